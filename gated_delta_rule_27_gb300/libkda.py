"""Python binding of libkda's C ABI (include/kda.h).

Argument marshalling only: every step of the recurrence runs in libkda's
CUDA kernels.  torch supplies device memory and streams.  There is no CPU or
PyTorch fallback: if libkda.so cannot be loaded, or a tensor is not on a CUDA
device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_BOUNDS = range(6)
KDA_F32, KDA_BF16 = 0, 1

SYMBOLS = ("kda_status_string", "kda_prefill_workspace_size", "kda_prefill_chunked", "kda_prefill_chunked_profiled",
           "kda_prefill_check", "kda_decode_step", "kda_prefill_chunked_noalloc", "kda_prefill_noalloc_check",
           "kda_decode_step_indexed", "kda_state_snapshot", "kda_state_restore", "kda_prefill_chunked_ex",
           "kda_decode_step_ex", "kda_short_conv_prefill", "kda_short_conv_decode")
# include/kda_testing.h (test hooks)
TESTING_SYMBOLS = ("kda_testing_set_plan", "kda_testing_set_fault")
PLAN_AUTO, PLAN_THREE, PLAN_CHAIN, PLAN_PIPE = -1, 0, 2, 3
FAULT_NONE, FAULT_NO_PUBLISH, FAULT_CHUNK_TABLE = 0, 1, 2
PREFILL_MAX_KERNELS = 4

_lib = None


class FusionOpts(ctypes.Structure):
    """kda_fusion_opts (include/kda.h): the fused q/k normalisation and gated output normalisation."""
    _fields_ = [("qk_l2norm", ctypes.c_int32), ("qk_eps", ctypes.c_float), ("out_gate", ctypes.c_void_p),
                ("out_weight", ctypes.c_void_p), ("out_eps", ctypes.c_float)]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, status_string(status)))


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libkda.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libkda.so is not built (%s); run gated_delta_rule_27_gb300.build" % _build.LIB)
    _lib = _declare(ctypes.CDLL(_build.LIB))
    return _lib


def load_debug() -> ctypes.CDLL:
    """Loads the bounds-checking build, libkda_debug.so (built on first use): the same C ABI, for tests."""
    _build.build(debug=True)
    return _declare(ctypes.CDLL(_build.DEBUG_LIB))


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Sets the argument and result types of libkda's entry points on a loaded library."""
    vp, i32, fp = ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
    lib.kda_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32, ctypes.c_int, i32]
    lib.kda_prefill_chunked.restype = ctypes.c_int
    lib.kda_prefill_chunked.argtypes = [vp, vp, vp, fp, fp, vp, i32, i32, i32, i32, i32, ctypes.c_int, i32,
                                        fp, vp, fp, vp, ctypes.c_size_t, vp]
    lib.kda_prefill_chunked_profiled.restype = ctypes.c_int
    lib.kda_prefill_chunked_profiled.argtypes = lib.kda_prefill_chunked.argtypes + [
        ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_char_p)]
    lib.kda_prefill_check.restype = ctypes.c_int
    lib.kda_prefill_check.argtypes = [vp, vp]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [vp, vp, vp, fp, fp, i32, i32, i32, i32, ctypes.c_int, fp, vp, vp]
    lib.kda_prefill_chunked_noalloc.restype = ctypes.c_int
    lib.kda_prefill_chunked_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_int,
                                                i32, vp, vp, vp, vp]
    lib.kda_prefill_noalloc_check.restype = ctypes.c_int
    lib.kda_prefill_noalloc_check.argtypes = [vp]
    lib.kda_prefill_chunked_ex.restype = ctypes.c_int
    lib.kda_prefill_chunked_ex.argtypes = lib.kda_prefill_chunked.argtypes + [ctypes.POINTER(FusionOpts)]
    lib.kda_decode_step_ex.restype = ctypes.c_int
    lib.kda_decode_step_ex.argtypes = lib.kda_decode_step.argtypes + [ctypes.POINTER(FusionOpts)]
    lib.kda_short_conv_prefill.restype = ctypes.c_int
    lib.kda_short_conv_prefill.argtypes = [vp, fp, vp, i32, i32, i32, i32, ctypes.c_int, fp, vp, fp, vp]
    lib.kda_short_conv_decode.restype = ctypes.c_int
    lib.kda_short_conv_decode.argtypes = [vp, fp, i32, i32, i32, ctypes.c_int, fp, vp, vp]
    lib.kda_decode_step_indexed.restype = ctypes.c_int
    lib.kda_decode_step_indexed.argtypes = [vp, vp, vp, fp, fp, vp, i32, i32, i32, i32, i32, ctypes.c_int, fp, vp,
                                            vp, vp]
    for name in ("kda_state_snapshot", "kda_state_restore"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = [fp, vp, i32, i32, i32, i32, i32, fp, vp, vp]
    lib.kda_testing_set_plan.restype = ctypes.c_int
    lib.kda_testing_set_plan.argtypes = [i32]
    lib.kda_testing_set_fault.restype = ctypes.c_int
    lib.kda_testing_set_fault.argtypes = [i32, ctypes.c_int64]
    return lib


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError("libkda takes bf16 or fp32 q/k/v, got %s" % t.dtype)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libkda takes device tensors; got a %s tensor" % t.device)
    if not t.is_contiguous():
        raise ValueError("libkda takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def kda_prefill_workspace_size(total_tokens: int, num_seqs: int, H: int, d_k: int, d_v: int, in_dtype: int,
                               chunk_size: int = 64) -> int:
    return int(load().kda_prefill_workspace_size(total_tokens, num_seqs, H, d_k, d_v, in_dtype, chunk_size))


def kda_prefill_chunked(q, k, v, g, beta, cu_seqlens, o, S0=None, S_final=None, workspace=None, chunk_size=64,
                        stream=None) -> None:
    """Calls kda_prefill_chunked on caller-owned device tensors (see include/kda.h)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if workspace is None:
        workspace = new_workspace(T, N, H, d_k, d_v, dt, chunk_size, q.device)
    rc = load().kda_prefill_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H,
                                    d_k, d_v, dt, chunk_size, _ptr(S0), _ptr(o), _ptr(S_final), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_chunked")


def kda_prefill_chunked_profiled(q, k, v, g, beta, cu_seqlens, o, events, S0=None, S_final=None, workspace=None,
                                 chunk_size=64, stream=None):
    """kda_prefill_chunked plus CUDA events around its kernels.

    `events` is a list of torch.cuda.Event (len >= PREFILL_MAX_KERNELS + 1,
    created with enable_timing=True and already initialised by a record).
    Returns the names of the launched kernels; events[i] precedes kernel i and
    events[len(names)] follows the last one.
    """
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if workspace is None:
        workspace = new_workspace(T, N, H, d_k, d_v, dt, chunk_size, q.device)
    n_ev = PREFILL_MAX_KERNELS + 1
    ev_arr = (ctypes.c_void_p * n_ev)(*[ctypes.c_void_p(e.cuda_event) for e in events[:n_ev]])
    n_k = ctypes.c_int32(0)
    names = (ctypes.c_char_p * PREFILL_MAX_KERNELS)()
    rc = load().kda_prefill_chunked_profiled(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T,
                                             H, d_k, d_v, dt, chunk_size, _ptr(S0), _ptr(o), _ptr(S_final),
                                             _ptr(workspace), workspace.numel() * workspace.element_size(),
                                             _stream(stream), ev_arr, ctypes.byref(n_k), names)
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_chunked_profiled")
    return [names[i].decode() for i in range(n_k.value)]


def kda_prefill_check(workspace, stream=None) -> int:
    return int(load().kda_prefill_check(_ptr(workspace), _stream(stream)))


def kda_prefill_noalloc_check(stream=None) -> int:
    return int(load().kda_prefill_noalloc_check(_stream(stream)))


def testing_set_plan(plan: int) -> None:
    """Test hook (include/kda_testing.h): force a launch plan of the tensor-core prefill (PLAN_AUTO restores)."""
    rc = load().kda_testing_set_plan(int(plan))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_testing_set_plan")


def testing_set_fault(fault: int, wait_limit_ns: int = 0) -> None:
    """Test hook (include/kda_testing.h): inject a fault and bound the flag waits (FAULT_NONE, 0 restores)."""
    rc = load().kda_testing_set_fault(int(fault), int(wait_limit_ns))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_testing_set_fault")


def kda_decode_step(q, k, v, g, beta, S_inout, o, stream=None) -> None:
    """Calls kda_decode_step on caller-owned device tensors (see include/kda.h)."""
    N, H, d_k = q.shape
    d_v = v.shape[2]
    rc = load().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), N, H, d_k, d_v, _dtype_code(q),
                                _ptr(S_inout), _ptr(o), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")


def fusion_opts(qk_l2norm=False, qk_eps=1e-6, out_gate=None, out_weight=None, out_eps=1e-6):
    """A kda_fusion_opts for the _ex entry points (None when nothing is fused)."""
    if not qk_l2norm and out_gate is None:
        return None
    return FusionOpts(1 if qk_l2norm else 0, float(qk_eps), _ptr(out_gate), _ptr(out_weight), float(out_eps))


def kda_prefill_chunked_ex(q, k, v, g, beta, cu_seqlens, o, S0=None, S_final=None, workspace=None, chunk_size=64,
                           stream=None, **fusion) -> None:
    """kda_prefill_chunked with the fused prologue / epilogue (keywords of fusion_opts)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    if workspace is None:
        workspace = new_workspace(T, N, H, d_k, d_v, dt, chunk_size, q.device)
    opts = fusion_opts(**fusion)
    rc = load().kda_prefill_chunked_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H,
                                       d_k, d_v, dt, chunk_size, _ptr(S0), _ptr(o), _ptr(S_final), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream),
                                       None if opts is None else ctypes.byref(opts))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_chunked_ex")


def kda_decode_step_ex(q, k, v, g, beta, S_inout, o, stream=None, **fusion) -> None:
    """kda_decode_step with the fused prologue / epilogue (keywords of fusion_opts)."""
    N, H, d_k = q.shape
    opts = fusion_opts(**fusion)
    rc = load().kda_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), N, H, d_k, v.shape[2],
                                   _dtype_code(q), _ptr(S_inout), _ptr(o), _stream(stream),
                                   None if opts is None else ctypes.byref(opts))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step_ex")


def kda_short_conv_prefill(x, w, cu_seqlens, y, conv_state=None, conv_state_out=None, stream=None) -> None:
    """kda_short_conv_prefill on x [T, C] (or [T, H, d], flattened), w [C, W]."""
    T = x.shape[0]
    C, W = w.shape
    rc = load().kda_short_conv_prefill(_ptr(x), _ptr(w), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, C, W,
                                       _dtype_code(x), _ptr(conv_state), _ptr(y), _ptr(conv_state_out),
                                       _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_short_conv_prefill")


def kda_short_conv_decode(x, w, conv_state, y, stream=None) -> None:
    """kda_short_conv_decode on x [N, C]: one token per sequence, conv_state [N, W - 1, C] rolled in place."""
    N = x.shape[0]
    C, W = w.shape
    rc = load().kda_short_conv_decode(_ptr(x), _ptr(w), N, C, W, _dtype_code(x), _ptr(conv_state), _ptr(y),
                                      _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_short_conv_decode")


def kda_decode_step_indexed(q, k, v, g, beta, seq_idx, S_pool, o, status=None, stream=None) -> None:
    """Calls kda_decode_step_indexed: one token for each listed pool slot (see include/kda.h)."""
    A, H, d_k = q.shape
    d_v = v.shape[2]
    rc = load().kda_decode_step_indexed(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(seq_idx), A,
                                        S_pool.shape[0], H, d_k, d_v, _dtype_code(q), _ptr(S_pool), _ptr(o),
                                        _ptr(status), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step_indexed")


def kda_state_snapshot(S_pool, seq_idx, S_saved, status=None, stream=None) -> None:
    """S_saved[i] = S_pool[seq_idx[i]] (kda_state_snapshot)."""
    num_slots, H, d_k, d_v = S_pool.shape
    rc = load().kda_state_snapshot(_ptr(S_pool), _ptr(seq_idx), seq_idx.numel(), num_slots, H, d_k, d_v,
                                   _ptr(S_saved), _ptr(status), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_state_snapshot")


def kda_state_restore(S_saved, seq_idx, S_pool, status=None, stream=None) -> None:
    """S_pool[seq_idx[i]] = S_saved[i] (kda_state_restore)."""
    num_slots, H, d_k, d_v = S_pool.shape
    rc = load().kda_state_restore(_ptr(S_saved), _ptr(seq_idx), seq_idx.numel(), num_slots, H, d_k, d_v,
                                  _ptr(S_pool), _ptr(status), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_state_restore")


def new_workspace(T, N, H, d_k, d_v, in_dtype, chunk_size, device) -> torch.Tensor:
    n = kda_prefill_workspace_size(T, N, H, d_k, d_v, in_dtype, chunk_size)
    if n == 0:
        raise KdaError(KDA_ERR_UNSUPPORTED, "kda_prefill_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def prefill(q, k, v, g, beta, cu_seqlens, S0=None, chunk_size=64, want_state=True, workspace=None, stream=None):
    """Allocates o (and S_final) with torch and runs kda_prefill_chunked; returns (o, S_final)."""
    T, H, d_k = q.shape
    N = cu_seqlens.numel() - 1
    o = torch.empty((T, H, v.shape[2]), dtype=v.dtype, device=q.device)
    S_final = torch.empty((N, H, d_k, v.shape[2]), dtype=torch.float32, device=q.device) if want_state else None
    kda_prefill_chunked(q, k, v, g, beta, cu_seqlens, o, S0=S0, S_final=S_final, workspace=workspace,
                        chunk_size=chunk_size, stream=stream)
    return o, S_final


def decode_step(q, k, v, g, beta, S_inout, stream=None):
    """Allocates o with torch, runs kda_decode_step (S_inout updated in place); returns o."""
    o = torch.empty_like(v)
    kda_decode_step(q, k, v, g, beta, S_inout, o, stream=stream)
    return o


NOALLOC_SCRATCH_BYTES = 64 << 20


def kda_prefill_chunked_noalloc(q, k, v, g, beta, cu_seqlens, o, S0=None, S_final=None, chunk_size=64,
                                stream=None) -> None:
    """Calls kda_prefill_chunked_noalloc: the prefill with the library's static scratch, no workspace argument.

    For callers that must not allocate device memory; see include/kda.h for
    the scratch limit and the rule that overlapping calls on one GPU race.
    """
    lib = load()
    T, H, d_k = q.shape
    N = cu_seqlens.numel() - 1
    rc = lib.kda_prefill_chunked_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, T, H,
                                         d_k, v.shape[2], _dtype_code(q), chunk_size, _ptr(S0), _ptr(o),
                                         _ptr(S_final), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_chunked_noalloc")
