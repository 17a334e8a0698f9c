"""tcgen05 descriptor encodings (kda_tc.cuh) against torch, through a one-CTA GEMM self-test.

The operand images are built here in the K-major 128-byte-swizzled layout the
tensor-core prefill uses (64 bf16 of K per 128-byte row, 8-row atoms of
1024 bytes, 16-byte chunks XORed with the row index); the GPU multiplies
them with tcgen05.mma and the 128 x N fp32 accumulator must equal A @ B^T.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_27_gb300 import libkda

pytestmark = pytest.mark.gpu


def sw128_image(X):
    """[R, K] bf16 matrix -> bytes of K/64 panels of R rows x 128 bytes, 128B-swizzled."""
    R, K = X.shape
    bits = X.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    img = np.zeros(R * K, dtype=np.uint16)
    for p in range(K // 64):
        for m in range(R):
            for c in range(8):
                chunk = c ^ (m & 7)
                dst = (p * R * 128 + m * 128 + chunk * 16) // 2
                img[dst:dst + 8] = bits[m, p * 64 + c * 8:p * 64 + c * 8 + 8]
    return img


def step_offsets(R, K):
    return [(s // 4) * R * 128 + (s % 4) * 32 for s in range(K // 16)]


def desc_base(lbo, sbo, swizzle=2):
    return ((lbo >> 4) << 16) | ((sbo >> 4) << 32) | (1 << 46) | (swizzle << 61)


def idesc(M, N, a_mn=False, b_mn=False):
    return (1 << 4) | (1 << 7) | (1 << 10) | (int(a_mn) << 15) | (int(b_mn) << 16) | ((N >> 3) << 17) | \
        ((M >> 4) << 24)


def mn_image(X):
    """[R, K] bf16 matrix -> MN-major 128B-swizzled bytes: R/64 chunks, each K rows of 64 R-elements (128 B)."""
    R, K = X.shape
    bits = X.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    img = np.zeros(R * K, dtype=np.uint16)
    for j in range(R // 64):
        for k in range(K):
            for c in range(8):
                chunk = c ^ (k & 7)
                dst = (j * K * 128 + k * 128 + chunk * 16) // 2
                img[dst:dst + 8] = bits[j * 64 + c * 8:j * 64 + c * 8 + 8, k]
    return img


def _selftest_fn():
    fn = libkda.load().kda_internal_tc_gemm_selftest
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong,
                   ctypes.c_ulonglong, ctypes.c_uint, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                   ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fn


@pytest.mark.parametrize("N,K", [(16, 128), (32, 128), (64, 128), (64, 64), (128, 64), (32, 64)])
def test_kmajor_sw128_gemm(N, K):
    lib = libkda.load()
    fn = lib.kda_internal_tc_gemm_selftest
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong,
                   ctypes.c_ulonglong, ctypes.c_uint, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                   ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    M = 128
    gen = torch.Generator().manual_seed(N * 1000 + K)
    A = torch.randn((M, K), generator=gen).to(torch.bfloat16)
    B = torch.randn((N, K), generator=gen).to(torch.bfloat16)
    a_img = torch.from_numpy(sw128_image(A).view(np.int16)).cuda()
    b_img = torch.from_numpy(sw128_image(B).view(np.int16)).cuda()
    steps = K // 16
    a_off = (ctypes.c_int * steps)(*step_offsets(M, K))
    b_off = (ctypes.c_int * steps)(*step_offsets(N, K))
    out = torch.full((M, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(a_img.data_ptr(), a_img.numel() * 2, b_img.data_ptr(), b_img.numel() * 2, desc_base(16, 1024),
            desc_base(16, 1024), idesc(M, N), steps, a_off, b_off, N, out.data_ptr(), status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0
    ref = A.float() @ B.float().T
    err = (out.cpu() - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), (err, out.cpu()[:4, :8], ref[:4, :8])


@pytest.mark.parametrize("M,N,K", [(128, 64, 64), (128, 16, 64)])
def test_mn_major_a_operand(M, N, K):
    """A stored MN-major (M contiguous per K row, 64-element M chunks LBO apart, 8-row K groups SBO apart)."""
    fn = _selftest_fn()
    gen = torch.Generator().manual_seed(M + N + K)
    A = torch.randn((M, K), generator=gen).to(torch.bfloat16)
    B = torch.randn((N, K), generator=gen).to(torch.bfloat16)
    a_img = torch.from_numpy(mn_image(A).view(np.int16)).cuda()
    b_img = torch.from_numpy(sw128_image(B).view(np.int16)).cuda()
    steps = K // 16
    a_off = (ctypes.c_int * steps)(*[s * 2048 for s in range(steps)])
    b_off = (ctypes.c_int * steps)(*step_offsets(N, K))
    out = torch.full((M, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = fn(a_img.data_ptr(), a_img.numel() * 2, b_img.data_ptr(), b_img.numel() * 2, desc_base(K * 128, 1024),
            desc_base(16, 1024), idesc(M, N, a_mn=True), steps, a_off, b_off, N, out.data_ptr(), status.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(status.item()) == 0
    ref = A.float() @ B.float().T
    err = (out.cpu() - ref).abs().max().item()
    assert err <= 1e-3 * ref.abs().max().item(), (err, out.cpu()[:4, :8], ref[:4, :8])
