"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments before it touches the device."""
import ctypes
import glob
import os
import re

import pytest

from gated_delta_rule_27_gb300 import libkda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            text = f.read()
        names.update(re.findall(r"KDA_API\s+[\w\s\*]*?\b(kda_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    assert {"kda_prefill_chunked", "kda_decode_step", "kda_prefill_workspace_size", "kda_status_string",
            "kda_prefill_check"} <= _declared_symbols()


def test_library_exports_every_declared_symbol():
    lib = libkda.load()
    for name in sorted(_declared_symbols()):
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings():
    assert libkda.status_string(0) == "KDA_OK"
    assert libkda.status_string(2) == "KDA_ERR_UNSUPPORTED"
    assert libkda.status_string(99) == "KDA_ERR_UNKNOWN"


def test_workspace_size():
    n = libkda.kda_prefill_workspace_size(4096, 1, 16, 128, 128, libkda.KDA_BF16, 64)
    assert n > 0 and n % 256 == 0
    # grows with tokens and documents, zero for unsupported sizes
    assert libkda.kda_prefill_workspace_size(8192, 1, 16, 128, 128, libkda.KDA_BF16, 64) > n
    assert libkda.kda_prefill_workspace_size(4096, 9, 16, 128, 128, libkda.KDA_BF16, 64) > n
    assert libkda.kda_prefill_workspace_size(4096, 1, 16, 32, 32, libkda.KDA_BF16, 64) == 0
    assert libkda.kda_prefill_workspace_size(4096, 1, 16, 128, 64, libkda.KDA_BF16, 64) == 0
    assert libkda.kda_prefill_workspace_size(4096, 1, 16, 128, 128, libkda.KDA_BF16, 48) == 0
    assert libkda.kda_prefill_workspace_size(-1, 1, 16, 128, 128, libkda.KDA_BF16, 64) == 0
    assert libkda.kda_prefill_workspace_size(0, 0, 1, 16, 16, libkda.KDA_F32, 0) > 0


def _prefill_raw(**kw):
    args = dict(q=None, k=None, v=None, g=None, beta=None, cu=None, N=1, T=64, H=1, dk=16, dv=16, dt=0, L=16,
                S0=None, o=None, Sf=None, ws=None, wsb=0, stream=None)
    args.update(kw)
    return libkda.load().kda_prefill_chunked(*args.values())


def test_prefill_rejects_bad_arguments_on_the_host():
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    assert _prefill_raw(dk=32, dv=32) == libkda.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(dk=16, dv=64) == libkda.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(L=8) == libkda.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(H=0) == libkda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(T=-5) == libkda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(dt=7) == libkda.KDA_ERR_INVALID_ARG
    assert _prefill_raw() == libkda.KDA_ERR_INVALID_ARG  # null pointers
    ok = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, cu=fake, o=ctypes.c_void_p(2 << 20))
    assert _prefill_raw(**ok) == libkda.KDA_ERR_INVALID_ARG  # no workspace
    assert _prefill_raw(**ok, ws=ctypes.c_void_p(3 << 20), wsb=16) == libkda.KDA_ERR_INVALID_ARG  # too small
    mis = dict(ok, q=ctypes.c_void_p((1 << 20) + 4))
    assert _prefill_raw(**mis, ws=ctypes.c_void_p(3 << 20), wsb=1 << 30) == libkda.KDA_ERR_INVALID_ARG
    alias = dict(ok, o=fake)
    assert _prefill_raw(**alias, ws=ctypes.c_void_p(3 << 20), wsb=1 << 30) == libkda.KDA_ERR_INVALID_ARG


def test_decode_rejects_bad_arguments_on_the_host():
    lib = libkda.load()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.kda_decode_step(None, None, None, None, None, 0, 1, 128, 128, 1, None, None, None) == libkda.KDA_OK
    assert lib.kda_decode_step(None, None, None, None, None, 4, 1, 128, 128, 1, None, None, None) == \
        libkda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, 4, 1, 96, 96, 1, fake, fake, None) == \
        libkda.KDA_ERR_UNSUPPORTED
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, 4, 0, 128, 128, 1, fake, fake, None) == \
        libkda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_step(fake, fake, fake, fake, fake, 4, 1, 128, 128, 1, fake, fake, None) == \
        libkda.KDA_ERR_INVALID_ARG  # o aliases q


def test_testing_hooks_check_their_arguments():
    lib = libkda.load()
    assert lib.kda_testing_set_plan(5) == libkda.KDA_ERR_INVALID_ARG
    assert lib.kda_testing_set_fault(3, 0) == libkda.KDA_ERR_INVALID_ARG
    assert lib.kda_testing_set_fault(libkda.FAULT_NO_PUBLISH, -1) == libkda.KDA_ERR_INVALID_ARG
    assert lib.kda_testing_set_plan(libkda.PLAN_AUTO) == libkda.KDA_OK
    assert lib.kda_testing_set_fault(libkda.FAULT_NONE, 0) == libkda.KDA_OK
