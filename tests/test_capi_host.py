"""C ABI host-side checks that need no GPU.

The library loads, exports every entry point include/rnn.h declares, and its
argument checks reject bad calls before touching CUDA (fake, never
dereferenced pointer values are fine here because validation fails first).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sequential_rnn_gb300 import build, _lib
    build.build()
    return _lib.load()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "rnn.h")).read()
    return sorted(set(re.findall(r"\b(rnn_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    from sequential_rnn_gb300 import _lib
    declared = _declared_symbols()
    assert set(declared) == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def _desc(**kw):
    from sequential_rnn_gb300._lib import rnn_desc_t
    d = dict(cell=0, dtype=1, T=8, B=4, NH=2, Dh=64, flags=0, cluster=0)
    d.update(kw)
    return rnn_desc_t(**d)


def _fwd(lib, desc, ws=0x1000, ws_bytes=256, wx=0x2000, r=0x3000, hseq=0x4000, stash=None):
    P = ctypes.c_void_p
    return lib.rnn_fwd(ctypes.byref(desc), P(wx), P(r), None, None, None, None, None, P(hseq),
                       None, None, None, None, P(stash) if stash else None, P(ws), ws_bytes, None)


def test_status_strings(lib):
    for s in range(8):
        assert lib.rnn_status_str(s)
    assert lib.rnn_status_str(99) == b"unknown status"


def test_sizes(lib):
    d = _desc(T=10, B=3, NH=2, Dh=64)
    assert lib.rnn_workspace_size(ctypes.byref(d), 0) >= 256
    assert lib.rnn_workspace_size(ctypes.byref(d), 1) >= 256 + 3 * 2 * 64 * 2
    assert lib.rnn_stash_size(ctypes.byref(d)) == 10 * 3 * 2 * 64 * 5 * 4
    assert lib.rnn_stash_size(ctypes.byref(_desc(cell=1, T=10, B=3, NH=2))) == 10 * 3 * 2 * 64 * 5 * 4
    assert lib.rnn_stash_size(ctypes.byref(_desc(cell=2, T=10, B=3, NH=2))) == 10 * 3 * 2 * 64 * 6 * 4
    gru = _desc(cell=1, T=10, B=3, NH=2, Dh=64)
    assert lib.rnn_workspace_size(ctypes.byref(gru), 1) >= 10 * 3 * 2 * 192 * 2
    assert lib.rnn_workspace_size(ctypes.byref(_desc(T=-1)), 0) == 0
    assert lib.rnn_workspace_size(None, 0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(cell=7), 1), (dict(dtype=5), 1), (dict(T=-1), 1), (dict(B=-2), 1), (dict(Dh=0), 1),
    (dict(cluster=-1), 1),
    (dict(Dh=48), 2), (dict(dtype=0, Dh=128), 2), (dict(Dh=512), 2), (dict(cluster=3), 2),
    (dict(Dh=64, cluster=16), 2), (dict(cell=1, Dh=64, cluster=8), 2), (dict(dtype=0, cluster=2), 2),
])
def test_invalid_descriptors(lib, kw, status):
    assert _fwd(lib, _desc(**kw)) == status


def test_null_and_small_workspace(lib):
    assert lib.rnn_fwd(None, *([None] * 14), 0, None) == 1
    assert _fwd(lib, _desc(), ws=0) == 1
    assert _fwd(lib, _desc(), ws_bytes=8) == 1
    assert _fwd(lib, _desc(), wx=0) == 1
    assert _fwd(lib, _desc(), hseq=0) == 1


def test_misaligned_pointers(lib):
    assert _fwd(lib, _desc(), wx=0x2008) == 3
    assert _fwd(lib, _desc(), r=0x3002) == 3
    assert _fwd(lib, _desc(), ws=0x1004) == 3


def test_train_flag_rules(lib):
    assert _fwd(lib, _desc(flags=1)) == 1                      # no stash
    assert _fwd(lib, _desc(cell=1, flags=1)) == 1
    assert _fwd(lib, _desc(dtype=0, flags=1), stash=0x5000) == 2  # training is bf16 only


def _bwd(lib, desc, ws=0x1000, ws_bytes=1 << 30, **ptr):
    P = ctypes.c_void_p
    names = ["R", "h0", "c0", "n0", "h_seq", "stash", "dh_seq", "dhT", "dcT", "dnT", "dWx", "dR",
             "db", "dh0", "dc0", "dn0"]
    base = dict(R=0x3000, h_seq=0x4000, stash=0x5000, dh_seq=0x6000, dWx=0x7000)
    base.update(ptr)
    args = [P(base[n]) if base.get(n) else None for n in names]
    return lib.rnn_bwd(ctypes.byref(desc), *args, P(ws) if ws else None, ws_bytes, None)


def test_backward_argument_checks(lib):
    assert _bwd(lib, _desc(dtype=0)) == 2                  # bf16 only
    assert _bwd(lib, _desc(Dh=48)) == 2
    assert _bwd(lib, _desc(), ws=0) == 1
    assert _bwd(lib, _desc(), ws_bytes=16) == 1
    assert _bwd(lib, _desc(), ws=0x1010) == 3               # workspace 256-aligned
    assert _bwd(lib, _desc(), stash=0) == 1
    assert _bwd(lib, _desc(cell=2), dWx=0x7008) == 3
    assert _bwd(lib, _desc(B=0)) == 0


def test_empty_batch_is_noop(lib):
    assert _fwd(lib, _desc(B=0)) == 0
    assert _fwd(lib, _desc(NH=0)) == 0


def _proj(lib, M=300, N=3072, K=768, x=0x1000, W=0x2000, bias=0, Wx=0x3000, ws=0x8000,
          ws_bytes=256):
    P = ctypes.c_void_p
    return lib.rnn_input_proj(M, N, K, P(x) if x else None, P(W) if W else None,
                              P(bias) if bias else None, P(Wx) if Wx else None,
                              P(ws) if ws else None, ws_bytes, None)


def test_input_proj_argument_checks(lib):
    assert _proj(lib, M=-1) == 1
    assert _proj(lib, N=0) == 1
    assert _proj(lib, K=0) == 1
    assert _proj(lib, ws=0) == 1
    assert _proj(lib, ws_bytes=128) == 1
    assert _proj(lib, ws=0x8010) == 3                       # workspace 256-aligned
    assert _proj(lib, K=12) == 2                            # K % 8
    assert _proj(lib, N=200) == 2                           # N % 16
    assert _proj(lib, M=65535 * 128 + 1) == 2
    assert _proj(lib, x=0) == 1
    assert _proj(lib, Wx=0) == 1
    assert _proj(lib, x=0x1008) == 3
    assert _proj(lib, W=0x2004) == 3
    assert _proj(lib, Wx=0x3002) == 3
    assert _proj(lib, bias=0x4002) == 3
    assert _proj(lib, M=0, x=0, Wx=0) == 0                  # empty input: no-op
