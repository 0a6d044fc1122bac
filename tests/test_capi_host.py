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


def test_exports_no_undeclared_c_symbols(lib):
    """Every unmangled function the library exports is one the header declares."""
    import shutil
    import subprocess
    from sequential_rnn_gb300 import _lib
    if shutil.which("nm") is None:
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {f[2] for f in (l.split() for l in out.splitlines())
                if len(f) == 3 and f[1] == "T" and not f[2].startswith(("_", "cuda", "cu"))}
    assert exported == set(_declared_symbols()), exported ^ set(_declared_symbols())


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
    for s in range(9):
        assert lib.rnn_status_str(s) and lib.rnn_status_str(s) != b"unknown status"
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
    (dict(Dh=64, cluster=16), 2), (dict(cell=1, Dh=32, cluster=8), 2), (dict(dtype=0, cluster=2), 2),
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
    # no work and no workspace: nothing touches the device (with a workspace the
    # call clears its status word, a device write these made-up pointers must not get)
    assert _bwd(lib, _desc(B=0), ws=0) == 0


def test_empty_batch_is_noop(lib):
    assert _fwd(lib, _desc(B=0), ws=0) == 0
    assert _fwd(lib, _desc(NH=0), ws=0) == 0


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
    assert _proj(lib, M=0, x=0, Wx=0, ws=0) == 1            # the workspace is checked first


def _stack(lib, desc=None, L=2, Din=96, chunk=16, x=0x1000, W0=0x2000, W=0x3000, R=0x4000,
           h_seq=0x5000, ws=0x10000, ws_bytes=None, **fp):
    P = ctypes.c_void_p
    desc = desc or _desc()
    if ws_bytes is None:
        ws_bytes = lib.rnn_stack_workspace_size(ctypes.byref(desc), L if 1 <= L <= 8 else 1,
                                                max(chunk, 1))
    f = {k: (P(fp[k]) if fp.get(k) else None)
         for k in ("b_ih", "bias", "h0", "c0", "n0", "m0", "hT", "cT", "nT", "mT")}
    return lib.rnn_stack_fwd(ctypes.byref(desc), L, Din, chunk, P(x) if x else None,
                             P(W0) if W0 else None, P(W) if W else None, f["b_ih"],
                             P(R) if R else None, f["bias"], f["h0"], f["c0"], f["n0"], f["m0"],
                             P(h_seq) if h_seq else None, f["hT"], f["cT"], f["nT"], f["mT"],
                             P(ws) if ws else None, ws_bytes, None)


def test_stack_workspace_size(lib):
    d = _desc()  # LSTM bf16, see _desc
    T, B, NH, Dh = d.T, d.B, d.NH, d.Dh
    al = lambda v: (v + 255) // 256 * 256
    dd = NH * Dh
    tc = min(16, T)
    want = 256 + al((2 - 1) * T * B * dd * 2) + 2 * al(tc * B * 4 * dd * 2) + 2 * 2 * 2 * al(B * dd * 4)
    assert lib.rnn_stack_workspace_size(ctypes.byref(d), 2, 16) == want
    assert lib.rnn_stack_workspace_size(ctypes.byref(d), 0, 16) == 0
    assert lib.rnn_stack_workspace_size(ctypes.byref(d), 9, 16) == 0
    assert lib.rnn_stack_workspace_size(ctypes.byref(d), 2, -1) == 0


def test_stack_argument_checks(lib):
    assert _stack(lib, L=0, ws_bytes=1 << 30) == 1
    assert _stack(lib, L=9, ws_bytes=1 << 30) == 1
    assert _stack(lib, chunk=-1, ws_bytes=1 << 30) == 1
    assert _stack(lib, Din=0) == 1
    assert _stack(lib, Din=12) == 2                        # Din % 8
    assert _stack(lib, desc=_desc(dtype=0)) == 2           # bf16 only
    assert _stack(lib, desc=_desc(flags=1)) == 2           # no training stash
    assert _stack(lib, desc=_desc(Dh=48)) == 2
    assert _stack(lib, ws_bytes=256) == 1
    assert _stack(lib, ws=0) == 1
    assert _stack(lib, ws=0x10010) == 3
    assert _stack(lib, x=0) == 1
    assert _stack(lib, W=0) == 1                           # L > 1 needs W_ih
    assert _stack(lib, R=0) == 1
    assert _stack(lib, x=0x1008) == 3
    assert _stack(lib, W0=0x2004) == 3
    assert _stack(lib, h0=0x6002) == 3
    assert _stack(lib, desc=_desc(B=0), ws=0) == 0         # empty batch: no-op


def _plan(lib, L=1, sms=148, **kw):
    out = (ctypes.c_int32 * 5)()
    st = lib.rnn_plan(ctypes.byref(_desc(**kw)), L, sms, out)
    return st, list(out)


@pytest.mark.parametrize("cell,Dh,NH,B,T,want", [
    (0, 64, 12, 16, 1024, 4),    # LSTM 12 x 64: the 4-CTA cluster (measured best)
    (1, 128, 6, 8, 2048, 4),     # GRU 6 x 128
    (2, 256, 4, 4, 4096, 8),     # sLSTM 4 x 256 (hi + lo h)
    (0, 768, 1, 16, 1024, 16),   # LSTM 1 x 768: only the 16-CTA split fits on chip
    (1, 32, 8, 16, 512, 1),      # GRU 32: one CTA per head is fastest
    (2, 64, 12, 4, 512, 4),      # sLSTM 12 x 64 with 4 batch rows (hi + lo in one n8 tile)
    (2, 128, 6, 3, 512, 4),      # sLSTM 6 x 128, 3 batch rows
    (2, 64, 12, 16, 512, 2),     # sLSTM 12 x 64, 16 batch rows (hi + lo operands)
])
def test_plan_picks_measured_best(lib, cell, Dh, NH, B, T, want):
    st, out = _plan(lib, cell=cell, Dh=Dh, NH=NH, B=B, T=T)
    assert st == 0 and out[0] == want, out
    rows = 4 if cell == 2 and B <= 4 and Dh <= 256 else 8  # batch rows per CTA
    nb = (B + rows - 1) // rows
    assert out[2] == NH * nb * want and out[3] == -(-out[2] // 148)


def test_plan_respects_constraints_and_occupancy(lib):
    # every automatic plan splits the head into whole unit groups and legal clusters
    for cell in (0, 1, 2):
        for Dh in (32, 64, 128, 256, 768):
            for NH, B in ((1, 4), (12, 16), (64, 256)):
                st, out = _plan(lib, cell=cell, Dh=Dh, NH=NH, B=B, T=256)
                assert st == 0, (cell, Dh)
                cs = out[0]
                ug = 16 if (cell == 1 and (Dh > 128 or Dh // cs > 64)) else 8
                assert cs in (1, 2, 4, 8, 16) and Dh % cs == 0 and (Dh // cs) % ug == 0
                assert (Dh // cs) // ug * 32 <= 1024
                assert cs > 1 or Dh <= 128
    # many heads and batch rows: waves over the SMs favour one CTA per head
    assert _plan(lib, Dh=64, NH=64, B=256)[1][0] == 1
    # few SMs: the 4-CTA split would need 4 waves
    assert _plan(lib, Dh=64, NH=12, B=16, sms=24)[1][0] == 1
    # an explicit cluster size is kept, and an impossible one is rejected
    assert _plan(lib, Dh=64, cluster=8)[1][0] == 8
    assert _plan(lib, Dh=256, cluster=2)[0] == 2
    assert _plan(lib, dtype=0)[0] == 2


def test_plan_for_stacked_layers(lib):
    # three 12 x 64 layers: one CTA per head so the layers' recurrences run side by side
    st, out = _plan(lib, L=3, Dh=64, NH=12, B=16, T=1024)
    assert st == 0 and out[0] == 1 and out[1] in (64, 128, 256), out
    assert 3 * out[2] <= 148
    # the workspace size follows the planned chunk
    d = _desc(Dh=64, NH=12, B=16, T=1024)
    assert lib.rnn_stack_workspace_size(ctypes.byref(d), 3, 0) == \
        lib.rnn_stack_workspace_size(ctypes.byref(d), 3, out[1])


def _fwd_host(lib, desc=None, chunk=0, wx=0x1000, r=0x2000, hseq=0x3000, ws=0x10000,
              ws_bytes=None):
    P = ctypes.c_void_p
    desc = desc or _desc()
    if ws_bytes is None:
        ws_bytes = lib.rnn_fwd_host_workspace_size(ctypes.byref(desc), max(chunk, 0))
    return lib.rnn_fwd_host(ctypes.byref(desc), chunk, P(wx) if wx else None,
                            P(r) if r else None, None, None, None, None, None,
                            P(hseq) if hseq else None, None, None, None, None,
                            P(ws) if ws else None, ws_bytes, None)


def test_fwd_host_workspace_size(lib):
    d = _desc(T=100, B=4, NH=2, Dh=64)   # LSTM bf16
    al = lambda v: (v + 255) // 256 * 256
    rows = 4 * 2
    for chunk, tc in ((0, 64), (10, 10), (500, 100)):
        want = 256 + 2 * al(tc * rows * 4 * 64 * 2) + 2 * al(tc * rows * 64 * 2) + 2 * 2 * al(rows * 64 * 4)
        assert lib.rnn_fwd_host_workspace_size(ctypes.byref(d), chunk) == want, chunk
    assert lib.rnn_fwd_host_workspace_size(ctypes.byref(d), -2) == 0
    # the automatic chunk is T/8 steps (at least 64)
    d = _desc(T=2048, B=4, NH=2, Dh=64)
    tc = 256
    want = 256 + 2 * al(tc * rows * 4 * 64 * 2) + 2 * al(tc * rows * 64 * 2) + 2 * 2 * al(rows * 64 * 4)
    assert lib.rnn_fwd_host_workspace_size(ctypes.byref(d), 0) == want


def test_fwd_host_argument_checks(lib):
    assert _fwd_host(lib, chunk=-1, ws_bytes=1 << 30) == 1
    assert _fwd_host(lib, desc=_desc(flags=1)) == 2          # no training stash
    assert _fwd_host(lib, desc=_desc(Dh=48)) == 2
    assert _fwd_host(lib, ws=0) == 1
    assert _fwd_host(lib, ws_bytes=256) == 1
    assert _fwd_host(lib, ws=0x10010) == 3
    assert _fwd_host(lib, wx=0) == 1
    assert _fwd_host(lib, hseq=0) == 1
    assert _fwd_host(lib, r=0) == 1
    assert _fwd_host(lib, r=0x2008) == 3
    assert _fwd_host(lib, desc=_desc(B=0), ws=0) == 0


def test_fwd_host_direct_mode_arguments(lib):
    """chunk = RNN_HOST_DIRECT (-1): the workspace is the forward's status word;
    chunks below it are invalid; an empty batch is a no-op; pointers the driver
    does not report as mapped host memory are refused (here: no device at all)."""
    d = _desc(T=100, B=4, NH=2, Dh=64)
    assert lib.rnn_fwd_host_workspace_size(ctypes.byref(d), -1) == 256
    assert lib.rnn_fwd_host_workspace_size(ctypes.byref(d), -2) == 0
    assert _fwd_host(lib, chunk=-2) == 1
    assert _fwd_host(lib, desc=_desc(B=0), chunk=-1, ws=0) == 0
    assert _fwd_host(lib, chunk=-1) == 1


def test_binding_constants_match_the_header():
    """Every enum value and #define of include/rnn.h that the binding mirrors
    has the header's value (read from the header text)."""
    import os
    import re
    from sequential_rnn_gb300 import _lib as L
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "rnn.h")).read()
    def value(expr):  # integer literals and `a << b` only
        m = re.fullmatch(r"(\d+)\s*<<\s*(\d+)", expr.strip())
        return int(m.group(1)) << int(m.group(2)) if m else int(expr)

    vals = {}
    for name, expr in re.findall(r"\b(RNN_[A-Z0-9_]+)\s*=\s*([^,}/\n]+)", hdr):
        vals[name] = value(expr)
    for name, expr in re.findall(r"#define\s+(RNN_[A-Z0-9_]+)\s+\(?(-?\d+)\)?", hdr):
        vals[name] = int(expr)
    mirrored = {"RNN_LSTM": L.RNN_LSTM, "RNN_GRU": L.RNN_GRU, "RNN_SLSTM": L.RNN_SLSTM,
                "RNN_F32": L.RNN_F32, "RNN_BF16": L.RNN_BF16, "RNN_FLAG_TRAIN": L.RNN_FLAG_TRAIN,
                "RNN_FLAG_H_BF16": L.RNN_FLAG_H_BF16,
                "RNN_FLAG_TEST_TIMEOUT": L.RNN_FLAG_TEST_TIMEOUT,
                "RNN_HOST_DIRECT": L.RNN_HOST_DIRECT}
    for name, v in mirrored.items():
        assert vals[name] == v, name
    for code, name in L.STATUS.items():
        assert vals[name] == code, name


def test_long_slstm_768_needs_the_bf16_h_flag(lib):
    """sLSTM heads above 256 units take h as one bf16 operand, whose deviation
    from the exact recurrence grows with T: past 768 steps the call is refused
    unless the caller sets RNN_FLAG_H_BF16 (host check, every entry point)."""
    from sequential_rnn_gb300._lib import RNN_FLAG_H_BF16
    assert _plan(lib, cell=2, Dh=768, NH=1, B=16, T=768)[0] == 0
    assert _plan(lib, cell=2, Dh=768, NH=1, B=16, T=769)[0] == 2
    assert _plan(lib, cell=2, Dh=768, NH=1, B=16, T=769, flags=RNN_FLAG_H_BF16)[0] == 0
    assert _plan(lib, cell=2, Dh=256, NH=1, B=16, T=100000)[0] == 0   # hi + lo operand: no bound
    assert _plan(lib, cell=0, Dh=768, NH=1, B=16, T=100000)[0] == 0   # LSTM: contractive
    assert _fwd(lib, _desc(cell=2, Dh=768, NH=1, T=769)) == 2
    d = _desc(cell=2, Dh=768, NH=1, T=769)
    assert lib.rnn_fwd_noalloc(ctypes.byref(d), *([None] * 15)) == 2
