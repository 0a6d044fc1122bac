"""GPU tests of the host-memory forward (rnn_fwd_host, needs a GB300).

Wx in pinned host memory, h_seq written back to host memory, the copies
pipelined with the recurrence over time chunks.  Every chunk continues from
the previous chunk's final state, so the results are bitwise those of one
rnn_fwd over the whole sequence (same launch plan), which is itself checked
against the fp64 oracle in the forward tests; one case here also compares
with the oracle directly.
"""
import numpy as np
import pytest
import torch

from oracle import rnn_oracle as O
from synth import make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from sequential_rnn_gb300 import build
    build.build()
    import sequential_rnn_gb300 as S
    return S


def both(S, d, chunk):
    cell = d["cell"]
    dt = torch.bfloat16 if d["dtype"] == "bf16" else torch.float32
    Wx_h = torch.from_numpy(np.ascontiguousarray(d["Wx"])).to(dt).pin_memory()
    R = torch.from_numpy(np.ascontiguousarray(d["R"])).to("cuda", dt)
    st = {k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda() for k in ("b", "h0", "c0", "n0", "m0")}
    sl = cell == "slstm"
    args = (R, st["b"], st["h0"], st["c0"] if cell != "gru" else None, st["n0"] if sl else None,
            st["m0"] if sl else None)
    ref = S.forward(cell, Wx_h.cuda(), *args)
    got = S.forward_host(cell, Wx_h, *args, chunk=chunk)
    torch.cuda.synchronize()
    return got, ref


@pytest.mark.parametrize("cell,dtype,Dh,B,NH,T,chunk", [
    ("lstm", "bf16", 64, 16, 12, 300, 0),     # automatic chunk (64 steps here)
    ("lstm", "bf16", 64, 5, 2, 37, 7),        # ragged last chunk
    ("gru", "bf16", 128, 8, 3, 50, 16),
    ("slstm", "bf16", 256, 4, 2, 40, 9),
    ("lstm", "f32", 64, 4, 1, 33, 10),
    ("gru", "bf16", 32, 3, 2, 12, 100),       # one chunk
    ("slstm", "bf16", 256, 4, 4, 40, 0),      # automatic: slow Wx stream -> direct reads
])
def test_fwd_host_equals_device_forward(S, cell, dtype, Dh, B, NH, T, chunk):
    d = make_inputs(cell, dtype, T, B, NH, Dh, seed=T + Dh, bias="normal0.1", states="random")
    got, ref = both(S, d, chunk)
    assert not got["h_seq"].is_cuda
    assert torch.equal(got["h_seq"], ref["h_seq"].cpu())
    for k in ("hT", "cT", "nT", "mT"):
        if k in ref:
            assert torch.equal(got[k], ref[k]), k


@pytest.mark.parametrize("cell,Dh,B,NH,T", [
    ("lstm", 64, 16, 12, 300), ("gru", 128, 5, 2, 41), ("slstm", 256, 4, 2, 40),
    ("slstm", 64, 9, 3, 17),
])
def test_fwd_host_direct_equals_device_forward(S, cell, Dh, B, NH, T):
    """RNN_HOST_DIRECT: the kernel streams Wx from and writes h_seq to the mapped
    pinned buffers; the arithmetic is the device forward's, bit for bit."""
    d = make_inputs(cell, "bf16", T, B, NH, Dh, seed=T + Dh + 1, bias="normal0.1", states="random")
    got, ref = both(S, d, S.RNN_HOST_DIRECT)
    assert torch.equal(got["h_seq"], ref["h_seq"].cpu())
    for k in ("hT", "cT", "nT", "mT"):
        if k in ref:
            assert torch.equal(got[k], ref[k]), k


def test_fwd_host_direct_rejects_unmapped_buffers(S):
    """Pageable host memory or device memory is refused before anything runs."""
    d = make_inputs("lstm", "bf16", 9, 3, 2, 64, seed=3)
    R = torch.from_numpy(d["R"]).to("cuda", torch.bfloat16)
    pageable = torch.from_numpy(d["Wx"]).to(torch.bfloat16)  # not pinned
    with pytest.raises(S.RnnError) as e:
        S.forward_host("lstm", pageable, R, chunk=S.RNN_HOST_DIRECT)
    assert "INVALID_ARG" in str(e.value)
    # device memory as the "host" h_seq, through the C ABI (the binding refuses it earlier)
    import ctypes
    from sequential_rnn_gb300 import _lib
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    desc = S.make_desc("lstm", "bf16", 9, 3, 2, 64)
    wx_pin = pageable.pin_memory()
    hs_dev = torch.empty((9, 3, 2, 64), dtype=torch.bfloat16, device="cuda")
    fin = [torch.empty((3, 2, 64), device="cuda") for _ in range(2)]
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st = _lib.load().rnn_fwd_host(ctypes.byref(desc), S.RNN_HOST_DIRECT, P(wx_pin), P(R), None, None,
                                  None, None, None, P(hs_dev), P(fin[0]), P(fin[1]), None, None,
                                  P(ws), 256, None)
    assert st == 1  # RNN_ERR_INVALID_ARG


def test_fwd_host_full_workload_against_oracle(S):
    d = workload_inputs("lstm_bf16_12x64_b16_t1024")
    got, _ = both(S, d, 0)
    ref = O.forward("lstm", d["Wx"], d["R"], d["b"], d["h0"], d["c0"])
    err = np.abs(got["h_seq"].float().numpy() - ref["h_seq"]).max()
    assert err <= 2e-2, err
