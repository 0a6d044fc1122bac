"""rnn_fwd_noalloc against rnn_fwd (needs a GB300).

The no-allocation entry point serves callers that cannot allocate device
memory at call time (a serving process that reserved its whole budget up
front, a latency-critical loop that must not risk an allocation's implicit
synchronisation).  It must give the same outputs as the regular entry point,
call after call: its scratch array is shared and keeps the last call's
contents, so two calls in a row are checked.  Collected last on purpose.
"""
import numpy as np
import pytest
import torch

from synth import make_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 bar of the parity tests


@pytest.fixture(scope="module")
def S():
    from sequential_rnn_gb300 import build
    build.build()
    import sequential_rnn_gb300 as S
    return S


@pytest.mark.parametrize("cell,Dh,B,NH,T,cluster", [
    ("lstm", 64, 13, 3, 40, 0),     # one CTA per head slice
    ("slstm", 256, 5, 2, 30, 0),    # thread-block cluster per head
    ("gru", 128, 8, 2, 25, 4),
])
def test_noalloc_matches_rnn_fwd_twice(S, cell, Dh, B, NH, T, cluster):
    d = make_inputs(cell, "bf16", T, B, NH, Dh, seed=11, bias="normal0.1", states="random")
    dt = torch.bfloat16
    Wx = torch.from_numpy(d["Wx"]).to("cuda", dt)
    R = torch.from_numpy(d["R"]).to("cuda", dt)
    f = {k: torch.from_numpy(d[k]).to("cuda", torch.float32) for k in ("b", "h0", "c0", "n0", "m0")}
    n0 = f["n0"] if cell == "slstm" else None
    m0 = f["m0"] if cell == "slstm" else None
    ref = S.forward(cell, Wx, R, f["b"], f["h0"], f["c0"], n0, m0, cluster=cluster)
    desc = ref["desc"]
    for call in range(2):
        h_seq = torch.full_like(ref["h_seq"], float("nan"))
        hT = torch.full_like(ref["hT"], float("nan"))
        cT = torch.full_like(ref["hT"], float("nan")) if cell != "gru" else None
        nT = torch.full_like(ref["hT"], float("nan")) if cell == "slstm" else None
        mT = torch.full_like(ref["hT"], float("nan")) if cell == "slstm" else None
        st = S.rnn_fwd_noalloc(desc, Wx, R, f["b"], f["h0"], f["c0"], n0, m0, h_seq, hT, cT, nT,
                               mT, None)
        assert st == 0, S.rnn_status_str(st)
        torch.cuda.synchronize()
        for name, got in (("h_seq", h_seq), ("hT", hT), ("cT", cT), ("nT", nT)):
            if got is None:
                continue
            err = (got.float() - ref[name].float()).abs().max().item()
            assert np.isfinite(err) and err <= TOL, (call, name, err)
