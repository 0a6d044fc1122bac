"""GPU parity of the input projection Wx = x W^T + b (tcgen05 GEMM, needs a GB300).

Compared element by element with the fp64 oracle on the same bf16 inputs.
The kernel sums in fp32 and rounds once to bf16, so per element
    |got - ref| <= 2^-8 |ref| + 1e-5 max|ref|
(half a bf16 ulp is 2^-9 |ref|; the fp32 sum error over K <= 4096 terms is far
below the absolute term).
"""
import numpy as np
import pytest
import torch

from oracle import rnn_oracle as O
from synth import make_inputs, make_projection_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from sequential_rnn_gb300 import build
    build.build()
    import sequential_rnn_gb300 as S
    return S


def dev(d):
    return (torch.from_numpy(d["x"]).to("cuda", torch.bfloat16),
            torch.from_numpy(d["W"]).to("cuda", torch.bfloat16),
            torch.from_numpy(d["b"]).to("cuda"))


def check(got, ref, label):
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), label
    tol = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max()
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (label, int(bad.sum()), float(np.abs(got - ref).max()))


@pytest.mark.parametrize("M,N,K", [
    (128, 128, 64),        # one tile, one k block
    (300, 208, 72),        # ragged rows, a partial column tile, a K tail of 8
    (1, 16, 8),            # smallest shape
    (257, 384, 1000),      # many k blocks, K tail
    (2048, 3072, 768),     # the 12 x 64 LSTM's projection at T*B = 2048
    (16384, 256, 64),      # 256-wide pair tiles (192-wide ones would leave pairs two tiles)
    (4096, 3072, 256),     # 192 pair tiles over 76 pairs: uneven waves, too many to split
    (2048, 2944, 64),      # 96 tiles: the last 20 run as halves, one half wholly past N
    (1280, 3904, 200),     # 80 tiles: the last 4 run as halves, one wholly past N; K tail
    (2048, 1024, 2048),    # K >= 2048: two pairs per cluster share x (multicast)
    (1000, 1536, 2104),    # the same with ragged rows and a K tail
    (5120, 1024, 2048),    # 40 two-pair units: more than one wave, the last ones as halves
])
def test_input_proj_matches_oracle(S, M, N, K):
    d = make_projection_inputs(M, N, K, seed=M + N + K)
    x, W, b = dev(d)
    got = S.input_proj(x, W, b)
    torch.cuda.synchronize()
    check(got, O.input_projection(d["x"], d["W"], d["b"]), f"{M}x{N}x{K}")


def test_input_proj_without_bias_and_batched_shape(S):
    d = make_projection_inputs(5 * 7, 96, 40, seed=3)
    x, W, _ = dev(d)
    got = S.input_proj(x.view(5, 7, 40), W)
    torch.cuda.synchronize()
    assert got.shape == (5, 7, 96)
    check(got.view(35, 96), O.input_projection(d["x"], d["W"]), "no bias")


def test_input_proj_full_size_sampled_rows(S):
    """T*B = 16384 rows of a d = 768 input onto 12 heads x 4 gates x 64: sampled rows."""
    M, N, K = 16384, 3072, 768
    d = make_projection_inputs(M, N, K, seed=11)
    x, W, b = dev(d)
    got = S.input_proj(x, W, b)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(M, 96, replace=False)
    # + rows of the last m tile, whose last eight tiles run as half tiles on 76 pairs
    rows = np.concatenate([rows, [0, 127, 128, M - 256, M - 129, M - 1]])
    ref = O.input_projection(d["x"][rows], d["W"], d["b"])
    check(got[torch.from_numpy(rows).cuda()], ref, "full size")


def test_projection_feeds_the_recurrence(S):
    """input_proj -> forward equals the oracle's projection -> recurrence."""
    T, B, NH, Dh, Din = 20, 6, 2, 64, 96
    p = make_projection_inputs(T * B, NH * 4 * Dh, Din, seed=21)
    r = make_inputs("lstm", "bf16", T, B, NH, Dh, seed=22, bias="forget1", states="random")
    x, W, bW = dev(p)
    Wx = S.input_proj(x.view(T, B, Din), W, bW).view(T, B, NH, 4 * Dh)
    g = {k: torch.from_numpy(np.ascontiguousarray(r[k])).cuda() for k in ("b", "h0", "c0")}
    R = torch.from_numpy(r["R"]).to("cuda", torch.bfloat16)
    out = S.forward("lstm", Wx, R, g["b"], g["h0"], g["c0"])
    torch.cuda.synchronize()
    Wx_ref = O.input_projection(p["x"], p["W"], p["b"]).reshape(T, B, NH, 4 * Dh)
    ref = O.forward("lstm", Wx_ref, r["R"], r["b"], r["h0"], r["c0"])
    err = np.abs(out["h_seq"].float().cpu().numpy() - ref["h_seq"]).max()
    assert err <= 2e-2, err
