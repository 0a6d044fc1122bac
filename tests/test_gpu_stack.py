"""GPU parity of stacked layers run as a wavefront over time chunks (needs a GB300).

rnn_stack_fwd runs layer l's chunk c once layer l-1 has finished chunk c, each
layer on its own stream.  Checked against the fp64 oracle's layers run one
after the other (bf16 tolerance, 2e-2 as for one layer: the inner layers' h is
rounded to bf16 once, as in the oracle's inputs of the next layer it is not,
so the tolerance covers one rounding per layer), and against the single-layer
entry points chained by hand (bitwise: same kernels, same inputs).
"""
import numpy as np
import pytest
import torch

from oracle import rnn_oracle as O
from synth import make_inputs, make_projection_inputs, round_bf16

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def S():
    from sequential_rnn_gb300 import build
    build.build()
    import sequential_rnn_gb300 as S
    return S


def layers(cell, T, B, NH, Dh, Din, L, seed):
    """Seeded weights of L layers (bf16 values) and random initial states."""
    G = O.GATES[cell]
    d = NH * Dh
    p0 = make_projection_inputs(T * B, G * d, Din, seed=seed)
    Wi = [make_projection_inputs(1, G * d, d, seed=seed + 100 + l) for l in range(1, L)]
    rec = [make_inputs(cell, "bf16", 1, B, NH, Dh, seed=seed + 200 + l, bias="normal0.1",
                       states="random") for l in range(L)]
    w = {"x": p0["x"].reshape(T, B, Din), "W_ih0": p0["W"],
         "W_ih": np.stack([q["W"] for q in Wi]) if L > 1 else None,
         "b_ih": np.stack([p0["b"]] + [q["b"] for q in Wi]),
         "R": np.stack([r["R"] for r in rec]), "b": np.stack([r["b"] for r in rec])}
    for k in ("h0", "c0", "n0", "m0"):
        w[k] = np.stack([r[k] for r in rec])
    return w


def to_dev(w):
    g = {}
    for k, v in w.items():
        if v is None:
            g[k] = None
        elif k in ("x", "W_ih0", "W_ih", "R"):
            g[k] = torch.from_numpy(np.ascontiguousarray(v)).to("cuda", torch.bfloat16)
        else:
            g[k] = torch.from_numpy(np.ascontiguousarray(v)).to("cuda", torch.float32)
    return g


def run(S, cell, g, chunk, cluster=0):
    sl = cell == "slstm"
    out = S.stack_forward(cell, g["x"], g["W_ih0"], g["W_ih"], g["b_ih"], g["R"], g["b"],
                          g["h0"], g["c0"] if cell != "gru" else None, g["n0"] if sl else None,
                          g["m0"] if sl else None, chunk=chunk, cluster=cluster)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("cell,T,B,NH,Dh,Din,L,chunk", [
    ("lstm", 40, 10, 2, 64, 96, 2, 16),     # ragged last chunk
    ("lstm", 33, 3, 1, 128, 64, 3, 5),
    ("gru", 29, 9, 2, 32, 40, 3, 7),
    ("slstm", 24, 5, 2, 64, 128, 2, 10),
    ("lstm", 6, 2, 1, 256, 48, 1, 4),       # one layer
])
def test_stack_matches_oracle(S, cell, T, B, NH, Dh, Din, L, chunk):
    w = layers(cell, T, B, NH, Dh, Din, L, seed=T + L)
    out = run(S, cell, to_dev(w), chunk)
    ref = O.stack_forward(cell, w["x"], w["W_ih0"], w["W_ih"], w["b_ih"], w["R"], w["b"],
                          w["h0"], w["c0"], w["n0"], w["m0"])
    for k in ("h_seq", "hT", "cT"):
        if k not in out:
            continue
        got = out[k].float().cpu().numpy()
        err = np.abs(got - ref[k]).max()
        if cell == "slstm" and k == "cT":
            err /= max(np.abs(ref[k]).max(), 1.0)
        assert err <= TOL, (cell, k, err)


@pytest.mark.parametrize("cluster", [1, 4])
def test_stack_chunking_is_bitwise(S, cluster):
    """With the CTAs per head fixed, the time chunk changes the schedule only.

    (With cluster = 0 the plan may pick another split for another chunk, and
    the one-CTA and cluster kernels differ in the last bits.)"""
    w = layers("lstm", 37, 6, 2, 64, 64, 3, seed=4)
    g = to_dev(w)
    a = run(S, "lstm", g, chunk=37, cluster=cluster)
    b = run(S, "lstm", g, chunk=8, cluster=cluster)
    c = run(S, "lstm", g, chunk=1, cluster=cluster)
    for k in ("h_seq", "hT", "cT"):
        assert torch.equal(a[k], b[k]) and torch.equal(a[k], c[k]), k


def test_stack_equals_chained_single_layers(S):
    """Full-size head shape (12 x 64, B=16, T=1024, d_in=768), three layers:
    the wavefront equals input_proj -> forward chained layer by layer."""
    cell, T, B, NH, Dh, Din, L = "lstm", 1024, 16, 12, 64, 768, 3
    w = layers(cell, T, B, NH, Dh, Din, L, seed=9)
    g = to_dev(w)
    cs = S.rnn_plan(S.make_desc(cell, "bf16", T, B, NH, Dh), L)["cluster"]
    out = run(S, cell, g, chunk=128, cluster=cs)
    inp = g["x"]
    for l in range(L):
        W = g["W_ih0"] if l == 0 else g["W_ih"][l - 1]
        Wx = S.input_proj(inp, W, g["b_ih"][l]).view(T, B, NH, 4 * Dh)
        f = S.forward(cell, Wx, g["R"][l], g["b"][l], g["h0"][l], g["c0"][l], cluster=cs)
        assert torch.equal(f["hT"], out["hT"][l]) and torch.equal(f["cT"], out["cT"][l]), l
        inp = f["h_seq"].view(T, B, NH * Dh)
    torch.cuda.synchronize()
    assert torch.equal(f["h_seq"], out["h_seq"])


def test_stack_zero_length_copies_states(S):
    w = layers("gru", 1, 3, 2, 64, 32, 2, seed=5)
    g = to_dev(w)
    g["x"] = g["x"][:0]
    out = run(S, "gru", g, chunk=4)
    assert torch.equal(out["hT"], g["h0"])
