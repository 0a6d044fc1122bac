"""The bounds-check build of the library (needs a GB300).

No sanitizer runs on the GPUs the library targets, so its recurrence kernels
can be built to check every index they compute (-DRNN_BOUNDS_CHECK ->
libsrnn_bc.so): global-memory element indices against their buffers' extents,
the main shared-memory offsets against the CTA's layout.  A failed check sets
RNN_ERR_BOUNDS in the call's status word and skips the access.

Ragged and edge-case shapes of every forward variant (one CTA per head, 2-, 8-
and 16-CTA clusters, the sLSTM hi + lo operand, fp32), of the backward, of the
host-memory forward (time chunks with ragged ends, direct reads of mapped host
Wx) and of the layer wavefront (per-chunk pointers into every layer's buffers)
run through that build in a child process (the library is chosen per process
by SRNN_BOUNDS_CHECK=1); every call must report a clean status, and every
output must equal, bit for bit, the normal build's on the same inputs (the
checks add no arithmetic).
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (cell, dtype, T, B, NH, Dh, CTAs per head (0: the plan's choice), training)
CASES = [
    ("lstm", "bf16", 9, 13, 3, 64, 0, False),
    ("lstm", "bf16", 7, 5, 2, 64, 1, True),
    ("gru", "bf16", 9, 5, 2, 128, 2, True),
    ("slstm", "bf16", 6, 3, 1, 256, 8, True),
    ("lstm", "bf16", 5, 9, 1, 768, 16, True),
    ("gru", "f32", 7, 3, 2, 32, 0, False),
    ("lstm", "f32", 11, 2, 1, 64, 0, False),
    ("slstm", "f32", 5, 3, 1, 64, 0, False),
]
# host-memory forward: (cell, dtype, T, B, NH, Dh, chunk (0: the plan's choice))
HOST_CASES = [
    ("lstm", "bf16", 37, 5, 2, 64, 7),
    ("gru", "bf16", 50, 8, 3, 128, 16),
    ("slstm", "bf16", 40, 4, 2, 256, 9),
    ("slstm", "bf16", 40, 4, 4, 256, 0),   # slow Wx stream: direct reads of host memory
    ("lstm", "f32", 33, 4, 1, 64, 10),
]
# layer wavefront: (cell, T, B, NH, Dh, Din, layers, chunk)
STACK_CASES = [
    ("lstm", 40, 10, 2, 64, 96, 2, 16),
    ("gru", 29, 9, 2, 32, 40, 3, 7),
    ("slstm", 24, 5, 2, 64, 128, 2, 10),
]

CHILD = r'''
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[3])
import sequential_rnn_gb300 as S
from synth import make_inputs, make_projection_inputs

cfg = json.loads(sys.argv[2])
out, stat = {}, {}
for i, (cell, dt, T, B, NH, Dh, cl, train) in enumerate(cfg["rec"]):
    d = make_inputs(cell, dt, T, B, NH, Dh, seed=100 + i, bias="normal0.1", states="random",
                    backward=train)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    dev = lambda k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda()
    Wx, R = dev("Wx").to(tdt), dev("R").to(tdt)
    sl = cell == "slstm"
    fw = S.forward(cell, Wx, R, dev("b"), dev("h0"), None if cell == "gru" else dev("c0"),
                   dev("n0") if sl else None, dev("m0") if sl else None, train=train,
                   cluster=cl, check=False)
    stat[f"{i}.fwd"] = S.rnn_read_status(fw["workspace"])
    for k in ("h_seq", "hT", "cT", "nT", "mT"):
        if k in fw:
            out[f"{i}.{k}"] = fw[k].float().cpu().numpy()
    if train:
        gr = S.backward(fw, R, dev("h0"), None if cell == "gru" else dev("c0"), dev("dh").to(tdt),
                        dev("dhT"), None if cell == "gru" else dev("dcT"),
                        n0=dev("n0") if sl else None, check=False)
        stat[f"{i}.bwd"] = S.rnn_read_status(gr["workspace"])
        for k in ("dWx", "dR", "db", "dh0", "dc0", "dn0"):
            if k in gr:
                out[f"{i}.{k}"] = gr[k].float().cpu().numpy()
for i, (cell, dt, T, B, NH, Dh, chunk) in enumerate(cfg["host"]):
    d = make_inputs(cell, dt, T, B, NH, Dh, seed=300 + i, bias="normal0.1", states="random")
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    dev = lambda k: torch.from_numpy(np.ascontiguousarray(d[k])).cuda()
    Wx_h = torch.from_numpy(np.ascontiguousarray(d["Wx"])).to(tdt).pin_memory()
    sl = cell == "slstm"
    fw = S.forward_host(cell, Wx_h, dev("R").to(tdt), dev("b"), dev("h0"),
                        None if cell == "gru" else dev("c0"), dev("n0") if sl else None,
                        dev("m0") if sl else None, chunk=chunk, check=False)
    torch.cuda.synchronize()
    stat[f"h{i}"] = S.rnn_read_status(fw["workspace"])
    for k in ("h_seq", "hT", "cT", "nT", "mT"):
        if k in fw:
            out[f"h{i}.{k}"] = fw[k].float().cpu().numpy()
for i, (cell, T, B, NH, Dh, Din, L, chunk) in enumerate(cfg["stack"]):
    G = 4 if cell != "gru" else 3
    d = NH * Dh
    p0 = make_projection_inputs(T * B, G * d, Din, seed=400 + i)
    Wi = [make_projection_inputs(1, G * d, d, seed=500 + 10 * i + l) for l in range(1, L)]
    rec = [make_inputs(cell, "bf16", 1, B, NH, Dh, seed=600 + 10 * i + l, bias="normal0.1",
                       states="random") for l in range(L)]
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    st = lambda k: cu(np.stack([r[k] for r in rec]))
    sl = cell == "slstm"
    try:
        o = S.stack_forward(cell, cu(p0["x"].reshape(T, B, Din)).bfloat16(), cu(p0["W"]).bfloat16(),
                            cu(np.stack([q["W"] for q in Wi])).bfloat16() if L > 1 else None,
                            cu(np.stack([p0["b"]] + [q["b"] for q in Wi])),
                            st("R").bfloat16(), st("b"), st("h0"), None if cell == "gru" else st("c0"),
                            st("n0") if sl else None, st("m0") if sl else None, chunk=chunk)
        torch.cuda.synchronize()
        stat[f"s{i}"] = 0
    except S.RnnError as e:
        stat[f"s{i}"] = e.status
        continue
    for k in ("h_seq", "hT", "cT", "nT", "mT"):
        if k in o:
            out[f"s{i}.{k}"] = o[k].float().cpu().numpy()
np.savez(sys.argv[1], **out)
with open(sys.argv[1] + ".json", "w") as f:
    json.dump(stat, f)
'''


def run_child(tmp_path, name, bounds_check):
    env = dict(os.environ)
    env.pop("SRNN_BOUNDS_CHECK", None)
    if bounds_check:
        env["SRNN_BOUNDS_CHECK"] = "1"
    path = str(tmp_path / f"{name}.npz")
    r = subprocess.run([sys.executable, "-c", CHILD, path, json.dumps({"rec": CASES, "host": HOST_CASES, "stack": STACK_CASES}), ROOT], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    with open(path + ".json") as f:
        stat = json.load(f)
    return dict(np.load(path)), stat


def test_bounds_check_build_is_clean_and_bitwise_equal(tmp_path):
    from sequential_rnn_gb300 import build
    build.build()
    build.build(bounds_check=True)
    ref, ref_stat = run_child(tmp_path, "normal", False)
    got, got_stat = run_child(tmp_path, "checked", True)
    n_calls = len(CASES) + sum(c[-1] for c in CASES) + len(HOST_CASES) + len(STACK_CASES)
    assert set(ref_stat) == set(got_stat) and len(got_stat) == n_calls
    assert all(v == 0 for v in ref_stat.values()), ref_stat
    bad = {k: v for k, v in got_stat.items() if v != 0}
    assert not bad, bad   # RNN_ERR_BOUNDS is 8
    assert set(ref) == set(got)
    for k in sorted(ref):
        assert np.array_equal(ref[k], got[k], equal_nan=True), k
