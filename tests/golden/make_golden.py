"""Write the regression fixtures in this folder.

Calls only the fp64 oracle (oracle/rnn_oracle.py) on tiny inputs that are
spelled out in the fixture itself, so a later change to the oracle's
arithmetic shows up as a diff here.  The inputs are fixed small dyadic-ish
values, not drawn from a generator, so the files do not depend on any RNG.
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
from oracle import rnn_oracle as O  # noqa: E402


def _vals(n, k):
    # deterministic small values in (-1, 1): ((i*k) mod 17 - 8) / 8
    return np.array([((i * k) % 17 - 8) / 8.0 for i in range(n)])


def case(cell, T=3, B=2, NH=2, Dh=2):
    G = O.GATES[cell]
    Wx = _vals(T * B * NH * G * Dh, 5).reshape(T, B, NH, G * Dh)
    R = 0.5 * _vals(NH * Dh * G * Dh, 7).reshape(NH, Dh, G * Dh)
    b = 0.25 * _vals(NH * G * Dh, 3).reshape(NH, G * Dh)
    h0 = 0.5 * _vals(B * NH * Dh, 11).reshape(B, NH, Dh)
    c0 = 0.5 * _vals(B * NH * Dh, 13).reshape(B, NH, Dh)
    dh = _vals(T * B * NH * Dh, 9).reshape(T, B, NH, Dh)
    inp = {"Wx": Wx, "R": R, "b": b, "h0": h0, "c0": c0, "dh": dh}
    fw = O.forward(cell, Wx, R, b, h0, c0)
    bw = O.backward(cell, Wx, R, b, h0, c0, dh_seq=dh)
    out = {k: v for k, v in fw.items() if not k.startswith("_")}
    out.update({k: v for k, v in bw.items()})
    return {"cell": cell, "source": "oracle/rnn_oracle.py (regression fixture)",
            "inputs": {k: v.tolist() for k, v in inp.items()},
            "outputs": {k: np.asarray(v).tolist() for k, v in out.items()}}


if __name__ == "__main__":
    for cell in ("lstm", "gru", "slstm"):
        with open(os.path.join(HERE, f"{cell}_tiny.json"), "w") as f:
            json.dump(case(cell), f, indent=1)
    print("written")
