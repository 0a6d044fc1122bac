"""Oracle against the fixtures in tests/golden (CPU only).

* lstm_hand_T1.txt: one LSTM step worked by hand from the cell equations.
* *_tiny.json: regression fixtures written by tests/golden/make_golden.py
  (oracle only), guarding the oracle's arithmetic against silent change.
"""
import json
import os

import numpy as np
import pytest

from oracle import rnn_oracle as O

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_hand_worked_lstm_step():
    with open(os.path.join(GOLD, "lstm_hand_T1.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    for ln in rows:
        lhs, rhs = ln.split("|")
        wx = np.array([float(v) for v in lhs.split()]).reshape(1, 1, 1, 4)
        c_exp, h_exp = (float(v) for v in rhs.split())
        o = O.lstm_forward(wx, np.zeros((1, 1, 4)), np.zeros((1, 4)))
        assert o["cT"].item() == pytest.approx(c_exp, abs=1e-15)
        assert o["hT"].item() == pytest.approx(h_exp, abs=1e-15)


@pytest.mark.parametrize("cell", ["lstm", "gru", "slstm"])
def test_tiny_regression_fixture(cell):
    with open(os.path.join(GOLD, f"{cell}_tiny.json")) as f:
        fx = json.load(f)
    i = {k: np.array(v) for k, v in fx["inputs"].items()}
    fw = O.forward(cell, i["Wx"], i["R"], i["b"], i["h0"], i["c0"])
    bw = O.backward(cell, i["Wx"], i["R"], i["b"], i["h0"], i["c0"], dh_seq=i["dh"])
    got = {**{k: v for k, v in fw.items() if not k.startswith("_")}, **bw}
    for k, v in fx["outputs"].items():
        np.testing.assert_allclose(got[k], np.array(v), rtol=0, atol=1e-14, err_msg=k)
