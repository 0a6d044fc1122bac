"""Plant plausible mistakes in the oracle (on the CPU) and check the pins fail.

Each mutant patches one helper of the oracle for the duration of a test; the
pins of test_oracle_pins must then catch it.  This shows the pins are
sensitive to a dropped term, a wrong sign or index, or a transposed operand.
"""
import numpy as np
import pytest

from oracle import rnn_oracle as O
import tests.test_oracle_pins as P


def _swap_gates(orig):
    def split(x, G):
        parts = orig(x, G)
        parts[0], parts[1] = parts[1], parts[0]
        return parts
    return split


MUTANTS = {
    # gate order i <-> f
    "swap_gates": ("_split", lambda o: _swap_gates(o)),
    # sign error inside the sigmoid
    "sigmoid_sign": ("_sigmoid", lambda o: (lambda x: 1.0 / (1.0 + np.exp(x)))),
    # heads paired with the wrong recurrent matrix
    "head_index": ("_recurrent", lambda o: (lambda h, R: o(h, R[::-1]))),
    # recurrent term dropped
    "no_recurrence": ("_recurrent", lambda o: (lambda h, R: 0.0 * o(h, R))),
    # transposed gradient operand: R instead of R^T in the backward contraction
    "bwd_transpose": ("_recurrent_T",
                      lambda o: (lambda dp, R: o(dp, R[..., ::-1]))),
    # upstream gradient of the final cell state ignored (LSTM and sLSTM)
    "lstm_drops_dcT": ("lstm_backward", lambda o: (lambda *a, **k: o(*a, **{**k, "dcT": None}))),
    "slstm_drops_dcT": ("slstm_backward", lambda o: (lambda *a, **k: o(*a, **{**k, "dcT": None}))),
    # normaliser carry of the sLSTM backward started with the wrong sign
    "slstm_dn_sign": ("slstm_backward",
                      lambda o: (lambda *a, **k: o(*a, **{**k, "dnT": None if k.get("dnT") is None
                                                          else -np.asarray(k["dnT"])}))),
    # upstream gradient of the final hidden state ignored (every cell)
    "drops_dhT": ("_bwd_common", lambda o: (lambda Wx, R, dh_seq, dhT: o(Wx, R, dh_seq, None))),
}

PINS = {
    "fwd_torch": lambda: [P.test_forward_matches_torch(c) for c in ("lstm", "gru")],
    "bwd_torch": lambda: [P.test_backward_matches_torch_autograd(c) for c in ("lstm", "gru")],
    "closed": lambda: (P.test_lstm_R0_closed_form(), P.test_gru_R0_closed_form(),
                       P.test_slstm_R0_weighted_average(), P.test_T1_scalar_closed_forms()),
    "fd": lambda: [P.test_backward_finite_differences(c) for c in ("lstm", "gru", "slstm")],
    "chunks": lambda: [P.test_backward_composes_over_chunks(c) for c in ("lstm", "gru", "slstm")],
    "unstab": lambda: P.test_slstm_equals_unstabilised_form(),
    "stab_pair": lambda: P.test_slstm_stabilised_gate_pair_has_a_unit_member(),
}


def _caught(monkeypatch, name):
    attr, make = MUTANTS[name]
    monkeypatch.setattr(O, attr, make(getattr(O, attr)))
    failed = []
    for pin, fn in PINS.items():
        try:
            fn()
        except AssertionError:
            failed.append(pin)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(monkeypatch, name):
    failed = _caught(monkeypatch, name)
    assert failed, f"mutant {name} passed every pin"
