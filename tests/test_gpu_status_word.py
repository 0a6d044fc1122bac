"""Every C-ABI call that launches nothing still leaves a clean status word (needs a GB300).

A caller may hand the library a workspace taken from a pool without clearing
it.  Each call that returns RNN_OK must leave its own device status in the
status word -- 0 when the call has no work (B, NH, T or M zero, or no
iterations) -- and never hand on what the memory held before.  The workspace
here starts with every bit set (the timeout bit included), so a call that
skips the clear reads as a timeout.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from sequential_rnn_gb300 import build
    build.build()
    import sequential_rnn_gb300 as S
    return S


def dirty(nbytes):
    return torch.full((max(nbytes, 256),), 0xFF, dtype=torch.uint8, device="cuda")


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("T,B", [(0, 3), (5, 0)])
@pytest.mark.parametrize("cell", ["lstm", "gru", "slstm"])
def test_forward_without_work(S, cell, T, B):
    desc = S.make_desc(cell, "bf16", T, B, 2, 64)
    ws = dirty(S.rnn_workspace_size(desc, 0) if B else 256)
    n = (B, 2, 64)
    st = S.rnn_fwd(desc, None, None, None, None, None, None, None, None, f32(*n), f32(*n),
                   f32(*n), f32(*n), None, ws)
    assert st == 0
    assert S.rnn_read_status(ws) == 0


@pytest.mark.parametrize("T,B", [(0, 3), (5, 0)])
def test_backward_without_work(S, T, B):
    desc = S.make_desc("lstm", "bf16", T, B, 2, 64, S.RNN_FLAG_TRAIN)
    ws = dirty(S.rnn_workspace_size(desc, 1) if B else 256)
    n = (B, 2, 64)
    dR, db = f32(2, 64, 256), f32(2, 256)
    st = S.rnn_bwd(desc, None, None, None, None, None, None, None, f32(*n), f32(*n), None, None,
                   dR, db, f32(*n), f32(*n), None, ws)
    assert st == 0
    assert S.rnn_read_status(ws) == 0


def test_input_projection_without_rows(S):
    ws = dirty(256)
    assert S.rnn_input_proj(0, 256, 64, None, None, None, None, ws) == 0
    assert S.rnn_read_status(ws) == 0


@pytest.mark.parametrize("T,B", [(0, 3), (5, 0)])
def test_stack_without_work(S, T, B):
    desc = S.make_desc("lstm", "bf16", T, B, 2, 64)
    ws = dirty(S.rnn_stack_workspace_size(desc, 2, 4) if B else 256)
    n = (2, B, 2, 64)
    st = S.rnn_stack_fwd(desc, 2, 64, 4, None, None, None, None, None, None, None, None, None,
                         None, None, f32(*n), f32(*n), None, None, ws)
    assert st == 0
    assert S.rnn_read_status(ws) == 0


@pytest.mark.parametrize("T,B", [(0, 3), (5, 0)])
def test_host_forward_without_work(S, T, B):
    desc = S.make_desc("gru", "bf16", T, B, 2, 64)
    ws = dirty(S.rnn_fwd_host_workspace_size(desc, 4) if B else 256)
    st = S.rnn_fwd_host(desc, 4, None, None, None, None, None, None, None, None, f32(B, 2, 64),
                        None, None, None, ws)
    assert st == 0
    assert S.rnn_read_status(ws) == 0


def test_sync_floor_without_iterations(S):
    desc = S.make_desc("lstm", "bf16", 8, 16, 12, 64)
    ws = dirty(256)
    assert S.rnn_sync_floor(desc, 0, ws) == 0
    assert S.rnn_read_status(ws) == 0
