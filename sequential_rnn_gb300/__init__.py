"""sequential_rnn_gb300: head-wise LSTM / GRU / sLSTM recurrence on GB300 (sm_103a).

Python binding of the C ABI in include/rnn.h.  The functions named like the C
entry points (``rnn_fwd``, ``rnn_bwd``, ...) take torch tensors (or None) and
only marshal arguments: device pointers, sizes and the current CUDA stream.
``forward`` / ``backward`` additionally allocate the outputs with torch and
raise ``RnnError`` on a non-OK status.  Every step of the recurrence runs in
the library's CUDA kernels; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (CELLS, DTYPES, RNN_BF16, RNN_F32, RNN_FLAG_H_BF16, RNN_FLAG_TEST_TIMEOUT,
                   RNN_FLAG_TRAIN, RNN_HOST_DIRECT,
                   STATUS, rnn_desc_t)

__all__ = ["RnnError", "make_desc", "rnn_workspace_size", "rnn_stash_size", "rnn_fwd", "rnn_bwd",
           "rnn_read_status", "rnn_sync_floor", "rnn_fwd_config", "rnn_status_str", "rnn_fwd_noalloc",
           "rnn_input_proj", "rnn_stack_workspace_size", "rnn_stack_fwd", "forward", "backward",
           "input_proj", "stack_forward", "rnn_plan", "rnn_fwd_host_workspace_size",
           "rnn_fwd_host", "forward_host", "GATES"]

GATES = {"lstm": 4, "gru": 3, "slstm": 4}


class RnnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({rnn_status_str(status)})")


def make_desc(cell: str, dtype: str, T: int, B: int, NH: int, Dh: int, flags: int = 0,
              cluster: int = 0) -> rnn_desc_t:
    return rnn_desc_t(CELLS[cell], DTYPES[dtype], T, B, NH, Dh, flags, cluster)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if t.numel() and not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _host_ptr(t):
    """Pointer of a contiguous host (preferably pinned) tensor."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ------------------------------------------------------ C-named wrappers --
def rnn_status_str(status: int) -> str:
    return _lib.load().rnn_status_str(int(status)).decode()


def rnn_workspace_size(desc: rnn_desc_t, pass_: int = 0) -> int:
    return int(_lib.load().rnn_workspace_size(ctypes.byref(desc), int(pass_)))


def rnn_stash_size(desc: rnn_desc_t) -> int:
    return int(_lib.load().rnn_stash_size(ctypes.byref(desc)))


def rnn_fwd_config(desc: rnn_desc_t):
    out = (ctypes.c_int32 * 6)()
    st = _lib.load().rnn_fwd_config(ctypes.byref(desc), out)
    if st:
        raise RnnError(st, "rnn_fwd_config")
    return dict(zip(("grid", "threads", "cluster", "nb", "smem", "kernel_id"), list(out)))


def rnn_fwd(desc, Wx, R, bias, h0, c0, n0, m0, h_seq, hT, cT, nT, mT, stash, workspace,
            stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return int(_lib.load().rnn_fwd(
        ctypes.byref(desc), _ptr(Wx), _ptr(R), _ptr(bias), _ptr(h0), _ptr(c0), _ptr(n0), _ptr(m0),
        _ptr(h_seq), _ptr(hT), _ptr(cT), _ptr(nT), _ptr(mT), _ptr(stash), _ptr(workspace),
        ws_bytes, _stream(stream)))


def rnn_fwd_noalloc(desc, Wx, R, bias, h0, c0, n0, m0, h_seq, hT, cT, nT, mT, stash,
                    device_status=None, stream=None) -> int:
    """rnn_fwd without a workspace, for callers that must not allocate device memory.

    ``device_status``: None or an int32 tensor (device, or pinned host) whose
    first element receives the call's device status word (0 = OK) on the stream.
    """
    if device_status is None:
        sp = None
    elif device_status.dtype != torch.int32 or device_status.numel() < 1:
        raise ValueError("device_status must be an int32 tensor")
    elif device_status.is_cuda:
        sp = _ptr(device_status)
    else:
        sp = _host_ptr(device_status)
    return int(_lib.load().rnn_fwd_noalloc(
        ctypes.byref(desc), _ptr(Wx), _ptr(R), _ptr(bias), _ptr(h0), _ptr(c0), _ptr(n0), _ptr(m0),
        _ptr(h_seq), _ptr(hT), _ptr(cT), _ptr(nT), _ptr(mT), _ptr(stash), sp, _stream(stream)))


def rnn_bwd(desc, R, h0, c0, n0, h_seq, stash, dh_seq, dhT, dcT, dnT, dWx, dR, db, dh0, dc0, dn0,
            workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return int(_lib.load().rnn_bwd(
        ctypes.byref(desc), _ptr(R), _ptr(h0), _ptr(c0), _ptr(n0), _ptr(h_seq), _ptr(stash),
        _ptr(dh_seq), _ptr(dhT), _ptr(dcT), _ptr(dnT), _ptr(dWx), _ptr(dR), _ptr(db), _ptr(dh0),
        _ptr(dc0), _ptr(dn0), _ptr(workspace), ws_bytes, _stream(stream)))


def rnn_input_proj(M: int, N: int, K: int, x, W, bias, Wx, workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return int(_lib.load().rnn_input_proj(int(M), int(N), int(K), _ptr(x), _ptr(W), _ptr(bias),
                                          _ptr(Wx), _ptr(workspace), ws_bytes, _stream(stream)))


def rnn_stack_workspace_size(desc: rnn_desc_t, L: int, chunk: int) -> int:
    return int(_lib.load().rnn_stack_workspace_size(ctypes.byref(desc), int(L), int(chunk)))


def rnn_stack_fwd(desc, L, Din, chunk, x, W_ih0, W_ih, b_ih, R, bias, h0, c0, n0, m0, h_seq, hT,
                  cT, nT, mT, workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return int(_lib.load().rnn_stack_fwd(
        ctypes.byref(desc), int(L), int(Din), int(chunk), _ptr(x), _ptr(W_ih0), _ptr(W_ih),
        _ptr(b_ih), _ptr(R), _ptr(bias), _ptr(h0), _ptr(c0), _ptr(n0), _ptr(m0), _ptr(h_seq),
        _ptr(hT), _ptr(cT), _ptr(nT), _ptr(mT), _ptr(workspace), ws_bytes, _stream(stream)))


def rnn_plan(desc: rnn_desc_t, L: int = 1, sms: int = 0) -> dict:
    out = (ctypes.c_int32 * 5)()
    st = _lib.load().rnn_plan(ctypes.byref(desc), int(L), int(sms), out)
    if st:
        raise RnnError(st, "rnn_plan")
    return dict(zip(("cluster", "chunk", "ctas", "waves", "us"), list(out)))


def rnn_fwd_host_workspace_size(desc: rnn_desc_t, chunk: int = 0) -> int:
    return int(_lib.load().rnn_fwd_host_workspace_size(ctypes.byref(desc), int(chunk)))


def rnn_fwd_host(desc, chunk, Wx_host, R, bias, h0, c0, n0, m0, h_seq_host, hT, cT, nT, mT,
                 workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return int(_lib.load().rnn_fwd_host(
        ctypes.byref(desc), int(chunk), _host_ptr(Wx_host), _ptr(R), _ptr(bias), _ptr(h0),
        _ptr(c0), _ptr(n0), _ptr(m0), _host_ptr(h_seq_host), _ptr(hT), _ptr(cT), _ptr(nT),
        _ptr(mT), _ptr(workspace), ws_bytes, _stream(stream)))


def rnn_read_status(workspace, stream=None) -> int:
    v = ctypes.c_int(0)
    st = _lib.load().rnn_read_status(_ptr(workspace), _stream(stream), ctypes.byref(v))
    if st:
        raise RnnError(st, "rnn_read_status")
    return int(v.value)


def rnn_sync_floor(desc, iters: int, workspace, stream=None) -> int:
    ws_bytes = workspace.numel() * workspace.element_size()
    return int(_lib.load().rnn_sync_floor(ctypes.byref(desc), int(iters), _ptr(workspace), ws_bytes,
                                          _stream(stream)))


# ------------------------------------------------------- conveniences ----
def _dtype_name(t: torch.Tensor) -> str:
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float32:
        return "f32"
    raise TypeError(f"unsupported dtype {t.dtype}")


def forward(cell: str, Wx, R, bias=None, h0=None, c0=None, n0=None, m0=None, *, train=False,
            cluster=0, h_bf16=False, test_timeout=False, stream=None, check=True):
    """Allocate outputs and run rnn_fwd.  Wx [T,B,NH,G*Dh], R [NH,Dh,G*Dh].

    ``h_bf16`` sets RNN_FLAG_H_BF16 (sLSTM: h_{t-1} enters the contraction as
    one bf16 value instead of a hi + lo pair).
    """
    T, B, NH, _ = Wx.shape
    Dh = R.shape[1]
    flags = ((RNN_FLAG_TRAIN if train else 0) | (RNN_FLAG_TEST_TIMEOUT if test_timeout else 0)
             | (RNN_FLAG_H_BF16 if h_bf16 else 0))
    desc = make_desc(cell, _dtype_name(Wx), T, B, NH, Dh, flags, cluster)
    dev = Wx.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"desc": desc,
           "h_seq": torch.empty((T, B, NH, Dh), dtype=Wx.dtype, device=dev),
           "hT": torch.empty((B, NH, Dh), **f32)}
    if cell != "gru":
        out["cT"] = torch.empty((B, NH, Dh), **f32)
    if cell == "slstm":
        out["nT"] = torch.empty((B, NH, Dh), **f32)
        out["mT"] = torch.empty((B, NH, Dh), **f32)
    out["workspace"] = torch.zeros(max(rnn_workspace_size(desc, 0), 256), dtype=torch.uint8, device=dev)
    out["stash"] = (torch.empty(max(rnn_stash_size(desc) // 4, 1), **f32) if train else None)
    st = rnn_fwd(desc, Wx, R, bias, h0, c0, n0, m0, out["h_seq"], out["hT"], out.get("cT"),
                 out.get("nT"), out.get("mT"), out["stash"], out["workspace"], stream)
    if st:
        raise RnnError(st, "rnn_fwd")
    if check:
        dst = rnn_read_status(out["workspace"], stream)
        if dst:
            raise RnnError(dst, "rnn_fwd (device)")
    return out


def backward(fwd: dict, R, h0, c0, dh_seq, dhT=None, dcT=None, *, n0=None, dnT=None, stream=None,
             check=True):
    """Run rnn_bwd after ``forward(..., train=True)``; returns the gradients."""
    desc = fwd["desc"]
    T, B, NH, Dh = desc.T, desc.B, desc.NH, desc.Dh
    cell = {v: k for k, v in CELLS.items()}[desc.cell]
    G = GATES[cell]
    dev = R.device
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"dWx": torch.empty((T, B, NH, G * Dh), dtype=R.dtype, device=dev),
         "dR": torch.empty((NH, Dh, G * Dh), **f32), "db": torch.empty((NH, G * Dh), **f32),
         "dh0": torch.empty((B, NH, Dh), **f32)}
    if cell != "gru":
        g["dc0"] = torch.empty((B, NH, Dh), **f32)
    if cell == "slstm":
        g["dn0"] = torch.empty((B, NH, Dh), **f32)
    ws = torch.zeros(rnn_workspace_size(desc, 1), dtype=torch.uint8, device=dev)
    st = rnn_bwd(desc, R, h0, c0, n0, fwd["h_seq"], fwd["stash"], dh_seq, dhT, dcT, dnT, g["dWx"],
                 g["dR"], g["db"], g["dh0"], g.get("dc0"), g.get("dn0"), ws, stream)
    if st:
        raise RnnError(st, "rnn_bwd")
    if check:
        dst = rnn_read_status(ws, stream)
        if dst:
            raise RnnError(dst, "rnn_bwd (device)")
    g["workspace"] = ws
    return g


def input_proj(x, W, bias=None, *, stream=None, check=True):
    """Wx = x W^T + bias through rnn_input_proj.

    x [..., K] bf16, W [N, K] bf16, bias [N] fp32 or None -> [..., N] bf16.
    With x [T, B, d] and W [NH*G*Dh, d] the result, viewed as [T, B, NH, G*Dh],
    is forward()'s Wx.
    """
    K = x.shape[-1]
    N = W.shape[0]
    M = x.numel() // K if K else 0
    out = torch.empty(tuple(x.shape[:-1]) + (N,), dtype=torch.bfloat16, device=x.device)
    ws = torch.empty(256, dtype=torch.uint8, device=x.device)  # the call clears its status word
    st = rnn_input_proj(M, N, K, x, W, bias, out, ws, stream)
    if st:
        raise RnnError(st, "rnn_input_proj")
    if check:
        dst = rnn_read_status(ws, stream)
        if dst:
            raise RnnError(dst, "rnn_input_proj (device)")
    return out


def stack_forward(cell: str, x, W_ih0, W_ih, b_ih, R, bias=None, h0=None, c0=None, n0=None,
                  m0=None, *, chunk=0, cluster=0, stream=None, check=True):
    """L stacked layers through rnn_stack_fwd (layer wavefront over time chunks).

    x [T, B, Din] bf16; W_ih0 [G*d, Din]; W_ih [L-1, G*d, d] or None; b_ih [L, G*d];
    R [L, NH, Dh, G*Dh] bf16; bias [L, NH, G*Dh]; states [L, B, NH, Dh] fp32 or None.
    chunk = 0 and cluster = 0 let the plan search choose.  Returns the last
    layer's h_seq and every layer's final states.
    """
    T, B, Din = x.shape
    L, NH, Dh = R.shape[0], R.shape[1], R.shape[2]
    desc = make_desc(cell, "bf16", T, B, NH, Dh, 0, cluster)
    dev = x.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"h_seq": torch.empty((T, B, NH, Dh), dtype=torch.bfloat16, device=dev),
           "hT": torch.empty((L, B, NH, Dh), **f32)}
    if cell != "gru":
        out["cT"] = torch.empty((L, B, NH, Dh), **f32)
    if cell == "slstm":
        out["nT"] = torch.empty((L, B, NH, Dh), **f32)
        out["mT"] = torch.empty((L, B, NH, Dh), **f32)
    nbytes = rnn_stack_workspace_size(desc, L, chunk)
    # no zero fill needed: the call clears its status word and writes every
    # intermediate before reading it
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    st = rnn_stack_fwd(desc, L, Din, chunk, x, W_ih0, W_ih, b_ih, R, bias, h0, c0, n0, m0,
                       out["h_seq"], out["hT"], out.get("cT"), out.get("nT"), out.get("mT"), ws,
                       stream)
    if st:
        raise RnnError(st, "rnn_stack_fwd")
    if check:
        dst = rnn_read_status(ws, stream)
        if dst:
            raise RnnError(dst, "rnn_stack_fwd (device)")
    return out


def forward_host(cell: str, Wx_host, R, bias=None, h0=None, c0=None, n0=None, m0=None, *,
                 h_seq_host=None, chunk=0, cluster=0, workspace=None, stream=None, check=True):
    """rnn_fwd_host: Wx_host [T,B,NH,G*Dh] and h_seq in pinned host memory, the
    copies pipelined with the recurrence over time chunks.  R and the states
    live on the device.  Returns h_seq (host) and the final states (device)."""
    T, B, NH, _ = Wx_host.shape
    Dh = R.shape[1]
    desc = make_desc(cell, _dtype_name(Wx_host), T, B, NH, Dh, 0, cluster)
    dev = R.device
    f32 = dict(dtype=torch.float32, device=dev)
    if h_seq_host is None:
        h_seq_host = torch.empty((T, B, NH, Dh), dtype=Wx_host.dtype, pin_memory=True)
    out = {"desc": desc, "h_seq": h_seq_host, "hT": torch.empty((B, NH, Dh), **f32)}
    if cell != "gru":
        out["cT"] = torch.empty((B, NH, Dh), **f32)
    if cell == "slstm":
        out["nT"] = torch.empty((B, NH, Dh), **f32)
        out["mT"] = torch.empty((B, NH, Dh), **f32)
    need = max(rnn_fwd_host_workspace_size(desc, chunk), 256)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    out["workspace"] = workspace
    st = rnn_fwd_host(desc, chunk, Wx_host, R, bias, h0, c0, n0, m0, h_seq_host, out["hT"],
                      out.get("cT"), out.get("nT"), out.get("mT"), workspace, stream)
    if st:
        raise RnnError(st, "rnn_fwd_host")
    if check:
        dst = rnn_read_status(workspace, stream)
        if dst:
            raise RnnError(dst, "rnn_fwd_host (device)")
    return out
