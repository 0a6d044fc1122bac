"""fp64 CPU oracle for the head-wise RNN recurrence (LSTM, GRU, sLSTM).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, the smoke check of ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA path; the two meet
only through the seeded inputs of the ``synth`` module.

What it computes (the FlashRNN pages, "FlashRNN: I/O-Aware Optimization of
Traditional RNNs on modern hardware", abstract, and the blog page "From a GPU
programming perspective, re-examining RNNs", paragraphs on register caching
and head-wise splitting):

* NH independent heads, each a small RNN with its own recurrent matrix
  R[h] of shape [Dh, G*Dh]; together they are one RNN whose recurrent matrix
  is block-diagonal (blog page, head-wise parallelisation paragraph).
* Per step t and head h the recurrent preactivation is
      pre_t = Wx_t + h_{t-1} @ R[h] + b[h]          (row-vector convention)
  where Wx_t is the precomputed input projection (the kernels consume it).
* Gate-major packing: column g*Dh + j of a G*Dh row is gate g of unit j.

The pages name the cells but print no equations; the plainest textbook
readings are used, written out below in the order the recurrence applies them:

* LSTM  (gates i, f, z, o):  i,f,o = sigmoid, z = tanh;
        c_t = f*c_{t-1} + i*z;  h_t = o*tanh(c_t).
* GRU   (gates r, z, n; PyTorch convention): with rec = h_{t-1} @ R + b,
        r = sigmoid(Wx_r + rec_r), z = sigmoid(Wx_z + rec_z),
        n = tanh(Wx_n + r*rec_n),  h_t = (1-z)*n + z*h_{t-1}.
* sLSTM (gates i, f, z, o; exponential input/forget gates, stabiliser m):
        m_t = max(f~ + m_{t-1}, i~),  i = exp(i~ - m_t),
        f = exp(f~ + m_{t-1} - m_t),  c_t = f*c + i*tanh(z~),
        n_t = f*n + i,  h_t = sigmoid(o~) * c_t / n_t.

Backward passes are textbook backpropagation through time of exactly these
forward graphs (the sLSTM stabiliser m is a reparametrisation the output h does
not depend on, so it is held at its forward values and carries no gradient).

The input projection that produces Wx from an input sequence x (the dense
step in front of the recurrence; the blog page's register-caching paragraph
separates the recurrent weight, kept on chip through the time loop, from the
input weight applied to all steps at once) is the plain definition
``Wx = x @ W^T + b``.

Everything is fp64 numpy; a library batched matmul is the only "primitive".
Optionally ``emulate_bf16_h`` rounds h_{t-1} to bf16 before the contraction,
mirroring a bf16 MMA operand, and (sLSTM) ``emulate_bf16_pair_h`` replaces it
by bf16(h) + bf16(h - bf16(h)), the two-part operand; both are diagnosis aids,
parity is checked against the plain fp64 run.
"""
from __future__ import annotations

import numpy as np

__all__ = ["GATES", "forward", "backward", "lstm_forward", "gru_forward",
           "slstm_forward", "lstm_backward", "gru_backward", "slstm_backward",
           "input_projection", "stack_forward"]

GATES = {"lstm": 4, "gru": 3, "slstm": 4}


# ----------------------------------------------------------------- helpers --
def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _recurrent(h_prev, R):
    """h_prev [B,NH,Dh] @ R [NH,Dh,G*Dh] per head -> [B,NH,G*Dh] (batched matmul)."""
    return np.matmul(h_prev.transpose(1, 0, 2), R).transpose(1, 0, 2)


def _recurrent_T(dpre, R):
    """dpre [B,NH,G*Dh] @ R[h]^T per head -> [B,NH,Dh] (batched matmul)."""
    return np.matmul(dpre.transpose(1, 0, 2), R.transpose(0, 2, 1)).transpose(1, 0, 2)


def _outer_sum(h_prev, dpre):
    """sum_b h_prev[b,h,:]^T dpre[b,h,:] per head -> [NH,Dh,G*Dh] (batched matmul)."""
    return np.matmul(h_prev.transpose(1, 2, 0), dpre.transpose(1, 0, 2))


def _split(x, G):
    """Split the last (gate-major) axis into G gate blocks."""
    return np.split(x, G, axis=-1)


def _to_bf16_f64(x):
    """Round fp64 values to the nearest bf16 (ties to even), back to fp64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _prep(Wx, R, b, states, names, Dh):
    Wx = np.asarray(Wx, np.float64)
    R = np.asarray(R, np.float64)
    T, B, NH, _ = Wx.shape
    b = np.zeros((NH, R.shape[2])) if b is None else np.asarray(b, np.float64)
    st = []
    for nm in names:
        v = states.get(nm)
        st.append(np.zeros((B, NH, Dh)) if v is None else np.array(v, np.float64))
    return Wx, R, b, st


# ----------------------------------------------------------------- forward --
def lstm_forward(Wx, R, b=None, h0=None, c0=None, emulate_bf16_h=False, keep=False):
    Dh = R.shape[1]
    Wx, R, b, (h, c) = _prep(Wx, R, b, {"h0": h0, "c0": c0}, ("h0", "c0"), Dh)
    T = Wx.shape[0]
    h_seq = np.empty(Wx.shape[:3] + (Dh,))
    saved = []
    for t in range(T):
        hin = _to_bf16_f64(h) if emulate_bf16_h else h
        pre = Wx[t] + _recurrent(hin, R) + b
        gi, gf, gz, go = _split(pre, 4)
        i, f, z, o = _sigmoid(gi), _sigmoid(gf), np.tanh(gz), _sigmoid(go)
        c_prev = c
        c = f * c + i * z
        h_prev = h
        h = o * np.tanh(c)
        h_seq[t] = h
        if keep:
            saved.append((h_prev, c_prev, i, f, z, o, c))
    out = {"h_seq": h_seq, "hT": h, "cT": c}
    if keep:
        out["_saved"] = saved
    return out


def gru_forward(Wx, R, b=None, h0=None, emulate_bf16_h=False, keep=False):
    Dh = R.shape[1]
    Wx, R, b, (h,) = _prep(Wx, R, b, {"h0": h0}, ("h0",), Dh)
    T = Wx.shape[0]
    h_seq = np.empty(Wx.shape[:3] + (Dh,))
    saved = []
    for t in range(T):
        hin = _to_bf16_f64(h) if emulate_bf16_h else h
        rec = _recurrent(hin, R) + b
        xr, xz, xn = _split(Wx[t], 3)
        rr, rz, rn = _split(rec, 3)
        r = _sigmoid(xr + rr)
        z = _sigmoid(xz + rz)
        n = np.tanh(xn + r * rn)
        h_prev = h
        h = (1.0 - z) * n + z * h
        h_seq[t] = h
        if keep:
            saved.append((h_prev, r, z, n, rn))
    out = {"h_seq": h_seq, "hT": h}
    if keep:
        out["_saved"] = saved
    return out


def slstm_forward(Wx, R, b=None, h0=None, c0=None, n0=None, m0=None,
                  emulate_bf16_h=False, keep=False, emulate_bf16_pair_h=False):
    Dh = R.shape[1]
    Wx, R, b, (h, c, n, m) = _prep(Wx, R, b, {"h0": h0, "c0": c0, "n0": n0, "m0": m0},
                                   ("h0", "c0", "n0", "m0"), Dh)
    T = Wx.shape[0]
    h_seq = np.empty(Wx.shape[:3] + (Dh,))
    saved = []
    for t in range(T):
        hin = _to_bf16_f64(h) if emulate_bf16_h else h
        if emulate_bf16_pair_h:  # h as the sum of two bf16 parts: bf16(h) + bf16(h - bf16(h))
            hi = _to_bf16_f64(h)
            hin = hi + _to_bf16_f64(h - hi)
        pre = Wx[t] + _recurrent(hin, R) + b
        gi, gf, gz, go = _split(pre, 4)
        m_new = np.maximum(gf + m, gi)
        i = np.exp(gi - m_new)
        f = np.exp(gf + m - m_new)
        z = np.tanh(gz)
        o = _sigmoid(go)
        c_prev, n_prev = c, n
        c = f * c + i * z
        n = f * n + i
        m = m_new
        h_prev = h
        h = o * c / n
        h_seq[t] = h
        if keep:
            saved.append((h_prev, c_prev, n_prev, i, f, z, o, c, n))
    out = {"h_seq": h_seq, "hT": h, "cT": c, "nT": n, "mT": m}
    if keep:
        out["_saved"] = saved
    return out


# ---------------------------------------------------------------- backward --
def _bwd_common(Wx, R, dh_seq, dhT):
    T, B, NH, _ = np.shape(Wx)
    Dh = R.shape[1]
    dh_seq = np.asarray(dh_seq, np.float64)
    dh_next = np.zeros((B, NH, Dh)) if dhT is None else np.array(dhT, np.float64)
    return T, dh_seq, dh_next


def lstm_backward(Wx, R, b=None, h0=None, c0=None, dh_seq=None, dhT=None, dcT=None):
    """Gradients of L = sum(h_seq * dh_seq) + sum(hT * dhT) + sum(cT * dcT).

    Returns dWx [T,B,NH,4Dh], dR [NH,Dh,4Dh], db [NH,4Dh], dh0, dc0 [B,NH,Dh].
    """
    fw = lstm_forward(Wx, R, b, h0, c0, keep=True)
    R = np.asarray(R, np.float64)
    T, dh_seq, dh_next = _bwd_common(Wx, R, dh_seq, dhT)
    dc_next = np.zeros_like(dh_next) if dcT is None else np.array(dcT, np.float64)
    dWx = np.zeros(np.shape(Wx))
    dR = np.zeros(R.shape)
    db = np.zeros((R.shape[0], R.shape[2]))
    for t in range(T - 1, -1, -1):
        h_prev, c_prev, i, f, z, o, c = fw["_saved"][t]
        dh = dh_seq[t] + dh_next
        tc = np.tanh(c)
        dc = dc_next + dh * o * (1.0 - tc * tc)
        d_o = dh * tc
        d_i = dc * z
        d_f = dc * c_prev
        d_z = dc * i
        dc_next = dc * f
        dpre = np.concatenate([d_i * i * (1.0 - i), d_f * f * (1.0 - f),
                               d_z * (1.0 - z * z), d_o * o * (1.0 - o)], axis=-1)
        dWx[t] = dpre
        dR += _outer_sum(h_prev, dpre)
        db += dpre.sum(axis=0)
        dh_next = _recurrent_T(dpre, R)
    return {"dWx": dWx, "dR": dR, "db": db, "dh0": dh_next, "dc0": dc_next}


def gru_backward(Wx, R, b=None, h0=None, dh_seq=None, dhT=None):
    """Gradients of L = sum(h_seq * dh_seq) + sum(hT * dhT) for the GRU.

    dWx differs from the recurrent-preactivation gradient on the n block
    (r multiplies only the recurrent part); db and dR follow the latter.
    """
    fw = gru_forward(Wx, R, b, h0, keep=True)
    R = np.asarray(R, np.float64)
    T, dh_seq, dh_next = _bwd_common(Wx, R, dh_seq, dhT)
    dWx = np.zeros(np.shape(Wx))
    dR = np.zeros(R.shape)
    db = np.zeros((R.shape[0], R.shape[2]))
    for t in range(T - 1, -1, -1):
        h_prev, r, z, n, rn = fw["_saved"][t]
        dh = dh_seq[t] + dh_next
        dn = dh * (1.0 - z)
        dz = dh * (h_prev - n)
        dn_pre = dn * (1.0 - n * n)
        dr = dn_pre * rn
        dr_pre = dr * r * (1.0 - r)
        dz_pre = dz * z * (1.0 - z)
        dWx[t] = np.concatenate([dr_pre, dz_pre, dn_pre], axis=-1)
        drec = np.concatenate([dr_pre, dz_pre, dn_pre * r], axis=-1)
        dR += _outer_sum(h_prev, drec)
        db += drec.sum(axis=0)
        dh_next = dh * z + _recurrent_T(drec, R)
    return {"dWx": dWx, "dR": dR, "db": db, "dh0": dh_next}


def slstm_backward(Wx, R, b=None, h0=None, c0=None, n0=None, m0=None, dh_seq=None,
                   dhT=None, dcT=None, dnT=None):
    """Gradients of L = sum(h_seq*dh_seq) + sum(hT*dhT) + sum(cT*dcT) + sum(nT*dnT).

    The stabiliser m only rescales (c, n) jointly and h = o*c/n is invariant to
    it, so m is held at its forward values (no gradient flows through the max).
    For any loss of h this is the exact gradient; the upstream terms on the
    stabilised final states cT, nT are differentiated with m_T held fixed,
    which is the convention under which backward passes over consecutive time
    chunks (final-state gradients of one chunk fed as dcT, dnT of the previous
    one) compose to the whole-sequence gradient.
    """
    fw = slstm_forward(Wx, R, b, h0, c0, n0, m0, keep=True)
    R = np.asarray(R, np.float64)
    T, dh_seq, dh_next = _bwd_common(Wx, R, dh_seq, dhT)
    dc_next = np.zeros_like(dh_next) if dcT is None else np.array(dcT, np.float64)
    dn_next = np.zeros_like(dh_next) if dnT is None else np.array(dnT, np.float64)
    dWx = np.zeros(np.shape(Wx))
    dR = np.zeros(R.shape)
    db = np.zeros((R.shape[0], R.shape[2]))
    for t in range(T - 1, -1, -1):
        h_prev, c_prev, n_prev, i, f, z, o, c, n = fw["_saved"][t]
        dh = dh_seq[t] + dh_next
        d_o = dh * c / n
        dc = dc_next + dh * o / n
        dn = dn_next - dh * o * c / (n * n)
        d_f = dc * c_prev + dn * n_prev
        d_i = dc * z + dn
        d_z = dc * i
        dc_next = dc * f
        dn_next = dn * f
        dpre = np.concatenate([d_i * i, d_f * f, d_z * (1.0 - z * z), d_o * o * (1.0 - o)],
                              axis=-1)
        dWx[t] = dpre
        dR += _outer_sum(h_prev, dpre)
        db += dpre.sum(axis=0)
        dh_next = _recurrent_T(dpre, R)
    return {"dWx": dWx, "dR": dR, "db": db, "dh0": dh_next, "dc0": dc_next, "dn0": dn_next}


# ------------------------------------------------------------- dispatchers --
def forward(cell, Wx, R, b=None, h0=None, c0=None, n0=None, m0=None, emulate_bf16_h=False):
    if cell == "lstm":
        return lstm_forward(Wx, R, b, h0, c0, emulate_bf16_h)
    if cell == "gru":
        return gru_forward(Wx, R, b, h0, emulate_bf16_h)
    if cell == "slstm":
        return slstm_forward(Wx, R, b, h0, c0, n0, m0, emulate_bf16_h)
    raise ValueError(cell)


def backward(cell, Wx, R, b=None, h0=None, c0=None, n0=None, m0=None, dh_seq=None,
             dhT=None, dcT=None, dnT=None):
    """Gradients of sum(h_seq*dh_seq) + sum(hT*dhT) (+ sum(cT*dcT), + sum(nT*dnT))
    for the cell; upstream terms a cell does not have are ignored."""
    if cell == "lstm":
        return lstm_backward(Wx, R, b, h0, c0, dh_seq=dh_seq, dhT=dhT, dcT=dcT)
    if cell == "gru":
        return gru_backward(Wx, R, b, h0, dh_seq=dh_seq, dhT=dhT)
    if cell == "slstm":
        return slstm_backward(Wx, R, b, h0, c0, n0, m0, dh_seq=dh_seq, dhT=dhT, dcT=dcT, dnT=dnT)
    raise ValueError(cell)


# --------------------------------------------------------- input projection --
def input_projection(x, W, b=None):
    """Wx[m, n] = sum_k x[m, k] W[n, k] + b[n] in fp64.

    x [M, K], W [N, K] (rows are output features, a linear layer's weight),
    b [N] or None.  With N = NH*G*Dh and M = T*B the result, reshaped to
    [T, B, NH, G*Dh], is the recurrence's Wx.
    """
    x = np.asarray(x, np.float64)
    W = np.asarray(W, np.float64)
    out = x @ W.T
    if b is not None:
        out = out + np.asarray(b, np.float64)[None, :]
    return out


# ------------------------------------------------------------ stacked layers --
def stack_forward(cell, x, W_ih0, W_ih, b_ih, R, b, h0=None, c0=None, n0=None, m0=None):
    """L stacked head-wise layers (the blog page's layer-level parallelism
    paragraph runs layers concurrently; the result is that of running them in
    order): layer 0 reads x [T, B, Din], layer l > 0 reads layer l-1's h_seq.

    W_ih0 [G*d, Din] and W_ih [L-1, G*d, d] (d = NH*Dh, rows ordered [NH, G*Dh]),
    b_ih [L, G*d] or None, R [L, NH, Dh, G*Dh], b [L, NH, G*Dh] or None, initial
    states [L, B, NH, Dh] or None.  Returns the last layer's h_seq and every
    layer's final states stacked over L.
    """
    x = np.asarray(x, np.float64)
    T, B, _ = x.shape
    L, NH, Dh = R.shape[0], R.shape[1], R.shape[2]
    G = GATES[cell]
    inp = x.reshape(T * B, -1)
    finals = {}
    out = None
    for l in range(L):
        W = W_ih0 if l == 0 else W_ih[l - 1]
        Wx = input_projection(inp, W, None if b_ih is None else b_ih[l]).reshape(T, B, NH, G * Dh)
        pick = (lambda s: None if s is None else s[l])
        out = forward(cell, Wx, R[l], pick(b), pick(h0), pick(c0), pick(n0), pick(m0))
        for k in ("hT", "cT", "nT", "mT"):
            if k in out:
                finals.setdefault(k, []).append(out[k])
        inp = out["h_seq"].reshape(T * B, NH * Dh)
    res = {"h_seq": out["h_seq"]}
    for k, v in finals.items():
        res[k] = np.stack(v)
    return res
