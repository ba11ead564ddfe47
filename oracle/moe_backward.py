"""CPU oracle for the backward pass of the DeepSeekMoE layer (gradients of the
layer output with respect to its input and weights), for a fixed routing.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle/moe_oracle.py``): only the tests
and bench.py's reference legs may import it; the CUDA path never does.  Plain
numpy, float64 throughout.

What is differentiated (pages: "DeepSeek-V3 详解" 2.2-2.3 and 4; "deepseek-v3-report"
load-balancing paragraph; "DeepSeek-V3 技术报告要点" section 1):
  out[t] = sum_s FFN_s(x_t) + sum_{j in C_t} g_j(t) FFN_{idx[t,j]}(x_t),
  g_j(t) = s_j / sum_{i in C_t} s_i,  s = sigmoid(x_t . w_router + o),
  FFN_e(x) = W_down,e (silu(W_gate,e x) * (W_up,e x)).
The chosen set C_t is the forward's selection: a discrete choice with no
gradient.  The selection bias b_i is used only to choose ("deepseek-v3-report":
b_i stays out of the gradient), so nothing here depends on it.

Chain rule, per token t and chosen slot j (y_j = FFN_{idx[t,j]}(x_t)):
  dy_j = g_j dout[t]            (shared experts: dy = dout[t])
  dg_j = <dout[t], y_j>
  ds_j = (dg_j - sum_i dg_i g_i) / sum_i s_i
  dz_j = ds_j s_j (1 - s_j);    dW_router[idx] += dz_j x_t;  dx_t += dz_j w_router[idx]
and per expert row (a = W_gate x, u = W_up x, h = silu(a) u, y = W_down h):
  dh = W_down^T dy;  dW_down += dy h^T
  da = dh * u * silu'(a),  silu'(a) = sigmoid(a) (1 + a (1 - sigmoid(a)));  du = dh * silu(a)
  dW_gate += da x^T;  dW_up += du x^T;  dx += W_gate^T da + W_up^T du.

parity: pinned by tests/test_oracle_backward.py (central finite differences of
the forward on tiny layers, the sum_j ds_j s_j = 0 identity of the gate
normalisation, the vanishing router gradient when every expert is identical,
and a single dense expert against torch's autograd).
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-_f64(z)))


def swiglu_expert_backward(x_rows, w_gate_up, w_down, dy) -> dict:
    """Gradients of y = W_down (silu(W_gate x) * (W_up x)) for rows x with upstream dy.

    Returns dx [n, d], dw_gate_up [2I, d], dw_down [d, I] and the row intermediates
    a, u, h, dh, da, du.
    """
    x = _f64(x_rows)
    dy = _f64(dy)
    wgu = _f64(w_gate_up)
    wd = _f64(w_down)
    I = wd.shape[1]
    wg, wu = wgu[:I], wgu[I:]
    a = x @ wg.T
    u = x @ wu.T
    sa = sigmoid(a)
    silu_a = a * sa
    h = silu_a * u
    dh = dy @ wd
    dw_down = dy.T @ h
    da = dh * u * sa * (1.0 + a * (1.0 - sa))
    du = dh * silu_a
    dw_gate_up = np.concatenate([da.T @ x, du.T @ x], axis=0)
    dx = da @ wg + du @ wu
    return dict(dx=dx, dw_gate_up=dw_gate_up, dw_down=dw_down, a=a, u=u, h=h, dh=dh, da=da, du=du)


def backward(x, w_router, w_gate_up, w_down, idx, dout, S, logit_offset=None) -> dict:
    """Layer gradients for the routing idx [T, k] (experts E..E+S-1 are shared).

    Returns dx [T, d], dw_router [E, d], dw_gate_up [E+S, 2I, d], dw_down [E+S, d, I],
    and per (token, slot): s, gate, dgate, ds, dz [T, k].
    """
    wgu = np.asarray(w_gate_up)
    wd = np.asarray(w_down)
    G = wgu.shape[0]
    r = backward_lazy(x, w_router, lambda e: (wgu[e], wd[e]), idx, dout, G - S, S, logit_offset,
                      dw_experts=range(G))
    dw_gate_up = np.zeros(wgu.shape)
    dw_down = np.zeros(wd.shape)
    for e, (gu, dn) in r.pop("dw").items():
        dw_gate_up[e] = gu
        dw_down[e] = dn
    return dict(r, dw_gate_up=dw_gate_up, dw_down=dw_down)


def backward_lazy(x, w_router, get_expert, idx, dout, E, S, logit_offset=None, dw_experts=(),
                  need_dx=True) -> dict:
    """The same gradients with the expert weights fetched one expert at a time
    (get_expert(e) -> (w_gate_up [2I, d], w_down [d, I])), for layers too large to
    hold every expert in float64.

    x, idx, dout may be any subset of the batch's tokens: dx, dz and the per-slot
    values are per token, while the weight gradients returned in dw = {e: (dW_gate_up,
    dW_down)} (experts in dw_experts) and dw_router sum over the given tokens only.
    need_dx=False skips the experts outside dw_experts (dx, dgate, ds, dz and
    dw_router are then not returned).
    """
    x = _f64(x)
    dout = _f64(dout)
    wr = _f64(w_router)
    idx = np.asarray(idx)
    T, d = x.shape
    k = idx.shape[1]
    want = set(int(e) for e in dw_experts)
    z = (x[:, None, :] * wr[idx]).sum(axis=2)  # logits of the chosen experts only
    if logit_offset is not None:
        z = z + _f64(logit_offset)[idx]
    s = sigmoid(z)
    ssum = s.sum(axis=1, keepdims=True)
    gate = s / ssum
    dx = np.zeros((T, d))
    dgate = np.zeros((T, k))
    dw = {}
    for sh in range(S):
        if not need_dx and E + sh not in want:
            continue
        wgu_e, wd_e = get_expert(E + sh)
        g = swiglu_expert_backward(x, wgu_e, wd_e, dout)
        dx += g["dx"]
        if E + sh in want:
            dw[E + sh] = (g["dw_gate_up"], g["dw_down"])
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0 or (not need_dx and e not in want):
            continue
        wgu_e, wd_e = get_expert(e)
        xe = x[tok]
        y = _forward_rows(xe, wgu_e, wd_e)
        dgate[tok, slot] = (dout[tok] * y).sum(axis=1)
        g = swiglu_expert_backward(xe, wgu_e, wd_e, gate[tok, slot][:, None] * dout[tok])
        np.add.at(dx, tok, g["dx"])
        if e in want:
            dw[e] = (g["dw_gate_up"], g["dw_down"])
    for e in want:  # experts without tokens here: zero gradients
        if e not in dw:
            wgu_e, wd_e = get_expert(e)
            dw[e] = (np.zeros(np.shape(wgu_e)), np.zeros(np.shape(wd_e)))
    out = dict(s=s, gate=gate, dw=dw)
    if not need_dx:
        return out
    ds = (dgate - (dgate * gate).sum(axis=1, keepdims=True)) / ssum
    dz = ds * s * (1.0 - s)
    dw_router = np.zeros(wr.shape)
    np.add.at(dw_router, idx.reshape(-1), (dz.reshape(-1, 1) * np.repeat(x, k, axis=0)))
    dx += (dz[:, :, None] * wr[idx]).sum(axis=1)
    out.update(dx=dx, dw_router=dw_router, dgate=dgate, ds=ds, dz=dz)
    return out


def _forward_rows(x_rows, w_gate_up, w_down) -> np.ndarray:
    """y = W_down (silu(W_gate x) * (W_up x)) in float64 (the forward expert)."""
    x = _f64(x_rows)
    wgu = _f64(w_gate_up)
    wd = _f64(w_down)
    I = wd.shape[1]
    a = x @ wgu[:I].T
    u = x @ wgu[I:].T
    return (a * sigmoid(a) * u) @ wd.T
