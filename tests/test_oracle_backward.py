"""Pins of the backward oracle (oracle/moe_backward.py) against things other than
itself: central finite differences of the forward layer on tiny shapes, the gate
normalisation identity, a special case with a known zero gradient, and a single
dense expert against torch's autograd."""
import numpy as np
import pytest
import torch

from oracle import moe_backward as BW
from oracle import moe_oracle as O


def _tiny(T=5, d=6, E=4, S=1, k=2, I=3, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    wr = 0.5 * rng.standard_normal((E, d))
    wgu = 0.4 * rng.standard_normal((E + S, 2 * I, d))
    wd = 0.4 * rng.standard_normal((E + S, d, I))
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    off = rng.uniform(-0.3, 0.3, E)
    idx = O.route(x, wr, bias, k, logit_offset=off)["idx"]
    return x, wr, wgu, wd, idx, off


def _layer(x, wr, wgu, wd, idx, S, off):
    """The forward layer in float64 for a fixed selection, built from the forward oracle's expert."""
    E = wr.shape[0]
    z = x @ wr.T + off[None, :]
    s = 1.0 / (1.0 + np.exp(-z))
    s_sel = np.take_along_axis(s, idx, axis=1)
    gate = s_sel / s_sel.sum(axis=1, keepdims=True)
    out = np.zeros_like(x)
    for sh in range(S):
        out += O.swiglu_expert(x, wgu[E + sh], wd[E + sh])
    for t in range(x.shape[0]):
        for j in range(idx.shape[1]):
            e = idx[t, j]
            out[t] += gate[t, j] * O.swiglu_expert(x[t:t + 1], wgu[e], wd[e])[0]
    return out


@pytest.mark.parametrize("S,k", [(1, 2), (0, 3), (2, 1)])
def test_backward_matches_finite_differences(S, k):
    x, wr, wgu, wd, idx, off = _tiny(S=S, k=k, seed=S * 10 + k)
    R = np.random.default_rng(7).standard_normal(x.shape)  # L = sum(out * R)
    g = BW.backward(x, wr, wgu, wd, idx, R, S, logit_offset=off)
    eps = 1e-6

    def check(arr, grad, name):
        flat = arr.reshape(-1)
        num = np.zeros(flat.size)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            lp = (_layer(x, wr, wgu, wd, idx, S, off) * R).sum()
            flat[i] = keep - eps
            lm = (_layer(x, wr, wgu, wd, idx, S, off) * R).sum()
            flat[i] = keep
            num[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad.reshape(-1), num, rtol=1e-6, atol=1e-8, err_msg=name)

    check(x, g["dx"], "dx")
    check(wr, g["dw_router"], "dw_router")
    check(wgu, g["dw_gate_up"], "dw_gate_up")
    check(wd, g["dw_down"], "dw_down")


def test_gate_normalisation_identity():
    # sum_j g_j = 1 for every token, so the affinity gradients satisfy sum_j ds_j s_j = 0
    x, wr, wgu, wd, idx, off = _tiny(T=9, E=6, k=3, seed=3)
    dout = np.random.default_rng(1).standard_normal(x.shape)
    g = BW.backward(x, wr, wgu, wd, idx, dout, 1, logit_offset=off)
    np.testing.assert_allclose((g["ds"] * g["s"]).sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["gate"].sum(axis=1), 1.0, atol=1e-14)


def test_router_gradient_vanishes_for_identical_experts():
    # all experts the same function and all chosen: out = FFN(x) whatever the gates are
    x, wr, wgu, wd, idx, off = _tiny(T=6, E=3, S=0, k=3, seed=4)
    wgu[:] = wgu[0]
    wd[:] = wd[0]
    dout = np.random.default_rng(2).standard_normal(x.shape)
    g = BW.backward(x, wr, wgu, wd, idx, dout, 0, logit_offset=off)
    assert np.abs(g["dw_router"]).max() < 1e-12
    assert np.abs(g["dz"]).max() < 1e-12


def test_single_dense_expert_against_autograd():
    # E = 1, k = 1, no shared expert: gate = 1, the layer is one SwiGLU FFN
    rng = np.random.default_rng(5)
    T, d, I = 7, 8, 5
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((1, d))
    wgu = 0.3 * rng.standard_normal((1, 2 * I, d))
    wd = 0.3 * rng.standard_normal((1, d, I))
    dout = rng.standard_normal((T, d))
    idx = np.zeros((T, 1), dtype=np.int32)
    g = BW.backward(x, wr, wgu, wd, idx, dout, 0)
    xt = torch.tensor(x, requires_grad=True)
    wgut = torch.tensor(wgu[0], requires_grad=True)
    wdt = torch.tensor(wd[0], requires_grad=True)
    a = xt @ wgut[:I].T
    u = xt @ wgut[I:].T
    y = (torch.nn.functional.silu(a) * u) @ wdt.T
    y.backward(torch.tensor(dout))
    np.testing.assert_allclose(g["dx"], xt.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dw_gate_up"][0], wgut.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dw_down"][0], wdt.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.abs(g["dw_router"]).max() == 0.0


def test_lazy_backward_on_token_subsets():
    # the subset uses the GPU tests rely on: dx of sampled tokens, dW of one expert from its own tokens
    x, wr, wgu, wd, idx, off = _tiny(T=12, E=5, S=1, k=2, seed=9)
    dout = np.random.default_rng(3).standard_normal(x.shape)
    full = BW.backward(x, wr, wgu, wd, idx, dout, 1, logit_offset=off)
    get = lambda e: (wgu[e], wd[e])
    tok = np.array([1, 4, 7])
    sub = BW.backward_lazy(x[tok], wr, get, idx[tok], dout[tok], 5, 1, off)
    np.testing.assert_allclose(sub["dx"], full["dx"][tok], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sub["dz"], full["dz"][tok], rtol=1e-13, atol=1e-13)
    e = int(idx[0, 0])
    mine = np.nonzero((idx == e).any(axis=1))[0]
    one = BW.backward_lazy(x[mine], wr, get, idx[mine], dout[mine], 5, 1, off, dw_experts=[e], need_dx=False)
    np.testing.assert_allclose(one["dw"][e][0], full["dw_gate_up"][e], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(one["dw"][e][1], full["dw_down"][e], rtol=1e-13, atol=1e-13)
    assert "dx" not in one
