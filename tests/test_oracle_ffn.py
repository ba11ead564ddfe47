"""Pins for the oracle's expert FFN and combine (CPU only).

Special cases reduce the layer to plain library routines (torch CPU, float64).
"""
import numpy as np
import torch
import torch.nn.functional as F

from oracle import moe_oracle as O


def _rand(rng, *shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def test_single_expert_is_a_plain_swiglu_ffn():
    # E=1, k=1, S=0: the gate is s/s = 1 and the layer is one SwiGLU FFN
    rng = np.random.default_rng(0)
    T, d, I = 33, 48, 20
    x = _rand(rng, T, d)
    wr = _rand(rng, 1, d)
    wgu = _rand(rng, 1, 2 * I, d, scale=d ** -0.5)
    wd = _rand(rng, 1, d, I, scale=I ** -0.5)
    res = O.forward(x, wr, np.zeros(1, np.float32), wgu, wd, k=1, S=0)
    xt = torch.from_numpy(x).double()
    g = xt @ torch.from_numpy(wgu[0, :I]).double().T
    u = xt @ torch.from_numpy(wgu[0, I:]).double().T
    ref = (F.silu(g) * u) @ torch.from_numpy(wd[0]).double().T
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_all_experts_chosen_is_a_dense_normalised_mixture():
    # k = E, b = 0: out = shared + sum_i s_i / sum(s) * y_i for every token
    rng = np.random.default_rng(1)
    T, d, I, E, S = 17, 32, 16, 5, 1
    x = _rand(rng, T, d)
    wr = _rand(rng, E, d, scale=0.3)
    wgu = _rand(rng, E + S, 2 * I, d, scale=d ** -0.5)
    wd = _rand(rng, E + S, d, I, scale=I ** -0.5)
    res = O.forward(x, wr, np.zeros(E, np.float32), wgu, wd, k=E, S=S)
    xt = torch.from_numpy(x).double()
    z = (xt @ torch.from_numpy(wr).double().T).float()
    s = torch.sigmoid(z).double()
    w = s / s.sum(1, keepdim=True)

    def expert(e):
        g = xt @ torch.from_numpy(wgu[e, :I]).double().T
        u = xt @ torch.from_numpy(wgu[e, I:]).double().T
        return (F.silu(g) * u) @ torch.from_numpy(wd[e]).double().T

    ref = expert(E)
    for e in range(E):
        ref = ref + w[:, e:e + 1] * expert(e)
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-5, atol=1e-6)


def test_shared_experts_add_ungated():
    # two shared experts and a routed part that is switched off by zero down weights
    rng = np.random.default_rng(2)
    T, d, I, E, S, k = 9, 16, 8, 4, 2, 2
    x = _rand(rng, T, d)
    wr = _rand(rng, E, d)
    wgu = _rand(rng, E + S, 2 * I, d, scale=0.25)
    wd = _rand(rng, E + S, d, I, scale=0.3)
    wd[:E] = 0.0
    res = O.forward(x, wr, np.zeros(E, np.float32), wgu, wd, k=k, S=S)
    xt = torch.from_numpy(x).double()
    ref = 0
    for e in (E, E + 1):
        g = xt @ torch.from_numpy(wgu[e, :I]).double().T
        u = xt @ torch.from_numpy(wgu[e, I:]).double().T
        ref = ref + (F.silu(g) * u) @ torch.from_numpy(wd[e]).double().T
    np.testing.assert_allclose(res["out"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_routed_output_is_gate_weighted_sum_of_chosen_experts():
    # distinguishes gate weighting, slot/expert pairing and gate-vs-up order
    rng = np.random.default_rng(3)
    T, d, I, E, S, k = 12, 16, 8, 6, 0, 3
    x = _rand(rng, T, d)
    wr = _rand(rng, E, d)
    wgu = _rand(rng, E, 2 * I, d, scale=0.25)
    wd = _rand(rng, E, d, I, scale=0.3)
    res = O.forward(x, wr, np.zeros(E, np.float32), wgu, wd, k=k, S=S)
    idx, gate = res["route"]["idx"], res["route"]["gate"]
    for t in range(T):
        xt = torch.from_numpy(x[t:t + 1]).double()
        acc = torch.zeros(1, d, dtype=torch.float64)
        for j in range(k):
            e = int(idx[t, j])
            g = xt @ torch.from_numpy(wgu[e, :I]).double().T
            u = xt @ torch.from_numpy(wgu[e, I:]).double().T
            acc += gate[t, j] * ((F.silu(g) * u) @ torch.from_numpy(wd[e]).double().T)
        np.testing.assert_allclose(res["out"][t], acc[0].numpy(), rtol=1e-12, atol=1e-12)


def test_forward_rows_matches_forward_on_subset():
    rng = np.random.default_rng(4)
    T, d, I, E, S, k = 40, 16, 8, 8, 1, 2
    x = _rand(rng, T, d)
    wr = _rand(rng, E, d)
    wgu = _rand(rng, E + S, 2 * I, d, scale=0.25)
    wd = _rand(rng, E + S, d, I, scale=0.3)
    full = O.forward(x, wr, np.zeros(E, np.float32), wgu, wd, k=k, S=S)
    rows = np.array([0, 7, 13, 39])
    sub = O.forward_rows(rows, x, full["route"], lambda e: (wgu[e], wd[e]), E, S)
    np.testing.assert_allclose(sub, full["out"][rows], rtol=1e-12, atol=1e-12)


def test_combine_hand_worked():
    # T = 2 tokens, k = 2 slots, S = 2 shared experts, d = 2.  Routed rows 0..3, then
    # shared expert 0 on tokens 0, 1 (rows 4, 5), shared expert 1 (rows 6, 7).
    y = np.array([[1, 0], [0, 1], [10, 0], [0, 10],
                  [100, 100], [200, 200],
                  [1000, 0], [0, 1000]], dtype=np.float64)
    gate = np.array([[0.75, 0.25], [0.6, 0.4]])
    inv_pos = np.array([[2, 0], [1, 3]])
    # token 0: 100 + 1000 (shared) + 0.75 * row 2 + 0.25 * row 0 = [1107.75, 100]
    # token 1: 200 + 1000 (shared) + 0.6 * row 1 + 0.4 * row 3   = [200, 1204.6]
    want = np.array([[1107.75, 100.0], [200.0, 1204.6]])
    got = O.combine(y, gate, inv_pos, T=2, k=2, S=2)
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-12)


def test_combine_of_permuted_expert_rows_is_the_layer():
    # the routed rows in permuted order (expert-major, tokens ascending) followed by the
    # shared rows, combined through inv_pos, give the layer output of forward()
    rng = np.random.default_rng(4)
    T, d, I, E, S, k = 23, 16, 8, 6, 2, 3
    x = _rand(rng, T, d)
    wr = _rand(rng, E, d, scale=0.5)
    wgu = _rand(rng, E + S, 2 * I, d, scale=d ** -0.5)
    wd = _rand(rng, E + S, d, I, scale=I ** -0.5)
    b = _rand(rng, E, scale=0.05)
    res = O.forward(x, wr, b, wgu, wd, k=k, S=S)
    r = res["route"]
    p = O.permutation(r["idx"], E)
    y = np.zeros((T * k + S * T, d))
    for e in range(E):
        lo, hi = p["offsets"][e], p["offsets"][e + 1]
        if hi > lo:
            y[lo:hi] = O.swiglu_expert(x[p["perm_token"][lo:hi]], wgu[e], wd[e])
    for s_id in range(S):
        y[T * k + s_id * T: T * k + (s_id + 1) * T] = O.swiglu_expert(x, wgu[E + s_id], wd[E + s_id])
    got = O.combine(y, r["gate"], p["inv_pos"], T, k, S)
    np.testing.assert_allclose(got, res["out"], rtol=1e-12, atol=1e-12)
