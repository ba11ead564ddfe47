"""CPU oracle for the DeepSeekMoE layer forward with auxiliary-loss-free routing.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product (the CUDA library and its Python binding) never calls it.
It shares no code with the CUDA path: it is plain numpy, float64 for every
matrix product, written to be read against the pages step by step.

Pages followed (titles and sections):
  [YDL]  "DeepSeek-V3 详解：用 1/30 的成本对齐 GPT-4o" (yudonglee.me),
         sections 2.2 (256 routed + 1 shared, top-8), 2.3 (Aux-Loss-Free Load
         Balancing: per-expert bias, update speed gamma = 0.001).
  [CSDN] "DeepSeek-V3 技术报告要点" (deepseek.csdn.net), section 3 table (hidden
         7168, expert intermediate 2048), section 4.2 (bias on the routing
         score, moved by the observed per-batch load), section 1 (SwiGLU FFN
         inside a pre-norm block).
  [DYN]  "deepseek-v3-report" (dynmi.github.io), model table (8 routed + 1 shared
         per token) and the load-balancing paragraph (overloaded expert: b_i
         down; idle expert: b_i up; b_i stays out of the gradient).
  [KC]   "拆解DeepSeek V3" (kongchang.com), section "让256个专家都干活" (the bias is
         added to each expert's routing score, not to the loss).

Readings where the pages are silent (each also listed in the design notes):
  * affinity s = sigmoid(z) of the router logit z = x . w_i (+ optional offset);
  * the bias is added to the affinity and used for selection only;
  * gates are the chosen unbiased affinities divided by their sum over the
    chosen k (no extra scaling factor);
  * top-k order: descending biased score, ties to the lower expert index;
  * shared experts are ungated (weight 1) independent SwiGLU experts;
  * the layer output excludes the residual;
  * bias update b_i += gamma * sign(T*k/E - count_i), sign(0) = 0, in float32.

Precision: float32 is used exactly where a float decides an integer (the routing
scores that are compared for selection), because the layer's router is kept in
bf16/FP32 ([YDL] section 4.3: sensitive operators keep high precision); every
other product is float64.

parity: pinned by tests/test_oracle_*.py (hand-worked 4x4 example in
tests/golden, brute-force top-k, invariants, reduction to a plain SwiGLU FFN,
dense-mixture special case, closed-form bias update, a hand-worked combine and
the combine of permuted expert rows against the layer forward).
"""
from __future__ import annotations

import numpy as np

NEAR_TIE = 1e-5


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- router


def router_logits(x, w_router, logit_offset=None) -> np.ndarray:
    """z[t, i] = sum_c x[t, c] * w_router[i, c] (+ o_i), returned as float32.

    The dot product is taken in float64 and rounded once to float32; the
    optional per-expert offset is then added in float32.
    """
    z = (_f64(x) @ _f64(w_router).T).astype(np.float32)
    if logit_offset is not None:
        z = z + np.asarray(logit_offset, dtype=np.float32)[None, :]
    return z


def affinity(z) -> np.ndarray:
    """s = 1 / (1 + exp(-z)) in float32 (sigmoid affinity)."""
    z = np.asarray(z, dtype=np.float32)
    one = np.float32(1.0)
    return one / (one + np.exp(-z))


def group_limit(v, n_group, topk_group, k):
    """Group-limited selection ("DeepSeek-V3 技术报告要点" section 9 table: n_group /
    topk_group; "DeepSeek-V3 详解" 2.4: a token's experts come from at most M nodes).

    Reading (the pages give no group score): experts form n_group contiguous groups;
    a group's score is the float32 sum, in descending order, of its ceil(k/topk_group)
    largest biased scores; the topk_group best groups are kept (ties to the lower group
    index) and every expert outside them gets -inf.  Returns (masked v, group_tie)
    where group_tie flags tokens whose kept/dropped group scores lie within NEAR_TIE.
    """
    v = np.asarray(v, dtype=np.float32)
    T, E = v.shape
    gsz = E // n_group
    m = -(-k // topk_group)
    vg = v.reshape(T, n_group, gsz)
    top_m = -np.sort(-vg, axis=2)[:, :, :m]
    gscore = np.zeros((T, n_group), dtype=np.float32)
    for j in range(m):
        gscore = (gscore + top_m[:, :, j]).astype(np.float32)
    gorder = np.argsort(-gscore, axis=1, kind="stable")
    keep = np.zeros((T, n_group), dtype=bool)
    np.put_along_axis(keep, gorder[:, :topk_group], True, axis=1)
    masked = np.where(np.repeat(keep, gsz, axis=1), v, np.float32(-np.inf)).astype(np.float32)
    if topk_group < n_group:
        gs = np.take_along_axis(gscore, gorder, axis=1).astype(np.float64)
        group_tie = (gs[:, topk_group - 1] - gs[:, topk_group]) < NEAR_TIE
    else:
        group_tie = np.zeros(T, dtype=bool)
    return masked, group_tie


def route(x, w_router, bias, k, logit_offset=None, n_group=0, topk_group=0) -> dict:
    """Biased top-k selection and unbiased normalised gates ([DYN], [KC], [YDL] 2.3).

    Returns a dict with
      idx   int32 [T, k]  chosen experts, descending biased score, ties -> lower index
      gate  float64 [T, k] s[t, idx] / sum_j s[t, idx_j]
      s     float32 [T, E] affinities;  v float32 [T, E] biased scores s + b
            (-inf outside the kept groups under group-limited routing)
      v_all float32 [T, E] biased scores s + b of every expert
      boundary_tie bool [T]: k-th and (k+1)-th biased scores within NEAR_TIE
      order_tie    bool [T]: two adjacent chosen scores within NEAR_TIE
    """
    z = router_logits(x, w_router, logit_offset)
    s = affinity(z)
    v = s + np.asarray(bias, dtype=np.float32)[None, :]
    v_all = v
    T, E = v.shape
    group_tie = np.zeros(T, dtype=bool)
    if n_group:
        v, group_tie = group_limit(v, n_group, topk_group, k)
    # stable sort of -v: equal scores keep ascending expert order
    order = np.argsort(-v, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    s_sel = np.take_along_axis(s, idx, axis=1).astype(np.float64)
    gate = s_sel / s_sel.sum(axis=1, keepdims=True)
    v_sorted = np.take_along_axis(v, order, axis=1).astype(np.float64)
    if k < E:
        boundary_tie = (v_sorted[:, k - 1] - v_sorted[:, k]) < NEAR_TIE
    else:
        boundary_tie = np.zeros(T, dtype=bool)
    if k > 1:
        order_tie = (np.diff(-v_sorted[:, :k], axis=1) < NEAR_TIE).any(axis=1)
    else:
        order_tie = np.zeros(T, dtype=bool)
    return dict(idx=idx, gate=gate, s=s, v=v, v_all=v_all, z=z, boundary_tie=boundary_tie | group_tie,
                order_tie=order_tie, group_tie=group_tie)


def expert_counts(idx, E) -> np.ndarray:
    """count_i = number of (token, slot) pairs routed to expert i (the observed load)."""
    return np.bincount(np.asarray(idx).reshape(-1), minlength=E).astype(np.int32)


def offsets_from_counts(counts) -> np.ndarray:
    """Exclusive prefix sum, length E+1, last entry = T*k."""
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    off[1:] = np.cumsum(counts)
    return off.astype(np.int32)


# ---------------------------------------------------------------- dispatch / combine


def permutation(idx, E) -> dict:
    """Group (token, slot) pairs by expert, token-ascending inside each expert.

    perm_token[p] = token of permuted row p; inv_pos[t, j] = row of (t, j).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.reshape(-1)  # row-major: token-major, then slot
    order = np.argsort(flat, kind="stable")
    perm_token = (order // k).astype(np.int32)
    inv_pos = np.empty(T * k, dtype=np.int32)
    inv_pos[order] = np.arange(T * k, dtype=np.int32)
    counts = expert_counts(idx, E)
    return dict(perm_token=perm_token, inv_pos=inv_pos.reshape(T, k),
                counts=counts, offsets=offsets_from_counts(counts))


def silu(a):
    a = _f64(a)
    return a / (1.0 + np.exp(-a))


def swiglu_expert(x_rows, w_gate_up, w_down) -> np.ndarray:
    """One SwiGLU expert ([CSDN] section 1): y = W_down (silu(W_gate x) * (W_up x)).

    w_gate_up [2I, d]: rows 0..I-1 are the gate projection, rows I..2I-1 the up
    projection.  w_down [d, I].  float64 throughout.
    """
    I = w_down.shape[1]
    wgu = _f64(w_gate_up)
    a = _f64(x_rows) @ wgu[:I].T
    u = _f64(x_rows) @ wgu[I:].T
    h = silu(a) * u
    return h @ _f64(w_down).T


def forward(x, w_router, bias, w_gate_up, w_down, k, S, logit_offset=None,
            route_result=None) -> dict:
    """Whole layer: route, group by expert, run experts, weighted combine + shared.

    out[t] = sum_s y_shared_s(x_t) + sum_j gate[t, j] * y_{idx[t, j]}(x_t)
    Experts E..E+S-1 in the weight arrays are the shared experts.
    """
    x = np.asarray(x)
    T, d = x.shape
    E = np.asarray(w_router).shape[0]
    r = route(x, w_router, bias, k, logit_offset) if route_result is None else route_result
    idx, gate = r["idx"], r["gate"]
    out = np.zeros((T, d), dtype=np.float64)
    for s_id in range(S):
        out += swiglu_expert(x, w_gate_up[E + s_id], w_down[E + s_id])
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        y = swiglu_expert(x[tok], w_gate_up[e], w_down[e])
        out[tok] += gate[tok, slot][:, None] * y
    return dict(out=out, route=r)


def forward_rows(tokens, x, route_result, get_expert, E, S) -> np.ndarray:
    """The layer output for a subset of tokens only (for large workloads).

    get_expert(e) -> (w_gate_up [2I, d], w_down [d, I]) as arrays.
    """
    tokens = np.asarray(tokens)
    xs = np.asarray(x)[tokens]
    idx = route_result["idx"][tokens]
    gate = route_result["gate"][tokens]
    out = np.zeros(xs.shape, dtype=np.float64)
    for s_id in range(S):
        wgu, wd = get_expert(E + s_id)
        out += swiglu_expert(xs, wgu, wd)
    for e in np.unique(idx):
        rows, slot = np.nonzero(idx == e)
        wgu, wd = get_expert(int(e))
        out[rows] += gate[rows, slot][:, None] * swiglu_expert(xs[rows], wgu, wd)
    return out


# ---------------------------------------------------------------- bias update


def bias_update(bias, counts, T, k, gamma=0.001) -> np.ndarray:
    """b_i <- b_i + gamma * sign(T*k/E - count_i)  ([YDL] 2.3, [DYN], [CSDN] 4.2).

    The sign is decided on integers (T*k against E*count_i), sign(0) = 0; the
    add is one float32 operation.
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.shape[0]
    sgn = np.sign(np.int64(T) * np.int64(k) - np.int64(E) * counts).astype(np.float32)
    return np.asarray(bias, dtype=np.float32) + np.float32(gamma) * sgn


def load_stats(counts) -> dict:
    c = np.asarray(counts, dtype=np.float64)
    return dict(max=float(c.max()), mean=float(c.mean()), max_over_mean=float(c.max() / c.mean()))


# ---------------------------------------------------------------- error metric


def max_rel_err(out, ref) -> float:
    """max |out - ref| / RMS(ref) over all compared elements."""
    out = _f64(out)
    ref = _f64(ref)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(out - ref)) / rms)


def combine(y, gate, inv_pos, T, k, S) -> np.ndarray:
    """out[t] = sum_s y[T*k + s*T + t] + sum_j gate[t, j] * y[inv_pos[t, j]] (float64)."""
    y = _f64(y)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for s_id in range(S):
        out += y[T * k + s_id * T: T * k + (s_id + 1) * T]
    g = _f64(gate)
    for j in range(k):
        out += g[:, j:j + 1] * y[np.asarray(inv_pos)[:, j]]
    return out
