"""Helpers shared by the GPU parity tests: oracle calls on torch tensors and the
routing comparison rule (bit-exact except at near-tied tokens, which must hold a
valid choice)."""
import numpy as np
import torch

from oracle import moe_oracle as O


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def oracle_route(x, w_router, bias, k, logit_offset=None, n_group=0, topk_group=0):
    return O.route(np64(x), np64(w_router), bias.cpu().numpy(), k,
                   None if logit_offset is None else logit_offset.cpu().numpy(), n_group=n_group,
                   topk_group=topk_group)


def check_routing(ref, idx, gate, counts, offsets, E, n_group=0, topk_group=0):
    """Returns the number of near-tied tokens; asserts everything else."""
    idx = idx.cpu().numpy()
    gate = gate.cpu().numpy().astype(np.float64)
    counts = counts.cpu().numpy()
    offsets = offsets.cpu().numpy()
    T, k = idx.shape
    rid = ref["idx"]
    btie, otie = ref["boundary_tie"], ref["order_tie"]
    clean = ~(btie | otie)
    # 1. tokens with no tie: indices equal, in order
    bad = np.nonzero(clean & np.any(idx != rid, axis=1))[0]
    assert bad.size == 0, f"{bad.size} untied tokens routed differently, first {bad[:5]}: {idx[bad[:3]]} vs {rid[bad[:3]]}"
    # 2. ties inside the chosen set only: same set
    only_order = otie & ~btie
    for t in np.nonzero(only_order)[0]:
        assert set(idx[t]) == set(rid[t]), t
    # 3. ties at the k-th place: the chosen set must be a valid top-k within 1e-5
    v = ref["v"].astype(np.float64)
    gtie = ref.get("group_tie", np.zeros(T, dtype=bool))
    if n_group:
        gsz = E // n_group
        for t in range(T):
            assert len({e // gsz for e in idx[t].tolist()}) <= topk_group, t
    for t in np.nonzero(btie & ~gtie)[0]:
        assert len(set(idx[t].tolist())) == k
        kth = np.sort(v[t])[::-1][k - 1]
        assert np.all(v[t][idx[t]] >= kth - O.NEAR_TIE), t
        must = np.nonzero(v[t] > kth + O.NEAR_TIE)[0]
        assert set(must.tolist()) <= set(idx[t].tolist()), t
    # 4. ties between kept and dropped groups: the groups used must be among the best
    #    topk_group within 1e-5, every group clearly better than the first dropped one
    #    must stay eligible, and no eligible expert left out may beat a chosen one
    for t in np.nonzero(gtie)[0]:
        assert len(set(idx[t].tolist())) == k, t
        va = ref["v_all"][t].astype(np.float64)
        m = -(-k // topk_group)
        gs = np.sort(va.reshape(n_group, gsz), axis=1)[:, ::-1][:, :m].sum(1)
        gsort = np.sort(gs)[::-1]
        used = {e // gsz for e in idx[t].tolist()}
        assert all(gs[g] >= gsort[topk_group - 1] - O.NEAR_TIE for g in used), t
        kept = used | set(np.nonzero(gs > gsort[topk_group] + O.NEAR_TIE)[0].tolist())
        weakest = va[idx[t]].min()
        for g in kept:
            for e in range(g * gsz, (g + 1) * gsz):
                if e not in set(idx[t].tolist()):
                    assert va[e] <= weakest + O.NEAR_TIE, (t, e)
    # gates: unbiased affinity of the chosen expert over the chosen sum
    s = ref["s"].astype(np.float64)
    s_sel = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    g_ref = s_sel / s_sel.sum(1, keepdims=True)
    np.testing.assert_allclose(gate, g_ref, rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(gate.sum(1), 1.0, rtol=0, atol=1e-5)
    # counts / offsets: the oracle's choice, with the GPU's valid choice at tied tokens
    use = np.where((btie | otie)[:, None], idx, rid)
    exp_counts = np.bincount(use.reshape(-1), minlength=E)
    np.testing.assert_array_equal(counts, exp_counts)
    np.testing.assert_array_equal(offsets, O.offsets_from_counts(exp_counts))
    return int((btie | otie).sum())


def rel_err(out, ref) -> float:
    return O.max_rel_err(np64(out) if isinstance(out, torch.Tensor) else out, ref)


BF16_HALF_ULP = 2.0 ** -8  # relative half-ulp of bf16 (8 significant bits)


def out_err(out, ref) -> float:
    """Computation error of a bf16 output against the float64 oracle, normalised by RMS(ref):
    max over elements of (|out - ref| - 2^-8 |ref|)+ / RMS(ref).  The 2^-8 |ref| term is the
    rounding of storing the exact value in bf16, which no bf16 output can avoid."""
    o = np64(out) if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.maximum(np.abs(o - ref) - BF16_HALF_ULP * np.abs(ref), 0.0)) / rms)


def fro_err(out, ref) -> float:
    """Relative Frobenius (RMS-normalised) error ||out - ref|| / ||ref|| over the compared
    elements: the bound a systematic error (a dropped term, a wrong index) cannot pass."""
    o = np64(out) if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(o - ref) / np.linalg.norm(ref))


def errs(out, ref) -> dict:
    """The three error figures the parity tests print: the gated computation error beyond
    bf16 storage rounding (out_err), the plain max/RMS and the relative Frobenius error."""
    return dict(out_err=out_err(out, ref), max_rms=rel_err(out, ref), fro=fro_err(out, ref))


# FP8 parity against the oracle's FP8 layer (the same simulated quantisation).  The GPU
# computes h in FP32, the oracle in float64; where h lies within that difference of a
# rounding midpoint the two sides pick neighbouring E4M3 codes.  Such a flip moves one
# element of h by one E4M3 step -- up to 32/448 of its tile's amax with amax / 448 scales
# and 32/256 with power-of-two scales, about 0.4-0.9 sigma of h since SwiGLU's
# heavy-tailed h puts a tile's amax 6-8 sigma out -- and reaches one output row through a
# column of W_down (elements ~ N(0, 1/sqrt(I))): some of that row's outputs move by a few
# per cent of the RMS, up to 0.1 x 0.143 x 8 = 11 % for the largest, while the Frobenius
# error barely changes.  A wrong scale, index or tile moves a large share of a whole tile
# (thousands to tens of thousands of elements).  So the FP8 gates are: relative Frobenius
# <= 5e-3 (the bf16 bound), at most 1e-3 of the elements beyond the bf16 bound
# (computation error beyond bf16 storage rounding > 2e-2 of the RMS; flips measured
# 1e-5..1e-4, a 2 % error on one tile of a V3 expert 6e-3), every element within 0.15.
FP8_TOL_FRO = 5e-3
FP8_TOL_FRAC = 1e-3
FP8_TOL_MAX = 0.15


def fp8_errs(out, ref) -> dict:
    """errs() plus the fraction of elements beyond the bf16 bound (see above)."""
    o = np64(out) if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    e = errs(o, ref)
    rms = np.sqrt(np.mean(ref * ref))
    dev = np.maximum(np.abs(o - ref) - BF16_HALF_ULP * np.abs(ref), 0.0) / rms
    e["frac_over"] = float(np.mean(dev > 2e-2))
    return e


def fp8_ok(e) -> bool:
    return e["fro"] <= FP8_TOL_FRO and e["frac_over"] <= FP8_TOL_FRAC and e["out_err"] <= FP8_TOL_MAX
