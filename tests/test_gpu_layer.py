"""GPU parity of the dispatch, expert FFN, combine and whole-layer calls against
the oracle, on seeded inputs shaped like the layer's workloads."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import inputs as I
from moe_testutil import check_routing, errs, np64, oracle_route, out_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_BF16 = 2e-2  # computation error / RMS(ref), on top of the bf16 storage rounding (see out_err)
TOL_FRO = 5e-3  # relative Frobenius error: h, y and out rounded to bf16 once each (about 2e-3 together)


def _assert_close(tag, got, want):
    e = errs(got, want)
    print(f"{tag}: out_err {e['out_err']:.3e}  max/RMS {e['max_rms']:.3e}  Frobenius {e['fro']:.3e}")
    assert e["out_err"] < TOL_BF16 and e["fro"] < TOL_FRO, tag


def _shape(cfg, fp8=False):
    return B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8)


@pytest.mark.parametrize("T,d,E,k", [(256, 256, 16, 2), (1000, 384, 20, 3), (4096, 2048, 64, 6), (3, 128, 8, 8)])
def test_permute_tables_and_rows(libmoe, T, d, E, k):
    cfg = I.MoEConfig("p", T, d, E, 1, k, 128, 0.05, seed=T)
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    ref = oracle_route(x, wr, torch.zeros(E), k)
    p = O.permutation(ref["idx"], E)
    s = _shape(cfg)
    idx = torch.tensor(ref["idx"], device=DEV)
    off = torch.tensor(p["offsets"], device=DEV)
    ws = B.alloc_workspace(s)
    xp, _, ptok, inv = B.moe_permute(s, x, idx, off, ws=ws)
    np.testing.assert_array_equal(ptok.cpu().numpy(), p["perm_token"])
    np.testing.assert_array_equal(inv.cpu().numpy(), p["inv_pos"])
    assert torch.equal(xp, x[ptok.long()])
    assert B.moe_get_device_status(ws) == 0


def test_permute_rejects_inconsistent_offsets(libmoe):
    cfg = I.CONFIGS["tiny"]
    s = _shape(cfg)
    x = I.make_x(cfg, DEV)
    idx = torch.zeros(cfg.T, cfg.k, dtype=torch.int32, device=DEV)
    idx[:, 1] = 1
    off = torch.zeros(cfg.E + 1, dtype=torch.int32, device=DEV)  # claims no rows at all
    ws = B.alloc_workspace(s)
    B.moe_permute(s, x, idx, off, ws=ws)
    assert B.moe_get_device_status(ws) == 7  # MOE_ERR_DEVICE
    assert B.moe_get_device_status(ws) == 0  # read clears it


def _expert_inputs(cfg):
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV)
    ref = oracle_route(x, wr, b, cfg.k)
    p = O.permutation(ref["idx"], cfg.E)
    wgu, wd = I.make_experts(cfg, DEV)
    return x, wr, b, ref, p, wgu, wd


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_expert_ffn_groups(libmoe, name):
    cfg = I.CONFIGS[name]
    x, wr, b, ref, p, wgu, wd = _expert_inputs(cfg)
    s = _shape(cfg)
    xp = x[torch.tensor(p["perm_token"], device=DEV).long()].contiguous()
    off = torch.tensor(p["offsets"], device=DEV)
    y = B.moe_expert_ffn(s, xp, None, x, off, wgu, wd)
    torch.cuda.synchronize()
    xn = np64(x)
    Tk = cfg.T * cfg.k
    yg = np64(y)
    # every routed group, shared experts on <= 512 tokens
    got, want = [], []
    for e in range(cfg.E):
        lo, hi = p["offsets"][e], p["offsets"][e + 1]
        if hi > lo:
            want.append(O.swiglu_expert(xn[p["perm_token"][lo:hi]], np64(wgu[e]), np64(wd[e])))
            got.append(yg[lo:hi])
    nt = min(cfg.T, 512)
    for si in range(cfg.S):
        want.append(O.swiglu_expert(xn[:nt], np64(wgu[cfg.E + si]), np64(wd[cfg.E + si])))
        got.append(yg[Tk + si * cfg.T: Tk + si * cfg.T + nt])
    _assert_close(f"{name}: expert FFN, every expert", np.concatenate(got), np.concatenate(want))


def test_combine(libmoe):
    cfg = I.CONFIGS["mid"]
    rng = np.random.default_rng(0)
    T, k, S, d = cfg.T, cfg.k, cfg.S, cfg.d
    y = torch.randn(T * k + S * T, d, device=DEV).to(torch.bfloat16)
    gate = torch.tensor(rng.dirichlet(np.ones(k), T).astype(np.float32), device=DEV)
    inv = torch.tensor(rng.permutation(T * k).reshape(T, k).astype(np.int32), device=DEV)
    out = B.moe_combine(_shape(cfg), y, gate, inv)
    ref = O.combine(np64(y), gate.cpu().numpy(), inv.cpu().numpy(), T, k, S)
    assert out_err(out, ref) < 1e-4  # an FP32 sum: only the bf16 store rounds


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_forward_full(libmoe, name):
    cfg = I.CONFIGS[name]
    x, wr, b, ref, p, wgu, wd = _expert_inputs(cfg)
    s = _shape(cfg)
    ws = B.alloc_workspace(s)
    out, idx, gate, counts = B.moe_forward(s, x, wr, b.clone(), wgu, wd, ws=ws)
    torch.cuda.synchronize()
    offsets = torch.tensor(O.offsets_from_counts(counts.cpu().numpy()))
    ties = check_routing(ref, idx, gate, counts, offsets, cfg.E)
    clean = np.nonzero(~(ref["boundary_tie"] | ref["order_tie"]))[0]
    tok = clean[:: max(1, cfg.T // 256)]  # every token of tiny, 256 spread tokens of mid
    yr = O.forward_rows(tok, np64(x), ref, lambda e: (np64(wgu[e]), np64(wd[e])), cfg.E, cfg.S)
    print(f"{name}: near-tied tokens {ties}")
    _assert_close(f"{name}: forward", np64(out)[tok], yr)
    out2, *_ = B.moe_forward(s, x, wr, b.clone(), wgu, wd, ws=ws)
    assert torch.equal(out, out2), "forward is deterministic"
    assert B.moe_get_device_status(ws) == 0


def _sampled_check(cfg, x, wr, b, wgu, wd, out, idx, gate, counts, logit_offset=None, n_tok=8):
    ref = oracle_route(x, wr, b, cfg.k, logit_offset)
    offsets = torch.tensor(O.offsets_from_counts(counts.cpu().numpy()))
    ties = check_routing(ref, idx, gate, counts, offsets, cfg.E)
    clean = np.nonzero(~(ref["boundary_tie"] | ref["order_tie"]))[0]
    rng = np.random.default_rng(cfg.T)
    tok = np.sort(rng.choice(clean, size=min(n_tok, clean.size), replace=False))
    cache = {}

    def get_expert(e):
        if e not in cache:
            cache.clear()
            cache[e] = (np64(wgu[e]), np64(wd[e]))
        return cache[e]

    yr = O.forward_rows(tok, np64(x), ref, get_expert, cfg.E, cfg.S)
    e = errs(np64(out)[tok], yr)
    print(f"{cfg.name}: sampled out_err {e['out_err']:.3e} (plain max/RMS {e['max_rms']:.3e}, "
          f"Frobenius {e['fro']:.3e})")
    assert e["fro"] < TOL_FRO
    return e["out_err"], ties


def test_skew_bias_trajectory(libmoe):
    """20 forward + bias-update steps on the Zipf-skewed decode workload; each step's
    routing is checked against the oracle and the bias bit for bit."""
    cfg = I.CONFIGS["skew"]
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    off = I.make_logit_offset(cfg, DEV)
    wgu, wd = I.make_experts(cfg, DEV)
    s = _shape(cfg)
    ws = B.alloc_workspace(s)
    bias = torch.zeros(cfg.E, dtype=torch.float32, device=DEV)
    loads = []
    for step in range(20):
        b_before = bias.clone()
        out, idx, gate, counts = B.moe_forward(s, x, wr, bias, wgu, wd, logit_offset=off, gamma=cfg.gamma,
                                               update_bias=True, ws=ws)
        torch.cuda.synchronize()
        ref = oracle_route(x, wr, b_before, cfg.k, off)
        offsets = torch.tensor(O.offsets_from_counts(counts.cpu().numpy()))
        check_routing(ref, idx, gate, counts, offsets, cfg.E)
        exp_b = O.bias_update(b_before.cpu().numpy(), counts.cpu().numpy(), cfg.T, cfg.k, cfg.gamma)
        np.testing.assert_array_equal(bias.cpu().numpy(), exp_b)
        st = O.load_stats(counts.cpu().numpy())
        loads.append(st["max_over_mean"])
        if step == 0:
            err, _ = _sampled_check(cfg, x, wr, b_before, wgu, wd, out, idx, gate, counts, logit_offset=off)
            assert err < TOL_BF16
    print("skew max/mean load per step:", " ".join(f"{v:.2f}" for v in loads))
    # overloaded experts were pushed down every step, underloaded ones up
    c0 = O.expert_counts(oracle_route(x, wr, torch.zeros(cfg.E), cfg.k, off)["idx"], cfg.E)
    hot = c0 > 2 * cfg.T * cfg.k / cfg.E  # strongly overloaded: still hot after 20 small steps
    assert np.all(bias.cpu().numpy()[hot] < 0)


def test_debug_wait_times_out(libmoe):
    s = _shape(I.CONFIGS["tiny"])
    ws = B.alloc_workspace(s)
    assert B.moe_get_device_status(ws) == 0
    B.moe_debug_wait_timeout(ws, 2000)
    assert B.moe_get_device_status(ws) == 6  # MOE_ERR_TIMEOUT
    assert B.moe_get_device_status(ws) == 0


def test_forward_group_limited(libmoe):
    cfg = I.CONFIGS["tiny"].with_(n_group=4, topk_group=2, k=3, seed=5)
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV)
    wgu, wd = I.make_experts(cfg, DEV)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, n_group=4, topk_group=2)
    out, idx, gate, counts = B.moe_forward(s, x, wr, b.clone(), wgu, wd)
    torch.cuda.synchronize()
    ref = oracle_route(x, wr, b, cfg.k, None, 4, 2)
    offsets = torch.tensor(O.offsets_from_counts(counts.cpu().numpy()))
    check_routing(ref, idx, gate, counts, offsets, cfg.E, 4, 2)
    clean = np.nonzero(~(ref["boundary_tie"] | ref["order_tie"]))[0]
    yr = O.forward_rows(clean, np64(x), ref, lambda e: (np64(wgu[e]), np64(wd[e])), cfg.E, cfg.S)
    _assert_close("group-limited forward", np64(out)[clean], yr)


def test_forward_no_tokens(libmoe):
    # T = 0: token buffers may be NULL; counts and offsets are zero, the bias is unchanged
    cfg = I.MoEConfig("empty", 0, 256, 16, 1, 2, 128, 0.02)
    s = _shape(cfg)
    wr = I.make_router(cfg, DEV)
    wgu, wd = I.make_experts(cfg, DEV)
    x = torch.empty(0, cfg.d, dtype=torch.bfloat16, device=DEV)
    bias = torch.full((cfg.E,), 0.25, dtype=torch.float32, device=DEV)
    ws = B.alloc_workspace(s)
    out, idx, gate, counts = B.moe_forward(s, x, wr, bias, wgu, wd, gamma=0.001, update_bias=True, ws=ws)
    _, _, c2, offsets = B.moe_route(s, x, wr, bias, ws=ws)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.d) and idx.shape == (0, cfg.k)
    assert not torch.any(counts) and not torch.any(c2) and not torch.any(offsets)
    assert torch.all(bias == 0.25)
    assert B.moe_get_device_status(ws) == 0
