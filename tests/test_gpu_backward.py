"""GPU parity of moe_backward (the layer's gradients for a fixed routing) against
the float64 backward oracle on the same seeded inputs and the oracle's own routing:
whole tensors on small layers (ragged expert groups, experts that get no token, two
shared experts, I not a multiple of 256), sampled tokens and one expert on the
V3-shaped layer, and run-to-run determinism.

Tolerances.  Two measures per output: out_err (the largest error beyond the bf16
rounding of the output itself, over the RMS of the reference) and the relative
Frobenius error.  The kernels keep a, u and dh in FP32, store h, dy = g dout,
[da du] and the per-row dx contributions in bf16 (relative rounding 2^-9 each)
and accumulate every contraction in FP32.  The same roundings replayed in float64
(a model of the kernels' arithmetic, not of their code) give out_err 0.011 /
0.012 (dx), 0.006 / 0.007 (dw_router), 0.021 / 0.054 (dw_gate_up) and 0.024 /
0.047 (dw_down) on the tiny / mid1k layers, Frobenius errors below 0.5 %; the
maximum grows with the number of elements.  The bounds leave about 1.5x over the
larger of those and of the measured values; a wrong index or a dropped term
moves the Frobenius error to O(1).
"""
import numpy as np
import pytest
import torch

from oracle import moe_backward as BW
from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import inputs as I
from moe_testutil import np64, oracle_route, out_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {"dx": 2.5e-2, "dw_router": 2e-2, "dw_gate_up": 8e-2, "dw_down": 8e-2}
TOL_FRO = 6e-3


def fro_err(got, ref) -> float:
    g = np64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(g - ref) / np.linalg.norm(ref))

CASES = {
    "tiny": I.CONFIGS["tiny"],
    # ragged groups, 2 shared experts, 4 experts that no token picks
    "ragged": I.MoEConfig("ragged", 300, 384, 20, 2, 3, 256, 0.05, bias_uniform=0.05, seed=5),
    # I = 1408 (not a multiple of 256), 64 + 2 experts, top-6
    "mid1k": I.CONFIGS["mid"].with_(name="mid1k", T=1024),
}
DEAD = {"ragged": 4}


def _inputs(cfg, dead=0):
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV)
    off = I.make_logit_offset(cfg, DEV)
    if dead:
        off = torch.zeros(cfg.E, dtype=torch.float32, device=DEV) if off is None else off
        off[:dead] = -40.0  # s ~ 4e-18: never among the top k
    wgu, wd = I.make_experts(cfg, DEV)
    dout = I.make_dout(cfg, DEV)
    ref = oracle_route(x, wr, b, cfg.k, off)
    idx = torch.tensor(ref["idx"], dtype=torch.int32, device=DEV)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    return s, x, wr, off, wgu, wd, dout, idx


def _run(s, x, wr, off, wgu, wd, dout, idx, ws=None):
    ws = B.alloc_backward_workspace(s) if ws is None else ws
    g = B.moe_backward(s, x, wr, wgu, wd, idx, dout, logit_offset=off, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    return g, ws


@pytest.mark.parametrize("name", list(CASES))
def test_backward_whole_tensors(libmoe, name):
    cfg = CASES[name]
    dead = DEAD.get(name, 0)
    s, x, wr, off, wgu, wd, dout, idx = _inputs(cfg, dead)
    (dx, dwr, dwgu, dwd), ws = _run(s, x, wr, off, wgu, wd, dout, idx)
    ref = BW.backward(np64(x), np64(wr), np64(wgu), np64(wd), idx.cpu().numpy(), np64(dout), cfg.S,
                      None if off is None else off.cpu().numpy())
    got = {"dx": dx, "dw_router": dwr, "dw_gate_up": dwgu, "dw_down": dwd}
    errs = {n: (out_err(g, ref[n]), fro_err(g, ref[n])) for n, g in got.items()}
    print(f"{name}: " + ", ".join(f"{n} {e:.3e} (fro {f:.2e})" for n, (e, f) in errs.items()))
    for n, (e, f) in errs.items():
        assert e < TOL[n] and f < TOL_FRO, (n, e, f)
    if dead:  # experts without tokens: exactly zero gradients
        assert not torch.any(dwgu[:dead]) and not torch.any(dwd[:dead]) and not torch.any(dwr[:dead])
    # deterministic: the same bits again
    dx2, dwr2, dwgu2, dwd2 = B.moe_backward(s, x, wr, wgu, wd, idx, dout, logit_offset=off, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2) and torch.equal(dwr, dwr2) and torch.equal(dwgu, dwgu2) and torch.equal(dwd, dwd2)


def test_backward_v3_sampled(libmoe):
    cfg = I.CONFIGS["v3"]
    s, x, wr, off, wgu, wd, dout, idx = _inputs(cfg)
    (dx, dwr, dwgu, dwd), ws = _run(s, x, wr, off, wgu, wd, dout, idx)
    del ws
    idx_np = idx.cpu().numpy()
    xn, dn, wrn = np64(x), np64(dout), np64(wr)
    cache = {}

    def get_expert(e):
        if e not in cache:
            cache.clear()
            cache[e] = (np64(wgu[e]), np64(wd[e]))
        return cache[e]

    # dx and dz of sampled tokens (every expert they picked, and the shared expert)
    tok = np.sort(np.random.default_rng(1).choice(cfg.T, size=4, replace=False))
    ref = BW.backward_lazy(xn[tok], wrn, get_expert, idx_np[tok], dn[tok], cfg.E, cfg.S)
    dxs = dx[torch.tensor(tok, device=DEV)]
    e_dx, f_dx = out_err(dxs, ref["dx"]), fro_err(dxs, ref["dx"])
    # dW of the routed expert with the fewest (non-zero) tokens, from its own tokens
    counts = np.bincount(idx_np.reshape(-1), minlength=cfg.E)
    e = int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    mine = np.nonzero((idx_np == e).any(axis=1))[0]
    one = BW.backward_lazy(xn[mine], wrn, get_expert, idx_np[mine], dn[mine], cfg.E, cfg.S, dw_experts=[e],
                           need_dx=False)
    e_gu, f_gu = out_err(dwgu[e], one["dw"][e][0]), fro_err(dwgu[e], one["dw"][e][0])
    e_dn, f_dn = out_err(dwd[e], one["dw"][e][1]), fro_err(dwd[e], one["dw"][e][1])
    print(f"v3: dx {e_dx:.3e} (fro {f_dx:.2e}; tokens {tok.tolist()}), expert {e} ({counts[e]} tokens): "
          f"dw_gate_up {e_gu:.3e} (fro {f_gu:.2e}), dw_down {e_dn:.3e} (fro {f_dn:.2e})")
    assert e_dx < TOL["dx"] and e_gu < TOL["dw_gate_up"] and e_dn < TOL["dw_down"]
    assert max(f_dx, f_gu, f_dn) < TOL_FRO
    # experts without tokens (if any) have zero gradients
    for z in np.nonzero(counts == 0)[0][:4]:
        assert not torch.any(dwgu[z]) and not torch.any(dwr[z])


def test_backward_degenerate_layers(libmoe):
    # every expert chosen by every token (k = E), no shared expert; gates normalise over all E
    cfg = I.MoEConfig("allk", 96, 256, 4, 0, 4, 128, 0.05, seed=11)
    s, x, wr, off, wgu, wd, dout, idx = _inputs(cfg)
    (dx, dwr, dwgu, dwd), _ = _run(s, x, wr, off, wgu, wd, dout, idx)
    ref = BW.backward(np64(x), np64(wr), np64(wgu), np64(wd), idx.cpu().numpy(), np64(dout), 0)
    for n, g in (("dx", dx), ("dw_router", dwr), ("dw_gate_up", dwgu), ("dw_down", dwd)):
        assert out_err(g, ref[n]) < TOL[n] and fro_err(g, ref[n]) < TOL_FRO, n


def test_backward_no_tokens(libmoe):
    # T = 0: nothing to differentiate, every weight gradient is zero
    s = B.make_shape(0, 256, 8, 1, 2, 128)
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    cfg = I.MoEConfig("empty", 0, 256, 8, 1, 2, 128, 0.05)
    wr = I.make_router(cfg, DEV)
    wgu, wd = I.make_experts(cfg, DEV)
    idx = torch.empty(0, 2, dtype=torch.int32, device=DEV)
    out = (torch.empty(0, 256, dtype=torch.bfloat16, device=DEV),
           torch.full((8, 256), 7.0, device=DEV),
           torch.full((9, 256, 256), 7.0, device=DEV).to(torch.bfloat16),
           torch.full((9, 256, 128), 7.0, device=DEV).to(torch.bfloat16))
    ws = B.alloc_backward_workspace(s)
    dx, dwr, dwgu, dwd = B.moe_backward(s, x, wr, wgu, wd, idx, x, ws=ws, out=out)
    torch.cuda.synchronize()
    assert not torch.any(dwr) and not torch.any(dwgu) and not torch.any(dwd)
    assert B.moe_get_device_status(ws) == 0


def test_backward_rejects_out_of_range_experts(libmoe):
    # an expert index outside [0, E) is caught on the device (MOE_ERR_DEVICE), nothing is
    # read or written out of bounds, and the workspace is usable again after the status read
    cfg = CASES["tiny"]
    s, x, wr, off, wgu, wd, dout, idx = _inputs(cfg)
    bad = idx.clone()
    bad[5, 1] = cfg.E
    ws = B.alloc_backward_workspace(s)
    B.moe_backward(s, x, wr, wgu, wd, bad, dout, logit_offset=off, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 7
    assert B.moe_get_device_status(ws) == 0
    B.moe_backward(s, x, wr, wgu, wd, idx, dout, logit_offset=off, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0


def test_forward_and_backward_at_the_largest_k_and_s(libmoe):
    # k = 16 of 32 routed experts and S = 8 shared experts (the library's limits)
    cfg = I.MoEConfig("maxks", 64, 256, 32, 8, 16, 128, 0.05, seed=21)
    s, x, wr, off, wgu, wd, dout, idx = _inputs(cfg)
    b = torch.zeros(cfg.E, dtype=torch.float32, device=DEV)
    out, fidx, gate, counts = B.moe_forward(s, x, wr, b, wgu, wd)
    (dx, dwr, dwgu, dwd), _ = _run(s, x, wr, off, wgu, wd, dout, idx)
    torch.cuda.synchronize()
    from oracle import moe_oracle as O
    ref_f = O.forward(np64(x), np64(wr), np.zeros(cfg.E, np.float32), np64(wgu), np64(wd), cfg.k, cfg.S)
    r = ref_f["route"]
    clean = ~(r["boundary_tie"] | r["order_tie"])
    assert np.array_equal(fidx.cpu().numpy()[clean], r["idx"][clean])
    assert out_err(np64(out)[clean], ref_f["out"][clean]) < 2e-2
    ref = BW.backward(np64(x), np64(wr), np64(wgu), np64(wd), idx.cpu().numpy(), np64(dout), cfg.S)
    for n, g in (("dx", dx), ("dw_router", dwr), ("dw_gate_up", dwgu), ("dw_down", dwd)):
        assert out_err(g, ref[n]) < TOL[n] and fro_err(g, ref[n]) < TOL_FRO, n
