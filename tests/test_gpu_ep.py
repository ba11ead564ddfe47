"""GPU parity of the expert-parallel path: moe_ep_regroup against a numpy restatement
(a stable sort of the received rows by local expert), bit for bit, and the whole
expert-parallel layer with G ranks emulated as threads of this process on one GPU
(exchanges as device copies, no kernel waiting on another) against moe_forward on
each rank's tokens -- bit for bit: every output element of the expert GEMMs is summed
over K in an order fixed by its feature block alone, whichever tokens share its tile --
and against the oracle."""
import threading

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import ep
from sparse_moe_layer_12_b300 import inputs as I
from moe_testutil import errs, np64, oracle_route

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _regroup_ref(counts, src, to_local):
    G, E_loc = counts.shape
    expert_of_row = np.concatenate([np.repeat(np.arange(E_loc), counts[s]) for s in range(G)])
    order = np.argsort(expert_of_row, kind="stable")
    if to_local:
        return src[order]
    dst = np.empty_like(src)
    dst[order] = src
    return dst


@pytest.mark.parametrize("G,E_loc,d,fp8", [(4, 8, 384, False), (2, 128, 256, True), (8, 32, 7168, False),
                                           (1, 4, 128, False)])
def test_regroup_bit_exact(libmoe, G, E_loc, d, fp8):
    rng = np.random.default_rng(G * E_loc)
    counts = rng.integers(0, 40, size=(G, E_loc)).astype(np.int32)
    counts[0, 0] = 0  # empty segments, first and in the middle
    counts[G // 2, E_loc // 2] = 0
    rows = int(counts.sum())
    if fp8:
        src = torch.randint(0, 255, (rows, d), dtype=torch.uint8, device=DEV).view(torch.float8_e4m3fn)
        ssc = torch.rand(rows, d // 128, device=DEV)
    else:
        src = torch.randn(rows, d, device=DEV).to(torch.bfloat16)
        ssc = None
    s = B.make_shape(16, 256, 16, 1, 2, 128)
    ws = B.alloc_workspace(s)
    c = torch.tensor(counts, device=DEV)
    dst, dsc, off = B.moe_ep_regroup(c, src, True, ws, src_scale=ssc)
    back, bsc, _ = B.moe_ep_regroup(c, dst, False, ws, src_scale=dsc)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    raw = src.view(torch.uint8) if fp8 else src.view(torch.int16)
    want = _regroup_ref(counts, raw.cpu().numpy(), True)
    got = (dst.view(torch.uint8) if fp8 else dst.view(torch.int16)).cpu().numpy()
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(off.cpu().numpy(), O.offsets_from_counts(counts.sum(0)))
    assert torch.equal(back.view(torch.uint8), src.view(torch.uint8))
    if fp8:
        np.testing.assert_array_equal(dsc.cpu().numpy(), _regroup_ref(counts, ssc.cpu().numpy(), True))
        assert torch.equal(bsc, ssc)


def test_regroup_rejects_inconsistent_counts(libmoe):
    s = B.make_shape(16, 256, 16, 1, 2, 128)
    ws = B.alloc_workspace(s)
    c = torch.tensor([[3, 4], [5, -1]], dtype=torch.int32, device=DEV)
    src = torch.zeros(11, 128, dtype=torch.bfloat16, device=DEV)
    _, _, off = B.moe_ep_regroup(c, src, True, ws)
    assert B.moe_get_device_status(ws) == 7  # MOE_ERR_DEVICE
    assert not torch.any(off)
    c = torch.tensor([[3, 4], [5, 0]], dtype=torch.int32, device=DEV)  # 12 rows claimed, 11 given
    B.moe_ep_regroup(c, src, True, ws)
    assert B.moe_get_device_status(ws) == 7


def _ep_layer(cfg, G, fp8=False, pow2=False):
    """Per-rank tokens, the layer's weights split over G ranks, and G CudaOps."""
    wr = I.make_router(cfg, DEV)
    bias = I.make_bias(cfg, DEV)
    if fp8:
        wgu, gs, wd, ds = I.make_experts_fp8(cfg, DEV, pow2=pow2)
    else:
        (wgu, wd), gs, ds = I.make_experts(cfg, DEV), None, None
    xs = [I.make_x(cfg.with_(seed=cfg.seed + 100 * r), DEV) for r in range(G)]
    ops = []
    for r in range(G):
        lo, hi = ep.expert_range(cfg.E, G, r)
        sc = None
        if fp8:
            sc = dict(gate_up_local=gs[lo:hi], down_local=ds[lo:hi], gate_up_shared=gs[cfg.E:],
                      down_shared=ds[cfg.E:])
        ops.append(ep.CudaOps(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, G, wr, wgu[lo:hi], wd[lo:hi], wgu[cfg.E:],
                              wd[cfg.E:], fp8=fp8, scales=sc, pow2=pow2))
    return wr, bias, wgu, wd, gs, ds, xs, ops


def _run_ep(cfg, G, ops, xs, bias):
    hub = ep.LocalTransport(G)
    res, failures = [None] * G, []
    biases = [bias.clone() for _ in range(G)]

    def run(r):
        try:
            rank = ep.EPRank(ops[r], hub.view(r), cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, r, G)
            res[r] = rank.forward(xs[r], biases[r], update_bias=True, gamma=cfg.gamma)
        except Exception as exc:
            failures.append(exc)
            hub._barrier.abort()

    th = [threading.Thread(target=run, args=(r,)) for r in range(G)]
    for t in th:
        t.start()
    for t in th:
        t.join(300)
    torch.cuda.synchronize()
    assert not failures, failures
    return res, biases


@pytest.mark.parametrize("name,G,T", [("tiny", 2, 256), ("mid", 4, 1024)])
def test_ep_layer_matches_forward(libmoe, name, G, T):
    cfg = I.CONFIGS[name].with_(T=T)
    wr, bias, wgu, wd, _, _, xs, ops = _ep_layer(cfg, G)
    res, biases = _run_ep(cfg, G, ops, xs, bias)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    counts_all = torch.zeros(cfg.E, dtype=torch.int32, device=DEV)
    for r in range(G):
        assert ops[r].device_status() == 0
        out, idx, gate, counts = res[r]
        ref_out, ref_idx, ref_gate, ref_counts = B.moe_forward(s, xs[r], wr, bias.clone(), wgu, wd)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx) and torch.equal(counts, ref_counts)
        e = errs(np64(out), np64(ref_out))
        print(f"{name} EP rank {r}/{G}: vs moe_forward bit-identical {torch.equal(out, ref_out)}, "
              f"out_err {e['out_err']:.2e} Frobenius {e['fro']:.2e}")
        assert torch.equal(out, ref_out)
        counts_all += counts
        # against the oracle on 64 of the rank's tokens
        ref = oracle_route(xs[r], wr, bias, cfg.k)
        clean = np.nonzero(~(ref["boundary_tie"] | ref["order_tie"]))[0][:64]
        yr = O.forward_rows(clean, np64(xs[r]), ref, lambda ex: (np64(wgu[ex]), np64(wd[ex])), cfg.E, cfg.S)
        eo = errs(np64(out)[clean], yr)
        print(f"{name} EP rank {r}/{G}: vs the oracle out_err {eo['out_err']:.2e} Frobenius {eo['fro']:.2e}")
        assert eo["out_err"] < 2e-2 and eo["fro"] < 5e-3
    want_b = O.bias_update(bias.cpu().numpy(), counts_all.cpu().numpy(), cfg.T * G, cfg.k, cfg.gamma)
    for r in range(G):
        np.testing.assert_array_equal(biases[r].cpu().numpy(), want_b)


@pytest.mark.parametrize("pow2", [False, True])
def test_ep_layer_fp8(libmoe, pow2):
    cfg = I.CONFIGS["tiny"]
    G = 2
    wr, bias, wgu, wd, gs, ds, xs, ops = _ep_layer(cfg, G, fp8=True, pow2=pow2)
    res, _ = _run_ep(cfg, G, ops, xs, bias)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8=True, pow2=pow2)
    for r in range(G):
        assert ops[r].device_status() == 0
        out = res[r][0]
        ref_out, *_ = B.moe_forward(s, xs[r], wr, bias.clone(), wgu, wd, w_gu_scale=gs, w_down_scale=ds)
        torch.cuda.synchronize()
        e = errs(np64(out), np64(ref_out))
        print(f"tiny fp8 (pow2 {pow2}) EP rank {r}/{G}: vs moe_forward bit-identical {torch.equal(out, ref_out)}, "
              f"out_err {e['out_err']:.2e} Frobenius {e['fro']:.2e}")
        assert torch.equal(out, ref_out)
