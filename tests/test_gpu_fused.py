"""The expert FFN with the dispatch fused into the gate/up GEMM's operand load
(routed rows gathered from x through the permutation table, moe_expert_ffn_gather)
against the expert FFN on the permuted copy (moe_permute -> moe_expert_ffn), on
the same routing.  Both run the same MMAs on the same operand bytes in the same
order, so y must agree bit for bit; the copy-based path is in turn checked
against the oracle in test_gpu_layer / test_gpu_fp8.  moe_forward, whichever
dispatch form it picks for the shape, must equal the step-by-step calls."""
import pytest
import torch

from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(cfg, fp8):
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV)
    if fp8:
        wgu, gs, wd, ds = I.make_experts_fp8(cfg, DEV)
    else:
        (wgu, wd), gs, ds = I.make_experts(cfg, DEV), None, None
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8=fp8, n_group=cfg.n_group,
                     topk_group=cfg.topk_group)
    return s, x, wr, b, wgu, gs, wd, ds


def _compare_ffn(cfg, fp8=False, off=None):
    s, x, wr, b, wgu, gs, wd, ds = _inputs(cfg, fp8)
    ws = B.alloc_workspace(s)
    idx, gate, counts, offsets = B.moe_route(s, x, wr, b, off, ws=ws)
    xp, xps, ptok, inv = B.moe_permute(s, x, idx, offsets, ws=ws)
    _, _, ptok2, inv2 = B.moe_permute(s, x, idx, offsets, ws=ws, rows=False)
    y_copy = B.moe_expert_ffn(s, xp, xps, x, offsets, wgu, wd, gs, ds, ws=ws)
    y_gath = B.moe_expert_ffn_gather(s, x, ptok2, offsets, wgu, wd, gs, ds, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    assert torch.equal(ptok, ptok2) and torch.equal(inv, inv2)
    diff = (y_gath.float() - y_copy.float()).abs().max().item()
    assert torch.equal(y_gath, y_copy), f"gathered FFN differs from the copy-based FFN (max |diff| {diff})"
    return counts


def _compare_forward(cfg, fp8=False, off=None):
    s, x, wr, b, wgu, gs, wd, ds = _inputs(cfg, fp8)
    ws = B.alloc_workspace(s)
    out, idx, gate, counts = B.moe_forward(s, x, wr, b.clone(), wgu, wd, logit_offset=off, w_gu_scale=gs,
                                           w_down_scale=ds, ws=ws)
    i2, g2, c2, offsets = B.moe_route(s, x, wr, b, off)
    if B.forward_gathers(s):
        _, _, ptok, inv = B.moe_permute(s, x, i2, offsets, rows=False)
        y = B.moe_expert_ffn_gather(s, x, ptok, offsets, wgu, wd, gs, ds)
    else:
        xp, xps, ptok, inv = B.moe_permute(s, x, i2, offsets)
        y = B.moe_expert_ffn(s, xp, xps, x, offsets, wgu, wd, gs, ds)
    ref = B.moe_combine(s, y, g2, inv)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    assert torch.equal(idx, i2) and torch.equal(gate, g2) and torch.equal(counts, c2)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("name", ["tiny", "mid", "v3grp"])
def test_gather_matches_copy_bf16(libmoe, name):
    _compare_ffn(I.CONFIGS[name])


@pytest.mark.parametrize("T,d,E,S,k,I_", [(77, 640, 5, 1, 5, 256), (1, 128, 8, 1, 8, 128), (3, 256, 16, 0, 2, 128),
                                          (1500, 256, 4, 2, 2, 384), (600, 384, 2, 1, 1, 128)])
def test_gather_ragged_bf16(libmoe, T, d, E, S, k, I_):
    # group sizes that are not multiples of 16, groups of > 256 tokens (several
    # chunks), single-token layers, no shared expert, several shared experts
    cfg = I.MoEConfig("rag", T, d, E, S, k, I_, 0.05, bias_uniform=0.1, seed=T + E)
    counts = _compare_ffn(cfg)
    if T >= 600:
        assert int(counts.max()) > 256


def test_gather_matches_copy_skew(libmoe):
    cfg = I.CONFIGS["skew"]
    _compare_ffn(cfg, off=I.make_logit_offset(cfg, DEV))


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_gather_matches_copy_fp8(libmoe, name):
    _compare_ffn(I.CONFIGS[name], fp8=True)


@pytest.mark.parametrize("T,d,E,S,k,I_", [(77, 640, 5, 1, 5, 256), (3, 256, 16, 0, 2, 128), (1500, 256, 4, 2, 2, 384)])
def test_gather_ragged_fp8(libmoe, T, d, E, S, k, I_):
    cfg = I.MoEConfig("rag", T, d, E, S, k, I_, 0.05, bias_uniform=0.1, seed=T + E)
    _compare_ffn(cfg, fp8=True)


def test_gather_matches_copy_v3(libmoe):
    _compare_ffn(I.CONFIGS["v3"])


def test_gather_matches_copy_v3fp8(libmoe):
    _compare_ffn(I.CONFIGS["v3fp8"], fp8=True)


@pytest.mark.parametrize("name,fp8", [("tiny", False), ("mid", False), ("tiny", True), ("mid", True)])
def test_forward_equals_steps(libmoe, name, fp8):
    cfg = I.CONFIGS[name]
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8=fp8)
    assert B.forward_gathers(s) == (cfg.T * cfg.k <= 4096)
    _compare_forward(cfg, fp8)


def test_forward_equals_steps_skew(libmoe):
    cfg = I.CONFIGS["skew"]
    _compare_forward(cfg, off=I.make_logit_offset(cfg, DEV))
