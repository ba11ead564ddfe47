"""moe_expert_ffn_static -- the expert FFN for callers that cannot allocate device
memory (a plugin whose host framework owns all device memory and offers no
workspace, or a serving loop that forbids cudaMalloc after start-up).  It runs the
same kernels as moe_expert_ffn on a fixed scratch array inside the library.

Checked through the C ABI against moe_expert_ffn, on two calls in a row (the
array keeps the previous call's contents), in bf16 and FP8, at decode-sized layers
that fit the array; a layer that does not fit must be refused before anything
runs; the device's free memory must not change across the calls; an inconsistent
offsets array must come back as MOE_ERR_DEVICE through the array's status word.
This file is collected last so that a run that stops at its first failure has
already run every other test."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import inputs as I
from moe_testutil import np64, oracle_route, out_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_BF16 = 2e-2


def _case(cfg):
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    ref = oracle_route(x, wr, I.make_bias(cfg, DEV), cfg.k)
    p = O.permutation(ref["idx"], cfg.E)
    wgu, wd = I.make_experts(cfg, DEV)
    xp = x[torch.tensor(p["perm_token"], device=DEV).long()].contiguous()
    off = torch.tensor(p["offsets"], device=DEV)
    return x, xp, off, wgu, wd


@pytest.mark.parametrize("cfg", [
    I.CONFIGS["tiny"],
    I.MoEConfig("decode", 256, 2048, 64, 2, 6, 1408, None, bias_uniform=0.05, seed=7),
    I.MoEConfig("decode2", 40, 1024, 32, 1, 4, 512, 0.02, seed=11),
], ids=lambda c: c.name)
def test_static_scratch_matches_workspace_call(libmoe, cfg):
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    x, xp, off, wgu, wd = _case(cfg)
    y_ref = B.moe_expert_ffn(s, xp, None, x, off, wgu, wd)
    for call in range(2):
        y = B.moe_expert_ffn_static(s, xp, None, x, off, wgu, wd)
        torch.cuda.synchronize()
        err = out_err(np64(y), np64(y_ref))
        assert err < TOL_BF16, f"call {call}: err {err:.3e}"
        assert torch.equal(y, y_ref), f"call {call}: same kernels, same schedule -> same bits"


def test_static_scratch_after_a_larger_layer(libmoe):
    # a second, smaller layer right after a larger one: stale contents must not leak
    big = I.MoEConfig("decode", 256, 2048, 64, 2, 6, 1408, None, seed=3)
    small = I.CONFIGS["tiny"]
    for cfg in (big, small):
        s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
        x, xp, off, wgu, wd = _case(cfg)
        y = B.moe_expert_ffn_static(s, xp, None, x, off, wgu, wd)
        y_ref = B.moe_expert_ffn(s, xp, None, x, off, wgu, wd)
        torch.cuda.synchronize()
        assert out_err(np64(y), np64(y_ref)) < TOL_BF16
        np.testing.assert_array_equal(y.view(torch.int16).cpu().numpy(), y_ref.view(torch.int16).cpu().numpy())


def test_static_scratch_refuses_layers_that_do_not_fit(libmoe):
    cfg = I.CONFIGS["v3"]  # T=8192 needs far more than the fixed array
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    t = torch.empty(16, dtype=torch.uint8, device=DEV)
    p = t.data_ptr()
    import ctypes
    code = B.load().moe_expert_ffn_static(ctypes.byref(s), p, None, p, p, p, None, p, None, p, None)
    assert code == 4  # MOE_ERR_WORKSPACE, nothing enqueued


def _fp8_case(cfg):
    x = I.make_x(cfg, DEV)
    ref = oracle_route(x, I.make_router(cfg, DEV), I.make_bias(cfg, DEV), cfg.k)
    p = O.permutation(ref["idx"], cfg.E)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8=True)
    idx = torch.tensor(ref["idx"], device=DEV)
    off = torch.tensor(p["offsets"], device=DEV)
    xp, xps, _, _ = B.moe_permute(s, x, idx, off)
    wgu_b, wd_b = I.make_experts(cfg, DEV)
    wgu, gs = B.moe_quantize_weights_fp8(wgu_b)
    wd, ds = B.moe_quantize_weights_fp8(wd_b)
    return s, x, xp, xps, off, wgu, gs, wd, ds


def test_static_scratch_fp8_matches_workspace_call(libmoe):
    # a decode-sized FP8 layer: E4M3 rows and 1x128 scales from moe_permute, weights
    # quantised per 128x128 by the library; the same bits as the workspace call, twice
    cfg = I.MoEConfig("decode_fp8", 96, 1024, 32, 1, 4, 512, 0.02, seed=13)
    s, x, xp, xps, off, wgu, gs, wd, ds = _fp8_case(cfg)
    y_ref = B.moe_expert_ffn(s, xp, xps, x, off, wgu, wd, gs, ds)
    for call in range(2):
        y = B.moe_expert_ffn_static(s, xp, xps, x, off, wgu, wd, gs, ds)
        torch.cuda.synchronize()
        assert B.moe_get_static_device_status() == 0
        assert torch.equal(y, y_ref), f"call {call}"


def test_static_scratch_allocates_nothing(libmoe):
    cfg = I.MoEConfig("decode", 256, 2048, 64, 2, 6, 1408, None, seed=7)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    x, xp, off, wgu, wd = _case(cfg)
    y = torch.empty(cfg.rows_total, cfg.d, dtype=torch.bfloat16, device=DEV)
    B.moe_expert_ffn_static(s, xp, None, x, off, wgu, wd, y=y)  # first call: modules loaded, address looked up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        B.moe_expert_ffn_static(s, xp, None, x, off, wgu, wd, y=y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device memory changed by {free0 - free1} bytes"
    assert B.moe_get_static_device_status() == 0


def test_static_scratch_reports_inconsistent_offsets(libmoe):
    # offsets[E] != T*k: the schedule kernel flags it (it reads offsets[0..E] only and
    # schedules no tile), and the status word of the array says so
    cfg = I.CONFIGS["tiny"]
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    x, xp, off, wgu, wd = _case(cfg)
    bad = off.clone()
    bad[-1] = cfg.T * cfg.k - 1
    B.moe_expert_ffn_static(s, xp, None, x, bad, wgu, wd)
    assert B.moe_get_static_device_status() == 7  # MOE_ERR_DEVICE
    assert B.moe_get_static_device_status() == 0  # the read clears it
    y = B.moe_expert_ffn_static(s, xp, None, x, off, wgu, wd)
    y_ref = B.moe_expert_ffn(s, xp, None, x, off, wgu, wd)
    torch.cuda.synchronize()
    assert B.moe_get_static_device_status() == 0
    assert torch.equal(y, y_ref)
