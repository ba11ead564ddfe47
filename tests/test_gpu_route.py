"""GPU parity of moe_route (through the C ABI) against the oracle router.

Indices, counts and offsets must match bit for bit, except at tokens whose
k-th and (k+1)-th (or two chosen) biased scores lie within 1e-5, where the
choice must be a valid one; gates within 2e-5 relative."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import inputs as I
from moe_testutil import check_routing, oracle_route

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_case(cfg, logit_offset=None, bias=None):
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV) if bias is None else bias
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, n_group=cfg.n_group, topk_group=cfg.topk_group)
    idx, gate, counts, offsets = B.moe_route(s, x, wr, b, logit_offset)
    ws = B.alloc_workspace(s)
    torch.cuda.synchronize()
    ref = oracle_route(x, wr, b, cfg.k, logit_offset, cfg.n_group, cfg.topk_group)
    ties = check_routing(ref, idx, gate, counts, offsets, cfg.E, cfg.n_group, cfg.topk_group)
    # deterministic run to run
    idx2, gate2, counts2, offsets2 = B.moe_route(s, x, wr, b, logit_offset, ws=ws)
    assert torch.equal(idx, idx2) and torch.equal(gate, gate2) and torch.equal(counts, counts2)
    assert B.moe_get_device_status(ws) == 0
    return ties


@pytest.mark.parametrize("name", ["tiny", "mid", "v3", "v3grp"])
def test_route_configs(libmoe, name):
    ties = _route_case(I.CONFIGS[name])
    print(f"{name}: near-tied tokens {ties}")


def test_route_skew_offsets(libmoe):
    cfg = I.CONFIGS["skew"]
    ties = _route_case(cfg, logit_offset=I.make_logit_offset(cfg, DEV))
    print(f"skew: near-tied tokens {ties}")


@pytest.mark.parametrize("T,d,E,k", [(200, 384, 20, 3), (1000, 256, 64, 16), (1, 128, 1, 1),
                                     (129, 128, 256, 8), (77, 640, 5, 5)])
def test_route_ragged(libmoe, T, d, E, k):
    cfg = I.MoEConfig("rag", T, d, E, 1, k, 128, 0.05, bias_uniform=0.1, seed=T + E)
    _route_case(cfg)


@pytest.mark.parametrize("T,d,E,k,ng,tg", [(500, 256, 64, 6, 8, 3), (130, 384, 256, 8, 8, 4), (77, 128, 32, 4, 4, 1),
                                           (300, 256, 16, 4, 4, 4)])
def test_route_group_limited(libmoe, T, d, E, k, ng, tg):
    cfg = I.MoEConfig("grp", T, d, E, 1, k, 128, 0.05, bias_uniform=0.1, seed=T + E, n_group=ng, topk_group=tg)
    _route_case(cfg)


def test_route_hand_worked_example(libmoe, golden_dir):
    # the 4x4 example padded to d = 128: exact integer logits, exact ties
    fx = json.load(open(os.path.join(golden_dir, "hand_4x4.json")))
    T, E, k = fx["T"], fx["E"], fx["k"]
    x = torch.zeros(T, 128, dtype=torch.bfloat16)
    x[:, :4] = torch.tensor(fx["x"], dtype=torch.bfloat16)
    wr = torch.zeros(E, 128, dtype=torch.bfloat16)
    wr[:, :4] = torch.tensor(fx["w_router"], dtype=torch.bfloat16)
    b = torch.tensor(fx["bias"], dtype=torch.float32)
    s = B.make_shape(T, 128, E, 1, k, 128)
    idx, gate, counts, offsets = B.moe_route(s, x.to(DEV), wr.to(DEV), b.to(DEV))
    ex = fx["expected"]
    np.testing.assert_array_equal(idx.cpu().numpy(), np.array(ex["idx"]))
    np.testing.assert_allclose(gate.cpu().numpy(), np.array(ex["gate"]), rtol=2e-6)
    np.testing.assert_array_equal(counts.cpu().numpy(), ex["counts"])
    np.testing.assert_array_equal(offsets.cpu().numpy(), ex["offsets"])


def test_bias_update_matches_oracle(libmoe):
    rng = np.random.default_rng(0)
    E, T, k = 256, 8192, 8
    s = B.make_shape(T, 128, E, 1, k, 128)
    b = torch.tensor(rng.uniform(-0.01, 0.01, E).astype(np.float32), device=DEV)
    counts = rng.multinomial(T * k, np.ones(E) / E).astype(np.int32)
    counts[:3] = T * k // E  # exact mean: no move
    c = torch.tensor(counts, device=DEV)
    ref = O.bias_update(b.cpu().numpy(), counts, T, k, 0.001)
    B.moe_bias_update(s, c, b, 0.001)
    np.testing.assert_array_equal(b.cpu().numpy(), ref)


def test_route_leaves_load_counters_clear(libmoe):
    """One launch per call: the load is summed in the workspace's control block, written
    out by the last block and cleared; calls of different shapes on one workspace."""
    big = B.make_shape(1000, 256, 64, 1, 6, 128)
    ws = B.alloc_workspace(big)
    for T, E, k, seed in [(1000, 64, 6, 1), (37, 16, 2, 2), (1000, 64, 6, 3), (513, 33, 8, 4)]:
        cfg = I.MoEConfig("ctl", T, 256, E, 1, k, 128, 0.05, bias_uniform=0.05, seed=seed)
        s = B.make_shape(T, 256, E, 1, k, 128)
        x, wr, b = I.make_x(cfg, DEV), I.make_router(cfg, DEV), I.make_bias(cfg, DEV)
        idx, gate, counts, offsets = B.moe_route(s, x, wr, b, ws=ws)
        torch.cuda.synchronize()
        want = np.bincount(idx.cpu().numpy().ravel(), minlength=E)
        np.testing.assert_array_equal(counts.cpu().numpy(), want)
        np.testing.assert_array_equal(offsets.cpu().numpy(), O.offsets_from_counts(want))
        assert not torch.any(ws[256:B.WS_CTRL_BYTES]), "load counters and ticket left clear"
        check_routing(oracle_route(x, wr, b, k), idx, gate, counts, offsets, E)
    assert B.moe_get_device_status(ws) == 0


@pytest.mark.parametrize("case", ["all_equal", "saturated"])
def test_route_degenerate_scores(libmoe, case):
    """Scores that defeat the candidate filter: every expert equal (x = 0: all of them
    candidates, the k lowest indices chosen, gates 1/k), and logits far beyond the
    sigmoid's range (s = 0 or 1 exactly, the choice made by the bias)."""
    cfg = I.MoEConfig("deg", 300, 512, 256, 1, 8, 128, 0.05, bias_uniform=0.01, seed=11)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    wr = I.make_router(cfg, DEV)
    if case == "all_equal":
        x = torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device=DEV)
        b = torch.zeros(cfg.E, dtype=torch.float32, device=DEV)
    else:
        x = (I.make_x(cfg, DEV).float() * 200.0).to(torch.bfloat16)
        b = I.make_bias(cfg, DEV)
    idx, gate, counts, offsets = B.moe_route(s, x, wr, b)
    torch.cuda.synchronize()
    if case == "all_equal":
        assert torch.equal(idx.cpu(), torch.arange(cfg.k, dtype=torch.int32).expand(cfg.T, cfg.k))
        assert torch.equal(gate.cpu(), torch.full((cfg.T, cfg.k), 1.0 / cfg.k))
    ties = check_routing(oracle_route(x, wr, b, cfg.k), idx, gate, counts, offsets, cfg.E)
    print(f"{case}: near-tied tokens {ties}")


def test_route_from_a_fresh_host_thread(libmoe):
    """The first library call of a host thread that has not used the CUDA runtime (buffers
    made by another thread) builds tensor maps before any runtime call."""
    import threading

    cfg = I.CONFIGS["tiny"]
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I)
    x, wr, b = I.make_x(cfg, DEV), I.make_router(cfg, DEV), I.make_bias(cfg, DEV)
    ws = B.alloc_workspace(s)
    out = {}
    bufs = [torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=DEV), torch.empty(cfg.T, cfg.k, device=DEV),
            torch.empty(cfg.E, dtype=torch.int32, device=DEV), torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)]
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()

    def run():  # ctypes only: no torch call in this thread
        import ctypes

        out["st"] = libmoe.moe_route(ctypes.byref(s), *(ctypes.c_void_p(t.data_ptr()) for t in (x, wr, b)), None,
                                     *(ctypes.c_void_p(t.data_ptr()) for t in bufs), ctypes.c_void_p(ws.data_ptr()),
                                     ws.numel(), ctypes.c_void_p(stream))
        out["sync"] = libmoe.moe_get_device_status(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(stream))

    t = threading.Thread(target=run)
    t.start()
    t.join(60)
    assert out == {"st": 0, "sync": 0}
    idx, gate, counts, offsets = B.moe_route(s, x, wr, b)
    assert torch.equal(bufs[0], idx) and torch.equal(bufs[1], gate) and torch.equal(bufs[2], counts)
    assert torch.equal(bufs[3], offsets)
