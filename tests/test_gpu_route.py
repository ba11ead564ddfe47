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
