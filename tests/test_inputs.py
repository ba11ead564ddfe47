"""The seeded generators give the shapes and distributions of the layer's workloads."""
import math

import numpy as np
import torch

from sparse_moe_layer_12_b300 import inputs as I


def test_configs_match_the_workloads():
    c = I.CONFIGS
    assert (c["tiny"].T, c["tiny"].d, c["tiny"].E, c["tiny"].S, c["tiny"].k, c["tiny"].I) == (256, 256, 16, 1, 2, 128)
    assert (c["mid"].T, c["mid"].d, c["mid"].E, c["mid"].S, c["mid"].k, c["mid"].I) == (4096, 2048, 64, 2, 6, 1408)
    assert (c["v3"].T, c["v3"].d, c["v3"].E, c["v3"].S, c["v3"].k, c["v3"].I) == (8192, 7168, 256, 1, 8, 2048)
    assert c["v3fp8"].T == 16384 and c["v3fp8"].fp8
    assert c["skew"].T == 256 and c["skew"].zipf_amp == 2.0
    # 2 * T * (k + S) * 3 * d * I at the V3 shape: 6.49 TFLOP
    assert abs(c["v3"].expert_flops() / 1e12 - 6.4938) < 1e-3


def test_generators_are_seeded_and_shaped():
    cfg = I.CONFIGS["tiny"]
    a = I.make_all(cfg)
    b = I.make_all(cfg)
    for key in ("x", "w_router", "bias", "w_gate_up", "w_down"):
        assert torch.equal(a[key], b[key]), key
    assert a["x"].shape == (256, 256) and a["x"].dtype == torch.bfloat16
    assert a["w_router"].shape == (16, 256)
    assert a["w_gate_up"].shape == (17, 256, 256) and a["w_down"].shape == (17, 256, 128)
    assert a["logit_offset"] is None and float(a["bias"].abs().max()) == 0.0
    # distributions
    assert abs(float(a["x"].float().std()) - 1.0) < 0.02
    assert abs(float(a["w_router"].float().std()) - 0.02) < 0.002
    assert abs(float(a["w_gate_up"].float().std()) - 1 / math.sqrt(256)) < 0.002
    assert abs(float(a["w_down"].float().std()) - 1 / math.sqrt(128)) < 0.002
    # one expert regenerates on its own
    wgu5, wd5 = I.make_expert(cfg, 5)
    assert torch.equal(wgu5, a["w_gate_up"][5]) and torch.equal(wd5, a["w_down"][5])


def test_mid_bias_and_skew_offsets():
    b = I.make_bias(I.CONFIGS["mid"])
    assert b.shape == (64,) and float(b.abs().max()) <= 0.05 and float(b.std()) > 0.02
    o = I.make_logit_offset(I.CONFIGS["skew"]).double().numpy()
    # a permutation of A * r^-1.1, r = 1..E
    ref = np.sort(2.0 * np.arange(1, 257, dtype=np.float64) ** -1.1)
    np.testing.assert_allclose(np.sort(o), ref, rtol=1e-6)
    assert abs(o.max() - 2.0) < 1e-6
