"""GPU parity of the FP8 path (E4M3, 1x128 activation tiles, 128x128 weight
blocks, FP32 accumulation) against the oracle's FP8 layer.

Codes and scales that both sides compute from the same bf16 inputs (x, weights)
must match bit for bit.  Float outputs are compared with the oracle's FP8 layer
under the same simulated quantisation with the FP8 gates of moe_testutil.fp8_ok
(relative Frobenius error <= 5e-3, at most 1e-3 of the elements beyond the bf16
bound, every element within 0.15 of the RMS: an E4M3 code of h that flips at a
rounding midpoint moves some of one row's outputs, a wrong scale, index or tile
moves thousands), and with the same layer left unquantised (x and h exact) at a
relative Frobenius error <= 6e-2: E4M3's three mantissa bits alone cost about 4.4 %
there, and the max error against the unquantised layer (20-30 % of the RMS) is
reported only."""
import numpy as np
import pytest
import torch

from oracle import fp8 as Q
from oracle import moe_oracle as O
from sparse_moe_layer_12_b300 import binding as B
from sparse_moe_layer_12_b300 import inputs as I
from moe_testutil import check_routing, errs, fp8_errs, fp8_ok, np64, oracle_route

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_FRO_UNQUANTISED = 6e-2


def _u8(t):
    return t.view(torch.uint8).cpu().numpy()


@pytest.mark.parametrize("T,d,E,k", [(256, 256, 16, 2), (1000, 2048, 64, 6), (37, 384, 8, 3)])
def test_permute_quantises_1x128_bit_exact(libmoe, T, d, E, k):
    cfg = I.MoEConfig("q", T, d, E, 1, k, 128, 0.05, seed=T)
    x = I.make_x(cfg, DEV)
    x[0, :128] = 0  # an all-zero tile
    x[1] *= 300.0  # large values
    ref = oracle_route(x, I.make_router(cfg, DEV), torch.zeros(E), k)
    p = O.permutation(ref["idx"], E)
    s = B.make_shape(T, d, E, 1, k, 128, fp8=True)
    xp, sc, ptok, inv = B.moe_permute(s, x, torch.tensor(ref["idx"], device=DEV),
                                      torch.tensor(p["offsets"], device=DEV))
    q_ref, sc_ref = Q.quantize_act_1x128(np64(x)[p["perm_token"]].astype(np.float32))
    np.testing.assert_array_equal(_u8(xp), q_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)


@pytest.mark.parametrize("G,N,K", [(2, 256, 256), (1, 4096, 7168), (3, 384, 1408 // 128 * 128)])
def test_weight_quantisation_bit_exact(libmoe, G, N, K):
    g = torch.Generator(device=DEV).manual_seed(G * N + K)
    w = (torch.randn(G, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w[0, :128, :128] = 0  # an all-zero block
    wq, ws = B.moe_quantize_weights_fp8(w)
    wn = w.float().cpu().numpy()
    for gi in range(G):
        q_ref, s_ref = Q.quantize_weight_128x128(wn[gi])
        np.testing.assert_array_equal(_u8(wq[gi]), q_ref)
        np.testing.assert_array_equal(ws[gi].cpu().numpy(), s_ref)


def _fp8_getter(wgu, gs, wd, ds):
    cache = {}

    def get(e):
        if e not in cache:
            cache.clear()
            cache[e] = (_u8(wgu[e]), gs[e].cpu().numpy(), _u8(wd[e]), ds[e].cpu().numpy())
        return cache[e]

    return get


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_fp8_forward(libmoe, name):
    cfg = I.CONFIGS[name]
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV)
    wgu, gs, wd, ds = I.make_experts_fp8(cfg, DEV)
    s = B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8=True)
    ws = B.alloc_workspace(s)
    out, idx, gate, counts = B.moe_forward(s, x, wr, b.clone(), wgu, wd, w_gu_scale=gs, w_down_scale=ds, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    ref = oracle_route(x, wr, b, cfg.k)
    offsets = torch.tensor(O.offsets_from_counts(counts.cpu().numpy()))
    ties = check_routing(ref, idx, gate, counts, offsets, cfg.E)
    clean = np.nonzero(~(ref["boundary_tie"] | ref["order_tie"]))[0]
    tok = clean[:: max(1, cfg.T // 128)]
    get = _fp8_getter(wgu, gs, wd, ds)
    yr = Q.fp8_forward_rows(tok, np64(x), ref, get, cfg.E, cfg.S)

    def get_unq(e):
        gq, gsc, dq, dsc = get(e)
        return Q.dequant_weight(gq, gsc), Q.dequant_weight(dq, dsc)

    yu = O.forward_rows(tok, np64(x), ref, get_unq, cfg.E, cfg.S)
    o = np64(out)[tok]
    e, eu = fp8_errs(o, yr), errs(o, yu)
    print(f"{name} fp8 (near ties {ties}): vs the oracle's FP8 layer out_err {e['out_err']:.3e} "
          f"max/RMS {e['max_rms']:.3e} Frobenius {e['fro']:.3e} beyond {e['frac_over']:.2e}; vs the unquantised layer "
          f"max/RMS {eu['max_rms']:.3e} Frobenius {eu['fro']:.3e}")
    assert fp8_ok(e)
    assert eu["fro"] < TOL_FRO_UNQUANTISED
    out2, *_ = B.moe_forward(s, x, wr, b.clone(), wgu, wd, w_gu_scale=gs, w_down_scale=ds, ws=ws)
    assert torch.equal(out, out2), "deterministic"
