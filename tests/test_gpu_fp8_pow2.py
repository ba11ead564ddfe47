"""GPU parity of the FP8 path with power-of-two block scales (MOE_FP8_E4M3_POW2: E4M3
codes, the smallest power of two above amax / 448 per 1x128 activation tile and per
128x128 weight block, applied by the block-scaled tensor-core MMA with FP32
accumulation) against the oracle's FP8 layer with the same scales.

Codes and scales computed on both sides from the same bf16 inputs match bit for bit.
Float outputs against the oracle's FP8 layer: the FP8 gates of moe_testutil.fp8_ok
(relative Frobenius error <= 5e-3, at most 1e-3 of the elements beyond the bf16 bound,
every element within 0.15 of the RMS -- with power-of-two scales one E4M3 step of h can
be 32/256 of its tile's amax); against the same layer with x and h left unquantised:
relative Frobenius error <= 6e-2."""
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


def _shape(cfg):
    return B.make_shape(cfg.T, cfg.d, cfg.E, cfg.S, cfg.k, cfg.I, fp8=True, pow2=True)


@pytest.mark.parametrize("T,d,E,k", [(256, 256, 16, 2), (1000, 2048, 64, 6), (37, 384, 8, 3)])
def test_permute_quantises_pow2_bit_exact(libmoe, T, d, E, k):
    cfg = I.MoEConfig("q", T, d, E, 1, k, 128, 0.05, seed=T)
    x = I.make_x(cfg, DEV)
    x[0, :128] = 0  # an all-zero tile
    x[1] *= 300.0
    x[2, 128:] *= 1e-30  # tiles far below 1, scales far below 2^-8
    ref = oracle_route(x, I.make_router(cfg, DEV), torch.zeros(E), k)
    p = O.permutation(ref["idx"], E)
    s = B.make_shape(T, d, E, 1, k, 128, fp8=True, pow2=True)
    xp, sc, _, _ = B.moe_permute(s, x, torch.tensor(ref["idx"], device=DEV), torch.tensor(p["offsets"], device=DEV))
    q_ref, sc_ref = Q.quantize_act_1x128(np64(x)[p["perm_token"]].astype(np.float32), pow2=True)
    np.testing.assert_array_equal(_u8(xp), q_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)


@pytest.mark.parametrize("G,N,K", [(2, 256, 256), (1, 4096, 7168)])
def test_weight_quantisation_pow2_bit_exact(libmoe, G, N, K):
    g = torch.Generator(device=DEV).manual_seed(G * N + K)
    w = (torch.randn(G, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    w[0, :128, :128] = 0
    wq, ws = B.moe_quantize_weights_fp8(w, pow2=True)
    wn = w.float().cpu().numpy()
    for gi in range(G):
        q_ref, s_ref = Q.quantize_weight_128x128(wn[gi], pow2=True)
        np.testing.assert_array_equal(_u8(wq[gi]), q_ref)
        np.testing.assert_array_equal(ws[gi].cpu().numpy(), s_ref)


def _getter(wgu, gs, wd, ds):
    cache = {}

    def get(e):
        if e not in cache:
            cache.clear()
            cache[e] = (_u8(wgu[e]), gs[e].cpu().numpy(), _u8(wd[e]), ds[e].cpu().numpy())
        return cache[e]

    return get


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_fp8_pow2_expert_ffn_every_expert(libmoe, name):
    cfg = I.CONFIGS[name]
    x = I.make_x(cfg, DEV)
    ref = oracle_route(x, I.make_router(cfg, DEV), I.make_bias(cfg, DEV), cfg.k)
    p = O.permutation(ref["idx"], cfg.E)
    s = _shape(cfg)
    wgu, gs, wd, ds = I.make_experts_fp8(cfg, DEV, pow2=True)
    xp, xps, _, _ = B.moe_permute(s, x, torch.tensor(ref["idx"], device=DEV), torch.tensor(p["offsets"], device=DEV))
    ws = B.alloc_workspace(s)
    y = B.moe_expert_ffn(s, xp, xps, x, torch.tensor(p["offsets"], device=DEV), wgu, wd, gs, ds, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    get = _getter(wgu, gs, wd, ds)
    xn, yg, Tk = np64(x), np64(y), cfg.T * cfg.k
    got, want = [], []
    for e in range(cfg.E):
        lo, hi = p["offsets"][e], p["offsets"][e + 1]
        if hi > lo:
            want.append(Q.fp8_swiglu_expert(xn[p["perm_token"][lo:hi]], *get(e), pow2=True))
            got.append(yg[lo:hi])
    nt = min(cfg.T, 512)
    for si in range(cfg.S):
        want.append(Q.fp8_swiglu_expert(xn[:nt], *get(cfg.E + si), pow2=True))
        got.append(yg[Tk + si * cfg.T: Tk + si * cfg.T + nt])
    got, want = np.concatenate(got), np.concatenate(want)
    e_ = fp8_errs(got, want)
    dev_ = np.abs(got - want) / np.sqrt(np.mean(want ** 2))
    worst = np.unravel_index(np.argmax(dev_), dev_.shape)
    print(f"{name} fp8-pow2 expert FFN, every expert: out_err {e_['out_err']:.3e} max/RMS {e_['max_rms']:.3e} "
          f"Frobenius {e_['fro']:.3e}; elements beyond 1e-2 of the RMS: {int((dev_ > 1e-2).sum())} of {dev_.size}, "
          f"worst at row {worst[0]} column {worst[1]}")
    assert fp8_ok(e_)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_fp8_pow2_forward(libmoe, name):
    cfg = I.CONFIGS[name]
    x = I.make_x(cfg, DEV)
    wr = I.make_router(cfg, DEV)
    b = I.make_bias(cfg, DEV)
    wgu, gs, wd, ds = I.make_experts_fp8(cfg, DEV, pow2=True)
    s = _shape(cfg)
    assert not B.forward_gathers(s)
    ws = B.alloc_workspace(s)
    out, idx, gate, counts = B.moe_forward(s, x, wr, b.clone(), wgu, wd, w_gu_scale=gs, w_down_scale=ds, ws=ws)
    torch.cuda.synchronize()
    assert B.moe_get_device_status(ws) == 0
    ref = oracle_route(x, wr, b, cfg.k)
    offsets = torch.tensor(O.offsets_from_counts(counts.cpu().numpy()))
    ties = check_routing(ref, idx, gate, counts, offsets, cfg.E)
    clean = np.nonzero(~(ref["boundary_tie"] | ref["order_tie"]))[0]
    tok = clean[:: max(1, cfg.T // 128)]
    get = _getter(wgu, gs, wd, ds)
    yr = Q.fp8_forward_rows(tok, np64(x), ref, get, cfg.E, cfg.S, pow2=True)

    def get_unq(e):
        gq, gsc, dq, dsc = get(e)
        return Q.dequant_weight(gq, gsc), Q.dequant_weight(dq, dsc)

    yu = O.forward_rows(tok, np64(x), ref, get_unq, cfg.E, cfg.S)
    o = np64(out)[tok]
    e, eu = fp8_errs(o, yr), errs(o, yu)
    print(f"{name} fp8-pow2 (near ties {ties}): vs the oracle's FP8 layer out_err {e['out_err']:.3e} "
          f"max/RMS {e['max_rms']:.3e} Frobenius {e['fro']:.3e}; vs the unquantised layer "
          f"max/RMS {eu['max_rms']:.3e} Frobenius {eu['fro']:.3e}")
    assert fp8_ok(e)
    assert eu["fro"] < TOL_FRO_UNQUANTISED
    out2, *_ = B.moe_forward(s, x, wr, b.clone(), wgu, wd, w_gu_scale=gs, w_down_scale=ds, ws=ws)
    assert torch.equal(out, out2), "deterministic"


def test_fp8_pow2_gather_is_refused(libmoe):
    cfg = I.CONFIGS["tiny"]
    s = _shape(cfg)
    x = I.make_x(cfg, DEV)
    wgu, gs, wd, ds = I.make_experts_fp8(cfg, DEV, pow2=True)
    ptok = torch.zeros(cfg.T * cfg.k, dtype=torch.int32, device=DEV)
    off = torch.zeros(cfg.E + 1, dtype=torch.int32, device=DEV)
    with pytest.raises(B.MoEError) as ei:
        B.moe_expert_ffn_gather(s, x, ptok, off, wgu, wd, gs, ds)
    assert ei.value.code == 2  # MOE_ERR_UNSUPPORTED
