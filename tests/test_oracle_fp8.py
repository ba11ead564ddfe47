"""Pins for the oracle's E4M3 codec and 1x128 / 128x128 quantisation (CPU only)."""
import numpy as np
import torch

from oracle import fp8 as Q


def test_decode_every_code_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    got = Q.e4m3_decode(codes)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert nan.sum() == 2  # only S.1111.111


def test_decode_spec_landmarks():
    assert Q.e4m3_decode(np.array([0x7E]))[0] == 448.0  # largest finite
    assert Q.e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6  # smallest normal
    assert Q.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9  # smallest subnormal
    assert Q.e4m3_decode(np.array([0x38]))[0] == 1.0  # exponent field 7 = bias
    assert Q.e4m3_decode(np.array([0xB8]))[0] == -1.0


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    parts = [
        rng.standard_normal(400_000) * 50.0,
        rng.standard_normal(200_000) * 2.0 ** -7,  # subnormal range
        rng.uniform(-464.0, 464.0, 200_000),
        rng.standard_normal(200_000),
    ]
    v = np.clip(np.concatenate(parts), -464.0, 464.0).astype(np.float32)
    # every exact midpoint between neighbouring codes (ties to even)
    vals = np.sort(Q.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = Q.e4m3_encode(v)
    np.testing.assert_array_equal(got, ref)


def test_encode_saturates_and_keeps_nan():
    v = np.array([448.0, 465.0, 1e4, -1e30, np.inf, -np.inf, np.nan], dtype=np.float32)
    got = Q.e4m3_encode(v)
    np.testing.assert_array_equal(got[:6], [0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE])
    assert got[6] == 0x7F


def test_act_tiles_are_1x128_per_token():
    rng = np.random.default_rng(1)
    R, C = 6, 384
    x = rng.standard_normal((R, C)).astype(np.float32)
    x[2] *= 1000.0  # one loud token
    x[4, 128:256] *= 1e-3  # one quiet tile
    x[5, 256:] = 0.0  # one empty tile
    q, sc = Q.quantize_act_1x128(x)
    assert q.shape == (R, C) and sc.shape == (R, 3) and sc.dtype == np.float32
    for r in range(R):
        for b in range(3):
            tile = x[r, b * 128:(b + 1) * 128]
            amax = np.float32(np.abs(tile).max())
            if amax == 0:
                assert sc[r, b] == 1.0 and np.all(q[r, b * 128:(b + 1) * 128] == 0)
                continue
            assert sc[r, b] == amax / np.float32(448.0)
            # the largest element lands on the largest code
            assert np.abs(Q.e4m3_decode(q[r, b * 128:(b + 1) * 128])).max() == 448.0
    deq = Q.dequant_act(q, sc)
    # error bound: half an E4M3 ulp, relative 2^-4 for normals, 2^-10 * scale for subnormals
    bound = np.maximum(np.abs(x) * 2.0 ** -4, np.repeat(sc, 128, axis=1) * 2.0 ** -10)
    assert np.all(np.abs(deq - x) <= bound * (1 + 1e-6))


def test_weight_blocks_are_128x128():
    rng = np.random.default_rng(2)
    N, K = 256, 384
    w = rng.standard_normal((N, K)).astype(np.float32)
    w[128:, 256:] *= 100.0
    q, sc = Q.quantize_weight_128x128(w)
    assert sc.shape == (2, 3)
    for i in range(2):
        for j in range(3):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert sc[i, j] == np.float32(np.abs(blk).max()) / np.float32(448.0)
    assert sc[1, 2] > 50 * sc[0, 0]
    deq = Q.dequant_weight(q, sc)
    assert np.max(np.abs(deq - w) / np.abs(w).max()) < 2.0 ** -4


def test_fp8_expert_close_to_unquantised():
    from oracle import moe_oracle as O
    rng = np.random.default_rng(3)
    T, d, I = 20, 256, 128
    x = rng.standard_normal((T, d)).astype(np.float32)
    wgu = (rng.standard_normal((2 * I, d)) / np.sqrt(d)).astype(np.float32)
    wd = (rng.standard_normal((d, I)) / np.sqrt(I)).astype(np.float32)
    gq, gs = Q.quantize_weight_128x128(wgu)
    dq, ds = Q.quantize_weight_128x128(wd)
    y8 = Q.fp8_swiglu_expert(x, gq, gs, dq, ds)
    y = O.swiglu_expert(x, wgu, wd)
    # E4M3 keeps 3 mantissa bits: the RMS error of a quantised product is a few
    # percent of the output RMS, whatever the length of the dot product
    rms_err = np.sqrt(np.mean((y8 - y) ** 2) / np.mean(y ** 2))
    assert 5e-3 < rms_err < 8e-2
    assert O.max_rel_err(y8, y) < 0.5


# ---- h quantisation inside the FP8 expert, pinned by hand-derived codes.
# x and every weight are exact in E4M3 with power-of-two scales, so the only
# rounding in the expert is the 1x128 quantisation of h along I ("DeepSeek-V3 详解"
# 4.2: activations scaled per 1x128 tile along the contraction dimension).  Every
# gate row is the same, so inside a token all a_i are equal and h_i / amax(tile)
# = u_i / max|u| over the tile: 448 * u_i / max|u| lands on a code picked by hand
# (each far from a midpoint between two codes), whatever the exact value of silu(a).

# tile 0 of I: up values (x 0.25 * x0) and the code 448 * v / 1.25 rounds to
_H_TILE0 = {1.25: 448.0, 1.0: 352.0, 0.875: 320.0, 0.5: 176.0, -0.75: -256.0, 0.0: 0.0, 0.0625: 22.0}
# tile 1 of I: amax 3.0 (not a power-of-two multiple of tile 0's, so a per-row
# scale would round tile 0 differently)
_H_TILE1 = {3.0: 448.0, 2.5: 384.0, -1.75: -256.0, 1.0: 144.0}


def _e4m3_codes(v):
    return torch.tensor(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _h_quant_case():
    d, I = 128, 256
    up = np.zeros(I)
    t0, t1 = list(_H_TILE0), list(_H_TILE1)
    for i in range(128):
        up[i] = t0[i % len(t0)]
        up[128 + i] = t1[i % len(t1)]
    # gate/up weight [2I, d]: only column 0 is non-zero; gate rows 1.0, up rows `up`;
    # every 128x128 block has scale 0.25
    w = np.zeros((2 * I, d))
    w[:I, 0] = 1.0
    w[I:, 0] = up
    wgu_q, wgu_sc = _e4m3_codes(w), np.full((2 * I // 128, 1), 0.25, np.float32)
    # down weight [d, I]: y_j = h_j + h_{128+j} (codes of 1.0, block scales 1.0)
    wd = np.zeros((d, I))
    wd[np.arange(128), np.arange(128)] = 1.0
    wd[np.arange(128), 128 + np.arange(128)] = 1.0
    wd_q, wd_sc = _e4m3_codes(wd), np.ones((1, 2), np.float32)
    # two tokens, x = x0 * e_0 with x0 = 1.75 and 3.5: amax / 448 = 2^-8 and 2^-7, exact
    x0 = np.array([1.75, 3.5])
    x = np.zeros((2, d), np.float32)
    x[:, 0] = x0
    return x, x0, up, wgu_q, wgu_sc, wd_q, wd_sc


def test_fp8_expert_quantises_h_per_1x128_along_I():
    x, x0, up, wgu_q, wgu_sc, wd_q, wd_sc = _h_quant_case()
    y = Q.fp8_swiglu_expert(x, wgu_q, wgu_sc, wd_q, wd_sc)
    for t in range(2):
        a = 0.25 * x0[t]  # gate: code 1.0 x block scale 0.25 x x0
        silu_a = float(torch.nn.functional.silu(torch.tensor(a, dtype=torch.float64)))
        hq = np.zeros(256)
        for tile, table, vmax in ((0, _H_TILE0, 1.25), (1, _H_TILE1, 3.0)):
            # h_i = silu(a) * 0.25 * x0 * up_i; the tile's scale is its amax / 448
            scale = silu_a * 0.25 * x0[t] * vmax / 448.0
            for i in range(tile * 128, tile * 128 + 128):
                hq[i] = table[up[i]] * scale
        want = hq[:128] + hq[128:]
        # float32 rounding of h and of the scale is the only slack left
        np.testing.assert_allclose(y[t], want, rtol=1e-6, atol=0)


def test_fp8_expert_h_rounding_is_visible():
    # the same case without any quantisation of h differs by far more than the pin's
    # tolerance, so the pin above cannot pass with h left unquantised
    x, x0, up, wgu_q, wgu_sc, wd_q, wd_sc = _h_quant_case()
    y = Q.fp8_swiglu_expert(x, wgu_q, wgu_sc, wd_q, wd_sc)
    wgu = Q.dequant_weight(wgu_q, wgu_sc)
    wd = Q.dequant_weight(wd_q, wd_sc)
    a = x.astype(np.float64) @ wgu[:256].T
    u = x.astype(np.float64) @ wgu[256:].T
    h = torch.nn.functional.silu(torch.from_numpy(a)).numpy() * u
    y_exact_h = h @ wd.T
    rel = np.abs(y - y_exact_h) / np.maximum(np.abs(y_exact_h), 1e-30)
    assert rel.max() > 1e-2


# ---- power-of-two scales (the smallest 2^e with amax <= 448 * 2^e)


def test_pow2_scale_closed_forms():
    eps = np.float32(2.0 ** -23)
    cases = [
        (448.0, 1.0),                      # amax = 448 exactly: scale 1, code 448
        (448.0 * (1 + eps), 2.0),          # one ulp above: the next power
        (224.0, 0.5),                      # 224 / 0.5 = 448
        (224.0 * (1 + eps), 1.0),
        (1.75, 2.0 ** -8),                 # 1.75 / 448 = 2^-8 exactly
        (1.75 * (1 + eps), 2.0 ** -7),
        (1.0, 2.0 ** -8),                  # 1 / 448 lies between 2^-9 and 2^-8
        (0.0, 1.0),                        # empty tile
        (448.0 * 2.0 ** 100, 2.0 ** 100),
        (1e-38, 2.0 ** -127),              # below 448 * 2^-127: the smallest one-byte scale
    ]
    amax = np.array([a for a, _ in cases], dtype=np.float32)
    got = Q.pow2_scale(amax)
    np.testing.assert_array_equal(got, np.array([s for _, s in cases], dtype=np.float32))


def test_pow2_scale_puts_the_tile_max_in_224_448():
    rng = np.random.default_rng(5)
    amax = (np.exp(rng.uniform(-60, 60, 100_000)) * rng.uniform(0.5, 1.0, 100_000)).astype(np.float32)
    sc = Q.pow2_scale(amax)
    m, _ = np.frexp(sc.astype(np.float64))
    assert np.all(m == 0.5)  # powers of two
    r = amax.astype(np.float64) / sc.astype(np.float64)
    assert np.all(r <= 448.0) and np.all(r > 224.0)


def test_pow2_tiles_codes_match_torch():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((9, 384)) * np.exp(rng.uniform(-8, 8, (9, 1)))).astype(np.float32)
    x[3, 128:256] = 0.0
    q, sc = Q.quantize_act_1x128(x, pow2=True)
    for r in range(9):
        for b in range(3):
            tile = x[r, b * 128:(b + 1) * 128]
            s = np.float32(sc[r, b])
            want = torch.from_numpy(tile / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(q[r, b * 128:(b + 1) * 128], want)
            if np.abs(tile).max() > 0:
                assert 224.0 <= np.abs(Q.e4m3_decode(q[r, b * 128:(b + 1) * 128])).max() <= 448.0
    wq, wsc = Q.quantize_weight_128x128(x[:, :256].repeat(128 // 9 + 1, axis=0)[:128], pow2=True)
    m, _ = np.frexp(wsc.astype(np.float64))
    assert np.all(m == 0.5)


def test_fp8_expert_pow2_quantises_h_per_1x128_along_I():
    # the hand case above with power-of-two activation scales: h's tile scale is the
    # power of two above amax / 448 and its codes are torch's E4M3 cast of h / scale
    x, x0, up, wgu_q, wgu_sc, wd_q, wd_sc = _h_quant_case()
    y = Q.fp8_swiglu_expert(x, wgu_q, wgu_sc, wd_q, wd_sc, pow2=True)
    for t in range(2):
        a = 0.25 * x0[t]
        silu_a = float(torch.nn.functional.silu(torch.tensor(a, dtype=torch.float64)))
        h = (silu_a * 0.25 * x0[t] * up).astype(np.float32)
        hq = np.zeros(256)
        for tile in range(2):
            seg = h[tile * 128:(tile + 1) * 128]
            amax = float(np.abs(seg).max())
            m, ex = np.frexp(amax)  # the power of two above amax / 448, restated
            s = 2.0 ** (ex - 9 if m <= 0.875 else ex - 8)
            codes = torch.from_numpy((seg / np.float32(s)).astype(np.float32)).to(torch.float8_e4m3fn)
            hq[tile * 128:(tile + 1) * 128] = codes.double().numpy() * s
        np.testing.assert_allclose(y[t], hq[:128] + hq[128:], rtol=1e-12, atol=0)
