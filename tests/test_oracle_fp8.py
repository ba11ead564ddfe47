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
