"""CPU oracle for the FP8 (E4M3) fine-grained quantisation of the expert GEMMs.

TEST INFRASTRUCTURE ONLY (same rule as moe_oracle: only tests, smoke() and the
bench's CPU-baseline legs import it; the product never does).

Pages followed:
  [YDL] "DeepSeek-V3 详解" (yudonglee.me), section 4.2 "V3 的 FP8 方案":
        activations scaled per 1x128 tile (one scale per token per 128
        channels), weights per 128x128 block; section 4.3: all GEMM
        accumulation in FP32.
  [DYN] "deepseek-v3-report" (dynmi.github.io), FP8 paragraph: 1x128 row tiles,
        128x128 blocks, FP32 accumulation.
  [KC]  "拆解DeepSeek V3" (kongchang.com), section "MLA 与 FP8": E4M3 range ~448.

E4M3 ("e4m3fn") is taken from the OCP 8-bit floating point specification:
1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, the
single NaN pattern S.1111.111, largest finite 448, smallest normal 2^-6,
smallest subnormal 2^-9.

Readings (pages silent): scale = amax / 448 in float32; an all-zero tile gets
scale 1; codes are round-to-nearest-even with saturation to +-448; v / scale is
one float32 division; the dequantised value is decode(code) * scale.  The pages
fix the granularity of the scales, not their format; the power-of-two variant
(pow2=True) takes the smallest power of two 2^e with amax <= 448 * 2^e (so the
tile maximum lands on a code in (224, 448]), e kept within [-127, 127], the
range of the one-byte exponent scales that a block-scaled tensor-core MMA applies.

parity: pinned by tests/test_oracle_fp8.py (every one of the 256 codes against
torch.float8_e4m3fn, random casts against torch, saturation and subnormal
closed forms, per-tile scale invariants; the quantisation of h inside the FP8
expert by a hand-derived case in which it is the only rounding, so that leaving
h unquantised, or tiling it along tokens or per whole row, fails; the power-of-two
scale by closed forms at and around the 448 * 2^e boundaries, and its codes
against torch's E4M3 cast).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8), float64; NaN for 0x7F / 0xFF."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


def e4m3_encode(v) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest, ties to even, saturating at 448."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    out = np.zeros(v.shape, dtype=np.uint8)
    nan = np.isnan(v)
    sign = np.signbit(v)
    a = np.abs(np.where(nan, 0.0, v))
    sat = a >= E4M3_MAX
    a = np.where(sat, 1.0, a)  # saturated lanes are overwritten below
    # subnormal range: units of 2^-9, rounding into code 8 (= 2^-6) is exact
    sub = a < 2.0 ** -6
    q_sub = np.rint(a / 2.0 ** -9)  # np.rint: round half to even
    # normal range: exponent e with 2^e <= a < 2^(e+1); 3 mantissa bits
    mant, ex = np.frexp(np.where(sub, 1.0, a))  # a = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1
    q = np.rint(a / np.exp2(e - 3.0))  # in [8, 16]
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)
    code_n = ((e + 7) << 3) | (q.astype(np.int64) - 8)
    code = np.where(sub, q_sub.astype(np.int64), code_n)
    code = np.where(sat, 0x7E, code)
    code = np.where(sign, code | 0x80, code)
    code = np.where(nan, 0x7F, code)
    out[...] = code.astype(np.uint8)
    return out


def pow2_scale(amax32) -> np.ndarray:
    """Smallest power of two 2^e with amax <= 448 * 2^e (1 for amax = 0), float32.

    With amax = m * 2^ex, m in [0.5, 1) (frexp): 448 * 2^e = 0.875 * 2^(9 + e), so
    e = ex - 9 when m <= 0.875 and ex - 8 otherwise; e is kept within [-127, 127]."""
    a = np.asarray(amax32, dtype=np.float32).astype(np.float64)
    m, ex = np.frexp(a)
    e = np.where(m <= 0.875, ex - 9, ex - 8)
    e = np.clip(e, -127, 127)
    sc = np.ldexp(np.float64(1.0), e).astype(np.float32)  # every 2^e in range is exact in float32
    return np.where(a == 0, np.float32(1.0), sc).astype(np.float32)


def _tile_scale(amax32: np.ndarray, pow2: bool = False) -> np.ndarray:
    if pow2:
        return pow2_scale(amax32)
    amax32 = amax32.astype(np.float32)
    sc = amax32 / np.float32(E4M3_MAX)
    return np.where(amax32 == 0, np.float32(1.0), sc).astype(np.float32)


def quantize_act_1x128(x, pow2: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Per-token 1x128 tiles: x [R, C] (C % 128 == 0) -> (codes uint8 [R, C], scale f32 [R, C/128])."""
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    t = x.reshape(R, C // 128, 128)
    amax = np.abs(t).max(axis=2)
    sc = _tile_scale(amax, pow2)
    q = e4m3_encode(t / sc[:, :, None])
    return q.reshape(R, C), sc


def quantize_weight_128x128(w, pow2: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """128x128 blocks: w [N, K] (both % 128 == 0) -> (codes [N, K], scale f32 [N/128, K/128])."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    b = w.reshape(N // 128, 128, K // 128, 128)
    amax = np.abs(b).max(axis=(1, 3))
    sc = _tile_scale(amax, pow2)
    q = e4m3_encode(b / sc[:, None, :, None])
    return q.reshape(N, K), sc


_LUT = None


def _decode_fast(q) -> np.ndarray:
    """e4m3_decode through a 256-entry table of its own values (for large arrays)."""
    global _LUT
    if _LUT is None:
        _LUT = e4m3_decode(np.arange(256, dtype=np.uint8))
    return _LUT[np.asarray(q, dtype=np.uint8)]


def dequant_act(q, sc) -> np.ndarray:
    R, C = q.shape
    return (_decode_fast(q).reshape(R, C // 128, 128) * np.asarray(sc, np.float64)[:, :, None]).reshape(R, C)


def dequant_weight(q, sc) -> np.ndarray:
    N, K = q.shape
    v = _decode_fast(q).reshape(N // 128, 128, K // 128, 128)
    return (v * np.asarray(sc, np.float64)[:, None, :, None]).reshape(N, K)


def fp8_swiglu_expert(x_rows, wgu_q, wgu_sc, wd_q, wd_sc, pow2: bool = False) -> np.ndarray:
    """One expert on the FP8 path with simulated quantisation.

    gate/up: x rows quantised per 1x128, weights per 128x128, products summed in
    float64 (the exact value the FP32-accumulating GEMM approximates); h is
    rounded to float32, quantised per 1x128 along I, and the down GEMM is taken
    the same way.  pow2: the activation scales (x and h) are powers of two (the
    weights' codes and scales are inputs).
    """
    I = wd_q.shape[1]
    xq, xs = quantize_act_1x128(x_rows, pow2)
    xa = dequant_act(xq, xs)
    wgu = dequant_weight(wgu_q, wgu_sc)
    a = xa @ wgu[:I].T
    u = xa @ wgu[I:].T
    h = (a / (1.0 + np.exp(-a))) * u
    hq, hs = quantize_act_1x128(h.astype(np.float32), pow2)
    return dequant_act(hq, hs) @ dequant_weight(wd_q, wd_sc).T


def fp8_forward_rows(tokens, x, route_result, get_expert_q, E, S, pow2: bool = False) -> np.ndarray:
    """Layer output on the FP8 path for a subset of tokens (simulated quantisation).

    get_expert_q(e) -> (wgu_q, wgu_sc, wd_q, wd_sc).
    """
    tokens = np.asarray(tokens)
    xs = np.asarray(x, dtype=np.float32)[tokens]
    idx = route_result["idx"][tokens]
    gate = route_result["gate"][tokens]
    out = np.zeros(xs.shape, dtype=np.float64)
    for s_id in range(S):
        out += fp8_swiglu_expert(xs, *get_expert_q(E + s_id), pow2=pow2)
    for e in np.unique(idx):
        rows, slot = np.nonzero(idx == e)
        out[rows] += gate[rows, slot][:, None] * fp8_swiglu_expert(xs[rows], *get_expert_q(int(e)), pow2=pow2)
    return out
