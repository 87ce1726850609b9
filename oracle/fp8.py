"""FP8 input preparation: incoherent processing and per-tile e4m3 quantisation.

Test infrastructure.  Source: "FlashAttention-Skalierung, Multi-GPU-Training und
Gewichtsquantisierung", section 1, bullet "Unterstützung geringer
FP8-Präzision": FP8 tensor cores double raw throughput; to keep outlier
activations from destroying FP8 precision the method scales small tiles
independently (block quantisation) and multiplies Q and K by random orthogonal
matrices before quantising (incoherent processing).  The pages fix neither the
matrix, the tile, the FP8 format nor the rounding; the readings taken here are:

* Rotation: M = diag(s) H_d, with s a seeded vector of +-1 signs and H_d the
  d x d Sylvester Walsh-Hadamard matrix (entries +-1, H H^T = d I).  M / sqrt(d)
  is orthogonal; the 1/sqrt(d) factor cancels in the quantised codes (they depend
  only on x / amax), so it is carried in the scores' scale instead:
  (Q M)(K M)^T = d * Q K^T.
* The same M multiplies Q and K (the pages name Q and K only); V is not rotated.
* Tile: 64 consecutive rows of one head times all d columns.
* Format: OCP FP8 E4M3 ("fn": bias 7, no infinities, one NaN pattern per sign,
  largest finite 448).  Rounding: round-to-nearest, ties to even, saturating
  to +-448.
* Per tile: amax = max |x|; the dequantisation scale is the power of two
  sigma = 2^e with e the smallest integer such that amax <= 448 * 2^e (e kept in
  [-126, 126] so that sigma and 1/sigma are normal fp32 numbers); codes =
  e4m3(x * 2^-e).  An all-zero tile has sigma = 1.  Because e4m3 is a
  floating-point format, a power-of-two scale costs no relative precision
  (amax / sigma lies in (224, 448]); it makes the scaling exact, and the
  dequantised values decode(code) * sigma exact in fp32 and bf16.

Because these codes are integers decided by floating point, the decision is made
in the kernel's precision (IEEE fp32) with the kernel's order of operations:
the rotation is the radix-2 fast Walsh-Hadamard transform with butterfly spans
1, 2, 4, ..., d/2 (each butterfly is one fp32 add and one fp32 subtract),
amax is exact, e is read from amax's fp32 bits, and ``x * 2^-e`` is one fp32
multiply (exact unless it leaves the normal range).  The transform is pinned against the float64 matrix product
``x @ diag(s) @ H`` within fp32 rounding bounds.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # smallest normal binade: 2^-6
E4M3_MANT_BITS = 3
E4M3_BIAS = 7


def sylvester_hadamard(d: int) -> np.ndarray:
    """d x d Sylvester Walsh-Hadamard matrix (float64, entries +-1); d a power of 2."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def fwht_f32(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Unnormalised rotation x -> (x * s) H_d along the last axis, in fp32.

    Radix-2 butterflies with spans 1, 2, ..., d/2, each an fp32 add/subtract, so
    the rounding is that of the kernel's transform.  ``signs`` is the +-1 vector s.
    """
    y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("last dimension must be a power of two")
    span = 1
    while span < d:
        shaped = y.reshape(y.shape[:-1] + (d // (2 * span), 2, span))
        a = shaped[..., 0, :]
        b = shaped[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(y.shape)
        span *= 2
    return y


def e4m3_round(x) -> np.ndarray:
    """Round values to the nearest OCP E4M3 value (ties to even), saturating at +-448.

    Works on the exact value of each input (float32 inputs are exact in float64).
    NaN stays NaN.  Returns float64.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    # log2 of a float64 can be off by one at exact powers of two; fix the binade.
    e = np.where(2.0 ** e > ax, e - 1, e)
    e = np.where(2.0 ** (e + 1) <= ax, e + 1, e)
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)          # subnormals share the 2^-6 binade's spacing
    ulp = 2.0 ** (e - E4M3_MANT_BITS)
    r = np.rint(ax / ulp) * ulp                      # np.rint rounds half to even
    r = np.minimum(r, E4M3_MAX)                      # satfinite
    return np.where(np.isnan(x), np.nan, np.copysign(r, x))


def e4m3_encode(x) -> np.ndarray:
    """Byte codes (uint8) of ``e4m3_round(x)``: sign << 7 | exponent << 3 | mantissa."""
    r = e4m3_round(x)
    sign = np.signbit(r).astype(np.uint8) << 7
    ar = np.abs(r)
    code = np.zeros(r.shape, dtype=np.uint8)
    nz = ar > 0
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(nz, ar, 1.0)))
    normal = nz & (e >= E4M3_MIN_NORMAL_EXP)
    sub = nz & ~normal
    # normal: value = 2^(E-7) * (1 + m/8)
    ef = (e + E4M3_BIAS).astype(np.int64)
    mant_n = np.rint((ar / 2.0 ** e - 1.0) * 8).astype(np.int64)
    # subnormal: value = 2^-6 * m/8 = m * 2^-9
    mant_s = np.rint(ar / 2.0 ** -9).astype(np.int64)
    code = np.where(normal, (ef << 3) | mant_n, code)
    code = np.where(sub, mant_s, code)
    code = np.where(np.isnan(r), 0x7F, code)
    return (code.astype(np.uint8) | sign)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of E4M3 byte codes (0x7F / 0xFF decode to NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(ef == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (ef - E4M3_BIAS))
    val = np.where((ef == 0xF) & (m == 0x7), np.nan, val)
    return s * val


def pow2_scale_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-126, 126]; 0 where amax == 0.

    amax (fp32, >= 0) = m * 2^e0 with m in [1, 2): 448 * 2^(e0-8) = 1.75 * 2^e0, so
    e = e0 - 8 when m <= 1.75 and e0 - 7 otherwise.  e0 and m come from the fp32
    bits (a subnormal amax gives e <= -134, clamped to -126).
    """
    a = np.asarray(amax, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.int64)
    field = (bits >> 23) & 0xFF
    mant = bits & 0x7FFFFF
    e = field - 127 - 8 + (mant > 0x600000)
    e = np.where(field == 0, -126, e)
    e = np.clip(e, -126, 126)
    return np.where(a == 0, 0, e).astype(np.int64)


def _quantise_tiles(x32: np.ndarray, tile: int):
    """Per-tile e4m3 codes and dequantisation scales of an fp32 array [..., N, d].

    Tiles are ``tile`` consecutive rows of the second-to-last axis (the last tile
    may be short).  Returns (codes uint8 [..., N, d], sigma float32 [..., ceil(N/tile)]).
    """
    *lead, N, d = x32.shape
    nt = -(-N // tile)
    codes = np.empty(x32.shape, dtype=np.uint8)
    sigma = np.empty(tuple(lead) + (nt,), dtype=np.float32)
    for t in range(nt):
        blk = x32[..., t * tile:(t + 1) * tile, :]
        amax = np.abs(blk).max(axis=(-2, -1)).astype(np.float32)
        e = pow2_scale_exponent(amax)
        sig = np.ldexp(np.float32(1), e).astype(np.float32)
        inv = np.ldexp(np.float32(1), -e).astype(np.float32)
        y = (blk * inv[..., None, None]).astype(np.float32)
        codes[..., t * tile:(t + 1) * tile, :] = e4m3_encode(y)
        sigma[..., t] = sig
    return codes, sigma


def fp8_prepare(q, k, v, signs, tile: int = 64):
    """Rotate Q and K, then block-quantise Q, K and V to e4m3.

    q, k, v: [B, H, N, d] (any float dtype; converted to fp32 exactly when they are
    fp32 or bf16).  signs: [d] of +-1.  Returns a dict with uint8 codes
    ``q8, k8, v8`` ([B,H,N,d]) and float32 dequantisation scales ``sq, sk, sv``
    ([B,H,ceil(N/tile)]), such that  Q diag(s) H ~= decode(q8) * sq  (per tile) and
    likewise for K;  V ~= decode(v8) * sv.
    """
    def f32(x):
        if hasattr(x, "detach"):
            import torch

            x = x.detach().to("cpu", torch.float32).numpy()
        return np.asarray(x, dtype=np.float32)

    q32, k32, v32 = f32(q), f32(k), f32(v)
    qr = fwht_f32(q32, signs)
    kr = fwht_f32(k32, signs)
    q8, sq = _quantise_tiles(qr, tile)
    k8, sk = _quantise_tiles(kr, tile)
    v8, sv = _quantise_tiles(v32, tile)
    return {"q8": q8, "k8": k8, "v8": v8, "sq": sq, "sk": sk, "sv": sv}


def fp8_dequantize(codes: np.ndarray, sigma: np.ndarray, tile: int = 64) -> np.ndarray:
    """float64 values decode(codes) * sigma(tile of the row), shapes as in fp8_prepare."""
    vals = e4m3_decode(codes)
    N = codes.shape[-2]
    rows_tile = np.arange(N) // tile
    return vals * sigma.astype(np.float64)[..., rows_tile][..., None]


# --------------------------------------------------- seeded rotation signs
#
# When the caller gives a 64-bit seed instead of a sign vector, the signs come
# from SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
# pseudorandom number generators", OOPSLA 2014; the generator as published in its
# reference implementation): state x starts at the seed; each output adds the
# constant 0x9E3779B97F4A7C15 to x (mod 2^64) and returns the mixed value
#     z = x;  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
#     z = (z ^ (z >> 27)) * 0x94D049BB133111EB;  z ^ (z >> 31)      (mod 2^64).
# Output c (0-based) thus depends only on (seed, c): the generator is counter-based.
# Column c's sign is -1 when the top bit of output c is set, else +1.  This is the
# library's definition of the seeded rotation; the library implements it in its own code.

_MASK64 = (1 << 64) - 1
_SPLITMIX_GAMMA = 0x9E3779B97F4A7C15


def splitmix64(seed: int, count: int) -> list[int]:
    """The first ``count`` SplitMix64 outputs from state ``seed`` (Python integers, exact)."""
    x = seed & _MASK64
    out = []
    for _ in range(count):
        x = (x + _SPLITMIX_GAMMA) & _MASK64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def seeded_rotation_signs(seed: int, d: int) -> np.ndarray:
    """The +-1 signs (int8 [d]) of the seeded rotation: sign of column c from output c's top bit."""
    return np.array([-1 if (z >> 63) else 1 for z in splitmix64(seed, d)], dtype=np.int8)
