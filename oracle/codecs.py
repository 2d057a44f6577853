"""Number formats of the MoE path, written from their bit-field definitions (fp64, numpy).

Sources on the pages:
  * MXFP4 weights = E2M1 codes with one E8M0 scale per 32 along K
    (moe_b12x_next.py, module docstring and ``_Geometry.__init__``: ``MXFP4_E8M0_K32``).
  * E8M0 decode is 2^(e-127) (hybrid_loader.py, ``_fp8_ne_transform._deq``).
  * NVFP4 weights = E2M1 with an E4M3 scale per 16 and a per-expert fp32 global scale
    (hybrid_loader.py, ``_deq_nv`` and the NVFP4 ``weight_scale_2`` tensors).
  * NF3 = 3-bit codes into an 8-entry LUT, 8 codes per 3 bytes, scale per 32
    (hybrid_loader.py, ``_NF3_VALS`` and ``_unpack_nf3``).
  * MXFP8 activations (E4M3 codes + E8M0 scale per 32) are produced inside the kernel
    (moe_b12x_next.py, module docstring "in-kernel MXFP8 activations"); the pages do not print
    the scale rule, so the OCP MX v1.0 rule is used: shared exponent = floor(log2 amax) - 8
    (8 = emax of E4M3), elements rounded to nearest-even and saturated to +-448.

Pinned by tests/test_oracle_codecs.py (hand-worked values in tests/golden/, exhaustive round
trips, and an independent library cast for the element rounding only).
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------- E2M1 (FP4)

def e2m1_value(code: int) -> float:
    """One E2M1 nibble: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
    Exponent 0 is subnormal: m * 0.5."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if e == 0 else (2.0 ** (e - 1)) * (1.0 + 0.5 * m)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


_E2M1_POS = E2M1_TABLE[:8]          # 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7)


def e2m1_encode_rne_sat(v) -> np.ndarray:
    """fp64 -> E2M1 code: nearest of the eight magnitudes, ties to the even code (mantissa bit
    0), saturating to 6; the sign bit is the input's sign (so -0 for a negative value that
    rounds to zero)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 6.0)
    lo = np.clip(np.searchsorted(_E2M1_POS, a, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    dlo = a - _E2M1_POS[lo]
    dhi = _E2M1_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x8, code).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """[..., n] bytes -> [..., 2n] nibble codes; element 2j is the low nibble of byte j."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0x0F) | ((c[..., 1::2] & 0x0F) << 4)


# ---------------------------------------------------------------------------- E8M0

def e8m0_value(b) -> np.ndarray:
    """E8M0 scale byte -> 2^(b-127); 0xFF is NaN."""
    b = np.asarray(b, dtype=np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, v)


# ---------------------------------------------------------------------------- E4M3 (fn)

def e4m3_value(code: int) -> float:
    """E4M3 'fn': sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
    Exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0
# positive finite magnitudes, codes 0..126, ascending
_E4M3_POS = E4M3_TABLE[:127]


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_rne_sat(v) -> np.ndarray:
    """fp64 -> E4M3 code: round to nearest, ties to even mantissa, saturate to +-448.
    NaN is never produced for finite input (the 'satfinite' rule).  The sign bit is the
    input's sign, so a negative value that rounds to zero gives -0 (0x80), as IEEE rounding
    keeps the sign of a zero result."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    # index of the largest grid value <= a
    lo = np.searchsorted(_E4M3_POS, a, side="right") - 1
    lo = np.clip(lo, 0, 126)
    hi = np.minimum(lo + 1, 126)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (lo % 2 == 1))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)


# ---------------------------------------------------------------------------- bf16

def bf16_round(v) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.  bf16 = 8 significant
    bits, exponent range of fp32 (normals down to 2^-126, subnormal step 2^-133)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = (v != 0) & np.isfinite(v)
    _, ex = np.frexp(v[nz])               # v = f * 2^ex, 0.5 <= |f| < 1
    e = ex.astype(np.int64) - 1            # floor(log2 |v|)
    q = np.maximum(e, -126) - 7            # exponent of one unit in the last place
    r = np.round(np.ldexp(v[nz], -q))      # numpy rounds half to even
    out[nz] = np.ldexp(r, q)
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    big = np.abs(out) >= 2.0 ** 128
    out[big] = np.copysign(np.inf, out[big])
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    r = bf16_round(v).astype(np.float32)
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def f32_round(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------- MXFP8 quantiser

MX_BLOCK = 32
E4M3_EMAX = 8


def biased_exponent(a) -> np.ndarray:
    """Biased binary exponent field of a non-negative value as an fp32 would store it:
    floor(log2 a) + 127 for normals, 0 for zero and fp32 subnormals."""
    a = np.asarray(a, dtype=np.float64)
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1 + 127
    return np.where(a >= 2.0 ** -126, e, 0)


def mxfp8_quantize(v: np.ndarray):
    """Quantise the last axis (a multiple of 32) to MXFP8.

    Per block of 32: amax = max |v|; scale byte s = clamp(E(amax) - 8, 0, 254) where E is the
    biased exponent (so the scale is 2^(floor(log2 amax) - 8)); code = E4M3 RNE-saturated
    value of v / 2^(s-127).  An all-zero block has scale byte 0 and zero codes.
    Returns (codes uint8 [..., K], scale bytes uint8 [..., K/32]).
    """
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    assert K % MX_BLOCK == 0
    blocks = v.reshape(v.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    s = np.clip(biased_exponent(amax) - E4M3_EMAX, 0, 254)
    scaled = np.ldexp(blocks, (127 - s)[..., None])
    codes = e4m3_encode_rne_sat(scaled).reshape(v.shape)
    return codes, s.astype(np.uint8)


def mxfp8_alternates(v: np.ndarray, rel: float, atol=0.0):
    """Elements whose MXFP8 rounding is decided by noise: the exact value lies within
    rel * |value| + atol of the midpoint between its two E4M3 neighbours (under the block scale
    the quantiser picks), so arithmetic that is exact only to that error may return either
    neighbour.  `atol` (a scalar or an array broadcasting against v) covers sums that cancel:
    their rounding error follows the size of the terms, not of the result.  Returns (mask,
    alternate dequantised value) with the same shape as v; where mask is False the alternate
    equals the nearest value."""
    v = np.asarray(v, dtype=np.float64)
    q, s = mxfp8_quantize(v)
    K = v.shape[-1]
    sc = np.repeat(e8m0_value(s), MX_BLOCK, axis=-1).reshape(v.shape)
    near = e4m3_decode(q) * sc                       # the quantiser's choice
    a = np.abs(v) / sc                                # magnitude in scaled units
    lo = np.clip(np.searchsorted(_E4M3_POS, np.minimum(a, E4M3_MAX), side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    mid = (_E4M3_POS[lo] + _E4M3_POS[hi]) / 2
    tol = rel * a + np.broadcast_to(np.asarray(atol, dtype=np.float64), v.shape) / sc
    mask = (np.abs(a - mid) <= tol) & (hi != lo) & (a < E4M3_MAX)
    other_mag = np.where(np.isclose(np.abs(near) / sc, _E4M3_POS[lo], rtol=0, atol=0),
                         _E4M3_POS[hi], _E4M3_POS[lo])
    alt = np.where(mask, np.copysign(other_mag * sc, v), near)
    return mask, alt


def bf16_alternates(v: np.ndarray, rel: float, atol=0.0):
    """As mxfp8_alternates for rounding to bf16: elements within rel * |value| + atol of the
    midpoint of their two bf16 neighbours, and the neighbour the nearest rounding did not
    pick."""
    v = np.asarray(v, dtype=np.float64)
    near = bf16_round(v)
    _, ex = np.frexp(np.where(v == 0, 1.0, v))
    ulp = np.ldexp(1.0, np.maximum(ex.astype(np.int64) - 1, -126) - 7)
    other = np.where(np.abs(v) >= np.abs(near), near + np.sign(v) * ulp, near - np.sign(v) * ulp)
    mid = (near + other) / 2
    mask = (np.abs(v - mid) <= rel * np.abs(v) + atol) & (v != 0)
    return mask, np.where(mask, other, near)


# ---------------------------------------------------------------------------- static FP8

def fp8_static_quantize(v, s):
    """Static per-tensor symmetric FP8 (hybrid_loader.py ``_build_kept_mxfp4``: the A8 opt-in
    selects ``kFp8StaticTensorSym`` for the kept experts, whose layer carries one fp32
    ``w13_input_scale`` / ``w2_input_scale``).  Reading (the page gives no arithmetic): each
    step in fp32 - the activation times the fp32 reciprocal of the scale, rounded to E4M3
    (nearest, ties to even, saturating at +-448) - and the dequantised value is code x s.
    Returns (codes uint8, dequantised values fp64) with the shape of v."""
    s32 = np.float32(s)
    inv = np.float32(1.0) / s32
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    codes = e4m3_encode_rne_sat((v32 * inv).astype(np.float64))
    return codes, e4m3_decode(codes) * np.float64(s32)


def fp8_static_alternates(v, s, rel: float, atol=0.0):
    """As mxfp8_alternates for the static per-tensor FP8 rounding of fp8_static_quantize: the
    elements whose scaled value v / s lies within rel * |v / s| + atol / s of the midpoint of its
    two E4M3 neighbours, and the neighbour's dequantised value."""
    v = np.asarray(v, dtype=np.float64)
    s64 = np.float64(np.float32(s))
    _, near = fp8_static_quantize(v, s)
    a = np.abs(v) / s64
    lo = np.clip(np.searchsorted(_E4M3_POS, np.minimum(a, E4M3_MAX), side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    mid = (_E4M3_POS[lo] + _E4M3_POS[hi]) / 2
    tol = rel * a + np.broadcast_to(np.asarray(atol, dtype=np.float64), v.shape) / s64
    mask = (np.abs(a - mid) <= tol) & (hi != lo) & (a < E4M3_MAX)
    other_mag = np.where(np.abs(near) / s64 == _E4M3_POS[lo], _E4M3_POS[hi], _E4M3_POS[lo])
    alt = np.where(mask, np.copysign(other_mag * s64, v), near)
    return mask, alt


# ---------------------------------------------------------------------------- NVFP4 activations

NV_BLOCK = 16


def nvfp4_quantize(v32: np.ndarray):
    """Quantise fp32 values (last axis a multiple of 16) to NVFP4 blocks of 16, every step in
    fp32 arithmetic (the decisions are taken in the precision the kernels use):
    vmax = max |v|;  scale code s = E4M3(fp32(vmax / 6)) (nearest-even, saturating);
    code = E2M1(fp32(v / E4M3value(s))) (nearest-even, saturating), all zero when s is 0.
    Returns (E2M1 codes uint8 [..., K], E4M3 scale codes uint8 [..., K/16])."""
    v = np.asarray(v32, dtype=np.float32)
    K = v.shape[-1]
    assert K % NV_BLOCK == 0
    blocks = v.reshape(v.shape[:-1] + (K // NV_BLOCK, NV_BLOCK))
    vmax = np.abs(blocks).max(axis=-1)
    s = e4m3_encode_rne_sat((vmax / np.float32(6.0)).astype(np.float32).astype(np.float64))
    sv = e4m3_decode(s).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blocks / sv[..., None]).astype(np.float32)
    codes = np.where((sv > 0)[..., None], e2m1_encode_rne_sat(q.astype(np.float64)), 0)
    return codes.reshape(v.shape).astype(np.uint8), s


def nvfp4_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    vals = E2M1_TABLE[np.asarray(codes, dtype=np.uint8)]
    K = vals.shape[-1]
    sc = e4m3_decode(scales)
    return (vals.reshape(vals.shape[:-1] + (K // NV_BLOCK, NV_BLOCK)) * sc[..., None]).reshape(
        vals.shape)


def nvfp4_alternates(v: np.ndarray, rel: float):
    """As mxfp8_alternates for NVFP4 blocks (under the scale the quantiser picks from v):
    elements whose scaled magnitude lies within rel of the midpoint of two E2M1 neighbours, and
    the dequantised value of the neighbour the nearest rounding did not pick."""
    v = np.asarray(v, dtype=np.float64)
    q, s = nvfp4_quantize(v.astype(np.float32))
    sc = np.repeat(e4m3_decode(s), NV_BLOCK, axis=-1).reshape(v.shape)
    near = nvfp4_dequantize(q, s)
    with np.errstate(divide="ignore", invalid="ignore"):
        a = np.where(sc > 0, np.abs(v) / sc, 0.0)
    lo = np.clip(np.searchsorted(_E2M1_POS, np.minimum(a, 6.0), side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    mid = (_E2M1_POS[lo] + _E2M1_POS[hi]) / 2
    mask = (np.abs(a - mid) <= rel * a) & (hi != lo) & (a < 6.0) & (sc > 0)
    picked_lo = np.abs(near) == _E2M1_POS[lo] * sc
    other = np.where(picked_lo, _E2M1_POS[hi], _E2M1_POS[lo]) * sc
    return mask, np.where(mask, np.copysign(other, v), near)


def mxfp8_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    vals = e4m3_decode(codes)
    K = vals.shape[-1]
    sc = e8m0_value(scales)
    return (vals.reshape(vals.shape[:-1] + (K // MX_BLOCK, MX_BLOCK)) * sc[..., None]).reshape(vals.shape)


# ---------------------------------------------------------------------------- NF3

# The 8-entry NF3 table exactly as printed (hybrid_loader.py, ``_NF3_VALS``).
NF3_LUT = (-1.0, -0.6047, -0.3563, -0.1275, 0.1275, 0.3563, 0.6047, 1.0)
NF3_GROUP = 32


def nf3_unpack(packed: np.ndarray, n_cols: int) -> np.ndarray:
    """[R, n_cols/8*3] bytes -> [R, n_cols] codes.  Each 3-byte group b0,b1,b2 forms the
    24-bit word b0 | b1<<8 | b2<<16 whose bits 3i..3i+2 are code i (hybrid_loader.py,
    ``_unpack_nf3``)."""
    p = np.asarray(packed, dtype=np.uint32)
    R = p.shape[0]
    p = p.reshape(R, n_cols // 8, 3)
    w24 = p[..., 0] | (p[..., 1] << 8) | (p[..., 2] << 16)
    codes = np.stack([(w24 >> (3 * i)) & 7 for i in range(8)], axis=-1)
    return codes.reshape(R, n_cols).astype(np.uint8)


def nf3_pack(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint32)
    R, n = c.shape
    c = c.reshape(R, n // 8, 8)
    w24 = np.zeros((R, n // 8), dtype=np.uint32)
    for i in range(8):
        w24 |= (c[..., i] & 7) << (3 * i)
    out = np.stack([w24 & 0xFF, (w24 >> 8) & 0xFF, (w24 >> 16) & 0xFF], axis=-1)
    return out.reshape(R, n // 8 * 3).astype(np.uint8)


def nf3_dequant(packed: np.ndarray, scale_codes: np.ndarray, n_cols: int) -> np.ndarray:
    """NF3 weight values as the page's unpack produces them: the LUT entry (held as fp32) times
    the fp32 value of the E4M3 group scale, the product rounded to bf16
    (``_unpack_nf3``: ``(nf[codes] * scale.float().repeat_interleave(32, 1)).to(bfloat16)``)."""
    codes = nf3_unpack(packed, n_cols)
    lut32 = np.array(NF3_LUT, dtype=np.float32)
    sc32 = e4m3_decode(scale_codes).astype(np.float32)
    prod32 = lut32[codes] * np.repeat(sc32, NF3_GROUP, axis=1)      # fp32 multiply
    return bf16_round(prod32.astype(np.float64))
