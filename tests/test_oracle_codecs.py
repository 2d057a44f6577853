"""Pins for oracle/codecs.py: hand-worked values (tests/golden/), exhaustive round trips and
properties fixed by the formats' definitions.  Nothing here re-uses the oracle's own tables to
produce an expected value."""
import math

import numpy as np
import pytest

from conftest import golden_lines
from oracle import codecs as C


def test_golden_scalar_formats():
    n = 0
    for f in golden_lines("codecs.txt"):
        kind = f[0]
        if kind == "e2m1":
            got = C.e2m1_value(int(f[1], 16))
            want = float(f[2])
            assert got == want and math.copysign(1, got) == math.copysign(1, want), f
        elif kind == "e8m0":
            assert float(C.e8m0_value(int(f[1]))) == float(f[2]), f
        elif kind == "e4m3":
            got = C.e4m3_value(int(f[1], 16))
            want = float(f[2])
            assert got == want and math.copysign(1, got) == math.copysign(1, want), f
        elif kind == "fp4byte":
            codes = C.unpack_fp4(np.array([[int(f[1], 16)]], dtype=np.uint8))[0]
            assert C.E2M1_TABLE[codes].tolist() == [float(f[2]), float(f[3])], f
        else:
            raise AssertionError(kind)
        n += 1
    assert n > 30


def test_e2m1_grid_properties():
    # magnitudes of the 8 positive codes are the OCP FP4 grid; the sign bit negates
    mags = [C.e2m1_value(c) for c in range(8)]
    assert mags == sorted(mags) and len(set(mags)) == 8
    for c in range(8):
        assert C.e2m1_value(c | 8) == -C.e2m1_value(c)
    # E2M1 values times 2 are integers (one mantissa bit, smallest step 0.5)
    assert all(float(2 * m).is_integer() for m in mags)


def test_fp4_pack_roundtrip_exhaustive():
    codes = np.array([[a, b] for a in range(16) for b in range(16)], dtype=np.uint8).reshape(1, -1)
    packed = C.pack_fp4(codes)
    assert packed.shape == (1, 256)
    assert sorted(packed[0].tolist()) == list(range(256))      # bijection on bytes
    assert np.array_equal(C.unpack_fp4(packed), codes)


def test_e4m3_table_properties():
    t = C.E4M3_TABLE
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2                                # only S.1111.111
    pos = t[:127]
    assert np.all(np.diff(pos) > 0)                              # strictly increasing grid
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    assert np.array_equal(t[128:255], -pos)                      # sign symmetry
    # within each binade 8 equal steps; the subnormal step equals the first normal step
    for e in range(1, 15):
        b = pos[8 * e: 8 * e + 8]
        assert np.allclose(np.diff(b), 2.0 ** (e - 10))
    assert np.allclose(np.diff(pos[:9]), 2.0 ** -9)


def test_e4m3_table_matches_library_cast():
    ml = pytest.importorskip("ml_dtypes")
    lib = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    ok = ~np.isnan(lib)
    assert np.array_equal(np.isnan(lib), np.isnan(C.E4M3_TABLE))
    assert np.array_equal(lib[ok], C.E4M3_TABLE[ok])


def test_e4m3_encode_roundtrip_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(C.e4m3_encode_rne_sat(C.e4m3_decode(codes)), codes)


def test_e4m3_encode_rounding_and_saturation():
    pos = C.E4M3_TABLE[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    got = C.e4m3_encode_rne_sat(mids)
    lo = np.arange(126)
    # ties go to the even code (even mantissa)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want)
    # just above / below a midpoint go to the nearer neighbour
    assert np.array_equal(C.e4m3_encode_rne_sat(np.nextafter(mids, np.inf)), lo + 1)
    assert np.array_equal(C.e4m3_encode_rne_sat(np.nextafter(mids, -np.inf)), lo)
    # saturation: everything >= 448 (incl. what would round to 480) maps to 0x7E
    assert C.e4m3_encode_rne_sat(np.array([448.0, 463.9, 464.0, 500.0, 1e30])).tolist() == [0x7E] * 5
    assert C.e4m3_encode_rne_sat(np.array([-1e30])).tolist() == [0xFE]


def test_e4m3_encode_matches_library_cast_in_range():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 10, 100)])
    v = v[np.abs(v) <= 440].astype(np.float32)        # library cast does not saturate
    lib = v.astype(ml.float8_e4m3fn).view(np.uint8)
    got = C.e4m3_encode_rne_sat(v.astype(np.float64))
    assert np.array_equal(lib, got)


def test_bf16_round_matches_library_cast():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(50000) * np.exp(rng.uniform(-30, 30, 50000))).astype(np.float32)
    lib = v.astype(ml.bfloat16).astype(np.float64)
    assert np.array_equal(C.bf16_round(v.astype(np.float64)), lib)


def test_bf16_round_by_definition():
    # values with <= 8 significant bits are fixed points; ties go to even
    assert C.bf16_round(np.array([1.0, 1.0 + 2 ** -7, 3.0, -255.0])).tolist() == [1.0, 1.0 + 2 ** -7, 3.0, -255.0]
    assert C.bf16_round(np.array([1.0 + 2 ** -8])).tolist() == [1.0]                      # tie -> even
    assert C.bf16_round(np.array([1.0 + 3 * 2 ** -8])).tolist() == [1.0 + 2 ** -6]        # tie -> even
    assert C.bf16_round(np.array([1.0 + 2 ** -8 + 2 ** -20])).tolist() == [1.0 + 2 ** -7]
    bits = C.f64_to_bf16_bits(np.array([1.0, -2.0, 0.0]))
    assert bits.tolist() == [0x3F80, 0xC000, 0x0000]
    assert C.bf16_bits_to_f64(np.array([0x3F80, 0x4049], dtype=np.uint16)).tolist() == [1.0, 3.140625]


def test_mxfp8_golden_blocks():
    n = 0
    for f in golden_lines("mxfp8_blocks.txt"):
        amax, probe, sbyte, code = float(f[0]), float(f[1]), int(f[2]), int(f[3], 16)
        block = np.zeros(32)
        block[0] = amax
        block[1] = probe
        q, s = C.mxfp8_quantize(block[None, :])
        assert int(s[0, 0]) == sbyte, f
        assert int(q[0, 1]) == code, f
        n += 1
    assert n >= 10


def test_mxfp8_properties():
    rng = np.random.default_rng(7)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    q, s = C.mxfp8_quantize(v)
    d = C.mxfp8_dequantize(q, s)
    blocks = v.reshape(64, 8, 32)
    amax = np.abs(blocks).max(-1)
    scale = 2.0 ** (s.astype(np.float64) - 127)
    # amax / scale lies in [256, 512): the block maximum uses the top binade of E4M3
    r = amax / scale
    assert np.all((r >= 256) & (r < 512))
    # per element error <= half an E4M3 step at the element's binade, or the saturation error
    err = np.abs(d - v).reshape(64, 8, 32)
    scaled = np.abs(blocks) / scale[..., None]
    binade = np.floor(np.log2(np.maximum(scaled, 2.0 ** -6)))
    half_step = 2.0 ** (binade - 3) / 2 * scale[..., None]
    sat = np.maximum(np.abs(blocks) - 448 * scale[..., None], 0)
    assert np.all(err <= half_step + sat + 1e-300)
    # scale-invariance: multiplying a block by 2^j shifts only the scale byte
    q2, s2 = C.mxfp8_quantize(v * 2.0 ** 5)
    assert np.array_equal(q2, q) and np.array_equal(s2.astype(int), s.astype(int) + 5)


def test_nf3_golden_and_roundtrip():
    for f in golden_lines("nf3.txt"):
        if f[0] == "lut":
            assert C.NF3_LUT[int(f[1])] == float(f[2])
            continue
        codes = np.array([[int(c) for c in f[0].split(",")]], dtype=np.uint8)
        packed = np.array([[int(b, 16) for b in f[1].split(",")]], dtype=np.uint8)
        assert np.array_equal(C.nf3_pack(codes), packed), f
        assert np.array_equal(C.nf3_unpack(packed, 8), codes), f
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 8, (5, 64)).astype(np.uint8)
    assert np.array_equal(C.nf3_unpack(C.nf3_pack(codes), 64), codes)
    raw = rng.integers(0, 256, (3, 24)).astype(np.uint8)
    assert np.array_equal(C.nf3_pack(C.nf3_unpack(raw, 64)), raw)


def test_nf3_dequant_definition():
    # one group of 32 codes (all code 6 = 0.6047) with scale 2.0 (E4M3 0x40), second group code 0
    codes = np.concatenate([np.full(32, 6), np.zeros(32)]).astype(np.uint8)[None, :]
    packed = C.nf3_pack(codes)
    sc = np.array([[0x40, 0x38]], dtype=np.uint8)
    d = C.nf3_dequant(packed, sc, 64)
    # 0.6047 as fp32 times 2 is exact in fp32; rounded to bf16 (8 significant bits)
    want0 = float(np.float32(0.6047) * np.float32(2.0))
    m, e = math.frexp(want0)
    want0 = round(m * 256) / 256 * 2 ** e
    assert np.all(d[0, :32] == want0)
    assert np.all(d[0, 32:] == -1.0)


def test_rounding_alternates():
    # scaled block: amax 256 -> scale byte 127 (scale 1); 1.0625 is the midpoint of 1.0 and 1.125
    v = np.zeros((1, 32))
    v[0, 0] = 256.0
    v[0, 1] = 1.0625 * (1 + 1e-6)      # just above the midpoint: nearest is 1.125
    v[0, 2] = 1.0625 * (1 - 1e-6)      # just below: nearest is 1.0
    v[0, 3] = 1.03                      # far from a midpoint
    mask, alt = C.mxfp8_alternates(v, 1e-4)
    assert mask[0, 1:3].tolist() == [True, True] and not mask[0, 3] and not mask[0, 0]
    assert alt[0, 1] == 1.0 and alt[0, 2] == 1.125
    assert alt[0, 3] == C.mxfp8_dequantize(*C.mxfp8_quantize(v))[0, 3]
    # bf16: 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7
    b = np.array([1 + 2 ** -8 + 1e-9, 1 + 2 ** -8 - 1e-9, 1.3])
    mask, alt = C.bf16_alternates(b, 1e-6)
    assert mask.tolist() == [True, True, False]
    assert alt[0] == 1.0 and alt[1] == 1 + 2 ** -7 and alt[2] == C.bf16_round(1.3)
    # the absolute part: 2^-20 * (1 + 2^-8) + 1e-9 is the midpoint of two tiny bf16 values plus
    # an offset far beyond 1e-6 of its size, but inside an absolute window of 2e-9
    t = np.array([2.0 ** -20 * (1 + 2 ** -8) + 1e-9, 0.5 + 1e-9])
    assert C.bf16_alternates(t, 1e-6)[0].tolist() == [False, False]
    mask, alt = C.bf16_alternates(t, 1e-6, atol=2e-9)
    assert mask.tolist() == [True, False] and alt[0] == 2.0 ** -20
    # MXFP8 with a per-element window: 1.0625 + 1e-3 is ambiguous only under atol 2e-3
    v[0, 1] = 1.0625 + 1e-3
    assert not C.mxfp8_alternates(v, 1e-4)[0][0, 1]
    atol = np.zeros_like(v)
    atol[0, 1] = 2e-3
    mask, alt = C.mxfp8_alternates(v, 1e-4, atol)
    assert mask[0, 1] and alt[0, 1] == 1.0 and not mask[0, 3]


def test_e2m1_encode_nearest_even_by_brute_force():
    """E2M1 encoding: for values on and between the grid (midpoints included), the code is the
    nearest of the eight magnitudes by exhaustive search, a tie takes the code with mantissa
    bit 0, magnitudes beyond 6 saturate, and the sign follows the input."""
    grid = C.E2M1_TABLE[:8]
    vals = np.concatenate([grid, (grid[1:] + grid[:-1]) / 2, np.linspace(0, 7, 113),
                           [6.0001, 1e9]])
    for v in vals:
        d = np.abs(grid - min(v, 6.0))
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert C.e2m1_encode_rne_sat(v) == want, v
        assert C.e2m1_encode_rne_sat(-v) == want | 8, v


def test_nvfp4_worked_block():
    """A block worked by hand: v = fp32(0.1 i), i = 0..15.  vmax / 6 = 0.25 = 2^-2, the E4M3
    code 0x28 (exponent field 5); v / 0.25 = 0, 0.4, 0.8, ..., 6 rounds to the E2M1 grid
    0, .5, 1, 1, 1.5, 2, 2, 3, 3, 4, 4, 4, 4, 6, 6, 6."""
    v = (np.arange(16, dtype=np.float32) * np.float32(0.1))[None, :]
    q, s = C.nvfp4_quantize(v)
    assert s.tolist() == [[0x28]]
    want = [0, .5, 1, 1, 1.5, 2, 2, 3, 3, 4, 4, 4, 4, 6, 6, 6]
    assert C.E2M1_TABLE[q[0]].tolist() == want
    assert np.allclose(C.nvfp4_dequantize(q, s)[0], np.array(want) * 0.25, rtol=0, atol=0)


def test_nvfp4_properties():
    """Random blocks: the scale is the E4M3 value nearest vmax / 6; every element is within
    half an E2M1 step (at its magnitude, in scaled units) of its dequantised value, except
    saturation past 6; zero blocks give zero codes; the alternates flag only near-midpoints."""
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((64, 64)) * 2.0 ** rng.integers(-8, 8, size=(64, 1))).astype(
        np.float32)
    v[3] = 0
    q, s = C.nvfp4_quantize(v)
    vmax = np.abs(v.reshape(64, 4, 16)).max(axis=-1) / 6
    sv = C.e4m3_decode(s)
    nxt = np.abs(C.E4M3_TABLE[np.minimum(s.astype(int) + 1, 126)] - vmax)
    prv = np.abs(C.E4M3_TABLE[np.maximum(s.astype(int) - 1, 0)] - vmax)
    assert np.all(np.abs(sv - vmax) <= np.minimum(nxt, prv) + 1e-30)
    assert np.all(q[3] == 0)
    x = np.abs(v.reshape(64, 4, 16)) / np.where(sv > 0, sv, 1)[..., None]
    deq = C.E2M1_TABLE[q.reshape(64, 4, 16) & 7]
    step = np.where(deq < 2, 0.5, np.where(deq < 4, 1.0, 2.0))
    ok = (np.abs(x - deq) <= step / 2 + 1e-6) | (x > 6)
    assert np.all(ok | (sv == 0)[..., None])
    mask, alt = C.nvfp4_alternates(v.astype(np.float64), 1e-4)
    near = C.nvfp4_dequantize(q, s)
    assert np.all(alt[~mask] == near[~mask])
    assert mask.mean() < 1e-2


# ---------------------------------------------------------------------------- static FP8

def test_fp8_static_worked_values():
    """Hand-worked: s = 0.5 (1 / s = 2 exactly): 1.3 -> 2.6 lies between the E4M3 neighbours 2.5
    (code 0x42: exponent 8, mantissa 2) and 2.75, nearer 2.5 -> 1.25; 300 -> 600 saturates to
    448 (0x7E) -> 224; -0.001 -> -0.002, nearest the subnormal 2^-9 (0x81) -> -2^-10; 0 -> 0.
    Ties go to the even mantissa: with s = 1, 2.625 (between 2.5 = 0x42 and 2.75 = 0x43) -> 2.5,
    2.875 (between 2.75 and 3.0 = 0x44) -> 3.0."""
    q, v = C.fp8_static_quantize(np.array([1.3, 300.0, -0.001, 0.0]), 0.5)
    assert q.tolist() == [0x42, 0x7E, 0x81, 0x00]
    assert v.tolist() == [1.25, 224.0, -2.0 ** -10, 0.0]
    q, v = C.fp8_static_quantize(np.array([2.625, 2.875, -2.625, 464.0, 1e9]), 1.0)
    assert q.tolist() == [0x42, 0x44, 0xC2, 0x7E, 0x7E]
    assert v.tolist() == [2.5, 3.0, -2.5, 448.0, 448.0]


def test_fp8_static_reciprocal_is_fp32():
    """The scaled value is the fp32 product with the fp32 reciprocal of the scale, not the
    exact quotient.  s = fp32(0.3), v = fp32 0x3DA33334 = 0.0796875059...: the exact quotient
    v / s = 0.265625009... lies just above the midpoint 0.265625 of the E4M3 neighbours 0.25
    (code 0x28) and 0.28125 (0x29), so it would round to 0x29; the fp32 product
    v x fp32(1 / s) is exactly 0.265625, a tie, which goes to the even code 0x28."""
    s = np.float32(0.3)
    v = np.array([0x3DA33334], dtype=np.uint32).view(np.float32)[0]
    assert float(np.float32(v * (np.float32(1.0) / s))) == 0.265625
    assert float(v) / float(s) > 0.265625
    q, deq = C.fp8_static_quantize(np.array([float(v)]), float(s))
    assert int(q[0]) == 0x28 and deq[0] == 0.25 * float(s)


def test_fp8_static_equals_mxfp8_when_the_block_scale_matches():
    """Closed form against the pinned MX quantiser: for a power-of-two scale s = 2^k and a
    block whose largest magnitude lies in [256 s, 512 s), the MX scale byte is 127 + k, so the
    MXFP8 codes of the block are the static FP8 codes (both round v / s to E4M3, saturating)."""
    rng = np.random.default_rng(5)
    for k in (-9, -3, 0, 4):
        s = 2.0 ** k
        v = rng.normal(0, 60 * s, size=(50, 32))
        v[:, 0] = rng.uniform(256 * s, 511 * s, size=50)
        qs, _ = C.fp8_static_quantize(v, s)
        qm, sm = C.mxfp8_quantize(v)
        assert np.all(sm == 127 + k)
        assert np.array_equal(qs, qm)


def test_fp8_static_matches_exhaustive_search():
    """Against a scalar exhaustive search (nearest of the 127 finite magnitudes, ties to the
    even code, saturating), on random values, exact midpoints and out-of-range values."""
    rng = np.random.default_rng(9)
    s = float(np.float32(0.0173))
    inv = np.float32(1.0) / np.float32(s)
    mids = (C.E4M3_TABLE[1:127] + C.E4M3_TABLE[:126]) / 2
    vals = np.concatenate([rng.normal(0, 3, 400), mids[::5] * s, [500 * s, -1e6, 0.0]])
    q, deq = C.fp8_static_quantize(vals, s)
    grid = [C.e4m3_value(c) for c in range(127)]
    for v, qc, d in zip(vals, q, deq):
        p = float(np.float32(np.float32(v) * inv))
        mag = min(abs(p), 448.0)
        c = min(range(127), key=lambda c: (abs(grid[c] - mag), c % 2))
        assert int(qc) & 0x7F == c
        assert d == math.copysign(grid[c], p) * float(np.float32(s)) or (c == 0 and d == 0)


def test_fp8_static_alternates_worked():
    """With s = 1: 2.6249 and 2.6251 sit within 1e-4 of the midpoint 2.625 of 2.5 and 2.75 -
    nearest 2.5 and 2.75, alternates 2.75 and 2.5; 2.55 is far from any midpoint (no
    alternate); with s = 0.25 the same scaled values give the same decisions, values x 0.25."""
    for s in (1.0, 0.25):
        v = np.array([2.6249, 2.6251, 2.55]) * s
        mask, alt = C.fp8_static_alternates(v, s, 1e-4)
        _, near = C.fp8_static_quantize(v, s)
        assert mask.tolist() == [True, True, False]
        assert (near / s).tolist() == [2.5, 2.75, 2.5]
        assert (alt / s).tolist() == [2.75, 2.5, 2.5]
