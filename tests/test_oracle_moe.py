"""Pins for oracle/moe.py: routing (hand-worked + brute force), SwiGLU closed forms, the forward
against a brute-force per-element loop, a closed-form layer, and the invariants the method fixes
(linearity in the router weights, padding rows, token-order invariance, w13 halves)."""
import math

import numpy as np
import pytest

from conftest import golden_lines
from oracle import codecs as C
from oracle import moe as O
import synth
from synth import moe_inputs as S


def _ints(s):
    return [int(v) for v in s.split(",")]


# ---------------------------------------------------------------------------- routing

def test_routing_golden():
    g = {f[0]: f[1:] for f in golden_lines("routing.txt")}
    E = int(g["E"][0])
    ids = np.array([_ints(r) for r in g["ids"]], dtype=np.int32)
    cnt, off, perm, slot_of = O.route(ids, E)
    assert cnt.tolist() == _ints(g["cnt"][0])
    assert off.tolist() == _ints(g["off"][0])
    assert perm.tolist() == _ints(g["perm"][0])
    assert slot_of.tolist() == _ints(g["slot_of"][0])


def _route_bruteforce(ids, E):
    flat = [int(v) for v in np.asarray(ids).ravel()]
    buckets = [[] for _ in range(E)]
    for f, e in enumerate(flat):
        if 0 <= e < E:
            buckets[e].append(f)
    perm = [f for b in buckets for f in b]
    slot_of = [-1] * len(flat)
    for p, f in enumerate(perm):
        slot_of[f] = p
    cnt = [len(b) for b in buckets]
    off = [0]
    for c in cnt:
        off.append(off[-1] + c)
    return cnt, off, perm, slot_of


@pytest.mark.parametrize("seed", range(6))
def test_routing_bruteforce(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 40))
    M, k = int(rng.integers(0, 50)), int(rng.integers(1, 9))
    ids = rng.integers(-3, E + 3, (M, k)).astype(np.int32)
    got = O.route(ids, E)
    want = _route_bruteforce(ids, E)
    for a, b in zip(got, want):
        assert list(np.asarray(a)) == list(b)


# ---------------------------------------------------------------------------- SwiGLU

def test_swiglu_closed_forms():
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    L = 7.0
    cases = [  # gate, up, expected
        (0.0, 5.0, 0.0),
        (1.0, 2.0, 1.0 * sig(1.0) * 2.0),
        (14.0, 14.0, 7.0 * sig(7.0) * 7.0),              # gate clamped from above, up too
        (-14.0, -14.0, -14.0 * sig(-14.0) * -7.0),       # gate not clamped from below
        (7.0, -7.0, 7.0 * sig(7.0) * -7.0),
    ]
    for g, u, want in cases:
        assert O.swiglu(np.array([g]), np.array([u]), L)[0] == pytest.approx(want, rel=1e-15)
    # no limit: silu(g) * u
    g = np.linspace(-20, 20, 41)
    u = np.linspace(-3, 3, 41)
    assert np.allclose(O.swiglu(g, u), g / (1 + np.exp(-g)) * u, rtol=1e-15)
    # alpha / beta form
    assert O.swiglu(np.array([2.0]), np.array([1.0]), 7.0, 1.702, 1.0)[0] == pytest.approx(
        2.0 * sig(1.702 * 2.0) * 2.0, rel=1e-15)


# ---------------------------------------------------------------------------- forward

def _tiny(quant, seed=0, E=6, H=64, I=32, layout=S.W13_UP_GATE):
    cfg = {"mxfp4": S.CONFIGS["tiny_w4a8"], "nvfp4": S.CONFIGS["w4a16_nvfp4"],
           "w4a8_nvfp4": S.CONFIGS["w4a8_nvfp4"], "w4a4_nvfp4": S.CONFIGS["w4a4_nvfp4"],
           "hybrid": S.CONFIGS["hybrid_nvfp4_nf3"],
           "hybrid_mx": S.CONFIGS["hybrid_mxfp4_nf3"]}[quant]
    if quant in ("hybrid", "hybrid_mx"):
        cfg = S.MoEConfig(**{**cfg.__dict__, "n_nvfp4": 2})
    ck = S.make_checkpoint(cfg, seed=seed, E=E, H=H, I=I, layout=layout)
    return cfg, ck


@pytest.mark.parametrize("quant,layout", [("mxfp4", 0), ("mxfp4", 1), ("nvfp4", 0), ("hybrid", 0),
                                          ("hybrid_mx", 0), ("hybrid_mx", 1), ("w4a8_nvfp4", 0),
                                          ("w4a4_nvfp4", 0), ("w4a4_nvfp4", 1)])
def test_forward_matches_bruteforce(quant, layout):
    cfg, ck = _tiny(quant, layout=layout)
    rng = np.random.default_rng(11)
    M, k = 5, 2
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    ids[4, 1] = -1
    ids[3, 0] = ck.E          # out of range: dropped
    w = S.router_weights(rng, M, k, "softmax", 1.0)
    lim = 7.0 if quant == "mxfp4" else math.inf
    a, f64 = O.moe_forward(ck, x, ids, w, lim, return_f64=True)
    b = O.moe_forward_bruteforce(ck, x, ids, w, lim)
    # both are fp64 sums of the same terms in different orders; the bf16 results agree except
    # where the fp64 sum sits within rounding noise of a bf16 midpoint
    da = C.bf16_bits_to_f64(a)
    db = C.bf16_bits_to_f64(b)
    assert np.mean(da == db) > 0.999
    assert np.allclose(da, db, rtol=2 ** -7, atol=0)


@pytest.mark.parametrize("quant", ["nvfp4", "hybrid_mx"])
def test_weight_on_input_matches_bruteforce(quant):
    """Router weights applied to fc1's input: the dgemm form against the element loop."""
    cfg, ck = _tiny(quant)
    rng = np.random.default_rng(21)
    M, k = 4, 2
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    ids[3, 1] = -1
    w = S.router_weights(rng, M, k, "sigmoid_norm", 2.5)
    a, _ = O.moe_forward(ck, x, ids, w, return_f64=True, weight_on_input=True)
    b = O.moe_forward_bruteforce(ck, x, ids, w, weight_on_input=True)
    da, db = C.bf16_bits_to_f64(a), C.bf16_bits_to_f64(b)
    assert np.mean(da == db) > 0.999
    assert np.allclose(da, db, rtol=2 ** -7, atol=0)


def test_weight_on_input_special_cases():
    """Weights 1 on the input give the standard layer exactly (x * 1 = x, combine weight 1);
    any other weight changes the SwiGLU's argument, so the results differ; W4A8 refuses."""
    cfg, ck = _tiny("hybrid")
    rng = np.random.default_rng(22)
    M, k = 5, 2
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    ones = np.ones((M, k), np.float32)
    _, f0 = O.moe_forward(ck, x, ids, ones, return_f64=True)
    _, f1 = O.moe_forward(ck, x, ids, ones, return_f64=True, weight_on_input=True)
    assert np.array_equal(f0, f1)
    halves = np.full((M, k), 0.5, np.float32)
    _, g0 = O.moe_forward(ck, x, ids, halves, return_f64=True)
    _, g1 = O.moe_forward(ck, x, ids, halves, return_f64=True, weight_on_input=True)
    assert not np.allclose(g0, g1)
    _, ck8 = _tiny("mxfp4")
    with pytest.raises(AssertionError):
        O.moe_forward(ck8, x[:, :ck8.H], ids % ck8.E, ones, weight_on_input=True)


def _nv_a8_case(seed, a_pow2):
    cfg, ck = _tiny("w4a8_nvfp4", seed=seed)
    rng = np.random.default_rng(seed + 1)
    if a_pow2 is not None:
        ck.a13 = (2.0 ** rng.integers(-a_pow2, a_pow2 + 1, size=ck.E)).astype(np.float32)
        ck.a2 = (2.0 ** rng.integers(-a_pow2, a_pow2 + 1, size=ck.E)).astype(np.float32)
    M, k = 6, 3
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    w = S.router_weights(rng, M, k, "softmax", 1.0)
    return ck, x, ids, w


def test_nvfp4_a8_power_of_two_gscales_drop_out():
    """MX scales are powers of two, so an activation global scale 2^k shifts every block scale
    by k and leaves the codes alone: the layer with power-of-two global scales equals the layer
    with global scales 1 exactly; a general global scale moves the MX grid and changes it."""
    ck, x, ids, w = _nv_a8_case(31, 6)
    _, f = O.moe_forward(ck, x, ids, w, return_f64=True)
    ck.a13 = np.ones(ck.E, np.float32)
    ck.a2 = np.ones(ck.E, np.float32)
    _, f1 = O.moe_forward(ck, x, ids, w, return_f64=True)
    assert np.array_equal(f, f1)
    ck.a13 = np.full(ck.E, 1.37, np.float32)
    _, f2 = O.moe_forward(ck, x, ids, w, return_f64=True)
    assert not np.array_equal(f, f2)


def test_nvfp4_a8_equals_w4a8_on_shared_values():
    """NVFP4 weights whose two E4M3 scales of each group of 32 are the same power of two
    (2^-9..2^8) and whose global scales are 1 are MXFP4 weights: with MXFP8 activations and
    unit activation global scales, the layer must equal the W4A8 (MXFP4 x MXFP8) layer exactly,
    pinning the mode to the W4A8 oracle."""
    ck, x, ids, w = _nv_a8_case(41, None)
    rng = np.random.default_rng(42)
    ck.a13 = np.ones(ck.E, np.float32)
    ck.a2 = np.ones(ck.E, np.float32)
    ck.g13 = np.ones(ck.E, np.float32)
    ck.g2 = np.ones(ck.E, np.float32)
    mx = S.Checkpoint(quant="mxfp4", E=ck.E, H=ck.H, I=ck.I, layout=ck.layout, w13=ck.w13,
                      w2=ck.w2)
    to_e4m3 = np.vectorize(lambda b: _e4m3_code_of_pow2(int(b) - 127), otypes=[np.uint8])
    for name, k in (("s13", ck.H // 32), ("s2", ck.I // 32)):
        e8 = rng.integers(118, 136, size=(ck.E, getattr(ck, name).shape[1], k), dtype=np.uint8)
        setattr(mx, name, e8)
        setattr(ck, name, np.repeat(to_e4m3(e8), 2, axis=-1))
    a, fa = O.moe_forward(ck, x, ids, w, return_f64=True)
    b, fb = O.moe_forward(mx, x, ids, w, return_f64=True)
    assert np.array_equal(fa, fb) and np.array_equal(a, b)


def test_w4a4_power_of_two_gscales_drop_out():
    """NVFP4 activations: scaling a block by 2^k moves vmax / 6 by 2^k, and while that stays in
    E4M3's normal range the scale code shifts by k exponent steps with the same E2M1 codes, so
    global scales that differ by powers of two give the same layer exactly."""
    cfg, ck = _tiny("w4a4_nvfp4", seed=51)
    rng = np.random.default_rng(52)
    M, k = 5, 2
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    w = S.router_weights(rng, M, k, "softmax", 1.0)
    # base scales that put a * x and a * h well inside E4M3's normal range (vmax / 6 >= 2^-6)
    h = O.slot_intermediate(ck, x, ids, math.inf)
    ck.a13 = np.full(ck.E, 64.0, np.float32)
    ck.a2 = np.full(ck.E, np.float32(2.0 ** np.ceil(np.log2(64.0 / np.abs(h).max()))))
    _, f0 = O.moe_forward(ck, x, ids, w, return_f64=True)
    ck.a13 = ck.a13 * (2.0 ** rng.integers(-2, 3, size=ck.E)).astype(np.float32)
    ck.a2 = ck.a2 * (2.0 ** rng.integers(-2, 3, size=ck.E)).astype(np.float32)
    _, f1 = O.moe_forward(ck, x, ids, w, return_f64=True)
    assert np.array_equal(f0, f1)
    ck.a13 = ck.a13 * np.float32(1.3)
    _, f2 = O.moe_forward(ck, x, ids, w, return_f64=True)
    assert not np.array_equal(f0, f2)


def _e4m3_code_of_pow2(j):
    """E4M3 (bias 7) code of 2^j, j in [-9, 8]: normal exponent field from 2^-6, subnormal
    mantissa below (value m * 2^-9)."""
    assert -9 <= j <= 8
    return (j + 7) << 3 if j >= -6 else 1 << (j + 9)


def test_mxfp4_kept_tier_equals_nvfp4_on_shared_values():
    """Hybrid layer with an MXFP4 kept tier (E2M1 x 2^(b-127) per 32) whose scales 2^-9..2^8
    are also E4M3 values: rewritten as an NVFP4 kept tier (the same E2M1 codes, each E8M0 scale
    as the E4M3 code of the same power of two for both groups of 16, global 1), the layer must
    give the identical fp64 result: the MXFP4 dequantisation is pinned to the NVFP4 one."""
    cfg, ck = _tiny("hybrid_mx", seed=3)
    rng = np.random.default_rng(12)
    for name in ("s13", "s2"):
        setattr(ck.nv, name, rng.integers(118, 136, size=getattr(ck.nv, name).shape,
                                          dtype=np.uint8))
    nv = S.Checkpoint(quant="nvfp4", E=ck.nv.E, H=ck.H, I=ck.I, layout=ck.layout,
                      w13=ck.nv.w13, w2=ck.nv.w2,
                      g13=np.ones(ck.nv.E, np.float32), g2=np.ones(ck.nv.E, np.float32))
    to_e4m3 = np.vectorize(lambda b: _e4m3_code_of_pow2(int(b) - 127), otypes=[np.uint8])
    nv.s13 = np.repeat(to_e4m3(ck.nv.s13), 2, axis=-1)
    nv.s2 = np.repeat(to_e4m3(ck.nv.s2), 2, axis=-1)
    ck_nv = S.Checkpoint(quant="hybrid", E=ck.E, H=ck.H, I=ck.I, layout=ck.layout, tier=ck.tier,
                         nv=nv, nf=ck.nf)
    M, k = 6, 3
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    w = S.router_weights(rng, M, k, "softmax", 1.0)
    a, fa = O.moe_forward(ck, x, ids, w, return_f64=True)
    b, fb = O.moe_forward(ck_nv, x, ids, w, return_f64=True)
    assert (ck.tier[ids] == S.TIER_NVFP4).any()
    assert np.array_equal(fa, fb) and np.array_equal(a, b)


def test_forward_full_tiny_config_bruteforce():
    cfg = S.CONFIGS["tiny_w4a8"]
    ck = S.make_checkpoint(cfg)
    x, ids, w = S.make_inputs(cfg, 4)
    a = O.moe_forward(ck, x, ids, w, cfg.swiglu_limit)
    b = O.moe_forward_bruteforce(ck, x, ids, w, cfg.swiglu_limit)
    da, db = C.bf16_bits_to_f64(a), C.bf16_bits_to_f64(b)
    assert np.mean(da == db) > 0.999 and np.allclose(da, db, rtol=2 ** -7, atol=0)


def test_forward_closed_form_identity_layer():
    """W13 up row i = one-hot at column i, gate row i = one-hot at column I+i (E2M1 1.0, scale
    1.0); W2 row r = one-hot at column r mod I.  Then up = x^[i], gate = x^[I+i],
    y[r] = q(h)[r mod I] and out = w * y, independent of everything else."""
    E, H, I = 2, 64, 32
    ck = S.Checkpoint(quant="mxfp4", E=E, H=H, I=I, layout=S.W13_UP_GATE)
    w13 = np.zeros((E, 2 * I, H), dtype=np.uint8)
    for i in range(I):
        w13[:, i, i] = 0x2                 # +1.0
        w13[:, I + i, I + i] = 0x2
    w13[1] = np.where(w13[1] == 0x2, 0x4, 0)   # expert 1: 2.0 everywhere instead
    ck.w13 = C.pack_fp4(w13)
    ck.s13 = np.full((E, 2 * I, H // 32), 127, dtype=np.uint8)
    w2 = np.zeros((E, H, I), dtype=np.uint8)
    for r in range(H):
        w2[:, r, r % I] = 0x2
    ck.w2 = C.pack_fp4(w2)
    ck.s2 = np.full((E, H, I // 32), 127, dtype=np.uint8)
    rng = np.random.default_rng(3)
    x = S.make_x(rng, 3, H)
    ids = np.array([[0], [1], [-1]], dtype=np.int32)
    w = np.array([[0.75], [1.5], [9.0]], dtype=np.float32)
    L = 7.0
    _, f64 = O.moe_forward(ck, x, ids, w, L, return_f64=True)
    xv = C.bf16_bits_to_f64(x)
    for t, scale in ((0, 1.0), (1, 2.0)):
        q, s = C.mxfp8_quantize(xv[t][None, :])
        xh = C.mxfp8_dequantize(q, s)[0]
        up, gate = scale * xh[:I], scale * xh[I:]
        h = [min(gg, L) / (1 + math.exp(-min(gg, L))) * max(-L, min(uu, L)) for gg, uu in zip(gate, up)]
        hq, hs = C.mxfp8_quantize(np.array(h)[None, :])
        hh = C.mxfp8_dequantize(hq, hs)[0]
        want = float(w[t, 0]) * np.array([hh[r % I] for r in range(H)])
        assert np.array_equal(f64[t], want)
    assert np.all(f64[2] == 0.0)


def _small_case(seed=21, quant="mxfp4"):
    cfg, ck = _tiny(quant, seed=seed, E=8, H=128, I=64)
    rng = np.random.default_rng(seed)
    M, k = 7, 3
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    w = S.router_weights(rng, M, k, "sigmoid_norm", 2.5)
    return ck, x, ids, w


@pytest.mark.parametrize("quant", ["mxfp4", "nvfp4", "hybrid"])
def test_linear_in_router_weights(quant):
    ck, x, ids, w = _small_case(quant=quant)
    _, f1 = O.moe_forward(ck, x, ids, w, 7.0, return_f64=True)
    _, f2 = O.moe_forward(ck, x, ids, 3.0 * w.astype(np.float64), 7.0, return_f64=True)
    assert np.allclose(f2, 3.0 * f1, rtol=1e-13, atol=1e-300)
    w_a = w.copy()
    w_a[:, 1:] = 0
    w_b = w - w_a
    _, fa = O.moe_forward(ck, x, ids, w_a, 7.0, return_f64=True)
    _, fb = O.moe_forward(ck, x, ids, w_b, 7.0, return_f64=True)
    assert np.allclose(fa + fb, f1, rtol=1e-12, atol=1e-12 * np.abs(f1).max())


def test_padding_and_invalid_ids():
    ck, x, ids, w = _small_case()
    ids2 = ids.copy()
    ids2[5:, :] = -1                 # padding rows
    ids2[0, 2] = ck.E                # out of range id
    ids2[1, 0] = -7
    out = O.moe_forward(ck, x, ids2, w, 7.0)
    assert np.all(out[5:] == 0)
    # a dropped slot contributes exactly what weight 0 on a valid id contributes
    ids3 = ids2.copy()
    w3 = w.copy()
    ids3[0, 2], w3[0, 2] = 0, 0.0
    ids3[1, 0], w3[1, 0] = 1, 0.0
    ids3[5:, :], w3[5:, :] = 2, 0.0
    _, fa = O.moe_forward(ck, x, ids2, w, 7.0, return_f64=True)
    _, fb = O.moe_forward(ck, x, ids3, w3, 7.0, return_f64=True)
    assert np.array_equal(fa, fb)


def test_token_order_invariance():
    ck, x, ids, w = _small_case()
    p = np.array([3, 0, 6, 1, 5, 2, 4])
    a = O.moe_forward(ck, x, ids, w, 7.0)
    b = O.moe_forward(ck, x[p], ids[p], w[p], 7.0)
    assert np.array_equal(a[p], b)


def test_swapped_w13_halves_detected():
    cfg = S.CONFIGS["tiny_w4a8"]
    ck = S.make_checkpoint(cfg)
    x, ids, w = S.make_inputs(cfg, 4)
    a, fa = O.moe_forward(ck, x, ids, w, 7.0, return_f64=True)
    ck.layout = S.W13_GATE_UP
    b = O.moe_forward(ck, x, ids, w, 7.0)
    rel, _ = O.row_errors(b, fa)
    assert np.all(rel > 0.2)          # far outside the 5e-3 bound


def test_zero_expert_contributes_nothing():
    ck, x, ids, w = _small_case()
    e = int(ids[0, 0])
    ck.w13 = ck.w13.copy()
    ck.w13[e] = 0
    _, fa = O.moe_forward(ck, x, ids, w, 7.0, return_f64=True)
    w0 = np.where(ids == e, 0.0, w)
    _, fb = O.moe_forward(ck, x, ids, w0, 7.0, return_f64=True)
    assert np.array_equal(fa, fb)


def test_row_subset_matches_full():
    ck, x, ids, w = _small_case()
    full = O.moe_forward(ck, x, ids, w, 7.0)
    sub = O.moe_forward(ck, x, ids, w, 7.0, rows=[1, 4])
    assert np.array_equal(sub[[1, 4]], full[[1, 4]])


def test_row_errors_bound_helper():
    ref = np.array([[1.0, 2.0, 3.0], [0.0, 0.0, 0.0]])
    got = C.f64_to_bf16_bits(ref)
    rel, mx = O.row_errors(got, ref)
    assert rel.tolist() == [0.0, 0.0] and mx.tolist() == [0.0, 0.0]
    bad = C.f64_to_bf16_bits(ref + np.array([[0.0, 0.0, 0.5], [0.0, 1.0, 0.0]]))
    rel, mx = O.row_errors(bad, ref)
    assert rel[0] > 0.1 and np.isinf(rel[1])
    # an outlier row: 1001.75 rounds to 1000 (bf16 spacing 4 there); its rounding error 1.75
    # alone is above 2e-2 of the row's rms, yet the correctly rounded output has no error beyond
    # its own rounding
    row = np.array([[1001.75] + [1.0] * 255])
    rms = np.sqrt((row ** 2).mean())
    rel, mx = O.row_errors(C.f64_to_bf16_bits(row), row)
    assert mx[0] == 0.0 and 0 < rel[0] < 2e-3 and 1.75 / rms > 0.02
    # the other neighbour (1004): the error 2.25 exceeds the half step 2 by 0.25
    off = C.f64_to_bf16_bits(row).copy()
    off[0, 0] = C.f64_to_bf16_bits(np.array([1004.0]))[0]
    _, mx = O.row_errors(off, row)
    assert mx[0] == 0.25 / rms
    # below the binade of 1.0 the half step is 2^-9: 0.5 + 2^-8 (one step up) is 2^-9 beyond
    small = np.array([[0.5, 0.5]])
    up = C.f64_to_bf16_bits(np.array([[0.5 + 2 ** -8, 0.5]]))
    _, mx = O.row_errors(up, small)
    assert mx[0] == 2 ** -9 / 0.5


def test_synth_recipes():
    cfg = S.CONFIGS["decode_w4a8"]
    ids, w = S.make_routing(cfg, 16)
    assert ids.shape == (16, 6) and np.all(ids[12:] == -1) and np.all(ids[:12] >= 0)
    assert np.allclose(w.sum(1), 2.5, rtol=1e-6)
    assert all(len(set(r)) == 6 for r in ids[:12].tolist())
    cfg = S.CONFIGS["prefill_w4a8_ep_i1152"]
    ids, w = S.make_routing(cfg, 128)
    assert ids.min() >= 0 and ids.max() < 192
    cfg = S.CONFIGS["hybrid_nvfp4_nf3"]
    ck = S.make_checkpoint(cfg, E=16, H=64, I=32)
    assert (ck.tier == S.TIER_NVFP4).sum() == 16 or ck.nv.E + ck.nf.E == 16


def test_slot_intermediate_matches_direct_dot_products():
    ck, x, ids, w = _small_case()
    h = O.slot_intermediate(ck, x, ids, 7.0)
    _, _, perm, _ = O.route(ids, ck.E)
    xq, xs = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
    xhat = C.mxfp8_dequantize(xq, xs)
    k = ids.shape[1]
    for p in (0, 5, len(perm) - 1):
        t, j = divmod(int(perm[p]), k)
        e = int(ids[t, j])
        codes = C.unpack_fp4(ck.w13[e])
        scale = np.repeat(C.e8m0_value(ck.s13[e]), 32, axis=1)
        rows = C.E2M1_TABLE[codes] * scale
        up = sum(rows[i] @ xhat[t] for i in [0])          # row 0 of the up half
        gate = rows[ck.I] @ xhat[t]                         # row 0 of the gate half
        g = min(gate, 7.0)
        u = max(-7.0, min(up, 7.0))
        assert h[p, 0] == pytest.approx(g / (1 + math.exp(-g)) * u, rel=1e-12, abs=1e-12)


# ---------------------------------------------------------------------------- acceptance helpers

def _other_neighbour(v, grid):
    """The two entries of the sorted non-negative grid that bracket |v| (lo <= |v| < hi)."""
    a = abs(v)
    lo = max(g for g in grid if g <= a)
    hi = min(g for g in grid if g > a)
    return lo, hi


def _flip_case(quant, woi, seed):
    """A tiny layer, one slot (t, j) and the intermediate element i of that slot whose exact
    value lies closest (relative to its size) to a rounding midpoint of the fc2 operand's
    format, with that element's other rounding worked out here from the format's grid: the
    E4M3 values (MXFP8 under the block's scale byte), the two bf16 bit patterns around the
    value, or the E2M1 values (NVFP4 under the block's E4M3 scale); with an activation global
    scale a2 the decision is taken on a2 * h and the operand is the value / a2."""
    cfg, ck = _tiny(quant, seed=seed)
    rng = np.random.default_rng(100 + seed)
    M, k = 3, 2
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    w = S.router_weights(rng, M, k, "sigmoid_norm", 2.5)
    lim = 7.0 if quant == "mxfp4" else math.inf
    t, j = 1, 1
    _, _, perm, slot_of = O.route(ids, ck.E)
    h = O.slot_intermediate(ck, x, ids, lim, topk_w=w, weight_on_input=woi)[slot_of[t * k + j]]
    e = int(ids[t, j])
    a2 = None if O.act_gscale(ck, "a2") is None else float(np.float32(O.act_gscale(ck, "a2")[e]))
    best = None
    for i in range(ck.I):
        if quant in ("mxfp4", "w4a8_nvfp4"):
            v = h * (1.0 if a2 is None else a2)
            q, s = C.mxfp8_quantize(v[None, :])
            sc = 2.0 ** (int(s[0, i // 32]) - 127)
            grid = sorted(set(C.E4M3_TABLE[:127].tolist()))
            near = C.mxfp8_dequantize(q, s)[0, i]
            val = v[i] / sc
        elif quant == "w4a4_nvfp4":
            v = (np.float32(a2) * h.astype(np.float32)).astype(np.float32)
            q, s = C.nvfp4_quantize(v[None, :])
            sc = float(C.E4M3_TABLE[s[0, i // 16]])
            grid = C.E2M1_TABLE[:8].tolist()
            near = C.nvfp4_dequantize(q, s)[0, i]
            val = float(v[i]) / sc
        else:
            bits = int(C.f64_to_bf16_bits(np.array([h[i]]))[0])
            cand = sorted(abs(float(C.bf16_bits_to_f64(np.array([b], np.uint16))[0]))
                          for b in (bits - 1, bits, bits + 1))
            sc, grid, near, val = 1.0, cand, float(C.bf16_round(h[i])), h[i]
        if val == 0 or abs(val) >= max(grid):
            continue
        lo, hi = _other_neighbour(val, grid)
        dist = abs(abs(val) - (lo + hi) / 2) / abs(val)
        other = hi if abs(near) == lo * sc else lo
        alt = math.copysign(other * sc, val) / (1.0 if a2 is None else a2)
        if best is None or dist < best[0]:
            best = (dist, i, alt)
    return ck, x, ids, w, lim, t, j, best


@pytest.mark.parametrize("quant,woi", [("mxfp4", False), ("nvfp4", False), ("nvfp4", True),
                                       ("w4a8_nvfp4", False), ("w4a4_nvfp4", False)])
def test_requant_alternatives_pinned_by_flipping(quant, woi):
    """oracle.moe.requant_alternatives against a forward recomputed with one decision flipped:
    the element-by-element brute force is run on the slot's fc2 operand with element i replaced
    by its other rounding (found above from the format's grid), and the change of the token's
    unrounded output must be one of the vectors the helper lists for that row - so a wrong sign,
    a missing router weight or a wrong column of W2 in the helper fails here."""
    ck, x, ids, w, lim, t, j, best = _flip_case(quant, woi, seed=3)
    dist, i, alt = best
    rel = max(1.5 * dist, 1e-9)
    alts = O.requant_alternatives(ck, x, ids, w, lim, rel=rel, rows=[t], weight_on_input=woi)[t]
    _, base = O.moe_forward_bruteforce(ck, x, ids, w, lim, weight_on_input=woi, return_f64=True)
    _, flip = O.moe_forward_bruteforce(ck, x, ids, w, lim, weight_on_input=woi,
                                       fc2_override={(t, j): {i: alt}}, return_f64=True)
    want = flip[t] - base[t]
    assert np.abs(want).max() > 0
    tol = 1e-12 * np.abs(base[t]).max()
    assert any(np.allclose(d, want, rtol=0, atol=tol) for d in alts), (quant, i, len(alts))
    # the other rows are untouched by a flip in row t's slot
    others = [r for r in range(ids.shape[0]) if r != t]
    assert np.array_equal(flip[others], base[others])


def test_nvfp4_alternates_worked_midpoints():
    """E2M1 midpoints under a chosen block scale: a block whose largest magnitude is 3 takes the
    E4M3 scale 0.5 (3 / 6), and each value 0.5 * m for a midpoint m of the E2M1 grid, nudged by
    one part in 10^5 above or below, has the grid value on that side as its nearest rounding and
    the one on the other side as its alternate; exact midpoints round to the even code."""
    mids = [(0.25, 0.0, 0.5), (0.75, 0.5, 1.0), (1.25, 1.0, 1.5), (1.75, 1.5, 2.0),
            (2.5, 2.0, 3.0), (3.5, 3.0, 4.0), (5.0, 4.0, 6.0)]
    for m, lo, hi in mids:
        for sign in (1.0, -1.0):
            v = np.zeros((1, 16))
            v[0, 0] = 3.0                                  # block maximum: scale 0.5
            v[0, 1] = sign * 0.5 * m * (1 + 1e-5)          # above the midpoint: nearest hi
            v[0, 2] = sign * 0.5 * m * (1 - 1e-5)          # below: nearest lo
            v[0, 3] = sign * 0.5 * (lo + (hi - lo) * 0.1)  # far from the midpoint
            mask, alt = C.nvfp4_alternates(v, 1e-4)
            q, s = C.nvfp4_quantize(v.astype(np.float32))
            assert s.tolist() == [[0x30]]                  # E4M3 0.5
            near = C.nvfp4_dequantize(q, s)[0]
            assert near[1] == sign * 0.5 * hi and near[2] == sign * 0.5 * lo, m
            assert mask[0].tolist()[:4] == [False, True, True, False], m
            assert alt[0, 1] == sign * 0.5 * lo and alt[0, 2] == sign * 0.5 * hi, m
            assert alt[0, 3] == near[3]
    # exact midpoints: ties to the even code (mantissa bit 0): 0.25 -> 0, 0.75 -> 1, 1.25 -> 1,
    # 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; the alternate is the odd neighbour
    v = np.zeros((1, 16))
    v[0, 0] = 3.0
    v[0, 1:8] = [0.5 * m for m, _, _ in mids]
    mask, alt = C.nvfp4_alternates(v, 1e-4)
    q, s = C.nvfp4_quantize(v.astype(np.float32))
    assert (C.nvfp4_dequantize(q, s)[0, 1:8] / 0.5).tolist() == [0, 1, 1, 2, 2, 4, 4]
    assert mask[0, 1:8].all()
    assert (alt[0, 1:8] / 0.5).tolist() == [0.5, 0.5, 1.5, 1.5, 3, 3, 6]


def test_tier_local_index_hand_map():
    """The hybrid layer's compact storage: each tier lists its experts in ascending id."""
    got = O.tier_local_index(np.array([3, 4, 3, 4, 4], np.int8))
    assert got == {0: (3, 0), 1: (4, 0), 2: (3, 1), 3: (4, 1), 4: (4, 2)}
    assert O.tier_local_index(np.array([4, 4, 4], np.int8)) == {0: (4, 0), 1: (4, 1), 2: (4, 2)}
    assert O.tier_local_index(np.array([3], np.int8)) == {0: (3, 0)}


def test_hybrid_expert_weights_hand_checkpoint():
    """A hybrid checkpoint written by hand, every expert's weights one constant: the kept tier
    (NVFP4, codes 0x22 = E2M1 1.0 in both nibbles) has E4M3 scales 1, 2, 3 for its experts 0, 1,
    2 and globals 1; the NF3 tier (codes all 7 = LUT 1.0, bytes 0xFF) has scales 4 and 8.  With
    tiers [3, 4, 3, 4, 4] the experts' values are 4, 1, 8, 2, 3 - in W13 and W2 alike - and the
    brute-force forward of one token through expert 2 alone is the closed form 8 * 8 * sum(x)."""
    E, H, I = 5, 32, 32
    tier = np.array([3, 4, 3, 4, 4], np.int8)
    nv = S.Checkpoint(quant="nvfp4", E=3, H=H, I=I)
    nv.w13 = np.full((3, 2 * I, H // 2), 0x22, np.uint8)
    nv.w2 = np.full((3, H, I // 2), 0x22, np.uint8)
    sc = np.array([0x38, 0x40, 0x44], np.uint8)        # E4M3 1.0, 2.0, 3.0
    nv.s13 = np.repeat(sc, 2 * I * H // 16).reshape(3, 2 * I, H // 16)
    nv.s2 = np.repeat(sc, H * I // 16).reshape(3, H, I // 16)
    nv.g13 = np.ones(3, np.float32)
    nv.g2 = np.ones(3, np.float32)
    nf = S.Checkpoint(quant="nf3", E=2, H=H, I=I)
    nf.w13 = np.full((2, 2 * I, 3 * H // 8), 0xFF, np.uint8)
    nf.w2 = np.full((2, H, 3 * I // 8), 0xFF, np.uint8)
    sf = np.array([0x48, 0x50], np.uint8)              # E4M3 4.0, 8.0
    nf.s13 = np.repeat(sf, 2 * I * H // 32).reshape(2, 2 * I, H // 32)
    nf.s2 = np.repeat(sf, H * I // 32).reshape(2, H, I // 32)
    ck = S.Checkpoint(quant="hybrid", E=E, H=H, I=I, tier=tier, nv=nv, nf=nf)
    for e, want in enumerate([4.0, 1.0, 8.0, 2.0, 3.0]):
        W13, W2, _ = O.expert_weights(ck, e)
        assert np.all(W13 == want) and np.all(W2 == want), e
    # one token through expert 2 (value 8): gate = up = 8 * sum(x), h = silu(g) * u rounded to
    # bf16, out = 8 * I * bf16(h) per output element (bf16 activations, no clamp)
    x = S.f32_to_bf16_bits(np.full((1, H), 0.0625, np.float32))
    ids = np.array([[2]], np.int32)
    w = np.ones((1, 1), np.float32)
    g = 8.0 * H * 0.0625
    h = float(C.bf16_round(g / (1 + math.exp(-g)) * g))
    _, f64 = O.moe_forward_bruteforce(ck, x, ids, w, return_f64=True)
    assert np.allclose(f64[0], 8.0 * I * h, rtol=1e-14, atol=0)


def test_ep_mask_foreign_hand_worked():
    """The EP slice's input recipe on a hand-worked batch: rank owning global experts 4..7.
    Row 0 owns global 5 (local 1): its foreign slot takes local 1.  Row 1 owns nothing: its
    slots take the batch's smallest owned local id (1).  Row 2 owns 7 and 6 (locals 3, 2).
    Weights of non-owned slots become 0."""
    ids = np.array([[5, 1], [9, -1], [7, 6]], np.int32)
    w = np.array([[0.5, 0.25], [0.75, 1.0], [0.125, 2.0]], np.float32)
    got_ids, got_w = S.ep_mask_foreign(ids, w, 4, 4)
    assert got_ids.tolist() == [[1, 1], [1, 1], [3, 2]]
    assert got_w.tolist() == [[0.5, 0.0], [0.0, 0.0], [0.125, 2.0]]
    # a batch that owns nothing: every slot id 0, weight 0
    got_ids, got_w = S.ep_mask_foreign(np.array([[0, 9]], np.int32), np.ones((1, 2), np.float32),
                                       4, 4)
    assert got_ids.tolist() == [[0, 0]] and got_w.tolist() == [[0.0, 0.0]]
    # the row's own smallest owned id wins over the batch's
    got_ids, _ = S.ep_mask_foreign(np.array([[4, 0], [7, 2]], np.int32),
                                   np.ones((2, 2), np.float32), 4, 4)
    assert got_ids.tolist() == [[0, 0], [3, 3]]


# ---------------------------------------------------------------------------- kept-tier A8

def _a8_case(seed=4):
    cfg, ck = _tiny("hybrid_mx", seed=seed)
    rng = np.random.default_rng(200 + seed)
    M, k = 6, 2
    x = S.make_x(rng, M, ck.H)
    ids = S.uniform_topk(rng, M, ck.E, k)
    w = S.router_weights(rng, M, k, "softmax", 1.0)
    return ck, x, ids, w


def test_kept_a8_forward_matches_bruteforce():
    """The A8 opt-in of the MXFP4 kept tier: the dgemm forward against the element loop, whose
    static FP8 rounding is its own exhaustive search (not codecs.fp8_static_quantize)."""
    ck, x, ids, w = _a8_case()
    tier = np.asarray(ck.tier)
    assert (tier[ids] == S.TIER_NVFP4).any() and (tier[ids] == S.TIER_NF3).any()
    a, f64 = O.moe_forward(ck, x, ids, w, return_f64=True, kept_a8=True)
    b, g64 = O.moe_forward_bruteforce(ck, x, ids, w, kept_a8=True, return_f64=True)
    assert np.allclose(f64, g64, rtol=1e-12, atol=1e-12 * np.abs(f64).max())
    # the opt-in changes the result (x and h go through FP8 for the kept experts)
    a16 = O.moe_forward(ck, x, ids, w, return_f64=True)[1]
    kept_rows = (tier[ids] == S.TIER_NVFP4).any(axis=1)
    assert not np.allclose(a16[kept_rows], f64[kept_rows], rtol=1e-6, atol=0)


def test_kept_a8_leaves_nf3_rows_and_matches_its_definition():
    """Rows routed only to NF3 experts are the A16 result exactly; for a kept expert the
    slot's output is W2 . fp8s(SwiGLU(W13 . fp8s(x, s13)), s2) with the weights dequantised by
    oracle.moe.expert_weights and fp8s the static quantiser - checked on one slot directly."""
    ck, x, ids, w = _a8_case(seed=6)
    tier = np.asarray(ck.tier)
    ids[0] = np.nonzero(tier == S.TIER_NF3)[0][:2]          # a row on NF3 experts only
    ids[1, 0] = np.nonzero(tier == S.TIER_NVFP4)[0][0]       # and one with a kept expert
    f8 = O.moe_forward(ck, x, ids, w, return_f64=True, kept_a8=True)[1]
    f16 = O.moe_forward(ck, x, ids, w, return_f64=True)[1]
    nf_rows = (tier[ids] == S.TIER_NF3).all(axis=1)
    assert nf_rows.any()
    assert np.array_equal(f8[nf_rows], f16[nf_rows])
    t, j = [(t, j) for t in range(ids.shape[0]) for j in range(ids.shape[1])
            if tier[ids[t, j]] == S.TIER_NVFP4][0]
    e = int(ids[t, j])
    W13, W2, _ = O.expert_weights(ck, e)
    xq = C.fp8_static_quantize(C.bf16_bits_to_f64(x[t]), ck.in13)[1]
    gate, up = O.split_w13(W13 @ xq, ck.I, ck.layout)
    y = W2 @ C.fp8_static_quantize(O.swiglu(gate, up), ck.in2)[1]
    one = np.zeros_like(ids)
    one[:] = -1
    one[t, j] = e
    single = O.moe_forward(ck, x, one, w, return_f64=True, kept_a8=True)[1][t]
    assert np.allclose(single, w[t, j] * y, rtol=1e-13, atol=1e-13 * np.abs(y).max())


def test_kept_a8_requant_alternatives_pinned_by_flipping():
    """requant_alternatives with the A8 opt-in: for a kept-tier slot, the intermediate element
    nearest (relative to its size) a static-FP8 midpoint is taken the other way in the element
    loop (its other E4M3 neighbour times s2, from the E4M3 grid), and the token's output change
    must be one of the vectors the helper lists."""
    ck, x, ids, w = _a8_case(seed=4)
    tier = np.asarray(ck.tier)
    k = ids.shape[1]
    t, j = [(t, j) for t in range(ids.shape[0]) for j in range(k)
            if tier[ids[t, j]] == S.TIER_NVFP4][0]
    _, _, perm, slot_of = O.route(ids, ck.E)
    h = O.slot_intermediate(ck, x, ids, kept_a8=True)[slot_of[t * k + j]]
    s2 = float(np.float32(ck.in2))
    grid = sorted(set(C.E4M3_TABLE[:127].tolist()))
    best = None
    for i in range(ck.I):
        a = abs(h[i]) / s2
        if a == 0 or a >= 448:
            continue
        lo, hi = _other_neighbour(a, grid)
        dist = abs(a - (lo + hi) / 2) / a
        near = float(C.fp8_static_quantize(np.array([h[i]]), ck.in2)[1][0])
        other = hi if abs(near) == lo * s2 else lo
        if best is None or dist < best[0]:
            best = (dist, i, math.copysign(other * s2, h[i]))
    dist, i, alt = best
    alts = O.requant_alternatives(ck, x, ids, w, rel=max(1.5 * dist, 1e-9), rows=[t],
                                  kept_a8=True)[t]
    _, base = O.moe_forward_bruteforce(ck, x, ids, w, kept_a8=True, return_f64=True)
    _, flip = O.moe_forward_bruteforce(ck, x, ids, w, kept_a8=True,
                                       fc2_override={(t, j): {i: alt}}, return_f64=True)
    want = flip[t] - base[t]
    assert np.abs(want).max() > 0
    tol = 1e-12 * np.abs(base[t]).max()
    assert any(np.allclose(d, want, rtol=0, atol=tol) for d in alts), (i, len(alts))
