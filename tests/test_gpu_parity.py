"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the same seeded inputs.

Bars: routing tables and MXFP8 activation codes / scales bit-exact; outputs per row within
rel-L2 <= 5e-3 and max|err| <= 2e-2 * rms(row) of the oracle evaluated on the same quantised
operands; deterministic mode bit-stable run to run and per token under token permutation."""
import math

import numpy as np
import pytest

from oracle import codecs as C
from oracle import moe as O
from synth import moe_inputs as S
from moe_cases import (H_CANCEL_ATOL, check_rows, oracle_rows, run_layer, small_cfg,
                        to_device, out_bits)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_route_count_gb300 import build
    build.build()


def _layer(ck, topk, max_m, limit, det, **kw):
    from serving_route_count_gb300 import MoELayer
    kw.setdefault("debug_copies", True)      # the tests read the quantised activations back
    return MoELayer(ck, topk, max_m, limit, det, **kw)


# ---------------------------------------------------------------------------- tiny config

@pytest.mark.parametrize("det", [0, 1])
def test_tiny_w4a8_all_rows(det):
    cfg = S.CONFIGS["tiny_w4a8"]
    ck = S.make_checkpoint(cfg)
    x, ids, w = S.make_inputs(cfg, 4)
    layer = _layer(ck, cfg.topk, 4, cfg.swiglu_limit, det)
    got = run_layer(layer, x, ids, w)
    check_rows(got, ck, x, ids, w, cfg.swiglu_limit)
    st, code = layer.device_error()
    assert st == 0 and code == 0


def test_tiny_routing_and_actq_bit_exact():
    cfg = S.CONFIGS["tiny_w4a8"]
    ck = S.make_checkpoint(cfg)
    x, ids, w = S.make_inputs(cfg, 4)
    layer = _layer(ck, cfg.topk, 4, cfg.swiglu_limit, 0)
    run_layer(layer, x, ids, w)
    torch.cuda.synchronize()
    route = O.route(ids, cfg.E)
    for a, b in zip(layer.routing(4), route):
        assert np.array_equal(a, b)
    xq, xs = layer.actq(4)
    q, s = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
    tok = route[2] // cfg.topk
    assert np.array_equal(xq, q[tok]) and np.array_equal(xs, s[tok])


# ---------------------------------------------------------------------------- small, ragged

@pytest.mark.parametrize("quant,det,backend", [("mxfp4", 0, 0), ("mxfp4", 1, 0), ("mxfp4", 0, 1),
                                               ("nvfp4", 0, 0), ("nvfp4", 1, 0), ("hybrid", 1, 0),
                                               ("hybrid", 0, 0)])
def test_small_ragged_all_rows(quant, det, backend):
    """E=16, H=1280 (one full and one partial 1024-wide K chunk), I=192 (fc2 K padded to 256),
    top-4, M=37 with padding rows and out-of-range ids: several tiles per expert and a tail."""
    cfg = small_cfg(quant)
    ck = S.make_checkpoint(cfg, seed=77, layout=S.W13_GATE_UP if det else S.W13_UP_GATE)
    rng = np.random.default_rng(78)
    M = 37
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 1.2)
    ids[-3:] = -1
    ids[2, 1] = cfg.E
    ids[5, 0] = -5
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    limit = 7.0 if quant == "mxfp4" else math.inf
    layer = _layer(ck, cfg.topk, 40, limit, det, backend=backend)
    got = run_layer(layer, x, ids, w)
    check_rows(got, ck, x, ids, w, limit)
    cnt, off, perm, slot_of = layer.routing(M)
    for a, b in zip((cnt, off, perm, slot_of), O.route(ids, cfg.E)):
        assert np.array_equal(a, b)
    if quant == "mxfp4":
        xq, xs = layer.actq(M)
        q, s = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
        tok = perm // cfg.topk
        assert np.array_equal(xq, q[tok]) and np.array_equal(xs, s[tok])


def test_swiglu_alpha_beta_and_no_clamp():
    cfg = small_cfg("mxfp4", E=8, H=256, I=128, topk=2)
    ck = S.make_checkpoint(cfg, seed=5)
    rng = np.random.default_rng(6)
    M = 9
    x = S.make_x(rng, M, cfg.H)
    ids = S.uniform_topk(rng, M, cfg.E, cfg.topk)
    w = S.router_weights(rng, M, cfg.topk, "softmax", 1.0)
    layer = _layer(ck, cfg.topk, M, 3.0, 0, alpha=1.702, beta=1.0)
    check_rows(run_layer(layer, x, ids, w), ck, x, ids, w, 3.0, alpha=1.702, beta=1.0)
    layer = _layer(ck, cfg.topk, M, math.inf, 1)
    check_rows(run_layer(layer, x, ids, w), ck, x, ids, w, math.inf)


# ---------------------------------------------------------------------------- invariants

def test_deterministic_bit_stable_and_permutation_invariant():
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=9)
    rng = np.random.default_rng(10)
    M = 33
    x = S.make_x(rng, M, cfg.H)
    ids = S.uniform_topk(rng, M, cfg.E, cfg.topk)
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 1.0)
    layer = _layer(ck, cfg.topk, M, 7.0, 1)
    a = run_layer(layer, x, ids, w)
    b = run_layer(layer, x, ids, w)
    assert np.array_equal(a, b)
    p = rng.permutation(M)
    c = run_layer(layer, x[p], ids[p], w[p])
    assert np.array_equal(a[p], c)


def test_edge_cases():
    from serving_route_count_gb300 import MoEError
    cfg = small_cfg("mxfp4", E=8, H=256, I=128, topk=2)
    ck = S.make_checkpoint(cfg, seed=3)
    rng = np.random.default_rng(4)
    layer = _layer(ck, 2, 8, 7.0, 1)
    # all ids invalid -> zero rows
    x = S.make_x(rng, 3, cfg.H)
    ids = np.array([[-1, 8], [-1, -1], [100, -7]], dtype=np.int32)
    w = np.ones((3, 2), np.float32)
    assert np.all(run_layer(layer, x, ids, w) == 0)
    # M = 1
    ids1 = np.array([[3, 5]], dtype=np.int32)
    got = run_layer(layer, x[:1], ids1, w[:1])
    check_rows(got, ck, x[:1], ids1, w[:1], 7.0)
    # capacity
    x9 = S.make_x(rng, 9, cfg.H)
    xt, it, wt = to_device(x9, np.zeros((9, 2), np.int32), np.ones((9, 2), np.float32))
    with pytest.raises(MoEError) as ei:
        layer(xt, it, wt)
    assert ei.value.status == 4
    # every expert hit by every token (max tile load), M = max_m
    ids8 = np.tile(np.array([[0, 1]], dtype=np.int32), (8, 1))
    x8 = S.make_x(rng, 8, cfg.H)
    got = run_layer(layer, x8, ids8, np.full((8, 2), 0.5, np.float32))
    check_rows(got, ck, x8, ids8, np.full((8, 2), 0.5, np.float32), 7.0)


def test_host_buffers_entry_point():
    cfg = S.CONFIGS["tiny_w4a8"]
    ck = S.make_checkpoint(cfg)
    x, ids, w = S.make_inputs(cfg, 4)
    layer = _layer(ck, cfg.topk, 4, cfg.swiglu_limit, 1)
    xh = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    ih = torch.from_numpy(ids).pin_memory()
    wh = torch.from_numpy(w).pin_memory()
    oh = torch.empty((4, cfg.H), dtype=torch.bfloat16).pin_memory()
    layer.run_host(xh, ih, wh, oh)
    got = oh.view(torch.int16).numpy().view(np.uint16)
    dev = run_layer(layer, x, ids, w)
    assert np.array_equal(got, dev)
    # the output written three ways: pinned (the kernel stores into it), pageable (staging
    # buffer and a copy), pinned but not 16-byte aligned (staging buffer and a copy)
    op = torch.empty((4, cfg.H), dtype=torch.bfloat16)
    layer.run_host(xh, ih, wh, op)
    assert np.array_equal(op.view(torch.int16).numpy().view(np.uint16), dev)
    raw = torch.zeros(4 * cfg.H + 4, dtype=torch.bfloat16).pin_memory()
    om = raw[4:].view(4, cfg.H)
    assert om.data_ptr() % 16 == 8
    layer.run_host(xh, ih, wh, om)
    assert np.array_equal(om.view(torch.int16).numpy().view(np.uint16), dev)
    assert not raw[:4].view(torch.int16).any()    # nothing written before the output rows


# ---------------------------------------------------------------------------- full sizes

@pytest.fixture(scope="module")
def decode_layer():
    cfg = S.CONFIGS["decode_w4a8"]
    ck = S.make_checkpoint(cfg)
    return cfg, ck


@pytest.mark.parametrize("det,fc1_kernel", [(0, 0), (1, 0), (0, 1), (1, 2)])
def test_decode_full_size_sampled(decode_layer, det, fc1_kernel):
    """E=384, H=7168, I=576, top-6 at M=16 (last 4 rows padding): routing bit-exact for the
    whole call, outputs of sampled rows against the oracle, padding rows exactly 0; with the
    automatic fc1 choice (stream-K here) and each fc1 kernel forced."""
    cfg, ck = decode_layer
    M = 16
    x, ids, w = S.make_inputs(cfg, M)
    layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, det, fc1_kernel=fc1_kernel)
    got = run_layer(layer, x, ids, w)
    route = O.route(ids, cfg.E)
    for a, b in zip(layer.routing(M), route):
        assert np.array_equal(a, b)
    xq, xs = layer.actq(M)
    q, s = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
    tok = route[2] // cfg.topk
    assert np.array_equal(xq, q[tok]) and np.array_equal(xs, s[tok])
    check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=[0, 7, 11, 12, 15])
    layer.close()


@pytest.mark.parametrize("cfg_name,M,det", [("prefill_w4a8", 1024, 1), ("prefill_w4a8", 2048, 0),
                                             ("prefill_w4a8_zipf", 4096, 1)])
def test_prefill_full_size_sampled(decode_layer, cfg_name, M, det):
    """E=384, H=7168, I=576, top-6 prefill calls (the decode layer's weights, the prefill
    routing recipe) at the three wide token-tile widths (32, 64 and 96 tokens at 16, 32 and 64
    expected slots per expert) with the persistent fc2: routing and activation codes
    bit-exact for the whole call, outputs of sampled rows against the oracle, and
    (deterministic mode) bit-identical repeats."""
    cfg, ck = decode_layer
    pcfg = S.CONFIGS[cfg_name]
    x, ids, w = S.make_inputs(pcfg, M)
    layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, det)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    route = O.route(ids, cfg.E)
    for a, b in zip(layer.routing(M), route):
        assert np.array_equal(a, b)
    xq, xs = layer.actq(M)
    q, s = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
    tok = route[2] // cfg.topk
    assert np.array_equal(xq, q[tok]) and np.array_equal(xs, s[tok])
    check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=[0, 1, M // 2, M - 1])
    if det:
        assert np.array_equal(run_layer(layer, x, ids, w), got)
    layer.close()


@pytest.mark.parametrize("M,det", [(16, 0), (512, 1)])
def test_prefill_ep_i1152_sampled(M, det):
    """The expert-parallel slice of the prefill config: E=192 local experts of 384, H=7168,
    I=1152 (nine full 128-row weight blocks per half), ids drawn over 384 experts with the
    foreign ones masked (weight 0, local id): routing bit-exact, sampled rows against the
    oracle."""
    cfg = S.CONFIGS["prefill_w4a8_ep_i1152"]
    ck = S.make_checkpoint(cfg)
    x, ids, w = S.make_inputs(cfg, M)
    layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, det)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    route = O.route(ids, cfg.E)
    for a, b in zip(layer.routing(M), route):
        assert np.array_equal(a, b)
    check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=[0, M // 3, M - 1])
    layer.close()


@pytest.mark.parametrize("quant,M,backend,fc1_kernel", [
    ("mxfp4", 5, 0, 0),       # one-launch routing + quantisation, fc1 tile list from the ids
    ("mxfp4", 16, 0, 2),      # stream-K fc1 with its own tile list from the ids
    ("mxfp4", 300, 0, 0),     # chunked routing over two 1024-slot chunks
    ("mxfp4", 40, 1, 0),      # CUDA-core backend: single-CTA routing kernel
    ("nvfp4", 8, 0, 0),       # one-launch routing + f16 conversion
    ("nvfp4", 100, 0, 0),     # single-CTA routing, then conversion
    ("w4a4_nvfp4", 20, 0, 0),  # NVFP4 activations: per-slot global scales of local experts
    ("w4a4_nvfp4", 90, 0, 0),
    ("w4a8_nvfp4", 20, 0, 0),
])
def test_expert_offset_on_device(quant, M, backend, fc1_kernel):
    """Expert parallelism on the device: a plan owning global experts [16, 32) of 48 takes
    global router ids (plus -1 padding).  Routing tables must equal the oracle's for the local
    ids with foreign ones dropped, and every row must match the oracle run on the adapter's
    own remap of the same inputs (foreign slots: weight 0, some local expert), which the
    dropped slots must reproduce."""
    cfg = small_cfg(quant)
    first, n_global = 16, 48
    ck = S.make_checkpoint(cfg, seed=3000 + M)
    rng = np.random.default_rng(4000 + M)
    x = S.make_x(rng, M, cfg.H)
    ids_g = S.zipf_topk(rng, M, n_global, cfg.topk, 0.6)
    ids_g[rng.random(ids_g.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, M, 7.0, 1, backend=backend, fc1_kernel=fc1_kernel,
                   first_expert=first)
    got = run_layer(layer, x, ids_g, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    lid = ids_g.astype(np.int64) - first
    local = np.where((lid >= 0) & (lid < cfg.E), lid, -1).astype(np.int32)
    assert (local >= 0).any() and (local < 0).any()
    for a, b in zip(layer.routing(M), O.route(local, cfg.E)):
        assert np.array_equal(a, b)
    ids_r, w_r = S.ep_mask_foreign(ids_g, w, first, cfg.E)
    check_rows(got, ck, x, ids_r, w_r, 7.0)
    # a row whose slots are all foreign gives 0 (the remap's weight-0 slots add exact zeros)
    none = ~(local >= 0).any(axis=1)
    assert np.all(got[none] == 0)
    layer.close()


@pytest.mark.parametrize("quant", ["mxfp4", "nvfp4", "w4a4_nvfp4"])
def test_run_chunked_above_capacity(quant):
    """M = 70 rows on a capacity-32 plan through the chunked entry point: three chunks (32, 32,
    6) in order on one scratch.  Deterministic mode: bit-identical to three separate calls, and
    every row within the bound of the oracle."""
    from serving_route_count_gb300 import moe_run_chunked
    cfg = small_cfg(quant)
    ck = S.make_checkpoint(cfg, seed=5000)
    rng = np.random.default_rng(5001)
    M, cap = 70, 32
    x = S.make_x(rng, M, cfg.H)
    ids = S.uniform_topk(rng, M, cfg.E, cfg.topk)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, cap, 7.0, 1)
    xt, it, wt = to_device(x, ids, w)
    out = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
    moe_run_chunked(layer.plan, layer.prep, layer.scratch, xt, it, wt, out)
    got = out_bits(out)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    sep = np.concatenate([run_layer(layer, x[s:s + cap], ids[s:s + cap], w[s:s + cap])
                          for s in range(0, M, cap)])
    assert np.array_equal(got, sep)
    check_rows(got, ck, x, ids, w, 7.0)
    layer.close()


@pytest.mark.parametrize("backend", [0, 1])
def test_hybrid_mx_scale_window(backend):
    """MXFP4 kept tier with scale bytes spread over the whole exact window (2^-40..2^-4: 36
    binades below the largest) plus 1 % of groups 80 binades further down, which prepare
    flushes to zero (terms below 2^-34 of the matrix's largest weights): every row within the
    bound of the oracle, which keeps them."""
    cfg = small_cfg("hybrid_mx", I=256)
    ck = S.make_checkpoint(cfg, seed=6100)
    rng = np.random.default_rng(6101)
    for name in ("s13", "s2"):
        sc = rng.integers(87, 124, size=getattr(ck.nv, name).shape, dtype=np.uint8)
        sc[rng.random(sc.shape) < 0.01] = 5
        setattr(ck.nv, name, sc)
    M = 24
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 0.8)
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 1.0)
    assert (ck.tier[ids] == S.TIER_NVFP4).any()
    layer = _layer(ck, cfg.topk, M, math.inf, 1, backend=backend)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, math.inf)
    layer.close()


def test_hybrid_mx_full_size_sampled():
    """The "v3" hybrid layer at full size (E=256, H=6144, I=512, top-8; 64 MXFP4 + 192 NF3
    experts, Zipf routing) at decode and prefill sizes: sampled rows against the oracle."""
    cfg = S.CONFIGS["hybrid_mxfp4_nf3"]
    ck = S.make_checkpoint(cfg)
    for M, rows in ((8, [0, 3, 7]), (512, [0, 255, 511])):
        x, ids, w = S.make_inputs(cfg, M)
        layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, 1)
        got = run_layer(layer, x, ids, w)
        st, code = layer.device_error()
        assert st == 0 and code == 0, code
        check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=rows)
        layer.close()


@pytest.mark.parametrize("quant,M,det,backend", [("nvfp4", 6, 1, 0), ("hybrid", 16, 0, 0),
                                                 ("hybrid_mx", 40, 1, 0), ("nvfp4", 300, 0, 0),
                                                 ("hybrid", 24, 1, 1), ("nvfp4", 4200, 1, 0)])
def test_router_weight_on_input(quant, M, det, backend):
    """Router weights applied to fc1's input (16-bit paths): one-launch, two-launch and (beyond
    4096 slots) chunked routing with the token-row conversion, several tile widths, both
    combines and the CUDA-core backend, against the oracle with the same option on every row;
    top-1 (the usual use) and top-4."""
    topk = 1 if M >= 100 else 4
    cfg = small_cfg(quant, I=256, topk=topk)
    ck = S.make_checkpoint(cfg, seed=7000 + M)
    rng = np.random.default_rng(7001 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, topk, 0.8)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, topk, M, math.inf, det, backend=backend, weight_on_input=True)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, math.inf, weight_on_input=True)
    layer.close()


@pytest.mark.parametrize("M,det", [(5, 1), (16, 0), (40, 1), (200, 0), (600, 1)])
def test_nvfp4_mxfp8_activations(M, det):
    """NVFP4 weights with MXFP8 activations and per-expert activation global scales, on the
    16-bit tensor-core kernels, at every token-tile width and both fc1 schedules: every row
    against the oracle, and fc2's operand - the MXFP8 value of a2 * h - code for code, except
    where fp32 noise decides a near-midpoint rounding (there it must be the other neighbour)."""
    cfg = small_cfg("w4a8_nvfp4", I=256)
    ck = S.make_checkpoint(cfg, seed=8000 + M)
    rng = np.random.default_rng(8001 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 0.8)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 1.0)
    layer = _layer(ck, cfg.topk, M, math.inf, det)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, math.inf)
    hq, _ = layer.intermediate(M)
    got_h = hq[:, : cfg.I].view(np.float16).astype(np.float64)
    h = O.slot_intermediate(ck, x, ids, math.inf)
    _, _, perm, _ = O.route(ids, cfg.E)
    a2 = ck.a2.astype(np.float64)[ids.reshape(-1)[perm]][:, None]
    q, sc = C.mxfp8_quantize(h * a2)
    want_h = C.mxfp8_dequantize(q, sc)
    amb, alt = C.mxfp8_alternates(h * a2, 1e-4)
    mism = got_h != want_h
    rate = float(mism.mean())
    assert np.all(amb[mism]), "a code differs where the rounding is not decided by fp32 noise"
    assert np.all(got_h[mism] == alt[mism])
    assert rate < 2e-3
    layer.close()


def test_nvfp4_mxfp8_activations_full_size_sampled():
    cfg = S.CONFIGS["w4a8_nvfp4"]
    ck = S.make_checkpoint(cfg)
    for M, rows in ((8, [0, 3, 7]), (512, [0, 255, 511])):
        x, ids, w = S.make_inputs(cfg, M)
        layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, 1)
        got = run_layer(layer, x, ids, w)
        st, code = layer.device_error()
        assert st == 0 and code == 0, code
        check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=rows)
        layer.close()


@pytest.mark.parametrize("M,det", [(5, 1), (16, 0), (40, 1), (100, 0), (300, 1)])
def test_w4a4_nvfp4(M, det):
    """NVFP4 weights x NVFP4 activations on the block-scaled FP4 tensor cores at every token-tile
    width (16 / 32 / 64), split and whole-K fc1, one- and two-launch routing, both combines:
    every row against the oracle, and fc2's operand - NVFP4 of a2 * h - scale for scale and
    value for value, except where fp32 noise decides a near-midpoint rounding (a block whose
    vmax / 6 sits at an E4M3 midpoint, or an element at an E2M1 midpoint)."""
    cfg = small_cfg("w4a4_nvfp4", I=256)
    ck = S.make_checkpoint(cfg, seed=9000 + M)
    rng = np.random.default_rng(9001 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 0.8)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 1.0)
    layer = _layer(ck, cfg.topk, M, math.inf, det)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    hq, hs = layer.intermediate(M)
    h = O.slot_intermediate(ck, x, ids, math.inf)
    _, _, perm, _ = O.route(ids, cfg.E)
    a2 = ck.a2.astype(np.float64)[ids.reshape(-1)[perm]][:, None]
    v = (h * a2).astype(np.float32)
    q, sc = C.nvfp4_quantize(v)
    Ip = hq.shape[1] * 2
    got_q = C.unpack_fp4(hq)
    # blocks: a different scale only where vmax / 6 lies at an E4M3 rounding midpoint
    vmax6 = np.abs(v.reshape(v.shape[0], -1, 16)).max(axis=-1) / 6.0
    bad_s = hs[:, : sc.shape[1]] != sc
    if bad_s.any():
        lo = C.e4m3_decode(np.minimum(sc, hs[:, : sc.shape[1]]))
        hi = C.e4m3_decode(np.maximum(sc, hs[:, : sc.shape[1]]))
        mid = (lo + hi) / 2
        assert np.all(np.abs(vmax6[bad_s] - mid[bad_s]) <= 1e-4 * vmax6[bad_s]), "scale flips"
    same = np.repeat(~bad_s, 16, axis=1)
    got_v = C.nvfp4_dequantize(got_q, hs)
    want_v = C.nvfp4_dequantize(q, sc)
    amb, alt = C.nvfp4_alternates(v.astype(np.float64), 1e-4)
    mism = (got_v != want_v) & same
    assert np.all(amb[mism]), "a code differs where the rounding is not decided by fp32 noise"
    assert np.all(got_v[mism] == alt[mism])
    assert mism.mean() < 2e-3
    check_rows(got, ck, x, ids, w, math.inf)
    if det:
        assert np.array_equal(run_layer(layer, x, ids, w), got)
    layer.close()


def test_w4a4_nvfp4_full_size_sampled():
    cfg = S.CONFIGS["w4a4_nvfp4"]
    ck = S.make_checkpoint(cfg)
    for M, rows in ((8, [0, 3, 7]), (512, [0, 255, 511])):
        x, ids, w = S.make_inputs(cfg, M)
        layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, 1)
        got = run_layer(layer, x, ids, w)
        st, code = layer.device_error()
        assert st == 0 and code == 0, code
        check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=rows)
        layer.close()


def test_run_host_packed_inputs():
    """moe_run_host with [x | ids | weights] back to back in one pinned buffer (one copy up)
    gives the same bits as with three separate host buffers (deterministic combine)."""
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=9100)
    rng = np.random.default_rng(9101)
    layer = _layer(ck, cfg.topk, 32, 7.0, 1)
    for M in (3, 32):
        x = S.make_x(rng, M, cfg.H)
        ids = S.uniform_topk(rng, M, cfg.E, cfg.topk)
        w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
        xb, kb = M * cfg.H * 2, M * cfg.topk * 4
        packed = torch.empty(xb + 2 * kb, dtype=torch.uint8).pin_memory()
        packed[:xb].copy_(torch.from_numpy(x.view(np.uint8).reshape(-1)))
        packed[xb:xb + kb].copy_(torch.from_numpy(ids.view(np.uint8).reshape(-1)))
        packed[xb + kb:].copy_(torch.from_numpy(w.view(np.uint8).reshape(-1)))
        o1 = torch.empty((M, cfg.H), dtype=torch.bfloat16).pin_memory()
        layer.run_host(packed[:xb].view(torch.bfloat16).view(M, cfg.H),
                       packed[xb:xb + kb].view(torch.int32).view(M, cfg.topk),
                       packed[xb + kb:].view(torch.float32).view(M, cfg.topk), o1)
        o2 = torch.empty((M, cfg.H), dtype=torch.bfloat16).pin_memory()
        layer.run_host(torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory(),
                       torch.from_numpy(ids).pin_memory(), torch.from_numpy(w).pin_memory(), o2)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        check_rows(out_bits(o1), ck, x, ids, w, 7.0)
    layer.close()


def _canon_fp4(a):
    lo, hi = a & 0x0F, a >> 4
    lo = np.where(lo == 8, 0, lo)
    hi = np.where(hi == 8, 0, hi)
    return (lo | (hi << 4)).astype(np.uint8)


@pytest.mark.parametrize("quant,layout", [("mxfp4", 0), ("mxfp4", 1), ("nvfp4", 1), ("hybrid", 0),
                                          ("hybrid_mx", 1), ("w4a8_nvfp4", 0),
                                          ("w4a4_nvfp4", 0)])
def test_prepare_roundtrip(quant, layout):
    """The prepared device layout holds every checkpoint byte: read back through the inverse
    permutation (moe_unprepare_weights) it equals the checkpoint - E2M1 nibbles after the
    -0 -> +0 rewrite, scales, NF3 planes, globals and activation global scales - for both w13
    stackings and every format."""
    from serving_route_count_gb300 import moe_unprepare_weights
    cfg = small_cfg(quant)
    ck = S.make_checkpoint(cfg, seed=9200, layout=layout)
    if ck.quant == "hybrid":
        nv, nf = ck.nv, ck.nf
        want = {"w13": nv.w13, "s13": nv.s13, "w2": nv.w2, "s2": nv.s2, "nf_w13": nf.w13,
                "nf_s13": nf.s13, "nf_w2": nf.w2, "nf_s2": nf.s2}
        if nv.quant == "nvfp4":
            want.update(g13=nv.g13, g2=nv.g2)
    else:
        want = {"w13": ck.w13, "s13": ck.s13, "w2": ck.w2, "s2": ck.s2}
        if ck.g13 is not None:
            want.update(g13=ck.g13, g2=ck.g2)
        if ck.a13 is not None:
            want.update(a1_gscale=ck.a13, a2_gscale=ck.a2)
    layer = _layer(ck, cfg.topk, 4, math.inf, 0)
    got = moe_unprepare_weights(layer.wp, layer.prep, want)
    for k, v in want.items():
        exp = _canon_fp4(v) if k in ("w13", "w2") else v
        assert np.array_equal(got[k], exp), k
    layer.close()


def _sample_rows(ids, M, seed, n=256):
    """All rows up to n; beyond, a seeded subset of n rows plus every padding row."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    pad = np.flatnonzero(~(ids >= 0).any(axis=1))
    return np.union1d(np.sort(rng.choice(M, n, replace=False)), pad)


def _full_size_both_modes(cfg, ck, M, layers=None):
    """One call of the full-size layer at M rows in each combine mode: every sampled row (all
    rows up to 256; a seeded 256-row subset plus all padding rows beyond) against the oracle,
    padding rows exactly 0, no device error, routing bit-exact, and in deterministic mode a
    bit-identical repeat.  ``layers`` ({det: layer}) reuses layers of a larger capacity."""
    x, ids, w = S.make_inputs(cfg, M)
    rows = _sample_rows(ids, M, seed=9000 + M)
    ref = oracle_rows(ck, x, ids, w, cfg.swiglu_limit, rows=rows)
    route = O.route(ids, ck.E)
    for det in (0, 1):
        layer = layers[det] if layers else _layer(ck, cfg.topk, M, cfg.swiglu_limit, det)
        got = run_layer(layer, x, ids, w)
        st, code = layer.device_error()
        assert st == 0 and code == 0, (M, det, code)
        for a, b in zip(layer.routing(M), route):
            assert np.array_equal(a, b), (M, det)
        check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=rows, ref_f64=ref)
        pad = ~(ids >= 0).any(axis=1)
        assert np.all(got[pad] == 0)
        if det:
            assert np.array_equal(run_layer(layer, x, ids, w), got), M
        if not layers:
            layer.close()


def test_decode_ladder_full_size_all_rows(decode_layer):
    """Every call of the decode ladder (E=384, H=7168, I=576, top-6, M = 1..8, 10, 12, 14, 16,
    last quarter of the rows padding) in both combine modes, every row against the oracle:
    the calls the bench times, on capacity-16 plans as the bench plans them, at their own
    split-K / stream-K fc1 and fc2 schedules."""
    cfg, ck = decode_layer
    layers = {det: _layer(ck, cfg.topk, 16, cfg.swiglu_limit, det) for det in (0, 1)}
    for M in cfg.m_list:
        _full_size_both_modes(cfg, ck, M, layers)
    for layer in layers.values():
        layer.close()


@pytest.fixture(scope="module")
def nvfp4_ck():
    return S.make_checkpoint(S.CONFIGS["w4a16_nvfp4"])


@pytest.mark.parametrize("M", [64, 512, 2048, 8192])
def test_nvfp4_full_size_sampled(nvfp4_ck, M):
    """NVFP4 W4A16 (E=256, H=6144, I=512, top-8) at its decode and prefill sizes, both
    combine modes: all rows up to 256, else 256 seeded rows."""
    _full_size_both_modes(S.CONFIGS["w4a16_nvfp4"], nvfp4_ck, M)


@pytest.mark.parametrize("M", [8, 2048])
def test_hybrid_full_size_sampled(M):
    """The hybrid layer (64 NVFP4 + 192 NF3 experts, Zipf 0.8 routing) at both of its sizes,
    both combine modes (deterministic is the configured one)."""
    cfg = S.CONFIGS["hybrid_nvfp4_nf3"]
    _full_size_both_modes(cfg, S.make_checkpoint(cfg), M)


# ---------------------------------------------------------------------------- tensor-core path

@pytest.mark.parametrize("M,det", [(5, 0), (16, 1), (37, 0), (100, 1), (200, 1), (600, 0)])
def test_w4a8_tensor_core_tile_widths(M, det):
    """W4A8 through the tcgen05 kernels at M covering every token-tile width (16 up to 16
    tokens; then 32, 64 and 96 by expected slots per expert: M = 37, 100, 200 / 600 here),
    experts with many tiles, and both fc1 schedules (split K for small M, whole K otherwise);
    E=16, H=1280 (10 K tiles), I=192 (two 128-row weight blocks, the second half empty), Zipf
    routing with dropped ids."""
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=1000 + M)
    rng = np.random.default_rng(2000 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 1.1)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, M, 7.0, det)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, 7.0)
    # the CUDA-core backend computes the same call independently
    simt = _layer(ck, cfg.topk, M, 7.0, det, backend=1)
    check_rows(run_layer(simt, x, ids, w), ck, x, ids, w, 7.0)
    xq, xs = layer.actq(M)
    _, _, perm, _ = layer.routing(M)
    q, s = C.mxfp8_quantize(C.bf16_bits_to_f64(x))
    assert np.array_equal(xq, q[perm // cfg.topk]) and np.array_equal(xs, s[perm // cfg.topk])


@pytest.mark.parametrize("M,det", [(1, 1), (3, 0), (9, 1), (16, 0)])
def test_w4a8_stream_k_fc1(M, det):
    """The persistent stream-K fc1 forced on small layers (E=16, H=1280: 10 K tiles per unit,
    far fewer than the grid's CTAs, so units split into many pieces and most CTAs hold none):
    every row against the oracle, the fc2 operand's codes against the oracle's requantisation
    within the near-midpoint reading, and (deterministic mode) bit-identical repeats."""
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=5000 + M)
    rng = np.random.default_rng(6000 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 1.1)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, M, 7.0, det, fc1_kernel=2)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, 7.0)
    if det:
        assert np.array_equal(run_layer(layer, x, ids, w), got)
    hq, hs = layer.intermediate(M)
    h = O.slot_intermediate(ck, x, ids, 7.0)
    q, s8 = C.mxfp8_quantize(h)
    got_h = C.mxfp8_dequantize(hq[:, : cfg.I], hs[:, : cfg.I // 32])
    want_h = C.mxfp8_dequantize(q, s8)
    amb, alt = C.mxfp8_alternates(h, 1e-4)
    mism = got_h != want_h
    assert np.all(amb[mism] & (got_h[mism] == alt[mism])), int(mism.sum())


@pytest.mark.parametrize("backend", [0, 1])
def test_w4a8_intermediate_requant(backend):
    """The fc2 operand h -> MXFP8 against the oracle's quantisation of the exact SwiGLU output:
    codes may differ only where the fp32 h sits within rounding noise of an E4M3 midpoint, so
    mismatches must be rare and each within one E4M3 step of the exact value."""
    cfg = small_cfg("mxfp4")
    M = 600
    ck = S.make_checkpoint(cfg, seed=1000 + M)
    rng = np.random.default_rng(2000 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 1.1)
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, M, 7.0, 0, backend=backend)
    run_layer(layer, x, ids, w)
    hq, hs = layer.intermediate(M)
    h = O.slot_intermediate(ck, x, ids, 7.0)
    q, s = C.mxfp8_quantize(h)
    I = cfg.I
    got = C.mxfp8_dequantize(hq[:, :I], hs[:, : I // 32])
    want = C.mxfp8_dequantize(q, s)
    mism = got != want
    rate = float(mism.mean())
    step = np.repeat(C.e8m0_value(s), 32, axis=1) * 2.0 ** np.floor(
        np.log2(np.maximum(np.abs(h) / np.repeat(C.e8m0_value(s), 32, axis=1), 2.0 ** -6))) / 8
    print(f"\nbackend {backend}: requant mismatches {int(mism.sum())} of {mism.size} "
          f"({rate:.2e}); rows with any: {int(mism.any(axis=1).sum())} of {mism.shape[0]}")
    amb, alt = C.mxfp8_alternates(h, 1e-4)
    assert np.all(amb[mism]), "a code differs where the rounding is not decided by fp32 noise"
    assert np.all(got[mism] == alt[mism])
    assert rate < 2e-3
    assert np.all(hq[:, I:] == 0)


@pytest.mark.parametrize("quant,M,det", [("nvfp4", 5, 0), ("hybrid", 16, 1), ("nvfp4", 37, 1),
                                         ("hybrid", 200, 0), ("hybrid", 600, 1),
                                         ("hybrid_mx", 5, 1), ("hybrid_mx", 40, 0),
                                         ("hybrid_mx", 200, 1)])
def test_w4a16_tensor_core_tile_widths(quant, M, det):
    """NVFP4, the NVFP4 + NF3 hybrid and the MXFP4 + NF3 hybrid through the 16-bit tcgen05
    kernels (weights expanded to f16) at every token-tile width, against the oracle on every
    row; the CUDA-core backend must agree too.  E=16 (5 kept experts), H=1280, I=256."""
    cfg = small_cfg(quant, I=256)
    ck = S.make_checkpoint(cfg, seed=3000 + M)
    rng = np.random.default_rng(4000 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 0.8)
    ids[rng.random(ids.shape) < 0.05] = -1
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 1.0)
    layer = _layer(ck, cfg.topk, M, math.inf, det)
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, math.inf)
    # intermediate h: bf16 rounding of the SwiGLU output, carried as f16.  bf16 values are exact
    # in f16 down to 2^-16 (f16 subnormal step 2^-24); below that the f16 subnormal rounding
    # applies, an absolute error under 2^-24 that no output can see.
    hq, _ = layer.intermediate(M)
    h = O.slot_intermediate(ck, x, ids, math.inf)
    got_h = hq[:, : cfg.I].view(np.float16).astype(np.float64)
    want_h = C.bf16_round(h)
    # ambiguity window: 1e-4 of the value, plus H_CANCEL_ATOL of the slot's rms for elements
    # whose gate or up projection cancels (fp32 sums err by the size of their terms)
    rms = np.sqrt(np.mean(h * h, axis=1, keepdims=True))
    amb, alt = C.bf16_alternates(h, 1e-4, H_CANCEL_ATOL * rms)
    big = np.abs(h) >= 2.0 ** -16
    mism = (got_h != want_h) & big
    # a mismatch is the other rounding of a near-midpoint value, or (a cancelled sum, whose
    # error exceeds an ulp of its small result) within the absolute window of the exact value
    near_exact = np.abs(got_h - h) <= np.abs(want_h - h) + H_CANCEL_ATOL * rms
    bad = mism & ~(amb & (got_h == alt)) & ~near_exact
    if bad.any():
        i = np.argwhere(bad)[:5]
        print("unexplained h mismatches:", int(bad.sum()),
              [(float(h[a, b]), float(want_h[a, b]), float(got_h[a, b]), float(rms[a, 0]))
               for a, b in i])
    assert not bad.any(), int(bad.sum())
    # tiny elements: f16 subnormal rounding (under 2^-24) on top of the same absolute window
    tiny_ok = np.abs(got_h - h) <= np.abs(want_h - h) + 2.0 ** -24 + H_CANCEL_ATOL * rms
    assert np.all(tiny_ok[~big])
    simt = _layer(ck, cfg.topk, M, math.inf, det, backend=1)
    check_rows(run_layer(simt, x, ids, w), ck, x, ids, w, math.inf)


@pytest.mark.parametrize("det", [0, 1])
def test_device_wait_timeout_recovers(det):
    """The bounded device waits, run out on purpose without a fault: with the wait probe on, fc1's
    MMA issuer waits 2 ms on a barrier nothing arrives on, so the call reports MOE_ERR_TIMEOUT
    through the device error word; its producers then give up their own waits after the 1 s
    bound and drain their copies.  The context and the plan stay usable: the next call, probe
    off, matches the oracle on every row and reports no error."""
    from serving_route_count_gb300 import moe_plan_set_wait_probe
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=8100 + det)
    rng = np.random.default_rng(8200 + det)
    M = 9
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 1.1)
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, M, 7.0, det, fc1_kernel=1)
    moe_plan_set_wait_probe(layer.plan, 2_000_000)
    run_layer(layer, x, ids, w)
    torch.cuda.synchronize()
    st, code = layer.device_error()
    assert st == 7 and code & 2, (st, code)
    moe_plan_set_wait_probe(layer.plan, 0)
    got = run_layer(layer, x, ids, w)
    assert layer.device_error() == (0, 0)
    check_rows(got, ck, x, ids, w, 7.0)


@pytest.mark.parametrize("M,det", [(5, 1), (16, 0), (40, 1), (200, 0), (1100, 0)])
def test_hybrid_mx_kept_a8(M, det):
    """The A8 opt-in of the MXFP4 kept tier (static per-tensor FP8 activations with the layer's
    two input scales) at tile widths 16 to 64, every routing path (one launch, two launches,
    and chunked routing with the token-row conversion beyond 4096 slots) and both combines: every
    row against the oracle; the kept tier's fc2 operand (h) code for code against the oracle's
    static FP8 decisions within the near-midpoint reading; NF3 slots unchanged (bf16 h)."""
    cfg = small_cfg("hybrid_mx", I=256)
    ck = S.make_checkpoint(cfg, seed=6200 + M)
    rng = np.random.default_rng(6300 + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 0.8)
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 1.0)
    assert (ck.tier[ids] == S.TIER_NVFP4).any() and (ck.tier[ids] == S.TIER_NF3).any()
    layer = _layer(ck, cfg.topk, M, math.inf, det, kept_a8=(ck.in13, ck.in2))
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, math.inf, kept_a8=True)
    if det:
        assert np.array_equal(run_layer(layer, x, ids, w), got)
    # fc2's operand: kept slots hold the static FP8 value of h divided by the scale (the
    # kernel keeps the E4M3 code value in f16), NF3 slots bf16(h)
    hqb, _ = layer.intermediate(M)
    hq = np.ascontiguousarray(hqb[:, : cfg.I]).view(np.float16).astype(np.float64)
    h = O.slot_intermediate(ck, x, ids, kept_a8=True)
    _, _, perm, _ = O.route(ids, cfg.E)
    kept = ck.tier[ids.reshape(-1)[perm]] == S.TIER_NVFP4
    s2 = float(np.float32(ck.in2))
    want_k = C.fp8_static_quantize(h[kept], ck.in2)[1] / s2
    mask, alt = C.fp8_static_alternates(h[kept], ck.in2, 1e-4)
    mism = hq[kept] != want_k
    assert np.all(mask[mism] & (hq[kept][mism] == alt[mism] / s2)), int(mism.sum())
    layer.close()


def test_hybrid_mx_kept_a8_full_size_sampled():
    """The A8 opt-in on the full-size "v3" hybrid layer (E=256, H=6144, I=512, top-8, 64 MXFP4
    + 192 NF3 experts, Zipf routing) at M = 8 and 512: sampled rows against the oracle."""
    cfg = S.CONFIGS["hybrid_mxfp4_nf3"]
    ck = S.make_checkpoint(cfg)
    for M, rows in ((8, [0, 3, 7]), (512, [0, 255, 511])):
        x, ids, w = S.make_inputs(cfg, M)
        layer = _layer(ck, cfg.topk, M, cfg.swiglu_limit, 1, kept_a8=(ck.in13, ck.in2))
        got = run_layer(layer, x, ids, w)
        st, code = layer.device_error()
        assert st == 0 and code == 0, code
        check_rows(got, ck, x, ids, w, cfg.swiglu_limit, rows=rows, kept_a8=True)
        layer.close()


@pytest.mark.parametrize("H,I,M,det", [(1408, 192, 9, 0), (1408, 320, 37, 1), (1408, 192, 200, 0),
                                       (1280, 448, 16, 1)])
def test_w4a8_fc2_paired_k_tails(H, I, M, det):
    """fc2's weights when I % 128 == 64: the 64-column K tails of row blocks 2j and 2j + 1 share
    one tile, an odd row block multiplying its half at a 64-column offset; with an odd number of
    128-row blocks (H = 1408: 11) the last tail has no partner.  Prepared bytes read back equal the
    checkpoint, and every row matches the oracle through the unit-per-CTA fc2 (small M) and the
    persistent one (M = 200), in both combines."""
    from serving_route_count_gb300 import moe_unprepare_weights
    cfg = small_cfg("mxfp4", H=H, I=I)
    ck = S.make_checkpoint(cfg, seed=9300 + I + M)
    rng = np.random.default_rng(9400 + I + M)
    x = S.make_x(rng, M, cfg.H)
    ids = S.zipf_topk(rng, M, cfg.E, cfg.topk, 1.1)
    w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
    layer = _layer(ck, cfg.topk, M, 7.0, det)
    want = {"w13": ck.w13, "s13": ck.s13, "w2": ck.w2, "s2": ck.s2}
    got_w = moe_unprepare_weights(layer.wp, layer.prep, want)
    for k, v in want.items():
        assert np.array_equal(got_w[k], _canon_fp4(v) if k in ("w13", "w2") else v), k
    got = run_layer(layer, x, ids, w)
    st, code = layer.device_error()
    assert st == 0 and code == 0, code
    check_rows(got, ck, x, ids, w, 7.0)
    if det:
        assert np.array_equal(run_layer(layer, x, ids, w), got)
    layer.close()
