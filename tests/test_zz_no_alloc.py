"""The allocation-free entry point (moe_run_static_scratch) against moe_run.

It exists for callers that cannot allocate device memory (a framework memory pool that exposes
no allocator to plug-ins, sandboxed runtimes, paths that must never allocate): the scratch lives
in a fixed array inside the library.  Two calls in a row, with different inputs, must each match
the caller-scratch entry point within the tolerance the parity tests use (and bit for bit in
deterministic mode, where both runs perform the same arithmetic).  This file is collected last
and also runs alone in a fresh process."""
import numpy as np
import pytest

from moe_cases import REL_L2_BOUND, MAX_ERR_BOUND, small_cfg, to_device, out_bits
from oracle import codecs as C
from oracle import moe as O
from synth import moe_inputs as S

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_route_count_gb300 import build
    build.build()


@pytest.mark.parametrize("det", [0, 1])
def test_static_scratch_matches_moe_run(det):
    from serving_route_count_gb300 import (MoELayer, moe_get_device_error_static,
                                           moe_run_static_scratch)
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=515)
    M = 37
    layer = MoELayer(ck, cfg.topk, M, 7.0, det)
    for call in range(2):
        rng = np.random.default_rng(600 + call)
        x = S.make_x(rng, M, cfg.H)
        ids = S.uniform_topk(rng, M, cfg.E, cfg.topk)
        ids[-2:] = -1
        w = S.router_weights(rng, M, cfg.topk, "sigmoid_norm", 2.5)
        xt, it, wt = to_device(x, ids, w)
        ref = out_bits(layer(xt, it, wt))
        out = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
        moe_run_static_scratch(layer.plan, layer.prep, xt, it, wt, out)
        got = out_bits(out)
        if det:
            assert np.array_equal(got, ref)
        rel, mx = O.row_errors(got, C.bf16_bits_to_f64(ref))
        assert np.all(rel <= REL_L2_BOUND) and np.all(mx <= MAX_ERR_BOUND), (call, rel.max(), mx.max())
        assert np.all(got[-2:] == 0)
        # the call's device error word lives in the library's array: read through the static
        # accessor (no bounded wait gave up, no device check failed)
        assert moe_get_device_error_static(layer.plan) == (0, 0)


@pytest.mark.parametrize("det", [0, 1])
def test_static_scratch_decode_layer(det):
    """The decode layer (E=384, H=7168, I=576, top-6) at capacity 16 fits the 16 MiB array in
    both combine modes.  Calls of M = 8 (split-K fc1) and M = 16 (the persistent stream-K fc1,
    whose partial-sum slots then live in the array too) match moe_run (bit for bit in
    deterministic mode)."""
    from serving_route_count_gb300 import (MoELayer, moe_get_device_error_static,
                                           moe_run_static_scratch, moe_scratch_bytes)
    cfg = S.CONFIGS["decode_w4a8"]
    ck = S.make_checkpoint(cfg)
    layer = MoELayer(ck, cfg.topk, 16, cfg.swiglu_limit, det)
    assert moe_scratch_bytes(layer.plan) <= 16 << 20
    for call, M in enumerate((8, 16)):
        x, ids, w = S.make_inputs(cfg, M)
        xt, it, wt = to_device(x, ids, w)
        ref = out_bits(layer(xt, it, wt))
        out = torch.empty((M, cfg.H), dtype=torch.bfloat16, device="cuda")
        moe_run_static_scratch(layer.plan, layer.prep, xt, it, wt, out)
        got = out_bits(out)
        if det:
            assert np.array_equal(got, ref), call
        rel, mx = O.row_errors(got, C.bf16_bits_to_f64(ref))
        assert np.all(rel <= REL_L2_BOUND) and np.all(mx <= MAX_ERR_BOUND), (call, rel.max(), mx.max())
        assert moe_get_device_error_static(layer.plan) == (0, 0)
    layer.close()


def test_static_scratch_rejects_large_plans():
    from serving_route_count_gb300 import MoEError, MoELayer, moe_run_static_scratch
    cfg = small_cfg("mxfp4")
    ck = S.make_checkpoint(cfg, seed=516)
    layer = MoELayer(ck, cfg.topk, 4096, 7.0, 1)     # scratch far above 16 MiB
    x = S.make_x(np.random.default_rng(1), 4, cfg.H)
    xt, it, wt = to_device(x, np.zeros((4, cfg.topk), np.int32), np.ones((4, cfg.topk), np.float32))
    out = torch.empty((4, cfg.H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoEError) as ei:
        moe_run_static_scratch(layer.plan, layer.prep, xt, it, wt, out)
    assert ei.value.status == 4
