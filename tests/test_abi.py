"""The C ABI library builds, loads and exports every function include/moe_gb300.h declares;
host-only entry points (planning, sizing, argument checks) behave as documented.  No call here
touches a GPU."""
import ctypes
import math

import pytest

from serving_route_count_gb300 import _lib, build
import serving_route_count_gb300 as moe


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.header_functions()
    assert "moe_run" in names and "moe_plan" in names and "moe_prepare_weights" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks a signature for {n}"


def test_version_and_status_strings(lib):
    assert "sm_103a" in moe.moe_version()
    assert _lib.load().moe_last_cuda_error().decode() == "cudaSuccess"
    assert moe.moe_status_str(0) == "ok"
    assert "capacity" in moe.moe_status_str(4)


def test_plan_weights_shapes_and_sizes(lib):
    E, H, I = 384, 7168, 576
    wp = moe.moe_plan_weights(E, H, I, moe.MOE_W4A8_MXFP4)
    n = moe.moe_prepared_bytes(wp)
    codes = E * (2 * I * H // 2 + H * 640 // 2)
    sf = E * (2 * 5 * (H // 128) * 512 + (H // 128) * 5 * 512)
    assert codes + sf <= n <= codes + sf + 4096
    moe.moe_destroy_weight_plan(wp)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_weights(8, 200, 128, moe.MOE_W4A8_MXFP4)         # H % 128 != 0
    assert ei.value.status == 2
    with pytest.raises(moe.MoEError):
        moe.moe_plan_weights(8, 256, 96, moe.MOE_W4A8_MXFP4)          # I % 64 != 0
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_weights(8, 256, 128, moe.MOE_W4A16_HYBRID)       # hybrid needs a tier map
    assert ei.value.status == 1
    with pytest.raises(moe.MoEError):
        moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A16_HYBRID, tier_of_expert=[4, 3, 5, 3])
    wp = moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A16_HYBRID, tier_of_expert=[4, 3, 3, 4])
    nv_bytes = moe.moe_prepared_bytes(wp)
    assert nv_bytes > 0
    moe.moe_destroy_weight_plan(wp)
    # MXFP4 kept tier: the NVFP4 sections plus the per-expert scale maxima of both matrices
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A16_HYBRID_MX)
    assert ei.value.status == 1
    wp = moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A16_HYBRID_MX, tier_of_expert=[4, 3, 3, 4])
    assert moe.moe_prepared_bytes(wp) == nv_bytes + 2 * 256
    moe.moe_destroy_weight_plan(wp)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_weights(4, 256, 128, 6)
    assert ei.value.status == 3


def test_plan_and_scratch_sizes(lib):
    p_atomic = moe.moe_plan(384, 7168, 576, 6, 16, moe.MOE_W4A8_MXFP4, 7.0, 0)
    p_det = moe.moe_plan(384, 7168, 576, 6, 16, moe.MOE_W4A8_MXFP4, 7.0, 1)
    a, d = moe.moe_scratch_bytes(p_atomic), moe.moe_scratch_bytes(p_det)
    assert a > 16 * 7168 * 4 and d > 96 * 7168 * 4
    assert moe.moe_io_bytes(p_det) >= 2 * 16 * 7168 * 2 + 2 * 96 * 4
    moe.moe_plan_set_swiglu_alpha_beta(p_det, 1.702, 1.0)
    moe.moe_destroy_plan(p_atomic)
    moe.moe_destroy_plan(p_det)
    with pytest.raises(moe.MoEError):
        moe.moe_plan(384, 7168, 576, 0, 16, moe.MOE_W4A8_MXFP4, 7.0, 0)       # top-k 0
    with pytest.raises(moe.MoEError):
        moe.moe_plan(384, 7168, 576, 6, 16, moe.MOE_W4A8_MXFP4, float("nan"), 0)
    with pytest.raises(moe.MoEError):
        moe.moe_plan(384, 7168, 576, 6, 16, 7, 7.0, 0)                        # bad quant mode
    p = moe.moe_plan(8, 256, 128, 2, 4, moe.MOE_W4A8_MXFP4, math.inf, 0)
    moe.moe_destroy_plan(p)


def test_run_argument_checks_without_gpu(lib):
    L = _lib.load()
    p = moe.moe_plan(8, 256, 128, 2, 4, moe.MOE_W4A8_MXFP4, 7.0, 0)
    wp = moe.moe_plan_weights(8, 256, 128, moe.MOE_W4A8_MXFP4)
    # null plan / weights
    assert L.moe_run(None, None, None, 0, None, None, None, None, 1, None) == 1
    # M > max_m -> capacity, before any device work
    fake = ctypes.c_void_p(1)
    assert L.moe_run(ctypes.c_void_p(p), fake, None, 0, None, None, None, None, 5, None) == 4
    # M == 0 is a no-op
    assert L.moe_run(ctypes.c_void_p(p), fake, None, 0, None, None, None, None, 0, None) == 0
    # negative M
    assert L.moe_run(ctypes.c_void_p(p), fake, None, 0, None, None, None, None, -1, None) == 1
    # null buffers with M > 0
    assert L.moe_run(ctypes.c_void_p(p), fake, None, 0, None, None, None, None, 2, None) == 1
    # prepare with a too small destination
    ck = _lib.MoeCheckpoint()
    out = ctypes.c_void_p()
    assert L.moe_prepare_weights(ctypes.c_void_p(wp), ctypes.byref(ck), ctypes.c_void_p(256), 16,
                                 None, ctypes.byref(out)) == 1
    moe.moe_destroy_plan(p)
    moe.moe_destroy_weight_plan(wp)


def test_static_error_word_arguments_without_gpu(lib):
    """moe_get_device_error_static checks its arguments and the plan's scratch size before any
    device call: a null plan or code pointer is MOE_ERR_ARG, a plan whose scratch exceeds the
    16 MiB array is MOE_ERR_CAPACITY."""
    L = _lib.load()
    code = ctypes.c_int(-1)
    assert L.moe_get_device_error_static(None, None, ctypes.byref(code)) == 1
    p = moe.moe_plan(8, 256, 128, 2, 4, moe.MOE_W4A8_MXFP4, 7.0, 0)
    assert L.moe_get_device_error_static(ctypes.c_void_p(p), None, None) == 1
    big = moe.moe_plan(16, 1280, 192, 4, 4096, moe.MOE_W4A8_MXFP4, 7.0, 1)
    assert moe.moe_scratch_bytes(big) > 16 << 20
    assert L.moe_get_device_error_static(ctypes.c_void_p(big), None, ctypes.byref(code)) == 4
    assert code.value == -1                     # nothing written on error
    moe.moe_destroy_plan(p)
    moe.moe_destroy_plan(big)


def test_16bit_modes_refuse_shapes_without_tensor_core_kernels(lib):
    """The 16-bit-operand modes run on tensor-core kernels whose fc2 K stages are 256 wide, so
    round_up(I, 128) must be a multiple of 256; other shapes are refused when planned (no silent
    switch to another kernel family).  The CUDA-core backend is an explicit cross-check for the
    supported shapes only."""
    for q in (moe.MOE_W4A16_NVFP4, moe.MOE_W4A16_HYBRID, moe.MOE_W4A16_HYBRID_MX,
              moe.MOE_W4A8_NVFP4, moe.MOE_W4A4_NVFP4):
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_plan(16, 1280, 576, 4, 8, q, math.inf, 0)     # Ip = 640
        assert ei.value.status in (2, 3), q
        p = moe.moe_plan(16, 1280, 512, 4, 8, q, math.inf, 0)      # Ip = 512
        moe.moe_destroy_plan(p)
    # W4A8 (MXFP4) has tensor-core kernels for every I % 64 == 0
    p = moe.moe_plan(16, 1280, 576, 4, 8, moe.MOE_W4A8_MXFP4, 7.0, 0)
    moe.moe_destroy_plan(p)


def test_w4a16_tiled_weight_sizes(lib):
    """NVFP4 and NF3 tiers are stored in tiles of 128 rows x 256 K per matrix: no padding at the
    config's shapes (I = 512, H = 6144), zero padding up to whole tiles otherwise."""
    E, H, I = 8, 6144, 512
    wp = moe.moe_plan_weights(E, H, I, moe.MOE_W4A16_NVFP4)
    codes = E * (2 * I * H // 2 + H * I // 2)
    scales = E * (2 * I * H // 16 + H * I // 16)
    assert codes + scales <= moe.moe_prepared_bytes(wp) <= codes + scales + 8 * 256 + 2 * E * 4
    moe.moe_destroy_weight_plan(wp)
    # I = 192: the fc1 row blocks (2 of 128 per half) and fc2's K (Ip = 256: one tile) padded
    wp = moe.moe_plan_weights(E, 1280, 192, moe.MOE_W4A16_NVFP4)
    tiles = E * (2 * 2 * 5 + 10 * 1)
    assert moe.moe_prepared_bytes(wp) >= tiles * (16384 + 2048)
    moe.moe_destroy_weight_plan(wp)


def test_launch_counts(lib):
    """Launches per call: calls of at most 256 flat slots route and quantise (or convert) in one
    launch; larger W4A8 calls, and other tensor-core calls beyond 4096 slots, in three (chunk
    counts, stable scatter, quantisation or conversion), other larger calls in two; then fc1,
    fc2, finalize.  The CUDA-core backend routes and converts in two and adds the SwiGLU
    launch."""
    p = moe.moe_plan(384, 7168, 576, 6, 4096, moe.MOE_W4A8_MXFP4, 7.0, 0)
    assert moe.moe_call_launches(p, 0) == 0
    assert moe.moe_call_launches(p, 16) == 4            # 96 slots
    assert moe.moe_call_launches(p, 42) == 4            # 252 slots
    assert moe.moe_call_launches(p, 43) == 6            # 258 slots
    assert moe.moe_call_launches(p, 4096) == 6
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_call_launches(p, 4097)
    assert ei.value.status == 4
    moe.moe_destroy_plan(p)
    p = moe.moe_plan(256, 6144, 512, 8, 64, moe.MOE_W4A16_NVFP4, float("inf"), 0)
    assert moe.moe_call_launches(p, 8) == 4             # 64 slots
    assert moe.moe_call_launches(p, 64) == 5            # 512 slots: one routing launch
    moe.moe_plan_set_backend(p, 1)
    assert moe.moe_call_launches(p, 8) == 6             # route, convert, fc1, act, fc2, finalize
    moe.moe_destroy_plan(p)
    p = moe.moe_plan(256, 6144, 512, 8, 1024, moe.MOE_W4A16_NVFP4, float("inf"), 0)
    assert moe.moe_call_launches(p, 512) == 5           # 4096 slots: one routing launch
    assert moe.moe_call_launches(p, 513) == 6           # 4104 slots: counts, scatter, conversion
    moe.moe_destroy_plan(p)



def test_expert_offset_arguments(lib):
    """The expert offset of an expert-parallel plan: any first id with first + E within int32;
    negative or overflowing offsets are argument errors."""
    p = moe.moe_plan(192, 7168, 1152, 6, 512, moe.MOE_W4A8_MXFP4, 7.0, 0)
    moe.moe_plan_set_expert_offset(p, 0)
    moe.moe_plan_set_expert_offset(p, 192)
    moe.moe_plan_set_expert_offset(p, 2**31 - 1 - 192)
    for bad in (-1, 2**31 - 192):
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_plan_set_expert_offset(p, bad)
        assert ei.value.status == 1
    moe.moe_destroy_plan(p)


def test_wait_probe_arguments(lib):
    """The device wait probe (a test hook): 0 turns it off, up to 1 s is accepted, more is an
    argument error, and a null plan is refused."""
    p = moe.moe_plan(8, 256, 128, 1, 16, moe.MOE_W4A8_MXFP4, 7.0, 0)
    moe.moe_plan_set_wait_probe(p, 2_000_000)
    moe.moe_plan_set_wait_probe(p, 1_000_000_000)
    moe.moe_plan_set_wait_probe(p, 0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_set_wait_probe(p, 1_000_000_001)
    assert ei.value.status == 1
    moe.moe_destroy_plan(p)
    assert lib.moe_plan_set_wait_probe(None, 0) == 1


def test_router_weight_on_input_arguments(lib):
    """Router weights on the input: 16-bit activation modes only (the pages refuse W4A8 too)."""
    p = moe.moe_plan(8, 256, 128, 1, 16, moe.MOE_W4A8_MXFP4, 7.0, 0)
    moe.moe_plan_set_router_weight_on_input(p, 0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_set_router_weight_on_input(p, 1)
    assert ei.value.status == 3
    moe.moe_destroy_plan(p)
    p = moe.moe_plan(8, 256, 256, 1, 16, moe.MOE_W4A16_NVFP4, float("inf"), 0)
    moe.moe_plan_set_router_weight_on_input(p, 1)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_set_router_weight_on_input(p, 2)
    assert ei.value.status == 1
    moe.moe_destroy_plan(p)


def test_nvfp4_a8_mode_limits(lib):
    """NVFP4 weights with MXFP8 activations: the tensor-core backend only, with round_up(I, 128)
    a multiple of 256; the activation global scales are part of the prepared buffer."""
    wp = moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A8_NVFP4)
    wp16 = moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A16_NVFP4)
    assert moe.moe_prepared_bytes(wp) == moe.moe_prepared_bytes(wp16) + 2 * 256
    moe.moe_destroy_weight_plan(wp)
    moe.moe_destroy_weight_plan(wp16)
    p = moe.moe_plan(8, 256, 256, 2, 16, moe.MOE_W4A8_NVFP4, float("inf"), 0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_set_backend(p, 1)
    assert ei.value.status == 3
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_set_router_weight_on_input(p, 1)
    assert ei.value.status == 3
    moe.moe_destroy_plan(p)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan(8, 256, 128, 2, 16, moe.MOE_W4A8_NVFP4, float("inf"), 0)   # Ip = 128
    assert ei.value.status == 2


def test_w4a4_mode_limits(lib):
    """NVFP4 weights with NVFP4 activations: the FP4 tensor-core kernels only; the prepared
    buffer holds the NVFP4 sections (scales in the kernels' atom layout, the same size) and the
    activation global scales."""
    wp = moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A4_NVFP4)
    wp8 = moe.moe_plan_weights(4, 256, 128, moe.MOE_W4A8_NVFP4)
    assert moe.moe_prepared_bytes(wp) == moe.moe_prepared_bytes(wp8)
    moe.moe_destroy_weight_plan(wp)
    moe.moe_destroy_weight_plan(wp8)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan(8, 256, 128, 2, 256, moe.MOE_W4A4_NVFP4, float("inf"), 0)   # Ip = 128
    assert ei.value.status == 3
    p = moe.moe_plan(8, 256, 256, 2, 256, moe.MOE_W4A4_NVFP4, float("inf"), 0)
    assert moe.moe_call_launches(p, 16) == 4            # 32 slots: one routing launch
    assert moe.moe_call_launches(p, 200) == 5           # 400 slots: routing, quantisation
    for setter, arg in ((moe.moe_plan_set_backend, 1),
                        (moe.moe_plan_set_router_weight_on_input, 1)):
        with pytest.raises(moe.MoEError) as ei:
            setter(p, arg)
        assert ei.value.status == 3
    moe.moe_destroy_plan(p)


def test_binding_constants_match_header(lib):
    """The binding's enum constants and the checkpoint struct follow include/moe_gb300.h."""
    import os
    import re
    from serving_route_count_gb300 import _lib
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "moe_gb300.h")).read()
    for name, val in re.findall(r"\b(MOE_W4A\w+|MOE_W13_\w+)\s*=\s*(\d+)", hdr):
        assert getattr(moe, name) == int(val), name
    body = re.search(r"typedef struct \{(.*?)\} moe_checkpoint;", hdr, re.S).group(1)
    fields = re.findall(r"\*\s*(\w+);", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
    assert fields == [f for f, _ in _lib.MoeCheckpoint._fields_]


def test_kept_a8_arguments(lib):
    """The MXFP4 kept tier's A8 opt-in: hybrid-MX plans only; both scales positive with finite
    nonzero fp32 reciprocals, or both 0 (off); refused beside router weights on the input and
    the CUDA-core backend, in either order."""
    p = moe.moe_plan(8, 256, 256, 2, 16, moe.MOE_W4A16_HYBRID_MX, float("inf"), 0)
    moe.moe_plan_set_kept_a8(p, 0.011, 0.018)
    moe.moe_plan_set_kept_a8(p, 0.0, 0.0)
    for a, b in ((-0.01, 0.02), (float("nan"), 0.02), (0.01, float("inf")), (1e-40, 0.02),
                 (0.01, 0.0), (0.0, 0.02)):
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_plan_set_kept_a8(p, a, b)
        assert ei.value.status == 1, (a, b)
    moe.moe_plan_set_kept_a8(p, 0.011, 0.018)
    for call in (lambda: moe.moe_plan_set_backend(p, 1),
                 lambda: moe.moe_plan_set_router_weight_on_input(p, 1)):
        with pytest.raises(moe.MoEError) as ei:
            call()
        assert ei.value.status == 3
    moe.moe_plan_set_kept_a8(p, 0.0, 0.0)
    moe.moe_plan_set_backend(p, 1)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_plan_set_kept_a8(p, 0.011, 0.018)
    assert ei.value.status == 3
    moe.moe_destroy_plan(p)
    for mode in (moe.MOE_W4A8_MXFP4, moe.MOE_W4A16_NVFP4, moe.MOE_W4A16_HYBRID):
        q = moe.moe_plan(8, 256, 256, 2, 16, mode, float("inf"), 0)
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_plan_set_kept_a8(q, 0.011, 0.018)
        assert ei.value.status == 3
        moe.moe_destroy_plan(q)
    assert lib.moe_plan_set_kept_a8(None, ctypes.c_float(0.0), ctypes.c_float(0.0)) == 1
