/*
 * moe_gb300.h - C ABI of the GB300 (sm_103a) routed mixture-of-experts expert computation.
 *
 *   out[t] = sum_j w[t,j] * expert_{id[t,j]}(x[t]),
 *   expert(x) = W2 . act(gate, up),  [up; gate] = W13 . x   (fc1, SwiGLU, fc2)
 *
 * Sources (web pages on the routed-MoE serving path):
 *   - "moe_b12x_next.py" (sglang adapter, docker-images/mia-tp4): module docstring (W4A8 =
 *     MXFP4 weights + in-kernel MXFP8 activations; w13 stacked [w3 (up); w1 (gate)]; ids
 *     outside [0, E) skipped, padding rows give 0; deterministic combine = per-slot route
 *     buffer + top-k sum), class _Geometry (plan_weights -> prepare_weights -> plan_execution
 *     -> bind -> run), _convert_layer (checkpoint shapes).
 *   - "hybrid_loader.py" (vLLM, docker-images/glm52-nf3-hybrid): NVFP4 / NF3 tiers, _unpack_nf3,
 *     _apply_ref (reference two-pass forward), the union staging + single top-k sum.
 *   - vLLM API page "fused_moe/b12x", class B12xExperts: _prepare_experts, _swiglu_params,
 *     apply.
 *
 * Conventions for every entry point:
 *   - All tensors are contiguous row-major.  Device pointers are CUDA device memory of the
 *     current device; "host" pointers are ordinary host memory.  The library never allocates
 *     device memory: the caller owns the prepared-weight buffer and the scratch buffer and
 *     passes their sizes (obtained from the *_bytes queries).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Calls return a moe_status; nothing is printed.  On error no kernel was launched unless the
 *     status is MOE_ERR_CUDA (a launch or copy failed; cudaGetLastError was cleared).
 *   - Handles are opaque host objects; destroy them with the matching moe_destroy_* call.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,          /* null pointer, negative size, buffer too small            */
  MOE_ERR_SHAPE = 2,        /* E/H/I/top-k outside what the kernels support             */
  MOE_ERR_UNSUPPORTED = 3,  /* quant mode / option combination not supported            */
  MOE_ERR_CAPACITY = 4,     /* M > max_m of the plan                                    */
  MOE_ERR_CAPTURING = 5,    /* planning / preparing while the stream is being captured  */
  MOE_ERR_CUDA = 6,         /* a CUDA runtime call failed                               */
  MOE_ERR_TIMEOUT = 7,      /* a bounded device-side wait gave up (see moe_get_device_error) */
  MOE_ERR_DEVICE = 8        /* a device-side check failed (see moe_get_device_error)    */
} moe_status;

typedef enum {
  /* MXFP4 weights (E2M1 + E8M0 per 32 along K), activations quantised in-kernel to MXFP8
   * (E4M3 + E8M0 per 32); "W4A8" of moe_b12x_next.py, module docstring. */
  MOE_W4A8_MXFP4 = 0,
  /* NVFP4 weights (E2M1 + E4M3 per 16 + one fp32 global per expert and matrix), bf16
   * activations; the kept tier of hybrid_loader.py (`_build_kept_b12x`, use_a16). */
  MOE_W4A16_NVFP4 = 1,
  /* Per-expert tier map: NVFP4 (tier 4) or NF3 (tier 3, 8-entry LUT x E4M3 per 32), bf16
   * activations, both tiers summed by one top-k sum (hybrid_loader.py, class docstring and
   * the union-staging path of `_apply_b12x_nf3`). */
  MOE_W4A16_HYBRID = 2,
  /* The same tier map with the kept tier in MXFP4 (E2M1 + UE8M0 per 32, no global scale) and
   * bf16 activations: hybrid_loader.py "v3" kept format `mxfp4_e8m0k32` (`create_weights`,
   * `_build_kept_mxfp4`, A16 default).  Prepare turns each UE8M0 scale 2^(b-127) into an f16
   * multiplier 2^(b - b_max + 13) with b_max the largest scale byte of the expert's matrix and
   * moves 2^(b_max - 140) into a per-matrix fp32 factor, so E2M1 x multiplier is exact in f16
   * for every group within 36 binades of the matrix's largest scale (groups further below are
   * flushed to zero: their terms are < 2^-34 of the matrix's largest weights). */
  MOE_W4A16_HYBRID_MX = 3,
  /* NVFP4 weights (as MOE_W4A16_NVFP4) with MXFP8 activations: B12xExperts quant mode
   * "w4a8_nvfp4" (`_supports_quant_scheme`: kNvfp4Static weights, kMxfp8Dynamic activations;
   * `_prepare_experts`: it needs the per-expert activation global scales a1_gscale / a2_gscale).
   * Each slot's fc1 input is MXFP8(a1[e] * x) / a1[e] (OCP MX rule on the fp32 products) and
   * fc2's is MXFP8(a2[e] * h) / a2[e]; runs on the tensor-core backend only, with
   * round_up(I, 128) a multiple of 256. */
  MOE_W4A8_NVFP4 = 4,
  /* NVFP4 weights with NVFP4 activations (W4A4): B12xExperts quant mode "nvfp4"
   * (kNvfp4Static weights x kNvfp4Dynamic activations; per-expert activation global scales
   * a1_gscale / a2_gscale required).  Each slot's fc1 input is NVFP4(a1[e] * x) / a1[e] and
   * fc2's NVFP4(a2[e] * h) / a2[e]: blocks of 16 with the E4M3 scale nearest vmax / 6 and E2M1
   * codes nearest-even of v / scale, in fp32.  Runs on block-scaled FP4 tensor-core kernels
   * (tcgen05 kind::mxf4nvf4) only, with H and round_up(I, 128) multiples of 256. */
  MOE_W4A4_NVFP4 = 5
} moe_quant_mode;

typedef enum {
  MOE_W13_UP_GATE = 0,  /* fc1 rows [w3 (up); w1 (gate)]: moe_b12x_next.py docstring       */
  MOE_W13_GATE_UP = 1   /* fc1 rows [w1 (gate); w3 (up)]: hybrid_loader.py weight_loader    */
} moe_w13_layout;

#define MOE_TIER_NVFP4 4
#define MOE_TIER_NF3 3

typedef struct moe_weight_plan moe_weight_plan;
typedef struct moe_prepared moe_prepared;
typedef struct moe_plan_s moe_plan_t;

/* Checkpoint-layout expert tensors (device pointers, contiguous), as listed by
 * moe_b12x_next.py `_convert_layer` (MXFP4) and hybrid_loader.py `create_weights` (NVFP4 / NF3).
 * For MOE_W4A16_HYBRID the fp4 fields hold the NVFP4 tier compacted over its experts (in
 * ascending expert id) and the nf3 fields the NF3 tier likewise; for MOE_W4A16_HYBRID_MX the
 * fp4 fields hold the kept tier in the MXFP4 layout below (compacted the same way).
 *   MXFP4: w13 [E, 2I, H/2] u8 (element 2j = low nibble of byte j), s13 [E, 2I, H/32] u8 E8M0,
 *          w2 [E, H, I/2] u8, s2 [E, H, I/32] u8 E8M0; g13 = g2 = NULL.
 *   NVFP4 (W4A16, W4A8_NVFP4, W4A4):
 *          w13 [E4, 2I, H/2], s13 [E4, 2I, H/16] u8 E4M3, g13 [E4] f32,
 *          w2 [E4, H, I/2],   s2 [E4, H, I/16] u8 E4M3,  g2 [E4] f32.
 *   NF3:   nf_w13 [E3, 2I, 3H/8] u8 (8 codes per 3 bytes, hybrid_loader.py _unpack_nf3),
 *          nf_s13 [E3, 2I, H/32] u8 E4M3, nf_w2 [E3, H, 3I/8] u8, nf_s2 [E3, H, I/32] u8 E4M3. */
typedef struct {
  const void* w13;
  const void* s13;
  const float* g13;
  const void* w2;
  const void* s2;
  const float* g2;
  const void* nf_w13;
  const void* nf_s13;
  const void* nf_w2;
  const void* nf_s2;
  /* MOE_W4A8_NVFP4 only (NULL otherwise): per-expert activation global scales [E] f32 of fc1's
   * input (a1_gscale = 1 / w13_input_scale) and of fc2's input (a2_gscale). */
  const float* a1_gscale;
  const float* a2_gscale;
} moe_checkpoint;

/* Weight plan: geometry and quant mode of one layer's experts (moe_b12x_next.py,
 * `_Geometry.__init__` -> fm.plan_weights; B12xExperts `_prepare_experts`).
 *   E, H, I   experts, hidden size, intermediate size (per rank).  Requires H % 128 == 0,
 *             I % 64 == 0 (moe_b12x_next.py `create_weights` checks), E >= 1.
 *   tier_of_expert  host [E] int8 of MOE_TIER_NVFP4 (the kept 4-bit tier: NVFP4, or MXFP4
 *             for MOE_W4A16_HYBRID_MX) / MOE_TIER_NF3 for MOE_W4A16_HYBRID(_MX),
 *             NULL otherwise.  Copied; the caller keeps ownership.
 * Errors: MOE_ERR_ARG (null out), MOE_ERR_SHAPE, MOE_ERR_UNSUPPORTED. */
moe_status moe_plan_weights(int E, int H, int I, int quant_mode, int w13_layout,
                            const int8_t* tier_of_expert, moe_weight_plan** out);

/* Size in bytes of the device buffer that moe_prepare_weights fills. */
moe_status moe_prepared_bytes(const moe_weight_plan* wp, size_t* bytes);

/* Repack checkpoint bytes into the device layout the kernels read (moe_b12x_next.py module
 * docstring: "the checkpoint bytes are repacked ... into ... PreparedExperts"; B12xExperts
 * `_prepare_experts`, incl. the FP4 zero-sign canonicalisation -0 -> +0).
 *   src       device checkpoint tensors (read only; not modified).
 *   dst       device buffer of at least moe_prepared_bytes bytes, 256-byte aligned; owned by the
 *             caller and referenced (not copied) by the returned handle, so it must outlive it.
 *   stream    the repack kernels run on it; the handle is usable by moe_run on the same stream
 *             right away (stream order).
 * Errors: MOE_ERR_ARG, MOE_ERR_CAPTURING (stream is capturing: B12xExperts refuses to
 * prepare under graph capture), MOE_ERR_CUDA. */
moe_status moe_prepare_weights(const moe_weight_plan* wp, const moe_checkpoint* src, void* dst,
                               size_t dst_bytes, void* stream, moe_prepared** out);

/* Execution plan for calls of up to max_m tokens (moe_b12x_next.py `_Geometry.build`:
 * fm.plan_execution per capacity; knob _DETERMINISTIC).
 *   topk          router top-k (1..16).
 *   max_m         capacity; moe_run with M > max_m returns MOE_ERR_CAPACITY.
 *   swiglu_limit  clamp of the SwiGLU (gate' = min(gate, L), up' = clamp(up, -L, L)); +inf for
 *                 no clamp.  alpha = 1, beta = 0 unless set with moe_plan_set_swiglu_alpha_beta.
 *   deterministic 0: fp32 atomic combine (run-to-run ulp differences possible);
 *                 1: per-slot route buffer + fixed-order top-k sum (bit-stable).
 * Shapes: the 16-bit-operand modes (W4A16 NVFP4, the hybrids, MOE_W4A8_NVFP4) need
 * round_up(I, 128) to be a multiple of 256 (their tensor-core fc2 runs 256-wide K stages);
 * W4A4 needs that and H % 256 == 0.  Other shapes are refused, never run on another kernel
 * family.
 * Errors: MOE_ERR_ARG, MOE_ERR_SHAPE, MOE_ERR_UNSUPPORTED. */
moe_status moe_plan(int E, int H, int I, int topk, int max_m, int quant_mode, float swiglu_limit,
                    int deterministic, moe_plan_t** out);

/* Optional alpha / beta of the clamped SwiGLU, h = gate' * sigmoid(alpha gate') * (up' + beta)
 * (B12xExperts `_swiglu_params`, SWIGLUOAI form). */
moe_status moe_plan_set_swiglu_alpha_beta(moe_plan_t* plan, float alpha, float beta);

/* Kernel family for later moe_run calls: 0 (default) = the tcgen05 tensor-core GEMMs (every mode
 * and shape moe_plan admits has them); 1 = CUDA-core GEMMs (a slower, independent path kept only
 * as an explicit cross-check; W4A16 NVFP4, the hybrids and W4A8 only).
 * Errors: MOE_ERR_ARG, MOE_ERR_UNSUPPORTED (backend 1 for MOE_W4A8_NVFP4 / MOE_W4A4_NVFP4). */
moe_status moe_plan_set_backend(moe_plan_t* plan, int backend);

/* fc1 kernel of the W4A8 tensor-core path at the 16-token tile width (calls with M <= 16):
 *   0 (default) automatic: the persistent stream-K kernel (the routed units' K tiles split
 *     evenly over all CTA slots) whenever its schedule fits (H / 128 < 130), else one
 *     (tile, row block) unit per CTA, split along K for small calls;
 *   1 always the unit-per-CTA kernel;  2 the stream-K kernel wherever its schedule fits.
 * Both give results within the same tolerance of the method (in deterministic mode each is
 * bit-stable on its own; the two differ in the rounding order of fc1's K sum).
 * Errors: MOE_ERR_ARG. */
moe_status moe_plan_set_fc1_kernel(moe_plan_t* plan, int choice);

/* Router weights on the input (B12xExperts `process_weights_after_loading`:
 * `apply_router_weight_on_input`, W4A16 only): on = 1 makes each slot's fc1 input
 * bf16(x * bf16(w)) (the weight cast to the activations' dtype and multiplied in it) and adds
 * the expert outputs with weight 1; on = 0 (default) weights the outputs.
 * Errors: MOE_ERR_ARG (plan NULL, on not 0/1), MOE_ERR_UNSUPPORTED (on = 1 for W4A8, which
 * the pages refuse too). */
moe_status moe_plan_set_router_weight_on_input(moe_plan_t* plan, int on);

/* A8 opt-in of the MXFP4 kept tier (hybrid_loader.py `_build_kept_mxfp4`: `HYBRID_MX_A8`
 * selects static per-tensor symmetric FP8 activations for the kept experts, with the layer's
 * `w13_input_scale` / `w2_input_scale`).  MOE_W4A16_HYBRID_MX plans only.  With both scales
 * > 0, each kept-tier slot's fc1 input is E4M3(fp32(x) * fp32(1 / w13_input_scale)) (nearest
 * even, saturating at +-448) times w13_input_scale, and its fc2 input the same of the fp32
 * SwiGLU output with w2_input_scale; the NF3 experts keep bf16 activations.  Both scales 0
 * turns it off (default).  Errors: MOE_ERR_ARG (plan NULL; a scale negative, NaN, infinite, or
 * one whose fp32 reciprocal is not finite and nonzero; one scale 0 and not the other),
 * MOE_ERR_UNSUPPORTED (another mode, router weights on the input, or the CUDA-core backend:
 * moe_plan_set_backend(plan, 1) and moe_plan_set_router_weight_on_input(plan, 1) are refused
 * the same way while it is on). */
moe_status moe_plan_set_kept_a8(moe_plan_t* plan, float w13_input_scale, float w2_input_scale);

/* Expert parallelism (moe_b12x_next.py `ep_remap` / `ep_remap_reference`): this plan's E
 * experts are the global experts [first_expert, first_expert + E).  topk_ids then hold global
 * ids; routing maps each to its local id (id - first_expert) on the device, and ids of other
 * ranks' experts (and padding) contribute nothing to out.  The adapter's remap gives such slots
 * weight 0 and some local expert; a weight-0 term adds an exact 0 to every output sum, so
 * dropping the slot gives the same out and skips its GEMM rows.  Default 0 (ids are local).
 * Errors: MOE_ERR_ARG (plan NULL, first_expert < 0 or first_expert + E > INT32_MAX). */
moe_status moe_plan_set_expert_offset(moe_plan_t* plan, int first_expert);

/* Test hook: on = 1 makes small W4A8 calls (at most 256 flat slots, tiles of <= 32 tokens),
 * whose fc1 quantises the activations itself stage by stage, also store the MXFP8 codes and
 * scales where moe_debug_actq reads them (other calls always do).  Default 0.
 * Errors: MOE_ERR_ARG. */
moe_status moe_plan_set_debug_copies(moe_plan_t* plan, int on);

/* Test hook for the device-side failure path: with ns > 0, the W4A8 fc1 kernel that runs one
 * (tile, row block) unit per CTA (calls whose units fit one wave) first makes its MMA issuer wait
 * up to ns nanoseconds on a barrier that no thread ever arrives on.  The wait runs out, sets the
 * timeout bit of the call's device error word (moe_get_device_error then returns
 * MOE_ERR_TIMEOUT), and the CTA stops issuing work, waits (with the normal 1 s bound) for the
 * copies it has in flight and returns: the call's output is then undefined, and the context and
 * the plan stay usable.  ns = 0 (default) turns it off.  Errors: MOE_ERR_ARG (ns > 1 s). */
moe_status moe_plan_set_wait_probe(moe_plan_t* plan, unsigned long long ns);

/* Size in bytes of the device scratch buffer moe_run needs (routing tables, quantised
 * activations, the fc1 -> fc2 intermediate, the combine buffer). */
moe_status moe_scratch_bytes(const moe_plan_t* plan, size_t* bytes);

/* One MoE layer call (moe_b12x_next.py `_Geometry._run` -> fm.run; hybrid_loader.py
 * run_w4a16_moe; B12xExperts `apply`).  All pointers are device memory:
 *   x            [M, H] bf16 hidden states.
 *   topk_ids     [M, topk] int32; ids outside [0, E) (e.g. -1 padding) contribute nothing.
 *   topk_weights [M, topk] fp32.
 *   out          [M, H] bf16, fully overwritten (rows without a valid id become 0).
 *   scratch      >= moe_scratch_bytes bytes, 256-byte aligned; its contents need no
 *                initialisation and are clobbered.  Calls that share a scratch buffer must be
 *                stream-ordered.
 * No host synchronisation and no allocation: the call can be captured in a CUDA graph.
 * M == 0 is a no-op.  Errors: MOE_ERR_ARG, MOE_ERR_CAPACITY, MOE_ERR_CUDA. */
moe_status moe_run(const moe_plan_t* plan, const moe_prepared* weights, void* scratch,
                   size_t scratch_bytes, const void* x, const int32_t* topk_ids,
                   const float* topk_weights, void* out, int M, void* stream);

/* moe_run for any M >= 0 (moe_b12x_next.py `_Geometry.forward`: the host loop over row chunks of
 * the largest capacity).  Rows [s, s + max_m) run as one moe_run each, in order, on the same
 * scratch and stream; every row's result is the one a single call of its chunk gives (so in
 * deterministic mode bit-identical to those calls).  Pointers, alignment and errors as moe_run;
 * the first failing chunk's status is returned and later chunks are not launched.  Graph
 * capture works as for moe_run. */
moe_status moe_run_chunked(const moe_plan_t* plan, const moe_prepared* weights, void* scratch,
                           size_t scratch_bytes, const void* x, const int32_t* topk_ids,
                           const float* topk_weights, void* out, int M, void* stream);

/* moe_run without a caller-provided scratch buffer (the pages have no counterpart of this entry
 * point).  It is for callers that cannot allocate device memory: code running under another
 * framework's memory pool with no allocator exposed to plug-ins, sandboxed or embedded runtimes
 * where cudaMalloc is unavailable after start-up, and paths that must never allocate.  The
 * scratch is a 16 MiB array compiled into the library (a file-scope __device__ variable): every
 * GPU that loads the library holds it until the process exits.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library call.
 *   Arguments as moe_run, without scratch.  Plans whose moe_scratch_bytes exceeds 16 MiB are
 *   rejected with MOE_ERR_CAPACITY (e.g. decode batches of the E=384, H=7168, I=576, top-6 layer
 *   fit: 11.7 MiB atomic / 13.8 MiB deterministic at max_m = 16, 10 MiB of it the fixed
 *   partial-sum slots of the persistent W4A8 fc1).
 *   The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *   that device current) and caches it; make that first call before any stream capture.
 *   All calls on a device share the array and it keeps the last call's contents; calls whose
 *   executions overlap on the GPU (other streams, other host threads) race on it and must be
 *   serialised by the caller.  Errors: as moe_run, plus MOE_ERR_CAPACITY as above. */
moe_status moe_run_static_scratch(const moe_plan_t* plan, const moe_prepared* weights,
                                  const void* x, const int32_t* topk_ids,
                                  const float* topk_weights, void* out, int M, void* stream);

/* moe_get_device_error for calls made with moe_run_static_scratch (no counterpart on the pages):
 * the device error word of those calls lives in the library's own array, which the caller cannot
 * name, so this reads (and clears) it there.  Synchronises `stream`.  *code = 0 when no
 * device-side check failed since the last read; the status is MOE_ERR_TIMEOUT / MOE_ERR_DEVICE
 * as for moe_get_device_error.  Like the run call it shares the array with every other static
 * call on the device: read it before the next call overwrites it.  The cached array address
 * assumes the device's primary context lives as long as the process (as for the run call).
 * Errors: MOE_ERR_ARG, MOE_ERR_CAPACITY (a plan the array cannot hold), MOE_ERR_CUDA. */
moe_status moe_get_device_error_static(const moe_plan_t* plan, void* stream, int* code);

/* Size of the device staging buffer moe_run_host needs (x, ids, weights and out of max_m rows). */
moe_status moe_io_bytes(const moe_plan_t* plan, size_t* bytes);

/* moe_run with HOST inputs and output: copies x / ids / weights host -> device into `io`
 * (>= moe_io_bytes, device), runs the layer, copies out device -> host and synchronises the
 * stream before returning.  Pinned host memory makes the copies asynchronous DMA.  When the
 * inputs sit back to back in one host buffer (ids_host = x_host + M*H*2 bytes, w_host =
 * ids_host + M*topk*4 bytes) they go up in one copy.  When out_host is page-locked memory the
 * device can address (cudaHostAlloc / cudaMallocHost under unified addressing, 16-byte aligned)
 * the finalize kernel writes the output rows into it directly and no device -> host copy is
 * made; the io buffer's output rows are then left untouched. */
moe_status moe_run_host(const moe_plan_t* plan, const moe_prepared* weights, void* scratch,
                        size_t scratch_bytes, void* io, size_t io_bytes, const void* x_host,
                        const int32_t* ids_host, const float* w_host, void* out_host, int M,
                        void* stream);

/* Test hook: the inverse of moe_prepare_weights, on the host.  Copies the prepared buffer of `w`
 * back (synchronises `stream`) and writes the checkpoint-layout tensors of the plan's mode into
 * the HOST buffers named by `dst` (the moe_checkpoint fields and shapes; the pointers are
 * written through): codes (E2M1 nibbles after the -0 -> +0 rewrite), block scales, NF3 codes
 * and scales, the NVFP4 globals and activation global scales where the mode has them (g13 /
 * g2 are not written for the MXFP4 kept tier, whose checkpoint has none; a kept-tier scale
 * that prepare flushed comes back as 0).  Errors: MOE_ERR_ARG, MOE_ERR_CUDA. */
moe_status moe_unprepare_weights(const moe_weight_plan* wp, const moe_prepared* w, void* stream,
                                 const moe_checkpoint* dst);

/* Reads and clears the device error word kept in `scratch` (synchronises `stream`).
 * *code = 0 when no device-side check failed since the last read. */
moe_status moe_get_device_error(const moe_plan_t* plan, void* scratch, void* stream, int* code);

/* Test hooks: after a moe_run on `stream`, copy routing tables / quantised activations of the
 * last call to host buffers (synchronises; the activations of small W4A8 calls only with
 * moe_plan_set_debug_copies on).  cnt [E], off [E+1], perm [S], slot_of [M*topk]
 * where S = off[E]; xq [S, H] E4M3 codes, xs [S, H/32] E8M0 bytes (W4A8 only), row p holding
 * the quantised row of token perm[p] / topk (buffers of M*topk rows suffice). */
moe_status moe_debug_routing(const moe_plan_t* plan, void* scratch, int M, int32_t* cnt,
                             int32_t* off, int32_t* perm, int32_t* slot_of, void* stream);
moe_status moe_debug_actq(const moe_plan_t* plan, void* scratch, int M, uint8_t* xq, uint8_t* xs,
                          void* stream);

/* Profiling hook.  With n_events >= 1 set, every later moe_run with this plan records
 * events[0] before its first kernel and events[i + 1] after stage i (up to n_events - 1 stages;
 * events are cudaEvent_t handles created by the caller with timing enabled).  Inside stream
 * capture the records become event-record nodes of the graph (cudaEventRecordExternal), so
 * graph replays time each stage on the device.  n_events = 0 turns it off.
 * moe_profile_stage_names returns the stage names of this plan's launch sequence, comma
 * separated, e.g. "route,actq,fc1,act,fc2,finalize". */
moe_status moe_plan_set_profile_events(moe_plan_t* plan, void* const* events, int n_events);
const char* moe_profile_stage_names(const moe_plan_t* plan);

/* Number of kernel launches moe_run makes for a call of M tokens with this plan and backend
 * (routing and activation quantisation or conversion - one launch for tensor-core calls of at
 * most 256 slots, three for larger W4A8 calls and for other tensor-core calls beyond 4096 slots,
 * two otherwise -, fc1, [SwiGLU on the CUDA-core path], fc2, finalize).  0 for M = 0.
 * Errors: MOE_ERR_ARG, MOE_ERR_CAPACITY (M > max_m). */
moe_status moe_call_launches(const moe_plan_t* plan, int M, int* launches);

/* Test hook: the fc2 activation operand of the last call in slot order (synchronises).
 * W4A8: hq [S, Ip] E4M3 codes and hs [S, Ip/32] E8M0 bytes (Ip = I rounded up to 128; columns
 * >= I are zero).  W4A4: hq [S, Ip/2] packed E2M1 codes and hs [S, Ip/16] E4M3 scales.
 * Other modes: hq receives [S, Ip] f16 values (bf16-rounded h, or the MXFP8 values of a2 * h
 * for MOE_W4A8_NVFP4), hs is not written.
 * Buffers of M*topk rows suffice. */
moe_status moe_debug_h(const moe_plan_t* plan, void* scratch, int M, void* hq, uint8_t* hs,
                       void* stream);

void moe_destroy_weight_plan(moe_weight_plan* wp);
void moe_destroy_prepared(moe_prepared* p);
void moe_destroy_plan(moe_plan_t* plan);
const char* moe_status_str(moe_status s);
/* Library version string, e.g. "moe_gb300 0.1 sm_103a". */
const char* moe_version(void);
/* Name of the CUDA error behind the last MOE_ERR_CUDA returned to this host thread (e.g.
 * "cudaErrorInvalidValue"), or "cudaSuccess" when there was none. */
const char* moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
