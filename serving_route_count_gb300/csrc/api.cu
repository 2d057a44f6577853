// api.cu - host implementation of the C ABI declared in include/moe_gb300.h: plans, buffer
// sizing, argument checks and the launch sequence of one MoE call.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "moe_common.cuh"
#include "tc_sched.cuh"
#include "tc_tile.cuh"
#include "../../include/moe_gb300.h"

namespace moe {
// route.cu
cudaError_t launch_route(const int32_t* ids, int Mk, int E, int ep_first, int tile_slots,
                         int max_tiles, const RunPtrs& r, cudaStream_t st);
cudaError_t launch_actq16_rows(const void* x, int M, int H, int topk, const RunPtrs& r,
                               const float* win, const int32_t* ids, int ep_first, int E,
                               void* z0, size_t z0_words, void* z1, size_t z1_words, void* z2,
                               size_t z2_words, KeptA8 ka8, cudaStream_t st);
cudaError_t launch_actq(const void* x, int M, int H, int topk, const RunPtrs& r, bool quant_x,
                        bool atoms, bool to_f16, const float* win, const float* ag,
                        const int32_t* ids, int ep_first, int E, bool nv4, void* z0,
                        size_t z0_words, void* z1, size_t z1_words, void* z2, size_t z2_words,
                        KeptA8 ka8, cudaStream_t st);
bool route_actq_small_supported(int Mk, int E);
int route_chunks(int Mk);
cudaError_t launch_route_count(const int32_t* ids, int Mk, int E, int ep_first,
                               const RunPtrs& r, cudaStream_t st);
cudaError_t launch_route_scatter(const int32_t* ids, int Mk, int E, int ep_first, int tile_slots,
                                 int max_tiles, const RunPtrs& r, cudaStream_t st);
cudaError_t launch_actq_rows(const void* x, int M, int H, int topk, const RunPtrs& r, void* z0,
                             size_t z0_words, void* z1, size_t z1_words, void* z2,
                             size_t z2_words, cudaStream_t st);
cudaError_t launch_route_actq_small(const int32_t* ids, int Mk, int E, int ep_first,
                                    int tile_slots, int max_tiles, const void* x, int H, int topk,
                                    const RunPtrs& r, bool atoms, bool to_f16, const float* win,
                                    const float* ag, bool nv4, bool skip_x, void* z0,
                                    size_t z0_words, void* z1, size_t z1_words, void* z2,
                                    size_t z2_words, KeptA8 ka8, cudaStream_t st);
// gemm_tc.cu
cudaError_t launch_tc_stage(int stage, const DevWeights& w, const RunPtrs& r, const PlanDims& d,
                            int bn, int tiles, int splits, const float* topk_w, int M,
                            const int32_t* ids, int max_tiles, const void* x, cudaStream_t st);
int tc_pick_bn(int M, int topk, int E, bool w4a8);
// gemm_tc_persist.cu
bool fc1_stream_preferred(int bn, int units);
size_t fc1_stream_part_bytes();
cudaError_t launch_fc1_stream(const DevWeights& w, const RunPtrs& r, const PlanDims& d, int bn,
                              int M, float* part, int32_t* tickets, const int32_t* ids,
                              int max_tiles, const void* x, cudaStream_t st);
bool fc2_persist_preferred(int bn, int units);
cudaError_t launch_fc2_persist(const DevWeights& w, const RunPtrs& r, const PlanDims& d, int bn,
                               int M, const float* topk_w, cudaStream_t st);
// gemm_simt.cu
cudaError_t launch_simt_stage(int stage, const DevWeights& w, const RunPtrs& r,
                              const PlanDims& d, int max_tiles, const void* x,
                              const float* topk_w, void* out, int M, cudaStream_t st);
// prepare.cu
cudaError_t launch_repack_fp4_tiled(const void* src, void* dst, int E, int halves, int rows,
                                    int src_cols, int dst_cols, int layout, int pair_I,
                                    cudaStream_t st);
cudaError_t launch_repack_sf_atoms(const void* src, void* dst, int E, int halves, int rows,
                                   int kblocks, int row_tiles, int k_tiles, int layout,
                                   cudaStream_t st);
// kind: 0 NVFP4 codes, 1 NVFP4 scales, 2 NF3 codes, 3 NF3 scales
cudaError_t launch_repack_mx16_scales(const void* src, void* dst, int32_t* kmax, float* g, int E,
                                      int halves, int rows, int src_k, int K, int layout,
                                      cudaStream_t st);
cudaError_t launch_repack_w16_tiled(int kind, const void* src, void* dst, int E, int halves,
                                    int rows, int src_k, int K, int layout, cudaStream_t st);
// gemm_tc4.cu
int tc4_pick_bn(int M);
cudaError_t launch_tc4_stage(int stage, const DevWeights& w, const RunPtrs& r, const PlanDims& d,
                             int bn, int tiles, int splits, const float* topk_w, int M,
                             cudaStream_t st);
// gemm_tc16.cu
// Flat slots beyond which the 16-bit and W4A4 tensor-core calls route over many CTAs and the
// 16-bit ones convert their activations token row by token row (measured: at 16,384 slots the
// one-CTA routing launch took ~54 us and the two changes cut 5-7 % of the call; at 512 both
// cost a few microseconds)
constexpr int kChunkedRouteSlots = 4096;
bool tc16_fc1_pair(int bn, int quant);
cudaError_t launch_tc16_stage(int stage, const DevWeights& w, const RunPtrs& r, const PlanDims& d,
                              int bn, int tiles, int splits, const float* topk_w, int M,
                              cudaStream_t st);
}  // namespace moe

using namespace moe;

struct moe_weight_plan {
  int E, H, I, Ip, quant, layout;
  int E4, E3;
  std::vector<int32_t> tier_map;  // (tier << 24) | local
  // section offsets in the prepared buffer
  size_t w13, s13, w2, s2, g13, g2, mxk13, mxk2, ag13, ag2, nf_w13, nf_s13, nf_w2, nf_s2, tmap,
      total;
};

struct moe_prepared {
  DevWeights w;
};

struct moe_plan_s {
  PlanDims d;
  Scratch s;
  size_t io_x, io_ids, io_w, io_out, io_total;
  std::vector<cudaEvent_t> prof;
};

namespace {

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return false;
  return cs != cudaStreamCaptureStatusNone;
}

// the CUDA error behind the last MOE_ERR_CUDA of this host thread (moe_last_cuda_error)
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda_error = e;
  (void)cudaGetLastError();
  return MOE_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kFc1CtasPerSm = 2;

// Tiles of a call of M tokens at tile width bn: at most one per slot, and at most
// ceil(S / bn) + (touched experts).
int call_tiles(const PlanDims& d, int max_tiles, int M, int bn) {
  const int Sm = M * d.topk;
  return std::min(max_tiles, std::min(Sm, cdiv(Sm, bn) + std::min(d.E, Sm)));
}

// K splits of the tensor-core fc1 so that small calls still put one CTA on most SMs.
// SMs of the current device (152 when there is none, e.g. when plans are sized on a host
// without a GPU), looked up once.
int device_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      sms = n;
    else
      sms = 152;
    (void)cudaGetLastError();
  }
  return sms;
}

// K splits of the unit-per-CTA fc1 so that small calls still fill the CTA slots: the most
// splits that keep the grid within one wave.  W4A8: two CTAs of the decode tile width per SM,
// at least 4 K tiles of 128 per split.  W4A16: one or two CTAs per SM (tc16_fc1_pair), at least
// 2 raw stages of 256 per split (measured: splitting calls with more units than SMs into
// several waves was slower).
int fc1_splits(const PlanDims& d, int tiles, int bn) {
  const int units = std::max(1, tiles * cdiv(d.I, 128));
  const bool a8 = d.quant == MOE_W4A8_MXFP4;
  const int per_sm = (a8 || d.quant == MOE_W4A4_NVFP4) ? kFc1CtasPerSm
                                                       : (tc16_fc1_pair(bn, d.quant) ? 2 : 1);
  const int slots = per_sm * device_sms();
  const int smax = a8 ? d.H / 128 / 4 : cdiv(d.H, 256) / 2;
  return std::max(1, std::min(std::min(slots / units, smax), 16));
}

moe_status check_geometry(int E, int H, int I, int quant) {
  if (E < 1 || E > 1024) return MOE_ERR_SHAPE;
  if (H < 128 || H % 128 != 0) return MOE_ERR_SHAPE;
  if (I < 64 || I % 64 != 0) return MOE_ERR_SHAPE;
  if ((long long)H * H > (1LL << 40) || (long long)I > (1 << 20)) return MOE_ERR_SHAPE;
  if (quant < 0 || quant > 5) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_UNSUPPORTED: return "unsupported mode";
    case MOE_ERR_CAPACITY: return "M exceeds the plan capacity";
    case MOE_ERR_CAPTURING: return "stream is capturing";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

const char* moe_version(void) { return "moe_gb300 0.1 sm_103a"; }

const char* moe_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

moe_status moe_plan_weights(int E, int H, int I, int quant_mode, int w13_layout,
                            const int8_t* tier_of_expert, moe_weight_plan** out) {
  if (out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  moe_status st = check_geometry(E, H, I, quant_mode);
  if (st != MOE_OK) return st;
  if (w13_layout != MOE_W13_UP_GATE && w13_layout != MOE_W13_GATE_UP) return MOE_ERR_ARG;
  const bool hybrid = quant_mode == MOE_W4A16_HYBRID || quant_mode == MOE_W4A16_HYBRID_MX;
  if (hybrid != (tier_of_expert != nullptr)) return MOE_ERR_ARG;
  moe_weight_plan* wp = new (std::nothrow) moe_weight_plan();
  if (wp == nullptr) return MOE_ERR_ARG;
  wp->E = E; wp->H = H; wp->I = I; wp->Ip = (int)align_up((size_t)I, 128);
  wp->quant = quant_mode; wp->layout = w13_layout;
  wp->E4 = E; wp->E3 = 0;
  if (hybrid) {
    wp->E4 = wp->E3 = 0;
    wp->tier_map.resize(E);
    for (int e = 0; e < E; ++e) {
      if (tier_of_expert[e] == MOE_TIER_NVFP4) {
        wp->tier_map[e] = (MOE_TIER_NVFP4 << 24) | wp->E4++;
      } else if (tier_of_expert[e] == MOE_TIER_NF3) {
        wp->tier_map[e] = (MOE_TIER_NF3 << 24) | wp->E3++;
      } else {
        delete wp;
        return MOE_ERR_ARG;
      }
    }
  }
  const size_t H_ = H, I_ = I, Ip = wp->Ip;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  const size_t E4 = wp->E4, E3 = wp->E3;
  // W4A16 tiles of 128 rows x 256 K per matrix (fc1: I x H, fc2: H x Ip)
  const size_t t13 = (size_t)2 * cdiv(I, 128) * cdiv(H, 256);
  const size_t t2 = (size_t)(H / 128) * cdiv((int)Ip, 256);
  if (quant_mode == MOE_W4A8_MXFP4) {
    wp->w13 = take(E4 * 2 * I_ * H_ / 2);
    wp->w2 = take(E4 * H_ * Ip / 2);
    wp->s13 = take(E4 * 2 * (size_t)cdiv(I, 128) * (H_ / 128) * 512);
    wp->s2 = take(E4 * (H_ / 128) * (Ip / 128) * 512);
    wp->g13 = wp->g2 = wp->mxk13 = wp->mxk2 = wp->ag13 = wp->ag2 = 0;
  } else {
    wp->w13 = take(E4 * t13 * kNvCodeTile);
    wp->w2 = take(E4 * t2 * kNvCodeTile);
    wp->s13 = take(E4 * t13 * kW16ScaleTile);
    wp->s2 = take(E4 * t2 * kW16ScaleTile);
    wp->g13 = take(E4 * 4);
    wp->g2 = take(E4 * 4);
    const bool mx = quant_mode == MOE_W4A16_HYBRID_MX;
    wp->mxk13 = mx ? take(E4 * 4) : 0;
    wp->mxk2 = mx ? take(E4 * 4) : 0;
    const bool act_g = quant_mode == MOE_W4A8_NVFP4 || quant_mode == MOE_W4A4_NVFP4;
    wp->ag13 = act_g ? take(E4 * 4) : 0;
    wp->ag2 = act_g ? take(E4 * 4) : 0;
  }
  wp->nf_w13 = take(E3 * t13 * kNfCodeTile);
  wp->nf_s13 = take(E3 * t13 * kW16ScaleTile);
  wp->nf_w2 = take(E3 * t2 * kNfCodeTile);
  wp->nf_s2 = take(E3 * t2 * kW16ScaleTile);
  wp->tmap = take((size_t)E * 4);
  wp->total = o;
  *out = wp;
  return MOE_OK;
}

moe_status moe_prepared_bytes(const moe_weight_plan* wp, size_t* bytes) {
  if (wp == nullptr || bytes == nullptr) return MOE_ERR_ARG;
  *bytes = wp->total;
  return MOE_OK;
}

moe_status moe_prepare_weights(const moe_weight_plan* wp, const moe_checkpoint* src, void* dst,
                               size_t dst_bytes, void* stream, moe_prepared** out) {
  if (wp == nullptr || src == nullptr || dst == nullptr || out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  if (dst_bytes < wp->total || !aligned(dst, 256)) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (capturing(st)) return MOE_ERR_CAPTURING;
  const bool fp4 = wp->E4 > 0, nf3 = wp->E3 > 0;
  if (fp4 && (src->w13 == nullptr || src->s13 == nullptr || src->w2 == nullptr ||
              src->s2 == nullptr))
    return MOE_ERR_ARG;
  const bool mx16 = wp->quant == MOE_W4A16_HYBRID_MX;
  if (fp4 && wp->quant != MOE_W4A8_MXFP4 && !mx16 && (src->g13 == nullptr || src->g2 == nullptr))
    return MOE_ERR_ARG;
  if (nf3 && (src->nf_w13 == nullptr || src->nf_s13 == nullptr || src->nf_w2 == nullptr ||
              src->nf_s2 == nullptr))
    return MOE_ERR_ARG;
  const bool nv_a8 = wp->quant == MOE_W4A8_NVFP4 || wp->quant == MOE_W4A4_NVFP4;
  if (nv_a8 && (src->a1_gscale == nullptr || src->a2_gscale == nullptr)) return MOE_ERR_ARG;
  uint8_t* base = static_cast<uint8_t*>(dst);
  const int E4 = wp->E4, E3 = wp->E3, H = wp->H, I = wp->I, Ip = wp->Ip, L = wp->layout;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  if (fp4) {
    if (wp->quant == MOE_W4A8_MXFP4) {
      chk(launch_repack_fp4_tiled(src->w13, base + wp->w13, E4, 2, I, H / 2, H / 2, L, 0, st));
      chk(launch_repack_fp4_tiled(src->w2, base + wp->w2, E4, 1, H, I / 2, Ip / 2, L,
                                  (I & 127) == 64 ? I : 0, st));
    } else {
      chk(launch_repack_w16_tiled(0, src->w13, base + wp->w13, E4, 2, I, H, H, L, st));
      chk(launch_repack_w16_tiled(0, src->w2, base + wp->w2, E4, 1, H, I, Ip, L, st));
    }
    if (wp->quant == MOE_W4A8_MXFP4) {
      chk(launch_repack_sf_atoms(src->s13, base + wp->s13, E4, 2, I, H / 32, cdiv(I, 128),
                                 H / 128, L, st));
      chk(launch_repack_sf_atoms(src->s2, base + wp->s2, E4, 1, H, I / 32, H / 128, Ip / 128, L,
                                 st));
    } else if (mx16) {
      // UE8M0 per 32 -> f16 multipliers + per-expert factors (in the NVFP4 global's place)
      chk(launch_repack_mx16_scales(src->s13, base + wp->s13,
                                    reinterpret_cast<int32_t*>(base + wp->mxk13),
                                    reinterpret_cast<float*>(base + wp->g13), E4, 2, I, H, H, L,
                                    st));
      chk(launch_repack_mx16_scales(src->s2, base + wp->s2,
                                    reinterpret_cast<int32_t*>(base + wp->mxk2),
                                    reinterpret_cast<float*>(base + wp->g2), E4, 1, H, I, Ip, L,
                                    st));
    } else {
      // NVFP4 scales: rows of the 16-bit path's tiles, or the W4A4 kernels' scale atoms
      const int kind = wp->quant == MOE_W4A4_NVFP4 ? 4 : 1;
      chk(launch_repack_w16_tiled(kind, src->s13, base + wp->s13, E4, 2, I, H, H, L, st));
      chk(launch_repack_w16_tiled(kind, src->s2, base + wp->s2, E4, 1, H, I, Ip, L, st));
      chk(cudaMemcpyAsync(base + wp->g13, src->g13, (size_t)E4 * 4, cudaMemcpyDeviceToDevice, st));
      chk(cudaMemcpyAsync(base + wp->g2, src->g2, (size_t)E4 * 4, cudaMemcpyDeviceToDevice, st));
      if (nv_a8) {
        chk(cudaMemcpyAsync(base + wp->ag13, src->a1_gscale, (size_t)E4 * 4,
                            cudaMemcpyDeviceToDevice, st));
        chk(cudaMemcpyAsync(base + wp->ag2, src->a2_gscale, (size_t)E4 * 4,
                            cudaMemcpyDeviceToDevice, st));
      }
    }
  }
  if (nf3) {
    chk(launch_repack_w16_tiled(2, src->nf_w13, base + wp->nf_w13, E3, 2, I, H, H, L, st));
    chk(launch_repack_w16_tiled(2, src->nf_w2, base + wp->nf_w2, E3, 1, H, I, Ip, L, st));
    chk(launch_repack_w16_tiled(3, src->nf_s13, base + wp->nf_s13, E3, 2, I, H, H, L, st));
    chk(launch_repack_w16_tiled(3, src->nf_s2, base + wp->nf_s2, E3, 1, H, I, Ip, L, st));
  }
  if (!wp->tier_map.empty())
    chk(cudaMemcpyAsync(base + wp->tmap, wp->tier_map.data(), wp->tier_map.size() * 4,
                        cudaMemcpyHostToDevice, st));
  if (e != cudaSuccess) return cuda_status(e);
  moe_prepared* p = new (std::nothrow) moe_prepared();
  if (p == nullptr) return MOE_ERR_ARG;
  DevWeights& w = p->w;
  w.quant = wp->quant; w.E = wp->E; w.H = H; w.I = I; w.Ip = Ip; w.E4 = E4; w.E3 = E3;
  w.fp4_tiled = wp->quant == MOE_W4A8_MXFP4 ? 1 : 0;
  w.mx_kept = mx16 ? 1 : 0;
  if (nv_a8) {
    w.ag13 = reinterpret_cast<const float*>(base + wp->ag13);
    w.ag2 = reinterpret_cast<const float*>(base + wp->ag2);
  }
  w.w13 = base + wp->w13; w.s13 = base + wp->s13; w.w2 = base + wp->w2; w.s2 = base + wp->s2;
  if (wp->quant != MOE_W4A8_MXFP4) {
    w.g13 = reinterpret_cast<const float*>(base + wp->g13);
    w.g2 = reinterpret_cast<const float*>(base + wp->g2);
  }
  w.nf_w13 = base + wp->nf_w13; w.nf_s13 = base + wp->nf_s13;
  w.nf_w2 = base + wp->nf_w2; w.nf_s2 = base + wp->nf_s2;
  w.tier_map = wp->tier_map.empty() ? nullptr : reinterpret_cast<const int32_t*>(base + wp->tmap);
  *out = p;
  return MOE_OK;
}

moe_status moe_plan(int E, int H, int I, int topk, int max_m, int quant_mode, float swiglu_limit,
                    int deterministic, moe_plan_t** out) {
  if (out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  moe_status st = check_geometry(E, H, I, quant_mode);
  if (st != MOE_OK) return st;
  if (topk < 1 || topk > 16 || max_m < 1 || max_m > (1 << 20)) return MOE_ERR_SHAPE;
  if (std::isnan(swiglu_limit) || swiglu_limit <= 0.f) return MOE_ERR_ARG;
  // The 16-bit-operand modes (W4A16 NVFP4, the hybrids, NVFP4 weights with MXFP8 activations)
  // run on tensor-core kernels whose fc2 K stages are 256 wide: other shapes are refused here
  // rather than sent to another kernel family
  if (quant_mode != MOE_W4A8_MXFP4 && quant_mode != MOE_W4A4_NVFP4 &&
      align_up((size_t)I, 128) % 256 != 0)
    return MOE_ERR_SHAPE;
  // W4A4: whole 256-wide K stages in both GEMMs (the activation scale atoms cover K exactly)
  if (quant_mode == MOE_W4A4_NVFP4 && (H % 256 != 0 || align_up((size_t)I, 128) % 256 != 0))
    return MOE_ERR_UNSUPPORTED;
  moe_plan_t* p = new (std::nothrow) moe_plan_t();
  if (p == nullptr) return MOE_ERR_ARG;
  PlanDims& d = p->d;
  d.E = E; d.H = H; d.I = I; d.Ip = (int)align_up((size_t)I, 128); d.topk = topk; d.max_m = max_m;
  d.quant = quant_mode; d.deterministic = deterministic ? 1 : 0;
  d.limit = swiglu_limit; d.alpha = 1.f; d.beta = 0.f; d.backend = 0; d.fc1_kernel = 0;
  d.ep_first = 0; d.w_on_input = 0; d.keep_act = 0; d.wait_probe_ns = 0;
  d.kept_a8 = 0; d.a8_s13 = d.a8_inv13 = d.a8_s2 = d.a8_inv2 = 0.f;
  const size_t Sm = (size_t)max_m * topk;
  Scratch& s = p->s;
  s.max_tiles = (int)std::min<size_t>(Sm, (Sm + kSimtSlots - 1) / kSimtSlots +
                                              std::min<size_t>((size_t)E, Sm));
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  const bool a8 = quant_mode == MOE_W4A8_MXFP4;
  const bool a4 = quant_mode == MOE_W4A4_NVFP4;     // packed E2M1 activations, 4X scale atoms
  s.ctrl = take(64 * 4);
  s.cnt = take((size_t)E * 4);
  s.off = take((size_t)(E + 1) * 4);
  s.perm = take(Sm * 4);
  s.slot_of = take(Sm * 4);
  s.tiles = take((size_t)s.max_tiles * 16);
  s.xq = a8 ? take(Sm * H) : (a4 ? take(Sm * H / 2) : 0);
  s.xs = a8 ? take(Sm * H / 32) : 0;
  // scale atom rows of the W4A8 tensor-core calls, padded for the widest tile (96 tokens) that
  // starts at the last slot position
  s.r16 = (int)Sm + 96;
  s.xs16 = a8 ? take((size_t)(H / 128) * s.r16 * 16) : (a4 ? take((size_t)(H / 64) * s.r16 * 16) : 0);
  s.hs16 = a8 ? take((size_t)(d.Ip / 128) * s.r16 * 16)
              : (a4 ? take((size_t)(d.Ip / 64) * s.r16 * 16) : 0);
  // fc1 output of the CUDA-core path, or the per-split partial sums of the tensor-core path
  // ([split][slot][2][Ip], one slice per split, summed in split order)
  size_t g_rows = Sm;
  for (int m = 1; m <= max_m; ++m) {
    const int bn_m = a4 ? tc4_pick_bn(m) : tc_pick_bn(m, topk, E, quant_mode == MOE_W4A8_MXFP4);
    const int sp = fc1_splits(d, call_tiles(d, s.max_tiles, m, bn_m), bn_m);
    if (sp > 1) g_rows = std::max(g_rows, (size_t)sp * m * topk);
  }
  s.g = take(g_rows * 2 * d.Ip * 4);
  s.tickets = take(align_up((size_t)s.max_tiles * cdiv(I, 128), 4) * 4);
  s.part = a8 ? take(fc1_stream_part_bytes()) : 0;
  s.rcc = take((size_t)route_chunks((int)Sm) * E * 4);
  s.hq = a8 ? take(Sm * d.Ip) : (a4 ? take(Sm * d.Ip / 2) : 0);
  s.hs = a8 ? take(Sm * d.Ip / 32) : 0;
  s.h16 = (a8 || a4) ? 0 : take(Sm * d.Ip * 2);
  s.x16 = (a8 || a4) ? 0 : take(Sm * H * 2);
  s.acc = d.deterministic ? 0 : take((size_t)max_m * H * 4);
  s.rbuf = d.deterministic ? take(Sm * H * 4) : 0;
  s.total = o;
  o = 0;
  p->io_x = take((size_t)max_m * H * 2);
  p->io_ids = take(Sm * 4);
  p->io_w = take(Sm * 4);
  p->io_out = take((size_t)max_m * H * 2);
  p->io_total = o;
  *out = p;
  return MOE_OK;
}

moe_status moe_plan_set_swiglu_alpha_beta(moe_plan_t* plan, float alpha, float beta) {
  if (plan == nullptr || std::isnan(alpha) || std::isnan(beta)) return MOE_ERR_ARG;
  plan->d.alpha = alpha;
  plan->d.beta = beta;
  return MOE_OK;
}

moe_status moe_scratch_bytes(const moe_plan_t* plan, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return MOE_ERR_ARG;
  *bytes = plan->s.total;
  return MOE_OK;
}

moe_status moe_io_bytes(const moe_plan_t* plan, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return MOE_ERR_ARG;
  *bytes = plan->io_total;
  return MOE_OK;
}

static RunPtrs resolve(const moe_plan_t* plan, void* scratch) {
  uint8_t* b = static_cast<uint8_t*>(scratch);
  const Scratch& s = plan->s;
  const bool a8 = plan->d.quant == MOE_W4A8_MXFP4;
  const bool a4 = plan->d.quant == MOE_W4A4_NVFP4;
  RunPtrs r;
  r.ctrl = reinterpret_cast<int32_t*>(b + s.ctrl);
  r.cnt = reinterpret_cast<int32_t*>(b + s.cnt);
  r.off = reinterpret_cast<int32_t*>(b + s.off);
  r.perm = reinterpret_cast<int32_t*>(b + s.perm);
  r.slot_of = reinterpret_cast<int32_t*>(b + s.slot_of);
  r.tiles = reinterpret_cast<int4*>(b + s.tiles);
  r.xq = (a8 || a4) ? b + s.xq : nullptr;
  r.xs = a8 ? b + s.xs : nullptr;
  r.xs16 = (a8 || a4) ? b + s.xs16 : nullptr;
  r.hs16 = (a8 || a4) ? b + s.hs16 : nullptr;
  r.r16 = s.r16;
  r.g = reinterpret_cast<float*>(b + s.g);
  r.tickets = reinterpret_cast<int32_t*>(b + s.tickets);
  r.part = a8 ? reinterpret_cast<float*>(b + s.part) : nullptr;
  r.rcc = reinterpret_cast<int32_t*>(b + s.rcc);
  r.hq = (a8 || a4) ? b + s.hq : nullptr;
  r.hs = a8 ? b + s.hs : nullptr;
  r.h16 = (a8 || a4) ? nullptr : reinterpret_cast<__nv_bfloat16*>(b + s.h16);
  r.x16 = (a8 || a4) ? nullptr : reinterpret_cast<uint16_t*>(b + s.x16);
  r.acc = plan->d.deterministic ? nullptr : reinterpret_cast<float*>(b + s.acc);
  r.rbuf = plan->d.deterministic ? reinterpret_cast<float*>(b + s.rbuf) : nullptr;
  return r;
}

namespace {
// Records profiling event i (if configured) on the stream of the call.
struct ProfRec {
  const std::vector<cudaEvent_t>* ev;
  cudaStream_t st;
  bool cap;
  void operator()(size_t i) const {
    if (i >= ev->size()) return;
    if (cap)
      cudaEventRecordWithFlags((*ev)[i], st, cudaEventRecordExternal);
    else
      cudaEventRecord((*ev)[i], st);
  }
};
}  // namespace

moe_status moe_plan_set_profile_events(moe_plan_t* plan, void* const* events, int n_events) {
  if (plan == nullptr || n_events < 0 || (n_events > 0 && events == nullptr)) return MOE_ERR_ARG;
  plan->prof.clear();
  for (int i = 0; i < n_events; ++i) plan->prof.push_back(static_cast<cudaEvent_t>(events[i]));
  return MOE_OK;
}

static bool use_tc(const PlanDims& d) { return d.backend == 0 && d.quant == MOE_W4A8_MXFP4; }
// W4A16 / hybrid on tensor cores (moe_plan admits only shapes with Ip % 256 == 0 for these
// modes, so backend 0 always runs them on tensor cores).
static bool use_tc16(const PlanDims& d) {
  return d.backend == 0 && d.quant != MOE_W4A8_MXFP4 && d.quant != MOE_W4A4_NVFP4;
}
// W4A4 runs on its block-scaled FP4 kernels only (moe_plan refuses the CUDA-core backend)
static bool use_tc4(const PlanDims& d) { return d.quant == MOE_W4A4_NVFP4; }

const char* moe_profile_stage_names(const moe_plan_t* plan) {
  if (plan == nullptr) return "";
  return (use_tc(plan->d) || use_tc16(plan->d) || use_tc4(plan->d))
             ? "route,actq,fc1,fc2,finalize"
             : "route,actq,fc1,act,fc2,finalize";
}

moe_status moe_plan_set_fc1_kernel(moe_plan_t* plan, int choice) {
  if (plan == nullptr || choice < 0 || choice > 2) return MOE_ERR_ARG;
  plan->d.fc1_kernel = choice;
  return MOE_OK;
}

moe_status moe_plan_set_router_weight_on_input(moe_plan_t* plan, int on) {
  if (plan == nullptr || (on != 0 && on != 1)) return MOE_ERR_ARG;
  if (on && (plan->d.quant == MOE_W4A8_MXFP4 || plan->d.quant == MOE_W4A8_NVFP4 ||
             plan->d.quant == MOE_W4A4_NVFP4 || plan->d.kept_a8))
    return MOE_ERR_UNSUPPORTED;
  plan->d.w_on_input = on;
  return MOE_OK;
}

moe_status moe_plan_set_kept_a8(moe_plan_t* plan, float w13_input_scale, float w2_input_scale) {
  if (plan == nullptr) return MOE_ERR_ARG;
  if (plan->d.quant != MOE_W4A16_HYBRID_MX) return MOE_ERR_UNSUPPORTED;
  if (w13_input_scale == 0.f && w2_input_scale == 0.f) {
    plan->d.kept_a8 = 0;
    plan->d.a8_s13 = plan->d.a8_inv13 = plan->d.a8_s2 = plan->d.a8_inv2 = 0.f;
    return MOE_OK;
  }
  // fp32 reciprocals, as the method takes them: finite and nonzero for scales in range
  const float inv13 = 1.0f / w13_input_scale, inv2 = 1.0f / w2_input_scale;
  if (!(w13_input_scale > 0.f) || !(w2_input_scale > 0.f) || !std::isfinite(w13_input_scale) ||
      !std::isfinite(w2_input_scale) || !std::isfinite(inv13) || !std::isfinite(inv2) ||
      inv13 == 0.f || inv2 == 0.f)
    return MOE_ERR_ARG;
  if (plan->d.w_on_input || plan->d.backend == 1) return MOE_ERR_UNSUPPORTED;
  plan->d.kept_a8 = 1;
  plan->d.a8_s13 = w13_input_scale;
  plan->d.a8_inv13 = inv13;
  plan->d.a8_s2 = w2_input_scale;
  plan->d.a8_inv2 = inv2;
  return MOE_OK;
}

moe_status moe_plan_set_debug_copies(moe_plan_t* plan, int on) {
  if (plan == nullptr || (on != 0 && on != 1)) return MOE_ERR_ARG;
  plan->d.keep_act = on;
  return MOE_OK;
}

moe_status moe_plan_set_wait_probe(moe_plan_t* plan, unsigned long long ns) {
  if (plan == nullptr || ns > 1000000000ull) return MOE_ERR_ARG;
  plan->d.wait_probe_ns = ns;
  return MOE_OK;
}

moe_status moe_plan_set_expert_offset(moe_plan_t* plan, int first_expert) {
  if (plan == nullptr || first_expert < 0 || first_expert > INT32_MAX - plan->d.E)
    return MOE_ERR_ARG;
  plan->d.ep_first = first_expert;
  return MOE_OK;
}

moe_status moe_plan_set_backend(moe_plan_t* plan, int backend) {
  if (plan == nullptr || backend < 0 || backend > 1) return MOE_ERR_ARG;
  if (backend == 1 && (plan->d.quant == MOE_W4A8_NVFP4 || plan->d.quant == MOE_W4A4_NVFP4 ||
                       plan->d.kept_a8))
    return MOE_ERR_UNSUPPORTED;
  plan->d.backend = backend;
  return MOE_OK;
}

moe_status moe_call_launches(const moe_plan_t* plan, int M, int* launches) {
  if (plan == nullptr || launches == nullptr || M < 0) return MOE_ERR_ARG;
  if (M > plan->d.max_m) return MOE_ERR_CAPACITY;
  const PlanDims& d = plan->d;
  if (M == 0) {
    *launches = 0;
    return MOE_OK;
  }
  const bool tc8 = use_tc(d), t16 = use_tc16(d) || use_tc4(d);
  if (tc8 || t16) {
    // routing and quantisation / conversion (one launch for calls of at most 256 flat slots;
    // beyond, three - counts, scatter, quantisation or conversion - for W4A8 and for the other
    // modes beyond kChunkedRouteSlots slots, else two), fc1, fc2, finalize
    const bool small = route_actq_small_supported(M * d.topk, d.E);
    const bool chunked = tc8 || M * d.topk > kChunkedRouteSlots;
    *launches = (small ? 1 : (chunked ? 3 : 2)) + 3;
    return MOE_OK;
  }
  // route, actq (when something needs it), fc1, act, fc2, finalize
  const bool actq = d.quant == MOE_W4A8_MXFP4 || !d.deterministic;
  *launches = 5 + (actq ? 1 : 0);
  return MOE_OK;
}

moe_status moe_run(const moe_plan_t* plan, const moe_prepared* weights, void* scratch,
                   size_t scratch_bytes, const void* x, const int32_t* topk_ids,
                   const float* topk_weights, void* out, int M, void* stream) {
  if (plan == nullptr || weights == nullptr) return MOE_ERR_ARG;
  if (M < 0) return MOE_ERR_ARG;
  if (M > plan->d.max_m) return MOE_ERR_CAPACITY;
  if (M == 0) return MOE_OK;
  if (scratch == nullptr || x == nullptr || topk_ids == nullptr || topk_weights == nullptr ||
      out == nullptr)
    return MOE_ERR_ARG;
  if (scratch_bytes < plan->s.total || !aligned(scratch, 256) || !aligned(x, 16) ||
      !aligned(out, 16) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4))
    return MOE_ERR_ARG;
  const PlanDims& d = plan->d;
  const DevWeights& w = weights->w;
  if (w.E != d.E || w.H != d.H || w.I != d.I || w.quant != d.quant) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const RunPtrs r = resolve(plan, scratch);
  const ProfRec prof{&plan->prof, st, !plan->prof.empty() && capturing(st)};
  const bool a8 = d.quant == MOE_W4A8_MXFP4;
  const bool tc8 = use_tc(d), t16 = use_tc16(d), t4 = use_tc4(d);
  const bool tc = tc8 || t16 || t4;
  const int Sm = M * d.topk;
  const int bn = t4 ? tc4_pick_bn(M) : (tc ? tc_pick_bn(M, d.topk, d.E, tc8) : kSimtSlots);
  const int tiles = call_tiles(d, plan->s.max_tiles, M, bn);
  const int RT = cdiv(d.I, 128);
  // 16-token tiles (decode sizes): the persistent stream-K fc1, when its 32-bit schedule
  // arithmetic fits the call (fc1_stream_preferred)
  const bool sk_ok = stream_schedule_fits((long long)tiles * RT, d.H / 128);
  const bool streamk = tc8 && bn == 16 && sk_ok &&
                       (d.fc1_kernel == 0 ? fc1_stream_preferred(bn, tiles * RT) : d.fc1_kernel == 2);
  const int splits = (tc && !streamk) ? fc1_splits(d, tiles, bn) : 1;
  // small tensor-core calls route and quantise (W4A8) or convert (16-bit path) in one launch
  const bool small = tc && route_actq_small_supported(Sm, d.E);
  // the W4A8 tensor-core kernels (16/32-token tiles) read activation-scale atoms from prepared
  // rows
  const bool atoms = tc8;
  // small W4A8 calls at tile widths <= 32: fc1 quantises the activations itself (the kernels
  // route in shared memory and know each tile's tokens), the routing launch only routes
  const bool fuse_x = tc8 && small && Sm <= kPreRouteSlots && bn <= 32;
  void* acc = d.deterministic ? nullptr : r.acc;
  const size_t acc_words = d.deterministic ? 0 : (size_t)M * d.H;
  void* g = nullptr;            // split partials are fully written before they are read
  const size_t g_words = 0;
  void* tk = (tc && (splits > 1 || streamk)) ? r.tickets : nullptr;
  const size_t tk_words = tk ? align_up((size_t)tiles * RT, 4) : 0;
  // router weights on the input (16-bit paths): they scale the f16 activations, and the
  // combine adds the expert outputs with weight 1
  const float* win = d.w_on_input ? topk_weights : nullptr;
  const float* wcomb = d.w_on_input ? nullptr : topk_weights;
  // the MXFP4 kept tier's A8 opt-in: its slots' activations are static FP8
  const KeptA8 ka8{d.kept_a8 ? w.tier_map : nullptr, d.a8_inv13};
  prof(0);
  cudaError_t e;
  if (small) {
    e = launch_route_actq_small(topk_ids, Sm, d.E, d.ep_first, bn, plan->s.max_tiles, x, d.H,
                                d.topk, r, atoms, t16, win, w.ag13, t4, fuse_x, acc, acc_words,
                                g, g_words, tk, tk_words, ka8, st);
    if (e != cudaSuccess) return cuda_status(e);
    prof(1);
  } else if (tc8) {
    // larger W4A8 calls: routing over many CTAs, quantisation straight into slot order
    e = launch_route_count(topk_ids, Sm, d.E, d.ep_first, r, st);
    if (e == cudaSuccess)
      e = launch_route_scatter(topk_ids, Sm, d.E, d.ep_first, bn, plan->s.max_tiles, r, st);
    if (e != cudaSuccess) return cuda_status(e);
    prof(1);
    e = launch_actq_rows(x, M, d.H, d.topk, r, acc, acc_words, g, g_words, tk, tk_words, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else {
    // the 16-bit and W4A4 tensor-core calls beyond kChunkedRouteSlots flat slots route over
    // many CTAs as W4A8 does (the same tables); smaller ones, and the CUDA-core path, in one
    if (tc && Sm > kChunkedRouteSlots) {
      e = launch_route_count(topk_ids, Sm, d.E, d.ep_first, r, st);
      if (e == cudaSuccess)
        e = launch_route_scatter(topk_ids, Sm, d.E, d.ep_first, bn, plan->s.max_tiles, r, st);
    } else {
      e = launch_route(topk_ids, Sm, d.E, d.ep_first, bn, plan->s.max_tiles, r, st);
    }
    if (e != cudaSuccess) return cuda_status(e);
    prof(1);
    if (t16 && tc && w.ag13 == nullptr && Sm > kChunkedRouteSlots) {
      // the f16 operand rows of large calls: each token row read once and stored at its slots'
      // positions (smaller calls convert slot by slot, over more threads)
      e = launch_actq16_rows(x, M, d.H, d.topk, r, win, topk_ids, d.ep_first, d.E, acc,
                             acc_words, g, g_words, tk, tk_words, ka8, st);
      if (e != cudaSuccess) return cuda_status(e);
    } else if (a8 || acc || g || t16 || t4) {
      e = launch_actq(x, M, d.H, d.topk, r, a8, atoms, t16, win, w.ag13, topk_ids, d.ep_first,
                      d.E, t4, acc, acc_words, g, g_words, tk, tk_words, ka8, st);
      if (e != cudaSuccess) return cuda_status(e);
    }
  }
  prof(2);
  if (tc) {
    if (t4)
      e = launch_tc4_stage(0, w, r, d, bn, tiles, splits, topk_weights, M, st);
    else if (streamk)
      e = launch_fc1_stream(w, r, d, bn, M, r.part, r.tickets, topk_ids, plan->s.max_tiles,
                            fuse_x ? x : nullptr, st);
    else
      e = tc8 ? launch_tc_stage(0, w, r, d, bn, tiles, splits, topk_weights, M, topk_ids,
                                plan->s.max_tiles, fuse_x ? x : nullptr, st)
              : launch_tc16_stage(0, w, r, d, bn, tiles, splits, topk_weights, M, st);
    if (e != cudaSuccess) return cuda_status(e);
    prof(3);
    if (t4)
      e = launch_tc4_stage(1, w, r, d, bn, tiles, 1, wcomb, M, st);
    else if (tc8 && fc2_persist_preferred(bn, tiles * (d.H / 128)))
      e = launch_fc2_persist(w, r, d, bn, M, topk_weights, st);
    else
      e = tc8 ? launch_tc_stage(1, w, r, d, bn, tiles, 1, topk_weights, M, nullptr, 0, nullptr,
                                st)
              : launch_tc16_stage(1, w, r, d, bn, tiles, 1, wcomb, M, st);
    if (e != cudaSuccess) return cuda_status(e);
    prof(4);
    e = launch_simt_stage(3, w, r, d, plan->s.max_tiles, x, topk_weights, out, M, st);
    if (e != cudaSuccess) return cuda_status(e);
    prof(5);
    return MOE_OK;
  }
  // fc1, SwiGLU + requant, fc2 + combine, finalize
  for (int stage = 0; stage < 4; ++stage) {
    e = launch_simt_stage(stage, w, r, d, plan->s.max_tiles, x, topk_weights, out, M, st);
    if (e != cudaSuccess) return cuda_status(e);
    prof(3 + stage);
  }
  return MOE_OK;
}

moe_status moe_run_chunked(const moe_plan_t* plan, const moe_prepared* weights, void* scratch,
                           size_t scratch_bytes, const void* x, const int32_t* topk_ids,
                           const float* topk_weights, void* out, int M, void* stream) {
  if (plan == nullptr || M < 0) return MOE_ERR_ARG;
  if (M > 0 && (x == nullptr || topk_ids == nullptr || topk_weights == nullptr || out == nullptr))
    return MOE_ERR_ARG;
  const int cap = plan->d.max_m, H = plan->d.H, k = plan->d.topk;
  for (int s = 0; s < M; s += cap) {
    const moe_status rc = moe_run(
        plan, weights, scratch, scratch_bytes, static_cast<const uint16_t*>(x) + (size_t)s * H,
        topk_ids + (size_t)s * k, topk_weights + (size_t)s * k,
        static_cast<uint16_t*>(out) + (size_t)s * H, std::min(cap, M - s), stream);
    if (rc != MOE_OK) return rc;
  }
  return MOE_OK;
}

moe_status moe_run_host(const moe_plan_t* plan, const moe_prepared* weights, void* scratch,
                        size_t scratch_bytes, void* io, size_t io_bytes, const void* x_host,
                        const int32_t* ids_host, const float* w_host, void* out_host, int M,
                        void* stream) {
  if (plan == nullptr) return MOE_ERR_ARG;
  if (M < 0) return MOE_ERR_ARG;
  if (M > plan->d.max_m) return MOE_ERR_CAPACITY;
  if (M == 0) return MOE_OK;
  if (io == nullptr || io_bytes < plan->io_total || !aligned(io, 256) || x_host == nullptr ||
      ids_host == nullptr || w_host == nullptr || out_host == nullptr)
    return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(io);
  const size_t xb = (size_t)M * plan->d.H * 2, kb = (size_t)M * plan->d.topk * 4;
  const uint8_t* xh = static_cast<const uint8_t*>(x_host);
  cudaError_t e = cudaSuccess;
  const uint8_t *dx, *dids, *dw;
  if (reinterpret_cast<const uint8_t*>(ids_host) == xh + xb &&
      reinterpret_cast<const uint8_t*>(w_host) == xh + xb + kb) {
    // [x | ids | w] in one host buffer: one copy, the same packing on the device (x rows are
    // multiples of 16 bytes, so ids and weights stay aligned)
    e = cudaMemcpyAsync(b + plan->io_x, x_host, xb + 2 * kb, cudaMemcpyHostToDevice, st);
    dx = b + plan->io_x;
    dids = dx + xb;
    dw = dids + kb;
  } else {
    e = cudaMemcpyAsync(b + plan->io_x, x_host, xb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(b + plan->io_ids, ids_host, kb, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(b + plan->io_w, w_host, kb, cudaMemcpyHostToDevice, st);
    dx = b + plan->io_x;
    dids = b + plan->io_ids;
    dw = b + plan->io_w;
  }
  if (e != cudaSuccess) return cuda_status(e);
  // page-locked output under unified addressing (cudaHostAlloc / cudaMallocHost memory): the
  // device addresses it directly, so finalize stores the rows there and no device -> host copy
  // follows; other host memory goes through the staging buffer and one copy
  void* dout = b + plan->io_out;
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, out_host) == cudaSuccess) {
    if (pa.type == cudaMemoryTypeHost && pa.devicePointer != nullptr &&
        aligned(pa.devicePointer, 16))
      dout = pa.devicePointer;
  } else {
    (void)cudaGetLastError();   // not a pointer CUDA knows: the copy path
  }
  moe_status s = moe_run(plan, weights, scratch, scratch_bytes, dx,
                         reinterpret_cast<const int32_t*>(dids),
                         reinterpret_cast<const float*>(dw), dout, M, stream);
  if (s != MOE_OK) return s;
  if (dout == b + plan->io_out)
    e = cudaMemcpyAsync(out_host, dout, xb, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e);
}

moe_status moe_get_device_error(const moe_plan_t* plan, void* scratch, void* stream, int* code) {
  if (plan == nullptr || scratch == nullptr || code == nullptr) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  int32_t* ctrl = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + plan->s.ctrl);
  cudaError_t e = cudaMemcpyAsync(&v, ctrl, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctrl, 0, 4, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  *code = v;
  if (v & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (v != 0) return MOE_ERR_DEVICE;
  return MOE_OK;
}

moe_status moe_debug_routing(const moe_plan_t* plan, void* scratch, int M, int32_t* cnt,
                             int32_t* off, int32_t* perm, int32_t* slot_of, void* stream) {
  if (plan == nullptr || scratch == nullptr || M < 0 || M > plan->d.max_m) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const RunPtrs r = resolve(plan, scratch);
  const int E = plan->d.E;
  std::vector<int32_t> hoff(E + 1);
  cudaError_t e = cudaMemcpyAsync(hoff.data(), r.off, (E + 1) * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  const int S = hoff[E];
  if (S < 0 || S > M * plan->d.topk) return MOE_ERR_DEVICE;
  if (off) std::memcpy(off, hoff.data(), (E + 1) * 4);
  if (cnt) e = cudaMemcpyAsync(cnt, r.cnt, E * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && perm && S > 0)
    e = cudaMemcpyAsync(perm, r.perm, (size_t)S * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && slot_of && M > 0)
    e = cudaMemcpyAsync(slot_of, r.slot_of, (size_t)M * plan->d.topk * 4, cudaMemcpyDeviceToHost,
                        st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e);
}

moe_status moe_debug_actq(const moe_plan_t* plan, void* scratch, int M, uint8_t* xq, uint8_t* xs,
                          void* stream) {
  if (plan == nullptr || scratch == nullptr || M < 0 || M > plan->d.max_m) return MOE_ERR_ARG;
  if (plan->d.quant != MOE_W4A8_MXFP4) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const RunPtrs r = resolve(plan, scratch);
  cudaError_t e = cudaSuccess;
  int32_t S = 0;
  e = cudaMemcpyAsync(&S, r.ctrl + 2, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  if (S < 0 || S > M * plan->d.topk) return MOE_ERR_DEVICE;
  if (xq && S) e = cudaMemcpyAsync(xq, r.xq, (size_t)S * plan->d.H, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && xs && S)
    e = cudaMemcpyAsync(xs, r.xs, (size_t)S * plan->d.H / 32, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e);
}

moe_status moe_debug_h(const moe_plan_t* plan, void* scratch, int M, void* hq, uint8_t* hs,
                       void* stream) {
  if (plan == nullptr || scratch == nullptr || M < 0 || M > plan->d.max_m) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const RunPtrs r = resolve(plan, scratch);
  int32_t S = 0;
  cudaError_t e = cudaMemcpyAsync(&S, r.ctrl + 2, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  if (S < 0 || S > M * plan->d.topk) return MOE_ERR_DEVICE;
  const size_t Ip = plan->d.Ip;
  if (plan->d.quant == MOE_W4A8_MXFP4) {
    if (hq && S) e = cudaMemcpyAsync(hq, r.hq, (size_t)S * Ip, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && hs && S)
      e = cudaMemcpyAsync(hs, r.hs, (size_t)S * Ip / 32, cudaMemcpyDeviceToHost, st);
  } else if (plan->d.quant == MOE_W4A4_NVFP4) {
    // packed E2M1 codes, and the E4M3 scales gathered from the atom rows [Ip/64][r16][16]
    if (hq && S) e = cudaMemcpyAsync(hq, r.hq, (size_t)S * Ip / 2, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && hs && S) {
      std::vector<uint8_t> rows((size_t)(Ip / 64) * r.r16 * 16);
      e = cudaMemcpyAsync(rows.data(), r.hs16, rows.size(), cudaMemcpyDeviceToHost, st);
      if (e == cudaSuccess) e = cudaStreamSynchronize(st);
      if (e == cudaSuccess)
        for (int q = 0; q < S; ++q)
          for (size_t g = 0; g < Ip / 16; ++g)
            hs[(size_t)q * (Ip / 16) + g] = rows[((g / 4) * r.r16 + q) * 16 + g % 4];
    }
  } else if (hq && S) {
    e = cudaMemcpyAsync(hq, r.h16, (size_t)S * Ip * 2, cudaMemcpyDeviceToHost, st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_status(e);
}

// ------------------------------------------------------------------ test hook: unprepare
// The inverse of the repack kernels of prepare.cu, on the host: each checkpoint byte is read back
// from its prepared position (through the same layout helpers), so a test can compare the
// device layout with the checkpoint byte for byte.
namespace {
struct Unprep {
  const std::vector<uint8_t>& P;
  const moe_weight_plan* wp;
  // checkpoint row of prepared fc1 matrix half `half`, row i
  int src_row(int half, int i) const { return (wp->layout == 0 ? half : 1 - half) * wp->I + i; }
};
// E4M3 scale code of a 16-group of an NVFP4 W4A4 4X atom tile
size_t atom4x_off(size_t mat, int r, int k, int rbs, int kts) {
  const int kk = k & 255, rr = r & 127;
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kW16ScaleTile + (size_t)(kk >> 6) * 512 +
         (size_t)((rr & 31) * 16 + (rr >> 5) * 4 + ((kk & 63) >> 4));
}
// UE8M0 byte of an MXFP4 kept-tier group from its f16 multiplier 2^(b - kmax + 13)
uint8_t mx_byte_of(uint16_t bits, int kmax) {
  if (bits == 0x7E00) return 0xFF;
  if (bits == 0) return 0;                                  // flushed group
  int j;
  if (bits >= 0x400) {
    j = (bits >> 10) - 15;
  } else {
    j = -24;
    for (uint16_t m = bits; m > 1; m >>= 1) ++j;
  }
  return (uint8_t)(j + kmax - 13);
}
}  // namespace

moe_status moe_unprepare_weights(const moe_weight_plan* wp, const moe_prepared* prepared,
                                  void* stream, const moe_checkpoint* dst) {
  if (wp == nullptr || prepared == nullptr || dst == nullptr) return MOE_ERR_ARG;
  const DevWeights& w = prepared->w;
  if (w.E != wp->E || w.H != wp->H || w.I != wp->I || w.quant != wp->quant) return MOE_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  std::vector<uint8_t> P(wp->total);
  cudaError_t e = cudaMemcpyAsync(P.data(), w.w13 - wp->w13, wp->total, cudaMemcpyDeviceToHost,
                                  st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  const int E4 = wp->E4, E3 = wp->E3, H = wp->H, I = wp->I, Ip = wp->Ip, q = wp->quant;
  const Unprep u{P, wp};
  auto out8 = [](const void* p) { return static_cast<uint8_t*>(const_cast<void*>(p)); };
  const uint8_t* b = P.data();
  const int rb1 = cdiv(I, 128), kt1 = cdiv(H, 256), rb2 = H / 128, kt2 = cdiv(Ip, 256);
  if (E4 > 0 && (dst->w13 == nullptr || dst->s13 == nullptr || dst->w2 == nullptr ||
                 dst->s2 == nullptr))
    return MOE_ERR_ARG;
  if (E3 > 0 && (dst->nf_w13 == nullptr || dst->nf_s13 == nullptr || dst->nf_w2 == nullptr ||
                 dst->nf_s2 == nullptr))
    return MOE_ERR_ARG;
  uint8_t *w13 = out8(dst->w13), *s13 = out8(dst->s13), *w2 = out8(dst->w2), *s2 = out8(dst->s2);
  if (q == MOE_W4A8_MXFP4) {
    for (int ex = 0; ex < E4; ++ex) {
      for (int half = 0; half < 2; ++half)
        for (int i = 0; i < I; ++i) {
          const size_t sr = (size_t)ex * 2 * I + u.src_row(half, i), mat = (size_t)ex * 2 + half;
          for (int c = 0; c < H / 2; ++c)
            w13[sr * (H / 2) + c] = b[wp->w13 + fp4_tiled_byte((size_t)E4 * 2, I, H, mat, i, 2 * c)];
          for (int kb = 0; kb < H / 32; ++kb)
            s13[sr * (H / 32) + kb] = b[wp->s13 + sf_atom_byte(rb1, H / 128, mat, i, kb)];
        }
      for (int r = 0; r < H; ++r) {
        const size_t sr = (size_t)ex * H + r;
        for (int c = 0; c < I / 2; ++c)
          w2[sr * (I / 2) + c] = b[wp->w2 + fp4_w2_byte((size_t)E4, H, Ip, I, ex, r, 2 * c)];
        for (int kb = 0; kb < I / 32; ++kb)
          s2[sr * (I / 32) + kb] = b[wp->s2 + sf_atom_byte(H / 128, Ip / 128, ex, r, kb)];
      }
    }
  } else if (E4 > 0) {
    // NVFP4 (16-bit, MXFP8-activation and W4A4 modes) or the MXFP4 kept tier
    const bool mx = q == MOE_W4A16_HYBRID_MX, a4x = q == MOE_W4A4_NVFP4;
    const int g = mx ? 32 : 16;
    auto scale = [&](size_t sec, size_t ksec, size_t mat, int r, int k, int rbs, int kts,
                     int ex) -> uint8_t {
      if (a4x) return b[sec + atom4x_off(mat, r, k, rbs, kts)];
      if (!mx) return b[sec + nv_scale_byte(mat, r, k, rbs, kts)];
      uint16_t bits;
      std::memcpy(&bits, &b[sec + mx16_scale_off(mat, r, k, rbs, kts)], 2);
      int32_t kmax;
      std::memcpy(&kmax, &b[ksec + (size_t)ex * 4], 4);
      return mx_byte_of(bits, kmax);
    };
    for (int ex = 0; ex < E4; ++ex) {
      for (int half = 0; half < 2; ++half)
        for (int i = 0; i < I; ++i) {
          const size_t sr = (size_t)ex * 2 * I + u.src_row(half, i), mat = (size_t)ex * 2 + half;
          for (int k = 0; k < H; k += 2)
            w13[sr * (H / 2) + k / 2] = b[wp->w13 + nv_code_byte(mat, i, k, rb1, kt1)];
          for (int k = 0; k < H; k += g)
            s13[sr * (H / g) + k / g] = scale(wp->s13, wp->mxk13, mat, i, k, rb1, kt1, ex);
        }
      for (int r = 0; r < H; ++r) {
        const size_t sr = (size_t)ex * H + r;
        for (int k = 0; k < I; k += 2)
          w2[sr * (I / 2) + k / 2] = b[wp->w2 + nv_code_byte(ex, r, k, rb2, kt2)];
        for (int k = 0; k < I; k += g)
          s2[sr * (I / g) + k / g] = scale(wp->s2, wp->mxk2, ex, r, k, rb2, kt2, ex);
      }
    }
    if (!mx && dst->g13 != nullptr && dst->g2 != nullptr) {
      std::memcpy(const_cast<float*>(dst->g13), &b[wp->g13], (size_t)E4 * 4);
      std::memcpy(const_cast<float*>(dst->g2), &b[wp->g2], (size_t)E4 * 4);
    }
    if (wp->ag13 != 0 && dst->a1_gscale != nullptr && dst->a2_gscale != nullptr) {
      std::memcpy(const_cast<float*>(dst->a1_gscale), &b[wp->ag13], (size_t)E4 * 4);
      std::memcpy(const_cast<float*>(dst->a2_gscale), &b[wp->ag2], (size_t)E4 * 4);
    }
  }
  if (E3 > 0) {
    uint8_t *nw13 = out8(dst->nf_w13), *ns13 = out8(dst->nf_s13), *nw2 = out8(dst->nf_w2),
            *ns2 = out8(dst->nf_s2);
    auto code = [&](size_t sec, size_t mat, int r, int k, int rbs, int kts) -> uint32_t {
      const uint32_t lo = (b[sec + nf_lo_byte(mat, r, k, rbs, kts)] >> (2 * (k & 3))) & 3u;
      const uint32_t hi = (b[sec + nf_hi_byte(mat, r, k, rbs, kts)] >> (k & 7)) & 1u;
      return lo | (hi << 2);
    };
    auto row_codes = [&](uint8_t* dstrow, size_t sec, size_t mat, int r, int K, int rbs, int kts) {
      for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t w24 = 0;
        for (int t = 0; t < 8; ++t) w24 |= code(sec, mat, r, k0 + t, rbs, kts) << (3 * t);
        dstrow[3 * (k0 / 8) + 0] = (uint8_t)(w24 & 0xFF);
        dstrow[3 * (k0 / 8) + 1] = (uint8_t)((w24 >> 8) & 0xFF);
        dstrow[3 * (k0 / 8) + 2] = (uint8_t)(w24 >> 16);
      }
    };
    for (int ex = 0; ex < E3; ++ex) {
      for (int half = 0; half < 2; ++half)
        for (int i = 0; i < I; ++i) {
          const size_t sr = (size_t)ex * 2 * I + u.src_row(half, i), mat = (size_t)ex * 2 + half;
          row_codes(nw13 + sr * (3 * H / 8), wp->nf_w13, mat, i, H, rb1, kt1);
          for (int k = 0; k < H; k += 32)
            ns13[sr * (H / 32) + k / 32] = b[wp->nf_s13 + nf_scale_byte(mat, i, k, rb1, kt1)];
        }
      for (int r = 0; r < H; ++r) {
        const size_t sr = (size_t)ex * H + r;
        row_codes(nw2 + sr * (3 * I / 8), wp->nf_w2, ex, r, I, rb2, kt2);
        for (int k = 0; k < I; k += 32)
          ns2[sr * (I / 32) + k / 32] = b[wp->nf_s2 + nf_scale_byte(ex, r, k, rb2, kt2)];
      }
    }
  }
  return MOE_OK;
}

void moe_destroy_weight_plan(moe_weight_plan* wp) { delete wp; }
void moe_destroy_prepared(moe_prepared* p) { delete p; }
void moe_destroy_plan(moe_plan_t* plan) { delete plan; }

}  // extern "C"
