// gemm_tc4.cu - W4A4 grouped GEMMs (NVFP4 weights x NVFP4 activations) on the 5th-generation
// tensor cores: tcgen05 kind::mxf4nvf4 with 4X scale vectors.
//
// B12xExperts quant mode "nvfp4" (vLLM fused_moe/b12x page: kNvfp4Static weights with
// kNvfp4Dynamic activations; `_prepare_experts` takes the per-expert activation global scales
// a1_gscale / a2_gscale).  Weights: E2M1 codes with an E4M3 scale per 16 along K and one fp32
// global per expert and matrix.  Activations: each slot's x (fc1) and h (fc2), times the
// expert's activation global scale in fp32, quantised to NVFP4 blocks of 16 (E4M3 scale
// nearest vmax / 6, E2M1 codes nearest-even of v / scale); the MMA multiplies codes and block
// scales of both operands exactly and accumulates in fp32, and the epilogue applies
// weight global / activation global.
//
// Same orientation and work split as the W4A8 kernels (gemm_tc.cu): weight rows are the 128-row
// MMA operand, the tile's tokens the N columns; one CTA per (tile, 128-row block[, K split]).
// A pipeline stage covers 256 K: the weight tiles are the 16-bit path's pre-swizzled 16 KB
// NVFP4 code tiles (one bulk copy each) with their scales prepared as four 512-byte tensor-
// memory atoms (one per K = 64 instruction), the activation tile comes by TMA (128-byte
// swizzle) and its scale atoms by bulk copies.  Warp 0 lane 0 loads, warp 1 lane 0 copies the
// scales to tensor memory and issues the MMAs, all four warps run the epilogue.
#include <algorithm>
#include <cstring>

#include <cuda_fp4.h>

#include "moe_common.cuh"
#include "tc_ptx.cuh"
#include "tc_sched.cuh"
#include "tc_tile.cuh"

namespace moe {

using namespace tc;

constexpr int k4TileA = kNvCodeTile;       // 128 rows x 256 K of packed E2M1
constexpr int k4SfTile = kW16ScaleTile;    // four 512-byte scale atoms (K = 64 each)

template <int BN, bool FC2>
struct Tc4Cfg {
  static constexpr int kMats = FC2 ? 1 : 2;
  static constexpr int kChunks = BN <= 32 ? 1 : BN / 32;    // 32-column MMAs
  static constexpr int kWidth = BN < 32 ? BN : 32;           // N of one MMA
  static constexpr int kB = BN * 128;                        // activation codes of a stage
  static constexpr int kSfb = kChunks * 2048;                // activation scale atoms
  // stage: weight tiles | weight scale atoms | activation tile | activation scale atoms
  static constexpr int kOffSfa = kMats * k4TileA;
  static constexpr int kOffB = kOffSfa + kMats * k4SfTile;   // multiple of 1024
  static constexpr int kOffSfb = kOffB + kB;
  static constexpr int kStage = (kOffSfb + kSfb + 1023) / 1024 * 1024;
  static constexpr int kStages = 2;                          // two CTAs per SM
  static constexpr int kSfCols = kMats * 16 + kChunks * 16;  // tensor-memory scale columns
  static constexpr int kColsD = kMats * BN;
  static constexpr int kCols = kColsD + kSfCols * kStages;
  static constexpr int kAlloc = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : 256;
  static_assert(kCols <= 256, "two CTAs per SM: at most 256 tensor-memory columns each");
  static_assert(BN == 16 || BN == 32 || BN == 64, "W4A4 token tile widths");
  static constexpr int kSmem = kStages * kStage + 1024;
};

struct Tc4Params {
  CUtensorMap tm_act;          // packed E2M1 activations [Sm][K/2] bytes, box 128 x min(BN, 32)
  const uint8_t* codes;        // weight code tiles (16 KB, pre-swizzled) [mats][RB][KT]
  const uint8_t* sfa;          // weight scale atoms, 2 KB per tile
  const uint8_t* sfb;          // activation scale atom rows [K/64][r16][16]
  int r16;
  const float* gscale;         // weight global of this matrix [E]
  const float* agscale;        // activation global of this GEMM's input [E]
  const float* agscale2;       // fc1: that of fc2's input (the requantised h)
  const int4* tiles;
  const int32_t* ctrl;
  int32_t* err;
  // fc1 outputs
  uint8_t* hq;                 // packed E2M1 [Sm][Ip/2]
  uint8_t* hs;                 // scale atom rows [Ip/64][r16][16]
  float* gacc;                 // [splits][Sm][2][Ip] split-K partial sums
  int32_t* tickets;
  // fc2 outputs
  const int32_t* perm;
  const float* topk_w;
  float* acc;
  float* rbuf;
  int K, I, Ip, RB, KT, Sm, splits, topk, deterministic, H;
  float limit, alpha, beta;
};

__device__ __forceinline__ float swiglu4(float gate, float up, float limit, float alpha,
                                         float beta) {
  const float g = fminf(gate, limit);
  const float u = fminf(fmaxf(up, -limit), limit);
  return g / (1.0f + expf(-alpha * g)) * (u + beta);
}

// NVFP4 requantisation of one token column of h for this warp's 32 features (two blocks of
// 16 lanes): v = a * h in fp32, block scale E4M3(vmax / 6), codes E2M1(v / scale); even lanes
// store the byte of their pair, lanes 0 and 16 the block's scale into the atom row.  All 32
// lanes call it with the same column.
__device__ __forceinline__ void nvfp4_store_h(float v, int lane, int pos, int f, int Ip,
                                              int r16, uint8_t* hq, uint8_t* hs) {
  float vmax = fabsf(v);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(vmax, 6.f));
  const float sv = e4m3_to_f32((uint8_t)sc);
  const uint32_t q =
      sv > 0.f ? (uint32_t)__nv_cvt_float_to_fp4(__fdiv_rn(v, sv), __NV_E2M1, cudaRoundNearest)
               : 0u;
  const uint32_t hi = __shfl_down_sync(0xffffffffu, q, 1);
  if ((lane & 1) == 0) hq[(size_t)pos * (Ip / 2) + f / 2] = (uint8_t)((q & 0xF) | ((hi & 0xF) << 4));
  if ((lane & 15) == 0) hs[((size_t)(f >> 6) * r16 + pos) * 16 + ((f & 63) >> 4)] = (uint8_t)sc;
}

template <int BN, bool FC2>
__global__ void __launch_bounds__(kTcThreads)
gemm_tc4_kernel(const __grid_constant__ Tc4Params p) {
  using Cfg = Tc4Cfg<BN, FC2>;
  constexpr int S = Cfg::kStages;
  constexpr int kMats = Cfg::kMats;
  __shared__ uint32_t s_tmem;
  tmem_alloc_first(&s_tmem, Cfg::kAlloc);
  pdl_wait_prev();             // routing tables and activations complete
  pdl_launch_next();
  const int tile = blockIdx.x;
  if (tile >= p.ctrl[1]) {
    tmem_exit_early(&s_tmem, Cfg::kAlloc);
    return;
  }
  const int4 td = p.tiles[tile];
  const int e = td.x, p0 = td.y, n = td.z;
  const int rb = blockIdx.y, split = blockIdx.z;
  const int kt0 = split * p.KT / p.splits, kt1 = (split + 1) * p.KT / p.splits;
  const int nk = kt1 - kt0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[S], empty[S], done;
  __shared__ int s_last, s_fail;
  __shared__ int s_f[BN];
  __shared__ float s_w[BN];

  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    s_fail = 0;
    fence_barrier_init();
  }
  if (tid == 64) prefetch_tmap(&p.tm_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;
  int issued = 0;
  auto stage = [&](int s) { return smem + s * Cfg::kStage; };
  constexpr int kAtomRows = BN < 32 ? BN : 32;
  constexpr uint32_t kTx = kMats * (k4TileA + k4SfTile) + Cfg::kB +
                           Cfg::kChunks * 4 * kAtomRows * 16;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
      int i = 0;
      for (; i < nk && ok; ++i) {
        const int s = i % S;
        if (i >= S) ok = mbar_wait(&empty[s], ((i / S) - 1) & 1, p.err);
        if (!ok) break;
        uint8_t* st = stage(s);
        const int kt = kt0 + i;
        mbar_arrive_expect_tx(&full[s], kTx);
        for (int m = 0; m < kMats; ++m) {
          const size_t t = w16_tile(FC2 ? (size_t)e : 2 * (size_t)e + m, rb, kt, p.RB, p.KT);
          bulk_load_hint(st + m * k4TileA, p.codes + t * k4TileA, k4TileA, &full[s], pol);
          bulk_load_hint(st + Cfg::kOffSfa + m * k4SfTile, p.sfa + t * k4SfTile, k4SfTile,
                         &full[s], pol);
        }
        for (int j = 0; j < Cfg::kChunks; ++j) {
          tma_load_2d(st + Cfg::kOffB + 4096 * j, &p.tm_act, kt * 128, p0 + 32 * j, &full[s]);
          for (int kb = 0; kb < 4; ++kb)
            bulk_load(st + Cfg::kOffSfb + 2048 * j + 512 * kb,
                      p.sfb + ((size_t)(kt * 4 + kb) * p.r16 + p0 + 32 * j) * 16,
                      kAtomRows * 16, &full[s]);
        }
      }
      issued = i;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mxf4nvf4(Cfg::kWidth);
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % S;
        ok = mbar_wait(&full[s], (i / S) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        uint8_t* st = stage(s);
        const uint32_t sfa = tmem + Cfg::kColsD + Cfg::kSfCols * s;
        const uint32_t sfb = sfa + kMats * 16;
#pragma unroll
        for (int m = 0; m < kMats; ++m)
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            tc_cp_sf(sfa + (m * 4 + kb) * 4, desc_sf(st + Cfg::kOffSfa + m * k4SfTile + 512 * kb));
#pragma unroll
        for (int j = 0; j < Cfg::kChunks; ++j)
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            tc_cp_sf(sfb + (j * 4 + kb) * 4, desc_sf(st + Cfg::kOffSfb + 2048 * j + 512 * kb));
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint32_t accum = (i > 0 || kb > 0) ? 1u : 0u;
#pragma unroll
          for (int j = 0; j < Cfg::kChunks; ++j) {
            const uint64_t bdesc = desc_sw128(st + Cfg::kOffB + 4096 * j + 32 * kb);
#pragma unroll
            for (int m = 0; m < kMats; ++m)
              mma_mxf4nvf4_4x(tmem + m * BN + 32 * j, desc_sw128(st + m * k4TileA + 32 * kb),
                              bdesc, idesc, sfa + (m * 4 + kb) * 4, sfb + (j * 4 + kb) * 4,
                              accum);
          }
        }
        tc_commit(&empty[s]);
      }
      tc_commit(&done);
    }
  } else if (FC2 && warp == 3) {
    for (int c = lane; c < n; c += 32) {
      const int f = p.perm[p0 + c];
      s_f[c] = f;
      s_w[c] = p.topk_w[f];
    }
  }

  __syncthreads();
  // one verdict per warp: the producer's or MMA issuer's lane may have given up a wait while the
  // other lanes did not, and the epilogue's TMEM loads and shuffles are warp-collective
  ok = __all_sync(0xffffffffu, mbar_wait(&done, 0, p.err) && ok);
  tc_fence_after();
  __syncwarp();
  const int row = rb * 128 + warp * 32 + lane;       // weight row of this lane
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  const float gs = p.gscale[e] / p.agscale[e];
  const float a_next = FC2 ? 0.f : p.agscale2[e];
  if (ok && nk > 0) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      float v0[16], v1[16];
      tmem_ld16(trow + c0, v0);
      if (!FC2) tmem_ld16(trow + BN + c0, v1);
      if (c0 >= n) continue;
      if (FC2) {
        // 16 token columns x this warp's 32 output features, read back transposed so that the
        // combine adds 16 bytes (4 features of one token) per atomic; the pipeline stages are
        // free once `done` has completed (every copy landed and was consumed)
        float(*sy)[32] = reinterpret_cast<float(*)[32]>(smem + warp * 2048);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sy[jj][lane] = v0[jj] * gs;
        __syncwarp();
        const int h4 = rb * 128 + warp * 32 + 4 * (lane & 7);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int cc = 4 * r + (lane >> 3);
          if (c0 + cc < n) {
            const float4 v = *reinterpret_cast<const float4*>(&sy[cc][4 * (lane & 7)]);
            const int f = s_f[c0 + cc];
            const float wt = s_w[c0 + cc];
            const float4 o = make_float4(wt * v.x, wt * v.y, wt * v.z, wt * v.w);
            if (p.deterministic)
              *reinterpret_cast<float4*>(p.rbuf + (size_t)f * p.H + h4) = o;
            else
              atomicAdd(reinterpret_cast<float4*>(p.acc + (size_t)(f / p.topk) * p.H + h4), o);
          }
        }
        __syncwarp();
        continue;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        if (c >= n) break;
        const int pos = p0 + c;
        if (!FC2) {
          if (p.splits == 1) {
            const float h = row < p.I ? swiglu4(v1[j] * gs, v0[j] * gs, p.limit, p.alpha, p.beta)
                                      : 0.f;
            nvfp4_store_h(h * a_next, lane, pos, row, p.Ip, p.r16, p.hq, p.hs);
          } else {
            float* gg = p.gacc + ((size_t)split * p.Sm + pos) * 2 * p.Ip;
            gg[row] = v0[j];
            gg[p.Ip + row] = v1[j];
          }
        } else {
          const float v = s_w[c] * (v0[j] * gs);
          const int f = s_f[c];
          if (p.deterministic)
            p.rbuf[(size_t)f * p.H + row] = v;
          else
            atomicAdd(&p.acc[(size_t)(f / p.topk) * p.H + row], v);
        }
      }
    }
  }
  if (!FC2 && p.splits > 1) __threadfence();
  if (!ok) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  // a wait gave up: let this CTA's copies land before its shared memory is released
  if (s_fail && warp == 0 && lane == 0) drain_stage_loads<S>(full, issued, p.err);
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc);
  if (!FC2 && p.splits > 1) {
    if (tid == 0) {
      __threadfence();
      const int t = atomicAdd(&p.tickets[tile * p.RB + rb], 1);
      s_last = (t == p.splits - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      // partial sums added in split order: the same result on every run
      for (int c = 0; c < n; ++c) {
        float up = 0.f, gt = 0.f;
        for (int sp = 0; sp < p.splits; ++sp) {
          const float* gg = p.gacc + ((size_t)sp * p.Sm + p0 + c) * 2 * p.Ip + row;
          up += __ldcg(gg);
          gt += __ldcg(gg + p.Ip);
        }
        const float h = row < p.I ? swiglu4(gt * gs, up * gs, p.limit, p.alpha, p.beta) : 0.f;
        nvfp4_store_h(h * a_next, lane, p0 + c, row, p.Ip, p.r16, p.hq, p.hs);
      }
    }
  }
}

// Persistent fc2 for decode and mid sizes (tile widths 16 and 32): each CTA takes a contiguous
// range of (tile, 128-row block) units and streams their weight stages through one 4-stage
// ring, so the loads of the next unit overlap the MMAs and the combine of the current one;
// the accumulators are double-buffered in tensor memory.  Warp 0 lane 0 loads, warp 1 lane 0
// issues, warps 4..7 run the combine (16-byte atomics after a transpose in shared memory).
constexpr int k4PThreads = 256;

template <int BN>
struct Tc4PersistCfg {
  using Base = Tc4Cfg<BN, true>;
  static constexpr int kStages = 4;
  static constexpr int kStage = Base::kStage;
  static constexpr int kCols = 2 * BN + Base::kSfCols * kStages;   // 2 accumulators + scales
  static constexpr int kAlloc = kCols <= 64 ? 64 : kCols <= 128 ? 128 : 256;
  static_assert(kCols <= 256, "two CTAs per SM: at most 256 tensor-memory columns each");
  static_assert(BN == 16 || BN == 32, "persistent W4A4 fc2 tile widths");
  static constexpr int kSmem = kStages * kStage + 1024;
};

template <int BN>
__global__ void __launch_bounds__(k4PThreads)
fc2_tc4_persist_kernel(const __grid_constant__ Tc4Params p) {
  using Cfg = Tc4PersistCfg<BN>;
  using B = typename Cfg::Base;
  constexpr int S = Cfg::kStages;
  __shared__ uint32_t s_tmem;
  tmem_alloc_first(&s_tmem, Cfg::kAlloc);
  pdl_wait_prev();             // fc1 complete, h and its scales visible
  pdl_launch_next();
  const int G = gridDim.x, c = blockIdx.x;
  const int units = p.ctrl[1] * p.RB;
  const int u_begin = (int)((long long)c * units / G);
  const int u_end = (int)((long long)(c + 1) * units / G);
  if (u_begin >= u_end) {
    tmem_exit_early(&s_tmem, Cfg::kAlloc);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[S], empty[S], acc_full[2], acc_empty[2];
  __shared__ int s_fail;
  __shared__ int s_f[BN];
  __shared__ float s_w[BN];
  __shared__ __align__(16) float s_y[4][16][32];

  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    s_fail = 0;
    fence_barrier_init();
  }
  if (tid == 64) prefetch_tmap(&p.tm_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;
  int issued = 0;
  auto stage = [&](int s) { return smem + s * Cfg::kStage; };
  constexpr int kAtomRows = BN < 32 ? BN : 32;
  constexpr uint32_t kTx = k4TileA + k4SfTile + B::kB + 4 * kAtomRows * 16;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
      int i = 0;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const int tile = u / p.RB, rb = u - tile * p.RB;
        const int4 td = p.tiles[tile];
        for (int kt = 0; kt < p.KT && ok; ++kt, ++i) {
          const int s = i % S;
          if (i >= S) ok = mbar_wait(&empty[s], ((i / S) - 1) & 1, p.err);
          if (!ok) break;
          uint8_t* st = stage(s);
          const size_t t = w16_tile((size_t)td.x, rb, kt, p.RB, p.KT);
          mbar_arrive_expect_tx(&full[s], kTx);
          bulk_load_hint(st, p.codes + t * k4TileA, k4TileA, &full[s], pol);
          bulk_load_hint(st + B::kOffSfa, p.sfa + t * k4SfTile, k4SfTile, &full[s], pol);
          tma_load_2d(st + B::kOffB, &p.tm_act, kt * 128, td.y, &full[s]);
          for (int kb = 0; kb < 4; ++kb)
            bulk_load(st + B::kOffSfb + 512 * kb,
                      p.sfb + ((size_t)(kt * 4 + kb) * p.r16 + td.y) * 16, kAtomRows * 16,
                      &full[s]);
        }
      }
      issued = i;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_mxf4nvf4(B::kWidth);
      int i = 0, j = 0;
      for (int u = u_begin; u < u_end && ok; ++u, ++j) {
        const int b = j & 1;
        if (j >= 2) ok = mbar_wait(&acc_empty[b], ((j >> 1) - 1) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + b * BN;
        for (int kt = 0; kt < p.KT && ok; ++kt, ++i) {
          const int s = i % S;
          ok = mbar_wait(&full[s], (i / S) & 1, p.err);
          if (!ok) break;
          tc_fence_after();
          uint8_t* st = stage(s);
          const uint32_t sfa = tmem + 2 * BN + B::kSfCols * s;
          const uint32_t sfb = sfa + 16;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            tc_cp_sf(sfa + kb * 4, desc_sf(st + B::kOffSfa + 512 * kb));
            tc_cp_sf(sfb + kb * 4, desc_sf(st + B::kOffSfb + 512 * kb));
          }
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            mma_mxf4nvf4_4x(d, desc_sw128(st + 32 * kb), desc_sw128(st + B::kOffB + 32 * kb),
                            idesc, sfa + kb * 4, sfb + kb * 4, (kt > 0 || kb > 0) ? 1u : 0u);
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[b]);
      }
    }
  } else if (warp >= 4) {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                  // row of the 128-row block
    float(*sy)[32] = s_y[quad];
    int j = 0, cur_tile = -1, n = 0;
    float gs = 0.f;
    for (int u = u_begin; u < u_end; ++u, ++j) {
      const int tile = u / p.RB, rb = u - tile * p.RB;
      if (tile != cur_tile) {
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int4 td = p.tiles[tile];
        n = td.z;
        gs = p.gscale[td.x] / p.agscale[td.x];
        if (row < n) {
          const int f = p.perm[td.y + row];
          s_f[row] = f;
          s_w[row] = p.topk_w[f];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        cur_tile = tile;
      }
      const int h4 = rb * 128 + quad * 32 + 4 * (lane & 7);
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[b], (j >> 1) & 1, p.err));
      tc_fence_after();
      __syncwarp();
      const uint32_t trow = tmem + b * BN + ((uint32_t)(quad * 32) << 16);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float y[16];
        tmem_ld16(trow + c0, y);
        if (!ok || c0 >= n) continue;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sy[jj][lane] = y[jj] * gs;
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int cc = 4 * r + (lane >> 3);
          if (c0 + cc < n) {
            const float4 v = *reinterpret_cast<const float4*>(&sy[cc][4 * (lane & 7)]);
            const int f = s_f[c0 + cc];
            const float wt = s_w[c0 + cc];
            const float4 o = make_float4(wt * v.x, wt * v.y, wt * v.z, wt * v.w);
            if (p.deterministic)
              *reinterpret_cast<float4*>(p.rbuf + (size_t)f * p.H + h4) = o;
            else
              atomicAdd(reinterpret_cast<float4*>(p.acc + (size_t)(f / p.topk) * p.H + h4), o);
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }
  if (!ok) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  // a wait gave up: let this CTA's copies land before its shared memory is released
  if (s_fail && warp == 0 && lane == 0) drain_stage_loads<S>(full, issued, p.err);
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc);
}

// ---------------------------------------------------------------------------------- host side

EncodeTiledFn tc_encode_fn();

// Packed E2M1 activations [rows][K/2] bytes: boxes of 128 bytes (256 K) x box_rows, 128-byte
// swizzle.
static bool tmap_fp4_act(CUtensorMap* tm, const void* base, int K, int rows, int box_rows) {
  EncodeTiledFn enc = tc_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool FC2>
static cudaError_t launch4(const Tc4Params& p, int tiles, cudaStream_t st) {
  using Cfg = Tc4Cfg<BN, FC2>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(gemm_tc4_kernel<BN, FC2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Cfg::kSmem);
    cudaFuncSetAttribute(gemm_tc4_kernel<BN, FC2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    attr = true;
  }
  dim3 grid(tiles, p.RB, FC2 ? 1 : p.splits);
  return launch_kernel(gemm_tc4_kernel<BN, FC2>, grid, dim3(kTcThreads), Cfg::kSmem, st, true,
                       p);
}

template <int BN>
static cudaError_t launch4_persist(const Tc4Params& p, int tiles, cudaStream_t st) {
  using Cfg = Tc4PersistCfg<BN>;
  static const int G = persistent_grid(fc2_tc4_persist_kernel<BN>, Cfg::kSmem, Cfg::kAlloc, 2,
                                       1 << 20);
  const int grid = std::max(1, std::min(G, tiles * p.RB));
  return launch_kernel(fc2_tc4_persist_kernel<BN>, dim3(grid), dim3(k4PThreads), Cfg::kSmem, st,
                       true, p);
}

// Token-tile width of the W4A4 kernels.
int tc4_pick_bn(int M) { return M <= 16 ? 16 : (M <= 64 ? 32 : 64); }

// stage 0: fc1 (+ SwiGLU, NVFP4 requantisation of h), stage 1: fc2 (+ combine).
cudaError_t launch_tc4_stage(int stage, const DevWeights& w, const RunPtrs& r, const PlanDims& d,
                             int bn, int tiles, int splits, const float* topk_w, int M,
                             cudaStream_t st) {
  const int Sm = M * d.topk;
  const bool fc2 = stage == 1;
  Tc4Params p;
  memset(&p, 0, sizeof(p));
  p.K = fc2 ? d.Ip : d.H;
  p.KT = cdiv(p.K, 256);
  if (!tmap_fp4_act(&p.tm_act, fc2 ? (const void*)r.hq : (const void*)r.xq, p.K, Sm,
                    bn < 32 ? bn : 32))
    return cudaErrorInvalidValue;
  p.codes = fc2 ? w.w2 : w.w13;
  p.sfa = fc2 ? w.s2 : w.s13;
  p.sfb = fc2 ? r.hs16 : r.xs16;
  p.r16 = r.r16;
  p.gscale = fc2 ? w.g2 : w.g13;
  p.agscale = fc2 ? w.ag2 : w.ag13;
  p.agscale2 = w.ag2;
  p.tiles = r.tiles; p.ctrl = r.ctrl; p.err = r.ctrl;
  p.hq = r.hq; p.hs = r.hs16; p.gacc = r.g; p.tickets = r.tickets;
  p.perm = r.perm; p.topk_w = topk_w; p.acc = r.acc; p.rbuf = r.rbuf;
  p.I = d.I; p.Ip = d.Ip; p.RB = fc2 ? d.H / 128 : cdiv(d.I, 128);
  p.Sm = Sm; p.splits = fc2 ? 1 : splits; p.topk = d.topk;
  p.deterministic = d.deterministic; p.H = d.H;
  p.limit = d.limit; p.alpha = d.alpha; p.beta = d.beta;
  switch (bn * 2 + (fc2 ? 1 : 0)) {
    case 32: return launch4<16, false>(p, tiles, st);
    case 33: return launch4_persist<16>(p, tiles, st);
    case 64: return launch4<32, false>(p, tiles, st);
    case 65: return launch4_persist<32>(p, tiles, st);
    case 128: return launch4<64, false>(p, tiles, st);
    case 129: return launch4<64, true>(p, tiles, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
