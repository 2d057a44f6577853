// route.cu - routing (per-expert histogram, prefix sum, stable slot permutation, GEMM tile
// list) and MXFP8 activation quantisation.
//
// Routing follows the pages' route planners (hybrid_loader.py: packed_route_indices /
// expert_offsets / block_expert_ids handed to run_w4a16_moe; moe_b12x_next.py knob
// _DIRECT_IDS: ids outside [0, E) are skipped).  The slots of expert e are listed in ascending
// flat index t*k + j, so the permutation is unique and can be compared bit for bit.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kMaxRouteExperts = 1024;  // shared-memory tables below

// Exclusive block scan of one value per thread over NW warps; returns the prefix, *total = sum.
template <int NW>
__device__ int block_excl_scan_n(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive prefix of warp sums
  }
  __syncthreads();
  int warp_base = warp ? s_warp[warp - 1] : 0;
  int t = s_warp[NW - 1];
  __syncthreads();
  *total = t;
  return warp_base + x - v;
}

// Exclusive block scan of one value per thread; returns the prefix, *total = sum.
__device__ int block_excl_scan(int v, int* total, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kRouteWarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive prefix of warp sums
  }
  __syncthreads();
  int warp_base = warp ? s_warp[warp - 1] : 0;
  int t = s_warp[kRouteWarps - 1];
  __syncthreads();
  *total = t;
  return warp_base + x - v;
}

// One CTA of 1024 threads routes the whole call.
//   cnt[e], off[e] (off[E] = S), perm[S] = flat slot ids grouped by expert in ascending order,
//   slot_of[f] = position of flat slot f or -1, tiles = {expert, first position, count} for
//   every run of up to `tile_slots` consecutive positions of one expert; ctrl[1] = tile count,
//   ctrl[2] = S.
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const int32_t* __restrict__ ids, int Mk, int E, int tile_slots, int max_tiles,
             int32_t* __restrict__ cnt, int32_t* __restrict__ off, int32_t* __restrict__ perm,
             int32_t* __restrict__ slot_of, int4* __restrict__ tiles, int32_t* __restrict__ ctrl,
             int ep_first) {
  __shared__ int s_cnt[kMaxRouteExperts];
  __shared__ int s_base[kMaxRouteExperts];
  __shared__ int s_wc[kRouteWarps][kMaxRouteExperts / 4];  // per-warp counts, 8 bits each
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait_prev();     // previous kernel of the call complete, its writes visible
  pdl_launch_next();

  if (tid == 0) ctrl[0] = 0;  // error word of this call
  for (int e = tid; e < E; e += kRouteThreads) s_cnt[e] = 0;
  for (int i = tid; i < kRouteWarps * (kMaxRouteExperts / 4); i += kRouteThreads)
    (&s_wc[0][0])[i] = 0;
  __syncthreads();
  for (int f = tid; f < Mk; f += kRouteThreads) {
    int e = local_expert(ids[f], ep_first, E);
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();

  // prefix over experts: thread t owns experts [t*per, t*per + per)
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  int local = 0, ltiles = 0;
  for (int i = 0; i < per; ++i) {
    int e = tid * per + i;
    if (e < E) {
      local += s_cnt[e];
      ltiles += (s_cnt[e] + tile_slots - 1) / tile_slots;
    }
  }
  int total;
  int base = block_excl_scan(local, &total, s_warp);
  int ttotal;
  int tbase = block_excl_scan(ltiles, &ttotal, s_warp);
  for (int i = 0; i < per; ++i) {
    int e = tid * per + i;
    if (e < E) {
      int c = s_cnt[e];
      cnt[e] = c;
      off[e] = base;
      s_base[e] = base;
      for (int p = 0; p < c; p += tile_slots) {
        if (tbase < max_tiles)
          tiles[tbase] = make_int4(e, base + p, min(tile_slots, c - p), 0);
        else
          set_error(ctrl, kErrTileOverflow);
        ++tbase;
      }
      base += c;
    }
  }
  if (tid == 0) {
    off[E] = total;
    ctrl[1] = min(ttotal, max_tiles);
    ctrl[2] = total;
  }
  __syncthreads();

  // stable scatter, 1024 flat slots per round in order
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = 0; r0 < Mk; r0 += kRouteThreads) {
    const int f = r0 + tid;
    int e = f < Mk ? local_expert(ids[f], ep_first, E) : -1;
    const bool valid = f < Mk && e >= 0 && e < E;
    const int key = valid ? e : (E + lane);  // invalid slots never match a valid one
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(peers & lt_mask);
    const int wcount = __popc(peers);
    const bool leader = rank == 0;
    // per-warp counts, 8 bits each (a warp has at most 32 slots of one expert)
    if (valid && leader) atomicAdd(&s_wc[warp][e >> 2], wcount << ((e & 3) * 8));
    __syncthreads();
    int pos = -1;
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += (s_wc[w][e >> 2] >> ((e & 3) * 8)) & 0xFF;
      pos = s_base[e] + before + rank;
    }
    __syncthreads();
    if (valid && leader) {
      atomicAdd(&s_base[e], wcount);
      atomicAnd(&s_wc[warp][e >> 2], ~(0xFF << ((e & 3) * 8)));
    }
    if (f < Mk) {
      slot_of[f] = pos;
      if (valid) {
        if (pos >= 0 && pos < total) perm[pos] = f;
        else set_error(ctrl, kErrRouteBounds);
      }
    }
    __syncthreads();
  }
}

// MXFP8 quantisation of x (W4A8) into slot order: one thread per block of 32 elements of the
// row of the token that owns slot position p, so every GEMM tile reads contiguous rows.
// The same launch clears the buffers that the later stages accumulate into.
// One block of 32 bf16 activations -> 32 E4M3 codes + the E8M0 scale byte (OCP MX rule:
// scale = 2^(floor(log2 amax) - 8), codes round to nearest even with saturation).
__device__ __forceinline__ uint32_t quantize_block32(const __nv_bfloat16* __restrict__ src_bf16,
                                                     uint8_t* __restrict__ q,
                                                     uint8_t* __restrict__ s8) {
  const uint4* src = reinterpret_cast<const uint4*>(src_bf16);
  const uint4 u[4] = {src[0], src[1], src[2], src[3]};
  uint32_t packed[8];
  const uint32_t s = mxfp8_block32(u, packed);
  uint4* dst = reinterpret_cast<uint4*>(q);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  *s8 = (uint8_t)s;
  return s;
}

struct ZeroRegion {
  void* ptr;
  size_t words;   // 4-byte words, a multiple of 4
};

// Eight bf16 values -> f16 (exact within the f16 range; `ok` cleared when one lies outside it).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 u, bool& ok) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
    ok &= fabsf(a) <= 65504.f && fabsf(b) <= 65504.f;
    o[j] = (uint32_t)__half_as_ushort(__float2half_rn(a)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Eight bf16 values scaled by a router weight already rounded to bf16: bf16(x * w) each (the
// product of two bf16 values is exact in fp32, then rounded to nearest even).
__device__ __forceinline__ uint4 bf16x8_scale(uint4 u, float wb) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = __uint_as_float(w[j] << 16) * wb;
    const float b = __uint_as_float(w[j] & 0xFFFF0000u) * wb;
    o[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Whether slot expert e takes the kept tier's static FP8 activations.
__device__ __forceinline__ bool kept_a8_expert(const KeptA8& k, int e) {
  return k.tiers != nullptr && e >= 0 && (k.tiers[e] >> 24) == kTierNVFP4;
}

// Eight bf16 values as static per-tensor FP8: the E4M3 code of fp32(x) * inv (nearest even,
// saturating at 448), stored as the f16 of the code's value (E4M3 values are exact in f16).
__device__ __forceinline__ uint4 bf16x8_to_fp8s_f16x8(uint4 u, float inv) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float a = e4m3_to_f32((uint8_t)f32_to_e4m3(__fmul_rn(__uint_as_float(w[j] << 16), inv)));
    const float b =
        e4m3_to_f32((uint8_t)f32_to_e4m3(__fmul_rn(__uint_as_float(w[j] & 0xFFFF0000u), inv)));
    o[j] = (uint32_t)__half_as_ushort(__float2half_rn(a)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(b)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// NVFP4 weights with MXFP8 activations: 32 activations times the expert's activation global
// scale `a` (fp32 products), quantised by the OCP MX rule (as quantize_block32) and stored as the
// f16 of each dequantised value E4M3 x 2^(s-127): exact while the block scale is within
// [2^-15, 2^7]; a larger one (values beyond f16) clears `ok`, a smaller one rounds the values'
// bits below 2^-24.
__device__ __forceinline__ void mx_roundtrip32_f16(const __nv_bfloat16* __restrict__ src_bf16,
                                                   float a, uint16_t* __restrict__ dst, bool& ok) {
  const uint4* src = reinterpret_cast<const uint4*>(src_bf16);
  float v[32];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    const uint4 u = src[qq];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[qq * 8 + 2 * j] = __uint_as_float(w[j] << 16) * a;
      v[qq * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * a;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint32_t s = mx_scale_byte(amax);
  const float inv = e8m0_inv_f32(s), sc = e8m0_to_f32(s);
  ok &= s <= 127 + 7;
  uint32_t o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float q0 = e4m3_to_f32((uint8_t)f32_to_e4m3(v[2 * j] * inv)) * sc;
    const float q1 = e4m3_to_f32((uint8_t)f32_to_e4m3(v[2 * j + 1] * inv)) * sc;
    o[j] = (uint32_t)__half_as_ushort(__float2half_rn(q0)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(q1)) << 16);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) d[qq] = make_uint4(o[4 * qq], o[4 * qq + 1], o[4 * qq + 2], o[4 * qq + 3]);
}

// NVFP4 activations (W4A4): 16 activations times the expert's activation global scale `a`
// (fp32 products) -> block scale E4M3(vmax / 6), E2M1 codes nearest-even of v / scale (zero
// when the scale is 0), packed two per byte (element 2i in the low nibble) into q8[0..7].
__device__ __forceinline__ uint32_t nvfp4_quant16(const __nv_bfloat16* __restrict__ src_bf16,
                                                  float a, uint8_t* __restrict__ q8) {
  const uint4* src = reinterpret_cast<const uint4*>(src_bf16);
  float v[16];
#pragma unroll
  for (int qq = 0; qq < 2; ++qq) {
    const uint4 u = src[qq];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[qq * 8 + 2 * j] = __uint_as_float(w[j] << 16) * a;
      v[qq * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * a;
    }
  }
  float vmax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) vmax = fmaxf(vmax, fabsf(v[j]));
  const uint32_t sc = f32_to_e4m3(__fdiv_rn(vmax, 6.f));
  const float sv = e4m3_to_f32((uint8_t)sc);
  uint32_t w2[2] = {0u, 0u};
  if (sv > 0.f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t c =
          (uint32_t)__nv_cvt_float_to_fp4(__fdiv_rn(v[j], sv), __NV_E2M1, cudaRoundNearest) & 0xF;
      w2[j >> 3] |= c << (4 * (j & 7));
    }
  }
  *reinterpret_cast<uint2*>(q8) = make_uint2(w2[0], w2[1]);
  return sc;
}

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

__global__ void __launch_bounds__(256)
actq_kernel(const __nv_bfloat16* __restrict__ x, int H, int topk, const int32_t* __restrict__ ctrl,
            const int32_t* __restrict__ perm, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
            uint8_t* __restrict__ xs16, int r16, uint16_t* __restrict__ x16,
            const float* __restrict__ win, const float* __restrict__ ag,
            const int32_t* __restrict__ ids, int ep_first, int E, uint8_t* __restrict__ xq4,
            uint8_t* __restrict__ xs4, int32_t* __restrict__ err, ZeroRegion z0, ZeroRegion z1,
            ZeroRegion z2, KeptA8 ka8) {
  pdl_wait_prev();
  pdl_launch_next();
  const size_t gtid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t gsz = (size_t)gridDim.x * blockDim.x;
  if (xq != nullptr) {
    const int nb = H / 32;
    const size_t nblk = (size_t)ctrl[2] * nb;
    for (size_t i = gtid; i < nblk; i += gsz) {
      const size_t p = i / nb;
      const int b = (int)(i % nb);
      const int t = perm[p] / topk;
      const uint32_t sb =
          quantize_block32(x + (size_t)t * H + b * 32, xq + p * H + b * 32, xs + p * nb + b);
      if (xs16 != nullptr) xs16[((size_t)(b >> 2) * r16 + p) * 16 + (b & 3)] = (uint8_t)sb;
    }
  }
  if (xq4 != nullptr) {
    // NVFP4 activations (W4A4): packed codes in slot order, scales in the atom rows
    const int nb = H / 16;
    const size_t nblk = (size_t)ctrl[2] * nb;
    for (size_t i = gtid; i < nblk; i += gsz) {
      const size_t p = i / nb;
      const int b = (int)(i % nb);
      const int f = perm[p];
      const int e = local_expert(ids[f], ep_first, E);
      const uint32_t sc = nvfp4_quant16(x + (size_t)(f / topk) * H + b * 16, ag[e],
                                        xq4 + p * (H / 2) + b * 8);
      xs4[((size_t)(b >> 2) * r16 + p) * 16 + (b & 3)] = (uint8_t)sc;
    }
  }
  if (x16 != nullptr && ag != nullptr) {
    // MXFP8 activations for NVFP4 weights, as f16 values in slot order
    const int nb = H / 32;
    const size_t nblk = (size_t)ctrl[2] * nb;
    bool range_ok = true;
    for (size_t i = gtid; i < nblk; i += gsz) {
      const size_t p = i / nb;
      const int b = (int)(i % nb);
      const int f = perm[p];
      const int e = local_expert(ids[f], ep_first, E);
      mx_roundtrip32_f16(x + (size_t)(f / topk) * H + b * 32, ag[e], x16 + p * H + b * 32,
                         range_ok);
    }
    if (!range_ok) atomicOr(err, kErrRange);
  } else if (x16 != nullptr) {
    // bf16 -> f16 copy in slot order for the 16-bit tensor-core path (exact within f16 range)
    const int nc = H / 8;
    const size_t nchunk = (size_t)ctrl[2] * nc;
    bool range_ok = true;
    for (size_t i = gtid; i < nchunk; i += gsz) {
      const size_t p = i / nc;
      const int c = (int)(i % nc);
      const int f = perm[p], t = f / topk;
      uint4 u = *reinterpret_cast<const uint4*>(x + (size_t)t * H + c * 8);
      if (ka8.tiers != nullptr && kept_a8_expert(ka8, local_expert(ids[f], ep_first, E))) {
        *reinterpret_cast<uint4*>(x16 + p * H + c * 8) = bf16x8_to_fp8s_f16x8(u, ka8.inv);
        continue;
      }
      if (win != nullptr) u = bf16x8_scale(u, bf16_round(win[f]));   // weight on the input
      *reinterpret_cast<uint4*>(x16 + p * H + c * 8) = bf16x8_to_f16x8(u, range_ok);
    }
    if (!range_ok) atomicOr(err, kErrRange);
  }
  const ZeroRegion zs[3] = {z0, z1, z2};
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    if (zs[r].ptr == nullptr) continue;
    uint4* a4 = reinterpret_cast<uint4*>(zs[r].ptr);
    for (size_t i = gtid; i < zs[r].words / 4; i += gsz) a4[i] = make_uint4(0, 0, 0, 0);
  }
}

// Small W4A8 calls (at most kSmallRouteSlots flat slots): routing and MXFP8 quantisation in one
// launch.  Every CTA routes the call in shared memory (the same tables as route_kernel: stable
// order, tiles of up to tile_slots positions), CTA 0 writes them out, and all CTAs quantise
// their share of the slot-ordered activation blocks and clear the accumulation buffers.
constexpr int kSmallRouteSlots = 256;
constexpr int kSmallRouteThreads = 256;

__global__ void __launch_bounds__(kSmallRouteThreads)
route_actq_small_kernel(const int32_t* __restrict__ ids, int Mk, int E, int tile_slots,
                        int max_tiles, const __nv_bfloat16* __restrict__ x, int H, int topk,
                        int32_t* __restrict__ cnt, int32_t* __restrict__ off,
                        int32_t* __restrict__ perm, int32_t* __restrict__ slot_of,
                        int4* __restrict__ tiles, int32_t* __restrict__ ctrl,
                        uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
                        uint8_t* __restrict__ xs16, int r16, uint16_t* __restrict__ x16,
                        const float* __restrict__ win, const float* __restrict__ ag,
                        uint8_t* __restrict__ xq4, uint8_t* __restrict__ xs4, ZeroRegion z0,
                        ZeroRegion z1, ZeroRegion z2, int ep_first, KeptA8 ka8) {
  constexpr int NW = kSmallRouteThreads / 32;
  __shared__ int s_ids[kSmallRouteSlots];
  __shared__ int s_perm[kSmallRouteSlots];
  __shared__ int s_warp[32];
  // per-expert counts, sized to E by the launch: a small footprint lets this kernel's CTAs sit
  // beside two CTAs of the next kernel (which launches as soon as this one starts) on an SM
  extern __shared__ int s_cnt[];
  const int tid = threadIdx.x;
  const bool writer = blockIdx.x == 0;
  pdl_wait_prev();
  pdl_launch_next();

  if (writer && tid == 0) ctrl[0] = 0;  // error word of this call
  for (int e = tid; e < E; e += kSmallRouteThreads) s_cnt[e] = 0;
  for (int f = tid; f < kSmallRouteSlots; f += kSmallRouteThreads) {
    const int e = f < Mk ? local_expert(ids[f], ep_first, E) : -1;
    s_ids[f] = (e >= 0 && e < E) ? e : -1;
  }
  __syncthreads();
  for (int f = tid; f < Mk; f += kSmallRouteThreads)
    if (s_ids[f] >= 0) atomicAdd(&s_cnt[s_ids[f]], 1);
  __syncthreads();

  // prefix over experts (thread t owns experts [t*per, t*per + per)), and over their tiles
  const int per = (E + kSmallRouteThreads - 1) / kSmallRouteThreads;
  int local = 0, ltiles = 0;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < E) {
      local += s_cnt[e];
      ltiles += (s_cnt[e] + tile_slots - 1) / tile_slots;
    }
  }
  int total, ttotal;
  int base = block_excl_scan_n<NW>(local, &total, s_warp);
  int tbase = block_excl_scan_n<NW>(ltiles, &ttotal, s_warp);
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < E) {
      const int c = s_cnt[e];
      if (writer) {
        cnt[e] = c;
        off[e] = base;
        for (int p = 0; p < c; p += tile_slots) {
          if (tbase < max_tiles)
            tiles[tbase] = make_int4(e, base + p, min(tile_slots, c - p), 0);
          else
            set_error(ctrl, kErrTileOverflow);
          ++tbase;
        }
      }
      s_cnt[e] = base;   // now the expert's first position
      base += c;
    }
  }
  if (writer && tid == 0) {
    off[E] = total;
    ctrl[1] = min(ttotal, max_tiles);
    ctrl[2] = total;
  }
  __syncthreads();
  // stable positions: earlier flat slots of the same expert come first
  for (int f = tid; f < Mk; f += kSmallRouteThreads) {
    const int e = s_ids[f];
    int pos = -1;
    if (e >= 0) {
      int rank = 0;
      for (int g = 0; g < f; ++g) rank += s_ids[g] == e;
      pos = s_cnt[e] + rank;
      s_perm[pos] = f;
      if (writer) perm[pos] = f;
    }
    if (writer) slot_of[f] = pos;
  }
  __syncthreads();

  // MXFP8 quantisation (W4A8) or the f16 copy (16-bit tensor-core path) of the slot-ordered
  // rows, as actq_kernel does
  const size_t gtid = (size_t)blockIdx.x * blockDim.x + tid;
  const size_t gsz = (size_t)gridDim.x * blockDim.x;
  if (xq != nullptr) {
    const int nb = H / 32;
    const size_t nblk = (size_t)total * nb;
    for (size_t i = gtid; i < nblk; i += gsz) {
      const size_t p = i / nb;
      const int b = (int)(i % nb);
      const int t = s_perm[p] / topk;
      const uint32_t sb =
          quantize_block32(x + (size_t)t * H + b * 32, xq + p * H + b * 32, xs + p * nb + b);
      if (xs16 != nullptr) xs16[((size_t)(b >> 2) * r16 + p) * 16 + (b & 3)] = (uint8_t)sb;
    }
  }
  if (xq4 != nullptr) {
    // NVFP4 activations (W4A4): packed codes in slot order, scales in the atom rows
    const int nb = H / 16;
    const size_t nblk = (size_t)total * nb;
    for (size_t i = gtid; i < nblk; i += gsz) {
      const size_t p = i / nb;
      const int b = (int)(i % nb);
      const int f = s_perm[p];
      const uint32_t sc = nvfp4_quant16(x + (size_t)(f / topk) * H + b * 16, ag[s_ids[f]],
                                        xq4 + p * (H / 2) + b * 8);
      xs4[((size_t)(b >> 2) * r16 + p) * 16 + (b & 3)] = (uint8_t)sc;
    }
  }
  if (x16 != nullptr && ag != nullptr) {
    // MXFP8 activations for NVFP4 weights, as f16 values in slot order
    const int nb = H / 32;
    const size_t nblk = (size_t)total * nb;
    bool range_ok = true;
    for (size_t i = gtid; i < nblk; i += gsz) {
      const size_t p = i / nb;
      const int b = (int)(i % nb);
      const int f = s_perm[p];
      mx_roundtrip32_f16(x + (size_t)(f / topk) * H + b * 32, ag[s_ids[f]],
                         x16 + p * H + b * 32, range_ok);
    }
    if (!range_ok) atomicOr(ctrl, kErrRange);
  } else if (x16 != nullptr) {
    const int nc = H / 8;
    const size_t nchunk = (size_t)total * nc;
    bool range_ok = true;
    for (size_t i = gtid; i < nchunk; i += gsz) {
      const size_t p = i / nc;
      const int c = (int)(i % nc);
      const int f = s_perm[p], t = f / topk;
      uint4 u = *reinterpret_cast<const uint4*>(x + (size_t)t * H + c * 8);
      if (kept_a8_expert(ka8, s_ids[f])) {
        *reinterpret_cast<uint4*>(x16 + p * H + c * 8) = bf16x8_to_fp8s_f16x8(u, ka8.inv);
        continue;
      }
      if (win != nullptr) u = bf16x8_scale(u, bf16_round(win[f]));   // weight on the input
      *reinterpret_cast<uint4*>(x16 + p * H + c * 8) = bf16x8_to_f16x8(u, range_ok);
    }
    if (!range_ok) atomicOr(ctrl, kErrRange);
  }
  const ZeroRegion zs[3] = {z0, z1, z2};
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    if (zs[r].ptr == nullptr) continue;
    uint4* a4 = reinterpret_cast<uint4*>(zs[r].ptr);
    for (size_t i = gtid; i < zs[r].words / 4; i += gsz) a4[i] = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------------------------------------
// Larger W4A8 calls: routing spread over CTAs of kChunkSlots flat slots each, then the MXFP8
// quantisation of the slot-ordered rows, in three launches.
//   route_count_kernel: per-chunk expert counts cc[c][e].
//   route_scatter_kernel: one CTA per chunk adds up the chunk counts into the expert totals and
//     its chunk's bases base[e] = off[e] + (slots of e in earlier chunks) and ranks the chunk's
//     slots (stable: by flat index within each expert, the same ranking as route_kernel's
//     rounds) into perm / slot_of; CTA 0 writes cnt / off / tiles / ctrl.
//   actq_rows_kernel: one warp per slot position quantises its token's row.
// Same tables and codes, bit for bit, as route_kernel + actq_kernel.
constexpr int kChunkSlots = 1024;

__global__ void __launch_bounds__(kRouteThreads)
route_count_kernel(const int32_t* __restrict__ ids, int Mk, int E, int32_t* __restrict__ ctrl,
                   int32_t* __restrict__ cc, int ep_first) {
  __shared__ int s_cnt[kMaxRouteExperts];
  const int tid = threadIdx.x, c = blockIdx.x;
  pdl_wait_prev();     // previous kernel of the call complete, its writes visible
  pdl_launch_next();
  if (c == 0 && tid == 0) ctrl[0] = 0;  // error word of this call
  for (int e = tid; e < E; e += kRouteThreads) s_cnt[e] = 0;
  __syncthreads();
  const int f = c * kChunkSlots + tid;
  if (f < Mk) {
    const int e = local_expert(ids[f], ep_first, E);
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += kRouteThreads) cc[(size_t)c * E + e] = s_cnt[e];
}

__global__ void __launch_bounds__(kRouteThreads)
route_scatter_kernel(const int32_t* __restrict__ ids, int Mk, int E, int tile_slots,
                     int max_tiles, const int32_t* __restrict__ cc, int32_t* __restrict__ cnt,
                     int32_t* __restrict__ off, int32_t* __restrict__ perm,
                     int32_t* __restrict__ slot_of, int4* __restrict__ tiles,
                     int32_t* __restrict__ ctrl, int ep_first) {
  __shared__ int s_base[kMaxRouteExperts];
  __shared__ int s_wc[kRouteWarps][kMaxRouteExperts / 4];  // per-warp counts, 8 bits each
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = gridDim.x, c = blockIdx.x;
  const bool writer = c == 0;
  pdl_wait_prev();     // chunk counts written
  pdl_launch_next();
  for (int i = tid; i < kRouteWarps * (kMaxRouteExperts / 4); i += kRouteThreads)
    (&s_wc[0][0])[i] = 0;

  // expert totals and this chunk's bases: thread t owns expert t (E <= kRouteThreads)
  int tot = 0, mine = 0;
  if (tid < E) {
    for (int q = 0; q < nch; ++q) {
      const int v = cc[(size_t)q * E + tid];
      mine += q < c ? v : 0;
      tot += v;
    }
  }
  int total, ttotal;
  const int base = block_excl_scan(tot, &total, s_warp);
  int tbase = block_excl_scan((tot + tile_slots - 1) / tile_slots, &ttotal, s_warp);
  if (tid < E) {
    s_base[tid] = base + mine;
    if (writer) {
      cnt[tid] = tot;
      off[tid] = base;
      for (int p = 0; p < tot; p += tile_slots, ++tbase) {
        if (tbase < max_tiles)
          tiles[tbase] = make_int4(tid, base + p, min(tile_slots, tot - p), 0);
        else
          set_error(ctrl, kErrTileOverflow);
      }
    }
  }
  if (writer && tid == 0) {
    off[E] = total;
    ctrl[1] = min(ttotal, max_tiles);
    ctrl[2] = total;
  }
  __syncthreads();

  const int f = c * kChunkSlots + tid;
  const int e = f < Mk ? local_expert(ids[f], ep_first, E) : -1;
  const bool valid = f < Mk && e >= 0 && e < E;
  const int key = valid ? e : (E + lane);  // invalid slots never match a valid one
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && rank == 0) atomicAdd(&s_wc[warp][e >> 2], __popc(peers) << ((e & 3) * 8));
  __syncthreads();
  if (f < Mk) {
    int pos = -1;
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += (s_wc[w][e >> 2] >> ((e & 3) * 8)) & 0xFF;
      pos = s_base[e] + before + rank;
      if (pos < total) {
        perm[pos] = f;
      } else {
        set_error(ctrl, kErrRouteBounds);
        pos = -1;
      }
    }
    slot_of[f] = pos;
  }
}

// MXFP8 quantisation of x into slot order, token by token: a token's row is read and quantised
// once and its codes stored at the slot position of each of its valid slots (slot_of).  Work
// items of one warp: 1024 consecutive elements of one token row (four segments of 256).  A lane
// loads one 16-byte chunk (8 elements) per segment - all four loads issued before any is used -
// four lanes share a block of 32 and its scale (amax over the group by shuffles), and the 16
// lanes of a 128-element K tile hand their four scales to one lane, which writes the tile's
// scale atom row (4 scale bytes, 12 zero bytes) with one 16-byte store.  Codes and scales are
// those of quantize_block32.  The same launch clears the buffers that the later stages
// accumulate into.
constexpr int kActqSegs = 4;

__global__ void __launch_bounds__(256)
actq_rows_kernel(const __nv_bfloat16* __restrict__ x, int M, int H, int topk,
                 const int32_t* __restrict__ slot_of, uint8_t* __restrict__ xq,
                 uint8_t* __restrict__ xs, uint8_t* __restrict__ xs16, int r16, ZeroRegion z0,
                 ZeroRegion z1, ZeroRegion z2) {
  pdl_wait_prev();
  pdl_launch_next();
  const int lane = threadIdx.x & 31;
  const size_t gtid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t gsz = (size_t)gridDim.x * blockDim.x;
  const int nb = H / 32, nc = H / 8;           // blocks, 16-byte chunks per row (nc % 16 == 0)
  const int per_row = (nc + 32 * kActqSegs - 1) / (32 * kActqSegs);   // work items per row
  const size_t items = (size_t)M * per_row;
  for (size_t it = gtid >> 5; it < items; it += gsz >> 5) {
    const size_t t = it / per_row;
    const int c0 = (int)(it - t * per_row) * 32 * kActqSegs;
    // slot positions of the token's top-k slots (-1: dropped), lane j holding slot j
    const int mypos = lane < topk ? slot_of[t * topk + lane] : -1;
    if (!__any_sync(0xffffffffu, mypos >= 0)) continue;   // padding row
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4 u[kActqSegs];
#pragma unroll
    for (int k = 0; k < kActqSegs; ++k) {
      const int c = c0 + 32 * k + lane;
      u[k] = c < nc ? src[c] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kActqSegs; ++k) {
      const int c = c0 + 32 * k + lane;
      const bool in = c < nc;                  // uniform per 16-lane half
      const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const uint32_t sc = mx_scale_byte(amax);
      const float inv = e8m0_inv_f32(sc);
      uint32_t q[2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
        q[h] = f32_to_e4m3(v[4 * h] * inv) | (f32_to_e4m3(v[4 * h + 1] * inv) << 8) |
               (f32_to_e4m3(v[4 * h + 2] * inv) << 16) | (f32_to_e4m3(v[4 * h + 3] * inv) << 24);
      const int g = lane & ~15;                // first lane of this K tile's 16
      const uint32_t atom = __shfl_sync(0xffffffffu, sc, g) |
                            (__shfl_sync(0xffffffffu, sc, g + 4) << 8) |
                            (__shfl_sync(0xffffffffu, sc, g + 8) << 16) |
                            (__shfl_sync(0xffffffffu, sc, g + 12) << 24);
      for (int j = 0; j < topk; ++j) {
        const int p = __shfl_sync(0xffffffffu, mypos, j);
        if (p < 0 || !in) continue;
        reinterpret_cast<uint2*>(xq + (size_t)p * H)[c] = make_uint2(q[0], q[1]);
        if ((c & 3) == 0) xs[(size_t)p * nb + (c >> 2)] = (uint8_t)sc;
        if ((c & 15) == 0)
          *reinterpret_cast<uint4*>(xs16 + ((size_t)(c >> 4) * r16 + p) * 16) =
              make_uint4(atom, 0u, 0u, 0u);
      }
    }
  }
  const ZeroRegion zs[3] = {z0, z1, z2};
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    if (zs[r].ptr == nullptr) continue;
    uint4* a4 = reinterpret_cast<uint4*>(zs[r].ptr);
    for (size_t i = gtid; i < zs[r].words / 4; i += gsz) a4[i] = make_uint4(0, 0, 0, 0);
  }
}

// bf16 -> f16 rows of the 16-bit tensor-core path in slot order, token by token (as
// actq_rows_kernel does for MXFP8): a warp takes 32 * kActqSegs 16-byte chunks of one token row,
// loads each once and stores it, converted, at the position of every valid slot of the token;
// the router weight on the input and the kept tier's static FP8 values apply per slot, as in
// actq_kernel.  The same launch clears the buffers that the later stages accumulate into.
__global__ void __launch_bounds__(256)
actq16_rows_kernel(const __nv_bfloat16* __restrict__ x, int M, int H, int topk,
                   const int32_t* __restrict__ slot_of, uint16_t* __restrict__ x16,
                   const float* __restrict__ win, const int32_t* __restrict__ ids, int ep_first,
                   int E, int32_t* __restrict__ err, ZeroRegion z0, ZeroRegion z1, ZeroRegion z2,
                   KeptA8 ka8) {
  pdl_wait_prev();
  pdl_launch_next();
  const int lane = threadIdx.x & 31;
  const size_t gtid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t gsz = (size_t)gridDim.x * blockDim.x;
  const int nc = H / 8;                        // 16-byte chunks per row
  const int per_row = (nc + 32 * kActqSegs - 1) / (32 * kActqSegs);
  const size_t items = (size_t)M * per_row;
  bool range_ok = true;
  for (size_t it = gtid >> 5; it < items; it += gsz >> 5) {
    const size_t t = it / per_row;
    const int c0 = (int)(it - t * per_row) * 32 * kActqSegs;
    // lane j: slot j of the token - its position (-1: dropped), whether its expert is a kept
    // tier expert with static FP8 activations, its router weight when that scales the input
    const size_t fj = t * topk + lane;
    const int mypos = lane < topk ? slot_of[fj] : -1;
    if (!__any_sync(0xffffffffu, mypos >= 0)) continue;   // padding row
    const bool my_a8 = mypos >= 0 && ka8.tiers != nullptr &&
                       kept_a8_expert(ka8, local_expert(ids[fj], ep_first, E));
    const float my_w = (mypos >= 0 && win != nullptr) ? bf16_round(win[fj]) : 1.f;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4 u[kActqSegs];
#pragma unroll
    for (int k = 0; k < kActqSegs; ++k) {
      const int c = c0 + 32 * k + lane;
      u[k] = c < nc ? src[c] : make_uint4(0, 0, 0, 0);
    }
    for (int j = 0; j < topk; ++j) {
      const int p = __shfl_sync(0xffffffffu, mypos, j);
      const bool a8 = __shfl_sync(0xffffffffu, my_a8 ? 1 : 0, j) != 0;
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      if (p < 0) continue;                     // uniform across the warp
#pragma unroll
      for (int k = 0; k < kActqSegs; ++k) {
        const int c = c0 + 32 * k + lane;
        if (c >= nc) continue;
        uint4 v = u[k];
        if (a8) {
          v = bf16x8_to_fp8s_f16x8(v, ka8.inv);
        } else {
          if (win != nullptr) v = bf16x8_scale(v, wj);   // weight on the input
          v = bf16x8_to_f16x8(v, range_ok);
        }
        *reinterpret_cast<uint4*>(x16 + (size_t)p * H + c * 8) = v;
      }
    }
  }
  if (!range_ok) atomicOr(err, kErrRange);
  const ZeroRegion zs[3] = {z0, z1, z2};
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    if (zs[r].ptr == nullptr) continue;
    uint4* a4 = reinterpret_cast<uint4*>(zs[r].ptr);
    for (size_t i = gtid; i < zs[r].words / 4; i += gsz) a4[i] = make_uint4(0, 0, 0, 0);
  }
}

int route_chunks(int Mk) { return (Mk + kChunkSlots - 1) / kChunkSlots; }

cudaError_t launch_route_count(const int32_t* ids, int Mk, int E, int ep_first,
                               const RunPtrs& r, cudaStream_t st) {
  static_assert(kMaxRouteExperts <= kRouteThreads, "one expert per thread");
  if (E > kMaxRouteExperts || Mk < 1) return cudaErrorInvalidValue;
  // first kernel of a call: an ordinary launch (the previous call may still read the tables)
  static const bool carveout = prefer_max_shared(route_count_kernel);
  (void)carveout;
  return launch_kernel(route_count_kernel, dim3(route_chunks(Mk)), dim3(kRouteThreads), 0, st,
                       false, ids, Mk, E, r.ctrl, r.rcc, ep_first);
}

cudaError_t launch_route_scatter(const int32_t* ids, int Mk, int E, int ep_first, int tile_slots,
                                 int max_tiles, const RunPtrs& r, cudaStream_t st) {
  if (E > kMaxRouteExperts || Mk < 1) return cudaErrorInvalidValue;
  static const bool carveout = prefer_max_shared(route_scatter_kernel);
  (void)carveout;
  return launch_kernel(route_scatter_kernel, dim3(route_chunks(Mk)), dim3(kRouteThreads), 0, st,
                       true, ids, Mk, E, tile_slots, max_tiles,
                       static_cast<const int32_t*>(r.rcc), r.cnt, r.off, r.perm, r.slot_of,
                       r.tiles, r.ctrl, ep_first);
}

cudaError_t launch_actq16_rows(const void* x, int M, int H, int topk, const RunPtrs& r,
                               const float* win, const int32_t* ids, int ep_first, int E,
                               void* z0, size_t z0_words, void* z1, size_t z1_words, void* z2,
                               size_t z2_words, KeptA8 ka8, cudaStream_t st) {
  if (H % 8 != 0 || topk > 32) return cudaErrorInvalidValue;
  const size_t items = (size_t)M * ((H / 8 + 32 * kActqSegs - 1) / (32 * kActqSegs));
  const size_t work = std::max(items * 32,
                               std::max(z0_words / 4, std::max(z1_words / 4, z2_words / 4)));
  const int blocks = (int)std::max<size_t>(1, std::min<size_t>((work + 255) / 256, 152 * 8));
  static const bool carveout = prefer_max_shared(actq16_rows_kernel);
  (void)carveout;
  return launch_kernel(actq16_rows_kernel, dim3(blocks), dim3(256), 0, st, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), M, H, topk,
                       static_cast<const int32_t*>(r.slot_of), r.x16, win, ids, ep_first, E,
                       r.ctrl, ZeroRegion{z0, z0_words}, ZeroRegion{z1, z1_words},
                       ZeroRegion{z2, z2_words}, ka8);
}

cudaError_t launch_actq_rows(const void* x, int M, int H, int topk, const RunPtrs& r, void* z0,
                             size_t z0_words, void* z1, size_t z1_words, void* z2,
                             size_t z2_words, cudaStream_t st) {
  if (H % 128 != 0) return cudaErrorInvalidValue;
  // a warp per 1024 elements of a token row; zeroing in 16-byte words
  if (topk > 32) return cudaErrorInvalidValue;
  const size_t items = (size_t)M * ((H / 8 + 32 * kActqSegs - 1) / (32 * kActqSegs));
  const size_t work = std::max(items * 32,
                               std::max(z0_words / 4, std::max(z1_words / 4, z2_words / 4)));
  const int blocks = (int)std::max<size_t>(1, std::min<size_t>((work + 255) / 256, 152 * 8));
  static const bool carveout = prefer_max_shared(actq_rows_kernel);
  (void)carveout;
  return launch_kernel(actq_rows_kernel, dim3(blocks), dim3(256), 0, st, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), M, H, topk,
                       static_cast<const int32_t*>(r.slot_of), r.xq, r.xs, r.xs16, r.r16,
                       ZeroRegion{z0, z0_words},
                       ZeroRegion{z1, z1_words}, ZeroRegion{z2, z2_words});
}

bool route_actq_small_supported(int Mk, int E) {
  return Mk <= kSmallRouteSlots && E <= kMaxRouteExperts;
}

cudaError_t launch_route_actq_small(const int32_t* ids, int Mk, int E, int ep_first,
                                    int tile_slots, int max_tiles, const void* x, int H,
                                    int topk, const RunPtrs& r, bool atoms, bool to_f16,
                                    const float* win, const float* ag, bool nv4, bool skip_x,
                                    void* z0, size_t z0_words, void* z1, size_t z1_words,
                                    void* z2, size_t z2_words, KeptA8 ka8, cudaStream_t st) {
  if (!route_actq_small_supported(Mk, E)) return cudaErrorInvalidValue;
  // skip_x: the consumer quantises the activations itself (W4A8 only), this launch routes and
  // clears
  const size_t act_work = skip_x ? 0 : (size_t)Mk * (to_f16 ? H / 8 : (nv4 ? H / 16 : H / 32));
  const size_t work = std::max(act_work,
                               std::max(z0_words / 4, std::max(z1_words / 4, z2_words / 4)));
  int blocks = (int)std::min<size_t>((work + kSmallRouteThreads - 1) / kSmallRouteThreads,
                                     152 * 4);
  // routing and zeroing only (fc1 quantises): a few CTAs, so that the SMs they sit on are free
  // for fc1's second CTA (one of this kernel and two of fc1 do not fit an SM's shared memory)
  if (skip_x) blocks = std::min(blocks, 16);
  if (blocks < 1) blocks = 1;
  // first kernel of a call: an ordinary launch (the previous call may still read the tables)
  static const bool carveout = prefer_max_shared(route_actq_small_kernel);
  (void)carveout;
  return launch_kernel(route_actq_small_kernel, dim3(blocks), dim3(kSmallRouteThreads),
                       (size_t)E * sizeof(int), st, false, ids, Mk, E, tile_slots, max_tiles,
                       reinterpret_cast<const __nv_bfloat16*>(x), H, topk, r.cnt, r.off, r.perm,
                       r.slot_of, r.tiles, r.ctrl, (to_f16 || nv4 || skip_x) ? nullptr : r.xq,
                       (to_f16 || nv4 || skip_x) ? nullptr : r.xs,
                       (atoms && !to_f16 && !nv4 && !skip_x) ? r.xs16 : nullptr, r.r16,
                       to_f16 ? r.x16 : nullptr, to_f16 ? win : nullptr,
                       (to_f16 || nv4) ? ag : nullptr, nv4 ? r.xq : nullptr,
                       nv4 ? r.xs16 : nullptr, ZeroRegion{z0, z0_words},
                       ZeroRegion{z1, z1_words}, ZeroRegion{z2, z2_words}, ep_first,
                       to_f16 ? ka8 : KeptA8{nullptr, 0.f});
}

cudaError_t launch_route(const int32_t* ids, int Mk, int E, int ep_first, int tile_slots,
                         int max_tiles, const RunPtrs& r, cudaStream_t st) {
  // first kernel of a call: an ordinary launch (the previous call may still read the tables)
  static const bool carveout = prefer_max_shared(route_kernel);
  (void)carveout;
  return launch_kernel(route_kernel, dim3(1), dim3(kRouteThreads), 0, st, false, ids, Mk, E,
                       tile_slots, max_tiles, r.cnt, r.off, r.perm, r.slot_of, r.tiles, r.ctrl,
                       ep_first);
}

cudaError_t launch_actq(const void* x, int M, int H, int topk, const RunPtrs& r, bool quant_x,
                        bool atoms, bool to_f16, const float* win, const float* ag,
                        const int32_t* ids, int ep_first, int E, bool nv4, void* z0,
                        size_t z0_words, void* z1, size_t z1_words, void* z2, size_t z2_words,
                        KeptA8 ka8, cudaStream_t st) {
  const size_t work = std::max(
      std::max(quant_x ? (size_t)M * topk * (H / 32) : (size_t)0,
               (to_f16 || nv4) ? (size_t)M * topk * (H / 8) : (size_t)0),
      std::max(z0_words / 4, std::max(z1_words / 4, z2_words / 4)));
  int blocks = (int)std::min<size_t>((work + 255) / 256, 152 * 8);
  if (blocks < 1) blocks = 1;
  static const bool carveout = prefer_max_shared(actq_kernel);
  (void)carveout;
  return launch_kernel(actq_kernel, dim3(blocks), dim3(256), 0, st, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), H, topk,
                       static_cast<const int32_t*>(r.ctrl), static_cast<const int32_t*>(r.perm),
                       quant_x ? r.xq : nullptr, quant_x ? r.xs : nullptr,
                       (quant_x && atoms) ? r.xs16 : nullptr, r.r16,
                       to_f16 ? r.x16 : nullptr, to_f16 ? win : nullptr,
                       (to_f16 || nv4) ? ag : nullptr, ids, ep_first, E, nv4 ? r.xq : nullptr,
                       nv4 ? r.xs16 : nullptr, r.ctrl,
                       ZeroRegion{z0, z0_words},
                       ZeroRegion{z1, z1_words}, ZeroRegion{z2, z2_words},
                       to_f16 ? ka8 : KeptA8{nullptr, 0.f});
}

}  // namespace moe
