// gemm_simt.cu - CUDA-core grouped GEMMs (fc1, fc2), the SwiGLU + requantisation step and the
// combine.  This is the general path: every quant mode and every M; weights are dequantised
// element by element in registers and multiplied in fp32.
//
// Math (hybrid_loader.py `_apply_ref`, moe_b12x_next.py module docstring):
//   fc1:  G[p, r] = sum_k W13_e[r, k] * xhat[t, k]          (rows r: [up | gate])
//   act:  h = min(g, L) * sigmoid(alpha * min(g, L)) * (clamp(u, -L, L) + beta)
//         W4A8: h -> MXFP8 (E4M3 + E8M0 per 32);  W4A16: h -> bf16
//   fc2:  y[p, c] = sum_i W2_e[c, i] * hhat[p, i]
//   combine: out[t] = sum_j w[t, j] * y[slot(t, j)]   (fp32 atomics, or a route buffer + a
//         fixed-order top-k sum; moe_b12x_next.py knob _DETERMINISTIC)
#include <algorithm>

#include "moe_common.cuh"

namespace moe {

__constant__ float c_nf3_lut[8] = {-1.0f, -0.6047f, -0.3563f, -0.1275f,
                                   0.1275f, 0.3563f,  0.6047f,  1.0f};

constexpr int kSimtThreads = 256;
constexpr int kSimtRowsPerCta = 32;     // 8 warps x 4 rows
constexpr int kSimtKChunk = 1024;

enum WeightKind { kKindMXFP4 = 0, kKindNVFP4 = 1, kKindNF3 = 2 };

struct SimtArgs {
  DevWeights w;
  RunPtrs r;
  const void* x;               // bf16 [M][H]
  const float* topk_w;         // [M][k] combine weights; nullptr: 1 (weights on the input)
  const float* win;            // [M][k] router weights applied to fc1's input, or nullptr
  int M, topk, H, I, Ip, E;
  int quant, deterministic;
};

// Weight kind and tier-local index of expert e.
__device__ __forceinline__ void resolve_expert(const DevWeights& w, int e, int& kind, int& le) {
  if (w.quant == kQuantW4A8) {
    kind = kKindMXFP4;
    le = e;
  } else if (w.quant == kQuantNVFP4) {
    kind = kKindNVFP4;
    le = e;
  } else {
    const int m = w.tier_map[e];
    kind = (m >> 24) == kTierNF3 ? kKindNF3 : kKindNVFP4;
    le = m & 0xFFFFFF;
  }
}

// Eight consecutive weights [k, k+8) of one row, dequantised to fp32 (exact for MXFP4/NVFP4;
// NF3 gives bf16(LUT * scale) as the NF3 unpack of hybrid_loader.py does).
//   FC2 selects the fc2 matrices; `row` is the matrix row (fc1: half * I + i, fc2: c).
template <bool FC2>
__device__ __forceinline__ void load_w8(const DevWeights& w, int kind, int le, int row, int k,
                                        float* out) {
  const int K = FC2 ? w.Ip : w.H;
  const int R = FC2 ? w.H : 2 * w.I;
  // W4A16 tiles: matrix and row within it, tiles per matrix
  const int half = FC2 ? 0 : row / w.I;
  const size_t mat = FC2 ? (size_t)le : (size_t)le * 2 + half;
  const int mr = FC2 ? row : row - half * w.I;
  const int rbs = cdiv(FC2 ? w.H : w.I, 128), kts = cdiv(K, 256);
  if (kind == kKindNF3) {
    const uint8_t* codes = FC2 ? w.nf_w2 : w.nf_w13;
    const uint32_t lo = *reinterpret_cast<const uint16_t*>(codes + nf_lo_byte(mat, mr, k, rbs, kts));
    const uint32_t hi = codes[nf_hi_byte(mat, mr, k, rbs, kts)];
    const float sc = e4m3_to_f32((FC2 ? w.nf_s2 : w.nf_s13)[nf_scale_byte(mat, mr, k, rbs, kts)]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t c = ((lo >> (2 * i)) & 3u) | (((hi >> i) & 1u) << 2);
      out[i] = __bfloat162float(__float2bfloat16_rn(c_nf3_lut[c] * sc));
    }
    return;
  }
  size_t cbyte;
  if (kind == kKindNVFP4) {
    cbyte = nv_code_byte(mat, mr, k, rbs, kts);
  } else if (w.fp4_tiled) {
    if (FC2) {
      if (k >= w.I) {          // the zero padding of K (not stored where tails are paired)
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = 0.f;
        return;
      }
      cbyte = fp4_w2_byte((size_t)w.E4, w.H, K, w.I, (size_t)le, row, k);
    } else {
      const int half = row / w.I;
      cbyte = fp4_tiled_byte((size_t)w.E4 * 2, w.I, K, (size_t)le * 2 + half, row - half * w.I, k);
    }
  } else {
    cbyte = ((size_t)le * R + row) * (size_t)(K / 2) + k / 2;
  }
  const uint32_t codes = *reinterpret_cast<const uint32_t*>((FC2 ? w.w2 : w.w13) + cbyte);
  float sc;
  if (kind == kKindMXFP4) {
    size_t byte;
    if (FC2) {
      byte = sf_atom_byte(w.H / 128, w.Ip / 128, (size_t)le, row, k / 32);
    } else {
      const int half = row / w.I, i = row - half * w.I;
      byte = sf_atom_byte(cdiv(w.I, 128), w.H / 128, (size_t)le * 2 + half, i, k / 32);
    }
    sc = e8m0_to_f32((FC2 ? w.s2 : w.s13)[byte]);
  } else if (w.mx_kept) {
    // MXFP4 kept tier of the 16-bit path: the group's prepared f16 multiplier
    sc = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(
        (FC2 ? w.s2 : w.s13) + mx16_scale_off(mat, mr, k, rbs, kts))));
  } else {
    sc = e4m3_to_f32((FC2 ? w.s2 : w.s13)[nv_scale_byte(mat, mr, k, rbs, kts)]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = e2m1_to_f32((codes >> (4 * i)) & 0xFu) * sc;
}

// Eight activations of slot position p at [k, k+8) as bf16 (exact for every operand the path
// produces: MXFP8 values have 4 significant bits).
template <bool FC2>
__device__ __forceinline__ uint4 load_a8(const SimtArgs& a, int p, int k) {
  const bool a8 = a.quant == kQuantW4A8;
  if (!FC2) {
    if (!a8) {
      const int f = a.r.perm[p], t = f / a.topk;
      const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.x) +
                                                      (size_t)t * a.H + k);
      if (a.win == nullptr) return u;
      const float wb = __bfloat162float(__float2bfloat16_rn(a.win[f]));
      const uint32_t in[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v0 = __uint_as_float(in[i] << 16) * wb;
        const float v1 = __uint_as_float(in[i] & 0xFFFF0000u) * wb;
        o[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v0)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v1)) << 16);
      }
      return make_uint4(o[0], o[1], o[2], o[3]);
    }
    // quantised activations are stored in slot order
    const uint2 q = *reinterpret_cast<const uint2*>(a.r.xq + (size_t)p * a.H + k);
    const float sc = e8m0_to_f32(a.r.xs[(size_t)p * (a.H / 32) + k / 32]);
    uint32_t qq[2] = {q.x, q.y};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t b = qq[i / 2] >> ((i & 1) * 16);
      const float v0 = e4m3_to_f32((uint8_t)(b & 0xFF)) * sc;
      const float v1 = e4m3_to_f32((uint8_t)((b >> 8) & 0xFF)) * sc;
      o[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v0)) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v1)) << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (!a8) return *reinterpret_cast<const uint4*>(a.r.h16 + (size_t)p * a.Ip + k);
  const uint2 q = *reinterpret_cast<const uint2*>(a.r.hq + (size_t)p * a.Ip + k);
  const float sc = e8m0_to_f32(a.r.hs[(size_t)p * (a.Ip / 32) + k / 32]);
  uint32_t qq[2] = {q.x, q.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t b = qq[i / 2] >> ((i & 1) * 16);
    const float v0 = e4m3_to_f32((uint8_t)(b & 0xFF)) * sc;
    const float v1 = e4m3_to_f32((uint8_t)((b >> 8) & 0xFF)) * sc;
    o[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v0)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v1)) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One CTA: one tile (<= 8 slot positions of one expert) x 32 weight rows, all of K.
// Lane l of a warp covers K offsets {l*8 + 256 g : g < 4} of each 1024-wide chunk, so weight
// loads are coalesced across lanes and activation reads are conflict-free 16-byte smem loads.
template <bool FC2>
__global__ void __launch_bounds__(kSimtThreads)
gemm_simt_kernel(SimtArgs a) {
  pdl_wait_prev();     // previous kernel of the call complete, its writes visible
  pdl_launch_next();
  const int tile = blockIdx.x;
  if (tile >= a.r.ctrl[1]) return;
  const int4 td = a.r.tiles[tile];
  const int e = td.x, p0 = td.y, n = td.z;
  int kind, le;
  resolve_expert(a.w, e, kind, le);
  const int K = FC2 ? a.Ip : a.H;
  const int R = FC2 ? a.H : 2 * a.I;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row0 = blockIdx.y * kSimtRowsPerCta + warp * 4;

  __shared__ __align__(16) __nv_bfloat16 s_act[kSimtSlots][kSimtKChunk];
  float acc[4][kSimtSlots];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int s = 0; s < kSimtSlots; ++s) acc[i][s] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kSimtKChunk) {
    __syncthreads();
    for (int gi = tid; gi < kSimtSlots * (kSimtKChunk / 8); gi += kSimtThreads) {
      const int s = gi / (kSimtKChunk / 8);
      const int kk = (gi % (kSimtKChunk / 8)) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (s < n && k0 + kk < K) v = load_a8<FC2>(a, p0 + s, k0 + kk);
      *reinterpret_cast<uint4*>(&s_act[s][kk]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = row0 + i;
      if (row >= R) break;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int kk = g * 256 + lane * 8;
        if (k0 + kk >= K) break;
        float wv[8];
        load_w8<FC2>(a.w, kind, le, row, k0 + kk, wv);
#pragma unroll
        for (int s = 0; s < kSimtSlots; ++s) {
          const uint4 av = *reinterpret_cast<const uint4*>(&s_act[s][kk]);
          const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
          float sum = acc[i][s];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            sum = fmaf(wv[2 * q], __uint_as_float(aw[q] << 16), sum);
            sum = fmaf(wv[2 * q + 1], __uint_as_float(aw[q] & 0xFFFF0000u), sum);
          }
          acc[i][s] = sum;
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int s = 0; s < kSimtSlots; ++s) {
      float v = acc[i][s];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[i][s] = v;
    }

  // lane (i*8 + s) writes element (row0 + i, slot s)
  const int i = lane >> 3, s = lane & 7;
  float v = 0.f;
#pragma unroll
  for (int ii = 0; ii < 4; ++ii)
#pragma unroll
    for (int ss = 0; ss < kSimtSlots; ++ss)
      if (ii == i && ss == s) v = acc[ii][ss];
  const int row = row0 + i;
  if (s >= n || row >= R) return;
  const int p = p0 + s;
  if (!FC2) {
    if (kind == kKindNVFP4 && a.w.g13 != nullptr) v *= a.w.g13[le];
    a.r.g[(size_t)p * (2 * a.I) + row] = v;
  } else {
    if (kind == kKindNVFP4 && a.w.g2 != nullptr) v *= a.w.g2[le];
    const int f = a.r.perm[p];
    const float wt = a.topk_w != nullptr ? a.topk_w[f] : 1.f;
    if (a.deterministic) {
      a.r.rbuf[(size_t)f * a.H + row] = wt * v;
    } else {
      atomicAdd(&a.r.acc[(size_t)(f / a.topk) * a.H + row], wt * v);
    }
  }
}

// SwiGLU + requantisation of the fc1 output: one thread per block of 32 intermediate columns.
__global__ void __launch_bounds__(256)
act_kernel(const float* __restrict__ g, const int32_t* __restrict__ ctrl, int I, int Ip,
           float limit, float alpha, float beta, int a8, uint8_t* __restrict__ hq,
           uint8_t* __restrict__ hs, __nv_bfloat16* __restrict__ h16) {
  pdl_wait_prev();     // previous kernel of the call complete, its writes visible
  pdl_launch_next();
  const int S = ctrl[2];
  const int nb = Ip / 32;
  const size_t total = (size_t)S * nb;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int p = (int)(idx / nb), b = (int)(idx % nb);
    float h[32];
    if (b * 32 >= I) {
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = 0.f;
    } else {
      const float* up = g + (size_t)p * 2 * I + b * 32;
      const float* gate = up + I;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float gg = fminf(gate[i], limit);
        const float uu = fminf(fmaxf(up[i], -limit), limit);
        h[i] = gg / (1.0f + expf(-alpha * gg)) * (uu + beta);
      }
    }
    if (a8) {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
      const uint32_t s = mx_scale_byte(amax);
      const float inv = e8m0_inv_f32(s);
      uint32_t packed[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        packed[i] = f32_to_e4m3(h[4 * i] * inv) | (f32_to_e4m3(h[4 * i + 1] * inv) << 8) |
                    (f32_to_e4m3(h[4 * i + 2] * inv) << 16) |
                    (f32_to_e4m3(h[4 * i + 3] * inv) << 24);
      uint4* dst = reinterpret_cast<uint4*>(hq + (size_t)p * Ip + b * 32);
      dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      hs[(size_t)p * nb + b] = (uint8_t)s;
    } else {
      __nv_bfloat16* dst = h16 + (size_t)p * Ip + b * 32;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[i] = __float2bfloat16_rn(h[i]);
    }
  }
}

// out[t, c] from the combine buffers: fp32 sum (atomic mode) or the fixed-order sum over the
// valid slots j = 0..k-1 of the route buffer (deterministic mode).  Eight columns per thread.
__global__ void __launch_bounds__(256)
finalize_kernel(int M, int H, int topk, int deterministic, const float* __restrict__ acc,
                const float* __restrict__ rbuf, const int32_t* __restrict__ slot_of,
                __nv_bfloat16* __restrict__ out) {
  pdl_wait_prev();     // previous kernel of the call complete, its writes visible
  pdl_launch_next();
  const size_t total = (size_t)M * (H / 8);
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(idx / (H / 8));
    const int c = (int)(idx % (H / 8)) * 8;
    float v[8];
    if (!deterministic) {
      const float4* a4 = reinterpret_cast<const float4*>(acc + (size_t)t * H + c);
      const float4 x0 = a4[0], x1 = a4[1];
      v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
      v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
      // slots in groups of 8: their indices, then their rows, all loads of a group in flight
      // together, added in slot order (the same sum on every run)
      for (int j0 = 0; j0 < topk; j0 += 8) {
        int so[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) so[j] = j0 + j < topk ? slot_of[t * topk + j0 + j] : -1;
        float4 r[8][2];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (so[j] >= 0) {
            const float4* r4 =
                reinterpret_cast<const float4*>(rbuf + (size_t)(t * topk + j0 + j) * H + c);
            r[j][0] = r4[0];
            r[j][1] = r4[1];
          } else {
            r[j][0] = r[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (so[j] < 0) continue;
          v[0] += r[j][0].x; v[1] += r[j][0].y; v[2] += r[j][0].z; v[3] += r[j][0].w;
          v[4] += r[j][1].x; v[5] += r[j][1].y; v[6] += r[j][1].z; v[7] += r[j][1].w;
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * q])) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * q + 1])) << 16);
    *reinterpret_cast<uint4*>(out + (size_t)t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Host-side launchers --------------------------------------------------------------------------

static cudaError_t launch_simt_fc(bool fc2, const SimtArgs& a, int max_tiles, cudaStream_t st) {
  const int R = fc2 ? a.H : 2 * a.I;
  dim3 grid(max_tiles, cdiv(R, kSimtRowsPerCta));
  static const bool carveout = prefer_max_shared(gemm_simt_kernel<true>) &&
                                prefer_max_shared(gemm_simt_kernel<false>);
  (void)carveout;
  return fc2 ? launch_kernel(gemm_simt_kernel<true>, grid, dim3(kSimtThreads), 0, st, true, a)
             : launch_kernel(gemm_simt_kernel<false>, grid, dim3(kSimtThreads), 0, st, true, a);
}

static cudaError_t launch_act(const RunPtrs& r, int Sm, int I, int Ip, float limit, float alpha,
                       float beta, int a8, cudaStream_t st) {
  const size_t total = (size_t)Sm * (Ip / 32);
  int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 16);
  if (blocks < 1) blocks = 1;
  static const bool carveout = prefer_max_shared(act_kernel);
  (void)carveout;
  return launch_kernel(act_kernel, dim3(blocks), dim3(256), 0, st, true,
                       static_cast<const float*>(r.g), static_cast<const int32_t*>(r.ctrl), I, Ip,
                       limit, alpha, beta, a8, r.hq, r.hs, r.h16);
}

static cudaError_t launch_finalize(int M, int H, int topk, int det, const RunPtrs& r, void* out,
                            cudaStream_t st) {
  const size_t total = (size_t)M * (H / 8);
  int blocks = (int)std::min<size_t>((total + 255) / 256, 152 * 16);
  if (blocks < 1) blocks = 1;
  static const bool carveout = prefer_max_shared(finalize_kernel);
  (void)carveout;
  return launch_kernel(finalize_kernel, dim3(blocks), dim3(256), 0, st, true, M, H, topk, det,
                       static_cast<const float*>(r.acc), static_cast<const float*>(r.rbuf),
                       static_cast<const int32_t*>(r.slot_of),
                       reinterpret_cast<__nv_bfloat16*>(out));
}

// stage 0: fc1, 1: SwiGLU + requant, 2: fc2 + combine, 3: finalize
cudaError_t launch_simt_stage(int stage, const DevWeights& w, const RunPtrs& r,
                              const PlanDims& d, int max_tiles, const void* x,
                              const float* topk_w, void* out, int M, cudaStream_t st) {
  SimtArgs a;
  a.w = w;
  a.r = r;
  a.x = x;
  // router weights on the input (16-bit activations only): fc1 reads bf16(x * bf16(w)), the
  // combine adds the expert outputs unweighted
  a.topk_w = d.w_on_input ? nullptr : topk_w;
  a.win = d.w_on_input ? topk_w : nullptr;
  a.M = M; a.topk = d.topk; a.H = d.H; a.I = d.I; a.Ip = d.Ip; a.E = d.E;
  a.quant = d.quant; a.deterministic = d.deterministic;
  const int Sm = M * d.topk;
  const int tiles = std::min(max_tiles, std::min(Sm, cdiv(Sm, kSimtSlots) + std::min(d.E, Sm)));
  switch (stage) {
    case 0: return launch_simt_fc(false, a, tiles, st);
    case 1:
      return launch_act(r, Sm, d.I, d.Ip, d.limit, d.alpha, d.beta,
                        d.quant == kQuantW4A8 ? 1 : 0, st);
    case 2: return launch_simt_fc(true, a, tiles, st);
    default: return launch_finalize(M, d.H, d.topk, d.deterministic, r, out, st);
  }
}

}  // namespace moe
