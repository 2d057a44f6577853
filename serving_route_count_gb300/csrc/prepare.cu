// prepare.cu - repack checkpoint-layout expert tensors into the device layout (moe_b12x_next.py
// module docstring: checkpoint bytes repacked into prepared experts at load; vLLM B12xExperts
// `_prepare_experts`, which also canonicalises FP4 zero signs, -0 -> +0).
//
// The device layout is documented in moe_common.cuh.  Every kernel here is a pure byte
// permutation (plus zero padding and the -0 -> +0 rewrite of E2M1 nibbles, a numerical no-op).
#include "moe_common.cuh"

namespace moe {

// fc1 row of half h (0 = up, 1 = gate), index i, in the checkpoint's stacking order.
__device__ __forceinline__ int src_row_fc1(int half, int i, int I, int layout) {
  // layout 0: [up; gate]; layout 1: [gate; up]
  return (layout == 0 ? half : 1 - half) * I + i;
}

__device__ __forceinline__ uint8_t canon_fp4_byte(uint8_t b) {
  uint8_t lo = b & 0xF, hi = b >> 4;
  if (lo == 0x8) lo = 0;
  if (hi == 0x8) hi = 0;
  return (uint8_t)(lo | (hi << 4));
}

#define GRID_STRIDE(i, n)                                                              \
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)(n); \
       i += (size_t)gridDim.x * blockDim.x)

// Packed FP4 rows -> the tile-contiguous layout (fp4_tiled_byte), zero padding of the row tail
// (src_cols .. dst_cols) and -0 -> +0.  src [E][halves*rows][src_cols], dst for
// mats = E*halves matrices of rows x (2*dst_cols) elements.
__global__ void repack_fp4_tiled_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                        int E, int halves, int rows, int src_cols, int dst_cols,
                                        int layout, int pair_I) {
  const size_t n = (size_t)E * halves * rows * dst_cols;
  const size_t n_mats = (size_t)E * halves;
  GRID_STRIDE(idx, n) {
    const int c = (int)(idx % dst_cols);
    const size_t rowid = idx / dst_cols;
    const int i = (int)(rowid % rows);
    const size_t mh = rowid / rows;
    const int half = (int)(mh % halves);
    const size_t e = mh / halves;
    uint8_t v = 0;
    if (c < src_cols) {
      const int sr = halves == 2 ? src_row_fc1(half, i, rows, layout) : i;
      v = canon_fp4_byte(src[(e * (size_t)(halves * rows) + sr) * src_cols + c]);
    }
    if (pair_I != 0) {
      // fc2 with paired 64-column tails: the padding columns are not stored (the partner block's
      // codes take their place)
      if (c < src_cols) dst[fp4_w2_byte(n_mats, rows, 2 * dst_cols, pair_I, mh, i, 2 * c)] = v;
    } else {
      dst[fp4_tiled_byte(n_mats, rows, 2 * dst_cols, mh, i, 2 * c)] = v;
    }
  }
}

// MXFP4 E8M0 scales -> SF atoms.  src [E][halves*rows][kblocks] (checkpoint stacking),
// dst atoms [E][halves][row_tiles][k_tiles][512]; padded rows / k-blocks get byte 0.
__global__ void repack_sf_atoms_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                       int E, int halves, int rows, int kblocks, int row_tiles,
                                       int k_tiles, int layout) {
  const size_t n = (size_t)E * halves * row_tiles * k_tiles * 512;
  GRID_STRIDE(idx, n) {
    const int b = (int)(idx & 511);
    size_t atom = idx >> 9;
    const int kt = (int)(atom % k_tiles);
    atom /= k_tiles;
    const int rt = (int)(atom % row_tiles);
    const size_t mh = atom / row_tiles;
    const int half = (int)(mh % halves);
    const size_t e = mh / halves;
    const int rr = (b >> 4) + 32 * ((b >> 2) & 3);
    const int kk = b & 3;
    const int r = rt * 128 + rr, kb = kt * 4 + kk;
    uint8_t v = 0;
    if (r < rows && kb < kblocks) {
      const int sr = halves == 2 ? src_row_fc1(half, r, rows, layout) : r;
      v = src[(e * (size_t)(halves * rows) + sr) * kblocks + kb];
    }
    dst[idx] = v;
  }
}

// W4A16 tiles (moe_common.cuh): every kernel below walks the destination bytes of
// mats = E*halves matrices of `rows` rows and K elements in tiles of 128 x 256, and reads the
// checkpoint row (fc1 halves in the checkpoint's stacking order) or writes 0 beyond it.

// NVFP4 codes (16 KB tiles, 128-byte swizzle), -0 -> +0.  src [E][halves*rows][src_k/2].
__global__ void repack_nv_codes_tiled_kernel(const uint8_t* __restrict__ src,
                                             uint8_t* __restrict__ dst, int E, int halves,
                                             int rows, int src_k, int K, int layout) {
  const int rbs = (rows + 127) / 128, kts = (K + 255) / 256;
  const size_t n = (size_t)E * halves * rbs * kts * kNvCodeTile;
  GRID_STRIDE(idx, n) {
    const int off = (int)(idx % kNvCodeTile);
    size_t t = idx / kNvCodeTile;
    const int kt = (int)(t % kts);
    t /= kts;
    const int rb = (int)(t % rbs);
    const size_t mat = t / rbs;
    const int rr = off >> 7, j = ((off >> 4) & 7) ^ (rr & 7), b = off & 15;
    const int r = rb * 128 + rr;
    const int cbyte = kt * 128 + j * 16 + b;          // packed byte within the row
    uint8_t v = 0;
    if (r < rows && 2 * cbyte < src_k) {
      const int half = (int)(mat % halves);
      const size_t e = mat / halves;
      const int sr = halves == 2 ? src_row_fc1(half, r, rows, layout) : r;
      v = canon_fp4_byte(src[(e * (size_t)(halves * rows) + sr) * (size_t)(src_k / 2) + cbyte]);
    }
    dst[idx] = v;
  }
}

// Scales of 16 bytes per row and tile: NVFP4 (`group` = 16 elements, 16 per tile) or NF3
// (`group` = 32 elements, 8 per tile, bytes 8..15 zero).  src [E][halves*rows][src_k/group].
__global__ void repack_w16_scales_tiled_kernel(const uint8_t* __restrict__ src,
                                               uint8_t* __restrict__ dst, int E, int halves,
                                               int rows, int src_k, int K, int group, int layout) {
  const int rbs = (rows + 127) / 128, kts = (K + 255) / 256;
  const int per_tile = 256 / group;
  const size_t n = (size_t)E * halves * rbs * kts * kW16ScaleTile;
  GRID_STRIDE(idx, n) {
    const int off = (int)(idx % kW16ScaleTile);
    size_t t = idx / kW16ScaleTile;
    const int kt = (int)(t % kts);
    t /= kts;
    const int rb = (int)(t % rbs);
    const size_t mat = t / rbs;
    const int rr = off >> 4, b = off & 15;
    const int r = rb * 128 + rr;
    const int g = kt * per_tile + b;
    uint8_t v = 0;
    if (b < per_tile && r < rows && g < src_k / group) {
      const int half = (int)(mat % halves);
      const size_t e = mat / halves;
      const int sr = halves == 2 ? src_row_fc1(half, r, rows, layout) : r;
      v = src[(e * (size_t)(halves * rows) + sr) * (size_t)(src_k / group) + g];
    }
    dst[idx] = v;
  }
}

// MXFP4 kept tier of the 16-bit path, step 1: per expert, the largest UE8M0 scale byte of the
// matrix (0xFF, NaN, left out) -> kmax[e], and the matrix's fp32 factor 2^(kmax - 140) -> g[e]
// (built from its bits: normal down to 2^-126, subnormal below).  One CTA per expert.
__global__ void mx_scale_max_kernel(const uint8_t* __restrict__ src, size_t per_expert,
                                    int32_t* __restrict__ kmax, float* __restrict__ g) {
  __shared__ int s_max[32];
  const size_t e = blockIdx.x;
  int m = -1;
  for (size_t i = threadIdx.x; i < per_expert; i += blockDim.x) {
    const int b = src[e * per_expert + i];
    if (b != 0xFF && b > m) m = b;
  }
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, s_max[w]);
    if (m < 0) m = 140;                       // no finite scale: factor 1
    const int x = m - 140;                    // factor exponent, -140 .. 114
    const uint32_t bits = x >= -126 ? (uint32_t)(x + 127) << 23 : 1u << (x + 149);
    kmax[e] = m;
    g[e] = __uint_as_float(bits);
  }
}

// Step 2: the scale tiles, each group's f16 multiplier 2^(b - kmax + 13): exponent j in
// [-23, 13] (normal from 2^-14, subnormal below); groups below 2^-23 flushed to 0, NaN kept.
__device__ __forceinline__ uint16_t mx_multiplier_f16(int b, int kmax) {
  if (b == 0xFF) return 0x7E00;
  const int j = b - kmax + 13;
  if (j < -23) return 0;
  return j >= -14 ? (uint16_t)((j + 15) << 10) : (uint16_t)(1u << (j + 24));
}

__global__ void repack_mx16_scales_tiled_kernel(const uint8_t* __restrict__ src,
                                                const int32_t* __restrict__ kmax,
                                                uint16_t* __restrict__ dst, int E, int halves,
                                                int rows, int src_k, int K, int layout) {
  const int rbs = (rows + 127) / 128, kts = (K + 255) / 256;
  const size_t n = (size_t)E * halves * rbs * kts * (kW16ScaleTile / 2);
  GRID_STRIDE(idx, n) {
    const int off = (int)(idx % (kW16ScaleTile / 2));
    size_t t = idx / (kW16ScaleTile / 2);
    const int kt = (int)(t % kts);
    t /= kts;
    const int rb = (int)(t % rbs);
    const size_t mat = t / rbs;
    const int rr = off >> 3, b = off & 7;
    const int r = rb * 128 + rr;
    const int grp = kt * 8 + b;
    uint16_t v = 0;
    if (r < rows && grp < src_k / 32) {
      const int half = (int)(mat % halves);
      const size_t e = mat / halves;
      const int sr = halves == 2 ? src_row_fc1(half, r, rows, layout) : r;
      v = mx_multiplier_f16(src[(e * (size_t)(halves * rows) + sr) * (size_t)(src_k / 32) + grp],
                            kmax[e]);
    }
    dst[idx] = v;
  }
}

// NVFP4 weight scales as the W4A4 kernels' tensor-memory atoms: per 128-row x 256-K tile four
// 512-byte atoms (one per K = 64 instruction), byte (r % 32) * 16 + (r / 32) * 4 + j of atom kb
// = the E4M3 scale of tile row r, group of 16 number 4 kb + j.  src [E][halves*rows][src_k/16].
__global__ void repack_nv_sf_atoms_kernel(const uint8_t* __restrict__ src,
                                          uint8_t* __restrict__ dst, int E, int halves, int rows,
                                          int src_k, int K, int layout) {
  const int rbs = (rows + 127) / 128, kts = (K + 255) / 256;
  const size_t n = (size_t)E * halves * rbs * kts * kW16ScaleTile;
  GRID_STRIDE(idx, n) {
    const int off = (int)(idx % kW16ScaleTile);
    size_t t = idx / kW16ScaleTile;
    const int kt = (int)(t % kts);
    t /= kts;
    const int rb = (int)(t % rbs);
    const size_t mat = t / rbs;
    const int kb = off >> 9, b = off & 511;
    const int rr = (b >> 4) + 32 * ((b >> 2) & 3), j = b & 3;
    const int r = rb * 128 + rr, g = kt * 16 + kb * 4 + j;
    uint8_t v = 0;
    if (r < rows && g < src_k / 16) {
      const int half = (int)(mat % halves);
      const size_t e = mat / halves;
      const int sr = halves == 2 ? src_row_fc1(half, r, rows, layout) : r;
      v = src[(e * (size_t)(halves * rows) + sr) * (size_t)(src_k / 16) + g];
    }
    dst[idx] = v;
  }
}

// NF3 code c of checkpoint row `sr` (3-byte groups of 8 codes), 0 beyond src_k.
__device__ __forceinline__ uint32_t nf3_code(const uint8_t* src, size_t row_base, int c,
                                             int src_k) {
  if (c >= src_k) return 0;
  const uint8_t* s = src + row_base + 3 * (c >> 3);
  const uint32_t w24 = (uint32_t)s[0] | ((uint32_t)s[1] << 8) | ((uint32_t)s[2] << 16);
  return (w24 >> (3 * (c & 7))) & 7u;
}

// NF3 codes -> 12 KB tiles of 2-bit and 1-bit planes.  src [E][halves*rows][3*src_k/8].
__global__ void repack_nf3_tiled_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                        int E, int halves, int rows, int src_k, int K,
                                        int layout) {
  const int rbs = (rows + 127) / 128, kts = (K + 255) / 256;
  const size_t n = (size_t)E * halves * rbs * kts * kNfCodeTile;
  GRID_STRIDE(idx, n) {
    const int off = (int)(idx % kNfCodeTile);
    size_t t = idx / kNfCodeTile;
    const int kt = (int)(t % kts);
    t /= kts;
    const int rb = (int)(t % rbs);
    const size_t mat = t / rbs;
    const int box = off >> 12, rr = (off >> 5) & 127, bb = off & 31;
    const int r = rb * 128 + rr;
    uint32_t v = 0;
    if (r < rows) {
      const int half = (int)(mat % halves);
      const size_t e = mat / halves;
      const int sr = halves == 2 ? src_row_fc1(half, r, rows, layout) : r;
      const size_t row_base = (e * (size_t)(halves * rows) + sr) * (size_t)(3 * src_k / 8);
      if (box < 2) {            // 2-bit plane byte: codes c0..c0+3, low two bits each
        const int c0 = kt * 256 + (box * 32 + bb) * 4;
        for (int i = 0; i < 4; ++i) v |= (nf3_code(src, row_base, c0 + i, src_k) & 3u) << (2 * i);
      } else {                  // 1-bit plane byte: codes c0..c0+7, bit 2 each
        const int c0 = kt * 256 + bb * 8;
        for (int i = 0; i < 8; ++i) v |= (nf3_code(src, row_base, c0 + i, src_k) >> 2) << i;
      }
    }
    dst[idx] = (uint8_t)v;
  }
}

static int grid_for(size_t n) {
  size_t b = (n + 255) / 256;
  if (b > 152 * 32) b = 152 * 32;
  return b < 1 ? 1 : (int)b;
}

cudaError_t launch_repack_fp4_tiled(const void* src, void* dst, int E, int halves, int rows,
                                    int src_cols, int dst_cols, int layout, int pair_I,
                                    cudaStream_t st) {
  const size_t n = (size_t)E * halves * rows * dst_cols;
  if (n == 0) return cudaSuccess;
  repack_fp4_tiled_kernel<<<grid_for(n), 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, E,
                                                       halves, rows, src_cols, dst_cols, layout,
                                                       pair_I);
  return cudaGetLastError();
}

cudaError_t launch_repack_sf_atoms(const void* src, void* dst, int E, int halves, int rows,
                                   int kblocks, int row_tiles, int k_tiles, int layout,
                                   cudaStream_t st) {
  const size_t n = (size_t)E * halves * row_tiles * k_tiles * 512;
  if (n == 0) return cudaSuccess;
  repack_sf_atoms_kernel<<<grid_for(n), 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, E,
                                                      halves, rows, kblocks, row_tiles, k_tiles,
                                                      layout);
  return cudaGetLastError();
}

// MXFP4 kept tier scales: src [E][halves*rows][src_k/32] UE8M0 -> per-expert kmax / factor g,
// then the f16 multiplier tiles.
cudaError_t launch_repack_mx16_scales(const void* src, void* dst, int32_t* kmax, float* g, int E,
                                      int halves, int rows, int src_k, int K, int layout,
                                      cudaStream_t st) {
  if (E == 0) return cudaSuccess;
  const uint8_t* s8 = static_cast<const uint8_t*>(src);
  mx_scale_max_kernel<<<E, 256, 0, st>>>(s8, (size_t)halves * rows * (src_k / 32), kmax, g);
  const size_t n = (size_t)E * halves * ((rows + 127) / 128) * ((K + 255) / 256) *
                   (kW16ScaleTile / 2);
  repack_mx16_scales_tiled_kernel<<<grid_for(n), 256, 0, st>>>(
      s8, kmax, static_cast<uint16_t*>(dst), E, halves, rows, src_k, K, layout);
  return cudaGetLastError();
}

cudaError_t launch_repack_w16_tiled(int kind, const void* src, void* dst, int E, int halves,
                                    int rows, int src_k, int K, int layout, cudaStream_t st) {
  const size_t tiles = (size_t)E * halves * ((rows + 127) / 128) * ((K + 255) / 256);
  if (tiles == 0) return cudaSuccess;
  const uint8_t* s8 = static_cast<const uint8_t*>(src);
  uint8_t* d8 = static_cast<uint8_t*>(dst);
  switch (kind) {
    case 0:   // NVFP4 codes
      repack_nv_codes_tiled_kernel<<<grid_for(tiles * kNvCodeTile), 256, 0, st>>>(
          s8, d8, E, halves, rows, src_k, K, layout);
      break;
    case 1:   // NVFP4 scales
      repack_w16_scales_tiled_kernel<<<grid_for(tiles * kW16ScaleTile), 256, 0, st>>>(
          s8, d8, E, halves, rows, src_k, K, 16, layout);
      break;
    case 2:   // NF3 codes
      repack_nf3_tiled_kernel<<<grid_for(tiles * kNfCodeTile), 256, 0, st>>>(
          s8, d8, E, halves, rows, src_k, K, layout);
      break;
    case 3:   // NF3 scales
      repack_w16_scales_tiled_kernel<<<grid_for(tiles * kW16ScaleTile), 256, 0, st>>>(
          s8, d8, E, halves, rows, src_k, K, 32, layout);
      break;
    case 4:   // NVFP4 scales as W4A4 tensor-memory atoms
      repack_nv_sf_atoms_kernel<<<grid_for(tiles * kW16ScaleTile), 256, 0, st>>>(
          s8, d8, E, halves, rows, src_k, K, layout);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
