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

// Row-wise copy with a per-row source mapping and zero padding of the row tail.
//   dst [mats][rows][dst_cols] <- src [mats][rows][src_cols]; fc1 mats interleave halves.
__global__ void repack_rows_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                   int E, int halves, int rows, int src_cols, int dst_cols,
                                   int layout, int canon_fp4) {
  const size_t n = (size_t)E * halves * rows * dst_cols;
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
      v = src[(e * (size_t)(halves * rows) + sr) * src_cols + c];
      if (canon_fp4) v = canon_fp4_byte(v);
    }
    dst[idx] = v;
  }
}

// Packed FP4 rows -> the tile-contiguous layout (fp4_tiled_byte), zero padding of the row tail
// (src_cols .. dst_cols) and -0 -> +0.  src [E][halves*rows][src_cols], dst for
// mats = E*halves matrices of rows x (2*dst_cols) elements.
__global__ void repack_fp4_tiled_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                        int E, int halves, int rows, int src_cols, int dst_cols,
                                        int layout) {
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
    dst[fp4_tiled_byte(n_mats, rows, 2 * dst_cols, mh, i, 2 * c)] = v;
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

// NF3: 3-byte groups of 8 codes -> per-row 2-bit plane + 1-bit plane (row tails padded with
// code 0 in both planes; their scale is 0, so the padded weights are exactly 0).
//   src [E][halves*rows][3*src_k/8], dst [E][halves][rows][3*dst_k/8]
__global__ void repack_nf3_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                  int E, int halves, int rows, int src_k, int dst_k, int layout) {
  const int groups = dst_k / 8;
  const size_t n = (size_t)E * halves * rows * groups;
  GRID_STRIDE(idx, n) {
    const int gi = (int)(idx % groups);
    const size_t rowid = idx / groups;
    const int i = (int)(rowid % rows);
    const size_t mh = rowid / rows;
    const int half = (int)(mh % halves);
    const size_t e = mh / halves;
    uint32_t w24 = 0;
    if (gi < src_k / 8) {
      const int sr = halves == 2 ? src_row_fc1(half, i, rows, layout) : i;
      const uint8_t* s = src + (e * (size_t)(halves * rows) + sr) * (size_t)(3 * src_k / 8) + 3 * gi;
      w24 = (uint32_t)s[0] | ((uint32_t)s[1] << 8) | ((uint32_t)s[2] << 16);
    }
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t code = (w24 >> (3 * c)) & 7u;
      lo |= (code & 3u) << (2 * c);
      hi |= (code >> 2) << c;
    }
    uint8_t* d = dst + rowid * (size_t)(3 * dst_k / 8);
    d[2 * gi] = (uint8_t)(lo & 0xFF);
    d[2 * gi + 1] = (uint8_t)(lo >> 8);
    d[dst_k / 4 + gi] = (uint8_t)hi;
  }
}

// NF3 E4M3 scales [E][halves*rows][src_k/32] -> [E][halves][rows][ceil(dst_k/256)][16]
__global__ void repack_nf3_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                         int E, int halves, int rows, int src_k, int dst_k,
                                         int layout) {
  const int kt = (dst_k + 255) / 256;
  const size_t n = (size_t)E * halves * rows * kt * 16;
  GRID_STRIDE(idx, n) {
    const int b = (int)(idx % (kt * 16));
    const size_t rowid = idx / (kt * 16);
    const int i = (int)(rowid % rows);
    const size_t mh = rowid / rows;
    const int half = (int)(mh % halves);
    const size_t e = mh / halves;
    const int g = (b >> 4) * 8 + (b & 15);       // K group of 32 elements
    uint8_t v = 0;
    if ((b & 15) < 8 && g < src_k / 32) {
      const int sr = halves == 2 ? src_row_fc1(half, i, rows, layout) : i;
      v = src[(e * (size_t)(halves * rows) + sr) * (src_k / 32) + g];
    }
    dst[idx] = v;
  }
}

static int grid_for(size_t n) {
  size_t b = (n + 255) / 256;
  if (b > 152 * 32) b = 152 * 32;
  return b < 1 ? 1 : (int)b;
}

cudaError_t launch_repack_rows(const void* src, void* dst, int E, int halves, int rows,
                               int src_cols, int dst_cols, int layout, int canon, cudaStream_t st) {
  const size_t n = (size_t)E * halves * rows * dst_cols;
  if (n == 0) return cudaSuccess;
  repack_rows_kernel<<<grid_for(n), 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, E, halves,
                                                  rows, src_cols, dst_cols, layout, canon);
  return cudaGetLastError();
}

cudaError_t launch_repack_fp4_tiled(const void* src, void* dst, int E, int halves, int rows,
                                    int src_cols, int dst_cols, int layout, cudaStream_t st) {
  const size_t n = (size_t)E * halves * rows * dst_cols;
  if (n == 0) return cudaSuccess;
  repack_fp4_tiled_kernel<<<grid_for(n), 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, E,
                                                       halves, rows, src_cols, dst_cols, layout);
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

cudaError_t launch_repack_nf3(const void* src, void* dst, int E, int halves, int rows, int src_k,
                              int dst_k, int layout, cudaStream_t st) {
  const size_t n = (size_t)E * halves * rows * (dst_k / 8);
  if (n == 0) return cudaSuccess;
  repack_nf3_kernel<<<grid_for(n), 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, E, halves,
                                                 rows, src_k, dst_k, layout);
  return cudaGetLastError();
}

cudaError_t launch_repack_nf3_scales(const void* src, void* dst, int E, int halves, int rows,
                                     int src_k, int dst_k, int layout, cudaStream_t st) {
  const size_t n = (size_t)E * halves * rows * ((dst_k + 255) / 256) * 16;
  if (n == 0) return cudaSuccess;
  repack_nf3_scales_kernel<<<grid_for(n), 256, 0, st>>>((const uint8_t*)src, (uint8_t*)dst, E,
                                                        halves, rows, src_k, dst_k, layout);
  return cudaGetLastError();
}

}  // namespace moe
