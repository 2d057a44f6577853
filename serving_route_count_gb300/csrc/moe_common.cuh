// moe_common.cuh - device layouts, scratch layout and small device helpers shared by the
// kernels of the GB300 routed-MoE library.  Host and device code include it.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>
#include <stdint.h>
#include <stddef.h>

namespace moe {

constexpr int kQuantW4A8 = 0;
constexpr int kQuantNVFP4 = 1;
constexpr int kQuantHybrid = 2;
constexpr int kQuantHybridMx = 3;   // hybrid with the kept tier in MXFP4
constexpr int kQuantW4A8Nv = 4;     // NVFP4 weights, MXFP8 activations
constexpr int kTierNVFP4 = 4;
constexpr int kTierNF3 = 3;

// Error word bits written by device-side checks (never a trap).
constexpr int kErrRouteBounds = 1;   // a routing index fell outside its table
constexpr int kErrTimeout = 2;       // a bounded wait gave up
constexpr int kErrTileOverflow = 4;  // more GEMM tiles than the plan reserved
constexpr int kErrRange = 8;         // a bf16 value outside the f16 range of the W4A16 MMA

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// ----------------------------------------------------------------------------------------------
// Prepared (device) weight layout.
//
// fc1 rows are stored as two halves [half 0 = up][half 1 = gate] whatever the checkpoint order,
// each half I rows of H (K) elements.  fc2 rows are H rows of Ip = round_up(I, 128) elements
// (zero codes beyond I), because the packed-FP4 TMA format needs a row length that is a
// multiple of 128 elements.
//
// FP4 codes: element 2j in the low nibble of byte j (checkpoint order).  MXFP4: tile-contiguous (fp4_tiled_byte): every 128-row x 128-K block is one 8 KB run
//   ([mats][rows/128][K/128][128][64 B]), the partial last row block of rows % 128 rows follows
//   all full blocks ([mats][K/128][rows % 128][64 B]), so each TMA box streams contiguous bytes.
// MXFP4 E8M0 scales ("SF atoms"): for each 128-row tile and each 128-wide K tile, 512 bytes
//   byte(r, kb) = (r % 32) * 16 + (r / 32) * 4 + kb     (r < 128 in the tile, kb < 4 blocks of 32)
//   atoms ordered [expert][half][row tile][k tile]  (fc1)  /  [expert][row tile][k tile]  (fc2).
// W4A16 tiers (NVFP4, NF3): tile-contiguous too, in tiles of 128 rows x 256 K of one matrix
//   ([mats][ceil(rows/128)][ceil(K/256)] tiles; rows and K beyond the matrix are zero), so that
//   a pipeline stage of a matrix is one bulk copy of codes and one of scales:
//   NVFP4 codes: 16 KB per tile, row r at r*128, its 16-byte chunk j (elements 32j..32j+31) at
//     chunk j ^ (r % 8) - the 128-byte swizzle the expanding warps read;
//   NVFP4 scales: 2 KB per tile, row r at r*16 (the E4M3 scales of its 16 groups of 16);
//   NF3 codes: 12 KB per tile, [3][128][32 B]: the row's 2-bit plane bytes 0..31 and 32..63 of
//     the tile (code c's low two bits at bits 2*(c%4) of byte c/4), then its 1-bit plane bytes
//     0..31 (bit 2 of code c at bit c%8 of byte c/8);
//   NF3 scales: 2 KB per tile, row r at r*16: the E4M3 scales of its 8 groups of 32, 8 zero.
//   MXFP4 kept tier of the 16-bit path: codes as NVFP4; scales 2 KB per tile, row r at r*16:
//     the f16 multipliers 2^(b - b_max + 13) of its 8 groups of 32 (b the UE8M0 byte, b_max
//     the largest of the expert's matrix, kept per expert with the fp32 factor 2^(b_max - 140)
//     in place of the NVFP4 global scale).
// ----------------------------------------------------------------------------------------------
struct DevWeights {
  int quant = 0;
  int E = 0, H = 0, I = 0, Ip = 0;
  int E4 = 0, E3 = 0;                 // experts in the fp4 tier / the NF3 tier
  int fp4_tiled = 0;                  // MXFP4 codes in the tile-contiguous layout
  // fp4 tier (MXFP4 or NVFP4)
  const uint8_t* w13 = nullptr;       // [E4][2][I][H/2] codes (tiled, see above)
  const uint8_t* s13 = nullptr;       // MXFP4 atoms / NVFP4 scale tiles
  const uint8_t* w2 = nullptr;        // [E4][H][Ip/2]
  const uint8_t* s2 = nullptr;        // MXFP4 atoms / NVFP4 [E4][H][Ip/16]
  const float* g13 = nullptr;         // [E4] NVFP4 global scales (MXFP4 kept tier: 2^shift)
  const float* g2 = nullptr;
  int mx_kept = 0;                    // kept tier MXFP4: scale tiles hold f16 multipliers
  const float* ag13 = nullptr;        // NVFP4 weights with MXFP8 activations: per-expert
  const float* ag2 = nullptr;         // activation global scales of fc1's / fc2's input ([E])
  // NF3 tier
  const uint8_t* nf_w13 = nullptr;    // NF3 code tiles of [E3][2] matrices I x H
  const uint8_t* nf_s13 = nullptr;    // NF3 scale tiles
  const uint8_t* nf_w2 = nullptr;     // [E3][H][3Ip/8] planes
  const uint8_t* nf_s2 = nullptr;     // NF3 scale tiles of [E3] matrices H x Ip
  const int32_t* tier_map = nullptr;  // [E]: (tier << 24) | local index
};

__host__ __device__ inline size_t fp4_tiled_byte(size_t n_mats, int rows, int K, size_t mat,
                                                 int r, int k) {
  const int rtf = rows >> 7, rem = rows & 127, kt_n = K >> 7;
  const int rt = r >> 7, rr = r & 127, kt = k >> 7, kb = (k & 127) >> 1;
  if (rt < rtf) return ((((mat * rtf + rt) * kt_n + kt) << 7) + rr) * 64 + kb;
  return n_mats * rtf * kt_n * 8192 + (((mat * kt_n + kt) * rem) + rr) * 64 + kb;
}

// fc2 codes of a W4A8 layer whose I % 128 == 64: the last K tile of a 128-row block holds 64
// columns, so the tails of row blocks 2j and 2j + 1 share the tile of block 2j (columns 0..63
// and 64..127; the tile of block 2j + 1 is unused).  fc2 reads the shared tile once from HBM for
// both blocks instead of two tiles half of zero codes.  Byte of elements k, k + 1 (k even) of
// row r of expert e's w2 (H rows, Kp = I rounded up to 128).
__host__ __device__ inline size_t fp4_w2_byte(size_t E, int H, int Kp, int I, size_t e, int r,
                                              int k) {
  const int kf = I & ~127;
  if ((I & 127) == 64 && k >= kf) {
    const int rb = r >> 7;
    return fp4_tiled_byte(E, H, Kp, e, ((rb & ~1) << 7) + (r & 127), k + 64 * (rb & 1));
  }
  return fp4_tiled_byte(E, H, Kp, e, r, k);
}
// Its code tile of row block rb, K tile kt ([E][H/128][Kp/128] tiles of 8 KB).
__host__ __device__ inline int fp4_w2_tile(int e, int rb, int kt, int RB, int KT, int pair) {
  return (e * RB + ((pair && kt == KT - 1) ? (rb & ~1) : rb)) * KT + kt;
}

// W4A16 tiles (see above): tile of matrix `mat`, row block rb, K tile kt.
__host__ __device__ inline size_t w16_tile(size_t mat, int rb, int kt, int rbs, int kts) {
  return (mat * (size_t)rbs + rb) * (size_t)kts + kt;
}
constexpr int kNvCodeTile = 16384, kNfCodeTile = 12288, kW16ScaleTile = 2048;
// NVFP4 code byte of elements k, k+1 (k even) of row r of matrix mat (rbs x kts tiles)
__host__ __device__ inline size_t nv_code_byte(size_t mat, int r, int k, int rbs, int kts) {
  const int rr = r & 127, kk = k & 255;
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kNvCodeTile + (size_t)rr * 128 +
         ((((kk >> 5) ^ (rr & 7))) << 4) + ((kk & 31) >> 1);
}
// NVFP4 scale byte of element k of row r
__host__ __device__ inline size_t nv_scale_byte(size_t mat, int r, int k, int rbs, int kts) {
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kW16ScaleTile + (size_t)(r & 127) * 16 +
         ((k & 255) >> 4);
}
// MXFP4 kept tier: byte offset of the f16 multiplier of element k of row r
__host__ __device__ inline size_t mx16_scale_off(size_t mat, int r, int k, int rbs, int kts) {
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kW16ScaleTile + (size_t)(r & 127) * 16 +
         ((k & 255) >> 5) * 2;
}
// NF3 2-bit plane byte of codes k..k+3 (k % 4 == 0) and 1-bit plane byte of codes k..k+7
// (k % 8 == 0) of row r
__host__ __device__ inline size_t nf_lo_byte(size_t mat, int r, int k, int rbs, int kts) {
  const int kk = k & 255;
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kNfCodeTile + (size_t)(kk >> 7) * 4096 +
         (size_t)(r & 127) * 32 + ((kk >> 2) & 31);
}
__host__ __device__ inline size_t nf_hi_byte(size_t mat, int r, int k, int rbs, int kts) {
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kNfCodeTile + 8192 + (size_t)(r & 127) * 32 +
         ((k & 255) >> 3);
}
// NF3 scale byte of element k of row r
__host__ __device__ inline size_t nf_scale_byte(size_t mat, int r, int k, int rbs, int kts) {
  return w16_tile(mat, r >> 7, k >> 8, rbs, kts) * kW16ScaleTile + (size_t)(r & 127) * 16 +
         ((k & 255) >> 5);
}

__host__ __device__ inline size_t sf_atom_byte(int row_tiles, int k_tiles, size_t mat, int r,
                                               int kb) {
  // mat = expert * halves + half (fc1) or expert (fc2)
  int rt = r >> 7, rr = r & 127, kt = kb >> 2, kk = kb & 3;
  size_t atom = (mat * (size_t)row_tiles + rt) * (size_t)k_tiles + kt;
  return atom * 512 + (size_t)((rr & 31) * 16 + (rr >> 5) * 4 + kk);
}

// ----------------------------------------------------------------------------------------------
// Scratch layout of one plan (byte offsets into the caller's scratch buffer).
// ----------------------------------------------------------------------------------------------
constexpr int kSimtSlots = 8;       // slots per tile of the CUDA-core GEMMs

struct Scratch {
  size_t ctrl;      // int32[64]: [0] error word, [1] n_tiles, [2] n_valid_slots
  size_t cnt;       // int32[E]
  size_t off;       // int32[E+1]
  size_t perm;      // int32[Sm]
  size_t slot_of;   // int32[Sm]
  size_t tiles;     // int4[max_tiles] {expert, first position, count, 0}
  size_t xq, xs;    // W4A8: u8 [Sm][H], u8 [Sm][H/32], one row per slot position
  // W4A8 calls with 16/32-token tiles: the E8M0 scales of x and of h again, laid out as the
  // tensor cores' scale atoms want them - per 128-wide K tile, one 16-byte row per slot position
  // (bytes 0..3 = the position's four scales of that K tile) - so a tile's atom is one bulk copy
  size_t xs16, hs16;  // u8 [H/128][r16][16], u8 [Ip/128][r16][16]
  int r16;            // rows per K tile: the positions of a 64-token call + 32 of padding
  size_t g;         // fp32 fc1 output [Sm][2][Ip] (CUDA-core path) / split-K partial sums
                    // [splits][Sm][2][Ip] (tensor-core paths)
  size_t tickets;   // int32 [max_tiles][ceil(I/128)] fc1 completion tickets
  size_t part;      // W4A8: fp32 partial sums of the stream-K fc1 (fixed-size slots)
  size_t rcc;       // W4A8: int32 [ceil(Sm / 1024)][E] chunked-routing counts + 1 ticket
  size_t hq, hs;    // W4A8: u8 [Sm][Ip], u8 [Sm][Ip/32]
  size_t h16;       // W4A16: bf16 [Sm][Ip] (CUDA-core path) or f16 (tensor-core path)
  size_t x16;       // W4A16 tensor-core path: f16 activations [Sm][H] in slot order
  size_t acc;       // fp32 [max_m][H]  (atomic combine)
  size_t rbuf;      // fp32 [max_m*topk][H]  (deterministic combine: one row per slot)
  size_t total;
  int max_tiles;
};

struct PlanDims {
  int E, H, I, Ip, topk, max_m, quant, deterministic;
  float limit, alpha, beta;
  int backend;      // 0: tensor cores where implemented, 1: CUDA-core path
  int fc1_kernel;   // W4A8 fc1 at 16-token tiles: 0 automatic, 1 unit per CTA, 2 stream-K
  int w_on_input;   // 16-bit paths: router weights scale fc1's input, the combine is unweighted
  int ep_first;     // global id of local expert 0; router ids outside [ep_first, ep_first + E)
                    // belong to other ranks and are dropped
  int keep_act;     // test hook: small W4A8 calls, whose fc1 quantises the activations itself,
                    // also store the codes where moe_debug_actq reads them
  unsigned long long wait_probe_ns;   // test hook (0: off): W4A8 fc1's MMA issuer first waits
                    // this long on a barrier nothing arrives on, so the wait runs out
  // A8 opt-in of the MXFP4 kept tier (hybrid MX mode): static FP8 input scales of fc1 / fc2
  // and their fp32 reciprocals
  int kept_a8;
  float a8_s13, a8_inv13, a8_s2, a8_inv2;
};

// The kept tier's A8 opt-in for an activation producer: the slots of experts whose tier-map
// entry is the kept tier (kTierNVFP4) get static per-tensor FP8 activations, E4M3 of
// fp32(x) * inv; tiers == nullptr: off.
struct KeptA8 {
  const int32_t* tiers;
  float inv;
};

// Local id of router id `id` on a plan that owns the global experts [first, first + E): id -
// first, or -1 for another rank's expert or padding.  Unsigned arithmetic, so no id overflows
// (first + E <= INT_MAX, checked when the offset is set).
__device__ __forceinline__ int local_expert(int id, int first, int E) {
  const unsigned u = static_cast<unsigned>(id) - static_cast<unsigned>(first);
  return u < static_cast<unsigned>(E) ? static_cast<int>(u) : -1;
}

// Pointers of one call, resolved from the scratch base.
struct RunPtrs {
  int32_t* ctrl;
  int32_t* cnt;
  int32_t* off;
  int32_t* perm;
  int32_t* slot_of;
  int4* tiles;
  uint8_t* xq;
  uint8_t* xs;
  uint8_t* xs16;
  uint8_t* hs16;
  int r16;
  float* g;
  int32_t* tickets;
  float* part;
  uint8_t* hq;
  uint8_t* hs;
  __nv_bfloat16* h16;
  uint16_t* x16;
  float* acc;
  float* rbuf;
  int32_t* rcc;     // chunked routing: per-chunk expert counts / bases, then a ticket
};

// ----------------------------------------------------------------------------------------------
// Device helpers
// ----------------------------------------------------------------------------------------------
// 2^(s-127) for an E8M0 byte (s = 255 is NaN by the format; never produced here).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  return s == 0 ? __int_as_float(0x00400000) : __int_as_float((int)(s << 23));
}

// 2^(127-s): the exact reciprocal of an E8M0 scale in fp32 (s in 0..254).
__device__ __forceinline__ float e8m0_inv_f32(uint32_t s) {
  return s == 254 ? __int_as_float(0x00400000) : __int_as_float((int)((254u - s) << 23));
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(__half(h));
}

// One E2M1 nibble (sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0) as fp32, times
// 2^-126: placing the three magnitude bits at fp32 bits 24..22 gives exactly that, subnormal
// case included (exponent 0 -> fp32 subnormal m * 2^-127 = m * 0.5 * 2^-126).
__device__ __forceinline__ float e2m1_scaled_down(uint32_t c) {
  return __int_as_float((int)(((c & 8u) << 28) | ((c & 7u) << 22)));
}
// E2M1 value of a nibble.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  return e2m1_scaled_down(c) * 0x1p126f;
}

// MXFP8 scale byte of a block whose largest magnitude is amax (OCP MX: floor(log2 amax) - 8,
// biased, clamped to the finite E8M0 range).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  int e = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  int s = e - 8;
  return (uint32_t)(s < 0 ? 0 : (s > 254 ? 254 : s));
}

// fp32 -> E4M3 code (round to nearest even, saturate to +-448).
__device__ __forceinline__ uint32_t f32_to_e4m3(float a) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ void set_error(int32_t* ctrl, int bit) { atomicOr(ctrl, bit); }

// One block of 32 bf16 activations (four 16-byte words, element 2j of a word in its low half)
// -> 32 E4M3 codes (eight words, element 4j + b in byte b of word j) and the E8M0 scale byte
// (OCP MX rule: scale = 2^(floor(log2 amax) - 8); codes round to nearest even and saturate).
__device__ __forceinline__ uint32_t mxfp8_block32(const uint4* u, uint32_t* packed) {
  float v[32];
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    const uint32_t w[4] = {u[qq].x, u[qq].y, u[qq].z, u[qq].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[qq * 8 + 2 * j] = __uint_as_float(w[j] << 16);
      v[qq * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const uint32_t s = mx_scale_byte(amax);
  const float inv = e8m0_inv_f32(s);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    packed[j] = f32_to_e4m3(v[4 * j] * inv) | (f32_to_e4m3(v[4 * j + 1] * inv) << 8) |
                (f32_to_e4m3(v[4 * j + 2] * inv) << 16) | (f32_to_e4m3(v[4 * j + 3] * inv) << 24);
  }
  return s;
}

// ----------------------------------------------------------------------------------------------
// Chained launches (programmatic dependent launch)
// ----------------------------------------------------------------------------------------------
// The kernels of one call are launched as a chain: each lets the next one launch once all of its
// own CTAs are running (pdl_launch_next), and each waits for the previous one to complete and
// its memory to be visible (pdl_wait_prev) before touching any buffer of the call.  A kernel that
// was launched without the chaining attribute returns from the wait at once.
__device__ __forceinline__ void pdl_wait_prev() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Asks for the largest shared-memory carveout for `kernel` (call once per kernel, from a
// static of its launch function).  An SM runs its CTAs under one carveout, so a kernel with
// little shared memory left at the default carveout keeps the tensor-core kernels chained after
// it off its SMs until its CTAs there end (measured: no fc1 CTA started on an SM while a
// routing CTA ran on it).
template <typename K>
inline bool prefer_max_shared(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess;
}

// Launches kernel<<<grid, block, smem, st>>>(args...); `chained` lets it start (up to its
// pdl_wait_prev) while the previous kernel of the stream is still running.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool chained, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace moe
