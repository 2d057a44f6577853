// gemm_tc16.cu - W4A16 grouped GEMMs (NVFP4 and NF3 weights, 16-bit activations) on the
// 5th-generation tensor cores.
//
// The NVFP4 kept tier and the NF3 tier of the hybrid layer (hybrid_loader.py: NVFP4 =
// E2M1 x E4M3 scale per 16 x per-expert fp32 global; NF3 = 8-entry LUT x E4M3 scale per 32,
// `_unpack_nf3`; "v3" MXFP4 kept tier = E2M1 x 2^(b-127) per 32, prepared as an f16 multiplier
// per group and a per-matrix power-of-two factor) run with bf16 activations.  There is no block-scaled MMA kind for a 16-bit
// operand, so the weights are expanded in shared memory ahead of the MMA (tcgen05 kind::f16):
//   NVFP4: E2M1 x E4M3 has at most 6 significant bits and lies in [2^-10, 2688]: exact in f16;
//   MXFP4: E2M1 x 2^j for j in [-23, 13] (the prepared multipliers): exact in f16;
//   NF3:   bf16(fp32(LUT[c]) x fp32(scale)) (the page's unpack) is exact in f16 for E4M3 scales;
//   activations: bf16 values are exact in f16 when |x| <= 65504 (larger values set an error
//   bit; values below 2^-14 lose low bits as f16 subnormals).
// So the MMA runs on f16 A and B (both operands must have the same type) with fp32 accumulation,
// and the per-expert NVFP4 global scale is applied in the fp32 epilogue.
//
// Same orientation and work split as the W4A8 kernels (gemm_tc.cu): weight rows are the
// 128-row MMA operand, the tile's tokens the N columns.  Roles (320 threads):
//   warp 0 lane 0   bulk copies of the raw weight tiles (codes + scales, 256-wide K stages)
//                   and TMA of the activation sub-tiles (64-wide K, 128-byte swizzle);
//   warp 1 lane 0   tcgen05.mma (4 MMAs of K = 16 per sub-tile and matrix) and commits;
//   warps 2..9      converters (two threads per weight row, one half of each sub-tile each)
//                   writing f16 sub-tiles in the 128-byte swizzled K-major layout; warps 2..5
//                   then run the epilogue from TMEM.
#include <algorithm>
#include <cstring>

#include "moe_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace tc;

constexpr int k16Threads = 320;           // producer, MMA issuer, 8 converter warps
constexpr int k16RawK = 256;              // K elements per raw stage
constexpr int k16SubK = 64;               // K elements per converted f16 sub-tile (128 B rows)
constexpr int k16RawCodes = 128 * 128;    // raw codes region per matrix (NVFP4: 128 x 128 B)
constexpr int k16RawScales = 128 * 16;    // raw scales region per matrix (128 rows x 16 B)

__constant__ float c_nf3_lut16[8] = {-1.0f, -0.6047f, -0.3563f, -0.1275f,
                                     0.1275f, 0.3563f,  0.6047f,  1.0f};

// PAIR: fc1 at two CTAs per SM (short rings; token tiles of at most 32, every 16-bit weight
// format)
template <int BN, bool FC2, bool PAIR = false>
struct Tc16Cfg {
  static constexpr int kMats = FC2 ? 1 : 2;
  static constexpr int kRaw = kMats * (k16RawCodes + k16RawScales);     // per raw stage
  static constexpr int kB = BN * 128;                                   // per B slot
  // The expanded f16 weights go to tensor memory (the MMA's A operand), not shared memory:
  // shared memory holds the raw stages and the activation sub-tiles only.  fc1 (one CTA per SM
  // by its tensor memory): 4 raw stages; fc2 (K = the intermediate size, a couple of raw
  // stages): 2, so that two CTAs fit an SM.
  static constexpr int kSr = (FC2 || PAIR) ? 2 : 4;
  // expanded sub-tiles: 3 when that keeps the allocation at 128 columns (fc2 at tiles of <= 32
  // tokens: four CTAs' worth of tensor memory per SM) or two CTAs fit (PAIR)
  static constexpr int kSa = (PAIR || (FC2 && BN <= 32)) ? 3 : 4;
  static constexpr int kSb = FC2 ? (BN <= 32 ? 8 : 4)
                                 : (BN <= 32 ? 8 : (BN <= 64 ? 6 : 4));
  static constexpr int kSmem = kSr * kRaw + kSb * kB + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory");
  // tensor memory: D (kMats x BN columns), then the expanded-A ring (kMats x 32 columns per
  // 64-wide sub-tile: two f16 per column)
  static constexpr int kColsD = kMats * BN;
  static constexpr int kA0 = (kColsD + 31) / 32 * 32;
  static constexpr int kASlot = kMats * 32;
  static constexpr int kCols = kA0 + kSa * kASlot;
  static constexpr int kAlloc = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128
                                : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "tensor memory");
};

struct Tc16Params {
  CUtensorMap tm_act;         // f16 [Sm][K] activations, boxes 64 x BN, 128-byte swizzle
  // weight tiles of 128 rows x 256 K per matrix (moe_common.cuh): one bulk copy each
  const uint8_t* nv_codes;    // NVFP4 codes, 16 KB tiles (128-byte swizzled rows)
  const uint8_t* nv_scales;   // NVFP4 scales, 2 KB tiles
  const uint8_t* nf_codes;    // NF3 planes, 12 KB tiles
  const uint8_t* nf_scales;   // NF3 scales, 2 KB tiles
  const int32_t* tier_map;    // hybrid: (tier << 24) | local; nullptr: every expert NVFP4
  const float* gscale;        // NVFP4 per-expert global of this matrix ([E4]); MXFP4 kept
                              // tier: the matrix's power-of-two factor
  int mx;                     // kept tier MXFP4 (f16 multiplier per group of 32)
  const float* agscale;       // MXFP8 activations: per-expert activation global scale of this
                              // GEMM's input ([E]); nullptr: 16-bit activations
  const float* agscale2;      // fc1 with MXFP8 activations: that of fc2's input (h)
  // A8 opt-in of the MXFP4 kept tier (0: off): the static FP8 input scale of this GEMM's
  // activations, which the kept tier's operands carry as E4M3 code values; and, for fc1, the
  // fp32 reciprocal of fc2's input scale, by which h is quantised
  float a8_s, a8_inv_next;
  int rb_in_x;                // grid (RB, tiles, splits) instead of (tiles, RB, splits)
  const int4* tiles;
  const int32_t* ctrl;
  int32_t* err;
  // fc1 outputs
  uint16_t* h16;              // f16 [Sm][Ip] (bf16-rounded SwiGLU output)
  float* gacc;                // [splits][Sm][2][Ip] split-K partial sums, one slice per split
  int32_t* tickets;
  // fc2 outputs
  const int32_t* perm;
  const float* topk_w;        // combine weights; nullptr: 1 (router weights on the input)
  float* acc;
  float* rbuf;
  int K, R, I, Ip, RB, KT, Sm, splits, topk, deterministic, H, nf3_row_bytes;
  float limit, alpha, beta;
};

__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}"
      : "=r"(out)
      : "r"(byte));
  return out;
}
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}"
      : "=r"(out)
      : "r"(two_bytes));
  return out;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_bcast(uint32_t f16bits) {
  return (f16bits & 0xFFFFu) | (f16bits << 16);
}

// NVFP4 row r, K sub-tile q (64 elements), half h (elements 32h..32h+31) -> 16 f16x2 words in
// K order (E2M1 x E4M3 scale, exact in f16).  Raw smem: the tile's 128-byte swizzled code rows
// (16-byte chunk j at j ^ (r % 8)) and 16-byte scale rows.  `mx`: the kept tier is MXFP4 and
// the scale row holds one f16 multiplier per group of 32 (the half's two bytes) instead of two
// E4M3 scales per half.
__device__ __forceinline__ void convert_nvfp4_half(const uint8_t* codes, const uint8_t* scales,
                                                   int r, int q, int h, bool mx, uint32_t* out) {
  const int sw = r & 7;
  const uint4 c = *reinterpret_cast<const uint4*>(codes + r * 128 + (((2 * q + h) ^ sw) << 4));
  const uint32_t sc4 = *reinterpret_cast<const uint32_t*>(scales + r * 16 + q * 4);
  const uint32_t raw = (sc4 >> (16 * h)) & 0xFFFF;
  uint32_t sc[2];
  if (mx) {
    sc[0] = sc[1] = f16x2_bcast(raw);
  } else {
    const uint32_t s2 = cvt_e4m3x2_f16x2(raw);
    sc[0] = f16x2_bcast(s2);
    sc[1] = f16x2_bcast(s2 >> 16);
  }
  const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t w = words[jj];
    const uint32_t s = sc[jj >> 1];
    out[4 * jj + 0] = hmul2(cvt_e2m1x2_f16x2(w & 0xFF), s);
    out[4 * jj + 1] = hmul2(cvt_e2m1x2_f16x2((w >> 8) & 0xFF), s);
    out[4 * jj + 2] = hmul2(cvt_e2m1x2_f16x2((w >> 16) & 0xFF), s);
    out[4 * jj + 3] = hmul2(cvt_e2m1x2_f16x2(w >> 24), s);
  }
}

// The eight NF3 levels of a scale group as f16 bytes for byte-permute look-ups: f16 of
// bf16(fp32(LUT[4 + i]) * scale) for i = 0..3 (codes 4..7), low bytes in tlo and high bytes in
// thp; thn holds the high bytes with the sign flipped.  Codes 3..0 are the negatives of codes
// 4..7 (the LUT is antisymmetric, and the product and both roundings are sign-symmetric), so
// code c reads entry c - 4 (c >= 4) or 7 - c (c < 4, from thn).
__device__ __forceinline__ void nf3_tables(float scale, uint32_t& tlo, uint32_t& thp,
                                           uint32_t& thn) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = __bfloat162float(__float2bfloat16_rn(c_nf3_lut16[4 + i] * scale));
    const uint32_t v = __half_as_ushort(__float2half_rn(a));
    lo |= (v & 0xFFu) << (8 * i);
    hi |= (v >> 8) << (8 * i);
  }
  tlo = lo;
  thp = hi;
  thn = hi ^ 0x80808080u;
}

// Byte-permute selectors of 8 codes: nibble k = c' of code k (low 2 bits at bits 2k..2k+1 of
// l16, high bit at bit k of h8), where c' = c - 4 for c >= 4 and 7 - c below, i.e. the low
// bits XOR 7 when the high bit is clear: the low bits and the high bits spread to nibbles,
// then one XOR.
__device__ __forceinline__ uint32_t nf3_sel8(uint32_t l16, uint32_t h8) {
  uint32_t x = l16;
  x = (x | (x << 8)) & 0x00FF00FFu;
  x = (x | (x << 4)) & 0x0F0F0F0Fu;
  x = (x | (x << 2)) & 0x33333333u;
  uint32_t y = h8;
  y = (y | (y << 12)) & 0x000F000Fu;
  y = (y | (y << 6)) & 0x03030303u;
  y = (y | (y << 3)) & 0x11111111u;
  return x ^ ((y ^ 0x11111111u) * 7u);
}

// NF3 row r, K sub-tile q (64 codes), half h (codes 32h..32h+31: one scale group) -> 16 f16x2
// words in K order.  Raw smem: 32-byte rows of the tile's 2-bit plane halves (bytes 0..31 at +0,
// 32..63 at +4096) and of its 1-bit plane (+8192).  Per 4 codes: the high bytes (with sign) by
// one byte permute over thp:thn, the low bytes by one over tlo, two more to interleave them.
__device__ __forceinline__ void convert_nf3_half(const uint8_t* codes, const uint8_t* scales,
                                                 int r, int q, int h, uint32_t* out) {
  const uint2 lo = *reinterpret_cast<const uint2*>(codes + (q >> 1) * 4096 + r * 32 +
                                                   (q & 1) * 16 + 8 * h);
  const uint32_t hi = *reinterpret_cast<const uint32_t*>(codes + 8192 + r * 32 + q * 8 + 4 * h);
  uint32_t tlo, thp, thn;
  nf3_tables(e4m3_to_f32(scales[r * 16 + q * 2 + h]), tlo, thp, thn);
  const uint32_t low[2] = {lo.x, lo.y};
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const uint32_t cs = nf3_sel8((low[jj >> 1] >> ((jj & 1) * 16)) & 0xFFFFu,
                                 (hi >> (jj * 8)) & 0xFFu);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const uint32_t sel = cs >> (16 * g);
      const uint32_t ph = __byte_perm(thp, thn, sel);
      const uint32_t pl = __byte_perm(tlo, tlo, sel & 0x3333u);
      out[4 * jj + 2 * g] = __byte_perm(pl, ph, 0x5140);
      out[4 * jj + 2 * g + 1] = __byte_perm(pl, ph, 0x7362);
    }
  }
}

__device__ __forceinline__ float swiglu16(float gate, float up, float limit, float alpha,
                                          float beta) {
  const float g = fminf(gate, limit);
  const float u = fminf(fmaxf(up, -limit), limit);
  return g / (1.0f + expf(-alpha * g)) * (u + beta);
}

// h (fp32) -> bf16 rounding (the method's intermediate) -> f16 bits for the next MMA.
__device__ __forceinline__ uint16_t h_to_f16(float h, int32_t* err) {
  const float hb = __bfloat162float(__float2bfloat16_rn(h));
  if (fabsf(hb) > 65504.f) atomicOr(err, kErrRange);
  return __half_as_ushort(__float2half_rn(hb));
}

// MXFP8 activations: h of one token column for this warp's 32 features (one MX block), times
// the expert's activation global scale a2, quantised by the OCP MX rule and returned as the f16
// of the dequantised value E4M3 x 2^(s-127) (exact while the block scale is at most 2^7: larger
// sets the range bit).  All 32 lanes call it with the same column.
// Static per-tensor FP8 (the kept tier's A8 opt-in): the E4M3 code of fp32(h * inv) (nearest
// even, saturating) as the f16 of the code's value (exact); the scale joins fc2's epilogue.
__device__ __forceinline__ uint16_t h_to_f16_fp8s(float h, float inv) {
  return __half_as_ushort(__float2half_rn(e4m3_to_f32((uint8_t)f32_to_e4m3(__fmul_rn(h, inv)))));
}

__device__ __forceinline__ uint16_t h_to_f16_mx(float h, float a2, int32_t* err) {
  const float v = h * a2;
  float amax = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const uint32_t s = mx_scale_byte(amax);
  if (s > 127 + 7) atomicOr(err, kErrRange);
  const float q = e4m3_to_f32((uint8_t)f32_to_e4m3(v * e8m0_inv_f32(s))) * e8m0_to_f32(s);
  return __half_as_ushort(__float2half_rn(q));
}

// The PAIR form asks the compiler for two CTAs per SM (<= 102 registers a thread): without the
// bound it took 168 and the register file held one CTA, whatever its shared and tensor memory.
template <int BN, bool FC2, bool PAIR>
__global__ void __launch_bounds__(k16Threads, PAIR ? 2 : 1)
gemm_tc16_kernel(const __grid_constant__ Tc16Params p) {
  using Cfg = Tc16Cfg<BN, FC2, PAIR>;
  constexpr int kMats = Cfg::kMats;
  __shared__ uint32_t s_tmem;
  tmem_alloc_first(&s_tmem, Cfg::kAlloc);
  pdl_wait_prev();     // previous kernel of the call complete, its writes visible
  // the row blocks of a tile are adjacent in launch order (while the tiles fit the grid's y),
  // so the CTAs that read the same activation tile run together and share it through L2
  const int tile = p.rb_in_x ? blockIdx.y : blockIdx.x;
  if (tile >= p.ctrl[1]) {
    tmem_exit_early(&s_tmem, Cfg::kAlloc);
    return;
  }
  const int4 td = p.tiles[tile];
  const int e = td.x, p0 = td.y, n = td.z;
  const int rb = p.rb_in_x ? blockIdx.x : blockIdx.y, split = blockIdx.z;
  const int kt0 = split * p.KT / p.splits, kt1 = (split + 1) * p.KT / p.splits;
  const int nraw = kt1 - kt0;               // raw stages (256-wide K)
  const int nsub = nraw * 4;                // 64-wide sub-tiles
  int le = e;
  bool nf3 = false;
  if (p.tier_map != nullptr) {
    const int m = p.tier_map[e];
    nf3 = (m >> 24) == kTierNF3;
    le = m & 0xFFFFFF;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* raw_base = smem;
  uint8_t* b_base = raw_base + Cfg::kSr * Cfg::kRaw;
  __shared__ __align__(8) uint64_t raw_full[Cfg::kSr], raw_empty[Cfg::kSr];
  __shared__ __align__(8) uint64_t a_full[Cfg::kSa], a_empty[Cfg::kSa];
  __shared__ __align__(8) uint64_t b_full[Cfg::kSb], b_empty[Cfg::kSb];
  __shared__ __align__(8) uint64_t done;
  __shared__ int s_last, s_fail;
  __shared__ int s_f[BN];          // fc2: flat slot index of each tile column
  __shared__ float s_w[BN];        // fc2: its router weight

  if (tid == 32) {
    for (int s = 0; s < Cfg::kSr; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 8);
    }
    for (int s = 0; s < Cfg::kSa; ++s) {
      mbar_init(&a_full[s], 8);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < Cfg::kSb; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(&done, 1);
    s_fail = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the next kernel may launch only once every CTA of this one holds its tensor memory (fc1
  // takes all of an SM's columns: a CTA of the next kernel allocating first would make it wait
  // for columns that are freed only after this kernel completes)
  pdl_launch_next();
  const uint32_t tmem = s_tmem;
  bool ok = true;
  int issued = 0, g = 0;   // raw stages filled, next activation sub-tile to load

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
      int i = 0;
      for (; i < nraw && ok; ++i) {
        const int s = i % Cfg::kSr;
        if (i >= Cfg::kSr) ok = mbar_wait(&raw_empty[s], ((i / Cfg::kSr) - 1) & 1, p.err);
        if (!ok) break;
        uint8_t* st = raw_base + s * Cfg::kRaw;
        const int kt = kt0 + i;
        const uint32_t code_bytes = nf3 ? kNfCodeTile : kNvCodeTile;
        mbar_arrive_expect_tx(&raw_full[s], kMats * (code_bytes + kW16ScaleTile));
        for (int m = 0; m < kMats; ++m) {
          const size_t tile = w16_tile(FC2 ? le : 2 * le + m, rb, kt, p.RB, p.KT);
          bulk_load_hint(st + m * k16RawCodes, (nf3 ? p.nf_codes : p.nv_codes) +
                         tile * code_bytes, code_bytes, &raw_full[s], pol);
          bulk_load_hint(st + kMats * k16RawCodes + m * k16RawScales,
                         (nf3 ? p.nf_scales : p.nv_scales) + tile * kW16ScaleTile, kW16ScaleTile,
                         &raw_full[s], pol);
        }
        // the four activation sub-tiles of this raw stage
        for (int q = 0; q < 4 && ok; ++q, ++g) {
          const int sb = g % Cfg::kSb;
          if (g >= Cfg::kSb) ok = mbar_wait(&b_empty[sb], ((g / Cfg::kSb) - 1) & 1, p.err);
          if (!ok) break;
          mbar_arrive_expect_tx(&b_full[sb], Cfg::kB);
          tma_load_2d(b_base + sb * Cfg::kB, &p.tm_act, kt * k16RawK + q * k16SubK, p0,
                      &b_full[sb]);
        }
      }
      issued = i;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((128u >> 4) << 24);
      for (int g = 0; g < nsub && ok; ++g) {
        const int sa = g % Cfg::kSa, sb = g % Cfg::kSb;
        ok = mbar_wait(&a_full[sa], (g / Cfg::kSa) & 1, p.err) &&
             mbar_wait(&b_full[sb], (g / Cfg::kSb) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t A = tmem + Cfg::kA0 + sa * Cfg::kASlot;
        const uint8_t* B = b_base + sb * Cfg::kB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = desc_sw128(B + 32 * kk);
          const uint32_t acc = (g > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
          for (int m = 0; m < kMats; ++m)
            mma_f16_ta(tmem + m * BN, A + m * 32 + 8 * kk, bd, idesc, acc);
        }
        tc_commit(&a_empty[sa]);
        tc_commit(&b_empty[sb]);
      }
      tc_commit(&done);
    }
  } else {
    // converters: two threads per row of the 128-row weight block, each expanding one half of
    // every 64-wide sub-tile into tensor memory (warps 2..5 the first half, 6..9 the second; a
    // warp handles the rows of its tensor-memory lane quadrant)
    const int r = 32 * (warp & 3) + lane, half = (warp - 2) >> 2;
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    if (FC2 && half == 0 && r < n) {
      // the combine's slot indices and router weights, read by these threads' epilogue
      const int f = p.perm[p0 + r];
      s_f[r] = f;
      s_w[r] = p.topk_w != nullptr ? p.topk_w[f] : 1.f;   // nullptr: weights on the input
    }
    int g = 0;
    for (int i = 0; i < nraw && ok; ++i) {
      const int s = i % Cfg::kSr;
      ok = mbar_wait_warp(&raw_full[s], (i / Cfg::kSr) & 1, p.err);
      if (!ok) break;
      const uint8_t* st = raw_base + s * Cfg::kRaw;
      for (int q = 0; q < 4 && ok; ++q, ++g) {
        const int sa = g % Cfg::kSa;
        if (g >= Cfg::kSa) ok = mbar_wait_warp(&a_empty[sa], ((g / Cfg::kSa) - 1) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < kMats; ++m) {
          const uint8_t* c = st + m * k16RawCodes;
          const uint8_t* sc = st + kMats * k16RawCodes + m * k16RawScales;
          uint32_t words[16];
          if (nf3)
            convert_nf3_half(c, sc, r, q, half, words);
          else
            convert_nvfp4_half(c, sc, r, q, half, p.mx != 0, words);
          tmem_st16(trow + Cfg::kA0 + sa * Cfg::kASlot + m * 32 + 16 * half, words);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&raw_empty[s]);
    }
  }

  // ---- epilogue (warps 2..5): TMEM lane quadrant = warp % 4
  if (warp >= 2 && warp < 6) {
    asm volatile("bar.sync 1, 128;" ::: "memory");         // s_f / s_w written (warps 2..5)
    // one verdict per warp (the epilogue's TMEM loads and shuffles are warp-collective)
    ok = __all_sync(0xffffffffu, mbar_wait(&done, 0, p.err) && ok);
    tc_fence_after();
    __syncwarp();
    const int quad = warp & 3;
    const int row = rb * 128 + quad * 32 + lane;           // weight row of this lane
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    // weight global (NVFP4) over the activation global (MXFP8 activations carry a * x)
    const float gs = ((!nf3 && p.gscale != nullptr) ? p.gscale[le] : 1.f) /
                     (p.agscale != nullptr ? p.agscale[e] : 1.f) *
                     ((!nf3 && p.a8_s != 0.f) ? p.a8_s : 1.f);
    const float a8_inv = nf3 ? 0.f : p.a8_inv_next;
    const float a_next = (!FC2 && p.agscale2 != nullptr) ? p.agscale2[e] : 0.f;
    if (ok && nsub > 0) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v0[16], v1[16];
        tmem_ld16(trow + c0, v0);
        if (!FC2) tmem_ld16(trow + BN + c0, v1);
        if (c0 >= n) continue;
        if (FC2) {
          // 16 token columns x this warp's 32 output features, read back transposed so that
          // the combine adds 16 bytes (4 features of one token) per atomic; the raw stages are
          // free once `done` has completed (every copy landed and was consumed)
          float(*sy)[32] = reinterpret_cast<float(*)[32]>(raw_base + quad * 2048);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) sy[jj][lane] = v0[jj] * gs;
          __syncwarp();
          const int h4 = rb * 128 + quad * 32 + 4 * (lane & 7);
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
              const float h = row < p.I ? swiglu16(v1[j] * gs, v0[j] * gs, p.limit, p.alpha,
                                                   p.beta)
                                        : 0.f;
              p.h16[(size_t)pos * p.Ip + row] =
                  a8_inv != 0.f ? h_to_f16_fp8s(h, a8_inv)
                  : p.agscale2 != nullptr ? h_to_f16_mx(h, a_next, p.err) : h_to_f16(h, p.err);
            } else {
              float* gg = p.gacc + ((size_t)split * p.Sm + pos) * 2 * p.Ip;
              gg[row] = v0[j];
              gg[p.Ip + row] = v1[j];
            }
          } else {
            const int f = s_f[c];
            const float v = s_w[c] * (v0[j] * gs);
            if (p.deterministic)
              p.rbuf[(size_t)f * p.H + row] = v;
            else
              atomicAdd(&p.acc[(size_t)(f / p.topk) * p.H + row], v);
          }
        }
      }
    }
  }
  if (!FC2 && p.splits > 1) __threadfence();
  if (!ok) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  // a wait gave up: let this CTA's copies land before its shared memory is released (its MMAs
  // completed or timed out at the wait on `done`)
  if (s_fail && warp == 0 && lane == 0) {
    drain_stage_loads<Cfg::kSr>(raw_full, issued, p.err);
    drain_stage_loads<Cfg::kSb>(b_full, g, p.err);
  }
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc);
  if (!FC2 && p.splits > 1) {
    if (tid == 0) {
      __threadfence();
      const int t = atomicAdd(&p.tickets[tile * p.RB + rb], 1);
      s_last = (t == p.splits - 1);
    }
    __syncthreads();
    if (s_last && warp >= 2 && warp < 6) {
      __threadfence();
      const int quad = warp & 3;
      const int row = rb * 128 + quad * 32 + lane;
      const float gs = ((!nf3 && p.gscale != nullptr) ? p.gscale[le] : 1.f) /
                       (p.agscale != nullptr ? p.agscale[e] : 1.f) *
                       ((!nf3 && p.a8_s != 0.f) ? p.a8_s : 1.f);
      const float a_next = p.agscale2 != nullptr ? p.agscale2[e] : 0.f;
      const float a8_inv = nf3 ? 0.f : p.a8_inv_next;
      // partial sums added in split order (the same result on every run), 16 columns at a
      // time with each split's 32 loads issued together
      for (int c0 = 0; c0 < n; c0 += 16) {
        float up[16], gt[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) up[j] = gt[j] = 0.f;
        for (int sp = 0; sp < p.splits; ++sp) {
          const float* gg = p.gacc + ((size_t)sp * p.Sm + p0 + c0) * 2 * p.Ip + row;
          float a[16], b[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // columns beyond the tile repeat its last one (a valid address) and add nothing
            const size_t jj = (size_t)min(j, n - 1 - c0);
            a[j] = __ldcg(gg + jj * 2 * p.Ip);
            b[j] = __ldcg(gg + jj * 2 * p.Ip + p.Ip);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (c0 + j < n) {
              up[j] += a[j];
              gt[j] += b[j];
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c0 + j < n) {
            const float h = row < p.I ? swiglu16(gt[j] * gs, up[j] * gs, p.limit, p.alpha, p.beta)
                                      : 0.f;
            p.h16[(size_t)(p0 + c0 + j) * p.Ip + row] =
                a8_inv != 0.f ? h_to_f16_fp8s(h, a8_inv)
                : p.agscale2 != nullptr ? h_to_f16_mx(h, a_next, p.err) : h_to_f16(h, p.err);
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn16)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn16 encode16() {
  static EncodeTiledFn16 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn16>(f);
  }
  return fn;
}

// f16 activations [rows][K] with boxes 64 x box_rows and 128-byte swizzle.
static bool tmap_f16(CUtensorMap* tm, const void* base, int K, int rows, int box_rows) {
  EncodeTiledFn16 enc = encode16();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool FC2, bool PAIR = false>
static cudaError_t launch16(const Tc16Params& p, int tiles, cudaStream_t st) {
  using Cfg = Tc16Cfg<BN, FC2, PAIR>;
  auto kernel = gemm_tc16_kernel<BN, FC2, PAIR>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    // all of the unified L1 / shared storage as shared memory
    cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    attr = true;
  }
  Tc16Params q = p;
  q.rb_in_x = tiles <= 65535 ? 1 : 0;
  const int sp = FC2 ? 1 : p.splits;
  const dim3 grid = q.rb_in_x ? dim3(p.RB, tiles, sp) : dim3(tiles, p.RB, sp);
  return launch_kernel(kernel, grid, dim3(k16Threads), Cfg::kSmem, st, true, q);
}

// fc1 of the 16-bit path at two CTAs per SM (token tiles of at most 32)
bool tc16_fc1_pair(int bn, int quant) {
  return bn <= 32 && (quant == kQuantNVFP4 || quant == kQuantW4A8Nv || quant == kQuantHybrid ||
                      quant == kQuantHybridMx);
}

// stage 0: fc1 (+ SwiGLU, h -> bf16 -> f16), stage 1: fc2 (+ combine).
cudaError_t launch_tc16_stage(int stage, const DevWeights& w, const RunPtrs& r, const PlanDims& d,
                              int bn, int tiles, int splits, const float* topk_w, int M,
                              cudaStream_t st) {
  const int Sm = M * d.topk;
  Tc16Params p;
  memset(&p, 0, sizeof(p));
  const bool fc2 = stage == 1;
  const int K = fc2 ? d.Ip : d.H;
  const int KT = (K + k16RawK - 1) / k16RawK;
  p.nv_codes = fc2 ? w.w2 : w.w13;
  p.nv_scales = fc2 ? w.s2 : w.s13;
  p.nf_codes = fc2 ? w.nf_w2 : w.nf_w13;
  p.nf_scales = fc2 ? w.nf_s2 : w.nf_s13;
  if (!tmap_f16(&p.tm_act, fc2 ? (const void*)r.h16 : (const void*)r.x16, K, Sm, bn))
    return cudaErrorInvalidValue;
  p.tier_map = w.tier_map;
  p.gscale = fc2 ? w.g2 : w.g13;
  p.mx = w.mx_kept;
  p.agscale = fc2 ? w.ag2 : w.ag13;
  p.agscale2 = fc2 ? nullptr : w.ag2;
  p.a8_s = d.kept_a8 ? (fc2 ? d.a8_s2 : d.a8_s13) : 0.f;
  p.a8_inv_next = (d.kept_a8 && !fc2) ? d.a8_inv2 : 0.f;
  p.tiles = r.tiles; p.ctrl = r.ctrl; p.err = r.ctrl;
  p.h16 = reinterpret_cast<uint16_t*>(r.h16); p.gacc = r.g; p.tickets = r.tickets;
  p.perm = r.perm; p.topk_w = topk_w; p.acc = r.acc; p.rbuf = r.rbuf;
  p.K = K; p.R = fc2 ? d.H : d.I; p.I = d.I; p.Ip = d.Ip; p.RB = fc2 ? d.H / 128 : cdiv(d.I, 128);
  p.KT = KT; p.Sm = Sm; p.splits = fc2 ? 1 : splits; p.topk = d.topk;
  p.deterministic = d.deterministic; p.H = d.H; p.nf3_row_bytes = 3 * K / 8;
  p.limit = d.limit; p.alpha = d.alpha; p.beta = d.beta;
  const bool pair = !fc2 && tc16_fc1_pair(bn, d.quant);
  switch (bn * 2 + (fc2 ? 1 : 0)) {
    case 32: return pair ? launch16<16, false, true>(p, tiles, st)
                         : launch16<16, false>(p, tiles, st);
    case 33: return launch16<16, true>(p, tiles, st);
    case 64: return pair ? launch16<32, false, true>(p, tiles, st)
                         : launch16<32, false>(p, tiles, st);
    case 65: return launch16<32, true>(p, tiles, st);
    case 128: return launch16<64, false>(p, tiles, st);
    case 129: return launch16<64, true>(p, tiles, st);
    case 256: return launch16<128, false>(p, tiles, st);
    default: return launch16<128, true>(p, tiles, st);
  }
}

}  // namespace moe
