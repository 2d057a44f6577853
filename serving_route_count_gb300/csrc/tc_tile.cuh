// tc_tile.cuh - pieces shared by the W4A8 tensor-core kernels: tile geometry, activation scale
// atoms, the SwiGLU + MXFP8 requantisation of an accumulator column, tensor maps.
#pragma once

#include <cuda.h>

#include "moe_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

using namespace tc;

constexpr int kTcThreads = 128;
constexpr int kTileBytesA = 128 * 128;   // 128 rows x 128 K of padded FP4 (1 byte / element)
// The packed-FP4 TMA format counts the bytes it reads from global memory (two elements per
// byte) as the transaction size, not the expanded shared-memory footprint.
constexpr int kTxBytesA = 128 * 128 / 2;

// Token columns of one block-scaled MMA.  A tile of BN tokens runs as ceil(BN / 32) MMAs of
// up to 32 columns each: the activation scales of a tile are BN consecutive 16-byte atom rows
// (bytes 0..3 = a token's four scales of the K tile), and each 32-row run of them is exactly the
// scale atom of a 32-column MMA, copied to tensor memory as is.
template <int BN>
struct NChunks {
  static constexpr int kCount = (BN + 31) / 32;
  static constexpr int kWidth = BN < 32 ? BN : 32;
  static_assert(BN % 16 == 0 && BN <= 96 && (BN <= 32 || BN % 32 == 0), "token tile width");
};

// What a tile of n tokens at tile width BN loads per K tile: up to 32 tokens the whole BN-row
// box; beyond, only the 32-row chunks that hold tokens (one 32-column MMA each), so that a
// wide tile of a cold expert costs no more than a narrow one.
template <int BN>
struct TileLoad {
  int nch;              // 32-column MMAs of the tile (1 up to 32 tokens)
  uint32_t b_bytes;     // activation codes
  uint32_t sf_bytes;    // activation scale atom rows
  __device__ __forceinline__ explicit TileLoad(int n) {
    if (BN <= 32) {
      nch = 1;
      b_bytes = BN * 128;
      sf_bytes = BN * 16;
    } else {
      nch = min(NChunks<BN>::kCount, (n + 31) >> 5);
      b_bytes = (uint32_t)nch * 4096;
      sf_bytes = (uint32_t)nch * 512;
    }
  }
  // activation codes of K offset k, slot positions p0.. (the map's boxes are BN rows up to
  // 32, else 32 rows)
  __device__ __forceinline__ void load_b(uint8_t* dst, const CUtensorMap* tm, int k, int p0,
                                         uint64_t* bar) const {
    if (BN <= 32) {
      tma_load_2d(dst, tm, k, p0, bar);
    } else {
      for (int j = 0; j < nch; ++j) tma_load_2d(dst + 4096 * j, tm, k, p0 + 32 * j, bar);
    }
  }
};
// Rows of the activation tensor map's box at tile width BN.
inline int act_box_rows(int bn) { return bn < 32 ? bn : 32; }

// Scale atom of BN activation rows for one K tile from a [j][BN] staging buffer (4 bytes per row:
// the row's four E8M0 bytes of that K tile): byte (n%32)*16 + (n/32)*4 + kb.
template <int BN>
static __device__ __forceinline__ void write_act_sf_rows(uint8_t* dst, const uint32_t* rows,
                                                         int lane) {
#pragma unroll
  for (int n = lane; n < BN; n += 32)
    *reinterpret_cast<uint32_t*>(dst + (n & 31) * 16 + (n >> 5) * 4) = rows[n];
}

// Routing of a small call in shared memory, ahead of the routing launch's tables: the experts
// of the GEMM tile list, built as the routing launch builds it (experts in ascending order,
// ceil(count / tile_slots) tiles each; ids outside [ep_first, ep_first + E) dropped), from the
// router ids alone.
// A kernel chained behind the routing launch may read the ids before waiting for it (the ids
// were complete when the routing launch passed its own wait), so it can request weights early.
// scratch: (E + kPreRouteTiles + 64) ints of shared memory; on return scratch[E + t] is the
// expert of tile t for t < min(tiles, kPreRouteTiles).  With `info` (PreRouteInfo, the kernel's
// own shared memory) it also keeps, per tile, its expert, token count, first slot position and
// index among its expert's tiles, and per flat slot the local expert id (-1 when dropped): what
// a kernel needs to gather the tile's activations itself.  Every thread of the CTA (NT threads)
// calls it; returns the tile count.
constexpr int kPreRouteSlots = 256;   // calls of at most this many flat slots
constexpr int kPreRouteTiles = 256;
struct PreRouteInfo {
  int te[kPreRouteTiles];             // expert | (token count << 16)
  int tp[kPreRouteTiles];             // first slot position | (index within the expert << 16)
  int16_t lid[kPreRouteSlots];        // local expert of each flat slot, -1 when dropped
};
template <int NT>
static __device__ int pre_route_tiles(const int32_t* ids, int Mk, int E, int ep_first,
                                      int tile_slots, int* scratch,
                                      PreRouteInfo* info = nullptr) {
  int* s_cnt = scratch;
  int* s_tile_e = scratch + E;
  int* s_red = scratch + E + kPreRouteTiles;       // [0, 32): tiles, [32, 64): slots per warp
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += NT) s_cnt[e] = 0;
  __syncthreads();
  for (int f = tid; f < Mk; f += NT) {
    const int e = local_expert(__ldcg(ids + f), ep_first, E);
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    if (info != nullptr) info->lid[f] = (int16_t)((e >= 0 && e < E) ? e : -1);
  }
  __syncthreads();
  const int per = (E + NT - 1) / NT;        // thread t: experts [t*per, t*per + per)
  int lt = 0, ls = 0;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e < E) {
      lt += (s_cnt[e] + tile_slots - 1) / tile_slots;
      ls += s_cnt[e];
    }
  }
  // exclusive scans of the per-thread tile and slot counts
  int incl = lt, incs = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    const int z = __shfl_up_sync(0xffffffffu, incs, o);
    if (lane >= o) {
      incl += y;
      incs += z;
    }
  }
  if (lane == 31) {
    s_red[warp] = incl;
    s_red[32 + warp] = incs;
  }
  __syncthreads();
  int before = 0, total = 0, before_s = 0;
  for (int w = 0; w < NT / 32; ++w) {
    before += w < warp ? s_red[w] : 0;
    before_s += w < warp ? s_red[32 + w] : 0;
    total += s_red[w];
  }
  int t = before + incl - lt, pos = before_s + incs - ls;
  for (int i = 0; i < per; ++i) {
    const int e = tid * per + i;
    if (e >= E) break;
    const int c = s_cnt[e];
    for (int j = 0; j * tile_slots < c; ++j, ++t) {
      if (t < kPreRouteTiles) {
        s_tile_e[t] = e;
        if (info != nullptr) {
          info->te[t] = e | (min(tile_slots, c - j * tile_slots) << 16);
          info->tp[t] = (pos + j * tile_slots) | (j << 16);
        }
      }
    }
    pos += c;
  }
  // the scratch lies in a pipeline stage that TMA writes next
  fence_proxy_async_smem();
  __syncthreads();
  return total;
}

// The tokens of tile t of a pre-routed small call: the flat slots of the tile's expert in
// ascending order, ranks [j * tile_slots, j * tile_slots + n), as token indices (slot / topk)
// into tok[0 .. n).  One warp calls it (a ballot per 32 flat slots).
static __device__ __forceinline__ void pre_route_tile_tokens(const PreRouteInfo& info, int t,
                                                             int Mk, int topk, int tile_slots,
                                                             int* tok) {
  const int lane = threadIdx.x & 31;
  const int e = info.te[t] & 0xFFFF, n = info.te[t] >> 16;
  const int r0 = (info.tp[t] >> 16) * tile_slots;
  int seen = 0;
  for (int f0 = 0; f0 < Mk && seen < r0 + n; f0 += 32) {
    const int f = f0 + lane;
    const bool mine = f < Mk && info.lid[f] == e;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    const int rank = seen + __popc(m & ((1u << lane) - 1u));
    if (mine && rank >= r0 && rank < r0 + n) tok[rank - r0] = f / topk;
    seen += __popc(m);
  }
  __syncwarp();
}

// In-kernel MXFP8 quantisation of a tile's activations, one K tile (128 activations per token)
// per pipeline stage, by 64 threads (two warps; thread q owns the (row, block) items q, q + 64,
// ...: row = item / 4, block of 32 = item % 4).  load() issues the bf16 loads of a K tile into
// registers; quant() turns them into E4M3 codes and E8M0 scales in registers; store() writes
// those straight into a stage: the B operand (BN rows of 128 codes, 16-byte chunk j of row r at
// chunk j ^ (r % 8): the 128-byte swizzle the MMA's descriptor reads) and its scale atom rows
// (row r: byte (r % 32) * 16 + (r / 32) * 4 + block).  Rows r >= n are written as zeros.  With
// xq / xs set, store() also writes the codes and scales row-major at slot position p0 + r (a
// copy for inspection).  The smem writes are generic-proxy stores: the caller fences them for
// the tensor cores (fence.proxy.async) before signalling the stage.
template <int BN>
struct ActQuant {
  static constexpr int kItems = BN * 4 / 64;
  static_assert(BN == 16 || BN == 32, "in-kernel quantisation at tile widths 16 / 32");
  struct Codes {
    uint32_t w[kItems][8];
    uint32_t sc[kItems];
  };
  const __nv_bfloat16* x;
  int H, q;
  __device__ __forceinline__ void load(uint4 (&v)[kItems][4], const int* tok, int n,
                                       int kt) const {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int item = q + 64 * it, r = item >> 2, b = item & 3;
      if (r < n) {
        const uint4* src =
            reinterpret_cast<const uint4*>(x + (size_t)tok[r] * H + kt * 128 + b * 32);
#pragma unroll
        for (int w = 0; w < 4; ++w) v[it][w] = __ldg(src + w);
      }
    }
  }
  __device__ __forceinline__ void quant(const uint4 (&v)[kItems][4], int n, Codes& c) const {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int r = (q + 64 * it) >> 2;
      if (r < n) {
        c.sc[it] = mxfp8_block32(v[it], c.w[it]);
      } else {
        c.sc[it] = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) c.w[it][j] = 0u;
      }
    }
  }
  __device__ __forceinline__ void store(const Codes& c, int n, int kt, uint8_t* b_tile,
                                        uint8_t* sf_rows, uint8_t* xq, uint8_t* xs,
                                        int p0) const {
#pragma unroll
    for (int it = 0; it < kItems; ++it) {
      const int item = q + 64 * it, r = item >> 2, b = item & 3;
      const uint32_t* w = c.w[it];
      uint8_t* row = b_tile + r * 128;
      *reinterpret_cast<uint4*>(row + (((2 * b) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(row + (((2 * b + 1) ^ (r & 7)) << 4)) =
          make_uint4(w[4], w[5], w[6], w[7]);
      sf_rows[(r & 31) * 16 + (r >> 5) * 4 + b] = (uint8_t)c.sc[it];
      if (xq != nullptr && r < n) {
        uint4* dq = reinterpret_cast<uint4*>(xq + (size_t)(p0 + r) * H + kt * 128 + b * 32);
        dq[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dq[1] = make_uint4(w[4], w[5], w[6], w[7]);
        xs[(size_t)(p0 + r) * (H / 32) + kt * 4 + b] = (uint8_t)c.sc[it];
      }
    }
  }
};

// Quantises the K tiles k0 .. k0 + len - 1 of one tile into the stages of fill numbers i0, i0 + 1,
// ... of an S-stage ring, signalling each stage's `full` barrier once per warp.  For each K tile
// the codes are computed and the loads of the K tile two ahead issued before waiting for the
// stage to be free (its `empty` phase, from the second lap on), so the load latency and the
// arithmetic overlap that wait.  Returns false when a wait gave up.
template <int BN, int S>
static __device__ __forceinline__ bool act_quant_run(
    const ActQuant<BN>& aq, const int* tok, int n, int k0, int len, int i0, uint8_t* smem,
    int stage_bytes, int off_b, int off_sf, uint64_t* full, uint64_t* empty, uint8_t* xq,
    uint8_t* xs, int p0, int32_t* err) {
  using V = uint4[ActQuant<BN>::kItems][4];
  V va, vb;
  typename ActQuant<BN>::Codes cq;
  const int lane = threadIdx.x & 31;
  if (len > 0) aq.load(va, tok, n, k0);
  if (len > 1) aq.load(vb, tok, n, k0 + 1);
  // K tile t from registers v (loaded two K tiles ago); v is reloaded with K tile t + 2
  auto step = [&](V& v, int t) -> bool {
    aq.quant(v, n, cq);
    if (t + 2 < len) aq.load(v, tok, n, k0 + t + 2);
    const int i = i0 + t, s = i % S;
    if (i >= S && !mbar_wait_warp(&empty[s], ((i / S) - 1) & 1, err)) return false;
    uint8_t* st = smem + s * stage_bytes;
    aq.store(cq, n, k0 + t, st + off_b, st + off_sf, xq, xs, p0);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&full[s]);
    return true;
  };
  for (int t = 0; t < len; t += 2) {
    if (!step(va, t)) return false;
    if (t + 1 < len && !step(vb, t + 1)) return false;
  }
  return true;
}

// A tile record of the routing launch for a kernel that planned its work from its own
// shared-memory routing of the ids (pre_route_tiles), read after waiting for the routing
// launch.  Both route the same ids, so the records agree; if the ids changed between the two
// reads (the caller modified them while the call ran), a tile the pre-routing counted may lie
// beyond the routing launch's list or hold an inconsistent record: such a tile reads as an
// empty tile of expert 0 (every copy and store stays inside its buffer) and sets the routing
// error bit.
static __device__ __forceinline__ int4 checked_tile(const int4* tiles, const int32_t* ctrl,
                                                    int tile, int E, int Sm, int bn,
                                                    int32_t* err) {
  const int4 td = tile < __ldcg(ctrl + 1) ? __ldcg(tiles + tile) : make_int4(-1, 0, 0, 0);
  if (td.x < 0 || td.x >= E || td.y < 0 || td.z < 1 || td.z > bn || td.y > Sm - td.z) {
    set_error(err, kErrRouteBounds);
    return make_int4(0, 0, 0, 0);
  }
  return td;
}

static __device__ __forceinline__ float swiglu(float gate, float up, float limit, float alpha,
                                               float beta) {
  const float g = fminf(gate, limit);
  const float u = fminf(fmaxf(up, -limit), limit);
  return g / (1.0f + expf(-alpha * g)) * (u + beta);
}

static __device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// h of one token column for the 32 features of this warp -> MXFP8 code + scale (row-major
// [rows][Ip/32], and, when hs16 is given, in the atom layout [Ip/128][r16][16]).
static __device__ __forceinline__ void requant_store(float h, int lane, size_t row, int Ip, int f,
                                                     uint8_t* hq, uint8_t* hs, uint8_t* hs16,
                                                     int r16) {
  const float amax = warp_max(fabsf(h));
  const uint32_t s = mx_scale_byte(amax);
  hq[row * Ip + f] = (uint8_t)f32_to_e4m3(h * e8m0_inv_f32(s));
  if (lane == 0) {
    hs[row * (Ip / 32) + (f >> 5)] = (uint8_t)s;
    if (hs16 != nullptr) hs16[((size_t)(f >> 7) * r16 + row) * 16 + ((f >> 5) & 3)] = (uint8_t)s;
  }
}

// Batches of P pieces x C columns of reduce_pieces: the 2 P C loads of a batch are issued
// together (one memory latency per batch), then added in piece order.  Every load reads a
// valid address - a piece or column beyond the last repeats the last one and its value is not
// added - so no load depends on a condition the compiler might evaluate after issuing it.
template <int P, int C, typename Base, typename Emit>
static __device__ __forceinline__ void reduce_pieces_small(int np, int n, size_t col_stride,
                                                           size_t gate_off, Base base,
                                                           Emit emit) {
  float up[C], gt[C];
#pragma unroll
  for (int jc = 0; jc < C; ++jc) up[jc] = gt[jc] = 0.f;
  for (int q0 = 0; q0 < np; q0 += P) {
    const float* bq[P];
#pragma unroll
    for (int jq = 0; jq < P; ++jq) bq[jq] = base(min(q0 + jq, np - 1));
    float a[P][C], b[P][C];
#pragma unroll
    for (int jq = 0; jq < P; ++jq) {
#pragma unroll
      for (int jc = 0; jc < C; ++jc) {
        const float* pp = bq[jq] + (size_t)min(jc, n - 1) * col_stride;
        a[jq][jc] = __ldcg(pp);
        b[jq][jc] = __ldcg(pp + gate_off);
      }
    }
#pragma unroll
    for (int jq = 0; jq < P; ++jq)
#pragma unroll
      for (int jc = 0; jc < C; ++jc)
        if (q0 + jq < np && jc < n) {
          up[jc] += a[jq][jc];
          gt[jc] += b[jq][jc];
        }
  }
#pragma unroll
  for (int jc = 0; jc < C; ++jc)
    if (jc < n) emit(jc, up[jc], gt[jc]);
}

// Adds `np` partial sums of this thread's accumulator row, in piece order 0..np-1, for the tile
// columns 0..n-1 and hands each column's (up, gate) total to emit(c, up, gate).  base(q) is the
// address of piece q's up value of column 0 (a valid address for every q < np); column c is at
// + c * col_stride, gate at + gate_off.  The piece addresses are computed once per piece and
// the loads issued 32 at a time - 16 pieces of one column, 8 of two or 4 of up to four columns,
// 16 columns of one piece beyond - so a reduction costs a few memory latencies, not one per
// piece (a decode call's unit of 56 K tiles split over ~10 CTAs reduces in one batch).  n and
// np are uniform across the warp (emit may use warp shuffles); n == 0 emits nothing.
template <typename Base, typename Emit>
static __device__ __forceinline__ void reduce_pieces(int np, int n, size_t col_stride,
                                                     size_t gate_off, Base base, Emit emit) {
  if (n <= 0) return;
  if (n <= 1) {
    reduce_pieces_small<16, 1>(np, n, col_stride, gate_off, base, emit);
    return;
  }
  if (n <= 2) {
    reduce_pieces_small<8, 2>(np, n, col_stride, gate_off, base, emit);
    return;
  }
  if (n <= 4) {
    reduce_pieces_small<4, 4>(np, n, col_stride, gate_off, base, emit);
    return;
  }
  for (int c0 = 0; c0 < n; c0 += 16) {
    float up[16], gt[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) up[j] = gt[j] = 0.f;
    for (int q = 0; q < np; ++q) {
      const float* bq = base(q);
      float a[16], b[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float* pp = bq + (size_t)min(c0 + j, n - 1) * col_stride;
        a[j] = __ldcg(pp);
        b[j] = __ldcg(pp + gate_off);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < n) {
          up[j] += a[j];
          gt[j] += b[j];
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c0 + j < n) emit(c0 + j, up[j], gt[j]);
  }
}

// ---------------------------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tc_encode_fn();
// Tile-contiguous packed FP4 weights: `tiles` runs of rows x 128 elements (64 B per row) as a 3-D
// tensor map whose boxes (128 elements x rows x 1) are whole tiles, expanded to one byte per
// element in shared memory.  rows or tiles of 0 leave the map unset (never used).
bool tmap_fp4(CUtensorMap* tm, const void* base, int rows, long long tiles);
// Byte matrix [rows][K] (E4M3 activations), boxes of 128 x box_rows.
bool tmap_u8(CUtensorMap* tm, const void* base, int K, int rows, int box_rows);

}  // namespace moe
