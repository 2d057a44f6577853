// gemm_tc_persist.cu - persistent, stream-K W4A8 fc1 for decode-size calls.
//
// Decode calls touch few experts (M = 16, top-6: ~66 experts x 5 weight blocks = ~330 units of
// 56 K tiles each), so one CTA per unit leaves a tail wave that runs a fraction of the SMs.
// Here a fixed grid of G CTAs (every SM times its resident CTAs) takes the units in full waves
// (whole units, data-parallel) and splits the K tiles of the remaining units evenly over all
// CTAs (stream-K).  A CTA streams its piece(s) first and then its whole units through one TMA
// pipeline; each segment (a run of one unit's K tiles) accumulates in one of two TMEM buffers,
// so the epilogue warps drain segment j while the MMA fills segment j + 1:
//   - a segment that covers its whole unit goes straight to SwiGLU + MXFP8 requantisation;
//   - a piece is stored as fp32 partial sums (the tile's token columns only) in a slot of its
//     CTA, and the CTA that completes the unit (ticket counting K tiles, no waiting) adds the
//     unit's pieces in K order - the same order on every run - and runs SwiGLU +
//     requantisation.
// Block-scaled MMA, layouts and operand staging are those of fc1_tc_kernel (gemm_tc.cu).
//
// Warps (256 threads): 0 TMA producer (lane 0), 1 MMA issuer (lane 0), 2..3 the activation
// quantisers of small calls (each stage's MXFP8 operand from the bf16 rows; idle when the
// routing launch's quantised rows are loaded instead), 4..7 epilogue (TMEM lane quadrant =
// warp % 4).
#include <algorithm>
#include <cstring>

#include "moe_common.cuh"
#include "tc_ptx.cuh"
#include "tc_tile.cuh"
#include "tc_sched.cuh"

namespace moe {

using namespace tc;

constexpr int kStreamThreads = 256;

template <int BN>
struct StreamCfg {
  static constexpr int kB = BN * 128;
  static constexpr int kStage = (2 * kTileBytesA + kB + 3 * 512 + 1023) / 1024 * 1024;
  static constexpr int kStages = 3;                      // two CTAs per SM
  static constexpr int kSfStage = 0;                     // scale atoms arrive by bulk copy
  static constexpr int kSmem = kStages * kStage + kSfStage + 1024;
  static constexpr int kAcc = 2 * BN;                    // one accumulator buffer: up | gate
  static constexpr int kCols = 2 * kAcc + 12 * kStages;
  static constexpr int kAlloc = kCols <= 64 ? 64 : kCols <= 128 ? 128 : 256;
  static constexpr int kPartFloats = 2 * BN * 128;       // one partial slot
};

struct StreamFc1Params {
  CUtensorMap tm_w13;        // full 128-row weight tiles
  CUtensorMap tm_w13_tail;   // partial last row tile
  CUtensorMap tm_x;          // E4M3 activations [Sm][H], boxes 128 x BN
  const uint8_t* sf13;
  const uint8_t* xs16;       // activation-scale atom rows [H/128][r16][16]
  const int4* tiles;
  const int32_t* ctrl;
  int32_t* err;
  uint8_t* hq;
  uint8_t* hs;
  uint8_t* hs16;             // h scales in the atom layout [Ip/128][r16][16]
  int r16;
  float* part;               // [2 * G][2][BN][128] partial accumulators
  int32_t* tickets;          // [units] K tiles completed
  int H, I, Ip, RT, KT, Sm, RTf, rem;
  float limit, alpha, beta;
  // small calls (Mk <= kPreRouteSlots): the router ids, to route in shared memory ahead of the
  // routing launch (null: wait for its tables)
  const int32_t* ids;
  int Mk, E, max_tiles, ep_first;
  // the bf16 hidden states, quantised to MXFP8 here stage by stage into the MMA's activation
  // operand (null: TMA loads of the routing launch's quantised rows); row block 0's codes are
  // also stored to xq / xs
  const __nv_bfloat16* x;
  int topk;
  uint8_t* xq;
  uint8_t* xs;
};

// A stage whose weights were requested before the routing was known for certain must be of the
// expert the stage turned out to need.
static __device__ __forceinline__ bool pre_e_check(int i, int pre, const int* pre_e, int e) {
  return i < pre && pre_e[i] != e;
}

template <int BN>
__global__ void __launch_bounds__(kStreamThreads)
fc1_stream_kernel(const __grid_constant__ StreamFc1Params p) {
  using Cfg = StreamCfg<BN>;
  constexpr int S = Cfg::kStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[S], empty[S], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_last, s_fail, s_npieces;
  __shared__ int s_pieces[kStreamMaxPieces];
  __shared__ PreRouteInfo s_info;
  __shared__ int s_tok[2][BN];      // each quantising warp's copy of its tile's token list
  // activations quantised here (the shared-memory routing knows each tile's tokens)
  const bool fused = p.x != nullptr && p.ids != nullptr;
  tmem_alloc_first(&s_tmem, Cfg::kAlloc);

  // Small calls route in shared memory (scratch in the last stage, before any copy lands
  // there), so the weights of the first stages are requested while the routing launch still
  // runs; larger calls wait for its tables.
  int* scratch = reinterpret_cast<int*>(smem + (S - 1) * Cfg::kStage);
  int n_tiles;
  if (p.ids != nullptr) {
    n_tiles = min(pre_route_tiles<kStreamThreads>(p.ids, p.Mk, p.E, p.ep_first, BN, scratch,
                                                  fused ? &s_info : nullptr),
                  p.max_tiles);
  } else {
    pdl_wait_prev();     // routing tables complete
    n_tiles = p.ctrl[1];
  }
  StreamWork wk;
  wk.init(n_tiles * p.RT, p.KT, gridDim.x, blockIdx.x);
  if (wk.nsteps <= 0) {
    tmem_exit_early(&s_tmem, Cfg::kAlloc);
    pdl_wait_prev();
    return;
  }
  // experts of the first stages' units (read before the producer's copies reach the scratch)
  int pre_e[S];
  int pre = 0;
  if (p.ids != nullptr && warp == 0 && lane == 0) {
    auto sg = wk.segs();
    int u, k0, len;
    while (pre < S && sg.next(u, k0, len)) {
      const int tile = u / p.RT;
      const int ex = tile < kPreRouteTiles ? scratch[p.E + tile] : -1;
      for (int kt = k0; kt < k0 + len && pre < S; ++kt) pre_e[pre++] = ex;
    }
  }

  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      // fused: the producer's arrival (weight bytes) and one per quantising warp
      mbar_init(&full[s], fused ? 3 : 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain, 1);
    s_fail = 0;
    fence_barrier_init();
  }
  if (tid == 64) prefetch_tmap(&p.tm_w13);
  if (tid == 96) prefetch_tmap(&p.tm_x);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;
  int issued = 0;                                   // stages filled by the TMA producer
  auto stage = [&](int s) { return smem + s * Cfg::kStage; };

  // the weight part of a stage: both halves' codes and scale atoms of K tile kt, row block fb
  // of expert ex; returns its byte count
  auto load_a = [&](uint8_t* st, int ex, int fb, int kt, uint64_t* bar, uint64_t pol,
                    bool expect_only) -> uint32_t {
    const uint32_t bytes = (fb < p.RTf ? 2 * kTxBytesA : 2 * p.rem * 64) + 2 * 512;
    if (expect_only) mbar_expect_tx(bar, bytes);
    if (fb < p.RTf) {
      tma_load_3d_hint(st, &p.tm_w13, 0, 0, ((2 * ex) * p.RTf + fb) * p.KT + kt, bar, pol);
      tma_load_3d_hint(st + kTileBytesA, &p.tm_w13, 0, 0,
                       ((2 * ex + 1) * p.RTf + fb) * p.KT + kt, bar, pol);
    } else {
      tma_load_3d_hint(st, &p.tm_w13_tail, 0, 0, (2 * ex) * p.KT + kt, bar, pol);
      tma_load_3d_hint(st + kTileBytesA, &p.tm_w13_tail, 0, 0, (2 * ex + 1) * p.KT + kt, bar,
                       pol);
    }
    const size_t a_up = ((size_t)(2 * ex) * p.RT + fb) * p.KT + kt;
    const size_t a_gt = ((size_t)(2 * ex + 1) * p.RT + fb) * p.KT + kt;
    bulk_load(st + 2 * kTileBytesA + Cfg::kB, p.sf13 + a_up * 512, 512, bar);
    bulk_load(st + 2 * kTileBytesA + Cfg::kB + 512, p.sf13 + a_gt * 512, 512, bar);
    return bytes;
  };
  if (warp == 0 && lane == 0 && pre > 0) {
    // weights of the first stages, before the routing launch completes; the stage barriers
    // expect their bytes now and are arrived on once the activation part is issued too
    const uint64_t pol = l2_evict_first_policy();
    auto sg = wk.segs();
    int u, k0, len, i = 0;
    while (i < pre && sg.next(u, k0, len)) {
      const int fb = u % p.RT;
      for (int kt = k0; kt < k0 + len && i < pre; ++kt, ++i) {
        if (pre_e[i] < 0) {   // tile beyond the shared-memory table: no early request
          pre = i;
          break;
        }
        if (fused) {
          // the weights are all the producer loads: it arrives now
          const uint32_t ab = (fb < p.RTf ? 2 * kTxBytesA : 2 * p.rem * 64) + 2 * 512;
          mbar_arrive_expect_tx(&full[i], ab);
          load_a(stage(i), pre_e[i], fb, kt, &full[i], pol, false);
        } else {
          load_a(stage(i), pre_e[i], fb, kt, &full[i], pol, true);
        }
      }
    }
  }
  if (!fused) {
    pdl_wait_prev();   // routing tables and activations complete
    // fc2 reads the routing tables before its own wait: it may launch only once every CTA of
    // this kernel has seen them complete
    pdl_launch_next();
    // the shared-memory routing planned the same tiles as the routing launch (see checked_tile)
    if (tid == 0 && n_tiles != min(__ldcg(p.ctrl + 1), p.max_tiles))
      set_error(p.err, kErrRouteBounds);
  }
  // a tile's (expert, first slot position, tokens): the shared-memory routing when fused (the
  // routing launch's tables are read only by the epilogue warps, after waiting for it)
  auto tile_of = [&](int tile) -> int4 {
    if (fused)
      return make_int4(s_info.te[tile] & 0xFFFF, s_info.tp[tile] & 0xFFFF, s_info.te[tile] >> 16,
                       0);
    return checked_tile(p.tiles, p.ctrl, tile, p.E, p.Sm, BN, p.err);
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
      int i = 0, cur_tile = -1, e = 0, p0 = 0;
      auto sg = wk.segs();
      int u, k0, len;
      while (ok && sg.next(u, k0, len)) {
        const int tile = u / p.RT, fb = u - tile * p.RT;
        if (tile != cur_tile) {
          cur_tile = tile;
          const int4 td = tile_of(tile);
          e = td.x;
          p0 = td.y;
        }
        for (int kt = k0; kt < k0 + len && ok; ++kt, ++i) {
          const int s = i % S;
          if (i >= S) ok = mbar_wait(&empty[s], ((i / S) - 1) & 1, p.err);
          if (!ok) break;
          uint8_t* st = stage(s);
          if (fused) {
            if (pre_e_check(i, pre, pre_e, e)) set_error(p.err, kErrRouteBounds);
            if (i >= pre) {
              const uint32_t ab = (fb < p.RTf ? 2 * kTxBytesA : 2 * p.rem * 64) + 2 * 512;
              mbar_arrive_expect_tx(&full[s], ab);
              load_a(st, e, fb, kt, &full[s], pol, false);
            }
            continue;
          }
          if (i < pre) {
            if (pre_e[i] != e) set_error(p.err, kErrRouteBounds);
            mbar_arrive_expect_tx(&full[s], Cfg::kB + BN * 16);
          } else {
            const uint32_t ab =
                (fb < p.RTf ? 2 * kTxBytesA : 2 * p.rem * 64) + 2 * 512;
            mbar_arrive_expect_tx(&full[s], ab + Cfg::kB + BN * 16);
            load_a(st, e, fb, kt, &full[s], pol, false);
          }
          tma_load_2d(st + 2 * kTileBytesA, &p.tm_x, kt * 128, p0, &full[s]);
          // activation-scale atom: the tile's prepared atom rows, one bulk copy
          bulk_load(st + 2 * kTileBytesA + Cfg::kB + 1024,
                    p.xs16 + ((size_t)kt * p.r16 + p0) * 16, BN * 16, &full[s]);
        }
      }
      issued = i;
    }
  } else if (fused && (warp == 2 || warp == 3)) {
    // warps 2..3: each stage's activation operand, quantised from the bf16 rows of the tile's
    // tokens (units of row block 0 also keep a copy of the codes in xq / xs)
    const ActQuant<BN> aq{p.x, p.H, tid - 64};
    int i = 0, cur_tile = -1, n = 0, p0 = 0;
    auto sg = wk.segs();
    int u, k0, len;
    while (ok && sg.next(u, k0, len)) {
      const int tile = u / p.RT, fb = u - tile * p.RT;
      if (tile != cur_tile) {
        // the new tile's token list, each warp its own copy (no barrier between the two)
        pre_route_tile_tokens(s_info, tile, p.Mk, p.topk, BN, s_tok[warp - 2]);
        cur_tile = tile;
        n = s_info.te[tile] >> 16;
        p0 = s_info.tp[tile] & 0xFFFF;
      }
      ok = act_quant_run<BN, S>(aq, s_tok[warp - 2], n, k0, len, i, smem, Cfg::kStage,
                                2 * kTileBytesA, 2 * kTileBytesA + Cfg::kB + 1024, full, empty,
                                fb == 0 ? p.xq : nullptr, p.xs, p0, p.err);
      i += len;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int i = 0, j = 0;
      auto sg = wk.segs();
      int u, k0, len;
      while (ok && sg.next(u, k0, len)) {
        const int b = j & 1;
        if (j >= 2) ok = mbar_wait(&acc_empty[b], ((j >> 1) - 1) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_up = tmem + b * Cfg::kAcc, d_gt = d_up + BN;
        for (int kt = 0; kt < len && ok; ++kt, ++i) {
          const int s = i % S;
          ok = mbar_wait(&full[s], (i / S) & 1, p.err);
          if (!ok) break;
          tc_fence_after();
          uint8_t* st = stage(s);
          const uint32_t sf = tmem + 2 * Cfg::kAcc + 12 * s;
          tc_cp_sf(sf + 0, desc_sf(st + 2 * kTileBytesA + Cfg::kB));
          tc_cp_sf(sf + 4, desc_sf(st + 2 * kTileBytesA + Cfg::kB + 512));
          tc_cp_sf(sf + 8, desc_sf(st + 2 * kTileBytesA + Cfg::kB + 1024));
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint32_t idesc = idesc_mxf8f6f4(kFmtE2M1, kFmtE4M3, BN, kb);
            const uint64_t bdesc = desc_sw128(st + 2 * kTileBytesA + 32 * kb);
            const uint32_t acc = (kt > 0 || kb > 0) ? 1u : 0u;
            mma_mxf8f6f4(d_up, desc_sw128(st + 32 * kb), bdesc, idesc, sf + 0, sf + 8, acc);
            mma_mxf8f6f4(d_gt, desc_sw128(st + kTileBytesA + 32 * kb), bdesc, idesc, sf + 4,
                         sf + 8, acc);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[b]);
        ++j;
      }
    }
  } else if (warp >= 4) {
    if (fused) {
      pdl_wait_prev();   // routing launch complete: its tables and cleared tickets
      pdl_launch_next();
      if (tid == 128 && n_tiles != min(__ldcg(p.ctrl + 1), p.max_tiles))
        set_error(p.err, kErrRouteBounds);
    }
    const int quad = warp & 3;
    const int row = quad * 32 + lane;                         // weight row within the block
    int j = 0;
    auto sg = wk.segs();
    int u, k0, len;
    for (; sg.next(u, k0, len); ++j) {
      const int k1 = k0 + len;
      const int tile = u / p.RT, fb = u - tile * p.RT;
      const int4 td = tile_of(tile);
      if (fused && tid == 128) {
        // the routing launch's record of the tile is the one routed here
        const int4 rt = checked_tile(p.tiles, p.ctrl, tile, p.E, p.Sm, BN, p.err);
        if (rt.x != td.x || rt.y != td.y || rt.z != td.z) set_error(p.err, kErrRouteBounds);
      }
      const int p0 = td.y, n = td.z;
      const int f = fb * 128 + row;
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[b], (j >> 1) & 1, p.err));
      tc_fence_after();
      __syncwarp();
      const uint32_t trow = tmem + b * Cfg::kAcc + ((uint32_t)(quad * 32) << 16);
      const bool whole = k0 == 0 && k1 == p.KT;
      float* part = whole ? nullptr
                          : p.part + (size_t)wk.own_slot(u) * Cfg::kPartFloats;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float up[16], gt[16];
        tmem_ld16(trow + c0, up);
        tmem_ld16(trow + BN + c0, gt);
        if (!ok || c0 >= n) continue;
        if (whole) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (c0 + jj < n) {
              const float h = f < p.I ? swiglu(gt[jj], up[jj], p.limit, p.alpha, p.beta) : 0.f;
              const size_t r = (size_t)(p0 + c0 + jj);
              requant_store(h, lane, r, p.Ip, f, p.hq, p.hs, p.hs16, p.r16);
            }
          }
        } else {
          // only the tile's n token columns are kept
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (c0 + jj < n) {
              part[(c0 + jj) * 128 + row] = up[jj];
              part[(BN + c0 + jj) * 128 + row] = gt[jj];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      if (!whole) {
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 4 && lane == 0) {
          const int t = atomicAdd(&p.tickets[u], len);
          s_last = (t + len == p.KT);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (s_last) {
          __threadfence();
          // the unit's pieces in K order (CTAs with empty ranges hold none), listed once by
          // one thread; the barrier is taken by all four warps, whatever their verdicts
          if (warp == 4 && lane == 0) s_npieces = wk.unit_pieces(u, s_pieces);
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (ok) reduce_pieces(
              s_npieces, n, (size_t)128, (size_t)BN * 128,
              [&](int qq) -> const float* {
                return p.part + (size_t)s_pieces[qq] * Cfg::kPartFloats + row;
              },
              [&](int cc, float up, float gt) {
                const float h = f < p.I ? swiglu(gt, up, p.limit, p.alpha, p.beta) : 0.f;
                const size_t r = (size_t)(p0 + cc);
                requant_store(h, lane, r, p.Ip, f, p.hq, p.hs, p.hs16, p.r16);
              });
        }
      }
    }
  }
  if (!ok) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  if (s_fail) {
    // a wait gave up: let this CTA's copies and MMAs land before its memory is released
    if (warp == 0 && lane == 0) drain_stage_loads<S>(full, issued, p.err);
    if (warp == 1 && lane == 0) {
      tc_commit(&drain);
      mbar_wait(&drain, 0, p.err);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc);
}

// ------------------------------------------------------------------------------------ fc2
// Persistent fc2: units are (tile, 128-row block of H) pairs of KT = Ip / 128 K tiles each.  In
// tile-major order the G CTAs take equal contiguous ranges of the flat (unit, K tile) steps when
// the combine is atomic (a unit cut between two CTAs adds both partial products) and of whole
// units when it is deterministic; an atomic call whose fp32 combine buffer is large takes whole
// units round robin in row-block-major order instead (Fc2Units).  The accumulators alternate between two TMEM buffers, so the combine
// of one segment overlaps the loads and MMAs of the next instead of ending the CTA.  The combine is
// that of fc2_tc_kernel (fp32 atomics into the token's row, or the weighted slot row of the
// route buffer); a separate finalize launch writes the output.

template <int BN>
struct PersistFc2Cfg {
  static constexpr int kB = BN * 128;
  static constexpr int kStage = (kTileBytesA + kB + 512 + BN * 16 + 1023) / 1024 * 1024;
  static constexpr int kStages = 3;                      // three CTAs per SM
  static constexpr int kSmem = kStages * kStage + 1024;
  static constexpr int kChunks = NChunks<BN>::kCount;
  static constexpr int kSf = 4 + 4 * kChunks;           // SFA, SFB chunks
  static constexpr int kCols = 2 * BN + kSf * kStages;  // two accumulators, scale ring
  static constexpr int kAlloc = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : 256;
  static_assert(kCols <= 256, "fc2 tensor memory");
};

struct PersistFc2Params {
  CUtensorMap tm_w2;         // packed FP4 tiles [E*RB*KT][128][128], box 128 x 128 x 1
  CUtensorMap tm_h;          // E4M3 [Sm][Ip], boxes 128 x BN
  const uint8_t* sf2;        // weight scale atoms [E][RB][KT][512]
  const uint8_t* hs16;       // h scale atom rows [Ip/128][r16][16]
  const int4* tiles;
  const int32_t* ctrl;
  int32_t* err;
  const int32_t* perm;
  const float* topk_w;
  float* acc;                // [M][H] atomic mode
  float* rbuf;               // [M*k][H] deterministic mode
  int H, KT, RB, Sm, topk, deterministic, r16;
  int pair;                  // I % 128 == 64: the last K tile's codes are paired (fp4_w2_tile)
  int rr;                    // whole units round robin in row-block-major order (Fc2Units)
};

template <int BN>
__global__ void __launch_bounds__(kStreamThreads)
fc2_persist_kernel(const __grid_constant__ PersistFc2Params p) {
  using Cfg = PersistFc2Cfg<BN>;
  constexpr int S = Cfg::kStages;
  pdl_launch_next();
  __shared__ __align__(8) uint64_t full[S], empty[S], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  // per epilogue warp (no barrier between them): the flat slot index of each column of its
  // current tile and that slot's router weight
  __shared__ int s_f[4][BN];
  __shared__ float s_w[4][BN];
  // per epilogue warp: 16 token columns x its 32 output features, read back transposed
  __shared__ __align__(16) float s_y[4][16][32];
  tmem_alloc_first(&s_tmem, Cfg::kAlloc);
  // The routing tables were complete before fc1 let this kernel launch (fc1 waits for the
  // routing launch first): the unit range and the weights of the first stages are read before
  // waiting for fc1's output (L2 reads: nothing of them is in this SM's L1).
  const int G = gridDim.x, c = blockIdx.x;
  const int n_tiles = __ldcg(&p.ctrl[1]);
  const int units = n_tiles * p.RB;
  // flat mode: this CTA's range [x0, x1) of the flat steps x = unit * KT + K tile, split evenly
  // when the combine is atomic (a unit cut between two CTAs adds both partial products to the
  // same outputs), whole units when it is deterministic (each slot's output is written once);
  // round-robin mode (large atomic calls): whole units c, c + G, ...
  int x0, x1;
  if (p.rr) {
    x0 = 0;
    x1 = c < units ? ((units - 1 - c) / G + 1) * p.KT : 0;   // this CTA's step count
  } else if (p.deterministic) {
    x0 = (int)((long long)c * units / G) * p.KT;
    x1 = (int)((long long)(c + 1) * units / G) * p.KT;
  } else {
    const long long T = (long long)units * p.KT;
    x0 = (int)(c * T / G);
    x1 = (int)((c + 1) * T / G);
  }
  const Fc2Units work{p.KT, p.RB, n_tiles, units, G, p.rr, x0, x1, c};
  if (x0 >= x1) {
    tmem_exit_early(&s_tmem, Cfg::kAlloc);
    pdl_wait_prev();
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain, 1);
    s_fail = 0;
    fence_barrier_init();
  }
  if (tid == 64) prefetch_tmap(&p.tm_w2);
  if (tid == 96) prefetch_tmap(&p.tm_h);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;
  int issued = 0;                                   // stages filled by the TMA producer
  auto stage = [&](int s) { return smem + s * Cfg::kStage; };
  // stage layout: A | B | SFA | SFB

  if (warp == 0 && lane == 0) {
    const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
    // weights of the first stages, before fc1 completes: the stage's barrier expects their
    // bytes now and is arrived on once the activation part is issued too
    int pre = 0;
    {
      Fc2Units pw = work;
      int tile, rb, k0, len;
      while (pre < S && pw.next(tile, rb, k0, len)) {
        const int e = __ldcg(reinterpret_cast<const int*>(p.tiles + tile));
        for (int kt = k0; kt < k0 + len && pre < S; ++kt, ++pre) {
          const size_t a = ((size_t)e * p.RB + rb) * p.KT + kt;
          mbar_expect_tx(&full[pre], kTxBytesA + 512);
          tma_load_3d_hint(stage(pre), &p.tm_w2, 0, 0,
                           fp4_w2_tile(e, rb, kt, p.RB, p.KT, p.pair), &full[pre], pol);
          bulk_load(stage(pre) + kTileBytesA + Cfg::kB, p.sf2 + a * 512, 512, &full[pre]);
        }
      }
    }
    pdl_wait_prev();     // fc1 complete, h visible
    int i = 0, cur_tile = -1, e = 0, p0 = 0;
    TileLoad<BN> tl(BN);
    Fc2Units sg = work;
    int tile, rb, k0, len;
    while (ok && sg.next(tile, rb, k0, len)) {
      if (tile != cur_tile) {
        cur_tile = tile;
        const int4 td = p.tiles[tile];
        e = td.x;
        p0 = td.y;
        tl = TileLoad<BN>(td.z);
      }
      for (int kt = k0; kt < k0 + len && ok; ++kt, ++i) {
        const int s = i % S;
        if (i >= S) ok = mbar_wait(&empty[s], ((i / S) - 1) & 1, p.err);
        if (!ok) break;
        uint8_t* st = stage(s);
        if (i < pre) {
          mbar_arrive_expect_tx(&full[s], tl.b_bytes + tl.sf_bytes);
        } else {
          const size_t a = ((size_t)e * p.RB + rb) * p.KT + kt;
          mbar_arrive_expect_tx(&full[s], kTxBytesA + tl.b_bytes + 512 + tl.sf_bytes);
          tma_load_3d_hint(st, &p.tm_w2, 0, 0, fp4_w2_tile(e, rb, kt, p.RB, p.KT, p.pair),
                           &full[s], pol);
          bulk_load(st + kTileBytesA + Cfg::kB, p.sf2 + a * 512, 512, &full[s]);
        }
        tl.load_b(st + kTileBytesA, &p.tm_h, kt * 128, p0, &full[s]);
        bulk_load(st + kTileBytesA + Cfg::kB + 512, p.hs16 + ((size_t)kt * p.r16 + p0) * 16,
                  tl.sf_bytes, &full[s]);
      }
    }
    issued = i;
  } else {
    pdl_wait_prev();     // previous kernels of the call complete
  }
  if (warp == 1) {
    if (lane == 0) {
      int i = 0, j = 0, cur_tile = -1;
      TileLoad<BN> tl(BN);
      Fc2Units sg = work;
      int tile, rb, k0, len;
      for (; ok && sg.next(tile, rb, k0, len); ++j) {
        if (tile != cur_tile) {
          cur_tile = tile;
          tl = TileLoad<BN>(p.tiles[tile].z);
        }
        const int b = j & 1;
        if (j >= 2) ok = mbar_wait(&acc_empty[b], ((j >> 1) - 1) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + b * BN;
        for (int kt = k0; kt < k0 + len && ok; ++kt, ++i) {
          const int s = i % S;
          ok = mbar_wait(&full[s], (i / S) & 1, p.err);
          if (!ok) break;
          tc_fence_after();
          uint8_t* st = stage(s);
          const uint32_t sf = tmem + 2 * BN + Cfg::kSf * s;
          tc_cp_sf(sf + 0, desc_sf(st + kTileBytesA + Cfg::kB));
#pragma unroll
          for (int jc = 0; jc < Cfg::kChunks; ++jc)
            if (jc < tl.nch)
              tc_cp_sf(sf + 4 + 4 * jc, desc_sf(st + kTileBytesA + Cfg::kB + 512 + 512 * jc));
          // a paired tail tile: two K steps, at columns 64.. of the tile for an odd row block
          const bool tail = p.pair && kt == p.KT - 1;
          const int a_off = (tail && (rb & 1)) ? 64 : 0;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            if (tail && kb >= 2) break;
            const uint32_t idesc = idesc_mxf8f6f4(kFmtE2M1, kFmtE4M3, NChunks<BN>::kWidth, kb);
#pragma unroll
            for (int jc = 0; jc < Cfg::kChunks; ++jc)
              if (jc < tl.nch)
                mma_mxf8f6f4(d + 32 * jc, desc_sw128(st + a_off + 32 * kb),
                           desc_sw128(st + kTileBytesA + 4096 * jc + 32 * kb), idesc, sf + 0,
                           sf + 4 + 4 * jc, (kt > k0 || kb > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[b]);
      }
    }
  } else if (warp >= 4) {
    const int quad = warp & 3;
    int j = 0, cur_tile = -1, n = 0;
    Fc2Units sg = work;
    int tile, rb, k0, len;
    for (; sg.next(tile, rb, k0, len); ++j) {
      if (tile != cur_tile) {
        // the combine's slot indices and router weights of the new tile, loaded by each warp
        // for itself before its accumulators are waited for (consecutive units of a flat
        // range share their tile; round-robin units change it every time)
        constexpr int NQ = (BN + 31) / 32;
        const int4 td = p.tiles[tile];
        n = td.z;
        int f[NQ];
        float wt[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) f[q] = lane + 32 * q < n ? p.perm[td.y + lane + 32 * q] : 0;
#pragma unroll
        for (int q = 0; q < NQ; ++q) wt[q] = lane + 32 * q < n ? p.topk_w[f[q]] : 0.f;
        __syncwarp();
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (lane + 32 * q < n) {
            s_f[quad][lane + 32 * q] = f[q];
            s_w[quad][lane + 32 * q] = wt[q];
          }
        __syncwarp();
        cur_tile = tile;
      }
      // after the transpose a lane holds four consecutive output features of one token
      const int h4 = rb * 128 + quad * 32 + 4 * (lane & 7);
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[b], (j >> 1) & 1, p.err));
      tc_fence_after();
      __syncwarp();
      const uint32_t trow = tmem + b * BN + ((uint32_t)(quad * 32) << 16);
      float(*sy)[32] = s_y[quad];
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float y[16];
        tmem_ld16(trow + c0, y);
        if (!ok || c0 >= n) continue;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) sy[jj][lane] = y[jj];
        __syncwarp();
        // one 16-byte combine per (token, 4 features): a quarter of the scalar atomics
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int cc = 4 * r + (lane >> 3);
          if (c0 + cc < n) {
            const float4 v = *reinterpret_cast<const float4*>(&sy[cc][4 * (lane & 7)]);
            const int f = s_f[quad][c0 + cc];
            const float wt = s_w[quad][c0 + cc];
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
  if (s_fail) {
    // a wait gave up: let this CTA's copies and MMAs land before its memory is released
    if (warp == 0 && lane == 0) drain_stage_loads<S>(full, issued, p.err);
    if (warp == 1 && lane == 0) {
      tc_commit(&drain);
      mbar_wait(&drain, 0, p.err);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc);
}

// ---------------------------------------------------------------------------------- host side

// The stream-K fc1 serves every call of 16-token tiles (decode sizes).  Its CTAs split the
// units the routing actually produced evenly over all CTA slots, where the one-unit-per-CTA
// kernel sizes its grid for the most tiles the call could have (one per routed slot), leaves
// the CTAs of absent tiles idle and gives each remaining CTA a whole unit: measured over the
// decode ladder M = 1..16 (E 384, H 7168, I 576, top-6), 725 us against 864 us per pass, and
// faster at every M.
bool fc1_stream_preferred(int bn, int units) {
  (void)units;
  return bn == 16;
}
// Scratch of its partial slots: 2 per CTA, each [2][16][128] fp32.
size_t fc1_stream_part_bytes() { return (size_t)2 * kStreamMaxCtas * 2 * 16 * 128 * 4; }

cudaError_t launch_fc1_stream(const DevWeights& w, const RunPtrs& r, const PlanDims& d, int bn,
                              int M, float* part, int32_t* tickets, const int32_t* ids,
                              int max_tiles, const void* x, cudaStream_t st) {
  if (bn != 16) return cudaErrorInvalidValue;
  StreamFc1Params p;
  memset(&p, 0, sizeof(p));
  p.RTf = d.I / 128;
  p.rem = d.I % 128;
  const long long kt = d.H / 128;
  const int Sm = M * d.topk;
  if (!tmap_fp4(&p.tm_w13, w.w13, 128, 2LL * d.E * p.RTf * kt) ||
      !tmap_fp4(&p.tm_w13_tail, w.w13 + (size_t)2 * d.E * p.RTf * kt * 8192, p.rem,
                2LL * d.E * kt) ||
      !tmap_u8(&p.tm_x, r.xq, d.H, Sm, bn))
    return cudaErrorInvalidValue;
  p.sf13 = w.s13; p.xs16 = r.xs16; p.hs16 = r.hs16; p.r16 = r.r16;
  p.tiles = r.tiles; p.ctrl = r.ctrl; p.err = r.ctrl;
  p.hq = r.hq; p.hs = r.hs; p.part = part; p.tickets = tickets;
  p.H = d.H; p.I = d.I; p.Ip = d.Ip; p.RT = cdiv(d.I, 128); p.KT = d.H / 128; p.Sm = Sm;
  p.limit = d.limit; p.alpha = d.alpha; p.beta = d.beta;
  p.ids = (ids != nullptr && Sm <= kPreRouteSlots) ? ids : nullptr;
  p.Mk = Sm; p.E = d.E; p.max_tiles = max_tiles; p.ep_first = d.ep_first;
  p.x = p.ids != nullptr ? static_cast<const __nv_bfloat16*>(x) : nullptr;
  p.topk = d.topk;
  p.xq = d.keep_act ? r.xq : nullptr;
  p.xs = r.xs;
  static const int G = persistent_grid(fc1_stream_kernel<16>, StreamCfg<16>::kSmem,
                                       StreamCfg<16>::kAlloc, 2, kStreamMaxCtas);
  return launch_kernel(fc1_stream_kernel<16>, dim3(G), dim3(kStreamThreads), StreamCfg<16>::kSmem,
                       st, true, p);
}

// The persistent fc2 serves every W4A8 tile width when the unit-per-CTA fc2 would run more
// than 5 waves of one unit per SM (measured: 39 -> 36 us at 3,750 units, 2-3 % faster calls at
// 1,000-2,000 units; slower than the unit-per-CTA kernel below ~2.5 waves).
bool fc2_persist_preferred(int bn, int units) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      sms = 152;
    }
  }
  return (bn == 16 || bn == 32 || bn == 64 || bn == 96) && units > 5 * sms;
}

template <int BN>
static cudaError_t launch_fc2_persist_bn(const PersistFc2Params& p, cudaStream_t st) {
  using Cfg = PersistFc2Cfg<BN>;
  static const int G = persistent_grid(fc2_persist_kernel<BN>, Cfg::kSmem, Cfg::kAlloc, 4,
                                       1 << 20);
  return launch_kernel(fc2_persist_kernel<BN>, dim3(G), dim3(kStreamThreads), Cfg::kSmem, st,
                       true, p);
}

constexpr size_t kFc2RoundRobinAccBytes = 32u << 20;

cudaError_t launch_fc2_persist(const DevWeights& w, const RunPtrs& r, const PlanDims& d, int bn,
                               int M, const float* topk_w, cudaStream_t st) {
  PersistFc2Params p;
  memset(&p, 0, sizeof(p));
  const int Sm = M * d.topk;
  p.RB = d.H / 128;
  p.KT = d.Ip / 128;
  p.pair = (d.I & 127) == 64 ? 1 : 0;
  if (!tmap_fp4(&p.tm_w2, w.w2, 128, (long long)d.E * p.RB * p.KT) ||
      !tmap_u8(&p.tm_h, r.hq, d.Ip, Sm, act_box_rows(bn)))
    return cudaErrorInvalidValue;
  p.sf2 = w.s2; p.hs16 = r.hs16; p.r16 = r.r16;
  p.tiles = r.tiles; p.ctrl = r.ctrl; p.err = r.ctrl;
  p.perm = r.perm; p.topk_w = topk_w; p.acc = r.acc; p.rbuf = r.rbuf;
  p.H = d.H; p.Sm = Sm; p.topk = d.topk; p.deterministic = d.deterministic;
  // round robin in row-block-major order once the fp32 combine buffer is a large part of L2
  // (measured at M = 4096, H = 7168: the 117 MB buffer's lines were evicted and fetched again
  // about three times over in tile-major order)
  p.rr = (!d.deterministic && (size_t)M * d.H * sizeof(float) > kFc2RoundRobinAccBytes) ? 1 : 0;
  if (bn == 16) return launch_fc2_persist_bn<16>(p, st);
  if (bn == 32) return launch_fc2_persist_bn<32>(p, st);
  if (bn == 64) return launch_fc2_persist_bn<64>(p, st);
  if (bn == 96) return launch_fc2_persist_bn<96>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace moe
