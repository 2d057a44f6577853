// gemm_tc.cu - W4A8 grouped GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// fc1 and fc2 of the routed MoE (moe_b12x_next.py module docstring: MXFP4 weights, in-kernel
// MXFP8 activations) as block-scaled MMAs of kind::mxf8f6f4: A = weights (E2M1, UE8M0 scale per
// 32 along K), B = activations (E4M3, UE8M0 per 32), fp32 accumulators in TMEM.
//
// Orientation ("swap AB"): the 128 rows of an MMA are weight rows (output features) and the N
// columns are the tile's tokens (slot positions of one expert), so decode calls with a handful
// of tokens per expert still use full 128-row MMAs and stream each touched weight byte once.
//
// Per CTA: one tile (<= BN slot positions of one expert) x one 128-row block of weights x one
// K range.  Warp roles in the main loop: warp 0 lane 0 issues TMA (weights and activations)
// and bulk copies (weight scale atoms); warp 2 writes the activations' scale atoms; warp 1
// lane 0 issues tcgen05.cp (scales -> TMEM) and tcgen05.mma.  All four warps run the
// epilogue from TMEM (lane = weight row, column = token).
//
// fc1 epilogue: h = SwiGLU(gate, up) (clamped), requantised to MXFP8 per 32 intermediate
// columns (the 32 rows of a warp), written as the fc2 activation operand.  With split K each
// split stores its partial sums in its own slice of an fp32 buffer, and the last CTA of the unit
// (atomic ticket, no waiting) adds the slices in split order - the same sum on every run - and
// runs the epilogue.
// fc2 epilogue: the combine (fp32 atomics into the token's row, or the weighted slot row of
// the deterministic route buffer).
#include <algorithm>
#include <cstring>

#include "moe_common.cuh"
#include "tc_ptx.cuh"
#include "tc_tile.cuh"

namespace moe {

using namespace tc;

template <int BN>
struct TcCfg {
  static constexpr int kB = BN * 128;                         // activation tile bytes
  // stage: weight tile(s) | activation tile | weight scale atom(s) | activation scale atom
  static constexpr int kStage1 = (2 * kTileBytesA + kB + 2 * 512 + BN * 16 + 1023) / 1024 * 1024;
  static constexpr int kStage2 = (kTileBytesA + kB + 512 + BN * 16 + 1023) / 1024 * 1024;
  // short rings, several CTAs per SM: a CTA keeps only a few stages in flight behind its one
  // producer thread, so more CTAs per SM stream more bytes at once (measured: fc2 at 2 stages
  // and 5 CTAs per SM runs 3x faster than at 6 stages and 1 CTA per SM)
  static constexpr int kStages1 = BN <= 16 ? 3 : 2;   // two CTAs per SM
  static constexpr int kStages2 = 2;
  static constexpr int kChunks = NChunks<BN>::kCount;
  static constexpr int kSf1 = 8 + 4 * kChunks;                // SFA_up, SFA_gate, SFB chunks
  static constexpr int kSf2 = 4 + 4 * kChunks;                // SFA, SFB chunks
  static constexpr int kCols1 = 2 * BN + kSf1 * kStages1;     // D_up, D_gate, scale ring
  static constexpr int kCols2 = BN + kSf2 * kStages2;
  static constexpr int pow2(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }
  static constexpr int kAlloc1 = pow2(kCols1);
  static constexpr int kAlloc2 = pow2(kCols2);
  static_assert(BN == 16 || BN == 32 || BN == 64 || BN == 96, "W4A8 token tile widths");
  // two CTAs per SM: tensor memory of at most 256 columns each
  static_assert(pow2(kCols1) <= 256, "fc1 tensor memory");
  static constexpr int kSmem1 = kStages1 * kStage1 + 1024;
  static constexpr int kSmem2 = kStages2 * kStage2 + 1024;
};

struct TcFc1Params {
  CUtensorMap tm_w13;        // packed FP4 full 128-row tiles [2E*RTf*KT][128][128], box 128x128x1
  CUtensorMap tm_w13_tail;   // partial last row tile [2E*KT][I%128][128], box 128 x (I%128) x 1
  CUtensorMap tm_x;          // E4M3 [Sm][H], box 128 x BN
  const uint8_t* sf13;       // weight scale atoms [E][2][RT][KT][512]
  const uint8_t* xs16;       // activation scales in the atom layout [H/128][r16][16]
  uint8_t* hs16;             // h scales in the atom layout [Ip/128][r16][16]
  int r16;
  const int4* tiles;
  const int32_t* ctrl;
  int32_t* err;
  uint8_t* hq;               // [Sm][Ip]
  uint8_t* hs;               // [Sm][Ip/32]
  float* gacc;               // [splits][Sm][2][Ip] split-K partial sums, one slice per split
  int32_t* tickets;          // [max_tiles][RT]
  int H, I, Ip, RT, KT, Sm, splits;
  int RTf, rem;              // full 128-row weight tiles per half, rows of the partial tile
  int fb_in_x;               // grid (RT, tiles, splits) instead of (tiles, RT, splits)
  float limit, alpha, beta;
  // small calls (Mk <= kPreRouteSlots): the router ids, to route in shared memory ahead of the
  // routing launch (null: wait for its tables)
  const int32_t* ids;
  int Mk, E, max_tiles, ep_first;
  // small calls at tile widths <= 32: the bf16 hidden states, which this kernel quantises to
  // MXFP8 itself, stage by stage, into the MMA's activation operand (null: TMA loads of the
  // routing launch's quantised rows); the codes of row block 0 are also stored to xq / xs
  const __nv_bfloat16* x;
  int topk;
  uint8_t* xq;               // [Sm][H] E4M3 copy of the quantised activations (row block 0)
  uint8_t* xs;               // [Sm][H/32] their E8M0 scales
  // test hook (0: off): the MMA issuer first waits this long on a barrier nothing arrives on;
  // the wait runs out, sets the timeout bit, and the CTA takes its failure path (no MMA, the
  // issued copies drained) - the bounded waits tested without a fault
  unsigned long long probe_ns;
};

struct TcFc2Params {
  CUtensorMap tm_w2;         // packed FP4 tiles [E*(H/128)*KT][128][128], box 128 x 128 x 1
  CUtensorMap tm_h;          // E4M3 [Sm][Ip], box 128 x BN
  const uint8_t* sf2;        // weight scale atoms [E][H/128][Ip/128][512]
  const uint8_t* hs16;       // h scales in the atom layout [Ip/128][r16][16]
  int r16;
  const int4* tiles;
  const int32_t* ctrl;
  int32_t* err;
  const int32_t* perm;
  const float* topk_w;
  float* acc;                // [M][H] atomic mode
  float* rbuf;               // [M*k][H] deterministic mode
  int H, Ip, KT, Sm, topk, deterministic;
  int pair;                  // I % 128 == 64: the last K tile's codes are paired (fp4_w2_tile)
};

template <int BN>
__global__ void __launch_bounds__(kTcThreads)
fc1_tc_kernel(const __grid_constant__ TcFc1Params p) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::kStages1;
  // the row blocks of a tile are adjacent in launch order (while the tiles fit the grid's y),
  // so the CTAs that read the same activation tile run together and share it through L2
  const int tile = p.fb_in_x ? blockIdx.y : blockIdx.x;
  const int fb = p.fb_in_x ? blockIdx.x : blockIdx.y, split = blockIdx.z;
  const int kt0 = split * p.KT / p.splits, kt1 = (split + 1) * p.KT / p.splits;
  const int nk = kt1 - kt0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[S], empty[S], done, never;
  __shared__ uint32_t s_tmem;
  __shared__ int s_last, s_fail;
  __shared__ PreRouteInfo s_info;
  __shared__ int s_tok[32];
  // activations quantised here (small calls, tiles of at most 32 tokens)
  const bool fused = BN <= 32 && p.x != nullptr && p.ids != nullptr;
  tmem_alloc_first(&s_tmem, Cfg::kAlloc1);

  // Small calls route in shared memory (scratch in the last stage, before any copy lands
  // there), so the weights of the first stages are requested while the routing launch still
  // runs; larger calls wait for its tables.
  int e_pre = -1, nt = 0, n_pre = 0, p0_pre = 0;
  if (p.ids != nullptr) {
    int* scratch = reinterpret_cast<int*>(smem + (S - 1) * Cfg::kStage1);
    nt = min(pre_route_tiles<kTcThreads>(p.ids, p.Mk, p.E, p.ep_first, BN, scratch,
                                         fused ? &s_info : nullptr),
             p.max_tiles);
    if (tile >= nt) {
      tmem_exit_early(&s_tmem, Cfg::kAlloc1);
      pdl_wait_prev();
      return;
    }
    if (tile < kPreRouteTiles) e_pre = scratch[p.E + tile];
    if (fused) {
      n_pre = s_info.te[tile] >> 16;
      p0_pre = s_info.tp[tile] & 0xFFFF;
      if (warp == 2) pre_route_tile_tokens(s_info, tile, p.Mk, p.topk, BN, s_tok);
    }
  } else {
    pdl_wait_prev();     // routing tables complete
    if (tile >= p.ctrl[1]) {
      tmem_exit_early(&s_tmem, Cfg::kAlloc1);
      return;
    }
  }

  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      // fused: the producer's arrival (weight bytes) and one per quantising warp
      mbar_init(&full[s], fused ? 3 : 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    mbar_init(&never, 1);      // the wait probe's barrier: no thread ever arrives on it
    s_fail = 0;
    fence_barrier_init();
  }
  if (tid == 64) prefetch_tmap(&p.tm_w13);
  if (tid == 96 && !fused) prefetch_tmap(&p.tm_x);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;
  int issued = 0;                                   // stages filled by the TMA producer
  auto stage = [&](int s) { return smem + s * Cfg::kStage1; };
  // stage layout: A_up | A_gate | B | SFA_up | SFA_gate | SFB
  const uint32_t a_bytes = fb < p.RTf ? 2 * kTxBytesA : 2 * p.rem * 64;
  // the weight part of a stage: both halves' codes and scale atoms of K tile kt of expert ex
  auto load_a = [&](uint8_t* st, int ex, int kt, uint64_t* bar, uint64_t pol) {
    if (fb < p.RTf) {
      tma_load_3d_hint(st, &p.tm_w13, 0, 0, ((2 * ex) * p.RTf + fb) * p.KT + kt, bar, pol);
      tma_load_3d_hint(st + kTileBytesA, &p.tm_w13, 0, 0,
                       ((2 * ex + 1) * p.RTf + fb) * p.KT + kt, bar, pol);
    } else {
      // partial row tile: rows >= I % 128 of the smem tile keep stale (finite) codes; their
      // accumulator rows are never read
      tma_load_3d_hint(st, &p.tm_w13_tail, 0, 0, (2 * ex) * p.KT + kt, bar, pol);
      tma_load_3d_hint(st + kTileBytesA, &p.tm_w13_tail, 0, 0, (2 * ex + 1) * p.KT + kt, bar,
                       pol);
    }
    const size_t a_up = ((size_t)(2 * ex) * p.RT + fb) * p.KT + kt;
    const size_t a_gt = ((size_t)(2 * ex + 1) * p.RT + fb) * p.KT + kt;
    bulk_load(st + 2 * kTileBytesA + Cfg::kB, p.sf13 + a_up * 512, 512, bar);
    bulk_load(st + 2 * kTileBytesA + Cfg::kB + 512, p.sf13 + a_gt * 512, 512, bar);
  };
  int pre = 0;                 // stages whose weights were requested before the wait
  if (warp == 0 && lane == 0 && e_pre >= 0) {
    const uint64_t pol = l2_evict_first_policy();
    pre = nk < S ? nk : S;
    for (int i = 0; i < pre; ++i) {
      // fused: the weights are all the producer loads, so it arrives now
      if (fused)
        mbar_arrive_expect_tx(&full[i], a_bytes + 2 * 512);
      else
        mbar_expect_tx(&full[i], a_bytes + 2 * 512);
      load_a(stage(i), e_pre, kt0 + i, &full[i], pol);
    }
  }
  int e, p0, n;
  if (fused) {
    // the tile as routed in shared memory; the routing launch's tables are only needed by the
    // epilogue (split tickets), which waits for that launch
    e = e_pre;
    p0 = p0_pre;
    n = n_pre;
  } else {
    pdl_wait_prev();           // routing tables and activations complete
    // fc2 reads the routing tables before its own wait: it may launch only once every CTA of
    // this kernel has seen them complete
    pdl_launch_next();
    // the shared-memory routing planned the same tiles as the routing launch (see checked_tile)
    if (p.ids != nullptr && tid == 0 && tile == 0 && fb == 0 && split == 0 &&
        nt != min(__ldcg(p.ctrl + 1), p.max_tiles))
      set_error(p.err, kErrRouteBounds);
    const int4 td = p.ids != nullptr ? checked_tile(p.tiles, p.ctrl, tile, p.E, p.Sm, BN, p.err)
                                      : p.tiles[tile];
    e = td.x;
    p0 = td.y;
    n = td.z;
    if (pre > 0 && e != e_pre) set_error(p.err, kErrRouteBounds);
  }
  const TileLoad<BN> tl(n);

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
        if (fused) {
          // the activations come from the quantising warps
          if (i >= pre) {
            mbar_arrive_expect_tx(&full[s], a_bytes + 2 * 512);
            load_a(st, e, kt, &full[s], pol);
          }
          continue;
        }
        if (i < pre) {
          mbar_arrive_expect_tx(&full[s], tl.b_bytes + tl.sf_bytes);
        } else {
          mbar_arrive_expect_tx(&full[s], a_bytes + tl.b_bytes + 2 * 512 + tl.sf_bytes);
          load_a(st, e, kt, &full[s], pol);
        }
        tl.load_b(st + 2 * kTileBytesA, &p.tm_x, kt * 128, p0, &full[s]);
        // activation-scale atom: the tile's prepared atom rows
        bulk_load(st + 2 * kTileBytesA + Cfg::kB + 1024, p.xs16 + ((size_t)kt * p.r16 + p0) * 16,
                  tl.sf_bytes, &full[s]);
      }
      issued = i;
    }
  } else if (fused && warp >= 2) {
    // warps 2..3: each stage's activation operand, quantised from the bf16 rows of the tile's
    // tokens (row block 0 also keeps a copy of the codes in xq / xs)
    if constexpr (BN <= 32) {
      const ActQuant<BN> aq{p.x, p.H, tid - 64};
      ok = act_quant_run<BN, S>(aq, s_tok, n, kt0, nk, 0, smem, Cfg::kStage1, 2 * kTileBytesA,
                                2 * kTileBytesA + Cfg::kB + 1024, full, empty,
                                fb == 0 ? p.xq : nullptr, p.xs, p0, p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (p.probe_ns != 0) ok = mbar_wait(&never, 0, p.err, p.probe_ns);
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % S;
        ok = mbar_wait(&full[s], (i / S) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        uint8_t* st = stage(s);
        const uint32_t sf = tmem + 2 * BN + Cfg::kSf1 * s;
        tc_cp_sf(sf + 0, desc_sf(st + 2 * kTileBytesA + Cfg::kB));
        tc_cp_sf(sf + 4, desc_sf(st + 2 * kTileBytesA + Cfg::kB + 512));
#pragma unroll
        for (int j = 0; j < Cfg::kChunks; ++j)
          if (j < tl.nch)
            tc_cp_sf(sf + 8 + 4 * j, desc_sf(st + 2 * kTileBytesA + Cfg::kB + 1024 + 512 * j));
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint32_t idesc = idesc_mxf8f6f4(kFmtE2M1, kFmtE4M3, NChunks<BN>::kWidth, kb);
          const uint32_t acc = (i > 0 || kb > 0) ? 1u : 0u;
#pragma unroll
          for (int j = 0; j < Cfg::kChunks; ++j) {
            if (j >= tl.nch) break;
            // columns 32j.. of the tile: B rows 32j.. (4 KB into the 128-byte-row tile)
            const uint64_t bdesc = desc_sw128(st + 2 * kTileBytesA + 4096 * j + 32 * kb);
            mma_mxf8f6f4(tmem + 32 * j, desc_sw128(st + 32 * kb), bdesc, idesc, sf + 0,
                         sf + 8 + 4 * j, acc);
            mma_mxf8f6f4(tmem + BN + 32 * j, desc_sw128(st + kTileBytesA + 32 * kb), bdesc, idesc,
                         sf + 4, sf + 8 + 4 * j, acc);
          }
        }
        tc_commit(&empty[s]);
      }
      tc_commit(&done);
    }
  }

  // ---- epilogue: all four warps, thread = weight row (feature), columns = tokens
  __syncwarp();
  if (fused) {
    pdl_wait_prev();           // routing launch complete: its tables and cleared tickets
    pdl_launch_next();
    // the shared-memory routing planned the same tiles as the routing launch (see checked_tile)
    if (tid == 0) {
      if (tile == 0 && fb == 0 && split == 0 && nt != min(__ldcg(p.ctrl + 1), p.max_tiles))
        set_error(p.err, kErrRouteBounds);
      const int4 td = checked_tile(p.tiles, p.ctrl, tile, p.E, p.Sm, BN, p.err);
      if (td.x != e || td.y != p0 || td.z != n) set_error(p.err, kErrRouteBounds);
    }
  }
  // one verdict per warp: the producer's or MMA issuer's lane may have given up a wait while the
  // other lanes did not, and the epilogue's TMEM loads and shuffles are warp-collective
  ok = __all_sync(0xffffffffu, mbar_wait(&done, 0, p.err) && ok);
  tc_fence_after();
  __syncwarp();
  const int f = fb * 128 + warp * 32 + lane;          // intermediate feature of this lane
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  if (ok && nk > 0) {
    if (p.splits == 1) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float up[16], gt[16];
        tmem_ld16(trow + c0, up);
        tmem_ld16(trow + BN + c0, gt);
        if (c0 >= n) continue;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c0 + j < n) {
            const float h = f < p.I ? swiglu(gt[j], up[j], p.limit, p.alpha, p.beta) : 0.f;
            const size_t row = (size_t)(p0 + c0 + j);
            requant_store(h, lane, row, p.Ip, f, p.hq, p.hs, p.hs16, p.r16);
          }
        }
      }
    } else {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float up[16], gt[16];
        tmem_ld16(trow + c0, up);
        tmem_ld16(trow + BN + c0, gt);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c0 + j < n) {
            float* g = p.gacc + ((size_t)split * p.Sm + p0 + c0 + j) * 2 * p.Ip;
            g[f] = up[j];
            g[p.Ip + f] = gt[j];
          }
        }
      }
    }
  }
  if (p.splits > 1) __threadfence();   // partial sums visible device-wide before the ticket
  if (!ok) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  // a wait gave up: let this CTA's copies land before its shared memory is released (its MMAs
  // completed or timed out at the wait on `done`)
  if (s_fail && warp == 0 && lane == 0) drain_stage_loads<S>(full, issued, p.err);
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc1);
  if (p.splits > 1) {
    if (tid == 0) {
      __threadfence();
      const int t = atomicAdd(&p.tickets[tile * p.RT + fb], 1);
      s_last = (t == p.splits - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      // partial sums added in split order: the same result on every run
      reduce_pieces(
          p.splits, n, (size_t)2 * p.Ip, (size_t)p.Ip,
          [&](int sp) -> const float* {
            return p.gacc + ((size_t)sp * p.Sm + p0) * 2 * p.Ip + f;
          },
          [&](int c, float up, float gt) {
            const float h = f < p.I ? swiglu(gt, up, p.limit, p.alpha, p.beta) : 0.f;
            const size_t row = (size_t)(p0 + c);
            requant_store(h, lane, row, p.Ip, f, p.hq, p.hs, p.hs16, p.r16);
          });
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(kTcThreads)
fc2_tc_kernel(const __grid_constant__ TcFc2Params p) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::kStages2;
  pdl_launch_next();
  __shared__ __align__(8) uint64_t full[S], empty[S], done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ int s_f[BN];          // flat slot index of each tile column
  __shared__ float s_w[BN];        // its router weight
  tmem_alloc_first(&s_tmem, Cfg::kAlloc2);
  // The routing tables were complete before fc1 let this kernel launch (fc1 waits for the
  // routing launch first), so the tile and the weights of the first stages are read before
  // waiting for fc1's output (L2 reads: nothing of them is in this SM's L1).
  const int tile = blockIdx.x;
  if (tile >= __ldcg(&p.ctrl[1])) {
    tmem_exit_early(&s_tmem, Cfg::kAlloc2);
    pdl_wait_prev();
    return;
  }
  const int4 td = __ldcg(&p.tiles[tile]);
  const int e = td.x, p0 = td.y, n = td.z;
  const TileLoad<BN> tl(n);
  const int rt = blockIdx.y;
  const int nk = p.KT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));

  if (tid == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
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
  auto stage = [&](int s) { return smem + s * Cfg::kStage2; };
  // stage layout: A | B | SFA | SFB

  if (warp == 0 && lane == 0) {
    const uint64_t pol = l2_evict_first_policy();   // weights: read once per call
    const int pre = nk < S ? nk : S;
    // weights of the first stages, before fc1 completes: the stage's barrier expects their
    // bytes now and is arrived on once the activation part is issued too
    for (int i = 0; i < pre; ++i) {
      const size_t a = ((size_t)e * (p.H / 128) + rt) * p.KT + i;
      mbar_expect_tx(&full[i], kTxBytesA + 512);
      tma_load_3d_hint(stage(i), &p.tm_w2, 0, 0, fp4_w2_tile(e, rt, i, p.H / 128, p.KT, p.pair),
                       &full[i], pol);
      bulk_load(stage(i) + kTileBytesA + Cfg::kB, p.sf2 + a * 512, 512, &full[i]);
    }
    pdl_wait_prev();     // fc1 complete, h visible
    int i = 0;
    for (; i < nk && ok; ++i) {
      const int s = i % S;
      if (i >= S) ok = mbar_wait(&empty[s], ((i / S) - 1) & 1, p.err);
      if (!ok) break;
      uint8_t* st = stage(s);
      if (i < pre) {
        mbar_arrive_expect_tx(&full[s], tl.b_bytes + tl.sf_bytes);
      } else {
        const size_t a = ((size_t)e * (p.H / 128) + rt) * p.KT + i;
        mbar_arrive_expect_tx(&full[s], kTxBytesA + tl.b_bytes + 512 + tl.sf_bytes);
        tma_load_3d_hint(st, &p.tm_w2, 0, 0, fp4_w2_tile(e, rt, i, p.H / 128, p.KT, p.pair),
                         &full[s], pol);
        bulk_load(st + kTileBytesA + Cfg::kB, p.sf2 + a * 512, 512, &full[s]);
      }
      tl.load_b(st + kTileBytesA, &p.tm_h, i * 128, p0, &full[s]);
      bulk_load(st + kTileBytesA + Cfg::kB + 512, p.hs16 + ((size_t)i * p.r16 + p0) * 16,
                tl.sf_bytes, &full[s]);
    }
    issued = i;
  } else {
    pdl_wait_prev();     // previous kernels of the call complete
  }
  if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % S;
        ok = mbar_wait(&full[s], (i / S) & 1, p.err);
        if (!ok) break;
        tc_fence_after();
        uint8_t* st = stage(s);
        const uint32_t sf = tmem + BN + Cfg::kSf2 * s;
        tc_cp_sf(sf + 0, desc_sf(st + kTileBytesA + Cfg::kB));
#pragma unroll
        for (int j = 0; j < Cfg::kChunks; ++j)
          if (j < tl.nch)
            tc_cp_sf(sf + 4 + 4 * j, desc_sf(st + kTileBytesA + Cfg::kB + 512 + 512 * j));
        // a paired tail tile: two K steps, at columns 64.. of the tile for an odd row block
        const bool tail = p.pair && i == nk - 1;
        const int a_off = (tail && (rt & 1)) ? 64 : 0;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          if (tail && kb >= 2) break;
          const uint32_t idesc = idesc_mxf8f6f4(kFmtE2M1, kFmtE4M3, NChunks<BN>::kWidth, kb);
#pragma unroll
          for (int j = 0; j < Cfg::kChunks; ++j)
            if (j < tl.nch)
              mma_mxf8f6f4(tmem + 32 * j, desc_sw128(st + a_off + 32 * kb),
                         desc_sw128(st + kTileBytesA + 4096 * j + 32 * kb), idesc, sf + 0,
                         sf + 4 + 4 * j, (i > 0 || kb > 0) ? 1u : 0u);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(&done);
    }
  } else if (warp == 3) {
    // warp 3: the combine's slot indices and router weights, loaded while the GEMM runs
    for (int c = lane; c < n; c += 32) {
      const int f = p.perm[p0 + c];
      s_f[c] = f;
      s_w[c] = p.topk_w[f];
    }
  }

  __syncthreads();                                    // s_f / s_w written
  // one verdict per warp: the producer's or MMA issuer's lane may have given up a wait while the
  // other lanes did not, and the epilogue's TMEM loads and shuffles are warp-collective
  ok = __all_sync(0xffffffffu, mbar_wait(&done, 0, p.err) && ok);
  tc_fence_after();
  __syncwarp();
  const int h = rt * 128 + warp * 32 + lane;          // output column of this lane
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  if (ok) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      float y[16];
      tmem_ld16(trow + c0, y);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j < n) {
          const int f = s_f[c0 + j];
          const float v = s_w[c0 + j] * y[j];
          if (p.deterministic)
            p.rbuf[(size_t)f * p.H + h] = v;
          else
            atomicAdd(&p.acc[(size_t)(f / p.topk) * p.H + h], v);
        }
      }
    }
  }
  if (!ok) s_fail = 1;
  tc_fence_before();
  __syncthreads();
  // a wait gave up: let this CTA's copies land before its shared memory is released (its MMAs
  // completed or timed out at the wait on `done`)
  if (s_fail && warp == 0 && lane == 0) drain_stage_loads<S>(full, issued, p.err);
  if (warp == 0) tmem_dealloc(tmem, Cfg::kAlloc2);
}

// ---------------------------------------------------------------------------------- host side

EncodeTiledFn tc_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool tmap_fp4(CUtensorMap* tm, const void* base, int rows, long long tiles) {
  EncodeTiledFn enc = tc_encode_fn();
  if (!enc) return false;
  if (tiles <= 0 || rows <= 0) return true;
  cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)tiles};
  cuuint64_t strides[2] = {64, (cuuint64_t)64 * rows};
  cuuint32_t box[3] = {128, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_u8(CUtensorMap* tm, const void* base, int K, int rows, int box_rows) {
  EncodeTiledFn enc = tc_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-tile width of the tensor-core kernels.  W4A8: 16-token tiles for decode calls (M <= 16);
// beyond, the width follows the expected slots per expert (M * topk / E under uniform routing),
// so that an expert's weights stream through the SMs about once per call: 32 up to 16 slots per
// expert, 64 up to 40, 96 beyond (2 CTAs per SM at every width: 2-stage rings, <= 256 tensor
// memory columns).  The 16-bit path keeps its M-based widths.
int tc_pick_bn(int M, int topk, int E, bool w4a8) {
  if (w4a8) {
    if (M <= 16) return 16;
    const long long slots = (long long)M * topk;
    if (slots <= 16LL * E) return 32;
    if (slots <= 40LL * E) return 64;
    return 96;
  }
  return M <= 16 ? 16 : (M <= 64 ? 32 : (M <= 512 ? 64 : 128));
}

template <int BN>
static cudaError_t launch_fc1_bn(const TcFc1Params& p, int tiles, cudaStream_t st) {
  using Cfg = TcCfg<BN>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(fc1_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Cfg::kSmem1);
    // all of the unified L1 / shared storage as shared memory
    cudaFuncSetAttribute(fc1_tc_kernel<BN>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    attr = true;
  }
  TcFc1Params q = p;
  q.fb_in_x = tiles <= 65535 ? 1 : 0;
  const dim3 grid = q.fb_in_x ? dim3(p.RT, tiles, p.splits) : dim3(tiles, p.RT, p.splits);
  return launch_kernel(fc1_tc_kernel<BN>, grid, dim3(kTcThreads), Cfg::kSmem1, st, true, q);
}

template <int BN>
static cudaError_t launch_fc2_bn(const TcFc2Params& p, int tiles, cudaStream_t st) {
  using Cfg = TcCfg<BN>;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(fc2_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Cfg::kSmem2);
    // all of the unified L1 / shared storage as shared memory
    cudaFuncSetAttribute(fc2_tc_kernel<BN>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    attr = true;
  }
  dim3 grid(tiles, p.H / 128);
  return launch_kernel(fc2_tc_kernel<BN>, grid, dim3(kTcThreads), Cfg::kSmem2, st, true, p);
}

// fc1 (stage 0) or fc2 (stage 1) of the W4A8 tensor-core path.
cudaError_t launch_tc_stage(int stage, const DevWeights& w, const RunPtrs& r, const PlanDims& d,
                            int bn, int tiles, int splits, const float* topk_w, int M,
                            const int32_t* ids, int max_tiles, const void* x,
                            cudaStream_t st) {
  const int Sm = M * d.topk;
  const int RT = cdiv(d.I, 128);
  if (stage == 0) {
    TcFc1Params p;
    memset(&p.tm_w13_tail, 0, sizeof(p.tm_w13_tail));
    p.RTf = d.I / 128;
    p.rem = d.I % 128;
    const long long kt = d.H / 128;
    if (!tmap_fp4(&p.tm_w13, w.w13, 128, 2LL * d.E * p.RTf * kt) ||
        !tmap_fp4(&p.tm_w13_tail, w.w13 + (size_t)2 * d.E * p.RTf * kt * 8192, p.rem, 2LL * d.E * kt))
      return cudaErrorInvalidValue;
    if (!tmap_u8(&p.tm_x, r.xq, d.H, Sm, act_box_rows(bn))) return cudaErrorInvalidValue;
    p.sf13 = w.s13; p.tiles = r.tiles; p.ctrl = r.ctrl; p.err = r.ctrl;
    p.hq = r.hq; p.hs = r.hs; p.gacc = r.g; p.tickets = r.tickets;
    p.xs16 = r.xs16; p.hs16 = r.hs16; p.r16 = r.r16;
    p.H = d.H; p.I = d.I; p.Ip = d.Ip; p.RT = RT; p.KT = d.H / 128; p.Sm = Sm;
    p.splits = splits; p.limit = d.limit; p.alpha = d.alpha; p.beta = d.beta;
    p.ids = (ids != nullptr && Sm <= kPreRouteSlots) ? ids : nullptr;
    p.Mk = Sm; p.E = d.E; p.max_tiles = max_tiles; p.ep_first = d.ep_first;
    // quantised here only when the call routes in shared memory at a width of <= 32 tokens
    p.x = (p.ids != nullptr && bn <= 32) ? static_cast<const __nv_bfloat16*>(x) : nullptr;
    p.topk = d.topk;
    p.probe_ns = d.wait_probe_ns;
    p.xq = d.keep_act ? r.xq : nullptr;
    p.xs = r.xs;
    switch (bn) {
      case 16: return launch_fc1_bn<16>(p, tiles, st);
      case 32: return launch_fc1_bn<32>(p, tiles, st);
      case 64: return launch_fc1_bn<64>(p, tiles, st);
      case 96: return launch_fc1_bn<96>(p, tiles, st);
      default: return cudaErrorInvalidValue;
    }
  }
  TcFc2Params p;
  if (!tmap_fp4(&p.tm_w2, w.w2, 128, (long long)d.E * (d.H / 128) * (d.Ip / 128)))
    return cudaErrorInvalidValue;
  if (!tmap_u8(&p.tm_h, r.hq, d.Ip, Sm, act_box_rows(bn))) return cudaErrorInvalidValue;
  p.sf2 = w.s2; p.tiles = r.tiles; p.ctrl = r.ctrl; p.err = r.ctrl;
  p.hs16 = r.hs16; p.r16 = r.r16;
  p.perm = r.perm; p.topk_w = topk_w; p.acc = r.acc; p.rbuf = r.rbuf;
  p.H = d.H; p.Ip = d.Ip; p.KT = d.Ip / 128; p.Sm = Sm; p.topk = d.topk;
  p.pair = (d.I & 127) == 64 ? 1 : 0;
  p.deterministic = d.deterministic;
  switch (bn) {
    case 16: return launch_fc2_bn<16>(p, tiles, st);
    case 32: return launch_fc2_bn<32>(p, tiles, st);
    case 64: return launch_fc2_bn<64>(p, tiles, st);
    case 96: return launch_fc2_bn<96>(p, tiles, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
