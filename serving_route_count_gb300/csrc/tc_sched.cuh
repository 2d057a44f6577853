// tc_sched.cuh - work schedules of the persistent W4A8 kernels: which (tile, 128-row block)
// units and which of their K tiles each CTA of a fixed grid processes.
#pragma once

#include <algorithm>

#include "moe_common.cuh"

namespace moe {

// Work of one CTA (G CTAs, U units of KT K steps).  With D = floor(U / G) full waves, the units
// D*G .. U-1 ("stream units") are split over all CTAs by K steps: CTA c gets the flat range
// [c*W/G, (c+1)*W/G) of their W = (U - D*G) * KT steps.  CTA c first streams that range, then
// its whole units c, c + G, ..., c + (D-1)*G, so the pieces' hand-over to the reducing CTA
// overlaps the whole units' streaming.
// All schedule arithmetic is 32-bit (the host admits a call only when W * G < 2^31, see
// stream_schedule_fits): a 64-bit division is a long software sequence on the GPU, and the
// reducing CTA of a unit enumerates its pieces on the critical path of the call.
constexpr int kStreamMaxPieces = 130;   // pieces of one unit: at most KT + 1 (KT <= 128)
struct StreamWork {
  int KT, G, c, D, first_stream_unit;   // first_stream_unit = D * G
  uint32_t W, q, rm;                    // stream steps of all CTAs, W / G, W % G
  uint32_t x0, x1;                      // this CTA's range of stream steps
  int own_first_unit;                   // stream unit holding step x0
  int n_sk, nsteps;                     // this CTA's stream steps; all its steps

  __device__ __forceinline__ void init(int units, int kt, int g, int cta) {
    KT = kt; G = g; c = cta;
    D = units / g;
    first_stream_unit = D * g;
    W = (uint32_t)(units - first_stream_unit) * (uint32_t)kt;
    q = W / (uint32_t)g;
    rm = W % (uint32_t)g;
    x0 = begin_of(cta);
    x1 = begin_of(cta + 1);
    own_first_unit = first_stream_unit + (int)(x0 / (uint32_t)kt);
    n_sk = (int)(x1 - x0);
    nsteps = n_sk + D * kt;
  }
  __device__ __forceinline__ uint32_t begin_of(int cta) const {
    return (uint32_t)cta * W / (uint32_t)G;
  }
  // Segments of this CTA in order: its stream range (split at unit boundaries), then its
  // whole units.  next() returns false after the last one.
  struct Segs {
    const StreamWork* w;
    uint32_t x;     // next flat stream step
    int dp;         // whole units handed out
    __device__ __forceinline__ bool next(int& u, int& k0, int& len) {
      if (x < w->x1) {
        const uint32_t kt = (uint32_t)w->KT;
        u = w->first_stream_unit + (int)(x / kt);
        k0 = (int)(x % kt);
        len = (int)min(kt - (uint32_t)k0, w->x1 - x);
        x += (uint32_t)len;
        return true;
      }
      if (dp < w->D) {
        u = w->c + dp * w->G;
        k0 = 0;
        len = w->KT;
        ++dp;
        return true;
      }
      return false;
    }
  };
  __device__ __forceinline__ Segs segs() const { return Segs{this, x0, 0}; }
  // partial slot of this CTA's piece of stream unit u: 2c for the unit its range starts in,
  // 2c + 1 for the one it ends in (no other piece of a range can be partial)
  __device__ __forceinline__ int own_slot(int u) const {
    return 2 * c + (u == own_first_unit ? 0 : 1);
  }
  // The partial slots of stream unit u's pieces in K order (the CTAs whose non-empty ranges
  // overlap its steps) into slots[]; returns their count.  One division pair, then the range
  // starts by an incremental recurrence (begin_of(c + 1) = begin_of(c) + q, + 1 when the
  // remainder wraps).
  __device__ int unit_pieces(int u, int* slots) const {
    const uint32_t xs = (uint32_t)(u - first_stream_unit) * (uint32_t)KT, xe = xs + KT;
    int cc = (int)(xs * (uint32_t)G / W);   // a CTA at or just before the owner of xs
    while (cc > 0 && begin_of(cc) > xs) --cc;
    uint32_t b = begin_of(cc), r = (uint32_t)cc * W % (uint32_t)G;
    int n = 0;
    for (; cc < G && b < xe; ++cc) {
      uint32_t nb = b + q, nr = r + rm;
      if (nr >= (uint32_t)G) {
        ++nb;
        nr -= (uint32_t)G;
      }
      if (nb > b && nb > xs && n < kStreamMaxPieces) slots[n++] = 2 * cc + (b >= xs ? 0 : 1);
      b = nb;
      r = nr;
    }
    return n;
  }
};


// The units of one CTA of the persistent fc2 (units = (tile, 128-row block of H) pairs of KT K
// tiles).  Flat mode: the steps [x, x1) of the units in tile-major order (unit = tile * RB + rb),
// cut at unit boundaries.  Round-robin mode: whole units c, c + G, c + 2G, ... in
// row-block-major order (unit = rb * n_tiles + tile), so that at any time the grid works on a
// narrow band of output column blocks and the combine's lines of that band stay in L2 while
// all their contributions arrive.  next() gives each segment's tile, row block, first K tile
// and length, in order; false after the last.
struct Fc2Units {
  int KT, RB, n_tiles, units, G, rr;
  int x, x1;     // flat mode
  int u;         // round-robin mode
  __device__ __forceinline__ bool next(int& tile, int& rb, int& k0, int& len) {
    if (rr) {
      if (u >= units) return false;
      rb = u / n_tiles;
      tile = u - rb * n_tiles;
      k0 = 0;
      len = KT;
      u += G;
      return true;
    }
    if (x >= x1) return false;
    const int uu = x / KT;
    k0 = x - uu * KT;
    len = min(KT - k0, x1 - x);
    x += len;
    tile = uu / RB;
    rb = uu - tile * RB;
    return true;
  }
};

// ---------------------------------------------------------------------------------- host side

constexpr int kStreamMaxCtas = 320;   // partial slots are reserved for this many CTAs

// Whether a stream-K schedule of `units` units of `kt` K steps fits the 32-bit arithmetic and
// the piece list of StreamWork for any grid of at most kStreamMaxCtas CTAs.
inline bool stream_schedule_fits(long long units, int kt) {
  return kt >= 1 && kt < kStreamMaxPieces && units * kt * kStreamMaxCtas < (1LL << 31);
}

// Resident CTAs of a persistent kernel: as many per SM as shared memory and tensor memory hold
// (`smem` dynamic bytes and `tmem_cols` columns per CTA), capped at `per_sm_cap` per SM and at
// `cap` in all.  (The occupancy query of the runtime reports one CTA per SM for any kernel that
// allocates tensor memory, although several are co-scheduled when both memories allow it.)
template <typename K>
inline int persistent_grid(K kernel, int smem, int tmem_cols, int per_sm_cap, int cap) {
  int sms = 0, dev = 0, sm_smem = 0, reserved = 0;
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // all of the unified L1 / shared storage as shared memory
  cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                       (int)cudaSharedmemCarveoutMaxShared);
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) fa.sharedSizeBytes = 0;
  const int per_cta = smem + (int)fa.sharedSizeBytes + reserved;
  int per_sm = std::min(sm_smem / std::max(per_cta, 1), 512 / std::max(tmem_cols, 32));
  per_sm = std::max(1, std::min(per_sm, per_sm_cap));
  (void)cudaGetLastError();
  return std::min(cap, per_sm * std::max(sms, 1));
}

}  // namespace moe
