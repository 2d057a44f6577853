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
struct StreamWork {
  int KT, G, c, D, first_stream_unit;   // first_stream_unit = D * G
  long long W, x0, x1;                  // stream steps of all CTAs; this CTA's range
  int n_sk, nsteps;                     // this CTA's stream steps; all its steps

  __device__ __forceinline__ void init(int units, int kt, int g, int cta) {
    KT = kt; G = g; c = cta;
    D = units / g;
    first_stream_unit = D * g;
    W = (long long)(units - first_stream_unit) * kt;
    x0 = begin_of(cta);
    x1 = begin_of(cta + 1);
    n_sk = (int)(x1 - x0);
    nsteps = n_sk + D * kt;
  }
  __device__ __forceinline__ long long begin_of(int cta) const { return (long long)cta * W / G; }
  // Segments of this CTA in order, without a division per K step: its stream range (split at
  // unit boundaries), then its whole units.  next() returns false after the last one.
  struct Segs {
    const StreamWork* w;
    long long x;    // next flat stream step
    int dp;         // whole units handed out
    __device__ __forceinline__ bool next(int& u, int& k0, int& len) {
      if (x < w->x1) {
        u = w->first_stream_unit + (int)(x / w->KT);
        k0 = (int)(x % w->KT);
        len = (int)min((long long)(w->KT - k0), w->x1 - x);
        x += len;
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
  // stream steps: CTA holding flat stream step x (ranges may be empty when G > W)
  __device__ __forceinline__ int cta_of(long long x) const {
    int cc = (int)((x * G) / W);
    while (cc + 1 < G && begin_of(cc + 1) <= x) ++cc;
    while (cc > 0 && begin_of(cc) > x) --cc;
    return cc;
  }
  // partial slot of CTA cc's piece of stream unit u: 2cc for the unit its range starts in,
  // 2cc + 1 for the one it ends in (no other piece of a range can be partial)
  __device__ __forceinline__ int part_slot(int cc, int u) const {
    const int first = first_stream_unit + (int)(begin_of(cc) / KT);
    return 2 * cc + (u == first ? 0 : 1);
  }
};

// ---------------------------------------------------------------------------------- host side

constexpr int kStreamMaxCtas = 320;   // partial slots are reserved for this many CTAs

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
