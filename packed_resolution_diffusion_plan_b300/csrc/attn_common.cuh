// Device helpers shared by the attention kernels: work decode and
// warp-uniform bounded waits.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace mf {

struct WorkItem {
  int sample;
  int head;
  int tile;       // 128-row tile index inside the sample
  int seq_start;  // first token of the sample in the pack
  int len;        // L_i
};

// Items are grouped per sample in longest-first order; inside a group the
// head is the slow index and the tile (kRows = 128) or tile pair (kRows =
// 256) the fast one, so CTAs that run at the same time share one head's K/V
// (or Q/dO) in L2.
template <int kRows = kTile>
__device__ __forceinline__ WorkItem decode_item(const AttnGeom& g, int item) {
  constexpr int col = kRows == kTile ? 1 : 2;  // order column of the first unit
  int lo = 0, hi = g.n_samples;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (g.order[4 * mid + col] * g.heads <= item) lo = mid; else hi = mid;
  }
  WorkItem w;
  w.sample = g.order[4 * lo];
  const int start = g.order[4 * lo + col];
  w.seq_start = g.cu_seqlens[w.sample];
  w.len = g.cu_seqlens[w.sample + 1] - w.seq_start;
  const int nt = (w.len + kRows - 1) / kRows;
  const int local = item - start * g.heads;
  w.head = local / nt;
  w.tile = local - w.head * nt;
  return w;
}

// Bounded wait whose outcome is the same in every lane of the warp, so that
// warp-collective tcgen05 instructions that follow stay convergent.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Teardown wait: bounded, but not cut short by the abort flag, used to let
// the CTA's own TMA copies / MMAs land before shared memory or TMEM is freed.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0u && globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

// (cos, sin) of rotation pair m (dims 2m, 2m+1, m < D/2) of a token at latent
// position p = (row, col) and frame f; text tokens (p.x < 0) are not rotated.
//   2 axes: pairs [0, D/4) turn by the row, [D/4, D/2) by the column; pair i
//           of a half at theta^(-2i/(D/2)) (plan table [grid][D/4]).
//   3 axes: pairs [0, D/16) turn by the frame (a slice of D/8 dims, table
//           [2][D/16]), the next 7D/32 by the row and the last 7D/32 by the
//           column (slices of 7D/16 dims, table [grid][7D/32]); pair i of an
//           a-dim slice at theta^(-2i/a).
template <int D>
__device__ __forceinline__ float2 rope_pair_cs(const AttnGeom& g, int m, int2 p, int f) {
  if (p.x < 0) return make_float2(1.f, 0.f);
  const float2* hw = reinterpret_cast<const float2*>(g.rope_cs);
  if (g.rope_axes == 3) {
    constexpr int nf = D / 16, nh = 7 * D / 32;
    if (m < nf) return __ldg(reinterpret_cast<const float2*>(g.rope_f) + f * nf + m);
    m -= nf;
    return m < nh ? __ldg(hw + p.x * nh + m) : __ldg(hw + p.y * nh + (m - nh));
  }
  constexpr int nh = D / 4;
  return m < nh ? __ldg(hw + p.x * nh + m) : __ldg(hw + p.y * nh + (m - nh));
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace mf
