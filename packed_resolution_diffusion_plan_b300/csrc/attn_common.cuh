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
// A drain that runs out raises the abort flag (if nothing did before), so
// that the CTA records a timeout instead of stalling silently.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0u && globaltimer_ns() - t0 > kWaitTimeoutNs) {
      if (*abort_flag == 0) *abort_flag = static_cast<int>(smem_u32(bar)) + 1;
      return;
    }
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

// RoPE factors of chunks [c_first, c_first + kChunks) of token `tok`'s row
// (logical 16-byte chunk c holds dims 8c .. 8c + 7, four rotation pairs):
// cs[i] = (cos, sin) of the chunk's four pairs; identity for text and for
// rows outside the sample (valid = false).  Only global loads: callers issue
// them before waiting for the tile, so that their latency overlaps the wait.
template <int D, int kChunks>
__device__ __forceinline__ void rope_row_cs(int c_first, long long tok, bool valid, const AttnGeom& g,
                                            float (&cs)[kChunks][8]) {
  const int2 p = valid ? reinterpret_cast<const int2*>(g.pos)[tok] : make_int2(-1, -1);
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int c = c_first + i;
    if (p.x < 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) { cs[i][2 * e] = 1.f; cs[i][2 * e + 1] = 0.f; }
    } else if (g.rope_axes == 2) {
      // 2 axes: the chunk's four pairs are consecutive frequencies of one half
      const int m0 = 4 * c;
      const int k0 = m0 % (D / 4);
      const int pp = m0 >= D / 4 ? p.y : p.x;
      const float4* tab = reinterpret_cast<const float4*>(g.rope_cs) + static_cast<size_t>(pp) * (D / 8) + k0 / 2;
      const float4 a0 = __ldg(tab), a1 = __ldg(tab + 1);
      cs[i][0] = a0.x; cs[i][1] = a0.y; cs[i][2] = a0.z; cs[i][3] = a0.w;
      cs[i][4] = a1.x; cs[i][5] = a1.y; cs[i][6] = a1.z; cs[i][7] = a1.w;
    } else {
      const int fr = g.frame[tok];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 v = rope_pair_cs<D>(g, 4 * c + e, p, fr);
        cs[i][2 * e] = v.x;
        cs[i][2 * e + 1] = v.y;
      }
    }
  }
}

// Rotates chunks [c_first, c_first + kChunks) of row r of a swizzled 128-row
// bf16 tile in shared memory into fp16 scale * R(x), in place, with the
// factors of rope_row_cs; a row outside the sample (valid = false) is zeroed,
// so that no value of the next sample, finite or not, takes part in this
// sample's products.  Returns the largest rotated magnitude.
template <int kChunks>
__device__ __forceinline__ float rotate_row_f16(uint8_t* tile, int r, int c_first, bool valid, float scale,
                                                const float (&cs)[kChunks][8]) {
  uint8_t* rowp = tile + r * 128;
  auto chunk_ptr = [&](int c) {
    return reinterpret_cast<uint4*>(rowp + (c >> 3) * 16384 + (((c & 7) ^ (r & 7)) << 4));
  };
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    uint4* ptr = chunk_ptr(c_first + i);
    if (!valid) {
      *ptr = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4 x = *ptr;
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x);
    uint32_t y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float c = cs[i][2 * e], sn = cs[i][2 * e + 1];
      const float x0 = bf16_lo(xw[e]), x1 = bf16_hi(xw[e]);
      const float y0 = fmaf(x0, c, -x1 * sn) * scale, y1 = fmaf(x0, sn, x1 * c) * scale;
      amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
      y[e] = pack_f16(y0, y1);
    }
    *ptr = make_uint4(y[0], y[1], y[2], y[3]);
  }
  return amax;
}

// SMs of the current device (cached per device): the persistent attention
// kernels launch one CTA per SM.
inline int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace mf
