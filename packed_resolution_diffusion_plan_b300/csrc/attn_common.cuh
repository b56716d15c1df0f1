// Device helpers shared by the attention kernels: work decode, warp-uniform
// bounded waits and the in-shared-memory 2D RoPE of one tile row.
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

// Row r of a 128-row bf16 tile of D columns (D/64 128-byte-swizzled halves)
// becomes, in place, fp16 of  mult * R(p) x :  the first D/2 columns turn by
// the latent row p.x, the rest by the column p.y, pair i of a half using
// table entry i of rope_cs (float [grid][D/4][2] = cos, sin); text rows
// (p.x < 0) are only scaled.  Returns the largest |value| written, so the
// caller can flag values beyond the fp16 range.
// kUnroll bounds how many 16-byte chunks the compiler may keep in flight
// (and so the registers the row needs).
template <int D, int kUnroll = D / 8>
__device__ __forceinline__ float rope_row_to_f16(uint8_t* tile, int r, int2 p, const float* rope_cs,
                                                 float mult) {
  constexpr int nf = D / 4;
  float amax = 0.f;
  if (p.x >= 0) {
    const float4* tab_row = reinterpret_cast<const float4*>(rope_cs) + static_cast<size_t>(p.x) * (nf / 2);
    const float4* tab_col = reinterpret_cast<const float4*>(rope_cs) + static_cast<size_t>(p.y) * (nf / 2);
#pragma unroll kUnroll
    for (int c16 = 0; c16 < D / 8; ++c16) {
      const int dim0 = c16 * 8;
      const int k0 = (dim0 % (D / 2)) / 2;  // multiple of 4
      const float4* tab = dim0 >= D / 2 ? tab_col : tab_row;
      const float4 a = __ldg(tab + k0 / 2);
      const float4 b = __ldg(tab + k0 / 2 + 1);
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      const float cs[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
        const float c = cs[2 * e] * mult, s = cs[2 * e + 1] * mult;
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
  } else {
#pragma unroll kUnroll
    for (int c16 = 0; c16 < D / 8; ++c16) {
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y0 = bf16_lo(w[e]) * mult, y1 = bf16_hi(w[e]) * mult;
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
  }
  return amax;
}

// The same rotation with the table's fp16 copy (rope_cs16: [grid][D/4] words
// of fp16 cos | fp16 sin << 16): one 16-byte load covers the four pairs of a
// 16-byte chunk, and the whole table of a 2048-pixel grid (16.5 KB) stays in
// the L1 cache that the 226 KB of shared tiles leave.
template <int D, int kUnroll = D / 8>
__device__ __forceinline__ float rope_row_to_f16_t16(uint8_t* tile, int r, int2 p, const uint32_t* rope_cs16,
                                                     float mult) {
  constexpr int nf = D / 4;
  float amax = 0.f;
  if (p.x >= 0) {
    const uint4* tab_row = reinterpret_cast<const uint4*>(rope_cs16) + static_cast<size_t>(p.x) * (nf / 4);
    const uint4* tab_col = reinterpret_cast<const uint4*>(rope_cs16) + static_cast<size_t>(p.y) * (nf / 4);
#pragma unroll kUnroll
    for (int c16 = 0; c16 < D / 8; ++c16) {
      const int dim0 = c16 * 8;
      const int k0 = (dim0 % (D / 2)) / 2;  // multiple of 4
      const uint4 t = __ldg((dim0 >= D / 2 ? tab_col : tab_row) + k0 / 4);
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      const uint32_t cs[4] = {t.x, t.y, t.z, t.w};
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&cs[e]));
        const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
        const float c = f.x * mult, s = f.y * mult;
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
  } else {
#pragma unroll kUnroll
    for (int c16 = 0; c16 < D / 8; ++c16) {
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y0 = bf16_lo(w[e]) * mult, y1 = bf16_hi(w[e]) * mult;
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
  }
  return amax;
}

// Zero row r of a 128-row tile of D columns (rows past a sample's end).
template <int D>
__device__ __forceinline__ void zero_row(uint8_t* tile, int r) {
#pragma unroll
  for (int c16 = 0; c16 < D / 8; ++c16)
    *reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7)) = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace mf
