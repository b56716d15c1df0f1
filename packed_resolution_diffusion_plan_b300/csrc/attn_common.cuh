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
// the latent row p.x, the rest by the column p.y, pair k of a half by angle
// pos * f_k; text rows (p.x < 0) are only scaled.  The first half reads the
// full table (rope_cs, float [grid][D/4][2]) at p.x, which a whole image row
// shares, so a warp's loads are broadcasts; the second half's rotation of
// position pos = 32 h + l is the product of the two-level table's entries
// e^{i 32h f_k} and e^{i l f_k} (rope_hl, float [2][D/4][32][2]): 16 KB that
// stay in L1 next to 226 KB of shared tiles, and a warp of consecutive
// tokens reads consecutive l.  Returns the largest |value| written, so the
// caller can flag values beyond the fp16 range.  kUnroll bounds the chunks
// whose loads are in flight together (and so the registers the row needs).
template <int D, bool kScale, int kUnroll = 2>
__device__ __forceinline__ float rope_row_to_f16(uint8_t* tile, int r, int2 p, const float* rope_cs,
                                                 const float* rope_hl, float mult) {
  constexpr int nf = D / 4;
  const float2* hi = reinterpret_cast<const float2*>(rope_hl);  // [nf][32]
  const float2* lo = hi + nf * 32;                              // [nf][32]
  float amax = 0.f;
  if (p.x >= 0) {
    const float2* full = reinterpret_cast<const float2*>(rope_cs) + static_cast<size_t>(p.x) * nf;
    const int hc = p.y >> 5, lc = p.y & 31;
    // first half: one full-table entry per pair
#pragma unroll kUnroll
    for (int c16 = 0; c16 < D / 16; ++c16) {
      const int k0 = c16 * 4;
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 F = __ldg(full + k0 + e);
        const float c = kScale ? F.x * mult : F.x, s = kScale ? F.y * mult : F.y;
        const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
    // second half: the product of the two-level table's entries
#pragma unroll kUnroll
    for (int c16 = D / 16; c16 < D / 8; ++c16) {
      const int k0 = (c16 - D / 16) * 4;
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 A = __ldg(hi + (k0 + e) * 32 + hc);
        const float2 B = __ldg(lo + (k0 + e) * 32 + lc);
        float c = fmaf(A.x, B.x, -A.y * B.y), s = fmaf(A.y, B.x, A.x * B.y);
        if (kScale) {
          c *= mult;
          s *= mult;
        }
        const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
        const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
  } else {
#pragma unroll 4
    for (int c16 = 0; c16 < D / 8; ++c16) {
      uint4* ptr = reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y0 = kScale ? bf16_lo(w[e]) * mult : bf16_lo(w[e]);
        const float y1 = kScale ? bf16_hi(w[e]) * mult : bf16_hi(w[e]);
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      *ptr = v;
    }
  }
  return amax;
}

// Part `part` of kParts of row r of a 128-row bf16 tile, rotated in place and
// rounded to fp16 like rope_row_to_f16: the part takes the same share of both
// halves (the first D/2 columns, which turn by the latent row, and the rest,
// which turn by the column), so that kParts threads sharing a row do equal
// work.  Rows at or past the sample's end (valid = false) become zero.
// Returns the largest |value| written.
template <int D, bool kScale, int kParts>
__device__ __forceinline__ float rope_part_row_to_f16(uint8_t* tile, int r, int part, int2 p, bool valid,
                                                      const float* rope_cs, const float* rope_hl, float mult) {
  constexpr int nf = D / 4;
  constexpr int kHalfChunks = D / 16;
  constexpr int n = kHalfChunks / kParts;
  static_assert(n * kParts == kHalfChunks, "parts must split a half into whole chunks");
  const int k0 = part * n;
  float amax = 0.f;
  auto chunk_ptr = [&](int c16) {
    return reinterpret_cast<uint4*>(tile + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7));
  };
  auto finish = [&](uint32_t (&w)[4], const float (&y)[8]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float y0 = kScale ? y[2 * e] * mult : y[2 * e], y1 = kScale ? y[2 * e + 1] * mult : y[2 * e + 1];
      amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
      w[e] = pack_f16(y0, y1);
    }
  };
  if (!valid) {
#pragma unroll
    for (int k = 0; k < n; ++k) {
      *chunk_ptr(k0 + k) = make_uint4(0, 0, 0, 0);
      *chunk_ptr(kHalfChunks + k0 + k) = make_uint4(0, 0, 0, 0);
    }
    return 0.f;
  }
  if (p.x < 0) {  // text row: scale and round only
#pragma unroll 2
    for (int k = 0; k < 2 * n; ++k) {
      uint4* ptr = chunk_ptr((k < n ? 0 : kHalfChunks - n) + k0 + k);
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
      float y[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        y[2 * e] = bf16_lo(w[e]);
        y[2 * e + 1] = bf16_hi(w[e]);
      }
      finish(*reinterpret_cast<uint32_t(*)[4]>(w), y);
      *ptr = v;
    }
    return amax;
  }
  // first half: (cos, sin) of p.x from the full table
  const float2* full = reinterpret_cast<const float2*>(rope_cs) + static_cast<size_t>(p.x) * nf;
#pragma unroll 2
  for (int k = k0; k < k0 + n; ++k) {
    uint4* ptr = chunk_ptr(k);
    uint4 v = *ptr;
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
    float y[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 F = __ldg(full + 4 * k + e);
      const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
      y[2 * e] = fmaf(x0, F.x, -x1 * F.y);
      y[2 * e + 1] = fmaf(x0, F.y, x1 * F.x);
    }
    finish(*reinterpret_cast<uint32_t(*)[4]>(w), y);
    *ptr = v;
  }
  // second half: the two-level factors of p.y
  const float2* hi = reinterpret_cast<const float2*>(rope_hl);  // [nf][32]
  const float2* lo = hi + nf * 32;                              // [nf][32]
  const int hc = p.y >> 5, lc = p.y & 31;
#pragma unroll 2
  for (int k = k0; k < k0 + n; ++k) {
    uint4* ptr = chunk_ptr(kHalfChunks + k);
    uint4 v = *ptr;
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
    float y[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 A = __ldg(hi + (4 * k + e) * 32 + hc);
      const float2 B = __ldg(lo + (4 * k + e) * 32 + lc);
      const float c = fmaf(A.x, B.x, -A.y * B.y), s = fmaf(A.y, B.x, A.x * B.y);
      const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
      y[2 * e] = fmaf(x0, c, -x1 * s);
      y[2 * e + 1] = fmaf(x0, s, x1 * c);
    }
    finish(*reinterpret_cast<uint32_t(*)[4]>(w), y);
    *ptr = v;
  }
  return amax;
}

// The same rotation of row r with its 16-byte chunks software-pipelined:
// chunk c + 1's row data and table entries are loaded before chunk c is
// rotated and stored (the in-place store would otherwise order every later
// load behind it), which roughly halves the row's latency at the cost of
// ~100 registers; rows at or past the sample's end (valid = false) become
// zero.  Used where the rotation of a streamed tile bounds the step (the
// forward's K tiles).
template <int D, bool kScale>
__device__ __forceinline__ float rope_row_to_f16_pipelined(uint8_t* tile, int r, int2 p, bool valid,
                                                           const float* rope_cs, const float* rope_hl, float mult) {
  constexpr int nf = D / 4;
  constexpr int kChunks = D / 8;
  const float2* hi = reinterpret_cast<const float2*>(rope_hl);  // [nf][32]
  const float2* lo = hi + nf * 32;                              // [nf][32]
  const uint32_t row_base = smem_u32(tile);
  auto addr = [&](int c16) { return row_base + (c16 >> 3) * 16384 + sw128_off(r, c16 & 7); };
  float amax = 0.f;
  if (!valid) {
#pragma unroll
    for (int c16 = 0; c16 < kChunks; ++c16) sts128(addr(c16), make_uint4(0, 0, 0, 0));
    return 0.f;
  }
  if (p.x < 0) {
#pragma unroll
    for (int c16 = 0; c16 < kChunks; ++c16) {
      uint4 v = lds128(addr(c16));
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y0 = kScale ? bf16_lo(w[e]) * mult : bf16_lo(w[e]);
        const float y1 = kScale ? bf16_hi(w[e]) * mult : bf16_hi(w[e]);
        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        w[e] = pack_f16(y0, y1);
      }
      sts128(addr(c16), v);
    }
    return amax;
  }
  const float2* full = reinterpret_cast<const float2*>(rope_cs) + static_cast<size_t>(p.x) * nf;
  const int hc = p.y >> 5, lc = p.y & 31;
  // first half: (cos, sin) from the full table at p.x; second half: the two
  // two-level factors of p.y
  auto load = [&](int c16, uint4& v, float2 (&a)[4], float2 (&b)[4]) {
    const int k0 = ((c16 * 8) % (D / 2)) / 2;
    v = lds128(addr(c16));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (c16 >= kChunks / 2) {
        a[e] = __ldg(hi + (k0 + e) * 32 + hc);
        b[e] = __ldg(lo + (k0 + e) * 32 + lc);
      } else {
        a[e] = __ldg(full + k0 + e);
        b[e] = make_float2(1.f, 0.f);
      }
    }
  };
  uint4 v_cur;
  float2 a_cur[4], b_cur[4];
  load(0, v_cur, a_cur, b_cur);
#pragma unroll
  for (int c16 = 0; c16 < kChunks; ++c16) {
    uint4 v_nxt;
    float2 a_nxt[4], b_nxt[4];
    if (c16 + 1 < kChunks) load(c16 + 1, v_nxt, a_nxt, b_nxt);
    uint32_t* w = reinterpret_cast<uint32_t*>(&v_cur);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float c = a_cur[e].x, s = a_cur[e].y;
      if (c16 >= kChunks / 2) {
        c = fmaf(a_cur[e].x, b_cur[e].x, -a_cur[e].y * b_cur[e].y);
        s = fmaf(a_cur[e].y, b_cur[e].x, a_cur[e].x * b_cur[e].y);
      }
      if (kScale) {
        c *= mult;
        s *= mult;
      }
      const float x0 = bf16_lo(w[e]), x1 = bf16_hi(w[e]);
      const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
      amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
      w[e] = pack_f16(y0, y1);
    }
    sts128(addr(c16), v_cur);
    if (c16 + 1 < kChunks) {
      v_cur = v_nxt;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a_cur[e] = a_nxt[e];
        b_cur[e] = b_nxt[e];
      }
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
