// Varlen joint attention backward with fused 2D RoPE (tcgen05 + TMA).
//
// Gradient of O = softmax(s R(Q) R(K)^T) V per sample and head with respect
// to the un-rotated Q, K and V (Mage-Flow review, section "Native-Resolution
// MMDiT": the packed attention is trained, so its backward runs on the same
// packs; the row log-sum-exp of the forward lets P be recomputed):
//   P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
//   dS = P * (dP - D), dq~ = s dS k~, dk~ = s dS^T q~, dq = R^T dq~, dk = R^T dk~.
//
// Three kernels:
//   bwd_pre      D = rowsum(dO * O) (float32 [heads, T]); zero the float32 dQ
//                accumulator.
//   bwd_main     one CTA per (sample, head, 128-row K/V tile); loops over the
//                sample's 128-row Q tiles with five tcgen05 MMAs per step:
//                  S^T  = k~ q~^T            (fp16 x fp16, TMEM cols 0..127)
//                  dP^T = V dO^T             (bf16 x bf16, TMEM cols 128..255)
//                  dV  += P^T dO             (bf16, TMEM, accumulated over Q tiles)
//                  dk~ += dS^T q~            (fp16, TMEM, accumulated)
//                  dQ   = dS k~              (fp16, reuses cols 0..D-1 of S^T)
//                P^T (bf16) and dS^T (fp16) are formed by the compute warps
//                in shared memory; dQ is added to the accumulator with vector
//                atomics; the epilogue writes dV and R^T dk~.
//   bwd_dq       dq = R^T (s * accumulator) as bf16.
// As in the forward, the rotated Q/K rows are fp16 (Q pre-scaled by
// s * log2 e) so S^T comes out in exp2 units.
#include "attn_common.cuh"

namespace mf {
namespace {

constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kRopeWarp0 = 6;
constexpr int kRopeThreads = 64;
constexpr int kComputeThreads = 128;
constexpr int kThreads = 8 * 32;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSqBytes = kTile * kTile * 2;  // P^T / dS^T tile
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffP = kOffDO + kTileBytes;
  static constexpr int kOffDS = kOffP + kSqBytes;
  static constexpr int kOffRow = kOffDS + kSqBytes;      // [2][2][128] float: lse2, D
  static constexpr int kSmemBytes = kOffRow + 2 * 2 * kTile * 4;
  static constexpr int kDynSmem = kSmemBytes + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D, kColDQ = 0;
  static constexpr uint32_t kTmemCols = 512;
};

// ---------------------------------------------------------------- bwd_pre
// One thread per (token, head, 8-column chunk); a group of D/8 lanes reduces
// one row.  Also zeroes the matching 8 accumulator floats.
template <int D>
__global__ void bwd_pre_kernel(const BwdArgs a) {
  constexpr int kChunks = D / 8;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rows = static_cast<long long>(a.g.total_tokens) * a.g.heads;
  const long long row = gid / kChunks;
  const int ch = static_cast<int>(gid % kChunks);
  float acc = 0.f;
  if (row < rows) {
    const uint4 o = reinterpret_cast<const uint4*>(a.o)[row * kChunks + ch];
    const uint4 g = reinterpret_cast<const uint4*>(a.dout)[row * kChunks + ch];
    const uint32_t* ow = reinterpret_cast<const uint32_t*>(&o);
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(&g);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      acc += bf16_lo(ow[e]) * bf16_lo(gw[e]) + bf16_hi(ow[e]) * bf16_hi(gw[e]);
    float4* z = reinterpret_cast<float4*>(a.dq_acc) + (row * kChunks + ch) * 2;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kChunks / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && ch == 0) {
    const long long tok = row / a.g.heads;
    const int h = static_cast<int>(row % a.g.heads);
    a.dsum[static_cast<long long>(h) * a.g.total_tokens + tok] = acc;
  }
}

// ---------------------------------------------------------------- bwd_dq
// dq = R^T (s * acc): one thread per (token, head, 8-column chunk).
template <int D>
__global__ void bwd_dq_kernel(const BwdArgs a) {
  constexpr int kChunks = D / 8;
  constexpr int nf = D / 4;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rows = static_cast<long long>(a.g.total_tokens) * a.g.heads;
  if (gid >= rows * kChunks) return;
  const long long row = gid / kChunks;
  const int ch = static_cast<int>(gid % kChunks);
  const long long tok = row / a.g.heads;
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc) + gid * 2;
  const float4 x0 = src[0], x1 = src[1];
  float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  const int2 p = reinterpret_cast<const int2*>(a.g.pos)[tok];
  uint32_t out[4];
  if (p.x >= 0) {
    const int dim0 = ch * 8;
    const int k0 = (dim0 % (D / 2)) / 2;
    const int pp = dim0 >= D / 2 ? p.y : p.x;
    const float4* tab = reinterpret_cast<const float4*>(a.g.rope_cs) + static_cast<size_t>(pp) * (nf / 2) + k0 / 2;
    const float4 c0 = __ldg(tab), c1 = __ldg(tab + 1);
    const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float c = cs[2 * e], s = cs[2 * e + 1];
      const float u0 = x[2 * e] * a.scale, u1 = x[2 * e + 1] * a.scale;
      out[e] = pack_bf16(fmaf(u0, c, u1 * s), fmaf(-u0, s, u1 * c));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = pack_bf16(x[2 * e] * a.scale, x[2 * e + 1] * a.scale);
  }
  reinterpret_cast<uint4*>(a.dq)[gid] = make_uint4(out[0], out[1], out[2], out[3]);
}

// ---------------------------------------------------------------- bwd_main
// 32 fp32 TMEM values of a row chunk -> R^T(p) (mult * v) as bf16 stored at dst.
// The chunk covers columns col0..col0+31 of a D-column row.
template <int D>
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16* dst, const uint32_t (&v)[32], int col0, float mult,
                                                int2 p, const float* rope_cs, bool inverse_rope) {
  constexpr int nf = D / 4;
  uint32_t packed[16];
  if (inverse_rope && p.x >= 0) {
    const int k0 = (col0 % (D / 2)) / 2;  // 16 pairs starting at frequency k0
    const int pp = col0 >= D / 2 ? p.y : p.x;
    const float4* tab = reinterpret_cast<const float4*>(rope_cs) + static_cast<size_t>(pp) * (nf / 2) + k0 / 2;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 cs = __ldg(tab + q);  // pairs 2q, 2q+1
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float c = e ? cs.z : cs.x, s = e ? cs.w : cs.y;
        const int m = 2 * q + e;
        const float u0 = __uint_as_float(v[2 * m]) * mult, u1 = __uint_as_float(v[2 * m + 1]) * mult;
        packed[m] = pack_bf16(fmaf(u0, c, u1 * s), fmaf(-u0, s, u1 * c));
      }
    }
  } else {
#pragma unroll
    for (int m = 0; m < 16; ++m)
      packed[m] = pack_bf16(__uint_as_float(v[2 * m]) * mult, __uint_as_float(v[2 * m + 1]) * mult);
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst + col0);
#pragma unroll
  for (int q = 0; q < 4; ++q) d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                const BwdArgs args) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_kv_full, bar_k_ready, bar_q_full, bar_q_ready, bar_do_full;
  __shared__ uint64_t bar_st_full, bar_ds_ready, bar_dv_done, bar_dk_done, bar_dq_full, bar_dq_free, bar_final;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_range;
  __shared__ WorkItem s_item;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar_kv_full, 1);
    mbar_init(&bar_k_ready, kRopeThreads);
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_ready, kRopeThreads);
    mbar_init(&bar_do_full, 1);
    mbar_init(&bar_st_full, 1);
    mbar_init(&bar_ds_ready, kComputeThreads);
    mbar_init(&bar_dv_done, 1);
    mbar_init(&bar_dk_done, 1);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dq_free, kComputeThreads);
    mbar_init(&bar_final, 1);
    s_abort = 0;
    s_range = 0;
    s_item = decode_item(args.g, blockIdx.x);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = s_tmem;
  const WorkItem w = s_item;             // w.tile = this CTA's K/V tile
  const int kv0 = w.seq_start + w.tile * kTile;
  const int kv_rows = min(kTile, w.len - w.tile * kTile);
  const int n_q = (w.len + kTile - 1) / kTile;
  const int xcol = w.head * D;
  const int T = args.g.total_tokens;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      mbar_arrive_expect_tx(&bar_kv_full, 2 * C::kTileBytes);
      for (int h = 0; h < C::kHalves; ++h) {
        tma_load_2d(smem + C::kOffK + h * 16384, &tk, &bar_kv_full, xcol + h * 64, kv0);
        tma_load_2d(smem + C::kOffV + h * 16384, &tv, &bar_kv_full, xcol + h * 64, kv0);
      }
      int i = 0, issued_do = 0, issued_q = 0;
      for (; i < n_q; ++i) {
        const int y = w.seq_start + i * kTile;
        if (i > 0 && !mbar_wait(&bar_dv_done, (i - 1) & 1, &s_abort)) break;
        mbar_arrive_expect_tx(&bar_do_full, C::kTileBytes);
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_2d(smem + C::kOffDO + h * 16384, &tdo, &bar_do_full, xcol + h * 64, y);
        issued_do = i + 1;
        if (i > 0 && !mbar_wait(&bar_dk_done, (i - 1) & 1, &s_abort)) break;
        mbar_arrive_expect_tx(&bar_q_full, C::kTileBytes);
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_2d(smem + C::kOffQ + h * 16384, &tq, &bar_q_full, xcol + h * 64, y);
        issued_q = i + 1;
      }
      wait_drain(&bar_kv_full, 0);
      if (issued_do) wait_drain(&bar_do_full, (issued_do - 1) & 1);
      if (issued_q) wait_drain(&bar_q_full, (issued_q - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t id_st = idesc_f16(kTile, kTile, false, false);   // k~ q~^T
      constexpr uint32_t id_dp = idesc_bf16(kTile, kTile, false, false);  // V dO^T
      constexpr uint32_t id_dv = idesc_bf16(kTile, D, false, true);       // P^T dO
      constexpr uint32_t id_dk = idesc_f16(kTile, D, false, true);        // dS^T q~
      constexpr uint32_t id_dq = idesc_f16(kTile, D, true, true);         // dS k~
      const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
      const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
      const uint32_t sP = smem_u32(smem + C::kOffP), sDS = smem_u32(smem + C::kOffDS);
      bool ok = mbar_wait(&bar_k_ready, 0, &s_abort) && mbar_wait(&bar_kv_full, 0, &s_abort);
      for (int i = 0; ok && i < n_q; ++i) {
        const uint32_t ph = i & 1;
        if (!mbar_wait(&bar_q_ready, ph, &s_abort) || !mbar_wait(&bar_do_full, ph, &s_abort) ||
            (i > 0 && !mbar_wait(&bar_dq_free, (i - 1) & 1, &s_abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColS, smem_desc(sK + off, 16, 1024), smem_desc(sQ + off, 16, 1024), id_st, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColDP, smem_desc(sV + off, 16, 1024), smem_desc(sDO + off, 16, 1024), id_dp, kk > 0);
        }
        mma_commit(&bar_st_full);
        if (!mbar_wait(&bar_ds_ready, ph, &s_abort)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColDV, smem_desc(sP + off, 16, 1024), smem_desc(sDO + kk * 2048, 16384, 1024), id_dv,
                 (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_dv_done);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColDK, smem_desc(sDS + off, 16, 1024), smem_desc(sQ + kk * 2048, 16384, 1024), id_dk,
                 (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_dk_done);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          mma_ss(tmem + C::kColDQ, smem_desc(sDS + kk * 2048, 16384, 1024), smem_desc(sK + kk * 2048, 16384, 1024),
                 id_dq, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_dq_full);
      }
      mma_commit(&bar_final);
      wait_drain(&bar_final, 0);
    }
  } else if (warp >= kRopeWarp0) {
    // fp16 k~ (once) and fp16 q~ * s * log2 e (per Q tile); rows past the
    // sample's end are zeroed.
    const int r = tid - kRopeWarp0 * 32;
    const int2* pos = reinterpret_cast<const int2*>(args.g.pos);
    const float* tab = args.g.rope_cs;
    float amax = 0.f;
    if (mbar_wait(&bar_kv_full, 0, &s_abort)) {
      uint8_t* kt = smem + C::kOffK;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int rr = r + u * kRopeThreads;
        if (rr < kv_rows) amax = fmaxf(amax, rope_row_to_f16<D>(kt, rr, pos[kv0 + rr], tab, 1.0f));
        else zero_row<D>(kt, rr);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bar_k_ready);
      for (int i = 0; i < n_q; ++i) {
        const int q0 = w.seq_start + i * kTile;
        const int q_rows = min(kTile, w.len - i * kTile);
        int2 pq[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) pq[u] = (r + u * kRopeThreads < q_rows) ? pos[q0 + r + u * kRopeThreads] : make_int2(-1, -1);
        if (!mbar_wait(&bar_q_full, i & 1, &s_abort)) break;
        uint8_t* qt = smem + C::kOffQ;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int rr = r + u * kRopeThreads;
          if (rr < q_rows) amax = fmaxf(amax, rope_row_to_f16<D>(qt, rr, pq[u], tab, args.scale_log2));
          else zero_row<D>(qt, rr);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar_q_ready);
      }
    }
    if (!(amax <= kF16Max)) s_range = 1;
  } else {
    // Compute warpgroup: thread t owns K/V row t of the tile (TMEM lane t)
    // for S^T, dP^T, dV, dk~, and query row t of the current Q tile for dQ.
    const int t = tid;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float* s_row = reinterpret_cast<float*>(smem + C::kOffRow);  // [2][lse2 | D][128]
    const bool kv_valid = t < kv_rows;
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      const int q0 = w.seq_start + i * kTile;
      const int q_rows = min(kTile, w.len - i * kTile);
      float* lse2 = s_row + (i & 1) * 2 * kTile;
      float* dsm = lse2 + kTile;
      {
        const bool vq = t < q_rows;
        const size_t idx = static_cast<size_t>(w.head) * T + q0 + t;
        lse2[t] = vq ? args.lse[idx] * kLog2e : 0.f;
        dsm[t] = vq ? args.dsum[idx] : 0.f;
      }
      named_bar_sync(1, kComputeThreads);
      if (!warp_wait(&bar_st_full, i & 1, &s_abort)) { ok = false; break; }
      tc_fence_after();
      uint8_t* Pt = smem + C::kOffP;
      uint8_t* DSt = smem + C::kOffDS;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tl + C::kColS + c * 32, sv);
        tmem_ld32(tl + C::kColDP + c * 32, dp);
        tmem_wait_ld(sv);
        tmem_wait_ld(dp);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int qq = c * 32 + 2 * e + u;
            const bool valid = kv_valid && qq < q_rows;
            const float p = valid ? ex2_approx(__uint_as_float(sv[2 * e + u]) - lse2[qq]) : 0.f;
            pv[u] = p;
            dv[u] = valid ? p * (__uint_as_float(dp[2 * e + u]) - dsm[qq]) : 0.f;
          }
          pw[e] = pack_bf16(pv[0], pv[1]);
          dw[e] = pack_f16(dv[0], dv[1]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = c * 4 + q;
          const uint32_t off = (ch >> 3) * 16384 + sw128_off(t, ch & 7);
          *reinterpret_cast<uint4*>(Pt + off) = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
          *reinterpret_cast<uint4*>(DSt + off) = make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_ds_ready);
      if (!warp_wait(&bar_dq_full, i & 1, &s_abort)) { ok = false; break; }
      tc_fence_after();
      // dQ row t (query q0 + t) += TMEM lane t, columns 0..D-1.
      float4* dst = reinterpret_cast<float4*>(args.dq_acc + (static_cast<size_t>(q0 + t) * args.g.heads + w.head) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + C::kColDQ + c * 32, v);
        tmem_wait_ld(v);
        if (t < q_rows) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            atomicAdd(dst + c * 8 + q, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
        }
      }
      tc_fence_before();
      mbar_arrive(&bar_dq_free);
    }
    if (ok && n_q > 0) {
      // The last dq_full commit covers every MMA, so dV and dk~ are final.
      tc_fence_after();
      const size_t rowoff = (static_cast<size_t>(kv0 + t) * args.g.heads + w.head) * D;
      const int2 pk = kv_valid ? reinterpret_cast<const int2*>(args.g.pos)[kv0 + t] : make_int2(-1, -1);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + C::kColDV + c * 32, v);
        tmem_wait_ld(v);
        if (kv_valid)
          store_row_chunk<D>(reinterpret_cast<__nv_bfloat16*>(args.dv) + rowoff, v, c * 32, 1.0f, pk,
                             args.g.rope_cs, false);
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tl + C::kColDK + c * 32, v);
        tmem_wait_ld(v);
        // TMEM holds dS^T (q~ * s * log2 e); dk~ = s dS^T q~ = ln 2 * TMEM.
        if (kv_valid)
          store_row_chunk<D>(reinterpret_cast<__nv_bfloat16*>(args.dk) + rowoff, v, c * 32, kLn2, pk,
                             args.g.rope_cs, true);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && (s_abort || s_range))
    atomicOr(args.g.status, (s_abort ? kStatusTimeout : 0) | (s_range ? kStatusRange : 0));
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  using C = BwdCfg<D>;
  const long long chunks = static_cast<long long>(a.g.total_tokens) * a.g.heads * (D / 8);
  const int threads = 256;
  const long long blocks = (chunks + threads - 1) / threads;
  bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  if (ev0 && (e = cudaEventRecord(ev0, stream)) != cudaSuccess) return e;
  bwd_main_kernel<D><<<a.g.n_items, kThreads, C::kDynSmem, stream>>>(tq, tk, tv, tdo, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev1 && (e = cudaEventRecord(ev1, stream)) != cudaSuccess) return e;
  bwd_dq_kernel<D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, int head_dim, cudaStream_t stream,
                            cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (a.g.n_items <= 0) return cudaSuccess;
  if (head_dim == 128) return launch_bwd_d<128>(a, tq, tk, tv, tdo, stream, ev_start, ev_stop);
  return launch_bwd_d<64>(a, tq, tk, tv, tdo, stream, ev_start, ev_stop);
}

}  // namespace mf
