// Varlen joint attention forward with fused 2D RoPE (tcgen05 + TMA).
//
// Per sample i and head h: O = softmax(s * R(Q) R(K)^T) V over the sample's
// own tokens, LSE = its row log-sum-exp (Mage-Flow review, section
// "Native-Resolution MMDiT": joint attention of concatenated text and image
// tokens, confined to each sample by cumulative offsets; Hugging Face paper
// page, Highlights "System-level speed": per-sample 2D RoPE).
//
// One CTA owns one 128-row Q tile of one (sample, head) and streams the
// sample's 128-row K/V tiles:
//   warp 4      TMA producer: Q once, then K/V tiles into a 2-stage ring
//   warps 6-7   RoPE: rotate the Q tile and each landed K tile in shared
//               memory (two rows per thread), so no rotated copy reaches HBM.
//               The rotated rows are stored as fp16 (Q pre-multiplied by
//               softmax_scale * log2 e): the logit MMA runs fp16 x fp16 ->
//               fp32, whose 11-bit significand keeps the rounding of the
//               rotated operands 8x below bf16's; S lands in TMEM already in
//               exp2 units.  P V stays bf16 x bf16 (V is a bf16 input).
//   warp 5      MMA issuer: S_j = Q K_j^T into TMEM (two S buffers), then
//               O += P_j V_j into a TMEM accumulator
//   warps 0-3   softmax: thread t owns query row t (TMEM lane t); online
//               softmax in the exp2 domain, P_j written to shared memory as
//               bf16, O rescaled in TMEM only when the running max grows by
//               more than 2^8, epilogue O / l and LSE
// Rows past the sample's end inside the last K/V tile are masked to -inf;
// Q rows past the end are computed but never stored.
#include "attn_common.cuh"

namespace mf {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPBytes = kTile * kTile * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + 2 * kTileBytes;
  static constexpr int kOffP = kOffV + 2 * kTileBytes;
  static constexpr int kSmemBytes = kOffP + 2 * kPBytes;
  static constexpr int kDynSmem = kSmemBytes + 1024;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kTmemCols = 512;
};

// 8 warps = 2 per SM sub-partition, which leaves up to 255 registers per
// thread for the softmax warps (128 fp32 logits live per thread).
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kRopeWarp0 = 6;
constexpr int kRopeThreads = 64;
constexpr int kThreads = 8 * 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_q_full, bar_q_rot, bar_final;
  __shared__ uint64_t bar_k_full[2], bar_k_rot[2], bar_v_full[2], bar_kv_empty[2];
  __shared__ uint64_t bar_s_full[2], bar_p_full[2], bar_pv_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_range;
  __shared__ WorkItem s_item;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_rot, kRopeThreads);
    mbar_init(&bar_final, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_rot[i], kRopeThreads);
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_kv_empty[i], 1);
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_full[i], kTile);
      mbar_init(&bar_pv_done[i], 1);
    }
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
  const WorkItem w = s_item;
  const int q0 = w.seq_start + w.tile * kTile;
  const int q_rows = min(kTile, w.len - w.tile * kTile);
  const int n_kv = (w.len + kTile - 1) / kTile;
  const int xcol = w.head * D;  // column of this head in the [T, heads*D] view

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(&bar_q_full, C::kTileBytes);
      for (int h = 0; h < C::kHalves; ++h)
        tma_load_2d(smem + C::kOffQ + h * 16384, &tq, &bar_q_full, xcol + h * 64, q0);
      int j = 0;
      for (; j < n_kv; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&bar_kv_empty[s], ((j >> 1) - 1) & 1, &s_abort)) break;
        const int y = w.seq_start + j * kTile;
        mbar_arrive_expect_tx(&bar_k_full[s], C::kTileBytes);
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_2d(smem + C::kOffK + s * C::kTileBytes + h * 16384, &tk, &bar_k_full[s], xcol + h * 64, y);
        mbar_arrive_expect_tx(&bar_v_full[s], C::kTileBytes);
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_2d(smem + C::kOffV + s * C::kTileBytes + h * 16384, &tv, &bar_v_full[s], xcol + h * 64, y);
      }
      // Let this CTA's own copies land before its shared memory is released.
      wait_drain(&bar_q_full, 0);
      for (int jj = max(0, j - 2); jj < j; ++jj) {
        wait_drain(&bar_k_full[jj & 1], (jj >> 1) & 1);
        wait_drain(&bar_v_full[jj & 1], (jj >> 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kTile, kTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kTile, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::kOffQ);
      const uint32_t sK = smem_u32(smem + C::kOffK);
      const uint32_t sV = smem_u32(smem + C::kOffV);
      const uint32_t sP = smem_u32(smem + C::kOffP);
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1;
        if (!mbar_wait(&bar_p_full[bb], (jj >> 1) & 1, &s_abort)) return false;
        if (!mbar_wait(&bar_v_full[bb], (jj >> 1) & 1, &s_abort)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t ad = smem_desc(sP + bb * C::kPBytes + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(sV + bb * C::kTileBytes + kk * 2048, 16384, 1024);
          mma_ss(tmem + C::kColO, ad, bd, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_pv_done[bb]);
        mma_commit(&bar_kv_empty[bb]);
        return true;
      };
      bool ok = mbar_wait(&bar_q_rot, 0, &s_abort);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&bar_k_rot[s], (j >> 1) & 1, &s_abort)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&bar_p_full[s], ((j - 2) >> 1) & 1, &s_abort)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + (s ? C::kColS1 : C::kColS0), smem_desc(sQ + off, 16, 1024),
                 smem_desc(sK + s * C::kTileBytes + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s_full[s]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(n_kv - 1);
      mma_commit(&bar_final);
      wait_drain(&bar_final, 0);
    }
  } else if (warp >= kRopeWarp0) {
    // Thread r prepares rows r and r + 64 of each tile for the logit MMA:
    // fp16 of R(pos) q * scale * log2(e) for Q, fp16 of R(pos) k for K;
    // rows past the sample's end are zeroed.
    const int r = tid - kRopeWarp0 * 32;
    const int2* pos = reinterpret_cast<const int2*>(args.g.pos);
    const float* tab = args.g.rope_cs;
    float amax = 0.f;
    int2 pq0 = make_int2(-1, -1), pq1 = make_int2(-1, -1);
    if (r < q_rows) pq0 = pos[q0 + r];
    if (r + kRopeThreads < q_rows) pq1 = pos[q0 + r + kRopeThreads];
    if (mbar_wait(&bar_q_full, 0, &s_abort)) {
      uint8_t* qt = smem + C::kOffQ;
      if (r < q_rows) amax = fmaxf(amax, rope_row_to_f16<D>(qt, r, pq0, tab, args.scale_log2));
      else zero_row<D>(qt, r);
      if (r + kRopeThreads < q_rows) amax = fmaxf(amax, rope_row_to_f16<D>(qt, r + kRopeThreads, pq1, tab, args.scale_log2));
      else zero_row<D>(qt, r + kRopeThreads);
      fence_proxy_async_smem();
      mbar_arrive(&bar_q_rot);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        const int kr = j * kTile + r;
        int2 pk0 = make_int2(-1, -1), pk1 = make_int2(-1, -1);
        if (kr < w.len) pk0 = pos[w.seq_start + kr];
        if (kr + kRopeThreads < w.len) pk1 = pos[w.seq_start + kr + kRopeThreads];
        if (!mbar_wait(&bar_k_full[s], (j >> 1) & 1, &s_abort)) break;
        uint8_t* kt = smem + C::kOffK + s * C::kTileBytes;
        if (kr < w.len) amax = fmaxf(amax, rope_row_to_f16<D>(kt, r, pk0, tab, 1.0f));
        else zero_row<D>(kt, r);
        if (kr + kRopeThreads < w.len) amax = fmaxf(amax, rope_row_to_f16<D>(kt, r + kRopeThreads, pk1, tab, 1.0f));
        else zero_row<D>(kt, r + kRopeThreads);
        fence_proxy_async_smem();
        mbar_arrive(&bar_k_rot[s]);
      }
    }
    if (!(amax <= kF16Max)) s_range = 1;
  } else {
    // Softmax warpgroup: thread `tid` owns query row `tid`.
    const int row = tid;
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int last_valid = w.len - (n_kv - 1) * kTile;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      if (!warp_wait(&bar_s_full[b], (j >> 1) & 1, &s_abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + (b ? C::kColS1 : C::kColS0) + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);
      if (j == n_kv - 1 && last_valid < kTile) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i >= last_valid) sr[c][i] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));
      const float m_new = fmaxf(m_run, mx);
      // P buffer b is free once PV_{j-2} has completed.
      if (j >= 2 && !warp_wait(&bar_pv_done[b], ((j - 2) >> 1) & 1, &s_abort)) { ok = false; break; }
      const bool need = m_new > m_run + kRescaleThreshold;
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (!warp_wait(&bar_pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, &s_abort)) { ok = false; break; }
        tc_fence_after();
        const float f = need ? ex2_approx(m_run - m_new) : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + C::kColO + c * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tl + C::kColO + c * 32, o);
        }
        tmem_wait_st();
      }
      if (need) {
        l_run *= ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      const float neg_m = -m_run;
      float rs = 0.f;
      uint8_t* Pb = smem + C::kOffP + b * C::kPBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p[e] = ex2_approx(__uint_as_float(sr[c][q * 8 + e]) + neg_m);
            rs += p[e];
          }
          const int ch = c * 4 + q;  // 16-byte chunk 0..15 of the 256-byte P row
          uint4 v = make_uint4(pack_bf16(p[0], p[1]), pack_bf16(p[2], p[3]), pack_bf16(p[4], p[5]),
                               pack_bf16(p[6], p[7]));
          *reinterpret_cast<uint4*>(Pb + (ch >> 3) * 16384 + sw128_off(row, ch & 7)) = v;
        }
      }
      l_run += rs;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_full[b]);
    }
    if (ok) ok = warp_wait(&bar_pv_done[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1, &s_abort);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const bool valid = row < q_rows;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(args.o) +
                            (static_cast<size_t>(q0 + row) * args.g.heads + w.head) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + C::kColO + c * 32, o);
        tmem_wait_ld(o);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            dst[q] = make_uint4(pack_bf16(__uint_as_float(o[q * 8 + 0]) * inv_l, __uint_as_float(o[q * 8 + 1]) * inv_l),
                                pack_bf16(__uint_as_float(o[q * 8 + 2]) * inv_l, __uint_as_float(o[q * 8 + 3]) * inv_l),
                                pack_bf16(__uint_as_float(o[q * 8 + 4]) * inv_l, __uint_as_float(o[q * 8 + 5]) * inv_l),
                                pack_bf16(__uint_as_float(o[q * 8 + 6]) * inv_l, __uint_as_float(o[q * 8 + 7]) * inv_l));
          }
        }
      }
      if (valid)
        args.lse[static_cast<size_t>(w.head) * args.g.total_tokens + q0 + row] = (m_run + __log2f(l_run)) * kLn2;
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
cudaError_t launch_fwd_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  using C = FwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  if (ev0 && (e = cudaEventRecord(ev0, stream)) != cudaSuccess) return e;
  attn_fwd_kernel<D><<<a.g.n_items, kThreads, C::kDynSmem, stream>>>(tq, tk, tv, a);
  e = cudaGetLastError();
  if (e == cudaSuccess && ev1) e = cudaEventRecord(ev1, stream);
  return e;
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, int head_dim, cudaStream_t stream,
                            cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (a.g.n_items <= 0) return cudaSuccess;
  if (head_dim == 128) return launch_fwd_d<128>(a, tq, tk, tv, stream, ev_start, ev_stop);
  return launch_fwd_d<64>(a, tq, tk, tv, stream, ev_start, ev_stop);
}

}  // namespace mf
