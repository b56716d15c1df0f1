// Varlen joint attention forward with fused 2D RoPE (tcgen05 + TMA).
//
// Per sample i and head h: O = softmax(s * R(Q) R(K)^T) V over the sample's
// own tokens, LSE = its row log-sum-exp (Mage-Flow review, section
// "Native-Resolution MMDiT": joint attention of concatenated text and image
// tokens, confined to each sample by cumulative offsets; Hugging Face paper
// page, Highlights "System-level speed": per-sample 2D RoPE).
//
// Two kernels:
//   fwd_pre    q~ = s log2(e) R(q) and k~ = R(k) as fp16 [T, heads, D], once per
//              token (the main kernel streams each K tile once per Q-tile pair
//              of its sample, so rotating there repeated the work that many
//              times).  fp16 keeps the rotation's rounding 8x below bf16's,
//              and with s log2(e) folded into q~ the logits land in TMEM
//              already in exp2 units.  A value beyond the fp16 range raises
//              the range status.
//   attn_fwd   one CTA owns a pair of 128-row Q tiles (256 query rows) of one
//              (sample, head) and streams the sample's 128-row k~/V tiles.
//              12 warps in three warpgroups:
//     WG0, WG1   softmax of Q tile 0 / 1: thread t owns query row t (TMEM
//                lane t); online softmax in the exp2 domain, O rescaled in
//                TMEM only when the running max grows by more than 2^8; P
//                written back into its S columns of TMEM as packed bf16;
//                epilogue O / l, LSE
//     WG2        warp 8: TMA producer (the q~ pair once; k~ into a 3-slot ring
//                freed right after both logit MMAs, V into a 2-slot ring);
//                warp 9: TMEM owner and single-thread MMA issuer:
//                  S_a = q~_a k~_j^T (smem x smem), O_a += P_a V_j (P from
//                  TMEM), in the ping-pong order QK_0(j), PV_1(j-1), QK_1(j),
//                  PV_0(j), so one tile's softmax overlaps the other tile's
//                  MMAs
// TMEM: S0 | S1 | O0 | O1 (128 + 128 + D + D columns of 512).  Registers are
// rebalanced with setmaxnreg (the warpgroup shares sum to the launch's
// 3 x 168 per thread).
// Rows past the sample's end: S columns past the end are masked to -inf
// (their P is exactly 0, so the V rows they meet add nothing), and Q rows
// past the end are never stored.
#include "attn_common.cuh"

namespace mf {
namespace {

template <int D>
struct FwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kOffQ = 0;                                 // Q0 | Q1
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kSmemBytes = kOffV + kVStages * kTileBytes;
  static constexpr int kDynSmem = kSmemBytes + 1024;
  static constexpr uint32_t kColS = 0;        // S_a at a * 128
  static constexpr uint32_t kColO = 256;      // O_a at 256 + a * D
  static constexpr uint32_t kTmemCols = 512;
};

constexpr int kThreads = 12 * 32;
constexpr int kCtrlWG = 2;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTimeoutKernelFwd = 1;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;
// Per-thread register shares after setmaxnreg; they add up to the launch's
// 3 x 168 per thread (65,536 / 384 rounded down to a multiple of 8).
constexpr uint32_t kRegsSoftmax = 208, kRegsCtrl = 88;
static_assert(2 * kRegsSoftmax + kRegsCtrl <= 3 * 168, "warpgroup register shares exceed the launch's registers");

// ---------------------------------------------------------------- fwd_pre
// One thread per (token, head, 8-column chunk): the chunk's four rotation
// pairs of q and k (rope_pair_cs: by the latent row and column, and with 3
// axes the frame; text tokens are not rotated), rounded to fp16.
template <int D>
__global__ void fwd_pre_kernel(const FwdArgs a) {
  constexpr int kChunks = D / 8;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rows = static_cast<long long>(a.g.total_tokens) * a.g.heads;
  if (gid >= rows * kChunks) return;
  const long long tok = gid / kChunks / a.g.heads;
  const int ch = static_cast<int>(gid % kChunks);
  // q, k rows are qk_stride elements apart (a plain tensor or a QKV row)
  const long long src = (tok * a.qk_stride + (gid / kChunks % a.g.heads) * D) / 8 + ch;
  const uint4 qv = reinterpret_cast<const uint4*>(a.q)[src];
  const uint4 kv = reinterpret_cast<const uint4*>(a.k)[src];
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(&qv);
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(&kv);
  const int2 p = reinterpret_cast<const int2*>(a.g.pos)[tok];
  const int fr = a.g.frame[tok];
  uint32_t qo[4], ko[4];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 cs = rope_pair_cs<D>(a.g, 4 * ch + e, p, fr);
    const float c = cs.x, sn = cs.y;
    const float q0 = bf16_lo(qw[e]), q1 = bf16_hi(qw[e]);
    const float k0 = bf16_lo(kw[e]), k1 = bf16_hi(kw[e]);
    const float yq0 = fmaf(q0, c, -q1 * sn) * a.scale_log2, yq1 = fmaf(q0, sn, q1 * c) * a.scale_log2;
    const float yk0 = fmaf(k0, c, -k1 * sn), yk1 = fmaf(k0, sn, k1 * c);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(yq0), fabsf(yq1)), fmaxf(fabsf(yk0), fabsf(yk1))));
    qo[e] = pack_f16(yq0, yq1);
    ko[e] = pack_f16(yk0, yk1);
  }
  reinterpret_cast<uint4*>(a.q_rot)[gid] = make_uint4(qo[0], qo[1], qo[2], qo[3]);
  reinterpret_cast<uint4*>(a.k_rot)[gid] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
  if (!(amax <= kF16Max)) atomicOr(a.g.status, kStatusRange);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // One block of barriers, so that a timeout record can name one by its
  // position: q_full 0, final 1, k_full 2.., k_free, v_full, v_free, s_full,
  // p_full, pv_done (two each for the last three).
  struct Bars {
    uint64_t q_full, final;
    uint64_t k_full[C::kKStages], k_free[C::kKStages];
    uint64_t v_full[C::kVStages], v_free[C::kVStages];
    uint64_t s_full[2], p_full[2], pv_done[2];
  };
  __shared__ Bars bars;
  uint64_t& bar_q_full = bars.q_full;
  uint64_t& bar_final = bars.final;
  uint64_t(&bar_k_full)[C::kKStages] = bars.k_full;
  uint64_t(&bar_k_free)[C::kKStages] = bars.k_free;
  uint64_t(&bar_v_full)[C::kVStages] = bars.v_full;
  uint64_t(&bar_v_free)[C::kVStages] = bars.v_free;
  uint64_t(&bar_s_full)[2] = bars.s_full;
  uint64_t(&bar_p_full)[2] = bars.p_full;
  uint64_t(&bar_pv_done)[2] = bars.pv_done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ WorkItem s_item;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
  if (tid == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_final, 1);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_free[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_full[i], kTile);
      mbar_init(&bar_pv_done[i], 1);
    }
    s_abort = 0;
    s_item = decode_item<2 * kTile>(args.g, blockIdx.x);
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
  const WorkItem w = s_item;                   // w.tile = pair index
  const int q0 = w.seq_start + w.tile * 2 * kTile;
  const int rows_left = w.len - w.tile * 2 * kTile;
  const int n_kv = (w.len + kTile - 1) / kTile;
  const int xcol = w.head * D;

  if (wg == kCtrlWG) {
    regs_dec<kRegsCtrl>();
    if (warp == kProducerWarp && lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(&bar_q_full, 2 * C::kTileBytes);
      for (int a = 0; a < 2; ++a)
        for (int h = 0; h < C::kHalves; ++h)
          tma_load_2d(smem + C::kOffQ + a * C::kTileBytes + h * 16384, &tq, &bar_q_full, xcol + h * 64,
                      q0 + a * kTile);
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      const bool drop = (args.g.debug & kDebugDropFwdKV) != 0;  // timeout-path tests only
      // K_j goes out one step ahead of V_j: the logit MMAs need it first.
      for (int j = 0; ok && j <= n_kv; ++j) {
        const int jk = j;  // K tile issued in this step
        if (jk < n_kv) {
          const int s = jk % C::kKStages;
          if (jk >= C::kKStages && !mbar_wait(&bar_k_free[s], (jk / C::kKStages - 1) & 1, &s_abort)) break;
          if (!drop) {
            mbar_arrive_expect_tx(&bar_k_full[s], C::kTileBytes);
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_2d(smem + C::kOffK + s * C::kTileBytes + h * 16384, &tk, &bar_k_full[s], xcol + h * 64,
                          w.seq_start + jk * kTile);
            k_issued = jk + 1;
          }
        }
        const int jv = j - 1;  // V tile issued in this step
        if (jv >= 0) {
          const int s = jv % C::kVStages;
          if (jv >= C::kVStages && !mbar_wait(&bar_v_free[s], (jv / C::kVStages - 1) & 1, &s_abort)) break;
          if (!drop) {
            mbar_arrive_expect_tx(&bar_v_full[s], C::kTileBytes);
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_2d(smem + C::kOffV + s * C::kTileBytes + h * 16384, &tv, &bar_v_full[s], xcol + h * 64,
                          w.seq_start + jv * kTile);
            v_issued = jv + 1;
          }
        }
      }
      // Let this CTA's own copies land before its shared memory is released.
      wait_drain(&bar_q_full, 0);
      for (int j = max(0, k_issued - C::kKStages); j < k_issued; ++j)
        wait_drain(&bar_k_full[j % C::kKStages], (j / C::kKStages) & 1);
      for (int j = max(0, v_issued - C::kVStages); j < v_issued; ++j)
        wait_drain(&bar_v_full[j % C::kVStages], (j / C::kVStages) & 1);
    } else if (warp == kMmaWarp && lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kTile, kTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kTile, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::kOffQ);
      const uint32_t sK = smem_u32(smem + C::kOffK);
      const uint32_t sV = smem_u32(smem + C::kOffV);
      auto issue_qk = [&](int a, int j) {
        const uint32_t kb = sK + (j % C::kKStages) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + C::kColS + a * kTile, sdesc<16, 1024>(sQ + a * C::kTileBytes + off), sdesc<16, 1024>(kb + off),
                 idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s_full[a]);
      };
      auto issue_pv = [&](int a, int j) {
        const uint32_t vb = sV + (j % C::kVStages) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(tmem + C::kColO + a * D, tmem + C::kColS + a * kTile + kk * 8, sdesc<16384, 1024>(vb + kk * 2048),
                 idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_pv_done[a]);
      };
      // Ping-pong order QK_0(j), PV_1(j-1), QK_1(j), PV_0(j), QK_0(j+1), ...:
      // each tile's softmax overlaps the other tile's MMAs, and the two
      // softmaxes never run at the same time.  S_a holds P_a until PV_a has
      // read it, so QK_a waits for the tile's previous PV_a.
      bool ok = mbar_wait(&bar_q_full, 0, &s_abort) && mbar_wait(&bar_k_full[0], 0, &s_abort);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j > 0) {
          if (!mbar_wait(&bar_p_full[1], (j - 1) & 1, &s_abort)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, j - 1);
          mma_commit(&bar_v_free[(j - 1) % C::kVStages]);
          if (!mbar_wait(&bar_pv_done[1], (j - 1) & 1, &s_abort)) { ok = false; break; }
          tc_fence_after();
        }
        issue_qk(1, j);
        mma_commit(&bar_k_free[j % C::kKStages]);
        if (!mbar_wait(&bar_p_full[0], j & 1, &s_abort) ||
            !mbar_wait(&bar_v_full[j % C::kVStages], (j / C::kVStages) & 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(0, j);
        if (j + 1 < n_kv) {
          if (!mbar_wait(&bar_k_full[(j + 1) % C::kKStages], ((j + 1) / C::kKStages) & 1, &s_abort) ||
              !mbar_wait(&bar_pv_done[0], j & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_qk(0, j + 1);
        }
      }
      if (ok && mbar_wait(&bar_p_full[1], (n_kv - 1) & 1, &s_abort)) {
        tc_fence_after();
        issue_pv(1, n_kv - 1);
        mma_commit(&bar_v_free[(n_kv - 1) % C::kVStages]);
      }
      mma_commit(&bar_final);
      wait_drain(&bar_final, 0);
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // Softmax warpgroup `a`: thread `row` owns query row `row` of Q tile a.
    const int a = wg;
    const int row = tid & (kTile - 1);
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colS = C::kColS + a * kTile, colO = C::kColO + a * D;
    const int last_valid = w.len - (n_kv - 1) * kTile;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(&bar_s_full[a], j & 1, &s_abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tl + colS + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_wait_ld(sr[c]);
      if (j == n_kv - 1 && last_valid < kTile) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i >= last_valid) sr[c][i] = __float_as_uint(-INFINITY);
      }
      // row max: three-input max into four independent chains
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          m4[i & 3] = fmax3(m4[i & 3], __uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
      const float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
      const float m_new = fmaxf(m_run, mx);
      const bool need = m_new > m_run + kRescaleThreshold;
      const bool rescale_o = j > 0 && __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (need) {
        alpha = ex2_approx(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
      }
      const uint64_t neg_m2 = f2_pack(-m_run, -m_run);
      uint64_t rs2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      // P as packed bf16 pairs over S's first 64 columns (all of S is in
      // registers already), 16 columns at a time so the logits die early;
      // S - m and the row sum run on fp32 pairs.
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          f2_unpack(f2_add(f2_pack(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), neg_m2), x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          rs2[i & 1] = f2_add(rs2[i & 1], f2_pack(p0, p1));
          pw[i] = pack_bf16(p0, p1);
        }
        tmem_st16(tl + colS + c * 16, pw);
      }
      float rsa, rsb, rsc, rsd;
      f2_unpack(rs2[0], rsa, rsb);
      f2_unpack(rs2[1], rsc, rsd);
      const float rs = (rsa + rsb) + (rsc + rsd);
      if (rescale_o) {
        // O_a is stable once PV_a(j-1) has completed; PV_a(j) is not issued
        // before p_full below.
        if (!warp_wait(&bar_pv_done[a], (j - 1) & 1, &s_abort)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + colO + c * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tl + colO + c * 32, o);
        }
      }
      tmem_wait_st();
      l_run += rs;
      tc_fence_before();
      mbar_arrive(&bar_p_full[a]);
    }
    if (ok) ok = warp_wait(&bar_pv_done[a], (n_kv - 1) & 1, &s_abort);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const int qrow = a * kTile + row;
      const bool valid = qrow < rows_left;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(args.o) +
                            (static_cast<size_t>(q0 + qrow) * args.g.heads + w.head) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + colO + c * 32, o);
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
        args.lse[static_cast<size_t>(w.head) * args.g.total_tokens + q0 + qrow] = (m_run + __log2f(l_run)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && s_abort) {
    const uint32_t a = static_cast<uint32_t>(s_abort) - 1u, base = smem_u32(&bars);
    record_timeout(args.g.status, args.g.timeout_info, kTimeoutKernelFwd,
                   a >= base && a < base + sizeof(Bars) ? (a - base) / 8 : 0xfffu);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  using C = FwdCfg<D>;
  const long long chunks = static_cast<long long>(a.g.total_tokens) * a.g.heads * (D / 8);
  fwd_pre_kernel<D><<<static_cast<unsigned>((chunks + 255) / 256), 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
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
