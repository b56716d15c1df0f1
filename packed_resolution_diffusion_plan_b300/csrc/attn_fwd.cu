// Varlen joint attention forward with fused 2D RoPE (tcgen05 + TMA).
//
// Per sample i and head h: O = softmax(s * R(Q) R(K)^T) V over the sample's
// own tokens, LSE = its row log-sum-exp (Mage-Flow review, section
// "Native-Resolution MMDiT": joint attention of concatenated text and image
// tokens, confined to each sample by cumulative offsets; Hugging Face paper
// page, Highlights "System-level speed": per-sample 2D RoPE).
//
// Two kernels:
//   fwd_pre    k~ = R(k) as fp16 [T, heads, D], once per token: the main
//              kernel streams each K tile once per Q-tile pair of its sample,
//              so rotating the streamed operand there would repeat the work
//              that many times.  fp16 keeps the rotation's rounding 8x below
//              bf16's.  A value beyond the fp16 range raises the range
//              status.  Thread 0 also zeroes the main kernel's work counter.
//   attn_fwd   a persistent kernel, one CTA per SM.  A work item is a pair of
//              128-row Q tiles (256 query rows) of one (sample, head); the
//              CTAs take items from a global counter in the plan's
//              longest-sample-first order, so the uneven per-sample L_i^2 is
//              balanced by whichever SM comes free first.  Per item the CTA
//              loads the raw bf16 Q pair, rotates it in shared memory (the
//              prologue: q~ = s log2(e) R(q) as fp16, so the logits land in
//              TMEM in exp2 units and no rotated Q copy goes to HBM), and
//              streams the sample's 128-row k~/V tiles.
//              12 warps in three warpgroups:
//     WG0, WG1   Q tile 0 / 1: thread t owns query row t (TMEM lane t).  The
//                prologue rotates the tile in place (thread t its row t);
//                then online softmax in the exp2 domain, O rescaled in TMEM
//                only when the running max grows by more than 2^8; P written
//                back into its S columns of TMEM as packed bf16; epilogue
//                O / l, LSE (while the other tile's MMAs go on)
//     WG2        warp 8: work counter and TMA producer (the raw Q pair per
//                item; k~ into a 3-slot ring freed right after both logit
//                MMAs, V into a 2-slot ring; the rings run on across items);
//                warp 9: TMEM owner and single-thread MMA issuer:
//                  S_a = q~_a k~_j^T (smem x smem), O_a += P_a V_j (P from
//                  TMEM), in the ping-pong order QK_0(j), PV_1(j-1), QK_1(j),
//                  PV_0(j), so one tile's softmax overlaps the other tile's
//                  MMAs;
//                warps 10-11: the zeroing of the last V tile's rows past the
//                sample's end
// Work items pass from the producer to the other roles through a two-slot
// ring in shared memory.  TMEM: S0 | S1 | O0 | O1 (128 + 128 + D + D columns
// of 512).  Registers are rebalanced with setmaxnreg (the warpgroup shares
// sum to the launch's 3 x 168 per thread).
// Rows past the sample's end: S columns past the end are replaced by -inf
// (their P is exactly 0), and the V rows they meet are zeroed, so that no
// value of the next sample, finite or not, reaches this sample's O; Q rows
// past the end are zeroed and never stored.
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
constexpr int kPrepWarp0 = 10;          // warps 10, 11: the V tail of ragged items
constexpr int kPrepThreads = 64;
constexpr uint32_t kTimeoutKernelFwd = 1;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
constexpr float kLn2 = 0.6931471805599453f;
// Arrivals on an item slot's "read" barrier: the MMA thread, the two prep
// warps and the eight softmax warps (one per warp).
constexpr uint32_t kItemReaders = 1 + 2 + 8;
// Per-thread register shares after setmaxnreg; they add up to the launch's
// 3 x 168 per thread (65,536 / 384 rounded down to a multiple of 8).
constexpr uint32_t kRegsSoftmax = 208, kRegsCtrl = 88;
static_assert(2 * kRegsSoftmax + kRegsCtrl <= 3 * 168, "warpgroup register shares exceed the launch's registers");

// ---------------------------------------------------------------- fwd_pre
// One thread per (token, head, 8-column chunk): the chunk's four rotation
// pairs of k (rope_pair_cs: by the latent row and column, and with 3 axes the
// frame; text tokens are not rotated), rounded to fp16.
template <int D>
__global__ void fwd_pre_kernel(const FwdArgs a) {
  constexpr int kChunks = D / 8;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid == 0) *a.work_counter = 0;
  const long long rows = static_cast<long long>(a.g.total_tokens) * a.g.heads;
  if (gid >= rows * kChunks) return;
  const long long tok = gid / kChunks / a.g.heads;
  const int ch = static_cast<int>(gid % kChunks);
  // k rows are qk_stride elements apart (a plain tensor or a QKV row)
  const long long src = (tok * a.qk_stride + (gid / kChunks % a.g.heads) * D) / 8 + ch;
  const uint4 kv = reinterpret_cast<const uint4*>(a.k)[src];
  const uint32_t* kw = reinterpret_cast<const uint32_t*>(&kv);
  const int2 p = reinterpret_cast<const int2*>(a.g.pos)[tok];
  const int fr = a.g.frame[tok];
  uint32_t ko[4];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 cs = rope_pair_cs<D>(a.g, 4 * ch + e, p, fr);
    const float c = cs.x, sn = cs.y;
    const float k0 = bf16_lo(kw[e]), k1 = bf16_hi(kw[e]);
    const float yk0 = fmaf(k0, c, -k1 * sn), yk1 = fmaf(k0, sn, k1 * c);
    amax = fmaxf(amax, fmaxf(fabsf(yk0), fabsf(yk1)));
    ko[e] = pack_f16(yk0, yk1);
  }
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
  // position: final 0, item_full 1-2, item_empty 3-4, q_full 5-6, q_ready
  // 7-8, q_empty 9-10, v_tail 11-12, v_fixed 13-14, k_full 15.., k_free,
  // v_full, v_free, s_full, p_full, pv_done (two each for the last three).
  // The last V tile of an item whose sample ends inside it (a "ragged" item)
  // lands on v_tail instead of its slot's v_full (whose phase the producer
  // completes with a plain arrival, so that the slot's phases stay in step):
  // the prep warps wait for that tile on v_tail, zero its rows past the
  // sample's end and arrive on v_fixed, which the MMA waits for instead.
  // Ragged item n uses v_tail / v_fixed n % 2: with one of each, two short
  // ragged items in a row could complete two phases before a waiter looked
  // (the next tail needs only the other V slot), and a parity wait would
  // then take the later phase for the one it wants.
  struct Bars {
    uint64_t final;
    uint64_t item_full[2], item_empty[2];
    uint64_t q_full[2], q_ready[2], q_empty[2];
    uint64_t v_tail[2], v_fixed[2];
    uint64_t k_full[C::kKStages], k_free[C::kKStages];
    uint64_t v_full[C::kVStages], v_free[C::kVStages];
    uint64_t s_full[2], p_full[2], pv_done[2];
  };
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ WorkItem s_item[2];   // decoded by the producer; sample < 0: no more work

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
  if (tid == 0) {
    mbar_init(&bars.final, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.item_full[i], 1);
      mbar_init(&bars.item_empty[i], kItemReaders);
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_ready[i], kTile);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], kTile);
      mbar_init(&bars.pv_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.v_tail[i], 1);
      mbar_init(&bars.v_fixed[i], kPrepThreads);
    }
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_free[i], 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_free[i], 1);
    }
    s_abort = 0;
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
  volatile int* abort_flag = &s_abort;

  // Item k of this CTA: wait for its slot and read it.  A whole warp
  // (whole_warp: the softmax and prep warps, whose waits must agree across
  // the warp) arrives once, from lane 0 after every lane has read; a single
  // thread (the MMA issuer) arrives itself.  w->sample < 0: no more work.
  // Returns false when the wait gave up.
  auto take_item = [&](int k, WorkItem* w, bool whole_warp) -> bool {
    const bool got = whole_warp ? warp_wait(&bars.item_full[k & 1], (k >> 1) & 1, abort_flag)
                                : mbar_wait(&bars.item_full[k & 1], (k >> 1) & 1, abort_flag);
    if (!got) return false;
    *w = s_item[k & 1];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(&bars.item_empty[k & 1]);
    return true;
  };

  if (wg == kCtrlWG) {
    regs_dec<kRegsCtrl>();
    if (warp == kProducerWarp && lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      const bool drop = (args.g.debug & kDebugDropFwdKV) != 0;  // timeout-path tests only
      // Per-CTA step counters are 32-bit (a CTA runs far fewer than 2^31 K/V
      // steps): the issuing thread derives ring slots and phases from them
      // every step, and a 64-bit division by the stage count is a long
      // multi-instruction sequence.
      int kc = 0, vc = 0;            // K / V tiles of the previous items (the rings' positions)
      int k_issued = 0, v_issued = 0;  // K / V loads issued so far
      int q_issued = 0;                    // Q tile loads issued so far
      int tail_issued = 0;                 // loads issued on v_tail
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (k >= 2 && !mbar_wait(&bars.item_empty[k & 1], ((k >> 1) - 1) & 1, abort_flag)) break;
        const int item = atomicAdd(args.work_counter, 1);
        WorkItem w;
        if (item < args.g.n_items) {
          w = decode_item<2 * kTile>(args.g, item);
        } else {
          w.sample = -1;
        }
        s_item[k & 1] = w;
        mbar_arrive(&bars.item_full[k & 1]);   // release: the slot write is visible to the waiters
        if (w.sample < 0) break;
        const int q0 = w.seq_start + w.tile * 2 * kTile;
        const int n_kv = (w.len + kTile - 1) / kTile;
        const bool ragged = w.len % kTile != 0;
        const int xcol = w.head * D;
        auto load_q = [&](int a) -> bool {
          if (k >= 1 && !mbar_wait(&bars.q_empty[a], (k - 1) & 1, abort_flag)) return false;
          mbar_arrive_expect_tx(&bars.q_full[a], C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(smem + C::kOffQ + a * C::kTileBytes + h * 16384, &tq, &bars.q_full[a], xcol + h * 64,
                        q0 + a * kTile);
          return true;
        };
        auto load_k = [&](int j) -> bool {
          const int g = kc + j;
          const int s = static_cast<int>(g % C::kKStages);
          if (g >= C::kKStages && !mbar_wait(&bars.k_free[s], (g / C::kKStages - 1) & 1, abort_flag)) return false;
          if (drop) return true;
          mbar_arrive_expect_tx(&bars.k_full[s], C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(smem + C::kOffK + s * C::kTileBytes + h * 16384, &tk, &bars.k_full[s], xcol + h * 64,
                        w.seq_start + j * kTile);
          k_issued = g + 1;
          return true;
        };
        auto load_v = [&](int j) -> bool {
          const int g = vc + j;
          const int s = static_cast<int>(g % C::kVStages);
          if (g >= C::kVStages && !mbar_wait(&bars.v_free[s], (g / C::kVStages - 1) & 1, abort_flag)) return false;
          if (drop) return true;
          uint64_t* bar = &bars.v_full[s];
          if (ragged && j == n_kv - 1) {
            mbar_arrive(bar);           // the slot's phase, without the data
            bar = &bars.v_tail[tail_issued & 1];
            ++tail_issued;
          }
          mbar_arrive_expect_tx(bar, C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(smem + C::kOffV + s * C::kTileBytes + h * 16384, &tv, bar, xcol + h * 64,
                        w.seq_start + j * kTile);
          v_issued = g + 1;
          return true;
        };
        // Q_0, K_0, Q_1, then K_j one step ahead of V_{j-1}: the logit MMAs
        // need K first, and Q_1 is free only after the previous item's last
        // QK_1.
        ok = load_q(0);
        if (ok) q_issued = 2 * k + 1;
        ok = ok && load_k(0) && load_q(1);
        if (ok) q_issued = 2 * k + 2;
        for (int j = 1; ok && j <= n_kv; ++j) {
          if (j < n_kv) ok = load_k(j);
          if (ok) ok = load_v(j - 1);
        }
        kc += n_kv;
        vc += n_kv;
      }
      // Let this CTA's own copies land before its shared memory is released
      // (q_issued counts Q tile loads: item k's tile a is load 2k + a).
      for (int i = q_issued > 2 ? q_issued - 2 : 0; i < q_issued; ++i) wait_drain(&bars.q_full[i & 1], (i >> 1) & 1, abort_flag);
      for (int g = k_issued > C::kKStages ? k_issued - C::kKStages : 0; g < k_issued; ++g)
        wait_drain(&bars.k_full[g % C::kKStages], (g / C::kKStages) & 1, abort_flag);
      for (int g = v_issued > C::kVStages ? v_issued - C::kVStages : 0; g < v_issued; ++g)
        wait_drain(&bars.v_full[g % C::kVStages], (g / C::kVStages) & 1, abort_flag);
      for (int t = tail_issued > 2 ? tail_issued - 2 : 0; t < tail_issued; ++t)
        wait_drain(&bars.v_tail[t & 1], (t >> 1) & 1, abort_flag);
    } else if (warp == kMmaWarp && lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kTile, kTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kTile, D, false, true);
      // Descriptor low halves of the operand tiles (K-major Q and K: 16-byte
      // leading and 1024-byte stride; MN-major V: two 64-element halves 16 KB
      // apart), built once per MMA group from an opaque base and advanced
      // per MMA by a constant add: the issuing thread's work per MMA is one
      // add and the issue itself, since issuing is what bounds this thread.
      const uint32_t s0 = smem_u32(smem);
      constexpr uint32_t kHi = sdesc_hi<1024>();
      auto klo = [&](int off) { return sdesc_lo<16>(opaque_u32(s0 + off)); };
      auto mlo = [&](int off) { return sdesc_lo<16384>(opaque_u32(s0 + off)); };
      auto issue_qk = [&](int a, int g) {
        const uint32_t qa = klo(C::kOffQ + a * C::kTileBytes);
        const uint32_t kb = klo(C::kOffK + static_cast<int>(g % C::kKStages) * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss_lh(tmem + C::kColS + a * kTile, qa + off, kb + off, kHi, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full[a]);
      };
      auto issue_pv = [&](int a, int g, bool first) {
        const uint32_t vb = mlo(C::kOffV + static_cast<int>(g % C::kVStages) * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts_lh(tmem + C::kColO + a * D, tmem + C::kColS + a * kTile + kk * 8, vb + kk * 128, kHi, idesc_pv,
                    (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bars.pv_done[a]);
      };
      int gs = 0;   // K/V steps of the previous items: the position of every per-step barrier
      int n_ragged = 0;   // items whose last V tile had rows past the sample's end
      bool ok = true;
      for (int k = 0; ok; ++k) {
        WorkItem w;
        if (!take_item(k, &w, false) || w.sample < 0) break;
        const int n_kv = (w.len + kTile - 1) / kTile;
        const bool ragged = w.len % kTile != 0;
        // Ping-pong order QK_0(j), PV_1(j-1), QK_1(j), PV_0(j), QK_0(j+1), ...:
        // each tile's softmax overlaps the other tile's MMAs, and the two
        // softmaxes never run at the same time.  S_a holds P_a until PV_a has
        // read it, so QK_a waits for the tile's previous PV_a (across items
        // too: the previous item's last PV_a).
        auto v_ready = [&](int j) -> bool {
          const int g = gs + j;
          if (ragged && j == n_kv - 1) return mbar_wait(&bars.v_fixed[n_ragged & 1], (n_ragged >> 1) & 1, abort_flag);
          return mbar_wait(&bars.v_full[g % C::kVStages], (g / C::kVStages) & 1, abort_flag);
        };
        ok = mbar_wait(&bars.q_ready[0], k & 1, abort_flag) &&
             mbar_wait(&bars.k_full[gs % C::kKStages], (gs / C::kKStages) & 1, abort_flag) &&
             (gs == 0 || mbar_wait(&bars.pv_done[0], (gs - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        issue_qk(0, gs);
        if (n_kv == 1) mma_commit(&bars.q_empty[0]);
        for (int j = 0; ok && j < n_kv; ++j) {
          const int g = gs + j;
          if (j > 0) {
            if (!mbar_wait(&bars.p_full[1], (g - 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_pv(1, g - 1, j == 1);
            mma_commit(&bars.v_free[(g - 1) % C::kVStages]);
            if (!mbar_wait(&bars.pv_done[1], (g - 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
          } else {
            if (!mbar_wait(&bars.q_ready[1], k & 1, abort_flag) ||
                (gs > 0 && !mbar_wait(&bars.pv_done[1], (gs - 1) & 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          issue_qk(1, g);
          mma_commit(&bars.k_free[g % C::kKStages]);
          if (j == n_kv - 1) mma_commit(&bars.q_empty[1]);
          if (!mbar_wait(&bars.p_full[0], g & 1, abort_flag) || !v_ready(j)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, g, j == 0);
          if (j + 1 < n_kv) {
            if (!mbar_wait(&bars.k_full[(g + 1) % C::kKStages], ((g + 1) / C::kKStages) & 1, abort_flag) ||
                !mbar_wait(&bars.pv_done[0], g & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk(0, g + 1);
            if (j + 2 == n_kv) mma_commit(&bars.q_empty[0]);
          }
        }
        if (ok && mbar_wait(&bars.p_full[1], (gs + n_kv - 1) & 1, abort_flag)) {
          tc_fence_after();
          issue_pv(1, gs + n_kv - 1, n_kv == 1);
          mma_commit(&bars.v_free[(gs + n_kv - 1) % C::kVStages]);
        } else {
          ok = false;
        }
        gs += n_kv;
        if (ragged) ++n_ragged;
      }
      mma_commit(&bars.final);
      wait_drain(&bars.final, 0, abort_flag);
    } else if (warp >= kPrepWarp0) {
      // The V tail of every ragged item (64 threads).
      const int t = tid - kPrepWarp0 * 32;
      int vc = 0;
      int n_ragged = 0;
      for (int k = 0;; ++k) {
        WorkItem w;
        if (!take_item(k, &w, true) || w.sample < 0) break;
        const int n_kv = (w.len + kTile - 1) / kTile;
        const int last_valid = w.len - (n_kv - 1) * kTile;
        if (last_valid < kTile) {
          // Zero the last V tile's rows past the sample's end (their P is 0,
          // but 0 times a non-finite value is not).
          const int g = vc + n_kv - 1;
          if (!warp_wait(&bars.v_tail[n_ragged & 1], (n_ragged >> 1) & 1, abort_flag)) break;
          uint8_t* vt = smem + C::kOffV + static_cast<int>(g % C::kVStages) * C::kTileBytes;
          for (int c = t; c < (kTile - last_valid) * 8 * C::kHalves; c += kPrepThreads) {
            const int r = last_valid + c / (8 * C::kHalves);
            const int rest = c % (8 * C::kHalves);
            *reinterpret_cast<uint4*>(vt + (rest >> 3) * 16384 + r * 128 + (rest & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          mbar_arrive(&bars.v_fixed[n_ragged & 1]);
          ++n_ragged;
        }
        vc += n_kv;
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // Softmax warpgroup `a`: thread `row` owns query row `row` of Q tile a.
    const int a = wg;
    const int row = tid & (kTile - 1);
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colS = C::kColS + a * kTile, colO = C::kColO + a * D;
    // Item k's prologue: take the item and rotate this warpgroup's Q tile
    // (rows past the sample's end zeroed) once its raw rows have landed.  It
    // runs for the next item before this item's epilogue, so that the next
    // logit MMA overlaps the epilogue.
    auto prologue = [&](int k, WorkItem* w) -> bool {
      if (!take_item(k, w, true)) return false;
      if (w->sample < 0) return true;
      const int qrow = a * kTile + row;
      const bool valid = qrow < w->len - w->tile * 2 * kTile;
      // the RoPE factors first: their loads overlap the wait for the tile
      float cs[D / 8][8];
      rope_row_cs<D, D / 8>(0, w->seq_start + w->tile * 2 * kTile + qrow, valid, args.g, cs);
      if (!warp_wait(&bars.q_full[a], k & 1, abort_flag)) return false;
      const float amax = rotate_row_f16<D / 8>(smem + C::kOffQ + a * C::kTileBytes, row, 0, valid,
                                               args.scale_log2, cs);
      if (!(amax <= kF16Max)) atomicOr(args.g.status, kStatusRange);
      fence_proxy_async_smem();
      mbar_arrive(&bars.q_ready[a]);
      return true;
    };
    int gs = 0;
    WorkItem w;
    bool ok = prologue(0, &w);
    for (int k = 0; ok && w.sample >= 0; ++k) {
      const int q0 = w.seq_start + w.tile * 2 * kTile;
      const int rows_left = w.len - w.tile * 2 * kTile;
      const int n_kv = (w.len + kTile - 1) / kTile;
      const int last_valid = w.len - (n_kv - 1) * kTile;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        const int g = gs + j;
        if (!warp_wait(&bars.s_full[a], g & 1, abort_flag)) { ok = false; break; }
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
          if (!warp_wait(&bars.pv_done[a], (g - 1) & 1, abort_flag)) { ok = false; break; }
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
        mbar_arrive(&bars.p_full[a]);
      }
      WorkItem next;
      if (ok) ok = prologue(k + 1, &next);
      if (ok) ok = warp_wait(&bars.pv_done[a], (gs + n_kv - 1) & 1, abort_flag);
      if (!ok) break;
      // Epilogue: O_a / l and the LSE.  The next item's PV_a, which
      // overwrites O_a, is issued only after this warpgroup's next p_full.
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
      tc_fence_before();
      if (valid)
        args.lse[static_cast<size_t>(w.head) * args.g.total_tokens + q0 + qrow] = (m_run + __log2f(l_run)) * kLn2;
      gs += n_kv;
      w = next;
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
  const int grid = a.g.n_items < sm_count() ? a.g.n_items : sm_count();
  attn_fwd_kernel<D><<<grid, kThreads, C::kDynSmem, stream>>>(tq, tk, tv, a);
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
