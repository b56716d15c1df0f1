// Varlen joint attention backward with fused 2D RoPE (tcgen05 + TMA).
//
// Gradient of O = softmax(s R(Q) R(K)^T) V per sample and head with respect
// to the un-rotated Q, K and V (Mage-Flow review, section "Native-Resolution
// MMDiT": the packed attention is trained, so its backward runs on the same
// packs; the row log-sum-exp of the forward lets P be recomputed):
//   P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
//   dS = P * (dP - D), dq = R^T (s dS R(k)), dk = R^T (s dS^T R(q)).
// The logit operands are fp16: q~ = s log2(e) R(q), a copy streamed from HBM,
// and k~ = R(k), rotated in the main kernel's prologue; dk~ = dS^T q~ and
// dq~ = dS k~ are taken back by dk_mult = ln 2 and dq_mult = s.
//
// Three kernels:
//   bwd_pre      D = rowsum(dO * O) (float32 [heads, T]); zero the float32 dQ
//                accumulator; q~ = s log2(e) R(q) as fp16 [T, heads, D],
//                rotated once per token (the main kernel streams every Q tile
//                once per K/V tile of its sample); zero the work counter.
//   bwd_main     a persistent kernel, one CTA per SM.  A work item is one
//                (sample, head, 128-row K/V tile); the CTAs take items from a
//                global counter in the plan's longest-sample-first order, so
//                the uneven per-sample L_i^2 is balanced by whichever SM comes
//                free first.  Per item the CTA loads the raw K tile and V,
//                rotates K in shared memory (the prologue: k~ = R(k) as fp16,
//                rows past the sample's end zeroed, no rotated K copy in
//                HBM), and streams the sample's 128-row q~/dO tiles (a
//                two-slot q~ ring, one dO slot; both run on across items).
//                Per Q tile i, five tcgen05 MMAs (TMEM columns: A = 0..127,
//                B = 128..255, dV = 256.., dK = 256 + D..):
//                  S^T_i  = k~ q~_i^T        fp16, smem x smem -> A
//                  dP^T_i = V dO_i^T         bf16, smem x smem -> B
//                  dV    += P^T_i dO_i       bf16, P^T from TMEM (A) x smem
//                  dk~   += dS^T_i q~_i      fp16, dS^T from TMEM (A) x smem
//                  dQ_i   = dS_i k~          fp16, smem x smem -> B; with
//                           head_dim 128 it is formed transposed (k~^T dS^T,
//                           TMEM lane = dimension), so that a warp's stores
//                           into the staging tile cover one 128-byte row
//                issued in the order dV_i, dK_i, dQ_i, S^T_{i+1}, dP^T_{i+1}:
//                the compute warps move dQ_i out of B while S^T_{i+1} runs.
//                12 warps:
//                  WG0, WG1  thread r owns K/V row r (TMEM lane r), WG c the
//                            query columns 64c..64c+63 (and, in the prologue,
//                            the dims c D/2 .. of its K row): P^T =
//                            exp2(S^T - LSE2) written back over its S^T
//                            columns as packed bf16, dS^T = P^T * (dP^T - D)
//                            as fp16 into TMEM (beside P^T, for dK) and shared
//                            memory (for dQ); the dQ epilogue (TMEM ->
//                            staging tile, half the tile each); at the end of
//                            the item dV and R^T dk~
//                  WG2       warp 8 work counter and TMA producer, warp 9
//                            TMEM owner and MMA issuer, warp 10 the dQ
//                            reducer: with head_dim 128 each half of dQ_i is
//                            staged in shared memory by its compute warpgroup
//                            (one in the staging tile, one in the q~_i slot,
//                            idle from dK_i until the producer refills it) and
//                            added into the float accumulator by one TMA
//                            reduce, so the compute warps never wait on the
//                            reduction traffic; warp 11 the per-tile -LSE2 / -D
//                            rows and, when the sample ends inside its last Q
//                            tile, the zeroing of that tile's q~ and dO rows
//                            past the end (so that no value of the next
//                            sample, finite or not, reaches this one)
//   bwd_dq       dq = R^T (dq_mult * accumulator) as bf16.
#include "attn_common.cuh"

namespace mf {
namespace {

constexpr int kThreads = 12 * 32;
constexpr int kCtrlWG = 2;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kReduceWarp = 10;
constexpr int kRowWarp = 11;
constexpr float kLog2e = 1.4426950408889634f;
// Per-thread register shares after setmaxnreg; they add up to the launch's
// 3 x 168 per thread (65,536 / 384 rounded down to a multiple of 8).
constexpr uint32_t kRegsCompute = 216, kRegsCtrl = 72;
static_assert(2 * kRegsCompute + kRegsCtrl <= 3 * 168, "warpgroup register shares exceed the launch's registers");

// Barriers and CTA-wide scalars of bwd_main, kept in dynamic shared memory
// after the tiles (the kernel has no static shared memory, so the dynamic
// base is the start of the CTA's window and the tiles stay 1024-aligned).
// A timeout record names a barrier by its position here: kv_full 0, kv_ready
// 1, kv_empty 2, acc_full 3, fin 4, item_full 5-6, item_empty 7-8, q_full
// 9-10, q_ready 11-12, q_free 13-14, do_full 15, do_free 16, q_tail 17-18,
// do_tail 19-20, tail_fixed 21-22, s_full 23, p_ready 24-25, dp_full 26,
// ds_ready 27-28, a_free 29, dq_full 30, dq_free 31, stage_full 32-33,
// stage_free 34, q_issued 35.
// The last Q tile of an item whose sample ends inside it (a "ragged" item)
// lands on q_tail / do_tail instead of its slots' q_full / do_full (whose
// phases the producer completes with plain arrivals, so that they stay in
// step); the row warp zeroes its rows past the end and arrives on
// tail_fixed, which the MMA issuer waits for instead.  Ragged item n uses
// the tail barriers n % 2: with one set, two short ragged items in a row
// could complete two phases of a tail barrier before its waiter looked (the
// next tail needs only the other q~ slot), and a parity wait would then
// take the later phase for the one it wants.
constexpr uint32_t kBwdBarriers = 36;
constexpr uint32_t kTimeoutKernelBwd = 2;
// Arrivals on an item slot's "read" barrier: the MMA thread, the reducer
// thread (head_dim 128 only: with 64, dQ leaves by atomics and the reducer
// warp has no role), the row warp and the eight compute warps (one per warp).
template <int D>
constexpr uint32_t item_readers() {
  return 1 + (D == 128 ? 1 : 0) + 1 + 8;
}
struct BwdCtl {
  uint64_t kv_full, kv_ready, kv_empty, acc_full, fin;
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[2], q_ready[2], q_free[2], do_full, do_free;
  uint64_t q_tail[2], do_tail[2], tail_fixed[2];
  uint64_t s_full, p_ready[2], dp_full, ds_ready[2], a_free, dq_full, dq_free;
  uint64_t stage_full[2], stage_free, q_issued;
  uint32_t tmem;
  int abort;
  WorkItem item[2];          // decoded by the producer; sample < 0: no more work
};

template <int D>
struct BwdCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSqBytes = kTile * kTile * 2;     // dS^T tile (fp16)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;       // 2 slots
  static constexpr int kOffDO = kOffQ + 2 * kTileBytes;  // 1 slot
  static constexpr int kOffDS = kOffDO + kTileBytes;
  static constexpr int kOffStage = kOffDS + kSqBytes;    // float [64 queries][D]: half a dQ tile
  static constexpr int kOffRow = kOffStage + 64 * D * 4; // [2 slots][LSE2[128] | D[128]] float
  static constexpr int kOffCtl = kOffRow + 2 * 2 * kTile * 4;
  static constexpr int kDynSmem = kOffCtl + 512;
  static constexpr uint32_t kColA = 0, kColB = 128, kColDV = 256, kColDK = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(sizeof(BwdCtl) <= 512, "control block");
  static_assert(offsetof(BwdCtl, tmem) == 8 * kBwdBarriers, "barrier block");
  static_assert(kDynSmem <= 232448, "shared memory");
};

// ---------------------------------------------------------------- bwd_pre
// One thread per (token, head, 8-column chunk); a group of D/8 lanes reduces
// one row of D.  The thread also zeroes the matching 8 accumulator floats and
// writes the chunk of q~ = s log2(e) R(q) as fp16 (rope_pair_cs; text is not
// rotated).  A value beyond the fp16 range raises the range status.
template <int D>
__global__ void bwd_pre_kernel(const BwdArgs a) {
  constexpr int kChunks = D / 8;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid == 0) *a.work_counter = 0;
  const long long rows = static_cast<long long>(a.g.total_tokens) * a.g.heads;
  const long long row = gid / kChunks;
  const int ch = static_cast<int>(gid % kChunks);
  float acc = 0.f;
  if (row < rows) {
    const uint4 o = reinterpret_cast<const uint4*>(a.o)[gid];
    const uint4 g = reinterpret_cast<const uint4*>(a.dout)[gid];
    const uint32_t* ow = reinterpret_cast<const uint32_t*>(&o);
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(&g);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      acc += bf16_lo(ow[e]) * bf16_lo(gw[e]) + bf16_hi(ow[e]) * bf16_hi(gw[e]);
    float4* z = reinterpret_cast<float4*>(a.dq_acc) + gid * 2;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    const long long tok = row / a.g.heads;
    const uint4 qv = reinterpret_cast<const uint4*>(a.q)[gid];
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(&qv);
    const int2 p = reinterpret_cast<const int2*>(a.g.pos)[tok];
    const int fr = a.g.frame[tok];
    uint32_t qo[4];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 cs = rope_pair_cs<D>(a.g, 4 * ch + e, p, fr);
      const float c = cs.x, sn = cs.y;
      const float q0 = bf16_lo(qw[e]), q1 = bf16_hi(qw[e]);
      const float yq0 = fmaf(q0, c, -q1 * sn) * a.scale_log2, yq1 = fmaf(q0, sn, q1 * c) * a.scale_log2;
      amax = fmaxf(amax, fmaxf(fabsf(yq0), fabsf(yq1)));
      qo[e] = pack_f16(yq0, yq1);
    }
    reinterpret_cast<uint4*>(a.q_rot)[gid] = make_uint4(qo[0], qo[1], qo[2], qo[3]);
    if (!(amax <= kF16Max)) atomicOr(a.g.status, kStatusRange);
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
// dq = R^T (dq_mult * acc): the accumulator holds dS k~, so s dS R(k) is
// ln 2 * acc when k~ carries the s log2(e) factor and s * acc when q~ does.
// One thread per (token, head, 8-column chunk).
template <int D>
__global__ void bwd_dq_kernel(const BwdArgs a) {
  constexpr int kChunks = D / 8;
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
  const int fr = a.g.frame[tok];
  uint32_t out[4];
  if (p.x >= 0) {
    float cs[8];
    if (a.g.rope_axes == 2) {
      // 2 axes: the chunk's 4 pairs are consecutive frequencies of one half
      const int dim0 = ch * 8;
      const int k0 = (dim0 % (D / 2)) / 2;
      const int pp = dim0 >= D / 2 ? p.y : p.x;
      const float4* tab = reinterpret_cast<const float4*>(a.g.rope_cs) + static_cast<size_t>(pp) * (D / 8) + k0 / 2;
      const float4 c0 = __ldg(tab), c1 = __ldg(tab + 1);
      cs[0] = c0.x; cs[1] = c0.y; cs[2] = c0.z; cs[3] = c0.w;
      cs[4] = c1.x; cs[5] = c1.y; cs[6] = c1.z; cs[7] = c1.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c = rope_pair_cs<D>(a.g, 4 * ch + e, p, fr);
        cs[2 * e] = c.x;
        cs[2 * e + 1] = c.y;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float c = cs[2 * e], s = cs[2 * e + 1];
      const float u0 = x[2 * e] * a.dq_mult, u1 = x[2 * e + 1] * a.dq_mult;
      out[e] = pack_bf16(fmaf(u0, c, u1 * s), fmaf(-u0, s, u1 * c));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) out[e] = pack_bf16(x[2 * e] * a.dq_mult, x[2 * e + 1] * a.dq_mult);
  }
  reinterpret_cast<uint4*>(a.dq)[gid] = make_uint4(out[0], out[1], out[2], out[3]);
}

// ---------------------------------------------------------------- bwd_main
// 32 fp32 TMEM values of a row chunk -> R^T(p, f) (mult * v) as bf16 stored at
// dst (or mult * v without the rotation).  The chunk covers columns
// col0..col0+31 of a D-column row, i.e. rotation pairs col0/2 .. col0/2 + 15.
template <int D>
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16* dst, const uint32_t (&v)[32], int col0, float mult,
                                                int2 p, int f, const AttnGeom& g, bool inverse_rope) {
  uint32_t packed[16];
  if (inverse_rope && p.x >= 0 && g.rope_axes == 2) {
    // 2 axes: the chunk's 16 pairs are consecutive frequencies of one half,
    // read two pairs per 16-byte load
    const int k0 = (col0 % (D / 2)) / 2;
    const int pp = col0 >= D / 2 ? p.y : p.x;
    const float4* tab = reinterpret_cast<const float4*>(g.rope_cs) + static_cast<size_t>(pp) * (D / 8) + k0 / 2;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 cs = __ldg(tab + q);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float c = e ? cs.z : cs.x, s = e ? cs.w : cs.y;
        const int m = 2 * q + e;
        const float u0 = __uint_as_float(v[2 * m]) * mult, u1 = __uint_as_float(v[2 * m + 1]) * mult;
        packed[m] = pack_bf16(fmaf(u0, c, u1 * s), fmaf(-u0, s, u1 * c));
      }
    }
  } else if (inverse_rope && p.x >= 0) {
#pragma unroll 4
    for (int m = 0; m < 16; ++m) {
      const float2 cs = rope_pair_cs<D>(g, col0 / 2 + m, p, f);
      const float c = cs.x, s = cs.y;
      const float u0 = __uint_as_float(v[2 * m]) * mult, u1 = __uint_as_float(v[2 * m + 1]) * mult;
      packed[m] = pack_bf16(fmaf(u0, c, u1 * s), fmaf(-u0, s, u1 * c));
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
                const __grid_constant__ CUtensorMap tdq, const BwdArgs args) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // The swizzled tiles need a 1024-byte aligned base; every thread sees the
  // same address, so a misaligned window makes the whole CTA leave at once.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(args.g.status, kStatusLayout);
    return;
  }
  BwdCtl& c = *reinterpret_cast<BwdCtl*>(smem + C::kOffCtl);
  float* rowbuf = reinterpret_cast<float*>(smem + C::kOffRow);
  volatile int* abort_flag = &c.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
  if (tid == 0) {
    mbar_init(&c.kv_full, 1);
    mbar_init(&c.kv_ready, 2 * kTile);
    mbar_init(&c.kv_empty, 1);
    mbar_init(&c.acc_full, 1);
    mbar_init(&c.fin, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.item_full[s], 1);
      mbar_init(&c.item_empty[s], item_readers<D>());
      mbar_init(&c.q_full[s], 1);
      mbar_init(&c.q_ready[s], 32);  // the row warp's lanes
      // head_dim 128: dK_i has read the slot, and the reducer has read the
      // dQ_i half staged in it (the producer, the row warp and warpgroup 1's
      // next staging wait on it)
      mbar_init(&c.q_free[s], D == 128 ? 2 : 1);
      mbar_init(&c.stage_full[s], kTile);
    }
    mbar_init(&c.do_full, 1);
    mbar_init(&c.do_free, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.q_tail[s], 1);
      mbar_init(&c.do_tail[s], 1);
      mbar_init(&c.tail_fixed[s], 32);
    }
    mbar_init(&c.s_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.p_ready[s], kTile);    // compute warpgroup s's P^T is in TMEM
      mbar_init(&c.ds_ready[s], kTile);   // its dS^T is in TMEM and shared memory
    }
    mbar_init(&c.dp_full, 1);
    mbar_init(&c.a_free, 1);
    mbar_init(&c.dq_full, 1);
    mbar_init(&c.dq_free, 2 * kTile);
    mbar_init(&c.stage_free, 1);
    mbar_init(&c.q_issued, 1);
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&c.tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = c.tmem;
  const int T = args.g.total_tokens;

  // Item k of this CTA: wait for its slot and read it.  A whole warp
  // (whole_warp: the compute and row warps, whose waits must agree across the
  // warp) arrives once, from lane 0 after every lane has read; a single
  // thread (the MMA issuer, the reducer) arrives itself.  w->sample < 0: no
  // more work.  Returns false when the wait gave up.
  auto take_item = [&](int k, WorkItem* w, bool whole_warp) -> bool {
    const bool got = whole_warp ? warp_wait(&c.item_full[k & 1], (k >> 1) & 1, abort_flag)
                                : mbar_wait(&c.item_full[k & 1], (k >> 1) & 1, abort_flag);
    if (!got) return false;
    *w = c.item[k & 1];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(&c.item_empty[k & 1]);
    return true;
  };

  if (wg == kCtrlWG) {
    regs_dec<kRegsCtrl>();
    if (warp == kProducerWarp && lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      const bool drop = (args.g.debug & kDebugDropBwdQdo) != 0;  // timeout-path tests only
      int gq = 0;            // Q tiles of the previous items (the position of every per-tile barrier)
      int q_loads = 0, do_loads = 0;   // q~ / dO loads issued (the index + 1 of the last)
      int kv_loads = 0, tail_loads = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (k >= 2 && !mbar_wait(&c.item_empty[k & 1], ((k >> 1) - 1) & 1, abort_flag)) break;
        const int item = atomicAdd(args.work_counter, 1);
        WorkItem w;
        if (item < args.g.n_items) {
          w = decode_item<kTile>(args.g, item);
        } else {
          w.sample = -1;
        }
        c.item[k & 1] = w;
        mbar_arrive(&c.item_full[k & 1]);   // release: the slot write is visible to the waiters
        if (w.sample < 0) break;
        const int n_q = (w.len + kTile - 1) / kTile;
        const bool ragged = w.len % kTile != 0;
        const int xcol = w.head * D;
        auto load_q = [&](int i) -> bool {
          const int g = gq + i;
          const int s = static_cast<int>(g & 1);
          if (g >= 2 && !mbar_wait(&c.q_free[s], ((g >> 1) - 1) & 1, abort_flag)) return false;
          if (drop) return true;
          uint64_t* bar = &c.q_full[s];
          if (ragged && i == n_q - 1) {
            mbar_arrive(bar);          // the slot's phase, without the data
            bar = &c.q_tail[tail_loads & 1];
          }
          q_loads = g + 1;
          mbar_arrive_expect_tx(bar, C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(smem + C::kOffQ + s * C::kTileBytes + h * 16384, &tq, bar, xcol + h * 64,
                        w.seq_start + i * kTile);
          return true;
        };
        auto load_do = [&](int i) -> bool {
          const int g = gq + i;
          // dO_i reuses the one slot once dV_{i-1} has read dO_{i-1}.
          if (g >= 1 && !mbar_wait(&c.do_free, (g - 1) & 1, abort_flag)) return false;
          if (drop) return true;
          uint64_t* bar = &c.do_full;
          if (ragged && i == n_q - 1) {
            mbar_arrive(bar);
            bar = &c.do_tail[tail_loads & 1];
            ++tail_loads;
          }
          do_loads = g + 1;
          mbar_arrive_expect_tx(bar, C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_2d(smem + C::kOffDO + h * 16384, &tdo, bar, xcol + h * 64, w.seq_start + i * kTile);
          return true;
        };
        // q~_0 first (its slot frees before the K/V tiles do), then the raw K
        // tile and V once the previous item's last MMAs have read them, then
        // dO_0 and the rest of the stream.
        ok = load_q(0);
        if (ok && k >= 1) ok = mbar_wait(&c.kv_empty, (k - 1) & 1, abort_flag);
        if (ok) {
          const int kv0 = w.seq_start + w.tile * kTile;
          mbar_arrive_expect_tx(&c.kv_full, 2 * C::kTileBytes);
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_2d(smem + C::kOffK + h * 16384, &tk, &c.kv_full, xcol + h * 64, kv0);
            tma_load_2d(smem + C::kOffV + h * 16384, &tv, &c.kv_full, xcol + h * 64, kv0);
          }
          kv_loads = k + 1;
          ok = load_do(0);
        }
        for (int i = 1; ok && i < n_q; ++i) {
          ok = load_q(i) && load_do(i);
          if (ok && i >= 2) mbar_arrive(&c.q_issued);  // the refill of the slot and dO_i are in the TMA queue
        }
        gq += n_q;
      }
      // Let this CTA's own copies land before its shared memory is released.
      if (kv_loads) wait_drain(&c.kv_full, (kv_loads - 1) & 1, abort_flag);
      for (int g = q_loads > 2 ? q_loads - 2 : 0; g < q_loads; ++g) wait_drain(&c.q_full[g & 1], (g >> 1) & 1, abort_flag);
      if (do_loads) wait_drain(&c.do_full, (do_loads - 1) & 1, abort_flag);
      for (int t = tail_loads > 2 ? tail_loads - 2 : 0; t < tail_loads; ++t) {
        wait_drain(&c.q_tail[t & 1], (t >> 1) & 1, abort_flag);
        wait_drain(&c.do_tail[t & 1], (t >> 1) & 1, abort_flag);
      }
    } else if (warp == kMmaWarp && lane == 0) {
      constexpr uint32_t id_st = idesc_f16(kTile, kTile, false, false);   // k~ q~^T
      constexpr uint32_t id_dp = idesc_bf16(kTile, kTile, false, false);  // V dO^T
      constexpr uint32_t id_dv = idesc_bf16(kTile, D, false, true);       // P^T dO
      constexpr uint32_t id_dk = idesc_f16(kTile, D, false, true);        // dS^T q~
      // dQ: head_dim 128 forms dQ^T = k~^T dS^T (M = dimension); head_dim 64
      // forms dQ = dS k~ (M = query row).
      constexpr uint32_t id_dq = D == 128 ? idesc_f16(D, kTile, true, true) : idesc_f16(kTile, D, true, true);
      // Descriptor low halves of the operand tiles (K-major: 16-byte leading
      // and 1024-byte stride; MN-major: two 64-element halves 16 KB apart),
      // rebuilt from an opaque base at each MMA group and advanced per MMA by
      // an add, so that the issuing thread keeps neither every MMA's
      // descriptor in registers (which spills) nor redoes the encoding.
      const uint32_t s0 = smem_u32(smem);
      constexpr uint32_t kHi = sdesc_hi<1024>();
      auto klo = [&](int off) { return sdesc_lo<16>(opaque_u32(s0 + off)); };
      auto mlo = [&](int off) { return sdesc_lo<16384>(opaque_u32(s0 + off)); };
      auto issue_s = [&](int s) {
        const uint32_t a = klo(C::kOffK), b = klo(C::kOffQ + s * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss_lh(tmem + C::kColA, a + off, b + off, kHi, id_st, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dp = [&]() {
        const uint32_t a = klo(C::kOffV), b = klo(C::kOffDO);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss_lh(tmem + C::kColB, a + off, b + off, kHi, id_dp, kk > 0 ? 1u : 0u);
        }
      };
      int gq = 0;
      int n_tail = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        WorkItem w;
        if (!take_item(k, &w, false) || w.sample < 0) break;
        const int n_q = (w.len + kTile - 1) / kTile;
        const bool ragged = w.len % kTile != 0;
        // Q tile i's q~ and dO are in place: its slot's q_full / the dO
        // slot's do_full, or for a ragged item's last tile the row warp's
        // tail_fixed (after the tail's rows past the sample's end are zeroed).
        auto q_in = [&](int i) -> bool {
          const int g = gq + i;
          if (ragged && i == n_q - 1) return mbar_wait(&c.tail_fixed[n_tail & 1], (n_tail >> 1) & 1, abort_flag);
          return mbar_wait(&c.q_full[g & 1], (g >> 1) & 1, abort_flag);
        };
        auto do_in = [&](int i) -> bool {
          const int g = gq + i;
          if (ragged && i == n_q - 1) return true;   // tail_fixed, waited by q_in
          return mbar_wait(&c.do_full, g & 1, abort_flag);
        };
        ok = mbar_wait(&c.kv_ready, k & 1, abort_flag) && q_in(0) &&
             (gq == 0 || mbar_wait(&c.a_free, (gq - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        issue_s(static_cast<int>(gq & 1));
        mma_commit(&c.s_full);
        ok = do_in(0) && (gq == 0 || mbar_wait(&c.dq_free, (gq - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        issue_dp();
        mma_commit(&c.dp_full);
        for (int i = 0; ok && i < n_q; ++i) {
          const int g = gq + i;
          const int s = static_cast<int>(g & 1), s1 = static_cast<int>((g + 1) & 1);
          const bool more = i + 1 < n_q;
          // dV += P^T_i dO_i, with P^T packed in the A columns each compute
          // warpgroup read its S^T from (query 64c.. at column 64c).  Both
          // dV and dK reduce over the tile's queries, of which warpgroup c
          // owns 64c..: each half is issued as soon as its warpgroup's
          // operand is in place (the four MMAs of warpgroup 0's half run
          // while warpgroup 1 still computes).
          for (int cw = 0; cw < 2; ++cw) {
            if (!mbar_wait(&c.p_ready[cw], g & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t b = mlo(C::kOffDO + cw * 64 * 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_lh(tmem + C::kColDV, tmem + C::kColA + 64 * cw + 8 * kk, b + kk * 128, kHi, id_dv,
                        (i > 0 || cw > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(&c.do_free);
          // dk~ += dS^T_i q~_i, with dS^T packed in the A columns beside P^T
          // (query 64c.. at column 64c + 32).
          for (int cw = 0; cw < 2; ++cw) {
            if (!mbar_wait(&c.ds_ready[cw], g & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t b = mlo(C::kOffQ + s * C::kTileBytes + cw * 64 * 128);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts_lh(tmem + C::kColDK, tmem + C::kColA + 32 + 64 * cw + 8 * kk, b + kk * 128, kHi, id_dk,
                        (i > 0 || cw > 0 || kk > 0) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(&c.a_free);  // dV_i and dK_i have read P^T and dS^T out of A
          mma_commit(&c.q_free[s]);
          // dQ_i into B (each compute warpgroup has read its dP^T_i before
          // its ds_ready).
          {
            const uint32_t bk = mlo(C::kOffK), bds = mlo(C::kOffDS);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              if (D == 128)
                mma_ss_lh(tmem + C::kColB, bk + kk * 128, bds + kk * 128, kHi, id_dq, kk > 0 ? 1u : 0u);
              else
                mma_ss_lh(tmem + C::kColB, bds + kk * 128, bk + kk * 128, kHi, id_dq, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&c.dq_full);
          if (!more) break;
          // S^T_{i+1} into A (dV_i and dK_i have read P^T_i and dS^T_i out of
          // it); it runs while the compute warps move dQ_i out of B.
          if (!q_in(i + 1) || !mbar_wait(&c.a_free, g & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          issue_s(s1);
          mma_commit(&c.s_full);
          // dP^T_{i+1} into B once dQ_i has been read out of it.
          if (!do_in(i + 1) || !mbar_wait(&c.dq_free, g & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          issue_dp();
          mma_commit(&c.dp_full);
        }
        // The item's last MMAs read K/V and complete dV, dK: the producer may
        // load the next item's tiles, the compute warps store dV and dK.
        mma_commit(&c.kv_empty);
        mma_commit(&c.acc_full);
        gq += n_q;
        if (ragged) ++n_tail;
      }
      mma_commit(&c.fin);
      wait_drain(&c.fin, 0, abort_flag);
    } else if (D == 128 && warp == kReduceWarp && lane == 0) {
      // Reducer: each staged half of dQ_i (64 queries x D floats) is added
      // into the accumulator by one TMA reduce.  Warpgroup 1's half sits in
      // the q~_i slot (free once dK_i has read it) and goes first; once the
      // TMA has read it the slot returns to the producer, and warpgroup 0's
      // half (in the staging tile) is issued only after the refill of the
      // slot and the next dO load (when the item has them), so that the TMA
      // unit, which takes its work in order, does not hold those loads behind
      // a second reduce.
      tma_prefetch_desc(&tdq);
      int gq = 0, qi_base = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        WorkItem w;
        if (!take_item(k, &w, false) || w.sample < 0) break;
        const int n_q = (w.len + kTile - 1) / kTile;
        for (int i = 0; i < n_q; ++i) {
          const int g = gq + i;
          const int y = w.seq_start + i * kTile;
          if (!mbar_wait(&c.stage_full[1], g & 1, abort_flag)) { ok = false; break; }
          tma_reduce_add_3d(&tdq, smem + C::kOffQ + static_cast<int>(g & 1) * C::kTileBytes, 0, w.head, y + 64);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&c.q_free[g & 1]);
          if (i + 2 < n_q && !mbar_wait(&c.q_issued, (qi_base + i) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait(&c.stage_full[0], g & 1, abort_flag)) { ok = false; break; }
          tma_reduce_add_3d(&tdq, smem + C::kOffStage, 0, w.head, y);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&c.stage_free);
        }
        gq += n_q;
        qi_base += n_q > 2 ? n_q - 2 : 0;
      }
      bulk_wait_group0();
    } else if (warp == kRowWarp) {
      // -LSE2 and -D of Q tile i's rows into the slot's row buffer, once the
      // compute warps are done with tile i - 2 (its dK has completed).
      // Queries past the sample's end get -LSE2 = -inf, hence P = 0, and
      // -D = 0.  For a ragged item's last tile, its q~ and dO rows past the
      // sample's end are zeroed once they land.
      int gq = 0;
      int n_tail = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        WorkItem w;
        if (!take_item(k, &w, true) || w.sample < 0) break;
        const int n_q = (w.len + kTile - 1) / kTile;
        for (int i = 0; i < n_q; ++i) {
          const int g = gq + i;
          const int s = static_cast<int>(g & 1);
          if (g >= 2 && !warp_wait(&c.q_free[s], ((g >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
          const int q0 = w.seq_start + i * kTile;
          const int valid_rows = min(kTile, w.len - i * kTile);
#pragma unroll
          for (int kq = 0; kq < kTile / 32; ++kq) {
            const int r = lane + 32 * kq;
            const bool valid = r < valid_rows;
            const size_t idx = static_cast<size_t>(w.head) * T + q0 + r;
            rowbuf[s * 2 * kTile + r] = valid ? -args.lse[idx] * kLog2e : -INFINITY;
            rowbuf[s * 2 * kTile + kTile + r] = valid ? -args.dsum[idx] : 0.f;
          }
          mbar_arrive(&c.q_ready[s]);
          if (valid_rows < kTile) {
            // the ragged item's last tile (only the last can be short)
            if (!warp_wait(&c.q_tail[n_tail & 1], (n_tail >> 1) & 1, abort_flag) ||
                !warp_wait(&c.do_tail[n_tail & 1], (n_tail >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* qt = smem + C::kOffQ + s * C::kTileBytes;
            uint8_t* dt = smem + C::kOffDO;
            for (int e = lane; e < (kTile - valid_rows) * 8 * C::kHalves; e += 32) {
              const int r = valid_rows + e / (8 * C::kHalves);
              const int rest = e % (8 * C::kHalves);
              const int off = (rest >> 3) * 16384 + r * 128 + (rest & 7) * 16;
              *reinterpret_cast<uint4*>(qt + off) = make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(dt + off) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            mbar_arrive(&c.tail_fixed[n_tail & 1]);
            ++n_tail;
          }
        }
        gq += n_q;
      }
    }
  } else {
    regs_inc<kRegsCompute>();
    // Thread r owns K/V row r (TMEM lane r); warpgroup cw the query columns
    // 64cw .. 64cw + 63 of S^T / dP^T.
    const int cw = wg;
    const int r = tid & (kTile - 1);
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint8_t* dst_ds = smem + C::kOffDS + cw * 16384;
    int gq = 0;
    WorkItem w;
    // dQ of Q tile g (TMEM B) into the float accumulator; warpgroup cw takes
    // half of it (queries 64cw ..) and releases B to the next dP^T as soon as
    // its loads land.  With head_dim 128 both halves are staged in shared
    // memory (float [64 queries][D], TMEM lane r = dimension r) for the
    // reducer's TMA reduce-adds: warpgroup 0's in the staging tile after its
    // next dS, warpgroup 1's right away in the q~ slot, which dK has finished
    // with.
    float dqv[64];
    auto dq_load = [&](int g, int i) -> bool {
      if (!warp_wait(&c.dq_full, g & 1, abort_flag)) return false;
      tc_fence_after();
      if (D == 128) {
        uint32_t v0[32], v1[32];
        tmem_ld32(tl + C::kColB + 64 * cw, v0);
        tmem_ld32(tl + C::kColB + 64 * cw + 32, v1);
        tmem_wait_ld(v0);
        tmem_wait_ld(v1);
        tc_fence_before();
        mbar_arrive(&c.dq_free);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          dqv[j] = __uint_as_float(v0[j]);
          dqv[32 + j] = __uint_as_float(v1[j]);
        }
      } else {
        // TMEM lane r = query r of the tile, columns = dimensions 32cw ..
        const int q0 = w.seq_start + i * kTile;
        const int q_rows = min(kTile, w.len - i * kTile);
        uint32_t v[32];
        tmem_ld32(tl + C::kColB + 32 * cw, v);
        tmem_wait_ld(v);
        tc_fence_before();
        mbar_arrive(&c.dq_free);
        if (r < q_rows) {
          float4* dst =
              reinterpret_cast<float4*>(args.dq_acc + (static_cast<size_t>(q0 + r) * args.g.heads + w.head) * D + 32 * cw);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            atomicAdd(dst + q, make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
        }
      }
      return true;
    };
    // vq: the tile's query rows inside the sample.  The rows past its end are
    // staged as zeros: the reduce adds them into the next sample's rows, and
    // with the sample's own non-finite k~ values 0 * k~ need not be 0.
    auto dq_stage = [&](int g, int vq) -> bool {
      if (D != 128) return true;
      // Neither half may run two phases ahead of the reducer's wait on its
      // stage_full barrier (a parity wait would then take the later phase for
      // the one it wants and never return).  Warpgroup 0 reuses the staging
      // tile only once the reducer has released it; warpgroup 1 stages tile g
      // only once the reducer has taken tile g - 1's half, i.e. after the
      // reducer's arrival on that slot's q_free (dK_{g-1} arrived long ago).
      if (cw == 0 && g >= 1 && !warp_wait(&c.stage_free, (g - 1) & 1, abort_flag)) return false;
      if (cw == 1 && g >= 1 && !warp_wait(&c.q_free[(g - 1) & 1], ((g - 1) >> 1) & 1, abort_flag)) return false;
      float* st = reinterpret_cast<float*>(smem + (cw == 0 ? C::kOffStage : C::kOffQ + static_cast<int>(g & 1) * C::kTileBytes)) + r;
      if (vq >= (cw + 1) * 64) {
#pragma unroll
        for (int j = 0; j < 64; ++j) st[j * D] = dqv[j];
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) st[j * D] = cw * 64 + j < vq ? dqv[j] : 0.f;
      }
      fence_proxy_async_smem();
      mbar_arrive(&c.stage_full[cw]);
      return true;
    };
    // The RoPE factors of the dims cw D/2 .. of this thread's K row of an
    // item.
    float cs[D / 16][8];
    auto k_row_cs = [&](const WorkItem& it) {
      const int kv0 = it.seq_start + it.tile * kTile;
      rope_row_cs<D, D / 16>(cw * (D / 16), kv0 + r, r < it.len - it.tile * kTile, args.g, cs);
    };
    // K prologue of item k: warpgroup cw rotates the dims cw D/2 .. of its
    // thread's K row into k~ = R(k) (rows past the sample's end zeroed).
    auto k_prologue = [&](int k, const WorkItem& it) -> bool {
      if (!warp_wait(&c.kv_full, k & 1, abort_flag)) return false;
      const float amax = rotate_row_f16<D / 16>(smem + C::kOffK, r, cw * (D / 16), r < it.len - it.tile * kTile,
                                                1.0f, cs);
      if (!(amax <= kF16Max)) atomicOr(args.g.status, kStatusRange);
      fence_proxy_async_smem();
      mbar_arrive(&c.kv_ready);
      return true;
    };
    bool ok = take_item(0, &w, true);
    if (ok && w.sample >= 0) {
      k_row_cs(w);
      ok = k_prologue(0, w);
    }
    for (int k = 0; ok && w.sample >= 0; ++k) {
      const int kv0 = w.seq_start + w.tile * kTile;
      const int kv_rows = min(kTile, w.len - w.tile * kTile);
      const int n_q = (w.len + kTile - 1) / kTile;
      const bool kv_valid = r < kv_rows;
      for (int i = 0; i < n_q; ++i) {
        const int g = gq + i;
        const int s = static_cast<int>(g & 1);
        // Warpgroup 1 stages dQ_{i-1} right away (its half frees a q~ slot);
        // warpgroup 0 keeps its half in registers until after its dS, so that
        // its exponentials never wait for the staging tile to drain.
        if (i > 0 && (!dq_load(g - 1, i - 1) || (cw == 1 && !dq_stage(g - 1, kTile)))) {
          ok = false;
          break;
        }
        if (!warp_wait(&c.q_ready[s], (g >> 1) & 1, abort_flag) || !warp_wait(&c.s_full, g & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float4* lse4 = reinterpret_cast<const float4*>(rowbuf + s * 2 * kTile + 64 * cw);          // -LSE2
        const float4* dsum4 = reinterpret_cast<const float4*>(rowbuf + s * 2 * kTile + kTile + 64 * cw);  // -D
        float p[64];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // query columns 64cw + 32hh .. + 31 -> packed TMEM columns 64cw + 16hh ..
          uint32_t sv[32];
          tmem_ld32(tl + C::kColA + 64 * cw + 32 * hh, sv);
          tmem_wait_ld(sv);
          uint32_t pw[16];
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 nl = lse4[8 * hh + j4];  // -LSE2 of four queries
            float* pp = p + 32 * hh + 4 * j4;
            float x0, x1, x2, x3;
            f2_unpack(f2_add(f2_pack(__uint_as_float(sv[4 * j4 + 0]), __uint_as_float(sv[4 * j4 + 1])),
                             f2_pack(nl.x, nl.y)), x0, x1);
            f2_unpack(f2_add(f2_pack(__uint_as_float(sv[4 * j4 + 2]), __uint_as_float(sv[4 * j4 + 3])),
                             f2_pack(nl.z, nl.w)), x2, x3);
            pp[0] = ex2_approx(x0);
            pp[1] = ex2_approx(x1);
            pp[2] = ex2_approx(x2);
            pp[3] = ex2_approx(x3);
            pw[2 * j4] = pack_bf16(pp[0], pp[1]);
            pw[2 * j4 + 1] = pack_bf16(pp[2], pp[3]);
          }
          tmem_st16(tl + C::kColA + 64 * cw + 16 * hh, pw);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&c.p_ready[cw]);
        if (!warp_wait(&c.dp_full, g & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // query columns 64cw + 32hh .. + 31 -> 16-byte chunks 4hh .. 4hh + 3
          uint32_t dp[32];
          tmem_ld32(tl + C::kColB + 64 * cw + 32 * hh, dp);
          tmem_wait_ld(dp);
          uint32_t dw[16];
          if (kv_valid) {
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 nd = dsum4[8 * hh + j4];  // -D of four queries
              const float* pp = p + 32 * hh + 4 * j4;
              float y0, y1, y2, y3;
              f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dp[4 * j4 + 0]), __uint_as_float(dp[4 * j4 + 1])),
                                      f2_pack(nd.x, nd.y)),
                               f2_pack(pp[0], pp[1])),
                        y0, y1);
              f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dp[4 * j4 + 2]), __uint_as_float(dp[4 * j4 + 3])),
                                      f2_pack(nd.z, nd.w)),
                               f2_pack(pp[2], pp[3])),
                        y2, y3);
              dw[2 * j4] = pack_f16(y0, y1);
              dw[2 * j4 + 1] = pack_f16(y2, y3);
            }
          } else {
            // K/V rows past the sample's end: dS^T = 0 keeps them out of dQ.
#pragma unroll
            for (int j = 0; j < 16; ++j) dw[j] = 0u;
          }
          // dS^T: packed fp16 into the dead S^T columns of A (the dK operand)
          // and into shared memory (the dQ operand)
          tmem_st16(tl + C::kColA + 64 * cw + 32 + 16 * hh, dw);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            *reinterpret_cast<uint4*>(dst_ds + sw128_off(r, 4 * hh + ch)) =
                make_uint4(dw[4 * ch], dw[4 * ch + 1], dw[4 * ch + 2], dw[4 * ch + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&c.ds_ready[cw]);
        if (i > 0 && cw == 0 && !dq_stage(g - 1, kTile)) { ok = false; break; }
      }
      if (ok) ok = dq_load(gq + n_q - 1, n_q - 1) && dq_stage(gq + n_q - 1, w.len - (n_q - 1) * kTile);
      WorkItem next;
      if (ok) ok = take_item(k + 1, &next, true);
      if (ok) ok = warp_wait(&c.acc_full, k & 1, abort_flag);
      if (!ok) break;
      // Every MMA of the item has completed: dV and dk~ are final.
      // Warpgroup cw stores columns cw * D/2 .. of its row, dV first; the
      // next item's K prologue runs between dV and dK, so that the next
      // item's first MMAs overlap the dK stores (they write TMEM A and B,
      // not dV or dK).  The next item's dV / dK MMAs, which overwrite them,
      // wait for this warpgroup's next p_ready / ds_ready.  (The RoPE
      // factors of the next K row are loaded right before its prologue:
      // loading them before the dV stores made the compiler spill.)
      tc_fence_after();
      const size_t rowoff = (static_cast<size_t>(kv0 + r) * args.g.heads + w.head) * D;
      const int2 pk = kv_valid ? reinterpret_cast<const int2*>(args.g.pos)[kv0 + r] : make_int2(-1, -1);
      const int fk = kv_valid ? args.g.frame[kv0 + r] : -1;
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col0 = cw * (D / 2) + 32 * cc;
        uint32_t v[32];
        tmem_ld32(tl + C::kColDV + col0, v);
        tmem_wait_ld(v);
        if (kv_valid)
          store_row_chunk<D>(reinterpret_cast<__nv_bfloat16*>(args.dv) + rowoff, v, col0, 1.0f, pk, fk, args.g,
                             false);
      }
      if (next.sample >= 0) { k_row_cs(next); if (!k_prologue(k + 1, next)) break; }
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col0 = cw * (D / 2) + 32 * cc;
        uint32_t v[32];
        tmem_ld32(tl + C::kColDK + col0, v);
        tmem_wait_ld(v);
        // TMEM holds dS^T q~; dk~ = dk_mult dS^T q~ (ln 2: q~ carries s log2 e).
        if (kv_valid)
          store_row_chunk<D>(reinterpret_cast<__nv_bfloat16*>(args.dk) + rowoff, v, col0, args.dk_mult, pk, fk,
                             args.g, true);
      }
      tc_fence_before();
      gq += n_q;
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
  if (tid == 0 && c.abort) {
    const uint32_t a = static_cast<uint32_t>(c.abort) - 1u, base = smem_u32(&c);
    record_timeout(args.g.status, args.g.timeout_info, kTimeoutKernelBwd,
                   a >= base && a < base + 8 * kBwdBarriers ? (a - base) / 8 : 0xfffu);
  }
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, cudaStream_t stream, cudaEvent_t ev0,
                         cudaEvent_t ev1) {
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
  const int grid = a.g.n_items < sm_count() ? a.g.n_items : sm_count();
  bwd_main_kernel<D><<<grid, kThreads, C::kDynSmem, stream>>>(tq, tk, tv, tdo, tdq, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ev1 && (e = cudaEventRecord(ev1, stream)) != cudaSuccess) return e;
  bwd_dq_kernel<D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, int head_dim, cudaStream_t stream,
                            cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  if (a.g.n_items <= 0) return cudaSuccess;
  if (head_dim == 128) return launch_bwd_d<128>(a, tq, tk, tv, tdo, tdq, stream, ev_start, ev_stop);
  return launch_bwd_d<64>(a, tq, tk, tv, tdo, tdq, stream, ev_start, ev_stop);
}

}  // namespace mf
