// Pack planner: prefix scan over per-sample token counts, the longest-first
// work order, per-token (row, col) ids and the 2D RoPE cos/sin table.
//
// Mage-Flow review (startedourmission.github.io), section "Native-Resolution
// MMDiT": variable-length latent token rows are packed back to back under a
// fixed token budget and attention is confined by per-sample cumulative
// offsets; section "Mage-VAE": an H x W px image becomes (H/16)(W/16) tokens.
#include "common.cuh"
#include "ptx.cuh"

namespace mf {
namespace {

constexpr int kPerThread = kPlanMaxSamples / kPlanThreads;  // 4

// Block-wide exclusive scan of one int64 per thread (1024 threads).
__device__ long long block_exclusive_scan(long long v, long long* s_warp, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = s_warp[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  long long before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
  *total = s_warp[31];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kPlanThreads) pack_scan_kernel(PlanArgs a) {
  __shared__ long long s_warp[32];
  __shared__ int32_t s_len[kPlanMaxSamples];
  __shared__ int32_t s_sorted[kPlanMaxSamples];
  __shared__ int s_npacked, s_maxlen, s_maxgrid;
  const int t = threadIdx.x;
  if (t == 0) {
    s_npacked = 0;
    s_maxlen = 0;
    s_maxgrid = 0;
  }
  // 1. token counts L_i = text + (H/16)(W/16); thread t owns samples 4t..4t+3.
  long long mine[kPerThread];
  long long local = 0;
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int i = t * kPerThread + u;
    long long L = 0;
    if (i < a.n) {
      const int32_t* s = a.samples + 4 * i;
      const int frames = s[3] == 0 ? 1 : s[3];
      L = static_cast<long long>(s[0]) + static_cast<long long>(frames) * (s[1] / 16) * (s[2] / 16);
      s_len[i] = static_cast<int32_t>(L);
    }
    mine[u] = L;
    local += L;
  }
  long long total_all;
  long long off = block_exclusive_scan(local, s_warp, &total_all);
  // 2. offsets, the packed prefix, maxima.
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int i = t * kPerThread + u;
    if (i < a.n) {
      const bool fits = (a.budget <= 0) || (off + mine[u] <= a.budget);
      if (fits) {
        a.cu_seqlens[i] = static_cast<int32_t>(off);
        atomicAdd(&s_npacked, 1);
        atomicMax(&s_maxlen, static_cast<int>(mine[u]));
        const int32_t* s = a.samples + 4 * i;
        atomicMax(&s_maxgrid, max(s[1] / 16, s[2] / 16));
      }
      off += mine[u];
    }
  }
  __syncthreads();
  const int np = s_npacked;
  // L_i > 0 for every valid sample, so the packed set is a prefix 0..np-1.
  // 3. longest-first order (stable: ties keep sample order).
  for (int i = t; i < np; i += kPlanThreads) {
    const int32_t Li = s_len[i];
    int rank = 0;
    for (int j = 0; j < np; ++j) {
      const int32_t Lj = s_len[j];
      rank += (Lj > Li) || (Lj == Li && j < i);
    }
    s_sorted[rank] = i;
  }
  __syncthreads();
  long long nt_local = 0, np_local = 0;
  long long nt_mine[kPerThread], np_mine[kPerThread];
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int r = t * kPerThread + u;
    long long nt = 0, npair = 0;
    if (r < np) {
      nt = (s_len[s_sorted[r]] + kTile - 1) / kTile;
      npair = (s_len[s_sorted[r]] + 2 * kTile - 1) / (2 * kTile);
    }
    nt_mine[u] = nt;
    np_mine[u] = npair;
    nt_local += nt;
    np_local += npair;
  }
  long long n_tiles, n_pairs;
  long long start = block_exclusive_scan(nt_local, s_warp, &n_tiles);
  long long pstart = block_exclusive_scan(np_local, s_warp, &n_pairs);
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int r = t * kPerThread + u;
    if (r < np) {
      a.order[4 * r] = s_sorted[r];
      a.order[4 * r + 1] = static_cast<int32_t>(start);
      a.order[4 * r + 2] = static_cast<int32_t>(pstart);
      a.order[4 * r + 3] = 0;
    }
    start += nt_mine[u];
    pstart += np_mine[u];
  }
  if (t == 0) {
    long long total = 0;
    for (int i = 0; i < np; ++i) total += s_len[i];
    a.cu_seqlens[np] = static_cast<int32_t>(total);
    a.scalars->n_packed = np;
    a.scalars->total_tokens = static_cast<int32_t>(total);
    a.scalars->max_seqlen = s_maxlen;
    a.scalars->max_grid = s_maxgrid;
    a.scalars->n_tiles = static_cast<int32_t>(n_tiles);
    a.scalars->n_pairs = static_cast<int32_t>(n_pairs);
    const PlanScalars& x = a.expect;
    const bool same = x.n_packed == np && x.total_tokens == total && x.max_seqlen == s_maxlen &&
                      x.max_grid == s_maxgrid && x.n_tiles == n_tiles && x.n_pairs == n_pairs;
    a.scalars->status = same ? 0 : kStatusPlan;
    a.scalars->timeout_info = 0;
  }
}

// Per-token ids: text -> (-1, -1), frame -1; image token j of a sample with
// gh x gw latents per frame -> frame j / (gh gw), then (r / gw, r % gw) with
// r = j % (gh gw).
__global__ void pack_pos_kernel(PlanArgs a) {
  const int tok = blockIdx.x * blockDim.x + threadIdx.x;
  const int total = a.scalars->total_tokens;
  if (tok >= total || tok >= a.token_bound) return;
  const int np = a.scalars->n_packed;
  int lo = 0, hi = np;  // find s with cu[s] <= tok < cu[s+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.cu_seqlens[mid] <= tok) lo = mid; else hi = mid;
  }
  const int32_t* s = a.samples + 4 * lo;
  const int j = tok - a.cu_seqlens[lo] - s[0];
  int2 p = make_int2(-1, -1);
  int f = -1;
  if (j >= 0) {
    const int gw = s[2] / 16, per_frame = (s[1] / 16) * gw;
    f = j / per_frame;
    const int r = j - f * per_frame;
    p = make_int2(r / gw, r % gw);
  }
  reinterpret_cast<int2*>(a.pos)[tok] = p;
  a.frame[tok] = f;
}

// cos/sin(p * theta^(-2i/a)) for the row/col slices of a dims (a = head_dim/2
// with 2 axes, 7 head_dim/16 with 3), i < a/2, p < grid_bound ([p][i] order);
// with 3 axes also the frame slice's (a_f = head_dim/8 dims) for frames 0, 1
// ([f][i] order, after the row/col entries in the index space).  Angles and
// sin/cos are evaluated in double and rounded to float once.
__global__ void rope_table_kernel(PlanArgs a) {
  const int a_hw = a.rope_axes == 3 ? 7 * a.head_dim / 16 : a.head_dim / 2;
  const int a_f = a.head_dim / 8;
  const int n_hw = a.grid_bound * (a_hw / 2);
  const int n_f = a.rope_axes == 3 ? 2 * (a_f / 2) : 0;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_hw + n_f) return;
  int p, i, width;
  if (idx < n_hw) {
    p = idx / (a_hw / 2);
    i = idx % (a_hw / 2);
    width = a_hw;
  } else {
    p = (idx - n_hw) / (a_f / 2);
    i = (idx - n_hw) % (a_f / 2);
    width = a_f;
  }
  const double f = pow(static_cast<double>(a.theta), -2.0 * i / width);
  double sv, cv;
  sincos(static_cast<double>(p) * f, &sv, &cv);
  const float2 v = make_float2(static_cast<float>(cv), static_cast<float>(sv));
  if (idx < n_hw) reinterpret_cast<float2*>(a.rope_cs)[idx] = v;
  else reinterpret_cast<float2*>(a.rope_f)[idx - n_hw] = v;
}

}  // namespace

cudaError_t launch_pack_plan(const PlanArgs& a, cudaStream_t stream) {
  pack_scan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.token_bound > 0) {
    pack_pos_kernel<<<(a.token_bound + 255) / 256, 256, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int a_hw = a.rope_axes == 3 ? 7 * a.head_dim / 16 : a.head_dim / 2;
  const int nt = a.grid_bound * (a_hw / 2) + (a.rope_axes == 3 ? a.head_dim / 8 : 0);
  if (a.grid_bound > 0) {
    rope_table_kernel<<<(nt + 255) / 256, 256, 0, stream>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace mf
