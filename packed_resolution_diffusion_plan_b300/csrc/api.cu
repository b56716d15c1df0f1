// C-ABI entry points of libmf (declared in include/mf.h): argument checks,
// workspace layout, TMA descriptor encoding and kernel launches.  No device
// memory is allocated here; every buffer comes from the caller.
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/mf.h"
#include "common.cuh"
#include "ptx.cuh"

namespace {

using mf::PlanScalars;

thread_local std::string g_last_cuda_error;
// One-shot event pair set by mf_record_main_kernel, consumed by the next
// attention call on this thread.
thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;
// Load-dropping flags of mf_debug_inject (MF_DEBUG_*), passed to the kernels.
static_assert(MF_DEBUG_DROP_FWD_KV == mf::kDebugDropFwdKV && MF_DEBUG_DROP_BWD_QDO == mf::kDebugDropBwdQdo,
              "debug flag values");
thread_local int32_t g_debug_flags = 0;

void take_events(cudaEvent_t* a, cudaEvent_t* b) {
  *a = g_ev_start;
  *b = g_ev_stop;
  g_ev_start = g_ev_stop = nullptr;
}

mf_status cuda_fail(cudaError_t e, const char* where) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
  g_last_cuda_error = buf;
  return MF_ERR_CUDA;
}

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- plan
struct PlanLayout {
  size_t off_scalars, off_samples, off_cu, off_order, off_pos, off_frame, off_rope, off_rope_f, bytes;
  int32_t token_bound, grid_bound;
  mf::PlanScalars expect;  // the plan's scalars, from the same greedy prefix rule as the device scan
};

// Latent frames of a sample (0 counts as 1).
int32_t sample_frames(const mf_sample& s) { return s.frames == 0 ? 1 : s.frames; }

mf_status check_samples(const mf_sample* samples, int32_t n, int32_t budget, int32_t head_dim,
                        int32_t rope_axes, PlanLayout* L) {
  if (n < 0 || (n > 0 && samples == nullptr) || budget < 0) return MF_ERR_INVALID_ARG;
  if (rope_axes != 2 && rope_axes != 3) return MF_ERR_INVALID_ARG;
  if (n > MF_MAX_SAMPLES) return MF_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  long long used = 0, n_tiles = 0, n_pairs = 0;
  int32_t gmax = 0, n_packed = 0, max_len = 0, max_grid = 0;
  bool stopped = false;
  for (int32_t i = 0; i < n; ++i) {
    const mf_sample& s = samples[i];
    // height = width = 0: a text-only sample (it must then have text)
    const bool text_only = s.height == 0 && s.width == 0 && s.text_len > 0;
    if (s.text_len < 0 || (!text_only && (s.height <= 0 || s.width <= 0)) || (s.height % 16) || (s.width % 16))
      return MF_ERR_INVALID_ARG;
    if (s.frames < 0 || s.frames > 2 || (sample_frames(s) == 2 && rope_axes != 3)) return MF_ERR_INVALID_ARG;
    const long long gh = s.height / 16, gw = s.width / 16;
    if (gh > MF_MAX_GRID || gw > MF_MAX_GRID) return MF_ERR_UNSUPPORTED;
    gmax = static_cast<int32_t>(std::max<long long>(gmax, std::max(gh, gw)));
    const long long len = s.text_len + sample_frames(s) * gh * gw;
    if (!stopped) {
      if (budget > 0 && used + len > budget) {
        stopped = true;
        if (i == 0) return MF_ERR_BUDGET;
      } else {
        used += len;
        if (used >= (1ll << 31)) return MF_ERR_INVALID_ARG;
        ++n_packed;
        max_len = static_cast<int32_t>(std::max<long long>(max_len, len));
        max_grid = static_cast<int32_t>(std::max<long long>(max_grid, std::max(gh, gw)));
        n_tiles += (len + mf::kTile - 1) / mf::kTile;
        n_pairs += (len + 2 * mf::kTile - 1) / (2 * mf::kTile);
      }
    }
  }
  L->expect = mf::PlanScalars{};
  L->expect.n_packed = n_packed;
  L->expect.total_tokens = static_cast<int32_t>(used);
  L->expect.max_seqlen = max_len;
  L->expect.max_grid = max_grid;
  L->expect.n_tiles = static_cast<int32_t>(n_tiles);
  L->expect.n_pairs = static_cast<int32_t>(n_pairs);
  L->token_bound = static_cast<int32_t>(used);
  L->grid_bound = gmax;
  size_t off = 0;
  L->off_scalars = off;
  off = align_up(off + sizeof(PlanScalars), 256);
  L->off_samples = off;
  off = align_up(off + static_cast<size_t>(n) * sizeof(mf_sample), 256);
  L->off_cu = off;
  off = align_up(off + static_cast<size_t>(n + 1) * sizeof(int32_t), 256);
  L->off_order = off;
  off = align_up(off + static_cast<size_t>(n) * 4 * sizeof(int32_t), 256);
  L->off_pos = off;
  off = align_up(off + static_cast<size_t>(L->token_bound) * 2 * sizeof(int32_t), 256);
  L->off_frame = off;
  off = align_up(off + static_cast<size_t>(L->token_bound) * sizeof(int32_t), 256);
  L->off_rope = off;
  // row/col table: pairs of the a-dim slices (a = head_dim/2 with 2 axes, 7 head_dim/16 with 3)
  const int a = rope_axes == 3 ? 7 * head_dim / 16 : head_dim / 2;
  off = align_up(off + static_cast<size_t>(gmax) * (a / 2) * 2 * sizeof(float), 256);
  L->off_rope_f = off;
  if (rope_axes == 3) off = align_up(off + static_cast<size_t>(2) * (head_dim / 16) * 2 * sizeof(float), 256);
  L->bytes = off;
  return MF_OK;
}

// ---------------------------------------------------------------- TMA
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// [rows, heads*head_dim] view of a [T, heads, head_dim] tensor of 16-bit
// elements; boxes of 128 rows x 64 columns, 128-byte swizzle, zero fill past
// the last row.
mf_status make_tmap(CUtensorMap* map, const void* base, int32_t rows, int32_t heads, int32_t head_dim,
                    int64_t row_elems = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    g_last_cuda_error = "cuTensorMapEncodeTiled entry point not available";
    return MF_ERR_CUDA;
  }
  const cuuint64_t cols = static_cast<cuuint64_t>(heads) * head_dim;
  cuuint64_t gdim[2] = {cols, static_cast<cuuint64_t>(rows)};
  // row_elems: elements from one token's row to the next (0 = cols, a plain
  // [T, heads, head_dim] tensor; 3 cols for the V third of a QKV projection)
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_elems > 0 ? row_elems : static_cast<int64_t>(cols)) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(mf::kTile)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
                   estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed with CUresult %d", static_cast<int>(r));
    g_last_cuda_error = buf;
    return MF_ERR_CUDA;
  }
  return MF_OK;
}

// float32 [rows][heads][head_dim] view of the dQ accumulator as a 3D tensor
// (dimension, head, token): boxes of head_dim x 1 x 64, no swizzle.
mf_status make_tmap_acc(CUtensorMap* map, const float* base, int32_t rows, int32_t heads, int32_t head_dim) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    g_last_cuda_error = "cuTensorMapEncodeTiled entry point not available";
    return MF_ERR_CUDA;
  }
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(head_dim) * 4, static_cast<cuuint64_t>(heads) * head_dim * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(head_dim), 1, 64};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled (dQ accumulator) failed with CUresult %d", static_cast<int>(r));
    g_last_cuda_error = buf;
    return MF_ERR_CUDA;
  }
  return MF_OK;
}

mf_status check_attn_common(const mf_plan* plan, int32_t heads, int32_t head_dim) {
  if (plan == nullptr || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (head_dim != plan->head_dim) return MF_ERR_INVALID_ARG;
  if (plan->total_tokens < 0 || plan->n_samples < 0) return MF_ERR_INVALID_ARG;
  if (plan->rope_axes != 2 && plan->rope_axes != 3) return MF_ERR_INVALID_ARG;
  if (plan->total_tokens > 0 &&
      (plan->cu_seqlens == nullptr || plan->pos == nullptr || plan->frame == nullptr || plan->rope_cs == nullptr ||
       (plan->rope_axes == 3 && plan->rope_f == nullptr) || plan->order == nullptr || plan->status == nullptr))
    return MF_ERR_INVALID_ARG;
  if (static_cast<long long>(plan->n_tiles) * heads >= (1ll << 31)) return MF_ERR_UNSUPPORTED;
  if (plan->n_pairs < 0 || plan->n_pairs > plan->n_tiles) return MF_ERR_INVALID_ARG;
  return MF_OK;
}

mf::AttnGeom make_geom(const mf_plan* plan, int32_t heads) {
  mf::AttnGeom g;
  g.cu_seqlens = plan->cu_seqlens;
  g.pos = plan->pos;
  g.rope_cs = plan->rope_cs;
  g.rope_f = plan->rope_f;
  g.frame = plan->frame;
  g.rope_axes = plan->rope_axes;
  g.order = plan->order;
  g.n_samples = plan->n_samples;
  g.total_tokens = plan->total_tokens;
  g.heads = heads;
  g.n_items = plan->n_tiles * heads;
  g.status = plan->status;
  // the timeout record sits two words after the status word (PlanScalars)
  static_assert(offsetof(mf::PlanScalars, timeout_info) - offsetof(mf::PlanScalars, status) == 2 * sizeof(int32_t),
                "timeout record beside the status word");
  g.timeout_info = plan->status + 2;
  g.debug = g_debug_flags;
  return g;
}

float resolve_scale(float s, int32_t head_dim) {
  return (s > 0.f && std::isfinite(s)) ? s : 1.0f / std::sqrt(static_cast<float>(head_dim));
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

extern "C" {

mf_status mf_pack_plan_workspace_size(const mf_sample* samples, int32_t n_samples, int32_t token_budget,
                                      int32_t head_dim, int32_t rope_axes, size_t* bytes) {
  if (bytes == nullptr) return MF_ERR_INVALID_ARG;
  PlanLayout L;
  mf_status st = check_samples(samples, n_samples, token_budget, head_dim, rope_axes, &L);
  if (st != MF_OK) return st;
  *bytes = L.bytes;
  return MF_OK;
}

mf_status mf_pack_plan(const mf_sample* samples, int32_t n_samples, int32_t token_budget, int32_t head_dim,
                       int32_t rope_axes, float rope_theta, void* workspace, size_t workspace_bytes,
                       mf_plan* plan_out, void* stream) {
  if (plan_out == nullptr || workspace == nullptr) return MF_ERR_INVALID_ARG;
  if (!(rope_theta > 0.f) || !std::isfinite(rope_theta)) return MF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MF_ERR_INVALID_ARG;
  PlanLayout L;
  mf_status st = check_samples(samples, n_samples, token_budget, head_dim, rope_axes, &L);
  if (st != MF_OK) return st;
  if (workspace_bytes < L.bytes) return MF_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  mf::PlanArgs a;
  a.samples = reinterpret_cast<const int32_t*>(ws + L.off_samples);
  a.n = n_samples;
  a.budget = token_budget;
  a.scalars = reinterpret_cast<PlanScalars*>(ws + L.off_scalars);
  a.cu_seqlens = reinterpret_cast<int32_t*>(ws + L.off_cu);
  a.order = reinterpret_cast<int32_t*>(ws + L.off_order);
  a.pos = reinterpret_cast<int32_t*>(ws + L.off_pos);
  a.frame = reinterpret_cast<int32_t*>(ws + L.off_frame);
  a.token_bound = L.token_bound;
  a.rope_cs = reinterpret_cast<float*>(ws + L.off_rope);
  a.rope_f = reinterpret_cast<float*>(ws + L.off_rope_f);
  a.grid_bound = L.grid_bound;
  a.head_dim = head_dim;
  a.rope_axes = rope_axes;
  a.theta = rope_theta;
  a.expect = L.expect;
  cudaError_t e;
  if (n_samples > 0) {
    e = cudaMemcpyAsync(ws + L.off_samples, samples, static_cast<size_t>(n_samples) * sizeof(mf_sample),
                        cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "mf_pack_plan: copy samples");
  }
  e = mf::launch_pack_plan(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "mf_pack_plan: launch");
  // The scalars come from the host pass above, so the call never waits on
  // `stream`; the device scan recomputes them and raises kStatusPlan if it
  // disagrees.
  plan_out->n_samples = L.expect.n_packed;
  plan_out->total_tokens = L.expect.total_tokens;
  plan_out->max_seqlen = L.expect.max_seqlen;
  plan_out->max_grid = L.expect.max_grid;
  plan_out->head_dim = head_dim;
  plan_out->n_tiles = L.expect.n_tiles;
  plan_out->n_pairs = L.expect.n_pairs;
  plan_out->cu_seqlens = a.cu_seqlens;
  plan_out->pos = a.pos;
  plan_out->frame = a.frame;
  plan_out->rope_axes = rope_axes;
  plan_out->rope_cs = a.rope_cs;
  plan_out->rope_f = rope_axes == 3 ? a.rope_f : nullptr;
  plan_out->order = a.order;
  plan_out->status = &a.scalars->status;
  return MF_OK;
}

mf_status mf_attn_fwd_workspace_size(int32_t total_tokens, int32_t heads, int32_t head_dim, size_t* bytes) {
  if (bytes == nullptr || total_tokens < 0 || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  const size_t rows = static_cast<size_t>(total_tokens) * heads;
  // fp16 k~ | the work counter of the persistent kernel
  *bytes = align_up(rows * head_dim * 2, 256) + 256;
  return MF_OK;
}

}  // extern "C"

namespace {

// The forward over q, k, v whose token rows are `stride` elements apart
// (heads * head_dim for plain tensors, 3 heads * head_dim for the thirds of a
// QKV projection).
mf_status attn_fwd_impl(const void* q, const void* k, const void* v, int64_t stride, const mf_plan* plan,
                        int32_t heads, int32_t head_dim, float softmax_scale, void* workspace,
                        size_t workspace_bytes, void* o, float* lse, void* stream, const char* who) {
  mf_status st = check_attn_common(plan, heads, head_dim);
  if (st != MF_OK) return st;
  if (plan->total_tokens == 0) return MF_OK;
  if (!q || !k || !v || !o || !lse || !workspace) return MF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return MF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MF_ERR_INVALID_ARG;
  size_t need = 0;
  if ((st = mf_attn_fwd_workspace_size(plan->total_tokens, heads, head_dim, &need)) != MF_OK) return st;
  if (workspace_bytes < need) return MF_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(plan->total_tokens) * heads;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  mf::FwdArgs a;
  a.g = make_geom(plan, heads);
  a.g.n_items = plan->n_pairs * heads;  // the forward works on 256-row tile pairs
  a.scale_log2 = resolve_scale(softmax_scale, head_dim) * kLog2e;
  a.q = q;
  a.k = k;
  a.qk_stride = stride;
  a.k_rot = ws;
  a.work_counter = reinterpret_cast<int32_t*>(ws + align_up(rows * head_dim * 2, 256));
  a.o = o;
  a.lse = lse;
  // The main kernel reads the raw Q rows (rotating them in its prologue) and
  // streams the rotated fp16 K copy that fwd_pre writes.
  CUtensorMap tq, tk, tv;
  if ((st = make_tmap(&tq, q, plan->total_tokens, heads, head_dim, stride)) != MF_OK) return st;
  if ((st = make_tmap(&tk, a.k_rot, plan->total_tokens, heads, head_dim)) != MF_OK) return st;
  if ((st = make_tmap(&tv, v, plan->total_tokens, heads, head_dim, stride)) != MF_OK) return st;
  cudaEvent_t ev0, ev1;
  take_events(&ev0, &ev1);
  cudaError_t e = mf::launch_attn_fwd(a, tq, tk, tv, head_dim, static_cast<cudaStream_t>(stream), ev0, ev1);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return MF_OK;
}

}  // namespace

extern "C" {

mf_status mf_attn_fwd(const void* q, const void* k, const void* v, const mf_plan* plan, int32_t heads,
                      int32_t head_dim, float softmax_scale, void* workspace, size_t workspace_bytes, void* o,
                      float* lse, void* stream) {
  return attn_fwd_impl(q, k, v, static_cast<int64_t>(heads) * head_dim, plan, heads, head_dim, softmax_scale,
                       workspace, workspace_bytes, o, lse, stream, "mf_attn_fwd");
}

mf_status mf_attn_fwd_qkv(const void* qkv, const mf_plan* plan, int32_t heads, int32_t head_dim,
                          float softmax_scale, void* workspace, size_t workspace_bytes, void* o, float* lse,
                          void* stream) {
  if (qkv == nullptr || heads < 1) return MF_ERR_INVALID_ARG;
  const int64_t C = static_cast<int64_t>(heads) * head_dim;
  const uint8_t* base = static_cast<const uint8_t*>(qkv);
  return attn_fwd_impl(base, base + C * 2, base + 2 * C * 2, 3 * C, plan, heads, head_dim, softmax_scale,
                       workspace, workspace_bytes, o, lse, stream, "mf_attn_fwd_qkv");
}

mf_status mf_attn_bwd_workspace_size(int32_t total_tokens, int32_t heads, int32_t head_dim, size_t* bytes) {
  if (bytes == nullptr || total_tokens < 0 || heads < 1) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  const size_t rows = static_cast<size_t>(total_tokens) * heads;
  // D | float32 dQ accumulator | fp16 q~ | the work counter of the persistent kernel
  *bytes = align_up(rows * sizeof(float), 256) + align_up(rows * head_dim * sizeof(float), 256) +
           align_up(rows * head_dim * 2, 256) + 256;
  return MF_OK;
}

}  // extern "C"

namespace {

// The backward: bwd_pre writes q~ = s log2(e) R(q) into the workspace beside
// D and the dQ accumulator; the main kernel rotates each K tile itself.
mf_status attn_bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, const mf_plan* plan, int32_t heads, int32_t head_dim, float softmax_scale,
                        void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv, void* stream,
                        const char* who) {
  mf_status st = check_attn_common(plan, heads, head_dim);
  if (st != MF_OK) return st;
  if (plan->total_tokens == 0) return MF_OK;
  if (!q || !k || !v || !o || !lse || !dout || !workspace || !dq || !dk || !dv) return MF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return MF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MF_ERR_INVALID_ARG;
  size_t need = 0;
  if ((st = mf_attn_bwd_workspace_size(plan->total_tokens, heads, head_dim, &need)) != MF_OK) return st;
  if (workspace_bytes < need) return MF_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(plan->total_tokens) * heads;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t off_acc = align_up(rows * sizeof(float), 256);
  const size_t off_qr = off_acc + align_up(rows * head_dim * sizeof(float), 256);
  const size_t off_ctr = off_qr + align_up(rows * head_dim * 2, 256);
  mf::BwdArgs a;
  a.g = make_geom(plan, heads);
  a.scale = resolve_scale(softmax_scale, head_dim);
  a.scale_log2 = a.scale * kLog2e;
  a.q = q;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dsum = reinterpret_cast<float*>(ws);
  a.dq_acc = reinterpret_cast<float*>(ws + off_acc);
  a.q_rot = ws + off_qr;
  a.work_counter = reinterpret_cast<int32_t*>(ws + off_ctr);
  // q~ carries s log2(e): dk~ = s dS^T R(q) = ln 2 (dS^T q~); k~ = R(k): dq~ = s (dS k~)
  a.dk_mult = 1.0f / kLog2e;
  a.dq_mult = a.scale;
  // The main kernel streams the fp16 q~ copy (16-bit elements: the tensor
  // maps only move bytes) and loads the raw K rows, which it rotates itself.
  CUtensorMap tq, tk, tv, tdo;
  if ((st = make_tmap(&tq, a.q_rot, plan->total_tokens, heads, head_dim)) != MF_OK) return st;
  if ((st = make_tmap(&tk, k, plan->total_tokens, heads, head_dim)) != MF_OK) return st;
  if ((st = make_tmap(&tv, v, plan->total_tokens, heads, head_dim)) != MF_OK) return st;
  if ((st = make_tmap(&tdo, dout, plan->total_tokens, heads, head_dim)) != MF_OK) return st;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  cudaEvent_t ev0, ev1;
  take_events(&ev0, &ev1);
  CUtensorMap tdq;
  if ((st = make_tmap_acc(&tdq, a.dq_acc, plan->total_tokens, heads, head_dim)) != MF_OK) return st;
  cudaError_t e = mf::launch_attn_bwd(a, tq, tk, tv, tdo, tdq, head_dim, static_cast<cudaStream_t>(stream), ev0, ev1);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return MF_OK;
}

}  // namespace

extern "C" {

mf_status mf_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, const mf_plan* plan, int32_t heads, int32_t head_dim,
                      float softmax_scale, void* workspace, size_t workspace_bytes, void* dq, void* dk,
                      void* dv, void* stream) {
  return attn_bwd_impl(q, k, v, o, lse, dout, plan, heads, head_dim, softmax_scale, workspace, workspace_bytes, dq,
                       dk, dv, stream, "mf_attn_bwd");
}

mf_status mf_check(const mf_plan* plan, void* stream) {
  if (plan == nullptr || plan->status == nullptr) return MF_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "mf_check: synchronize");
  // status, n_pairs, timeout record (PlanScalars from the status word on)
  int32_t words[3] = {0, 0, 0};
  e = cudaMemcpyAsync(words, plan->status, sizeof(words), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "mf_check: read status");
  const int32_t status = words[0];
  if (status != 0) {
    e = cudaMemsetAsync(plan->status, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->status + 2, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "mf_check: clear status");
    if (status & mf::kStatusTimeout) {
      const uint32_t info = static_cast<uint32_t>(words[2]);
      char buf[160];
      snprintf(buf, sizeof(buf), "a bounded wait timed out in %s: first at barrier %u, %u CTA(s)",
               (info >> 28) == 1 ? "attn_fwd_kernel" : (info >> 28) == 2 ? "bwd_main_kernel" : "a kernel",
               (info >> 16) & 0xfffu, info & 0xffffu);
      g_last_cuda_error = buf;
    }
    if (status & mf::kStatusPlan) {
      g_last_cuda_error = "the device pack scan disagreed with the host's plan scalars";
      return MF_ERR_CUDA;
    }
    if (status & mf::kStatusLayout) {
      g_last_cuda_error = "a kernel found its shared memory misaligned and did no work";
      return MF_ERR_CUDA;
    }
    if (status & mf::kStatusPairing) return MF_ERR_INVALID_ARG;
    return (status & mf::kStatusTimeout) ? MF_ERR_TIMEOUT : MF_ERR_RANGE;
  }
  return MF_OK;
}

mf_status mf_record_main_kernel(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return MF_ERR_INVALID_ARG;
  g_ev_start = static_cast<cudaEvent_t>(start_event);
  g_ev_stop = static_cast<cudaEvent_t>(stop_event);
  return MF_OK;
}

const char* mf_status_string(mf_status status) {
  switch (status) {
    case MF_OK: return "ok";
    case MF_ERR_INVALID_ARG: return "invalid argument";
    case MF_ERR_UNSUPPORTED: return "unsupported configuration";
    case MF_ERR_BUDGET: return "first sample exceeds the token budget";
    case MF_ERR_CUDA: return "CUDA error";
    case MF_ERR_TIMEOUT: return "a kernel wait timed out";
    case MF_ERR_RANGE: return "a rotated Q/K value exceeded the fp16 range of the logit product";
  }
  return "unknown status";
}

const char* mf_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

mf_status mf_cfg_combine(const void* o, const mf_plan* plan, int32_t heads, int32_t head_dim, float guidance,
                         void* out, void* stream) {
  mf_status st = check_attn_common(plan, heads, head_dim);
  if (st != MF_OK) return st;
  if (plan->n_samples % 2 != 0 || !std::isfinite(guidance)) return MF_ERR_INVALID_ARG;
  if (plan->total_tokens == 0) return MF_OK;
  if (!o || !out || !aligned16(o) || !aligned16(out)) return MF_ERR_INVALID_ARG;
  const mf::AttnGeom g = make_geom(plan, heads);
  cudaError_t e = mf::launch_cfg_combine(o, g, head_dim, guidance, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mf_cfg_combine");
  return MF_OK;
}

// Plan checks shared by the chain calls (they read only the offsets).
mf_status check_chain(const mf_plan* plan, int32_t hidden) {
  if (plan == nullptr || hidden <= 0) return MF_ERR_INVALID_ARG;
  if (plan->total_tokens < 0 || plan->n_samples < 0) return MF_ERR_INVALID_ARG;
  if (plan->total_tokens > 0 && plan->cu_seqlens == nullptr) return MF_ERR_INVALID_ARG;
  return MF_OK;
}

mf_status mf_norm_modulate(const void* x, const mf_plan* plan, int32_t hidden, const void* shift,
                           const void* scale, float eps, void* y, void* stream) {
  mf_status st = check_chain(plan, hidden);
  if (st != MF_OK) return st;
  const int k = hidden / 1024;
  if (hidden % 1024 != 0 || !(k == 1 || k == 2 || k == 3 || k == 4 || k == 6 || k == 8)) return MF_ERR_UNSUPPORTED;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return MF_ERR_INVALID_ARG;
  if (plan->total_tokens == 0) return MF_OK;
  if (!x || !shift || !scale || !y) return MF_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(shift) || !aligned16(scale) || !aligned16(y)) return MF_ERR_INVALID_ARG;
  mf::AttnGeom g = make_geom(plan, 1);
  cudaError_t e = mf::launch_norm_modulate(x, g, hidden, shift, scale, eps, y, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mf_norm_modulate");
  return MF_OK;
}

mf_status mf_gate_residual(const void* x, const void* z, const mf_plan* plan, int32_t hidden, const void* gate,
                           void* out, void* stream) {
  mf_status st = check_chain(plan, hidden);
  if (st != MF_OK) return st;
  if (hidden % 8 != 0) return MF_ERR_UNSUPPORTED;
  if (plan->total_tokens == 0) return MF_OK;
  if (!x || !z || !gate || !out) return MF_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(z) || !aligned16(gate) || !aligned16(out)) return MF_ERR_INVALID_ARG;
  mf::AttnGeom g = make_geom(plan, 1);
  cudaError_t e = mf::launch_gate_residual(x, z, g, hidden, gate, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mf_gate_residual");
  return MF_OK;
}

mf_status mf_debug_inject(int32_t flags) {
  if (flags & ~(MF_DEBUG_DROP_FWD_KV | MF_DEBUG_DROP_BWD_QDO)) return MF_ERR_INVALID_ARG;
  g_debug_flags = flags;
  return MF_OK;
}

}  // extern "C"
