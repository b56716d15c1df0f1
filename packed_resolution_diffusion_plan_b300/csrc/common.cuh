// Parameter blocks and launch declarations shared by the C-ABI layer and the
// kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mf {

constexpr int kTile = 128;            // rows per Q tile and per KV tile
constexpr int kPlanThreads = 1024;    // one CTA runs the pack scan
constexpr int kPlanMaxSamples = 4096;

// Scalars the pack-plan kernel writes for the host (one 32-byte block).
struct PlanScalars {
  int32_t n_packed;
  int32_t total_tokens;
  int32_t max_seqlen;
  int32_t max_grid;
  int32_t n_tiles;
  int32_t status;
  int32_t n_pairs;
  int32_t timeout_info;   // record_timeout's word (0: no wait timed out)
};

struct PlanArgs {
  const int32_t* samples;   // device [n][4] (text_len, height_px, width_px, frames)
  int32_t n;
  int32_t budget;           // 0 = none
  PlanScalars* scalars;
  int32_t* cu_seqlens;      // [n+1]
  int32_t* order;           // [n][4]
  int32_t* pos;             // [token_bound][2]
  int32_t* frame;           // [token_bound]
  int32_t token_bound;
  float* rope_cs;           // [grid_bound][a/2][2], a = the row/col slice width
  float* rope_f;            // [2][head_dim/16][2] (3 axes), else unused
  int32_t grid_bound;
  int32_t head_dim;
  int32_t rope_axes;        // 2 or 3
  float theta;
  PlanScalars expect;       // the host's scalars for this pack (the scan checks its own against them)
};

cudaError_t launch_pack_plan(const PlanArgs& a, cudaStream_t stream);

// Attention work decode: the plan's order list holds, per sample sorted by
// length (longest first), the sample index, its first 128-row tile index and
// its first 256-row tile-pair index in that order; a CTA item is (sorted
// sample, head, tile or pair) with the tile / pair fastest.
// AttnGeom::debug bits (the C ABI's MF_DEBUG_* values): the TMA producer of
// the forward / backward main kernel drops its streamed-tile loads, so that
// the consumers' bounded waits run out (tests of the timeout path).
constexpr int32_t kDebugDropFwdKV = 1;
constexpr int32_t kDebugDropBwdQdo = 2;

struct AttnGeom {
  const int32_t* cu_seqlens;
  const int32_t* pos;
  const float* rope_cs;
  const float* rope_f;
  const int32_t* frame;
  int32_t rope_axes;
  const int32_t* order;
  int32_t n_samples;
  int32_t total_tokens;
  int32_t heads;
  int32_t n_items;          // work units (tiles or pairs) * heads
  int32_t* status;
  int32_t* timeout_info;    // the plan's timeout record (PlanScalars::timeout_info)
  int32_t debug;            // MF_DEBUG_* flags of mf_debug_inject (0 in normal use)
};

struct FwdArgs {
  AttnGeom g;
  float scale_log2;          // softmax_scale * log2(e), folded into the fp16 Q operand
  const void* q;             // bf16, token rows qk_stride elements apart, [heads, D] each
  const void* k;
  int64_t qk_stride;         // heads * D, or 3 heads * D for a QKV projection's rows
  void* k_rot;               // fp16 [T, heads, D] R(k)
  int32_t* work_counter;     // the persistent kernel's next work item (zeroed by fwd_pre)
  void* o;                   // bf16 [T, heads, D]
  float* lse;                // [heads, T]
};

// The memory-bound chains around a joint-attention block (chain.cu).
cudaError_t launch_norm_modulate(const void* x, const AttnGeom& g, int hidden, const void* shift, const void* scale,
                                 float eps, void* y, cudaStream_t stream);
cudaError_t launch_gate_residual(const void* x, const void* z, const AttnGeom& g, int hidden, const void* gate,
                                 void* out, cudaStream_t stream);

// guided = u + g (c - u) on the conditional image rows of each (cond, uncond)
// sample pair of the pack.
cudaError_t launch_cfg_combine(const void* o, const AttnGeom& g, int head_dim, float guidance, void* out,
                               cudaStream_t stream);

// ev_start / ev_stop (may be null) are recorded around the main kernel.
cudaError_t launch_attn_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, int head_dim, cudaStream_t stream,
                            cudaEvent_t ev_start, cudaEvent_t ev_stop);

struct BwdArgs {
  AttnGeom g;
  float scale;               // softmax_scale
  float scale_log2;          // softmax_scale * log2(e), folded into the fp16 q~ copy
  const void* q;             // bf16 [T, heads, D]
  const void* o;
  const void* dout;
  const float* lse;
  float* dsum;               // [heads, T] rowsum(dO * O)
  void* q_rot;               // fp16 [T, heads, D] q~ = s log2(e) R(q), written by bwd_pre
  float dk_mult;             // dk~ = dk_mult * (dS^T q~) = ln 2 * (dS^T q~)
  float dq_mult;             // dq~ = dq_mult * (dS k~) = s * (dS k~), k~ = R(k) unscaled
  float* dq_acc;             // [T, heads, D] float32 accumulator (zeroed by bwd_pre)
  int32_t* work_counter;     // the persistent kernel's next work item (zeroed by bwd_pre)
  void* dq;
  void* dk;
  void* dv;
};

// tdq: float32 [T][heads][D] view of the dQ accumulator, boxes of 64 tokens
// of one head (used with head_dim 128).
cudaError_t launch_attn_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq, int head_dim,
                            cudaStream_t stream, cudaEvent_t ev_start, cudaEvent_t ev_stop);

}  // namespace mf
