// The memory-bound chains around one joint-attention block, each fused into a
// single pass over HBM.
//
// Mage-Flow review, kernel-fusion section: normalisation, adaptive
// modulation, RoPE application, gating and the residual add are memory-bound
// chains that, run as separate kernels, re-read and re-write large
// activations; fused, only the final output is written.  The pages do not
// give the operations' exact form; the plainest reading for a diffusion
// transformer block is used:
//   norm_modulate   y = LN(x) (1 + scale_s) + shift_s   (LayerNorm over the
//                   hidden size, no affine, eps inside the square root;
//                   per-sample modulation vectors of the sample s a token
//                   belongs to)
//   gate_residual   out = x + gate_s * z                 (after the output
//                   projection)
// The RoPE application of the chain runs in the attention forward's first
// pass, which reads q and k straight from the QKV projection's rows
// (mf_attn_fwd_qkv).
#include "common.cuh"
#include "ptx.cuh"

namespace mf {
namespace {

// Sample of token `tok`: the s with cu[s] <= tok < cu[s + 1].
__device__ __forceinline__ int sample_of(const int32_t* cu, int n, int tok) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= tok) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = bf16_lo(w[e]);
    f[2 * e + 1] = bf16_hi(w[e]);
  }
}

// One CTA of 128 threads per token row of kNch * 1024 elements: every thread
// keeps its kNch 8-element chunks in registers, so x is read once.
template <int kNch>
__global__ void __launch_bounds__(128) norm_modulate_kernel(const uint4* x, const int32_t* cu, int n_samples,
                                                            const uint4* shift, const uint4* scale, float eps,
                                                            uint4* y) {
  constexpr int C8 = kNch * 128;  // uint4 chunks per row
  __shared__ float red[2][4];
  const int tok = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float v[kNch][8];
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < kNch; ++c) {
    unpack8(x[static_cast<size_t>(tok) * C8 + c * 128 + t], v[c]);
#pragma unroll
    for (int e = 0; e < 8; ++e) sum += v[c][e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[0][warp] = sum;
  __syncthreads();
  const float mean = (red[0][0] + red[0][1] + red[0][2] + red[0][3]) * (1.0f / (kNch * 1024));
  float sq = 0.f;
#pragma unroll
  for (int c = 0; c < kNch; ++c)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float d = v[c][e] - mean;
      sq += d * d;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0) red[1][warp] = sq;
  __syncthreads();
  const float var = (red[1][0] + red[1][1] + red[1][2] + red[1][3]) * (1.0f / (kNch * 1024));
  const float rstd = rsqrtf(var + eps);
  const int s = sample_of(cu, n_samples, tok);
#pragma unroll
  for (int c = 0; c < kNch; ++c) {
    float sh[8], sc[8];
    unpack8(__ldg(shift + static_cast<size_t>(s) * C8 + c * 128 + t), sh);
    unpack8(__ldg(scale + static_cast<size_t>(s) * C8 + c * 128 + t), sc);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16(fmaf((v[c][2 * e] - mean) * rstd, 1.0f + sc[2 * e], sh[2 * e]),
                       fmaf((v[c][2 * e + 1] - mean) * rstd, 1.0f + sc[2 * e + 1], sh[2 * e + 1]));
    y[static_cast<size_t>(tok) * C8 + c * 128 + t] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One thread per 8-element chunk: out = x + gate_s * z.
__global__ void gate_residual_kernel(const uint4* x, const uint4* z, const int32_t* cu, int n_samples,
                                     const uint4* gate, long long chunks, int c8, uint4* out) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= chunks) return;
  const int tok = static_cast<int>(gid / c8), ch = static_cast<int>(gid % c8);
  const int s = sample_of(cu, n_samples, tok);
  float xv[8], zv[8], gv[8];
  unpack8(x[gid], xv);
  unpack8(z[gid], zv);
  unpack8(__ldg(gate + static_cast<size_t>(s) * c8 + ch), gv);
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    w[e] = pack_bf16(fmaf(gv[2 * e], zv[2 * e], xv[2 * e]), fmaf(gv[2 * e + 1], zv[2 * e + 1], xv[2 * e + 1]));
  out[gid] = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

cudaError_t launch_norm_modulate(const void* x, const AttnGeom& g, int hidden, const void* shift, const void* scale,
                                 float eps, void* y, cudaStream_t stream) {
  const int T = g.total_tokens;
  if (T == 0) return cudaSuccess;
  const uint4 *xi = static_cast<const uint4*>(x), *sh = static_cast<const uint4*>(shift),
              *sc = static_cast<const uint4*>(scale);
  uint4* yo = static_cast<uint4*>(y);
  switch (hidden / 1024) {
    case 1: norm_modulate_kernel<1><<<T, 128, 0, stream>>>(xi, g.cu_seqlens, g.n_samples, sh, sc, eps, yo); break;
    case 2: norm_modulate_kernel<2><<<T, 128, 0, stream>>>(xi, g.cu_seqlens, g.n_samples, sh, sc, eps, yo); break;
    case 3: norm_modulate_kernel<3><<<T, 128, 0, stream>>>(xi, g.cu_seqlens, g.n_samples, sh, sc, eps, yo); break;
    case 4: norm_modulate_kernel<4><<<T, 128, 0, stream>>>(xi, g.cu_seqlens, g.n_samples, sh, sc, eps, yo); break;
    case 6: norm_modulate_kernel<6><<<T, 128, 0, stream>>>(xi, g.cu_seqlens, g.n_samples, sh, sc, eps, yo); break;
    case 8: norm_modulate_kernel<8><<<T, 128, 0, stream>>>(xi, g.cu_seqlens, g.n_samples, sh, sc, eps, yo); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_gate_residual(const void* x, const void* z, const AttnGeom& g, int hidden, const void* gate,
                                 void* out, cudaStream_t stream) {
  const long long chunks = static_cast<long long>(g.total_tokens) * (hidden / 8);
  if (chunks == 0) return cudaSuccess;
  gate_residual_kernel<<<static_cast<unsigned>((chunks + 255) / 256), 256, 0, stream>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(z), g.cu_seqlens, g.n_samples,
      static_cast<const uint4*>(gate), chunks, hidden / 8, static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace mf
