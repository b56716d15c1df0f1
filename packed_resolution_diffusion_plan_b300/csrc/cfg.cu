// Classifier-free guidance over a pack of (conditional, unconditional) sample
// pairs.
//
// Mage-Flow review, section on classifier-free guidance: the conditional and
// unconditional branches run in one packed forward.  The pages do not print
// the combination; the standard reading is used:
//     guided = u + g (c - u)
// for the image rows of each pair, with samples 2p (conditional) and 2p + 1
// (unconditional) of the pack.  Image rows end each sample and both members
// of a pair have the same number of them, so row j from the end of one pairs
// with row j from the end of the other whatever their text lengths.
#include "../../include/mf.h"
#include "common.cuh"
#include "ptx.cuh"

namespace mf {
namespace {

// One thread per (token, head, 8-column chunk); only the conditional
// samples' image rows write.  A row whose partner does not sit at the same
// latent position (the pair's image sizes differ) is skipped and raises
// kStatusPairing.
template <int D>
__global__ void cfg_combine_kernel(const void* o, const AttnGeom g, float guidance, void* out) {
  constexpr int kChunks = D / 8;
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rows = static_cast<long long>(g.total_tokens) * g.heads;
  if (gid >= rows * kChunks) return;
  const long long row = gid / kChunks;
  const int ch = static_cast<int>(gid % kChunks);
  const int tok = static_cast<int>(row / g.heads);
  const int h = static_cast<int>(row % g.heads);
  const int2* pos = reinterpret_cast<const int2*>(g.pos);
  if (pos[tok].x < 0) return;  // text row
  int lo = 0, hi = g.n_samples;  // sample s with cu[s] <= tok < cu[s+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (g.cu_seqlens[mid] <= tok) lo = mid; else hi = mid;
  }
  if (lo & 1) return;  // unconditional sample: read, not written
  // Same image size: the partner row has the same latent position (and
  // frame); anything else means the pair's images differ.
  const int partner = tok - g.cu_seqlens[lo + 1] + g.cu_seqlens[lo + 2];
  const int2 pt = pos[tok];
  if (partner < g.cu_seqlens[lo + 1] || pos[partner].x != pt.x || pos[partner].y != pt.y ||
      g.frame[partner] != g.frame[tok]) {
    atomicOr(g.status, kStatusPairing);
    return;
  }
  const long long prow = static_cast<long long>(partner) * g.heads + h;
  const uint4 c = reinterpret_cast<const uint4*>(o)[gid];
  const uint4 u = reinterpret_cast<const uint4*>(o)[prow * kChunks + ch];
  const uint32_t* cw = reinterpret_cast<const uint32_t*>(&c);
  const uint32_t* uw = reinterpret_cast<const uint32_t*>(&u);
  uint32_t r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float u0 = bf16_lo(uw[e]), u1 = bf16_hi(uw[e]);
    r[e] = pack_bf16(fmaf(guidance, bf16_lo(cw[e]) - u0, u0), fmaf(guidance, bf16_hi(cw[e]) - u1, u1));
  }
  reinterpret_cast<uint4*>(out)[gid] = make_uint4(r[0], r[1], r[2], r[3]);
}

}  // namespace

cudaError_t launch_cfg_combine(const void* o, const AttnGeom& g, int head_dim, float guidance, void* out,
                               cudaStream_t stream) {
  const long long chunks = static_cast<long long>(g.total_tokens) * g.heads * (head_dim / 8);
  if (chunks == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((chunks + 255) / 256);
  if (head_dim == 128) cfg_combine_kernel<128><<<blocks, 256, 0, stream>>>(o, g, guidance, out);
  else cfg_combine_kernel<64><<<blocks, 256, 0, stream>>>(o, g, guidance, out);
  return cudaGetLastError();
}

}  // namespace mf
