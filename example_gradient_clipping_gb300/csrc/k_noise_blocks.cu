// The Gaussian mechanism and the 1/B average over several blocks of one flat gradient in
// one launch, each block with its own bound ([FastClip] section 2; [ThreeTools] section 2
// for per-layer bounds): grad[e] <- (grad[e] + sigma C_b z_e) / B for e in block b, z_e lane
// e % 4 of normal4(e / 4) -- the arithmetic of the single-block noise pass, so the result
// equals one dp_add_noise call per block.  Work items are the Philox blocks (four flat
// indices) each block touches; a block boundary inside a Philox block gives that Philox
// block to both neighbours, each writing only its own elements.
#include <algorithm>

#include "common.cuh"

namespace dpk {

__global__ void __launch_bounds__(256) add_noise_blocks_kernel(float* __restrict__ grad, NoiseBlocks nb, float invB,
                                                               uint64_t seed,
                                                               const unsigned long long* __restrict__ seed_dev) {
  pdl_trigger();
  pdl_wait();
  if (seed_dev) seed = *seed_dev;
  const uint64_t total = nb.qcum[nb.count];
  for (uint64_t q = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total;
       q += (uint64_t)gridDim.x * blockDim.x) {
    int b = 0;
    while (b + 1 < nb.count && nb.qcum[b + 1] <= q) ++b;     // blocks in flat order, few of them
    const uint64_t lo = nb.off[b], hi = lo + nb.n[b];
    const uint64_t e0 = ((lo >> 2) + (q - nb.qcum[b])) << 2;  // first flat index of the Philox block
    float z[4];
    normal4(e0 >> 2, seed, 0u, z);
    const float sc = nb.sc[b];
    float* g = grad + e0;
    if (e0 >= lo && e0 + 4 <= hi && (reinterpret_cast<uintptr_t>(g) & 15u) == 0) {
      float4 v = __ldcs(reinterpret_cast<const float4*>(g));
      v.x = fmaf(sc, z[0], v.x) * invB;
      v.y = fmaf(sc, z[1], v.y) * invB;
      v.z = fmaf(sc, z[2], v.z) * invB;
      v.w = fmaf(sc, z[3], v.w) * invB;
      __stcs(reinterpret_cast<float4*>(g), v);
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (e0 + r >= lo && e0 + r < hi) g[r] = fmaf(sc, z[r], g[r]) * invB;
    }
  }
}

}  // namespace dpk

namespace dph {
using namespace dpk;

cudaError_t launch_add_noise_blocks(float* grad, const NoiseBlocks& nb, float invB, uint64_t seed,
                                    const unsigned long long* seed_dev, cudaStream_t s) {
  const uint64_t total = nb.qcum[nb.count];
  if (!total) return cudaSuccess;
  const unsigned blocks = (unsigned)std::min<uint64_t>((total + 255) / 256, 152ull * 16);
  launch_pdl(add_noise_blocks_kernel, blocks, 256, 0, s, grad, nb, invB, seed, seed_dev);
  return cudaGetLastError();
}

}  // namespace dph
