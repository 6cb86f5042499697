// Clipped sum from kept per-example gradients.
//
// When a layer's norm was formed by instantiating g_i ([MixGhost] section 3, the
// FastGradClip side of the mixed clipping), the instantiating kernel can also store g_i
// and b_i; the clipped sum is then the weighted gradient dW = sum_i c_i g_i, db =
// sum_i c_i b_i formed from the stored per-sample gradients, as the Opacus approach of
// [MixGhost] section 2 ("Previous arts") does -- fast but memory-costly -- at the 2BpD
// time of its Appendix C.5, instead of a second contraction over the T rows (2BTpD).
//
// kept_wsum_direct_kernel: a block per chunk of kPer 4-element items of the per-example
// layout, over all B examples: its kGroups thread groups sum c_i g_i over consecutive
// example ranges in order, eight to sixteen examples' loads in flight (two batches of eight,
// the next issued before the current is summed), then the groups' sums are added in group
// order, one thread per element, and written straight to their weight (or bias) positions
// (conv: mapping the kernel's tile column order back to the weight layout) -- one launch and
// one read of the kept gradients, no partial sums.  With nz on, each output also gets its noise and the 1/B
// scale on the way out, z drawn at its flat index with the noise pass's arithmetic (so the
// result is the same as the sum followed by that pass).  Small layers (fewer item blocks than
// half the SMs: VGG-11's first conv layer has 7) split the examples over blockIdx.y as well;
// each split's group-ordered sums go to a partial row, and kept_wsum_finish_kernel adds the
// splits in order and writes as above.
#include <algorithm>

#include "tc.cuh"

namespace dpk {

constexpr int kPer = 64, kGroups = 8;   // items per block, example groups (512 threads)

// Weight position of element f of a kept gradient's per-example layout: conv_kk == 0 the
// weight layout itself; else tile columns col = (c / 64 * kk + tap) * 64 + c % 64 of rows n,
// stored [n][col] (width D) or column-quad major ([col / 4][n][4]), mapped to n * D + c * kk + tap.
__device__ __forceinline__ long kept_pos(size_t f, int p, int D, int kk, int quad) {
  if (kk == 0) return (long)f;
  int n, col;
  if (quad) {
    const size_t qd = f / (4 * (size_t)p), r = f - qd * 4 * (size_t)p;
    n = (int)(r >> 2);
    col = (int)(qd * 4 + (r & 3));
  } else {
    n = (int)(f / D);
    col = (int)(f - (size_t)n * D);
  }
  const int blk = col >> 6, tap = blk % kk, c = (blk / kk) * 64 + (col & 63);
  if (c * kk >= D) return -1;   // (no such channel)
  return (long)n * D + (long)c * kk + tap;
}

// Sum v of element i (0..3) of item it to its weight or bias position, with the accumulate
// flag and the fused noise.
__device__ __forceinline__ void kept_write1(size_t it, int i, size_t iw, float v, int p, int D, int kk, int quad,
                                            float* __restrict__ dW, float* __restrict__ db, int accumulate,
                                            const NoiseArgs& nz, uint64_t seed) {
  if (it < iw) {
    const long m = kept_pos(it * 4 + i, p, D, kk, quad);
    if (m >= 0) {
      if (accumulate) v += dW[m];
      if (nz.on) v = fmaf(nz.sc, noise_z1(nz.off_a + (uint64_t)m, seed), v) * nz.invB;
      dW[m] = v;
    }
  } else {
    const size_t j = (it - iw) * 4 + i;
    if (accumulate) v += db[j];
    if (nz.on) v = fmaf(nz.sc, noise_z1(nz.off_b + j, seed), v) * nz.invB;
    db[j] = v;
  }
}

__global__ void __launch_bounds__(kPer * kGroups) kept_wsum_direct_kernel(
    const float* __restrict__ keep, const float* __restrict__ keep_b, const float* __restrict__ factors, int B,
    size_t nw, int p, int D, int kk, int quad, float* __restrict__ dW, float* __restrict__ db, int accumulate,
    NoiseArgs nz, float4* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  const uint64_t seed = nz.on && nz.seed_dev ? (uint64_t)*nz.seed_dev : nz.seed;
  __shared__ float4 red[kGroups][kPer];
  const size_t iw = nw / 4, items = iw + (keep_b ? (size_t)p / 4 : 0);
  const int lane_item = threadIdx.x % kPer, grp = threadIdx.x / kPer;
  const size_t it = (size_t)blockIdx.x * kPer + lane_item;
  // this block's examples: split blockIdx.y of gridDim.y, then group grp of kGroups
  const int es = (B + gridDim.y - 1) / gridDim.y, sb = blockIdx.y * es, se = min(B, sb + es);
  const int eg = (es + kGroups - 1) / kGroups, e0 = sb + grp * eg, e1 = min(se, e0 + eg);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (it < items) {
    const bool w = it < iw;
    const float* src = w ? keep + it * 4 : keep_b + (it - iw) * 4;
    const size_t stride = w ? nw : (size_t)p;
    // examples e0 .. e1 - 1 in batches of eight, summed in example order; the next batch's
    // loads are issued before the current batch is summed, so eight to sixteen are in flight
    float4 va[8], vb[8];
    float ca[8], cb[8];
    auto load = [&](float4 (&v)[8], float (&c)[8], int e) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (e + q < e1) {
          v[q] = __ldcs(reinterpret_cast<const float4*>(src + (size_t)(e + q) * stride));
          c[q] = __ldg(factors + e + q);
        }
      }
    };
    auto add = [&](const float4 (&v)[8], const float (&c)[8], int e) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (e + q < e1) {
          acc.x = fmaf(c[q], v[q].x, acc.x);
          acc.y = fmaf(c[q], v[q].y, acc.y);
          acc.z = fmaf(c[q], v[q].z, acc.z);
          acc.w = fmaf(c[q], v[q].w, acc.w);
        }
      }
    };
    if (e0 < e1) load(va, ca, e0);
    for (int e = e0; e < e1; e += 16) {
      if (e + 8 < e1) load(vb, cb, e + 8);
      add(va, ca, e);
      if (e + 16 < e1) load(va, ca, e + 16);
      if (e + 8 < e1) add(vb, cb, e + 8);
    }
  }
  red[grp][lane_item] = acc;
  __syncthreads();
  // one thread per element of the block's items: the groups' sums added in group order
  if (threadIdx.x < 4 * kPer) {
    const int li = threadIdx.x >> 2, i = threadIdx.x & 3;
    const size_t iti = (size_t)blockIdx.x * kPer + li;
    if (iti < items) {
      const float* r = reinterpret_cast<const float*>(&red[0][0]);
      float v = r[li * 4 + i];
#pragma unroll
      for (int g = 1; g < kGroups; ++g) v += r[(g * kPer + li) * 4 + i];
      if (part) reinterpret_cast<float*>(part + (size_t)blockIdx.y * items + iti)[i] = v;
      else kept_write1(iti, i, iw, v, p, D, kk, quad, dW, db, accumulate, nz, seed);
    }
  }
}

// The splits' partial rows added in split order, then written as the one-launch kernel does.
__global__ void __launch_bounds__(256) kept_wsum_finish_kernel(const float4* __restrict__ part, int splits, size_t iw,
                                                               size_t items, int p, int D, int kk, int quad,
                                                               float* __restrict__ dW, float* __restrict__ db,
                                                               int accumulate, NoiseArgs nz) {
  pdl_trigger();
  pdl_wait();
  const uint64_t seed = nz.on && nz.seed_dev ? (uint64_t)*nz.seed_dev : nz.seed;
  for (size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (size_t)gridDim.x * blockDim.x) {
    float4 s = part[it];
    for (int k = 1; k < splits; ++k) {
      const float4 t = part[(size_t)k * items + it];
      s.x += t.x;
      s.y += t.y;
      s.z += t.z;
      s.w += t.w;
    }
    kept_write1(it, 0, iw, s.x, p, D, kk, quad, dW, db, accumulate, nz, seed);
    kept_write1(it, 1, iw, s.y, p, D, kk, quad, dW, db, accumulate, nz, seed);
    kept_write1(it, 2, iw, s.z, p, D, kk, quad, dW, db, accumulate, nz, seed);
    kept_write1(it, 3, iw, s.w, p, D, kk, quad, dW, db, accumulate, nz, seed);
  }
}

}  // namespace dpk

namespace dph {
using namespace dpk;

// Example splits: one unless the item blocks fill less than half the SMs; then enough to
// give about two blocks per SM, each split at least 64 examples.
static int kept_splits(int B, int p, int D) {
  const long blocks = (long)(((size_t)p * D / 4 + p / 4 + kPer - 1) / kPer);
  if (blocks * 2 >= 152) return 1;
  return (int)std::max<long>(1, std::min<long>((304 + blocks - 1) / blocks, B / 64));
}

size_t kept_sum_ws_bytes(int B, int p, int D) {
  const int s = kept_splits(B, p, D);
  return s > 1 ? (size_t)s * ((size_t)p * D / 4 + p / 4) * 16 : 256;
}

cudaError_t launch_kept_sum(int B, int p, int D, int conv_kk, const float* keep, const float* keep_b,
                            const float* factors, float* dW, float* db, int accumulate, cudaStream_t s, bool quad,
                            NoiseArgs* nz, void* ws) {
  if (((size_t)p * D) % 4 || p % 4) return cudaErrorInvalidValue;
  const bool bias = db && keep_b;
  const size_t nw = (size_t)p * D;
  const size_t items = nw / 4 + (bias ? (size_t)p / 4 : 0);
  NoiseArgs none = {};
  const NoiseArgs& na = nz && nz->on ? *nz : none;
  const int splits = kept_splits(B, p, D);
  float4* part = splits > 1 ? static_cast<float4*>(ws) : nullptr;
  if (splits > 1 && !ws) return cudaErrorInvalidValue;
  launch_pdl(kept_wsum_direct_kernel, dim3((unsigned)((items + kPer - 1) / kPer), (unsigned)splits), kPer * kGroups,
             0, s, keep, bias ? keep_b : nullptr, factors, B, nw, p, D, conv_kk, quad ? 1 : 0, dW, db, accumulate, na,
             part);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && splits > 1) {
    const unsigned blocks = (unsigned)std::min<size_t>((items + 255) / 256, 152 * 4);
    launch_pdl(kept_wsum_finish_kernel, blocks, 256, 0, s, (const float4*)part, splits, nw / 4, items, p, D, conv_kk,
               quad ? 1 : 0, dW, db, accumulate, na);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && nz && nz->on) {
    nz->applied_a = 1;
    nz->applied_b = bias ? 1 : nz->applied_b;
  }
  return e;
}

}  // namespace dph
