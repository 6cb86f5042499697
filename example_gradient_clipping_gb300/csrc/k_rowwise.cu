// HBM-bound and tiny kernels: one-row norms, clip factors, Gaussian noise, adaptive bound.
#include <algorithm>

#include "common.cuh"

namespace dpk {

// ---------------------------------------------------------------------------
// One-row norm ([FastClip] eq. 6: the per-example gradient of a one-row linear
// layer is the outer product g a^T, so ||g a^T||_F^2 = ||a||^2 ||g||^2; the bias
// gradient is g itself).  One warp per example, 16-byte vector loads when the
// rows are 16-byte aligned, warp-shuffle reduction.
template <class E>
__device__ __forceinline__ float row_sqsum(const E* __restrict__ x, int n, int lane, bool vec) {
  float acc = 0.f;
  constexpr int kVec = 16 / sizeof(E);
  int j0 = 0;
  if (vec) {
    const int nv = n / kVec;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    for (int v = lane; v < nv; v += 32) {
      uint4 w = __ldg(xv + v);
      const E* e = reinterpret_cast<const E*>(&w);
#pragma unroll
      for (int q = 0; q < kVec; ++q) { const float f = to_f(e[q]); acc = fmaf(f, f, acc); }
    }
    j0 = nv * kVec;
  }
  for (int j = j0 + lane; j < n; j += 32) { const float f = to_f(x[j]); acc = fmaf(f, f, acc); }
  return warp_sum(acc);
}

template <class E>
__global__ void __launch_bounds__(256) t1_norm_kernel(Geom g, const E* __restrict__ A,
                                                      const E* __restrict__ G, float* __restrict__ out,
                                                      bool vec_a, bool vec_g) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int w0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (vec_a && vec_g) {
    // Vector path: each warp takes two examples per pass (i and i + warps) and has the loads
    // of both rows of both examples in flight together; the grid is capped, so warps pass
    // over many examples instead of retiring after one.
    constexpr int kVec = 16 / sizeof(E);
    const int nva = g.d / kVec, nvg = g.p / kVec, nv = max(nva, nvg);
    for (int i = w0; i < g.B; i += 2 * warps) {
      const int i2 = i + warps;
      const bool two = i2 < g.B;
      const uint4* av = reinterpret_cast<const uint4*>(A + (size_t)i * g.d);
      const uint4* gv = reinterpret_cast<const uint4*>(G + (size_t)i * g.p);
      const uint4* av2 = reinterpret_cast<const uint4*>(A + (size_t)(two ? i2 : i) * g.d);
      const uint4* gv2 = reinterpret_cast<const uint4*>(G + (size_t)(two ? i2 : i) * g.p);
      float xa = 0.f, xg = 0.f, ya = 0.f, yg = 0.f;
#pragma unroll 2
      for (int v = lane; v < nv; v += 32) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 wa = v < nva ? __ldg(av + v) : z, wg = v < nvg ? __ldg(gv + v) : z;
        const uint4 wa2 = (two && v < nva) ? __ldg(av2 + v) : z, wg2 = (two && v < nvg) ? __ldg(gv2 + v) : z;
        const E* ea = reinterpret_cast<const E*>(&wa);
        const E* eg = reinterpret_cast<const E*>(&wg);
        const E* ea2 = reinterpret_cast<const E*>(&wa2);
        const E* eg2 = reinterpret_cast<const E*>(&wg2);
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          const float fa = to_f(ea[q]), fg = to_f(eg[q]), fa2 = to_f(ea2[q]), fg2 = to_f(eg2[q]);
          xa = fmaf(fa, fa, xa);
          xg = fmaf(fg, fg, xg);
          ya = fmaf(fa2, fa2, ya);
          yg = fmaf(fg2, fg2, yg);
        }
      }
      const E* a = A + (size_t)i * g.d;
      const E* gg = G + (size_t)i * g.p;
      for (int j = nva * kVec + lane; j < g.d; j += 32) { const float f = to_f(a[j]); xa = fmaf(f, f, xa); }
      for (int j = nvg * kVec + lane; j < g.p; j += 32) { const float f = to_f(gg[j]); xg = fmaf(f, f, xg); }
      if (two) {
        const E* a2 = A + (size_t)i2 * g.d;
        const E* g2 = G + (size_t)i2 * g.p;
        for (int j = nva * kVec + lane; j < g.d; j += 32) { const float f = to_f(a2[j]); ya = fmaf(f, f, ya); }
        for (int j = nvg * kVec + lane; j < g.p; j += 32) { const float f = to_f(g2[j]); yg = fmaf(f, f, yg); }
      }
      const float sa = warp_sum(xa), sg = warp_sum(xg), ta = warp_sum(ya), tg = warp_sum(yg);
      if (lane == 0) {
        out[i] = sa * sg + (g.has_bias ? sg : 0.f);
        if (two) out[i2] = ta * tg + (g.has_bias ? tg : 0.f);
      }
    }
    return;
  }
  for (int i = w0; i < g.B; i += warps) {
    const E* a = A + (size_t)i * g.d;
    const E* gg = G + (size_t)i * g.p;
    const float sa = row_sqsum(a, g.d, lane, vec_a);
    const float sg = row_sqsum(gg, g.p, lane, vec_g);
    if (lane == 0) out[i] = sa * sg + (g.has_bias ? sg : 0.f);
  }
}

// ---------------------------------------------------------------------------
// One-row clipped sum: dW[j, m] = sum_i c_i g_i[j] a_i[m], db[j] = sum_i c_i g_i[j]
// (the reweighted sum of [FastClip] section 5 for T = 1: a sum of scaled outer
// products).  Thread -> (j, four consecutive m); a warp reads a_i[m .. m+127]
// coalesced and broadcasts g_i[j]; examples are split over blockIdx.y into partials.
template <class E>
__global__ void __launch_bounds__(256) t1_sum_kernel(Geom g, const E* __restrict__ A, const E* __restrict__ G,
                                                     const float* __restrict__ factors, int ex_per_split,
                                                     float* __restrict__ part_w, float* __restrict__ part_b,
                                                     int accumulate) {
  pdl_trigger();
  pdl_wait();
  const int mq = (g.d + 3) / 4;                      // m quads per row
  const long n_th = (long)g.p * mq;
  const int i0 = blockIdx.y * ex_per_split, i1 = min(g.B, i0 + ex_per_split);
  for (long q = blockIdx.x * (long)blockDim.x + threadIdx.x; q < n_th; q += (long)gridDim.x * blockDim.x) {
    const int j = (int)(q / mq), m0 = (int)(q - (long)j * mq) * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, bacc = 0.f;
    // eight examples' loads in flight per pass, accumulated in example order
    for (int ib = i0; ib < i1; ib += 8) {
      float cg[8], av[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = ib + u;
        cg[u] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) av[u][r] = 0.f;
        if (i < i1) {
          cg[u] = __ldg(factors + i) * to_f(G[(size_t)i * g.p + j]);
          const E* a = A + (size_t)i * g.d + m0;
#pragma unroll
          for (int r = 0; r < 4; ++r)
            if (m0 + r < g.d) av[u][r] = to_f(a[r]);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = fmaf(cg[u], av[u][r], acc[r]);
        bacc += cg[u];
      }
    }
    // partials of split blockIdx.y, or (one split, accumulate) the output itself
    float* out = part_w + ((size_t)blockIdx.y * g.p + j) * g.d + m0;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (m0 + r < g.d) out[r] = accumulate ? out[r] + acc[r] : acc[r];
    if (part_b && m0 == 0) {
      float* ob = part_b + (size_t)blockIdx.y * g.p + j;
      *ob = accumulate ? *ob + bacc : bacc;
    }
  }
}

// ---------------------------------------------------------------------------
// Clip factors: c = 1 if n <= C else C/n ([FastClip] section 2); flat sums the
// layers' squared norms first, per-layer keeps them apart ([ThreeTools] section 2).
struct Bounds { float C[64]; };

__global__ void clip_factors_kernel(const float* __restrict__ sq, int B, int L, int per_layer,
                                    Bounds bounds, const float* __restrict__ Cdev,
                                    float* __restrict__ out, unsigned* status) {
  pdl_trigger();
  pdl_wait();
  const int n_out = per_layer ? B * L : B;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n_out; e += gridDim.x * blockDim.x) {
    float s, C;
    if (per_layer) {
      const int l = e / B;
      s = sq[e];
      C = Cdev ? Cdev[l] : bounds.C[l];
    } else {
      s = 0.f;
      for (int l = 0; l < L; ++l) s += sq[(size_t)l * B + e];
      C = Cdev ? Cdev[0] : bounds.C[0];
    }
    const float n = sqrtf(s);
    float c;
    if (!isfinite(n)) {
      c = 0.f;
      atomicOr(status, kStatusNonfinite);
    } else {
      c = (n <= C) ? 1.f : C / n;
    }
    out[e] = c;
  }
}

// ---------------------------------------------------------------------------
// Gaussian mechanism + 1/B: grad[j] = (grad[j] + sc * z_{offset+j}) * invB.
// One thread per pair of Philox blocks (eight consecutive elements of the global index)
// per pass: both loads are issued first, then the two generator chains run side by side
// (the kernel is bound by the generator's arithmetic at large sizes); float4 load/store
// when the four lie in range and are 16-byte aligned.
__device__ __forceinline__ void noise_block_store(float* __restrict__ grad, size_t n, int64_t j0, bool vec, float4 v,
                                                  const float (&z)[4], float sc, float invB) {
  if (vec) {
    v.x = fmaf(sc, z[0], v.x) * invB;
    v.y = fmaf(sc, z[1], v.y) * invB;
    v.z = fmaf(sc, z[2], v.z) * invB;
    v.w = fmaf(sc, z[3], v.w) * invB;
    __stcs(reinterpret_cast<float4*>(grad + j0), v);
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t j = j0 + r;
      if (j >= 0 && j < (int64_t)n) grad[j] = fmaf(sc, z[r], grad[j]) * invB;
    }
  }
}

// The common case, flat offset % 4 == 0 and grad 16-byte aligned, with fewer than 2^31
// Philox blocks: block b covers grad[4b .. 4b+3], every block full but possibly the last;
// 32-bit indices and no alignment tests per block (the pass is bound by its arithmetic).
template <int NB>
__global__ void __launch_bounds__(256) add_noise_aligned_kernel(float* __restrict__ grad, uint32_t n4, uint32_t tail,
                                                                float sc, float invB, uint64_t seed, uint64_t q0,
                                                                const unsigned long long* __restrict__ seed_dev) {
  pdl_trigger();
  pdl_wait();
  if (seed_dev) seed = *seed_dev;
  const PhiloxKey key = philox_key(seed);
  const uint32_t nb = n4 + (tail ? 1u : 0u);          // blocks touched
  const uint32_t stride = NB * gridDim.x * blockDim.x;
  for (uint32_t b = NB * (blockIdx.x * blockDim.x + threadIdx.x); b < nb; b += stride) {
    float4* g4 = reinterpret_cast<float4*>(grad) + b;
    float4 xa = make_float4(0.f, 0.f, 0.f, 0.f), xb = xa;
    if (b < n4) xa = __ldcs(g4);
    if (NB == 2 && b + 1 < n4) xb = __ldcs(g4 + 1);
    float za[4], zb[4];
    normal4(q0 + b, key, 0u, za);
    if (NB == 2) normal4(q0 + b + 1, key, 0u, zb);
    const size_t n = (size_t)n4 * 4 + tail;
    noise_block_store(grad, n, (int64_t)b * 4, b < n4, xa, za, sc, invB);
    if (NB == 2 && b + 1 < nb) noise_block_store(grad, n, (int64_t)(b + 1) * 4, b + 1 < n4, xb, zb, sc, invB);
  }
}

template <int NB>
__global__ void __launch_bounds__(256) add_noise_kernel(float* __restrict__ grad, size_t n, float sc,
                                                        float invB, uint64_t seed, uint64_t offset,
                                                        const unsigned long long* __restrict__ seed_dev) {
  pdl_trigger();
  pdl_wait();
  if (seed_dev) seed = *seed_dev;
  const PhiloxKey key = philox_key(seed);
  const uint64_t q0 = offset >> 2;
  const uint64_t q1 = (offset + n + 3) >> 2;  // one past the last block touched
  const uint64_t stride = NB * (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t qa = q0 + NB * ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x); qa < q1; qa += stride) {
    const uint64_t qb = qa + 1;
    const bool has_b = NB == 2 && qb < q1;
    const int64_t ja = (int64_t)(qa << 2) - (int64_t)offset, jb = ja + 4;   // index of lane 0 in grad
    const bool va = ja >= 0 && ja + 4 <= (int64_t)n && ((reinterpret_cast<uintptr_t>(grad + ja) & 15u) == 0);
    const bool vb = has_b && jb >= 0 && jb + 4 <= (int64_t)n &&
                    ((reinterpret_cast<uintptr_t>(grad + jb) & 15u) == 0);
    float4 xa = make_float4(0.f, 0.f, 0.f, 0.f), xb = xa;
    if (va) xa = __ldcs(reinterpret_cast<const float4*>(grad + ja));
    if (vb) xb = __ldcs(reinterpret_cast<const float4*>(grad + jb));
    float za[4], zb[4];
    normal4(qa, key, 0u, za);
    if (NB == 2) normal4(qb, key, 0u, zb);
    noise_block_store(grad, n, ja, va, xa, za, sc, invB);
    if (has_b) noise_block_store(grad, n, jb, vb, xb, zb, sc, invB);
  }
}

// ---------------------------------------------------------------------------
// Adaptive bound ([ThreeTools] section 3): C_next = alpha/B (sum_i min(n_i, C_l2)
// + sigma_l2 C_l2 z), C_l2_next = beta C_next.  One block per layer (layer0 + blockIdx.x,
// norms sq[blockIdx.x * B ..], bound Cl2.C[blockIdx.x], out[2 * blockIdx.x ..]); fp64
// accumulation; with seed_dev the seed is read from device memory.
__global__ void __launch_bounds__(256) adaptive_bound_kernel(const float* __restrict__ sq, int B, Bounds Cl2,
                                                             float alpha, float beta, float sigma_l2,
                                                             uint64_t seed,
                                                             const unsigned long long* __restrict__ seed_dev,
                                                             int layer0, float* __restrict__ out,
                                                             unsigned* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ double part[8];
  const float C_l2 = Cl2.C[blockIdx.x];
  const float* sql = sq + (size_t)blockIdx.x * B;
  double acc = 0.0;
  for (int i = threadIdx.x; i < B; i += blockDim.x) {
    const float n = sqrtf(sql[i]);
    // a non-finite norm raises the status (as the clip factors do) and counts as a norm
    // at the bound, min(inf, C_l2) = C_l2
    if (!isfinite(n)) atomicOr(status, kStatusNonfinite);
    acc += isfinite(n) ? (double)fminf(n, C_l2) : (double)C_l2;
  }
  acc = warp_sum_d(acc);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += part[w];
    float z[4];
    const uint64_t e = (uint64_t)(layer0 + (int)blockIdx.x);
    normal4(e >> 2, seed_dev ? (uint64_t)*seed_dev : seed, 1u, z);
    const double cn = (double)alpha / (double)B * (tot + (double)sigma_l2 * (double)C_l2 * (double)z[e & 3]);
    out[2 * blockIdx.x] = (float)cn;
    out[2 * blockIdx.x + 1] = (float)((double)beta * cn);
  }
}

}  // namespace dpk

namespace dph {
using namespace dpk;

cudaError_t launch_t1_norm(const Geom& g, int dtype, const void* A, const void* G, float* out,
                           cudaStream_t s) {
  const int warps_per_block = 8;
  // about eight resident blocks per SM; warps then pass over many examples
  const int blocks = std::min((g.B + warps_per_block - 1) / warps_per_block, 152 * 8);
  const size_t es = dtype == DP_FP32 ? 4 : 2;
  const bool va = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && ((g.d * es) % 16 == 0);
  const bool vg = ((reinterpret_cast<uintptr_t>(G) & 15u) == 0) && ((g.p * es) % 16 == 0);
  if (dtype == DP_FP32)
    launch_pdl(t1_norm_kernel<float>, blocks, 256, 0, s, g, (const float*)A, (const float*)G, out, va, vg);
  else
    launch_pdl(t1_norm_kernel<__nv_bfloat16>, blocks, 256, 0, s, g, (const __nv_bfloat16*)A,
                                                         (const __nv_bfloat16*)G, out, va, vg);
  return cudaGetLastError();
}

cudaError_t launch_clip_factors(const float* sq, int B, int L, int per_layer, const float* C,
                                float* out, unsigned* status, cudaStream_t s) {
  Bounds b{};
  const int nC = per_layer ? L : 1;
  for (int l = 0; l < nC && l < 64; ++l) b.C[l] = C[l];
  // more than 64 per-layer bounds are rejected by the caller
  const int n_out = per_layer ? B * L : B;
  const int blocks = (n_out + 255) / 256;
  launch_pdl(clip_factors_kernel, blocks > 0 ? blocks : 1, 256, 0, s, sq, B, L, per_layer, b, nullptr, out,
                                                              status);
  return cudaGetLastError();
}

cudaError_t launch_add_noise(float* grad, size_t n, float sc, float invB, uint64_t seed,
                             uint64_t offset, const unsigned long long* seed_dev, cudaStream_t s) {
  const uint64_t blocks4 = ((offset + n + 3) >> 2) - (offset >> 2);
  const uint64_t cap = 152ull * 8ull;   // grid-stride beyond 8 resident blocks per SM
  // two Philox blocks per thread and pass once the grid is full anyway, else one
  const bool two = blocks4 >= 2 * cap * 256;
  uint64_t grid = (blocks4 + (two ? 511 : 255)) / (two ? 512 : 256);
  if (grid > cap) grid = cap;
  if (grid == 0) grid = 1;
  const bool aligned = (offset & 3) == 0 && (reinterpret_cast<uintptr_t>(grad) & 15u) == 0 &&
                       blocks4 < ((uint64_t)1 << 31) - 2;
  if (aligned) {
    const uint32_t n4 = (uint32_t)(n >> 2), tail = (uint32_t)(n & 3);
    if (two)
      launch_pdl(add_noise_aligned_kernel<2>, (unsigned)grid, 256, 0, s, grad, n4, tail, sc, invB, seed, offset >> 2,
                 seed_dev);
    else
      launch_pdl(add_noise_aligned_kernel<1>, (unsigned)grid, 256, 0, s, grad, n4, tail, sc, invB, seed, offset >> 2,
                 seed_dev);
  } else if (two) {
    launch_pdl(add_noise_kernel<2>, (unsigned)grid, 256, 0, s, grad, n, sc, invB, seed, offset, seed_dev);
  } else {
    launch_pdl(add_noise_kernel<1>, (unsigned)grid, 256, 0, s, grad, n, sc, invB, seed, offset, seed_dev);
  }
  return cudaGetLastError();
}

cudaError_t launch_adaptive_bound(const float* sq, int B, int L, const float* C_l2, float alpha, float beta,
                                  float sigma_l2, uint64_t seed, const unsigned long long* seed_dev, int layer0,
                                  float* out, unsigned* status, cudaStream_t s) {
  if (L < 1 || L > 64) return cudaErrorInvalidValue;
  Bounds b{};
  for (int l = 0; l < L; ++l) b.C[l] = C_l2[l];
  launch_pdl(adaptive_bound_kernel, (unsigned)L, 256, 0, s, sq, B, b, alpha, beta, sigma_l2, seed, seed_dev, layer0,
             out, status);
  return cudaGetLastError();
}

// Examples per split of the one-row clipped sum: enough splits to give the SMs about two
// blocks each, 8 to 32 examples per split (one to four passes of eight loads in flight; the
// cap also bounds each thread's fp32 accumulation chain).
static int t1_sum_eps(const Geom& g) {
  const long n_th = (long)g.p * ((g.d + 3) / 4);
  const long bx = std::min<long>((n_th + 255) / 256, 152L * 8);
  const long want = std::max<long>(1, (2L * 152 + bx - 1) / bx);
  const long eps = std::min<long>(32, std::max<long>(8, (g.B + want - 1) / want));
  return (int)std::min<long>(g.B, eps);
}
int t1_sum_splits(const Geom& g) { const int e = t1_sum_eps(g); return (g.B + e - 1) / e; }
size_t t1_sum_ws_bytes(const Geom& g) {
  return (size_t)t1_sum_splits(g) * ((size_t)g.p * g.d + g.p) * sizeof(float);
}

cudaError_t launch_t1_sum(const Geom& g, int dtype, const void* A, const void* G, const float* factors, float* dW,
                          float* db, int accumulate, float* ws, cudaStream_t s, NoiseArgs* nz) {
  const int eps = t1_sum_eps(g), splits = t1_sum_splits(g);
  const bool direct = splits == 1;           // one split writes dW and db itself
  float* part_w = direct ? dW : ws;
  float* part_b = db ? (direct ? db : ws + (size_t)splits * g.p * g.d) : nullptr;
  const int acc = direct ? accumulate : 0;
  const long n_th = (long)g.p * ((g.d + 3) / 4);
  dim3 grid((unsigned)std::min<long>((n_th + 255) / 256, 152L * 8), (unsigned)splits);
  if (dtype == DP_FP32)
    launch_pdl(t1_sum_kernel<float>, grid, 256, 0, s, g, (const float*)A, (const float*)G, factors, eps, part_w, part_b,
               acc);
  else
    launch_pdl(t1_sum_kernel<__nv_bfloat16>, grid, 256, 0, s, g, (const __nv_bfloat16*)A, (const __nv_bfloat16*)G,
                                                      factors, eps, part_w, part_b, acc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || direct) return e;
  const size_t nw = (size_t)g.p * g.d;
  return launch_reduce_splits2(SplitSeg{part_w, nw, nw, dW}, SplitSeg{part_b, (size_t)g.p, db ? (size_t)g.p : 0, db},
                               splits, accumulate, s, nz);
}

}  // namespace dph
