// SIMT (FFMA) kernels for every norm and sum path, any dtype and shape.
//
// They serve fp32 layers (whose 1e-5 tolerance rules out reduced-precision tensor
// cores) and shapes the tensor-core kernels do not take.  All accumulate in fp32.
#include <algorithm>

#include "common.cuh"

namespace dpk {

constexpr int kBM = 64, kBN = 64, kBK = 16, kThreads = 256;

// ---------------------------------------------------------------------------
// Row-contraction tile: acc += sum_{r in [r0, r1)} w(r) X(r, m) Y(r, n) for the
// 64x64 tile at (m0, n0), X = output grads (m < p), Y = (unfolded) inputs (n < D),
// row r = i*T + t.  This is the per-example gradient G_i^T U(A_i) when the rows
// are one example's, and the reweighted contraction sum_i c_i G_i^T U(A_i)
// ([FastClip] section 5, the reweighted loss) when they span the batch.
// With colsum != nullptr, threads 0..63 also accumulate sum_r w(r) X(r, m0+tid).
template <class E, bool SCALE>
__device__ __forceinline__ void rows_tile(const Geom& g, const E* __restrict__ A,
                                          const E* __restrict__ G, const float* __restrict__ w,
                                          int m0, int n0, long r0, long r1, float acc[4][4],
                                          float* colsum, float (*Xs)[kBM + 4],
                                          float (*Ys)[kBN + 4]) {
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  for (long rb = r0; rb < r1; rb += kBK) {
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int kk, mm;
      if (!g.conv) { mm = tid & 63; kk = (tid >> 6) + 4 * q; }
      else { kk = tid & 15; mm = (tid >> 4) + 16 * q; }
      const long r = rb + kk;
      const int m = m0 + mm;
      float v = 0.f;
      if (r < r1 && m < g.p) {
        const int i = (int)(r / g.T), t = (int)(r - (long)i * g.T);
        v = ld_g(G, g, i, t, m);
        if (SCALE) v *= w[i];
      }
      Xs[kk][mm] = v;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int kk, nn;
      if (!g.conv) { nn = tid & 63; kk = (tid >> 6) + 4 * q; }
      else { kk = tid & 15; nn = (tid >> 4) + 16 * q; }
      const long r = rb + kk;
      const int n = n0 + nn;
      float v = 0.f;
      if (r < r1 && n < g.D) {
        const int i = (int)(r / g.T), t = (int)(r - (long)i * g.T);
        v = ld_a(A, g, i, t, n);
      }
      Ys[kk][nn] = v;
    }
    __syncthreads();
    if (colsum && tid < kBM) {
      float s = 0.f;
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) s += Xs[kk][tid];
      *colsum += s;
    }
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Ys[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
  }
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0)
    for (int j = 0; j < (int)(blockDim.x >> 5); ++j) t += red[j];
  return t;  // valid in thread 0
}

// Clipped sum, split over rows: ws[split] holds the partial [p, D] and ws_db[split] [p].
template <class E>
__global__ void __launch_bounds__(kThreads) simt_clipped_sum_kernel(Geom g, const E* __restrict__ A,
                                                                    const E* __restrict__ G,
                                                                    const float* __restrict__ fac,
                                                                    float* __restrict__ ws,
                                                                    float* __restrict__ ws_db,
                                                                    long rows_per_split) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float Xs[kBK][kBM + 4];
  __shared__ __align__(16) float Ys[kBK][kBN + 4];
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN, split = blockIdx.z;
  const long R = (long)g.B * g.T;
  const long r0 = (long)split * rows_per_split;
  const long r1 = min(R, r0 + rows_per_split);
  float acc[4][4] = {};
  float cs = 0.f;
  const bool do_db = (blockIdx.y == 0) && ws_db;
  rows_tile<E, true>(g, A, G, fac, m0, n0, r0, r1, acc, do_db ? &cs : nullptr, Xs, Ys);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float* out = ws + (size_t)split * g.p * g.D;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + ty * 4 + u;
    if (m >= g.p) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int n = n0 + tx * 4 + v;
      if (n < g.D) out[(size_t)m * g.D + n] = acc[u][v];
    }
  }
  if (do_db && threadIdx.x < kBM && m0 + threadIdx.x < g.p)
    ws_db[(size_t)split * g.p + m0 + threadIdx.x] = cs;
}

// out[e] (+)= sum_s ws[s*n + e]  (fixed order: deterministic)
// With nz.on, the reductions below also add the Gaussian noise of element e (flat index
// noff + e) and the 1/B scale on the way out, as the separate noise pass does.
__device__ __forceinline__ float with_noise(const NoiseArgs& nz, uint64_t seed, uint64_t e, float v) {
  return nz.on ? fmaf(nz.sc, noise_z1(e, seed), v) * nz.invB : v;
}

__global__ void reduce_splits_kernel(const float* __restrict__ ws, int splits, size_t n,
                                     float* __restrict__ out, int accumulate, NoiseArgs nz, uint64_t noff) {
  pdl_trigger();
  pdl_wait();
  const uint64_t seed = nz.on && nz.seed_dev ? (uint64_t)*nz.seed_dev : nz.seed;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    float s = accumulate ? out[e] : 0.f;
    for (int k = 0; k < splits; ++k) s += ws[(size_t)k * n + e];
    out[e] = with_noise(nz, seed, noff + e, s);
  }
}

// Two segments (the weight and the bias of one layer) in one pass; V = 4: float4 items
// (every base 16-byte aligned, strides and lengths multiples of 4), V = 1: floats.  Each
// element adds its splits in ascending order, eight loads in flight.
template <int V>
__global__ void reduce_splits2_kernel(SplitSeg a, SplitSeg b, int splits, int accumulate, NoiseArgs nz) {
  pdl_trigger();
  pdl_wait();
  const uint64_t seed = nz.on && nz.seed_dev ? (uint64_t)*nz.seed_dev : nz.seed;
  const size_t ia = a.n / V, items = ia + b.n / V;
  for (size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (size_t)gridDim.x * blockDim.x) {
    const bool first = it < ia;
    const size_t off = (first ? it : it - ia) * V;
    const float* src = (first ? a.ws : b.ws) + off;
    const size_t stride = first ? a.stride : b.stride;
    float* out = (first ? a.out : b.out) + off;
    float acc[V];
    if (accumulate) {
      if constexpr (V == 4) {
        const float4 o = *reinterpret_cast<const float4*>(out);
        acc[0] = o.x; acc[1] = o.y; acc[2] = o.z; acc[3] = o.w;
      } else {
        acc[0] = out[0];
      }
    } else {
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = 0.f;
    }
    for (int k0 = 0; k0 < splits; k0 += 8) {
      float v[8][V];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (k0 + j >= splits) break;
        const float* p = src + (size_t)(k0 + j) * stride;
        if constexpr (V == 4) {
          const float4 t = *reinterpret_cast<const float4*>(p);
          v[j][0] = t.x; v[j][1] = t.y; v[j][2] = t.z; v[j][3] = t.w;
        } else {
          v[j][0] = p[0];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (k0 + j >= splits) break;
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] += v[j][q];
      }
    }
    if (nz.on) {
      const uint64_t e0 = (first ? nz.off_a : nz.off_b) + off;
      float z[V];
      if constexpr (V == 4) noise_z4(e0, seed, z);
      else z[0] = noise_z1(e0, seed);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = fmaf(nz.sc, z[q], acc[q]) * nz.invB;
    }
    if constexpr (V == 4) *reinterpret_cast<float4*>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else out[0] = acc[0];
  }
}

// Many splits of a short vector: one warp per element, lanes stride over the splits,
// then a fixed butterfly (deterministic).
__global__ void reduce_splits_warp_kernel(const float* __restrict__ ws, int splits, size_t n,
                                          float* __restrict__ out, int accumulate, NoiseArgs nz, uint64_t noff) {
  pdl_trigger();
  pdl_wait();
  const uint64_t seed = nz.on && nz.seed_dev ? (uint64_t)*nz.seed_dev : nz.seed;
  const int lane = threadIdx.x & 31;
  const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
  for (size_t e = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; e < n; e += nw) {
    float s = 0.f;
    for (int k = lane; k < splits; k += 32) s += ws[(size_t)k * n + e];
    s = warp_sum(s);
    if (lane == 0) out[e] = with_noise(nz, seed, noff + e, accumulate ? out[e] + s : s);
  }
}

// Very many splits of a short vector: one block per element, threads stride over the
// splits, then a fixed tree over the block (deterministic).
__global__ void reduce_splits_block_kernel(const float* __restrict__ ws, int splits, size_t n,
                                           float* __restrict__ out, int accumulate, NoiseArgs nz, uint64_t noff) {
  pdl_trigger();
  pdl_wait();
  const uint64_t seed = nz.on && nz.seed_dev ? (uint64_t)*nz.seed_dev : nz.seed;
  __shared__ float red[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (size_t e = blockIdx.x; e < n; e += gridDim.x) {
    float s = 0.f;
    for (int k = threadIdx.x; k < splits; k += blockDim.x) s += ws[(size_t)k * n + e];
    s = warp_sum(s);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (warp == 0) {
      float t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
      t = warp_sum(t);
      if (lane == 0) out[e] = with_noise(nz, seed, noff + e, accumulate ? out[e] + t : t);
    }
    __syncthreads();
  }
}

// Instantiated norm: CTA (bx, by, i) forms the 64x64 tile of g_i = G_i^T U(A_i)
// over all T rows of example i, squares and sums it ([MixGhost] Appendix C.4).
// CTAs with by == 0 also form the bias gradient sum_t G_i[t, :] of their rows.
template <class E>
__global__ void __launch_bounds__(kThreads) simt_inst_kernel(Geom g, const E* __restrict__ A,
                                                             const E* __restrict__ G,
                                                             float* __restrict__ ws_w,
                                                             float* __restrict__ ws_b) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) float Xs[kBK][kBM + 4];
  __shared__ __align__(16) float Ys[kBK][kBN + 4];
  __shared__ float red[kThreads / 32];
  const int i = blockIdx.z;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  float acc[4][4] = {};
  float cs = 0.f;
  const bool do_b = (blockIdx.y == 0);
  rows_tile<E, false>(g, A, G, nullptr, m0, n0, (long)i * g.T, (long)(i + 1) * g.T, acc,
                      do_b ? &cs : nullptr, Xs, Ys);
  float sq = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) sq = fmaf(acc[u][v], acc[u][v], sq);
  const float tot = block_sum(sq, red);
  if (threadIdx.x == 0)
    ws_w[((size_t)i * gridDim.x + blockIdx.x) * gridDim.y + blockIdx.y] = tot;
  if (do_b) {
    const float bsq = block_sum(threadIdx.x < kBM ? cs * cs : 0.f, red);
    if (threadIdx.x == 0) ws_b[(size_t)i * gridDim.x + blockIdx.x] = bsq;
  }
}

// Ghost norm ([MixGhost] eq. 2.7): for example i and the block pair (tb <= sb) of
// 32-row blocks, sum_{t in tb, s in sb} (U U^T)_{ts} (G G^T)_{ts}, doubled off the
// diagonal (both Grams are symmetric).  The sum of the G-Gram entries is the bias
// norm ||sum_t g_t||^2 and is returned beside it.
constexpr int kGT = 32;

template <class E, bool GRAD>
__device__ __forceinline__ void gram_tile(const Geom& g, const E* __restrict__ X, int i, int t0,
                                          int s0, float acc[2][2], float (*Ts)[kGT + 1],
                                          float (*Ss)[kGT + 1]) {
  const int tid = threadIdx.x;
  const int K = GRAD ? g.p : g.D;
  const int tx = tid & 15, ty = tid >> 4;
  // contiguous dimension of the source: linear rows are contiguous in k; conv
  // inputs and conv grads are contiguous in t.
  const bool k_fast = !g.conv;
  for (int k0 = 0; k0 < K; k0 += kGT) {
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int kk, tt;
      if (k_fast) { kk = tid & 31; tt = (tid >> 5) + 8 * q; }
      else { tt = tid & 31; kk = (tid >> 5) + 8 * q; }
      const int k = k0 + kk;
      float a = 0.f, b = 0.f;
      if (k < K) {
        const int t = t0 + tt, s = s0 + tt;
        if (t < g.T) a = GRAD ? ld_g(X, g, i, t, k) : ld_a(X, g, i, t, k);
        if (s < g.T) b = GRAD ? ld_g(X, g, i, s, k) : ld_a(X, g, i, s, k);
      }
      Ts[kk][tt] = a;
      Ss[kk][tt] = b;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kGT; ++kk) {
      const float a0 = Ts[kk][ty * 2], a1 = Ts[kk][ty * 2 + 1];
      const float b0 = Ss[kk][tx * 2], b1 = Ss[kk][tx * 2 + 1];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
  }
}

template <class E>
__global__ void __launch_bounds__(kThreads) simt_ghost_kernel(Geom g, const E* __restrict__ A,
                                                              const E* __restrict__ G,
                                                              float* __restrict__ ws_h,
                                                              float* __restrict__ ws_g) {
  pdl_trigger();
  pdl_wait();
  __shared__ float Ts[kGT][kGT + 1];
  __shared__ float Ss[kGT][kGT + 1];
  __shared__ float red[kThreads / 32];
  const int i = blockIdx.y, pair = blockIdx.x;
  const int nb = (g.T + kGT - 1) / kGT;
  int tb = 0, rem = pair;
  while (rem >= nb - tb) { rem -= nb - tb; ++tb; }
  const int sb = tb + rem;
  float ga[2][2] = {}, gg[2][2] = {};
  gram_tile<E, false>(g, A, i, tb * kGT, sb * kGT, ga, Ts, Ss);
  gram_tile<E, true>(g, G, i, tb * kGT, sb * kGT, gg, Ts, Ss);
  const float wgt = (tb == sb) ? 1.f : 2.f;
  float h = 0.f, s = 0.f;
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int v = 0; v < 2; ++v) { h = fmaf(ga[u][v], gg[u][v], h); s += gg[u][v]; }
  const float H = block_sum(h * wgt, red);
  const float S = block_sum(s * wgt, red);
  if (threadIdx.x == 0) {
    ws_h[(size_t)i * gridDim.x + pair] = H;
    ws_g[(size_t)i * gridDim.x + pair] = S;
  }
}

// out[i] = sum_j ws1[i*n1 + j] + bias * sum_j ws2[i*n2 + j]  (one warp per example)
__global__ void reduce_norm_kernel(const float* __restrict__ ws1, int n1, const float* __restrict__ ws2,
                                   int n2, int B, int bias, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= B) return;
  float a = 0.f, b = 0.f;
  for (int j = lane; j < n1; j += 32) a += ws1[(size_t)i * n1 + j];
  if (bias)
    for (int j = lane; j < n2; j += 32) b += ws2[(size_t)i * n2 + j];
  a = warp_sum(a);
  b = warp_sum(b);
  if (lane == 0) out[i] = a + (bias ? b : 0.f);
}

}  // namespace dpk

namespace dph {
using namespace dpk;

static inline int cdiv(long a, long b) { return (int)((a + b - 1) / b); }

size_t simt_sum_splits(const Geom& g) {
  const long tiles = (long)cdiv(g.p, kBM) * cdiv(g.D, kBN);
  const long R = (long)g.B * g.T;
  long splits = cdiv(2 * 152, tiles);
  splits = std::min<long>(splits, cdiv(R, 256));
  splits = std::max<long>(1, std::min<long>(splits, 64));
  return (size_t)splits;
}

cudaError_t launch_simt_clipped_sum(const Geom& g, int dtype, const void* A, const void* G,
                                    const float* factors, float* dW, float* db, int accumulate,
                                    float* ws, int splits, cudaStream_t s) {
  const long R = (long)g.B * g.T;
  const long rps = ((R + splits - 1) / splits + kBK - 1) / kBK * kBK;
  float* ws_db = db ? ws + (size_t)splits * g.p * g.D : nullptr;
  dim3 grid(cdiv(g.p, kBM), cdiv(g.D, kBN), splits);
  if (dtype == DP_FP32)
    launch_pdl(simt_clipped_sum_kernel<float>, grid, kThreads, 0, s, g, (const float*)A, (const float*)G,
                                                              factors, ws, ws_db, rps);
  else
    launch_pdl(simt_clipped_sum_kernel<__nv_bfloat16>, grid, kThreads, 0, s, g, (const __nv_bfloat16*)A, (const __nv_bfloat16*)G, factors, ws, ws_db, rps);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t n = (size_t)g.p * g.D;
  const NoiseArgs none = {};
  launch_pdl(reduce_splits_kernel, (unsigned)std::min<size_t>((n + 255) / 256, 152 * 8), 256, 0, s, ws, splits, n, dW,
             accumulate, none, (uint64_t)0);
  if (db) {
    launch_pdl(reduce_splits_kernel, (unsigned)((g.p + 255) / 256), 256, 0, s, ws_db, splits, (size_t)g.p, db,
               accumulate, none, (uint64_t)0);
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_splits(const float* ws, int splits, size_t n, float* out, int accumulate,
                                 cudaStream_t s, const NoiseArgs* nz, uint64_t noff) {
  const NoiseArgs none = {};
  const NoiseArgs& na = (nz && nz->on) ? *nz : none;
  if (splits >= 512 && n <= ((size_t)1 << 14)) {
    const unsigned blocks = (unsigned)std::min<size_t>(n, 152 * 8);
    launch_pdl(reduce_splits_block_kernel, blocks ? blocks : 1, 256, 0, s, ws, splits, n, out, accumulate, na, noff);
    return cudaGetLastError();
  }
  if (splits >= 16 && n <= ((size_t)1 << 16)) {
    const size_t blocks = std::min<size_t>((n * 32 + 255) / 256, 152 * 8);
    launch_pdl(reduce_splits_warp_kernel, (unsigned)(blocks ? blocks : 1), 256, 0, s, ws, splits, n, out, accumulate,
               na, noff);
    return cudaGetLastError();
  }
  const size_t blocks = std::min<size_t>((n + 255) / 256, 152 * 8);
  launch_pdl(reduce_splits_kernel, (unsigned)(blocks ? blocks : 1), 256, 0, s, ws, splits, n, out, accumulate, na,
             noff);
  return cudaGetLastError();
}

cudaError_t launch_reduce_splits2(SplitSeg a, SplitSeg b, int splits, int accumulate, cudaStream_t s,
                                  NoiseArgs* nz) {
  if (!b.out) b.n = 0;
  const bool noise = nz && nz->on;
  if (splits >= 16 && std::max(a.n, b.n) <= ((size_t)1 << 16)) {
    // many splits of short vectors: the warp- and block-per-element kernels (packed layouts),
    // with or without the noise, so that a noised call sums in the same order as a plain one
    cudaError_t e = launch_reduce_splits(a.ws, splits, a.n, a.out, accumulate, s, nz, noise ? nz->off_a : 0);
    if (noise) nz->applied_a = 1;
    if (e != cudaSuccess || !b.n) return e;
    if (b.stride == b.n) {
      e = launch_reduce_splits(b.ws, splits, b.n, b.out, accumulate, s, nz, noise ? nz->off_b : 0);
      if (noise) nz->applied_b = 1;
      return e;
    }
    a.n = 0;   // a strided bias segment: the kernel below takes it alone
  }
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const bool v4 = al(a.ws) && al(a.out) && al(b.ws) && al(b.out) && a.stride % 4 == 0 && a.n % 4 == 0 &&
                  b.stride % 4 == 0 && b.n % 4 == 0;
  const size_t items = v4 ? (a.n + b.n) / 4 : a.n + b.n;
  if (!items) return cudaSuccess;
  NoiseArgs off = {};
  const NoiseArgs& na = noise ? *nz : off;
  const unsigned blocks = (unsigned)std::min<size_t>((items + 255) / 256, 152 * 8);
  if (v4) launch_pdl(reduce_splits2_kernel<4>, blocks, 256, 0, s, a, b, splits, accumulate, na);
  else launch_pdl(reduce_splits2_kernel<1>, blocks, 256, 0, s, a, b, splits, accumulate, na);
  if (noise) nz->applied_a = nz->applied_b = 1;
  return cudaGetLastError();
}

size_t simt_ghost_ws_floats(const Geom& g) {
  const long nb = cdiv(g.T, kGT);
  return (size_t)2 * g.B * (nb * (nb + 1) / 2);
}

cudaError_t launch_simt_ghost(const Geom& g, int dtype, const void* A, const void* G, float* out,
                              float* ws, cudaStream_t s) {
  const int nb = cdiv(g.T, kGT);
  const int npairs = nb * (nb + 1) / 2;
  float* ws_h = ws;
  float* ws_g = ws + (size_t)g.B * npairs;
  dim3 grid(npairs, g.B);
  if (dtype == DP_FP32)
    launch_pdl(simt_ghost_kernel<float>, grid, kThreads, 0, s, g, (const float*)A, (const float*)G, ws_h, ws_g);
  else
    launch_pdl(simt_ghost_kernel<__nv_bfloat16>, grid, kThreads, 0, s, g, (const __nv_bfloat16*)A,
                                                               (const __nv_bfloat16*)G, ws_h, ws_g);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(reduce_norm_kernel, cdiv(g.B, 8), 256, 0, s, ws_h, npairs, ws_g, npairs, g.B, g.has_bias, out);
  return cudaGetLastError();
}

size_t simt_inst_ws_floats(const Geom& g) {
  const long tm = cdiv(g.p, kBM), tn = cdiv(g.D, kBN);
  return (size_t)g.B * (tm * tn + tm);
}

cudaError_t launch_simt_inst(const Geom& g, int dtype, const void* A, const void* G, float* out,
                             float* ws, cudaStream_t s) {
  const int tm = cdiv(g.p, kBM), tn = cdiv(g.D, kBN);
  float* ws_w = ws;
  float* ws_b = ws + (size_t)g.B * tm * tn;
  dim3 grid(tm, tn, g.B);
  if (dtype == DP_FP32)
    launch_pdl(simt_inst_kernel<float>, grid, kThreads, 0, s, g, (const float*)A, (const float*)G, ws_w, ws_b);
  else
    launch_pdl(simt_inst_kernel<__nv_bfloat16>, grid, kThreads, 0, s, g, (const __nv_bfloat16*)A,
                                                              (const __nv_bfloat16*)G, ws_w, ws_b);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(reduce_norm_kernel, cdiv(g.B, 8), 256, 0, s, ws_w, tm * tn, ws_b, tm, g.B, g.has_bias, out);
  return cudaGetLastError();
}

}  // namespace dph
