// Row layout of a convolution for the tensor-core kernels (bf16, exact copies).
//
// The per-example gradient of a conv layer is F^{-1}(G_i)^T U(a_i) ([MixGhost]
// section 3.1, eq. 3.1: U is the unfold of the input, F^{-1} flattens the output
// gradient over positions).  These kernels write both factors in the row layout of
// a linear layer, so the linear tensor-core kernels serve conv layers unchanged:
//   U[i, t, m]  = x_i[c, zo*s - pad_z + kd*dil, ho*s - pad_h + kh*dil, wo*s - pad + kw*dil]
//                 (0 outside the input), t = (zo*Hout + ho)*Wout + wo,
//                 m = ((c*k_z + kd)*k_h + kh)*k + kw  (the order of a PyTorch weight;
//                 conv2d: k_z = 1, k_h = k; conv1d: one input row, k_z = k_h = 1; conv3d:
//                 a cubic kernel, the 2-D staging kernel does not take it),
//                 m < Dp: columns D <= m < Dp (Dp = D rounded up to 8) are zero
//   Gt[i, t, j] = G_i[j, t]   (the NCHW output gradient, transposed per example; a
//                 channels-last output gradient is already in this layout)
// Channels-last inputs (x_i stored [Z, H, W, Cin]) are read with their own strides.
#include <algorithm>

#include "tc.cuh"

namespace dpk {

// One CTA per example: the example's whole input ([Cin, H, W] or, channels last,
// [H, W, Cin]: contiguous either way) is staged in shared memory with 16-byte loads, then
// its T output rows are written with 16-byte stores, each gathered from shared memory
// (zero outside the image).
__global__ void unfold_rows_smem_kernel(Geom g, int Dp, const __nv_bfloat16* __restrict__ x,
                                        __nv_bfloat16* __restrict__ U) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) __nv_bfloat16 xs[];     // [Cin][H][W] or [H][W][Cin]
  const int kk = g.kh * g.k;
  const int cpr = Dp >> 3;                                // 16-byte chunks per output row
  const int HW = g.H * g.W;
  const int n_in = g.Cin * HW;
  const int cs = g.nhwc ? 1 : HW, ps = g.nhwc ? g.Cin : 1;   // channel and pixel strides
  for (int i = blockIdx.x; i < g.B; i += gridDim.x) {
    const __nv_bfloat16* xi = x + (size_t)i * n_in;
    if ((n_in & 7) == 0) {
      for (int q = threadIdx.x; q < (n_in >> 3); q += blockDim.x)
        reinterpret_cast<uint4*>(xs)[q] = reinterpret_cast<const uint4*>(xi)[q];
    } else {
      for (int q = threadIdx.x; q < n_in; q += blockDim.x) xs[q] = xi[q];
    }
    __syncthreads();
    __nv_bfloat16* out = U + (size_t)i * g.T * Dp;
    const int nch = g.T * cpr;
    for (int q = threadIdx.x; q < nch; q += blockDim.x) {
      const int t = q / cpr, m0 = (q - t * cpr) * 8;
      const int ho = t / g.Wout, wo = t - ho * g.Wout;
      const int hb = ho * g.stride - g.padh, wb = wo * g.stride - g.pad;
      // (c, kh, kw) of m0 once, then stepped along the chunk (no per-element division)
      int c = m0 / kk, r = m0 - c * kk;
      int kh = r / g.k, kw = r - kh * g.k;
      __align__(16) __nv_bfloat16 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int h = hb + kh * g.dil, w = wb + kw * g.dil;
        v[j] = (m0 + j < g.D && h >= 0 && h < g.H && w >= 0 && w < g.W) ? xs[c * cs + (h * g.W + w) * ps]
                                                                         : __float2bfloat16_rn(0.f);
        if (++kw == g.k) {
          kw = 0;
          if (++kh == g.kh) { kh = 0; ++c; }
        }
      }
      *reinterpret_cast<uint4*>(out + (size_t)q * 8) = *reinterpret_cast<const uint4*>(v);
    }
    __syncthreads();
  }
}

// Fallback when the staged rows do not fit in shared memory: one thread per 16-byte
// output chunk, gathered from global memory.
__global__ void unfold_rows_kernel(Geom g, int Dp, const __nv_bfloat16* __restrict__ x,
                                   __nv_bfloat16* __restrict__ U, size_t n_chunks) {
  pdl_trigger();
  pdl_wait();
  const int cpr = Dp >> 3;
  const int khk = g.kh * g.k, kk = g.kz * khk;
  const int hw = g.Hout * g.Wout;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n_chunks;
       q += (size_t)gridDim.x * blockDim.x) {
    const size_t row = q / cpr;
    const int m0 = (int)(q - row * cpr) * 8;
    const int i = (int)(row / g.T), t = (int)(row - (size_t)i * g.T);
    const int zo = t / hw, t2 = t - zo * hw;
    const int ho = t2 / g.Wout, wo = t2 - ho * g.Wout;
    const __nv_bfloat16* xi = x + (size_t)i * g.Cin * g.Z * g.H * g.W;
    __align__(16) __nv_bfloat16 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int m = m0 + j;
      const int c = m / kk, r = m - c * kk;
      const int kd = r / khk, r2 = r - kd * khk;
      const int kh = r2 / g.k, kw = r2 - kh * g.k;
      const int z = zo * g.stride - g.padz + kd * g.dil;
      const int h = ho * g.stride - g.padh + kh * g.dil;
      const int w = wo * g.stride - g.pad + kw * g.dil;
      const bool in = m < g.D && z >= 0 && z < g.Z && h >= 0 && h < g.H && w >= 0 && w < g.W;
      const size_t pix = ((size_t)z * g.H + h) * g.W + w;
      v[j] = in ? xi[g.nhwc ? pix * g.Cin + c : (size_t)c * g.Z * g.H * g.W + pix] : __float2bfloat16_rn(0.f);
    }
    *reinterpret_cast<uint4*>(U + q * 8) = *reinterpret_cast<const uint4*>(v);
  }
}

// Per example [p, T] -> [T, p] (T % 8 == 0, p % 8 == 0) through registers, no shared memory.
// A warp takes a tile of 8 * JC rows j by 8 * TQ pixels t (TQ = 4, 2 or 1 as T allows, JC =
// 32 / TQ); each lane loads one 8 x 8 block (eight 16-byte pieces of consecutive rows),
// transposes it with byte permutes and stores eight 16-byte pieces of consecutive pixel rows.
// One load instruction of the warp covers 16 * TQ contiguous bytes of each of JC rows, one
// store instruction 16 * JC contiguous bytes of each of TQ pixel rows.  With kScale, every
// value of example i is multiplied by scale[i] in fp32 and rounded to bf16 once, and with
// `bias_part` each tile writes the partial scale[i] * sum_t G[i, j, t] over its pixels to
// bias_part[(i * nt + tile) * p + j] (nt pixel tiles per example).
struct RowsJob {
  int T, p, tq, nt, njb;                 // pixel chunks per tile, pixel tiles, row tiles
  const __nv_bfloat16* src;
  __nv_bfloat16* dst;
  long units;                            // B * nt * njb warp tiles
};

__host__ __device__ __forceinline__ int rows_tile_tq(int T) { return T >= 32 ? 4 : T >= 16 ? 2 : 1; }

__device__ __forceinline__ uint32_t u4_word(const uint4& q, int k) {
  return k == 0 ? q.x : k == 1 ? q.y : k == 2 ? q.z : q.w;
}

template <bool kScale>
__global__ void __launch_bounds__(256, kScale ? 3 : 4) transpose_rows_reg_kernel(RowsJob j0, RowsJob j1,
                                                                    const float* __restrict__ scale,
                                                                    float* __restrict__ bias_part) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long nwarps = ((long)gridDim.x * blockDim.x) >> 5;
  for (long uu = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5; uu < j0.units + j1.units; uu += nwarps) {
    const bool second = uu >= j0.units;
    const RowsJob J = second ? j1 : j0;
    const long u = second ? uu - j0.units : uu;
    const long per = (long)J.nt * J.njb;
    const int i = (int)(u / per);
    const int rem = (int)(u - (long)i * per);
    const int tb = rem / J.njb, jb = rem - tb * J.njb;     // pixel tile, row tile
    const int tq = lane % J.tq, jc = lane / J.tq;
    const int t = (tb * J.tq + tq) * 8, j = (jb * (32 / J.tq) + jc) * 8;
    const bool ok = t < J.T && j < J.p;
    const size_t base = (size_t)i * J.T * J.p;
    uint4 a[8];
    if (ok) {
      const __nv_bfloat16* src = J.src + base + (size_t)j * J.T + t;
#pragma unroll
      for (int r = 0; r < 8; ++r) a[r] = __ldcs(reinterpret_cast<const uint4*>(src + (size_t)r * J.T));
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) a[r] = make_uint4(0u, 0u, 0u, 0u);
    }
    const float sc = kScale ? __ldg(scale + i) : 1.f;
    float bs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    __nv_bfloat16* dst = J.dst + base + (size_t)t * J.p + j;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      // pixel s of the block: channel pair (2v, 2v + 1) from rows 2v and 2v + 1, the value in
      // the low (s even) or high half of their word s / 2
      const uint32_t sel = (s & 1) ? 0x7632u : 0x5410u;
      uint32_t w[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) w[v] = __byte_perm(u4_word(a[2 * v], s >> 1), u4_word(a[2 * v + 1], s >> 1), sel);
      if (kScale) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float lo = __uint_as_float(w[v] << 16), hi = __uint_as_float(w[v] & 0xffff0000u);
          bs[2 * v] += lo;
          bs[2 * v + 1] += hi;
          const __nv_bfloat162 h = __floats2bfloat162_rn(sc * lo, sc * hi);
          w[v] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      if (ok) *reinterpret_cast<uint4*>(dst + (size_t)s * J.p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (kScale && bias_part) {
      // the TQ lanes of one row chunk hold consecutive pixel chunks: add across them
#pragma unroll
      for (int r = 0; r < 8; ++r)
        for (int o = 1; o < J.tq; o <<= 1) bs[r] += __shfl_xor_sync(0xffffffffu, bs[r], o);
      if (tq == 0 && j < J.p) {
        float* bp = bias_part + ((size_t)i * J.nt + tb) * J.p + j;
#pragma unroll
        for (int r = 0; r < 8; ++r) bp[r] = sc * bs[r];
      }
    }
  }
}

// Per example [p, T] -> [T, p] for T < 8 (p % 8 == 0): one thread per (example, 8 rows
// j0 .. j0+7), whose 8 x T values are contiguous (T 16-byte loads); each pixel's eight values
// are picked out in registers and stored as one 16-byte piece.  Scale and bias partial (one
// per example: bias_part[i * p + j]) as above.
template <int T>
__global__ void transpose_rows_few_kernel(int B, int p, const __nv_bfloat16* __restrict__ G,
                                          __nv_bfloat16* __restrict__ Gt, const float* __restrict__ scale,
                                          float* __restrict__ bias_part) {
  pdl_trigger();
  pdl_wait();
  const int cp = p >> 3;
  const size_t n = (size_t)B * cp;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const size_t i = q / cp;
    const int j0 = (int)(q - i * cp) * 8;
    const uint4* src = reinterpret_cast<const uint4*>(G + (i * p + j0) * T);
    uint4 a[T];
#pragma unroll
    for (int k = 0; k < T; ++k) a[k] = __ldcs(src + k);
    const float sc = scale ? __ldg(scale + i) : 1.f;
    float bs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = 0; t < T; ++t) {
      uint32_t w[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        // value (row r, pixel t) is element r * T + t of the block: 16-byte piece / 8, word / 2, half
        const int e0 = 2 * v * T + t, e1 = (2 * v + 1) * T + t;
        const uint32_t x = u4_word(a[e0 >> 3], (e0 & 7) >> 1), y = u4_word(a[e1 >> 3], (e1 & 7) >> 1);
        w[v] = __byte_perm(x, y, ((e0 & 1) ? 0x32u : 0x10u) | ((e1 & 1) ? 0x7600u : 0x5400u));
      }
      if (scale) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float lo = __uint_as_float(w[v] << 16), hi = __uint_as_float(w[v] & 0xffff0000u);
          bs[2 * v] += lo;
          bs[2 * v + 1] += hi;
          const __nv_bfloat162 h = __floats2bfloat162_rn(sc * lo, sc * hi);
          w[v] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      *reinterpret_cast<uint4*>(Gt + (i * T + t) * p + j0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (bias_part) {
#pragma unroll
      for (int r = 0; r < 8; ++r) bias_part[i * p + j0 + r] = sc * bs[r];
    }
  }
}

// Rows with T % 8 != 0, T > 8 (p % 8 == 0): one thread per (example, 8 outputs j0 .. j0+7),
// over all T pixels: gathers eight rows of G_i per pixel, one 16-byte store each.
__global__ void transpose_rows_short_kernel(int B, int T, int p, const __nv_bfloat16* __restrict__ G,
                                            __nv_bfloat16* __restrict__ Gt, const float* __restrict__ scale,
                                            float* __restrict__ bias_part) {
  pdl_trigger();
  pdl_wait();
  const int cp = p >> 3;
  const size_t n = (size_t)B * cp;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const size_t i = q / cp;
    const int j0 = (int)(q - i * cp) * 8;
    const __nv_bfloat16* src = G + (i * p + j0) * T;
    const float sc = scale ? __ldg(scale + i) : 1.f;
    float bsum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int t = 0; t < T; ++t) {
      __align__(16) __nv_bfloat16 v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const __nv_bfloat16 x = src[(size_t)r * T + t];
        bsum[r] += __bfloat162float(x);
        v[r] = scale ? __float2bfloat16_rn(sc * __bfloat162float(x)) : x;
      }
      *reinterpret_cast<uint4*>(Gt + (i * T + t) * p + j0) = *reinterpret_cast<const uint4*>(v);
    }
    if (bias_part) {
#pragma unroll
      for (int r = 0; r < 8; ++r) bias_part[i * p + j0 + r] = sc * bsum[r];
    }
  }
}

// Channels-last output gradients are rows [B, T, p] already: bf16(c_i G) in place of the
// scaled transpose, with the bias partial c_i sum_t G[i, t, j] of each example (p % 8 == 0).
// Thread = (example, 8 channels); consecutive threads read consecutive 16-byte chunks of a
// row, four rows in flight.
__global__ void scale_rows_kernel(int B, int T, int p, const __nv_bfloat16* __restrict__ G,
                                  __nv_bfloat16* __restrict__ Gs, const float* __restrict__ scale,
                                  float* __restrict__ bias_part) {
  pdl_trigger();
  pdl_wait();
  const int cp = p >> 3;
  const size_t n = (size_t)B * cp;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const size_t i = q / cp;
    const int j0 = (int)(q - i * cp) * 8;
    const float sc = __ldg(scale + i);
    float bsum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int t0 = 0; t0 < T; t0 += 4) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (t0 + u < T) raw[u] = __ldcs(reinterpret_cast<const uint4*>(G + (i * T + t0 + u) * p + j0));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (t0 + u >= T) break;
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw[u]);
        __align__(16) __nv_bfloat16 v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float f = __bfloat162float(x[r]);
          bsum[r] += f;
          v[r] = __float2bfloat16_rn(sc * f);
        }
        *reinterpret_cast<uint4*>(Gs + (i * T + t0 + u) * p + j0) = *reinterpret_cast<const uint4*>(v);
      }
    }
    if (bias_part) {
#pragma unroll
      for (int r = 0; r < 8; ++r) bias_part[i * p + j0 + r] = sc * bsum[r];
    }
  }
}

// General fallback: 32 x 33 tiles, 2-byte accesses.
__global__ void transpose_rows_kernel(int B, int T, int p, const __nv_bfloat16* __restrict__ G,
                                      __nv_bfloat16* __restrict__ Gt) {
  pdl_trigger();
  pdl_wait();
  __shared__ __nv_bfloat16 tile[32][33];
  const int t0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  for (int i = blockIdx.z; i < B; i += gridDim.z) {
    const size_t off = (size_t)i * T * p;
    for (int y = threadIdx.y; y < 32; y += blockDim.y) {
      const int j = j0 + y, t = t0 + threadIdx.x;
      if (j < p && t < T) tile[y][threadIdx.x] = G[off + (size_t)j * T + t];
    }
    __syncthreads();
    for (int y = threadIdx.y; y < 32; y += blockDim.y) {
      const int t = t0 + y, j = j0 + threadIdx.x;
      if (j < p && t < T) Gt[off + (size_t)t * p + j] = tile[threadIdx.x][y];
    }
    __syncthreads();
  }
}

// dW[j, m] (+)= Wp[j, m] for m < D (the padded columns are dropped).
__global__ void compact_cols_kernel(const float* __restrict__ Wp, int p, int D, int Dp, float* __restrict__ dW,
                                    int accumulate) {
  pdl_trigger();
  pdl_wait();
  const size_t n = (size_t)p * D;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const size_t j = q / D, m = q - j * D;
    const float v = Wp[j * Dp + m];
    dW[q] = accumulate ? dW[q] + v : v;
  }
}

constexpr int kUnfoldSmemMax = 160 * 1024;

}  // namespace dpk

namespace dph {
using namespace dpk;

int conv_rows_width(const Geom& g) { return (g.D + 7) / 8 * 8; }

cudaError_t launch_conv_rows(const Geom& g, const void* x, const void* G, void* U, void* Gt, cudaStream_t s,
                             const float* scale, float* db, int accumulate, float* bias_part, NoiseArgs* nz) {
  const int Dp = conv_rows_width(g);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* Ub = static_cast<__nv_bfloat16*>(U);
  const size_t stage = (size_t)g.Cin * g.H * g.W * sizeof(__nv_bfloat16);
  if (g.Z == 1 && g.kz == 1 && stage <= (size_t)kUnfoldSmemMax) {     // 1-D and 2-D inputs staged whole
    if (stage > 48 * 1024) {
      int dev = 0;
      cudaGetDevice(&dev);
      static bool attr_set[64] = {};
      if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(unfold_rows_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kUnfoldSmemMax);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
      }
    }
    const unsigned blocks = (unsigned)std::min<long>(g.B, 152L * 16);
    launch_plain(unfold_rows_smem_kernel, blocks, 256, stage, s, g, Dp, xb, Ub);
  } else {
    const size_t n_chunks = (size_t)g.B * g.T * (Dp / 8);
    const size_t blocks = std::min<size_t>((n_chunks + 255) / 256, (size_t)152 * 16);
    launch_plain(unfold_rows_kernel, (unsigned)(blocks ? blocks : 1), 256, 0, s, g, Dp, xb, Ub, n_chunks);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (scale) return launch_scaled_rows(g.B, g.T, g.p, G, Gt, scale, db, accumulate, bias_part, s, g.nhwc != 0, nz);
  if (g.nhwc) return cudaSuccess;        // channels last: G is already the rows the kernels read
  return launch_transpose_rows(g.B, g.T, g.p, G, Gt, s);
}

int transpose_bias_parts(int B, int T) {
  if (T % 8 == 0) return B * ((T + 8 * rows_tile_tq(T) - 1) / (8 * rows_tile_tq(T)));
  return B;
}

static RowsJob rows_job(int B, int T, int p, const void* src, void* dst) {
  RowsJob J;
  J.T = T;
  J.p = p;
  J.tq = rows_tile_tq(T);
  J.nt = (T + 8 * J.tq - 1) / (8 * J.tq);
  J.njb = (p + 8 * (32 / J.tq) - 1) / (8 * (32 / J.tq));
  J.src = static_cast<const __nv_bfloat16*>(src);
  J.dst = static_cast<__nv_bfloat16*>(dst);
  J.units = (long)B * J.nt * J.njb;
  return J;
}

static void launch_rows_reg(const RowsJob& a, const RowsJob& b, const float* scale, float* bias_part, cudaStream_t s) {
  const long warps = a.units + b.units;
  const unsigned blocks = (unsigned)std::max<long>(1, std::min<long>((warps + 7) / 8, 152L * 16));
  if (scale)
    launch_plain(transpose_rows_reg_kernel<true>, blocks, 256, 0, s, a, b, scale, bias_part);
  else
    launch_plain(transpose_rows_reg_kernel<false>, blocks, 256, 0, s, a, b, scale, bias_part);
}

template <int T>
static void launch_rows_few(int B, int p, const __nv_bfloat16* G, __nv_bfloat16* Gt, const float* scale,
                            float* bias_part, cudaStream_t s) {
  const size_t n = (size_t)B * (p / 8);
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)152 * 16);
  launch_plain(transpose_rows_few_kernel<T>, blocks ? blocks : 1, 256, 0, s, B, p, G, Gt, scale, bias_part);
}

cudaError_t launch_transpose_rows(int B, int T, int p, const void* src, void* dst, cudaStream_t s,
                                  const float* scale, float* bias_part) {
  const auto* Gb = static_cast<const __nv_bfloat16*>(src);
  auto* Gtb = static_cast<__nv_bfloat16*>(dst);
  if (T % 8 == 0 && p % 8 == 0) {
    RowsJob none = rows_job(B, T, p, src, dst);
    none.units = 0;
    launch_rows_reg(rows_job(B, T, p, src, dst), none, scale, bias_part, s);
  } else if (p % 8 == 0 && T < 8) {
    switch (T) {
      case 1: launch_rows_few<1>(B, p, Gb, Gtb, scale, bias_part, s); break;
      case 2: launch_rows_few<2>(B, p, Gb, Gtb, scale, bias_part, s); break;
      case 3: launch_rows_few<3>(B, p, Gb, Gtb, scale, bias_part, s); break;
      case 4: launch_rows_few<4>(B, p, Gb, Gtb, scale, bias_part, s); break;
      case 5: launch_rows_few<5>(B, p, Gb, Gtb, scale, bias_part, s); break;
      case 6: launch_rows_few<6>(B, p, Gb, Gtb, scale, bias_part, s); break;
      default: launch_rows_few<7>(B, p, Gb, Gtb, scale, bias_part, s); break;
    }
  } else if (p % 8 == 0) {
    const size_t n = (size_t)B * (p / 8);
    const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)152 * 16);
    launch_plain(transpose_rows_short_kernel, blocks ? blocks : 1, 256, 0, s, B, T, p, Gb, Gtb, scale, bias_part);
  } else {
    if (scale || bias_part) return cudaErrorInvalidValue;   // scaled copies need p % 8 == 0
    dim3 grid((T + 31) / 32, (p + 31) / 32, std::min(B, 65535));
    launch_plain(transpose_rows_kernel, grid, dim3(32, 8), 0, s, B, T, p, Gb, Gtb);
  }
  return cudaGetLastError();
}

cudaError_t launch_transpose_rows2(int B, int T0, int p0, const void* src0, void* dst0, int T1, int p1, const void* src1,
                                   void* dst1, cudaStream_t s) {
  if (T0 % 8 || p0 % 8 || T1 % 8 || p1 % 8) {
    const cudaError_t e = launch_transpose_rows(B, T0, p0, src0, dst0, s);
    return e != cudaSuccess ? e : launch_transpose_rows(B, T1, p1, src1, dst1, s);
  }
  launch_rows_reg(rows_job(B, T0, p0, src0, dst0), rows_job(B, T1, p1, src1, dst1), nullptr, nullptr, s);
  return cudaGetLastError();
}

cudaError_t launch_scaled_rows(int B, int T, int p, const void* G, void* Gt, const float* factors, float* db,
                               int accumulate, float* bias_part, cudaStream_t s, bool rows_in, NoiseArgs* nz) {
  if (rows_in) {   // channels last: scale in place of the transpose, one bias partial per example
    if (p % 8) return cudaErrorInvalidValue;
    const size_t n = (size_t)B * (p / 8);
    const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)152 * 16);
    launch_plain(scale_rows_kernel, blocks ? blocks : 1, 256, 0, s, B, T, p,
                 static_cast<const __nv_bfloat16*>(G), static_cast<__nv_bfloat16*>(Gt), factors,
                 db ? bias_part : nullptr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !db) return e;
    return conv_bias_reduce(bias_part, B, p, db, accumulate, s, nz);
  }
  cudaError_t e = launch_transpose_rows(B, T, p, G, Gt, s, factors, db ? bias_part : nullptr);
  if (e != cudaSuccess || !db) return e;
  return conv_bias_reduce(bias_part, transpose_bias_parts(B, T), p, db, accumulate, s, nz);
}

size_t scaled_rows_bias_bytes(int B, int T, int p) {
  return ((size_t)transpose_bias_parts(B, T) * p * 4 + 255) & ~size_t(255);
}

cudaError_t launch_compact_cols(const float* Wp, int p, int D, int Dp, float* dW, int accumulate, cudaStream_t s) {
  const size_t n = (size_t)p * D;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)152 * 8);
  launch_plain(compact_cols_kernel, blocks ? blocks : 1, 256, 0, s, Wp, p, D, Dp, dW, accumulate);
  return cudaGetLastError();
}

}  // namespace dph
