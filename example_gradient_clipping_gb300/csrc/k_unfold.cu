// Row layout of a convolution for the tensor-core kernels (bf16, exact copies).
//
// The per-example gradient of a conv layer is F^{-1}(G_i)^T U(a_i) ([MixGhost]
// section 3.1, eq. 3.1: U is the unfold of the input, F^{-1} flattens the output
// gradient over positions).  These two kernels write both factors in the row layout
// of a linear layer, so the linear tensor-core kernels serve conv layers unchanged:
//   U[i, t, m]  = x_i[c, ho*s - pad + kh*dil, wo*s - pad + kw*dil]  (0 outside the image)
//                 t = ho*Wout + wo,  m = c*k*k + kh*k + kw  (torch.nn.functional.unfold order)
//   Gt[i, t, j] = G_i[j, t]   (the NCHW output gradient, transposed per example)
#include <algorithm>

#include "common.cuh"

namespace dpk {

// One thread writes 8 consecutive m of one row (16-byte store); D % 8 == 0.
__global__ void unfold_rows_kernel(Geom g, const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ U,
                                   size_t n_chunks) {
  const int cpr = g.D >> 3;                           // chunks per row
  const int kk = g.k * g.k;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n_chunks;
       q += (size_t)gridDim.x * blockDim.x) {
    const size_t row = q / cpr;
    const int m0 = (int)(q - row * cpr) * 8;
    const int i = (int)(row / g.T), t = (int)(row - (size_t)i * g.T);
    const int ho = t / g.Wout, wo = t - ho * g.Wout;
    const __nv_bfloat16* xi = x + (size_t)i * g.Cin * g.H * g.W;
    __align__(16) __nv_bfloat16 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int m = m0 + j;
      const int c = m / kk, r = m - c * kk;
      const int kh = r / g.k, kw = r - kh * g.k;
      const int h = ho * g.stride - g.pad + kh * g.dil;
      const int w = wo * g.stride - g.pad + kw * g.dil;
      v[j] = (h >= 0 && h < g.H && w >= 0 && w < g.W) ? xi[((size_t)c * g.H + h) * g.W + w]
                                                      : __float2bfloat16_rn(0.f);
    }
    *reinterpret_cast<uint4*>(U + q * 8) = *reinterpret_cast<const uint4*>(v);
  }
}

// Per example [p, T] -> [T, p] through a 32 x 33 shared tile.
__global__ void transpose_rows_kernel(int B, int T, int p, const __nv_bfloat16* __restrict__ G,
                                      __nv_bfloat16* __restrict__ Gt) {
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

}  // namespace dpk

namespace dph {
using namespace dpk;

cudaError_t launch_conv_rows(const Geom& g, const void* x, const void* G, void* U, void* Gt, cudaStream_t s) {
  const size_t n_chunks = (size_t)g.B * g.T * (g.D / 8);
  const size_t blocks = std::min<size_t>((n_chunks + 255) / 256, (size_t)152 * 16);
  unfold_rows_kernel<<<(unsigned)(blocks ? blocks : 1), 256, 0, s>>>(
      g, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(U), n_chunks);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 grid((g.T + 31) / 32, (g.p + 31) / 32, std::min(g.B, 65535));
  transpose_rows_kernel<<<grid, dim3(32, 8), 0, s>>>(g.B, g.T, g.p, static_cast<const __nv_bfloat16*>(G),
                                                      static_cast<__nv_bfloat16*>(Gt));
  count_launch();
  return cudaGetLastError();
}

}  // namespace dph
