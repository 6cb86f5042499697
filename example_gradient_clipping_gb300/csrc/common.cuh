// Shared device/host helpers of libdpclip (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dpclip.h"

namespace dpk {

// Device status bits (ORed into the status word; dp_check_status maps them).
constexpr unsigned kStatusNonfinite = 1u;
constexpr unsigned kStatusTimeout = 2u;

// Geometry of one layer's per-example contraction, resolved on the host.
// Linear: row t of example i is A[i, t, :] / G[i, t, :].
// Conv2d: row t = (ho, wo) of the unfolded input U(a_i) and of F^{-1}(G_i).
struct Geom {
  int B, T, D, p;             // examples, rows, (unfolded) input width, outputs
  int d;                      // linear input width (== D for linear)
  int Cin, H, W, k, stride, pad, dil, Hout, Wout;
  int kh, padh;               // kernel height and vertical padding: k and pad (conv2d, conv3d),
                              // 1 and 0 (conv1d: one input row, a 1 x k kernel)
  int Z, Zout, kz, padz;      // input depth, output depth, kernel depth, depth padding: conv3d,
                              // else 1, 1, 1, 0
  int conv;                   // 0 linear, 1 conv1d, conv2d or conv3d
  int nhwc;                   // conv: A and G channels last ([.., H, W, C]), else channels first
  int has_bias;
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Output-gradient element X(i, t, j), j < p.
template <class E>
__device__ __forceinline__ float ld_g(const E* __restrict__ G, const Geom& g, int i, int t, int j) {
  if (!g.conv || g.nhwc) return to_f(G[((size_t)i * g.T + t) * g.p + j]);
  return to_f(G[((size_t)i * g.p + j) * g.T + t]);
}

// (Unfolded) input element Y(i, t, m), m < D; zero outside the image (padding).
template <class E>
__device__ __forceinline__ float ld_a(const E* __restrict__ A, const Geom& g, int i, int t, int m) {
  if (!g.conv) return to_f(A[((size_t)i * g.T + t) * g.d + m]);
  // m = ((c*kz + kd)*kh + kh_)*k + kw, t = (zo*Hout + ho)*Wout + wo (PyTorch unfold order)
  const int kk = g.kz * g.kh * g.k;
  const int c = m / kk, r = m - c * kk;
  const int khk = g.kh * g.k;
  const int kd = r / khk, r2 = r - kd * khk;
  const int kh = r2 / g.k, kw = r2 - kh * g.k;
  const int hw = g.Hout * g.Wout;
  const int zo = t / hw, t2 = t - zo * hw;
  const int ho = t2 / g.Wout, wo = t2 - ho * g.Wout;
  const int z = zo * g.stride - g.padz + kd * g.dil;
  const int h = ho * g.stride - g.padh + kh * g.dil;
  const int w = wo * g.stride - g.pad + kw * g.dil;
  if (z < 0 || z >= g.Z || h < 0 || h >= g.H || w < 0 || w >= g.W) return 0.f;
  if (g.nhwc) return to_f(A[((((size_t)i * g.Z + z) * g.H + h) * g.W + w) * g.Cin + c]);
  return to_f(A[((((size_t)i * g.Cin + c) * g.Z + z) * g.H + h) * g.W + w]);
}

// Programmatic dependent launch: every library kernel is launched with programmatic
// stream serialization, lets the next kernel in the stream start launching once all of
// its CTAs are running (pdl_trigger), and waits for the previous kernel in the stream to
// complete, with its memory visible, before its first global-memory access (pdl_wait) --
// except the tensor-core kernels of linear layers, whose loads of the caller's A and G
// (which no library kernel writes) may precede the wait.  Kernels that do not use these
// (another library's) keep ordinary stream order.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Philox4x32-10 block function (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 products,
// XOR of the high halves into the other words and the round key, a word
// permutation, and a Weyl-sequence key schedule.  The round keys depend on the seed
// alone, so a kernel that draws many blocks under one seed builds them once
// (philox_key) and each block costs the products and XORs only.
struct PhiloxOut { uint32_t x[4]; };
struct PhiloxKey { uint32_t k0[10], k1[10]; };

__device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
  PhiloxKey k;
  k.k0[0] = (uint32_t)seed;
  k.k1[0] = (uint32_t)(seed >> 32);
#pragma unroll
  for (int r = 1; r < 10; ++r) {
    k.k0[r] = k.k0[r - 1] + kW0;
    k.k1[r] = k.k1[r - 1] + kW1;
  }
  return k;
}

__device__ __forceinline__ PhiloxOut philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                   const PhiloxKey& key) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one 32x32->64 product gives both halves
    const uint64_t p0 = (uint64_t)kM0 * c0, p1 = (uint64_t)kM1 * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ key.k0[r], n2 = (uint32_t)(p0 >> 32) ^ c3 ^ key.k1[r];
    c0 = n0; c1 = (uint32_t)p1; c2 = n2; c3 = (uint32_t)p0;
  }
  PhiloxOut o;
  o.x[0] = c0; o.x[1] = c1; o.x[2] = c2; o.x[3] = c3;
  return o;
}

// Uniform in (0, 1) from the top 23 bits of a word: (floor(x/2^9) + 1/2)/2^23, exact in fp32.
__device__ __forceinline__ float u01_from_word(uint32_t x) {
  return __uint2float_rn(x >> 9) * 0x1p-23f + 0x1p-24f;
}

// Four standard normals of Philox block q of stream `stream` under the key of a seed:
// Box-Muller on (u0, u1) and (u2, u3).  The radius sqrt(-2 ln u) is formed as x * rsqrt(x)
// (x > 0 since u < 1): within a few ulp, and two instructions instead of a rounded sqrt.
// The angle 2 pi u is taken as pi + theta, theta = 2 pi (u - 1/2) in [-pi, pi), whose sine
// and cosine come from the hardware approximations (absolute error about 2^-21.4 there):
// the accurate sincospi cost the noise pass a quarter of its throughput, and the error it
// leaves in z is at most the radius (< 5.8) times ~6e-7, under 4e-6.
__device__ __forceinline__ void normal4(uint64_t q, const PhiloxKey& key, uint32_t stream, float z[4]) {
  const PhiloxOut o = philox4x32_10((uint32_t)q, (uint32_t)(q >> 32), stream, 0u, key);
  const float u0 = u01_from_word(o.x[0]), u1 = u01_from_word(o.x[1]);
  const float u2 = u01_from_word(o.x[2]), u3 = u01_from_word(o.x[3]);
  const float x01 = -2.f * logf(u0), x23 = -2.f * logf(u2);
  const float r01 = x01 * rsqrtf(x01);
  const float r23 = x23 * rsqrtf(x23);
  float s1, c1, s3, c3;
  __sincosf(6.283185307f * (u1 - 0.5f), &s1, &c1);   // sin, cos of 2 pi u1 - pi
  __sincosf(6.283185307f * (u3 - 0.5f), &s3, &c3);
  z[0] = -r01 * c1; z[1] = -r01 * s1; z[2] = -r23 * c3; z[3] = -r23 * s3;
}

__device__ __forceinline__ void normal4(uint64_t q, uint64_t seed, uint32_t stream, float z[4]) {
  normal4(q, philox_key(seed), stream, z);
}

// One vector of split partials: split k at ws + k*stride (n floats), summed into out.
struct SplitSeg {
  const float* ws;
  size_t stride, n;
  float* out;
};

// The Gaussian mechanism and the 1/B average applied by a clipped sum's final pass, with
// the arithmetic of the separate noise pass: x <- (x + sc z_e) * invB, z_e lane e % 4 of
// normal4(e / 4) in stream 0, e the element's index in the flat parameter vector.
struct NoiseArgs {
  int on;
  float sc, invB;
  uint64_t seed;
  const unsigned long long* seed_dev;   // non-null: the seed is read here when the kernel runs
  uint64_t off_a, off_b;                // flat index of the first element of segment a / b
  int applied_a, applied_b;             // host: set by the launcher that fused it (dW, db)
};

// Up to 64 blocks of a flat gradient with their noise scales (sigma * C_b), in increasing
// offset order, not overlapping; qcum[b] = Philox blocks touched by blocks 0 .. b-1.
constexpr int kMaxNoiseBlocks = 64;
struct NoiseBlocks {
  int count;
  uint64_t off[kMaxNoiseBlocks], n[kMaxNoiseBlocks];
  float sc[kMaxNoiseBlocks];
  uint64_t qcum[kMaxNoiseBlocks + 1];
};

// z_e for the four consecutive flat indices e0 .. e0+3 (one or two Philox blocks).
__device__ __forceinline__ void noise_z4(uint64_t e0, uint64_t seed, float z[4]) {
  const int m = (int)(e0 & 3);
  float a[4];
  normal4(e0 >> 2, seed, 0u, a);
  if (m == 0) {
    z[0] = a[0]; z[1] = a[1]; z[2] = a[2]; z[3] = a[3];
    return;
  }
  float b[4];
  normal4((e0 >> 2) + 1, seed, 0u, b);
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int k = m + r;   // 1 .. 6: lane k of a, then of b
    z[r] = k == 1 ? a[1] : k == 2 ? a[2] : k == 3 ? a[3] : k == 4 ? b[0] : k == 5 ? b[1] : b[2];
  }
}

__device__ __forceinline__ float noise_z1(uint64_t e, uint64_t seed) {
  float a[4];
  normal4(e >> 2, seed, 0u, a);
  const int m = (int)(e & 3);
  return m == 0 ? a[0] : m == 1 ? a[1] : m == 2 ? a[2] : a[3];
}

}  // namespace dpk

// Host-side launchers implemented by the kernel translation units.
namespace dph {
using dpk::Geom;
// Counts kernels the library launched (reported by dp_launch_count).
void count_launch(unsigned n = 1);

// Launch with programmatic stream serialization (see pdl_wait); counts the launch.
// `pdl` false gives ordinary stream order (the kernel's pdl_wait is then a no-op): the
// conv layout and im2col kernels, where overlapping launches measured slower.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
  count_launch();
  return e;
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  return launch_k(true, kernel, grid, block, smem, s, static_cast<Args&&>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                         Args&&... args) {
  return launch_k(false, kernel, grid, block, smem, s, static_cast<Args&&>(args)...);
}
// Counts kernels the library launched (reported by dp_launch_count).
// Descriptor validation and the thread-local error message, shared by entry points.
dp_status geom_from_desc(const dp_layer_desc* d, Geom* g);
dp_status set_error(dp_status st, const char* msg);
cudaError_t launch_t1_norm(const Geom& g, int dtype, const void* A, const void* G, float* out,
                           cudaStream_t s);
// One-row (T = 1) linear clipped sum, FFMA, example splits reduced in a fixed order.
int t1_sum_splits(const Geom& g);
size_t t1_sum_ws_bytes(const Geom& g);
cudaError_t launch_t1_sum(const Geom& g, int dtype, const void* A, const void* G, const float* factors, float* dW,
                          float* db, int accumulate, float* ws, cudaStream_t s, dpk::NoiseArgs* nz = nullptr);
cudaError_t launch_clip_factors(const float* sq, int B, int L, int per_layer, const float* C,
                                float* out, unsigned* status, cudaStream_t s);
cudaError_t launch_add_noise(float* grad, size_t n, float sc, float invB, uint64_t seed,
                             uint64_t offset, const unsigned long long* seed_dev, cudaStream_t s);
cudaError_t launch_add_noise_blocks(float* grad, const dpk::NoiseBlocks& nb, float invB, uint64_t seed,
                                    const unsigned long long* seed_dev, cudaStream_t s);
// Adaptive bounds of layers layer0 .. layer0 + L - 1 (1 <= L <= 64) in one launch: norms
// sq [L, B], bounds C_l2 (host, L), out [L, 2]; with seed_dev the seed is read on the device.
cudaError_t launch_adaptive_bound(const float* sq, int B, int L, const float* C_l2, float alpha, float beta,
                                  float sigma_l2, uint64_t seed, const unsigned long long* seed_dev, int layer0,
                                  float* out, unsigned* status, cudaStream_t s);
// out[e] (+)= sum_k ws[k*n + e], fixed order; with nz->on also the noise of flat index
// noff + e and the 1/B scale.
cudaError_t launch_reduce_splits(const float* ws, int splits, size_t n, float* out, int accumulate,
                                 cudaStream_t s, const dpk::NoiseArgs* nz = nullptr, uint64_t noff = 0);
// The weight and bias reductions of one clipped sum in one launch (segments: dpk::SplitSeg).
// With nz->on the same pass adds the noise and the 1/B scale to both segments (nz->applied_a
// and applied_b are then set; with the short-vector kernels it is left for a noise pass).
using dpk::SplitSeg;
using dpk::NoiseArgs;
cudaError_t launch_reduce_splits2(SplitSeg a, SplitSeg b, int splits, int accumulate, cudaStream_t s,
                                  NoiseArgs* nz = nullptr);
// SIMT (FFMA) paths: any dtype/shape.
size_t simt_sum_splits(const Geom& g);
cudaError_t launch_simt_clipped_sum(const Geom& g, int dtype, const void* A, const void* G,
                                    const float* factors, float* dW, float* db, int accumulate,
                                    float* ws, int splits, cudaStream_t s);
size_t simt_ghost_ws_floats(const Geom& g);
cudaError_t launch_simt_ghost(const Geom& g, int dtype, const void* A, const void* G, float* out,
                              float* ws, cudaStream_t s);
size_t simt_inst_ws_floats(const Geom& g);
cudaError_t launch_simt_inst(const Geom& g, int dtype, const void* A, const void* G, float* out,
                             float* ws, cudaStream_t s);
}  // namespace dph
