// Tensor-core (tcgen05 / TMEM / TMA) kernels of libdpclip: declarations.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace dph {
using dpk::Geom;
// Clipped sum as one reweighted GEMM over the batch rows (bf16 in, fp32 accumulate).
bool tc_sum_supported(const Geom& g);
size_t tc_sum_ws_bytes(const Geom& g);
cudaError_t launch_tc_sum(const Geom& g, const void* A, const void* G, const float* factors,
                          float* dW, float* db, int accumulate, float* ws, unsigned* status,
                          cudaStream_t s, dpk::NoiseArgs* nz = nullptr);
// The same GEMM over rows whose G part already holds bf16(c_i G) (no bias).
cudaError_t launch_tc_sum_prescaled(const Geom& g, const void* A, const void* Gs, float* dW, int accumulate,
                                    float* ws, unsigned* status, cudaStream_t s, dpk::NoiseArgs* nz = nullptr);
// Clipped sum with per-example TMEM accumulation and fp32 scaling (rows per example >= 64).
bool tc_sumx_supported(const Geom& g);
size_t tc_sumx_ws_bytes(const Geom& g);
cudaError_t launch_tc_sumx(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                           float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s,
                           dpk::NoiseArgs* nz = nullptr, bool early = false);
// Instantiated norm ||G_i^T A_i||^2 (+ bias) from the same per-example TMEM products
// (shapes as tc_sumx_supported).
size_t tc_inst_ws_bytes(const Geom& g);
// With `keep`, every example's gradient is also written to keep [B, p, D] and its bias to
// keep_b [B, p] (fp32) for the kept-gradient clipped sum.
cudaError_t launch_tc_inst(const Geom& g, const void* A, const void* G, float* out, float* ws,
                           unsigned* status, cudaStream_t s, float* keep = nullptr, float* keep_b = nullptr,
                           bool early = false);
// Clipped sum from kept per-example gradients: dW (+)= sum_i c_i g_i, db (+)= sum_i c_i b_i
// (2pD flop per example, one read of the kept gradients).  conv_kk > 0: g_i in the conv
// kernel's tile column order with that many filter taps (mapped back to [p, Cin, k, k]);
// `quad`: g_i stored column-quad major, [D / 4][p][4] (the shifted-tile kernel's stores).
// With nz on, the noise and the 1/B scale in the same pass (nz->applied_* set).
size_t kept_sum_ws_bytes(int B, int p, int D);
cudaError_t launch_kept_sum(int B, int p, int D, int conv_kk, const float* keep, const float* keep_b,
                            const float* factors, float* dW, float* db, int accumulate, cudaStream_t s,
                            bool quad = false, dpk::NoiseArgs* nz = nullptr, void* ws = nullptr);
// Diagnostic: one kernel whose bounded wait runs out (timeout status, TMEM released).
cudaError_t launch_selftest_wait(unsigned* status, unsigned long long* waited_ns, cudaStream_t s);
// Stride-1 "same" conv layers over 64 input channels: every filter tap a shifted view of one
// input tile (NHWC copy of a channels-first input and channels-last rows of G in the workspace).
bool tc_halo_supported(const Geom& g);
size_t tc_halo_ws_bytes(const Geom& g);
// ||g_i||^2 -> out [B]; with `keep`, g_i [B, p, D] in the conv tile column order and b_i [B, p].
cudaError_t launch_tc_halo_norm(const Geom& g, const void* A, const void* G, float* out, void* ws, unsigned* status,
                                cudaStream_t s, float* keep = nullptr, float* keep_b = nullptr);
// Conv layers whose unfolded width plus bias is at most 64 (first layers over a few input
// channels): the unfold formed on chip from the example's input, G read as it lies.
bool tc_unfold_supported(const Geom& g);
size_t tc_unfold_ws_bytes(const Geom& g, bool norm);
// ||g_i||^2 -> out [B]; with `keep`, g_i [B, p, D] (weight layout) and b_i [B, p] as well.
cudaError_t launch_tc_unfold_norm(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                  unsigned* status, cudaStream_t s, float* keep = nullptr, float* keep_b = nullptr);
// dW (+)= sum_i c_i g_i, db (+)= sum_i c_i b_i (example splits summed in a fixed order).
cudaError_t launch_tc_unfold_sum(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                                 float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s,
                                 dpk::NoiseArgs* nz = nullptr);
// Ghost norm from per-example Gram tiles (bf16 in, fp32 accumulate).
bool tc_ghost_supported(const Geom& g);
size_t tc_ghost_ws_bytes(const Geom& g);
cudaError_t launch_tc_ghost(const Geom& g, const void* A, const void* G, float* out, float* ws,
                            unsigned* status, cudaStream_t s, bool early = false);
// Conv layer -> row layout of a linear layer (bf16): unfolded input U [B, T, D] and the
// output gradient transposed per example, Gt [B, T, p].
// U has conv_rows_width(g) = D rounded up to 8 columns (the extra ones zero).
int conv_rows_width(const Geom& g);
// With `scale`, Gt holds bf16(scale[i] * G) (the clip factors applied once, for the
// row-scaled clipped sum) and db (if given) receives the bias sum (see launch_scaled_rows).
cudaError_t launch_conv_rows(const Geom& g, const void* x, const void* G, void* U, void* Gt, cudaStream_t s,
                             const float* scale = nullptr, float* db = nullptr, int accumulate = 0,
                             float* bias_part = nullptr, dpk::NoiseArgs* nz = nullptr);
// Per example [p, T] -> [T, p] (bf16): the output gradient's row layout, and NCHW -> NHWC.
cudaError_t launch_transpose_rows(int B, int T, int p, const void* src, void* dst, cudaStream_t s,
                                  const float* scale = nullptr, float* bias_part = nullptr);
// Two such transposes (same B) in one launch.
cudaError_t launch_transpose_rows2(int B, int T0, int p0, const void* src0, void* dst0, int T1, int p1, const void* src1,
                                   void* dst1, cudaStream_t s);
// Gt = bf16(c_i G_i^T) for the row-scaled clipped sum, and db (+)= sum_i c_i sum_t G[i, :, t]
// from fp32 partial sums taken on the way (bias_part: scaled_rows_bias_bytes).
cudaError_t launch_scaled_rows(int B, int T, int p, const void* G, void* Gt, const float* factors, float* db,
                               int accumulate, float* bias_part, cudaStream_t s, bool rows_in = false,
                               dpk::NoiseArgs* nz = nullptr);
size_t scaled_rows_bias_bytes(int B, int T, int p);
// Conv layers with the unfold done by TMA im2col loads (Cin % 64 == 0, T % 8 == 0, T >= 64):
// instantiated norm and clipped sum; the workspace holds an NHWC copy of the input.
bool tc_conv_supported(const Geom& g);
size_t tc_conv_ws_bytes(const Geom& g, bool norm);
// With `keep`, every example's gradient is also written to keep [B, p, D] in the kernel's
// tile column order ((channel block * k*k + tap) * 64 + channel) and its bias to keep_b [B, p].
cudaError_t launch_tc_conv_norm(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                unsigned* status, cudaStream_t s, float* keep = nullptr, float* keep_b = nullptr);
// reuse_xh: the workspace already holds the NHWC copy of the input (a norm call left it).
cudaError_t launch_tc_conv_sum(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                               float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s,
                               bool reuse_xh = false, dpk::NoiseArgs* nz = nullptr);
// im2col map (bf16, 128-byte swizzle, 64 channels per pixel) over an NHWC copy of a conv input.
bool encode_im2col_bf16(CUtensorMap* map, const void* Xh, const Geom& g, int pixels);
// dW[j, m] (+)= sum over splits of part[s, j, col(m)], col mapping the weight column
// m = c*kk + tap to the im2col tile column (c/64 * kk + tap) * 64 + c % 64; `quad`: part's
cudaError_t launch_conv_reduce(const float* part, int splits, int p, int ncols, int kk, float* dW, int accumulate,
                               cudaStream_t s);
// A conv sum's bias: db (+)= the splits of part_db [splits, p] in order, with nz's noise
// (nz->applied_b is then set).
cudaError_t conv_bias_reduce(const float* part_db, int splits, int p, float* db, int accumulate, cudaStream_t s,
                             dpk::NoiseArgs* nz = nullptr);
// Row-scaled clipped sum of a conv layer (Cin % 64 == 0) with im2col loads for the input.
bool tc_sum_conv_supported(const Geom& g);
size_t tc_sum_conv_ws_bytes(const Geom& g);
// reuse_xh: the workspace already holds the NHWC copy of the input (a norm call left it).
cudaError_t launch_tc_sum_conv(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                               float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s,
                               bool reuse_xh = false, dpk::NoiseArgs* nz = nullptr);
// Ghost norm of a conv layer (Cin % 64 == 0) with im2col loads for the input Gram.
bool tc_ghost_conv_supported(const Geom& g);
size_t tc_ghost_conv_ws_bytes(const Geom& g);
cudaError_t launch_tc_ghost_conv(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                 unsigned* status, cudaStream_t s);
// dW[j, m] (+)= Wp[j, m] for j < p, m < D (Wp rows of Dp floats).
cudaError_t launch_compact_cols(const float* Wp, int p, int D, int Dp, float* dW, int accumulate, cudaStream_t s);
// 2D/3D bf16 tensor map (dims innermost first, strides in bytes), 128-byte swizzle unless
// `swizzle` is false; elements outside the tensor read as zero.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, bool swizzle = true);
}  // namespace dph
