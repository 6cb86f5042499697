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
                          cudaStream_t s);
// Clipped sum with per-example TMEM accumulation and fp32 scaling (rows per example >= 64).
bool tc_sumx_supported(const Geom& g);
size_t tc_sumx_ws_bytes(const Geom& g);
cudaError_t launch_tc_sumx(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                           float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s);
// Instantiated norm ||G_i^T A_i||^2 (+ bias) from the same per-example TMEM products
// (shapes as tc_sumx_supported).
size_t tc_inst_ws_bytes(const Geom& g);
cudaError_t launch_tc_inst(const Geom& g, const void* A, const void* G, float* out, float* ws,
                           unsigned* status, cudaStream_t s);
// Ghost norm from per-example Gram tiles (bf16 in, fp32 accumulate).
bool tc_ghost_supported(const Geom& g);
size_t tc_ghost_ws_bytes(const Geom& g);
cudaError_t launch_tc_ghost(const Geom& g, const void* A, const void* G, float* out, float* ws,
                            unsigned* status, cudaStream_t s);
// Conv layer -> row layout of a linear layer (bf16): unfolded input U [B, T, D] and the
// output gradient transposed per example, Gt [B, T, p].
// U has conv_rows_width(g) = D rounded up to 8 columns (the extra ones zero).
int conv_rows_width(const Geom& g);
cudaError_t launch_conv_rows(const Geom& g, const void* x, const void* G, void* U, void* Gt, cudaStream_t s);
// Per example [p, T] -> [T, p] (bf16): the output gradient's row layout, and NCHW -> NHWC.
cudaError_t launch_transpose_rows(int B, int T, int p, const void* src, void* dst, cudaStream_t s);
// Conv layers with the unfold done by TMA im2col loads (Cin % 64 == 0, T % 8 == 0, T >= 64):
// instantiated norm and clipped sum; the workspace holds an NHWC copy of the input.
bool tc_conv_supported(const Geom& g);
size_t tc_conv_ws_bytes(const Geom& g, bool norm);
cudaError_t launch_tc_conv_norm(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                unsigned* status, cudaStream_t s);
cudaError_t launch_tc_conv_sum(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                               float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s);
// dW[j, m] (+)= Wp[j, m] for j < p, m < D (Wp rows of Dp floats).
cudaError_t launch_compact_cols(const float* Wp, int p, int D, int Dp, float* dW, int accumulate, cudaStream_t s);
// 2D/3D bf16 tensor map with 128-byte swizzle (dims innermost first, strides in bytes).
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);
}  // namespace dph
