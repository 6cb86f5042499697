// Clipped sum as one reweighted GEMM on the 5th-generation tensor cores.
//
//   dW[j, m] = sum_r c_{r/T} G[r, j] A[r, m],   db[j] = sum_r c_{r/T} G[r, j],   r < R = B*T
//
// ([FastClip] section 5: the gradient of the reweighted loss sum_i c_i l_i is the
// clipped sum; [MixGhost] section 3.2: the second back-propagation's weight GEMM.)
// MMA view: D[M = p-tile, N = d-tile] += G^T[M, K] A[K, N] over K = batch rows; both
// operands are MN-major in memory (rows of G and A are contiguous along p and d).
//
// Per CTA: one 128 x 256 output tile over a contiguous range of rows (split-K).
//   warps 0, 6 TMA producers (alternate stages): per stage up to two 64x64 boxes of G and
//              four of A (128B swizzle); boxes wholly past p or D are not loaded
//   warp 1     MMA issuer: four 128xNx16 tcgen05.mma per stage into TMEM, N the tile's
//              columns inside D rounded up to 16 (narrow layers issue narrow MMAs)
//   warps 2-5  scale: multiply each row of the G tile in shared memory by its example's
//              clip factor (zero outside the CTA's rows) and accumulate the bias sums;
//              then the epilogue: TMEM -> registers -> fp32 partial tile.
// Partials [split, p, d] are reduced in a fixed order (deterministic) by a second kernel.
// Wide tiles (rows already scaled, p >= 256): 256 x 256 per CTA as two M = 128 accumulators
// in TMEM sharing each stage's A boxes, so a CTA reads 64 KB per 64 rows for twice the MMA
// work of a 48 KB narrow stage (the TMA delivery into an SM, not the tensor core, bounds
// the narrow tile).
#include <algorithm>
#include <cudaTypedefs.h>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tcsum {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_TILE = BN * BK * 2;            // 32 KB: four 64-column boxes
constexpr int BOX = 64 * BK * 2;               // 8 KB
constexpr int kThreads = 224;
constexpr int PSTR = BN + 4;                   // staged output row stride (floats)
template <bool kWide> struct Cfg {
  static constexpr int TM = kWide ? 2 * BM : BM;          // output rows per CTA
  static constexpr int STAGES = kWide ? 3 : 4;
  static constexpr int G_TILE = TM * BK * 2;              // 16 KB (two boxes) or 32 KB (four)
  static constexpr int STAGE = G_TILE + A_TILE;
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
  static_assert(BM * PSTR * 4 <= STAGES * STAGE, "staging fits in the stage buffers");
};

struct Params {
  const float* factors;
  float* ws;        // [splits, p, d]
  float* ws_db;     // [splits, p] or null
  unsigned* status;
  long R, rows_per_split;
  int T, p, d;
  // conv layers (Cin % 64 == 0): mapA is a TMA im2col map over an NHWC copy of the
  // input; unfolded column block q (64 wide) is channel block q / (k*k), tap q % (k*k)
  int conv, Wout, k, stride, pad, dil;
  // the G rows already hold bf16(c_i G) (written so by the transpose that made them):
  // no scaling pass, the MMA takes each stage as it lands; the bias is summed elsewhere
  int prescaled;
};

// Column block q of the unfolded rows starting at batch row `row` (64 rows).
__device__ __forceinline__ void load_a_block(const Params& P, const CUtensorMap* map, uint64_t* bar, void* dst,
                                             int q, int row) {
  if (!P.conv) {
    ptx::tma_load_2d(map, bar, dst, 64 * q, row);
    return;
  }
  const int taps = P.k * P.k, cc = q / taps, tap = q - cc * taps;
  const int kh = tap / P.k, kw = tap - kh * P.k;
  const int e = row / P.T, t = row - e * P.T;
  const int ho = t / P.Wout, wo = t - ho * P.Wout;
  ptx::tma_load_im2col_4d(map, bar, dst, cc * 64, wo * P.stride - P.pad, ho * P.stride - P.pad, e,
                          (uint16_t)(kw * P.dil), (uint16_t)(kh * P.dil));
}

template <bool kWide>
__global__ void __launch_bounds__(kThreads, 1)
tc_sum_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapA,
              Params P) {
  using C = Cfg<kWide>;
  constexpr int STAGES = C::STAGES, STAGE = C::STAGE, G_TILE = C::G_TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint64_t* scaled = full + STAGES;
  uint64_t* empty = scaled + STAGES;
  uint64_t* accum = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * C::TM, n0 = blockIdx.y * BN, split = blockIdx.z;
  const long r0 = (long)split * P.rows_per_split;
  const long r1 = min(P.R, r0 + P.rows_per_split);
  const int nk = (int)((r1 - r0 + BK - 1) / BK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&scaled[s], 4);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(accum, 1);
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mapG);
    ptx::prefetch_tensormap(&mapA);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kWide ? 512 : 256);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();   // the next kernel in the stream may start launching
  pdl_wait();      // the previous kernel has completed; its writes are visible

  // boxes inside the layer: G boxes along p, A boxes along D; MMA width N along D
  const int ng = min(C::TM / 64, (P.p - m0 + 63) / 64), na = min(4, (P.d - n0 + 63) / 64);
  const int nacc = (ng + 1) / 2;   // accumulators with rows inside p (1, or 2 for wide tiles)
  const int n_mma = min(BN, (P.d - n0 + 15) / 16 * 16);
  if (warp == 0 || warp == 6) {
    // TMA producers (whole warp; the elected lane issues); producer pr loads stages k % 2 == pr
    const int pr = warp == 6 ? 1 : 0;
    int last = -1;
    for (int k = pr; k < nk; k += 2) {
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait(&empty[s], ((k / STAGES) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) break;
      uint8_t* st = smem + s * STAGE;
      const int row = (int)(r0 + (long)k * BK);
      if (ptx::elect_one()) {
        ptx::mbar_arrive_expect_tx(&full[s], (uint32_t)(ng + na) * BOX);
        for (int j = 0; j < ng; ++j) ptx::tma_load_2d(&mapG, &full[s], st + j * BOX, m0 + 64 * j, row);
        for (int j = 0; j < na; ++j) load_a_block(P, &mapA, &full[s], st + G_TILE + j * BOX, n0 / 64 + j, row);
      }
      __syncwarp();
      last = k;
    }
    if (*abort && lane == 0) {   // let this producer's copies in flight land before the CTA exits
      for (int k = max(pr, last - STAGES + 1); k <= last; ++k)
        if ((k & 1) == pr) ptx::mbar_wait_drain(&full[k % STAGES], (k / STAGES) & 1);
    }
  } else if (warp == 1) {
    // MMA issuer (whole warp; the elected lane issues)
    for (int k = 0; k < nk; ++k) {
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait(P.prescaled ? &full[s] : &scaled[s], (k / STAGES) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) break;
      // the scale warps fenced their writes to the async proxy before arriving
      const uint32_t g = ptx::smem_u32(smem + s * STAGE);
      // 16 rows per MMA = two 8-row groups of 1024 B; MN chunks of 64 are 8 KB apart
      const uint64_t da = ptx::sdesc_sw128(g, BOX, 1024);
      const uint64_t db = ptx::sdesc_sw128(g + G_TILE, BOX, 1024);
      const uint32_t idesc = ptx::idesc_bf16_f32(BM, n_mma, 1, 1);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          ptx::umma_bf16(tmem, ptx::sdesc_add(da, kk * 2048), ptx::sdesc_add(db, kk * 2048), idesc, (k | kk) != 0);
          // the second accumulator: G boxes 2 and 3 (outputs m0+128 ..), the same A boxes
          if (kWide && nacc > 1)
            ptx::umma_bf16(tmem + 256, ptx::sdesc_add(da, 2 * BOX + kk * 2048),
                           ptx::sdesc_add(db, kk * 2048), idesc, (k | kk) != 0);
        }
        ptx::umma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (ptx::elect_one()) ptx::umma_commit(accum);
    __syncwarp();
  } else {
    // ---- scale warps (128 threads) ----
    const int t = threadIdx.x - 64;
    const int j = t & 7;            // row phase within each 8-row group
    const int cg = t >> 3;          // 16 column groups of 8 elements: box (0/1) and 16-byte chunk
    const int box = cg >> 3, q = cg & 7;
    float dbacc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) dbacc[e] = 0.f;
    bool ok = true;
    for (int k = 0; k < nk && ok && !P.prescaled; ++k) {
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait(&full[s], (k / STAGES) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      uint8_t* gt = smem + s * STAGE + box * BOX;
      const long rowbase = r0 + (long)k * BK;
#pragma unroll
      for (int rr = 0; rr < BK / 8; ++rr) {
        if (box >= ng) break;         // box not loaded (past p): nothing to scale
        const int r = rr * 8 + j;
        const long row = rowbase + r;
        const float c = (row < r1) ? __ldg(P.factors + (int)row / P.T) : 0.f;
        // 128-byte swizzle: the 16-byte chunk q of row r sits at chunk q ^ (r % 8)
        uint4* ptr = reinterpret_cast<uint4*>(gt + r * 128 + ((q ^ j) << 4));
        uint4 v = *ptr;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(h[e]);
          f.x *= c;
          f.y *= c;
          dbacc[2 * e] += f.x;
          dbacc[2 * e + 1] += f.y;
          h[e] = __floats2bfloat162_rn(f.x, f.y);
        }
        *ptr = v;
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&scaled[s]);
    }
    // bias partial sums: the 8 threads sharing a column group are lanes 8u..8u+7
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float v = dbacc[e];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      dbacc[e] = v;
    }
    if (ok && P.ws_db && !P.prescaled && blockIdx.y == 0 && j == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int col = m0 + box * 64 + q * 8 + e;
        if (col < P.p) P.ws_db[(size_t)split * P.p + col] = dbacc[e];
      }
    }
    // ---- epilogue: each thread drains one accumulator row (TMEM lane) into a shared
    // staging tile (the stage buffers are idle once the last MMA completed), then the
    // four warps write whole rows, so the stores coalesce.  All four warps pass the
    // barrier, also after an abort.
    const bool w = ok && ptx::mbar_wait(accum, 0, abort, P.status);
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    float* stg = reinterpret_cast<float*>(smem);
    const bool got = __all_sync(0xffffffffu, w);
    for (int h = 0; h < nacc; ++h) {
      if (h > 0) asm volatile("bar.sync 1, 128;" ::: "memory");   // the staging tile is free again
      if (got) {
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < (n_mma + 31) / 32; ++c) {
          float v[32];
          ptx::tmem_ld32(tmem + h * 256 + ((uint32_t)(quarter * 32) << 16) + c * 32, v);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(stg + row * PSTR + c * 32 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
      if (!*abort) {
        const int t = threadIdx.x - 64, nc4 = (n_mma + 3) / 4;
        const bool vec = (P.d & 3) == 0;
        for (int item = t; item < BM * nc4; item += 128) {
          const int r = item / nc4, c4 = item - r * nc4;
          const int m = m0 + h * BM + r, n = n0 + c4 * 4;
          if (m >= P.p) continue;
          const float4 o = *reinterpret_cast<const float4*>(stg + r * PSTR + c4 * 4);
          float* out = P.ws + ((size_t)split * P.p + m) * P.d + n;
          if (vec && n + 4 <= P.d) {
            *reinterpret_cast<float4*>(out) = o;
          } else {
            const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (n + q < P.d) out[q] = ov[q];
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 32) ptx::mbar_wait_drain(accum, 0);   // MMAs in flight
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kWide ? 512 : 256);
  }
}

}  // namespace tcsum
}  // namespace dpk

namespace dph {
using namespace dpk;

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int cdiv_i(long a, long b) { return (int)((a + b - 1) / b); }

// Split of the batch rows over CTAs: enough splits to cover the SMs with output
// tiles, each split a whole number of 64-row stages and every split non-empty.
static void tc_sum_split(const Geom& g, int* splits_out, long* rows_per_split, bool wide = false);

// Wide tiles for rows that arrive scaled (the conv row layout) when p fills them and each
// CTA still runs at least 24 stages (with fewer, the two accumulators' drains outweigh the
// saved loads: VGG-11's 2x2 layers ran 10% slower wide, its 8x8 and 4x4 layers 6-19% faster).
static bool tc_sum_wide(const Geom& g, bool prescaled) {
  if (!prescaled || g.p < 256) return false;
  int splits;
  long rps;
  tc_sum_split(g, &splits, &rps, true);
  return rps >= 24 * tcsum::BK;
}

static void tc_sum_split(const Geom& g, int* splits_out, long* rows_per_split, bool wide) {
  const long tiles = (long)cdiv_i(g.p, wide ? 2 * tcsum::BM : tcsum::BM) * cdiv_i(g.D, tcsum::BN);
  const long R = (long)g.B * g.T;
  long splits = std::max<long>(1, 152 / tiles);
  splits = std::min<long>(splits, std::max<long>(1, R / (4 * tcsum::BK)));
  long rps = (R + splits - 1) / splits;
  rps = (rps + tcsum::BK - 1) / tcsum::BK * tcsum::BK;
  *splits_out = (int)((R + rps - 1) / rps);
  *rows_per_split = rps;
}

// Splits of either tile width (the workspace covers both).
static int tc_sum_splits(const Geom& g) {
  int s, sw;
  long rps;
  tc_sum_split(g, &s, &rps, false);
  tc_sum_split(g, &sw, &rps, true);
  return std::max(s, sw);
}

bool tc_sum_supported(const Geom& g) {
  // linear layers whose rows are 16-byte multiples (TMA strides); boxes past the edges read zeros
  return !g.conv && (g.p % 8 == 0) && (g.D % 8 == 0) && g.p >= 8 && g.D >= 8 &&
         (long)g.B * g.T < (1L << 31);
}

size_t tc_sum_ws_bytes(const Geom& g) {
  return (size_t)tc_sum_splits(g) * ((size_t)g.p * g.D + g.p) * sizeof(float);
}

// The row-scaled GEMM over maps already built (ma: tiled rows or im2col), partials
// into ws, then the fixed-order reduction (conv: with the column map back to the
// weight layout).
static cudaError_t run_tc_sum(const Geom& g, const CUtensorMap& mg, const CUtensorMap& ma, const float* factors,
                              float* dW, float* db, int accumulate, float* ws, unsigned* status, cudaStream_t s,
                              bool prescaled = false, NoiseArgs* nz = nullptr);

cudaError_t launch_tc_sum(const Geom& g, const void* A, const void* G, const float* factors,
                          float* dW, float* db, int accumulate, float* ws, unsigned* status,
                          cudaStream_t s, NoiseArgs* nz) {
  const long R = (long)g.B * g.T;
  CUtensorMap mg, ma;
  const uint64_t dg[2] = {(uint64_t)g.p, (uint64_t)R}, sg[1] = {(uint64_t)g.p * 2};
  const uint64_t da[2] = {(uint64_t)g.D, (uint64_t)R}, sa[1] = {(uint64_t)g.D * 2};
  const uint32_t box[2] = {64, tcsum::BK};
  if (!encode_tmap_bf16(&mg, G, 2, dg, sg, box) || !encode_tmap_bf16(&ma, A, 2, da, sa, box))
    return cudaErrorInvalidValue;
  return run_tc_sum(g, mg, ma, factors, dW, db, accumulate, ws, status, s, false, nz);
}

cudaError_t launch_tc_sum_prescaled(const Geom& g, const void* A, const void* Gs, float* dW, int accumulate,
                                    float* ws, unsigned* status, cudaStream_t s, NoiseArgs* nz) {
  const long R = (long)g.B * g.T;
  CUtensorMap mg, ma;
  const uint64_t dg[2] = {(uint64_t)g.p, (uint64_t)R}, sg[1] = {(uint64_t)g.p * 2};
  const uint64_t da[2] = {(uint64_t)g.D, (uint64_t)R}, sa[1] = {(uint64_t)g.D * 2};
  const uint32_t box[2] = {64, tcsum::BK};
  if (!encode_tmap_bf16(&mg, Gs, 2, dg, sg, box) || !encode_tmap_bf16(&ma, A, 2, da, sa, box))
    return cudaErrorInvalidValue;
  return run_tc_sum(g, mg, ma, nullptr, dW, nullptr, accumulate, ws, status, s, true, nz);
}

// Conv layers with Cin % 64 == 0: the unfolded rows come from TMA im2col loads over an
// NHWC copy of the input, the output gradient from its row layout [B*T, p].  Workspace:
// the NHWC copy, the row layout of G, then the split partials.
bool tc_sum_conv_supported(const Geom& g) {
  if (g.kh != g.k || g.padh != g.pad || g.Z != 1 || g.kz != 1) return false;   // square 2D kernels (TMA im2col)
  return g.conv && g.Cin % 64 == 0 && g.p % 8 == 0 && g.stride <= 8 && g.pad <= 127 &&
         g.dil * (g.k - 1) - g.pad <= 128 && (double)g.B * g.H * g.W * g.Cin < 4e9 &&
         (long)g.B * g.T < (1L << 31);
}

static size_t al256s(size_t n) { return (n + 255) & ~size_t(255); }

size_t tc_sum_conv_ws_bytes(const Geom& g) {
  return al256s((size_t)g.B * g.H * g.W * g.Cin * 2) + al256s((size_t)g.B * g.T * g.p * 2) +
         al256s(tc_sum_ws_bytes(g)) + scaled_rows_bias_bytes(g.B, g.T, g.p);
}

cudaError_t launch_tc_sum_conv(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                               float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s, bool reuse_xh,
                               NoiseArgs* nz) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* Xh = w;
  void* Gt = w + al256s((size_t)g.B * g.H * g.W * g.Cin * 2);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(Gt) + al256s((size_t)g.B * g.T * g.p * 2));
  float* part_db = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(part) + al256s(tc_sum_ws_bytes(g)));
  // channels-last inputs are the im2col source themselves; else an NHWC copy (or the one a
  // norm call left in the workspace)
  cudaError_t e = (reuse_xh || g.nhwc) ? cudaSuccess : launch_transpose_rows(g.B, g.H * g.W, g.Cin, A, Xh, s);
  if (e != cudaSuccess) return e;
  if (g.nhwc) Xh = const_cast<void*>(A);
  // bf16(c_i G_i^T) and db in one pass, written right before the GEMM reads it (L2-hot);
  // rereading a norm call's unscaled rows and scaling them in the GEMM measured slower
  e = launch_scaled_rows(g.B, g.T, g.p, G, Gt, factors, db, accumulate, part_db, s, g.nhwc != 0, nz);
  if (e != cudaSuccess) return e;
  const long R = (long)g.B * g.T;
  CUtensorMap mg, ma;
  const uint64_t dg[2] = {(uint64_t)g.p, (uint64_t)R}, sg[1] = {(uint64_t)g.p * 2};
  const uint32_t box[2] = {64, tcsum::BK};
  if (!encode_tmap_bf16(&mg, Gt, 2, dg, sg, box) || !encode_im2col_bf16(&ma, Xh, g, tcsum::BK))
    return cudaErrorInvalidValue;
  return run_tc_sum(g, mg, ma, nullptr, dW, nullptr, accumulate, part, status, s, true, nz);
}

static cudaError_t run_tc_sum(const Geom& g, const CUtensorMap& mg, const CUtensorMap& ma, const float* factors,
                              float* dW, float* db, int accumulate, float* ws, unsigned* status, cudaStream_t s,
                              bool prescaled, NoiseArgs* nz) {
  const long R = (long)g.B * g.T;
  const bool wide = tc_sum_wide(g, prescaled);
  int splits;
  long rps;
  tc_sum_split(g, &splits, &rps, wide);
  tcsum::Params P;
  P.factors = factors;
  P.ws = ws;
  P.ws_db = (db && !prescaled) ? ws + (size_t)splits * g.p * g.D : nullptr;
  P.prescaled = prescaled ? 1 : 0;
  P.status = status;
  P.R = R;
  P.rows_per_split = rps;
  P.T = g.T;
  P.p = g.p;
  P.d = g.D;
  P.conv = g.conv;
  P.Wout = g.Wout;
  P.k = g.k;
  P.stride = g.stride;
  P.pad = g.pad;
  P.dil = g.dil;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64][2] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev][wide]) {
    cudaError_t e = wide ? cudaFuncSetAttribute(tcsum::tc_sum_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                tcsum::Cfg<true>::SMEM)
                         : cudaFuncSetAttribute(tcsum::tc_sum_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                tcsum::Cfg<false>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev][wide] = true;
  }
  dim3 grid(cdiv_i(g.p, wide ? 2 * tcsum::BM : tcsum::BM), cdiv_i(g.D, tcsum::BN), splits);
  if (wide) launch_pdl(tcsum::tc_sum_kernel<true>, grid, tcsum::kThreads, tcsum::Cfg<true>::SMEM, s, mg, ma, P);
  else launch_pdl(tcsum::tc_sum_kernel<false>, grid, tcsum::kThreads, tcsum::Cfg<false>::SMEM, s, mg, ma, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!g.conv) {
    const size_t nw = (size_t)g.p * g.D;
    return launch_reduce_splits2(SplitSeg{ws, nw, nw, dW},
                                 SplitSeg{P.ws_db, (size_t)g.p, P.ws_db ? (size_t)g.p : 0, db}, splits, accumulate, s,
                                 nz);
  }
  e = launch_conv_reduce(ws, splits, g.p, g.D, g.k * g.k, dW, accumulate, s);
  if (e != cudaSuccess) return e;
  if (P.ws_db) e = conv_bias_reduce(P.ws_db, splits, g.p, db, accumulate, s, nz);
  return e;
}

}  // namespace dph
