// Convolution layers on the tensor cores with the unfold done by the TMA unit.
//
// The per-example gradient of a conv layer is P_i = F^{-1}(G_i)^T U(a_i) ([MixGhost]
// section 3.1, eq. 3.1).  Here U(a_i) is never written out: a TMA im2col load brings
// one [64 pixels x 64 channels] block of U for one filter tap straight from an NHWC
// copy of the input (zero outside the image), and the NCHW output gradient G_i
// [p, T] is the K-major A operand as it lies in memory.  Per CTA: one 128 x 256 tile
// of P (128 outputs x four im2col blocks = 256 unfolded columns), per example in one
// of two TMEM buffers.
//   norm mode: the epilogue adds up P_i^2 over the tile -> part[tile, i]; a fixed-order
//              sum over the tiles gives ||g_i||^2 (the instantiated norm of [MixGhost]
//              section 3).  With `keep` it also stores P_i (tile column order) and b_i
//              for the kept-gradient clipped sum.
//   sum mode:  the epilogue folds c_i P_i into fp32 registers (the clip factor of
//              [FastClip] section 5 applied in fp32) over the CTA's examples and
//              writes a partial tile; a fixed-order reduction over the example splits
//              maps the columns back to the weight layout [p, Cin, k, k].
//   bias:      the last column tile carries one more 64-column block of constant ones in
//              every stage buffer (written once; the TMA never touches it), so the MMA
//              also forms b_i = sum_t G_i[:, t] (every column of that block), accumulated
//              in fp32 like the rest: its square joins the norm partial, c_i b_i the db
//              partial of the CTA's split.
// Columns of the tile: block q = cc * k*k + tap (channel block cc of 64, filter tap
// kh*k + kw), 64 channels each; the weight column is (64 cc + c) * k*k + tap.
// Roles (384 threads): warps 0 and 2 TMA producers (alternate stages), warp 1 MMA
// issuer, warp 3 idle, warps 4-11 epilogue (two per TMEM lane quarter, 128 columns).
#include <algorithm>
#include <cudaTypedefs.h>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tcconv {

constexpr int BM = 128, BN = 256, STAGES = 4;
constexpr int BOX = 64 * 64 * 2;             // 8 KB: 64 rows x 128 B
constexpr int STAGE = 6 * BOX;               // G [128 outputs x 64 pixels], then 4 im2col blocks
constexpr int kThreads = 384;
constexpr int kEpiFirst = 4, kEpiWarps = 8;
constexpr int SMEM = STAGES * STAGE + 1024 + 512;
constexpr int PSTR = BN + 4;                 // staged output row stride (floats)
static_assert(BM * PSTR * 4 <= STAGES * STAGE, "staging fits in the stage buffers");
// A = G (K-major: pixels contiguous; channels-last output gradients: MN-major, outputs
// contiguous, two 64-output boxes), B = im2col blocks (MN-major: channels contiguous);
// the instruction's N is the tile's block count x 64

struct Params {
  const float* factors;   // sum mode
  float* part;            // norm: [tiles, B]; sum: [splits, p, ncols]
  float* part_db;         // sum mode with bias: [splits, p]
  int bias;               // the layer has a bias
  unsigned* status;
  int B, T, p, Wout, k, stride, pad, dil;
  int items;              // im2col blocks per pixel block: k*k*Cin/64
  int nk;                 // 64-pixel stages per example
  int ex_per_split;
  int ncols;              // items * 64
  float* keep;            // norm mode, or null: every example's gradient [B, p, ncols] in tile
                          // column order ((cc * k*k + tap) * 64 + c), and its bias [B, p]
  float* keep_b;
  int g_mn;               // G channels last ([B, T, p]): the A operand is MN-major
};

struct Ctl {
  uint64_t full[STAGES], empty[STAGES], accum[2], tfree[2], drain;
  uint32_t tmem;
  int abort;
  float red[2][8];
};

__device__ __forceinline__ void producer(const Params& P, const CUtensorMap* mG, const CUtensorMap* mX,
                                         uint8_t* smem, Ctl* c, int e0, int e1, int m0, int q0, int nitems,
                                         int pr) {
  volatile int* abort = &c->abort;
  const int kk = P.k * P.k;
  const uint32_t bytes = (uint32_t)(2 + nitems) * BOX;
  int k = 0, last = -1;
  bool live = true;
  for (int e = e0; e < e1 && live; ++e) {
    for (int u = 0; u < P.nk; ++u, ++k) {
      if ((k & 1) != pr) continue;
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait(&c->empty[s], ((k / STAGES) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      uint8_t* st = smem + s * STAGE;
      if (ptx::elect_one()) {
        ptx::mbar_arrive_expect_tx(&c->full[s], bytes);
        const int t0 = u * 64;
        if (P.g_mn) {             // [64 pixels x 64 outputs] twice: outputs m0.. and m0+64..
          ptx::tma_load_3d(mG, &c->full[s], st, m0, t0, e);
          ptx::tma_load_3d(mG, &c->full[s], st + BOX, m0 + 64, t0, e);
        } else {
          ptx::tma_load_3d(mG, &c->full[s], st, t0, m0, e);
        }
        const int ho = t0 / P.Wout, wo = t0 - ho * P.Wout;
        const int wb = wo * P.stride - P.pad, hb = ho * P.stride - P.pad;
        for (int j = 0; j < nitems; ++j) {
          const int q = q0 + j, cc = q / kk, tap = q - cc * kk;
          const int kh = tap / P.k, kw = tap - kh * P.k;
          ptx::tma_load_im2col_4d(mX, &c->full[s], st + (2 + j) * BOX, cc * 64, wb, hb, e,
                                  (uint16_t)(kw * P.dil), (uint16_t)(kh * P.dil));
        }
      }
      __syncwarp();
      last = k;
    }
  }
  if (*abort && (threadIdx.x & 31) == 0) {
    for (int q = max(0, last - STAGES + 1); q <= last; ++q)
      if ((q & 1) == pr) ptx::mbar_wait_drain(&c->full[q % STAGES], (q / STAGES) & 1);
  }
}

__device__ __forceinline__ void mma_issuer(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0,
                                           int e1, int nblocks) {
  volatile int* abort = &c->abort;
  const uint32_t idesc = ptx::idesc_bf16_f32(BM, 64 * nblocks, P.g_mn ? 1 : 0, 1);   // the tile's blocks only
  const int a_kstep = P.g_mn ? 2048 : 32;           // bytes per 16 pixels of the A operand
  int k = 0;
  bool live = true;
  for (int e = e0; e < e1 && live; ++e) {
    const int x = e - e0, b = x & 1;
    if (x >= 2) {
      const bool w = ptx::mbar_wait(&c->tfree[b], ((x >> 1) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) break;
    }
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem + b * 256;
    for (int u = 0; u < P.nk; ++u, ++k) {
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait(&c->full[s], (k / STAGES) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      const uint32_t g = ptx::smem_u32(smem + s * STAGE);
      // A: 128 rows of 128 B (64 pixels), K step of 16 pixels = 32 B; MN-major: two boxes of
      // 64 pixel rows x 128 B (64 outputs), BOX apart, K step of 16 pixels = 2048 B
      const uint64_t da = P.g_mn ? ptx::sdesc_sw128(g, BOX, 1024) : ptx::sdesc_sw128(g, 16, 1024);
      // B: 64-pixel rows of 128 B per block, blocks BOX apart, K step of 16 pixels = 2048 B
      const uint64_t dbd = ptx::sdesc_sw128(g + 2 * BOX, BOX, 1024);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::umma_bf16(d_tmem, ptx::sdesc_add(da, kk * a_kstep), ptx::sdesc_add(dbd, kk * 2048), idesc,
                         (u | kk) != 0);
        ptx::umma_commit(&c->empty[s]);
      }
      __syncwarp();
    }
    if (live) {
      if (ptx::elect_one()) ptx::umma_commit(&c->accum[b]);
      __syncwarp();
    }
  }
}

// Warps 4-11.  Every epilogue warp walks all of the CTA's examples (also after an
// abort) so the per-example barrier of the norm mode is always complete.
template <bool kNorm>
__device__ __forceinline__ void epilogue(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0, int e1,
                                         int m0, int q0, int nitems, int ones_slot) {
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = (warp - kEpiFirst) >> 2;
  // bias: the ones block (slot ones_slot of the tile, or -1) holds b_i in every column;
  // this thread's rows take it from the first column when the slot is in its half
  const bool my_ones = ones_slot >= 0 && (ones_slot >> 1) == half;
  const int ones_ch = (ones_slot & 1) * 4;              // 16-column chunk of that column
  // this thread's 128 columns are blocks 2*half and 2*half + 1 of the tile
  const bool v0 = 2 * half < nitems, v1 = 2 * half + 1 < nitems;
  const size_t tile = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
  float acc[kNorm ? 1 : 128];
  if constexpr (!kNorm) {
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] = 0.f;
  }
  bool ok = true;
  for (int e = e0; e < e1; ++e) {
    const int x = e - e0, b = x & 1;
    float ss = 0.f;
    if (ok) {
      const bool w = ptx::mbar_wait(&c->accum[b], (x >> 1) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) ok = false;
    }
    if (ok) {
      ptx::tc_fence_after();
      const float cf = kNorm ? 0.f : __ldg(P.factors + e);
      const uint32_t base = tmem + b * 256 + half * 128 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
      for (int ch = 0; ch < 8; ch += 2) {
        float a0[16], a1[16];
        ptx::tmem_ld16(base + ch * 16, a0);
        ptx::tmem_ld16(base + ch * 16 + 16, a1);
        ptx::tmem_wait_ld();
        if constexpr (kNorm) {
          const int m = m0 + quarter * 32 + lane;
          if (ch < 4 ? v0 : v1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              ss = fmaf(a0[j], a0[j], ss);
              ss = fmaf(a1[j], a1[j], ss);
            }
            if (P.keep && m < P.p) {   // 32 consecutive tile columns of row m: one 128-byte line
              float4* dst = reinterpret_cast<float4*>(P.keep + ((size_t)e * P.p + m) * P.ncols + (size_t)q0 * 64 +
                                                      half * 128 + ch * 16);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                dst[j] = make_float4(a0[4 * j], a0[4 * j + 1], a0[4 * j + 2], a0[4 * j + 3]);
                dst[4 + j] = make_float4(a1[4 * j], a1[4 * j + 1], a1[4 * j + 2], a1[4 * j + 3]);
              }
            }
          }
          if (my_ones && ch == ones_ch) {
            ss = fmaf(a0[0], a0[0], ss);   // ||b_i||^2, once per row
            if (P.keep_b && m < P.p) P.keep_b[(size_t)e * P.p + m] = a0[0];
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            acc[ch * 16 + j] = fmaf(cf, a0[j], acc[ch * 16 + j]);
            acc[ch * 16 + 16 + j] = fmaf(cf, a1[j], acc[ch * 16 + 16 + j]);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c->tfree[b]);
    }
    if constexpr (kNorm) {
      ss = warp_sum(ss);
      if (lane == 0) c->red[b][warp - kEpiFirst] = ss;
      asm volatile("bar.sync 2, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (threadIdx.x == 32 * kEpiFirst && !*abort) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kEpiWarps; ++w) t += c->red[b][w];
        P.part[tile * P.B + e] = t;
      }
    }
  }
  if constexpr (!kNorm) {
    // stage the partial tile in shared memory (the stage buffers are idle once the last
    // MMA completed), then write whole rows so the stores coalesce; every epilogue warp
    // passes the barrier
    const int row = quarter * 32 + lane;
    const int et = threadIdx.x - 32 * kEpiFirst;      // 0..255
    float* stg = reinterpret_cast<float*>(smem);
    if (ok) {
#pragma unroll
      for (int j = 0; j < 128; j += 4)
        *reinterpret_cast<float4*>(stg + row * PSTR + half * 128 + j) =
            make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    }
    asm volatile("bar.sync 2, %0;" ::"r"(32 * kEpiWarps) : "memory");
    if (*abort) return;
    if (ones_slot >= 0 && P.part_db && et < BM && m0 + et < P.p)      // sum_i c_i b_i of row et
      P.part_db[(size_t)blockIdx.z * P.p + m0 + et] = stg[et * PSTR + ones_slot * 64];
    const int nc4 = nitems * 16;                      // float4s per row of this tile
    for (int item = threadIdx.x - 32 * kEpiFirst; item < BM * nc4; item += 32 * kEpiWarps) {
      const int r = item / nc4, c4 = item - r * nc4;
      const int m = m0 + r;
      if (m >= P.p) continue;
      *reinterpret_cast<float4*>(P.part + ((size_t)blockIdx.z * P.p + m) * P.ncols + (size_t)q0 * 64 + c4 * 4) =
          *reinterpret_cast<const float4*>(stg + r * PSTR + c4 * 4);
    }
  }
}

__device__ __forceinline__ void finish(Ctl* c, uint32_t tmem) {
  ptx::tc_fence_before();
  __syncthreads();
  if (*(volatile int*)&c->abort && threadIdx.x == 32) {
    ptx::umma_commit(&c->drain);   // arrives once every MMA issued so far has completed
    ptx::mbar_wait_drain(&c->drain, 0);
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
tc_conv_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapX, Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* c = reinterpret_cast<Ctl*>(smem + STAGES * STAGE);
  const int warp = threadIdx.x >> 5;
  const int m0 = blockIdx.x * BM, q0 = blockIdx.y * 4;
  const int nitems = max(0, min(4, P.items - q0));
  // the ones block follows the last im2col block (a tile of its own when that tile is full)
  const int ones_slot = (P.bias && P.items >= q0 && P.items < q0 + 4) ? P.items - q0 : -1;
  const int nblocks = nitems + (ones_slot >= 0 ? 1 : 0);
  const int e0 = blockIdx.z * P.ex_per_split;
  const int e1 = min(P.B, e0 + P.ex_per_split);

  if (ones_slot >= 0) {   // constant ones in that block of every stage buffer (bf16 1.0 = 0x3F80)
    for (int q = threadIdx.x; q < STAGES * (BOX / 16); q += blockDim.x) {
      const int s = q / (BOX / 16), o = q % (BOX / 16);
      reinterpret_cast<uint4*>(smem + s * STAGE + (2 + ones_slot) * BOX)[o] =
          make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    }
    ptx::fence_proxy_async_smem();         // visible to the tensor core
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&c->full[s], 1);
      ptx::mbar_init(&c->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&c->accum[b], 1);
      ptx::mbar_init(&c->tfree[b], kEpiWarps);
    }
    ptx::mbar_init(&c->drain, 1);
    c->abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mapG);
    ptx::prefetch_tensormap(&mapX);
  }
  if (warp == 1) ptx::tmem_alloc(&c->tmem, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c->tmem;
  pdl_trigger();   // the next kernel in the stream may start launching
  pdl_wait();      // the previous kernel has completed; its writes are visible

  if (warp >= kEpiFirst) {
    ptx::regs_inc<216>();
    epilogue<kNorm>(P, smem, c, tmem, e0, e1, m0, q0, nitems, ones_slot);
    finish(c, tmem);
  } else {
    ptx::regs_dec<64>();
    if (warp == 0 || warp == 2)
      producer(P, &mapG, &mapX, smem, c, e0, e1, m0, q0, nitems, warp >> 1);
    else if (warp == 1)
      mma_issuer(P, smem, c, tmem, e0, e1, nblocks);
    finish(c, tmem);
  }
}

// dW[j, m] (+)= sum_s part[s, j, n(m)] in split order; n(m) maps the weight column
// m = c*k*k + tap to the tile column (64*(c/64)*k*k + 64*tap + c%64).  (The noise of a fused
// call is not drawn here: one output per thread would draw a whole Philox block per output,
// which measured slower than the separate four-outputs-per-block noise pass on the large
// layers; grouping four outputs per thread instead starved the small layers of threads.)
__global__ void conv_reduce_kernel(const float* __restrict__ part, int splits, int p, int ncols, int kk,
                                   float* __restrict__ dW, int accumulate) {
  pdl_trigger();
  pdl_wait();
  const size_t n = (size_t)p * ncols;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(q / ncols), m = (int)(q - (size_t)j * ncols);
    const int cch = m / kk, tap = m - cch * kk;
    const int col = ((cch >> 6) * kk + tap) * 64 + (cch & 63);
    float s = 0.f;
    for (int sp = 0; sp < splits; ++sp) s += part[((size_t)sp * p + j) * ncols + col];
    dW[q] = accumulate ? dW[q] + s : s;
  }
}

}  // namespace tcconv
}  // namespace dpk

namespace dph {
using namespace dpk;

static int cdiv_c(long a, long b) { return (int)((a + b - 1) / b); }
static size_t al256(size_t n) { return (n + 255) & ~size_t(255); }

static PFN_cuTensorMapEncodeIm2col_v12000 im2col_fn() {
  static PFN_cuTensorMapEncodeIm2col_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(p);
  }
  return fn;
}

bool tc_conv_supported(const Geom& g) {
  if (!g.conv || g.Cin % 64 || g.T % 8 || g.T < 64 || g.p < 8) return false;
  if (g.nhwc && g.p % 8) return false;     // channels-last G rows: 16-byte TMA strides
  if (g.kh != g.k || g.padh != g.pad || g.Z != 1 || g.kz != 1) return false;   // square 2D kernels (TMA im2col)
  if (g.stride > 8 || g.pad > 127 || g.dil * (g.k - 1) - g.pad > 128 || g.dil * (g.k - 1) > 65535) return false;
  return (double)g.B * g.H * g.W * g.Cin < 4e9;
}

struct ConvPlan {
  int tm, tn, tiles, items, splits, eps;
};

static ConvPlan conv_plan(const Geom& g, bool norm) {
  ConvPlan c;
  c.items = g.k * g.k * (g.Cin / 64);
  c.tm = cdiv_c(g.p, tcconv::BM);
  c.tn = cdiv_c(c.items + (g.has_bias ? 1 : 0), 4);   // + the ones block of the bias
  c.tiles = c.tm * c.tn;
  const long want = std::max<long>(1, std::min<long>(g.B, 152 / c.tiles));
  c.eps = cdiv_c(g.B, want);
  c.splits = cdiv_c(g.B, c.eps);
  (void)norm;
  return c;
}

// The NHWC copy of an NCHW input for the im2col loads (channels-last inputs need none),
// then the kernel's partials.
static size_t nhwc_bytes(const Geom& g) { return g.nhwc ? 0 : al256((size_t)g.B * g.H * g.W * g.Cin * 2); }

// The im2col source of a call: channels-last inputs are their own; else an NHWC copy in
// the workspace (or the one a norm call left there).  The output gradient is read as it
// lies either way ([p, T] K-major, or channels last [T, p] MN-major).
static cudaError_t conv_layouts(const Geom& g, const void* A, const void* G, void* ws, bool reuse_xh,
                                const void** Xh, const void** Gc, cudaStream_t s) {
  *Gc = G;
  if (g.nhwc) {
    *Xh = A;
    return cudaSuccess;
  }
  *Xh = ws;
  return reuse_xh ? cudaSuccess : launch_transpose_rows(g.B, g.H * g.W, g.Cin, A, ws, s);   // NCHW -> NHWC
}

size_t tc_conv_ws_bytes(const Geom& g, bool norm) {
  const ConvPlan c = conv_plan(g, norm);
  if (norm) return nhwc_bytes(g) + al256((size_t)c.tiles * g.B * 4);
  return nhwc_bytes(g) + al256((size_t)c.splits * g.p * c.items * 64 * 4) + al256((size_t)c.splits * g.p * 4);
}

// im2col map over the NHWC copy [B, H, W, Cin]: the bounding box's corners are the
// padding (lower -pad, upper pad - dil*(k-1)), so its positions are the output pixels'
// top-left input positions; the element strides are the conv stride; 64 channels
// (128 bytes, one swizzled row) per pixel and `pixels` pixels per load.
bool encode_im2col_bf16(CUtensorMap* map, const void* Xh, const Geom& g, int pixels) {
  auto fn = im2col_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)g.Cin, (cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.B};
  const cuuint64_t str[3] = {(cuuint64_t)g.Cin * 2, (cuuint64_t)g.W * g.Cin * 2, (cuuint64_t)g.H * g.W * g.Cin * 2};
  const int lo[2] = {-g.pad, -g.pad};
  const int hi[2] = {g.pad - g.dil * (g.k - 1), g.pad - g.dil * (g.k - 1)};
  const cuuint32_t es[4] = {1, (cuuint32_t)g.stride, (cuuint32_t)g.stride, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(Xh), dims, str, lo, hi, 64,
                        (cuuint32_t)pixels, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool encode_maps(const Geom& g, const void* Xh, const void* G, CUtensorMap* mG, CUtensorMap* mX) {
  if (g.nhwc) {     // [B, T, p]: boxes of 64 outputs x 64 pixels
    const uint64_t dg[3] = {(uint64_t)g.p, (uint64_t)g.T, (uint64_t)g.B};
    const uint64_t sg[2] = {(uint64_t)g.p * 2, (uint64_t)g.T * g.p * 2};
    const uint32_t box[3] = {64, 64, 1};
    if (!encode_tmap_bf16(mG, G, 3, dg, sg, box)) return false;
  } else {
    const uint64_t dg[3] = {(uint64_t)g.T, (uint64_t)g.p, (uint64_t)g.B};
    const uint64_t sg[2] = {(uint64_t)g.T * 2, (uint64_t)g.p * g.T * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!encode_tmap_bf16(mG, G, 3, dg, sg, box)) return false;
  }
  return encode_im2col_bf16(mX, Xh, g, 64);
}

cudaError_t launch_conv_reduce(const float* part, int splits, int p, int ncols, int kk, float* dW, int accumulate,
                               cudaStream_t s) {
  const size_t n = (size_t)p * ncols;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, (size_t)152 * 8);
  launch_plain(tcconv::conv_reduce_kernel, blocks ? blocks : 1, 256, 0, s, part, splits, p, ncols, kk, dW, accumulate);
  return cudaGetLastError();
}

cudaError_t conv_bias_reduce(const float* part_db, int splits, int p, float* db, int accumulate, cudaStream_t s,
                             NoiseArgs* nz) {
  const cudaError_t e = launch_reduce_splits(part_db, splits, (size_t)p, db, accumulate, s, nz, nz ? nz->off_b : 0);
  if (nz && nz->on) nz->applied_b = 1;
  return e;
}

template <bool kNorm>
static cudaError_t launch_kernel(const Geom& g, const ConvPlan& c, const CUtensorMap& mG, const CUtensorMap& mX,
                                 const tcconv::Params& P, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcconv::tc_conv_kernel<kNorm>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tcconv::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(c.tm, c.tn, c.splits);
  launch_plain(tcconv::tc_conv_kernel<kNorm>, grid, tcconv::kThreads, tcconv::SMEM, s, mG, mX, P);
  return cudaGetLastError();
}

static tcconv::Params base_params(const Geom& g, const ConvPlan& c, unsigned* status) {
  tcconv::Params P = {};
  P.g_mn = g.nhwc;
  P.status = status;
  P.B = g.B;
  P.T = g.T;
  P.p = g.p;
  P.Wout = g.Wout;
  P.k = g.k;
  P.stride = g.stride;
  P.pad = g.pad;
  P.dil = g.dil;
  P.items = c.items;
  P.nk = cdiv_c(g.T, 64);
  P.ex_per_split = c.eps;
  P.ncols = c.items * 64;
  return P;
}

cudaError_t launch_tc_conv_norm(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                unsigned* status, cudaStream_t s, float* keep, float* keep_b) {
  const ConvPlan c = conv_plan(g, true);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* part = reinterpret_cast<float*>(w + nhwc_bytes(g));
  const void *Xh, *Gc;
  cudaError_t e = conv_layouts(g, A, G, w, false, &Xh, &Gc, s);
  if (e != cudaSuccess) return e;
  CUtensorMap mG, mX;
  if (!encode_maps(g, Xh, Gc, &mG, &mX)) return cudaErrorInvalidValue;
  tcconv::Params P = base_params(g, c, status);
  P.part = part;
  P.bias = g.has_bias;
  P.keep = keep;
  P.keep_b = g.has_bias ? keep_b : nullptr;
  e = launch_kernel<true>(g, c, mG, mX, P, s);
  if (e != cudaSuccess) return e;
  return launch_reduce_splits(part, c.tiles, (size_t)g.B, out, 0, s);
}

cudaError_t launch_tc_conv_sum(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                               float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s, bool reuse_xh,
                               NoiseArgs* nz) {
  const ConvPlan c = conv_plan(g, false);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* part = reinterpret_cast<float*>(w + nhwc_bytes(g));
  float* part_db = reinterpret_cast<float*>(w + nhwc_bytes(g) + al256((size_t)c.splits * g.p * c.items * 64 * 4));
  const void *Xh, *Gc;
  cudaError_t e = conv_layouts(g, A, G, w, reuse_xh, &Xh, &Gc, s);
  if (e != cudaSuccess) return e;
  CUtensorMap mG, mX;
  if (!encode_maps(g, Xh, Gc, &mG, &mX)) return cudaErrorInvalidValue;
  tcconv::Params P = base_params(g, c, status);
  P.factors = factors;
  P.part = part;
  P.part_db = db ? part_db : nullptr;
  P.bias = g.has_bias;                       // the plan's tiles include the ones block
  e = launch_kernel<false>(g, c, mG, mX, P, s);
  if (e != cudaSuccess) return e;
  e = launch_conv_reduce(part, c.splits, g.p, c.items * 64, g.k * g.k, dW, accumulate, s);
  if (e != cudaSuccess || !db) return e;
  return conv_bias_reduce(part_db, c.splits, g.p, db, accumulate, s, nz);
}


}  // namespace dph
