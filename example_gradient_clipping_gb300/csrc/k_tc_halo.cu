// Stride-1 "same" convolutions over 64 input channels on the tensor cores: the filter's rows
// on the M side (shifted views of the output gradient), its columns on the N side (shifted
// views of the input), one tile of each per stage.
//
// Column block (kh, kw) of the per-example gradient P_i = F^{-1}(G_i)^T U(a_i) ([MixGhost]
// section 3.1, eq. 3.1) is
//     P_i[n, (kh, kw, c)] = sum_t G_i[t, n] a_i[t + shift(kh, kw), c]
// over the output pixels t laid out in padded rows (width Wp = W + 2 pad; the pad columns hold
// no output and G = 0 there; the input is laid out the same way, its pad columns and rows zero),
// shift(kh, kw) = (kh dil - pad) Wp + (kw dil - pad).  With shift = b(kw) - a(kh),
// b(kw) = kw dil - pad and a(kh) = -(kh dil - pad) Wp, and q = t - a(kh):
//     P_i[n, (kh, kw, c)] = sum_q G_i[q + a(kh), n] a_i[q + b(kw), c].
// So one MMA (M = 128, N = 64 k, K = 16 pixels q) forms the blocks of two filter rows and all k
// columns: A = the output gradient at q + a(kh) for two kh (the two 64-row halves of an MN-major
// operand, LBO = their distance), B = the input at q + b(kw) for every kw (k chunks of 64
// channels, MN-major, LBO = dil pixels).  Both operands are views into one TMA box each per
// stage (padded rows; the box's zero fill forms the padding), so a pixel arrives once per stage
// rather than once per tap.  Wide N is what keeps the tensor pipe busy: an M = 128, K = 16
// instruction took about 40 ns at any N up to 128 on this part and 50 ns at N = 192 (3x3),
// whatever M.  The filter rows pair up on M (3x3: rows 2 and 1, then row 0 with an unused
// half), so p <= 64; wider layers (whose P_i would not fit in TMEM at once) stay on the im2col
// kernels.
// norm mode: ||P_i||^2 + ||b_i||^2 per example, with b_i = sum_t G_i[t, :] summed by the
// epilogue warps from the channels-last output gradient in global memory while the example's
// MMAs run (shared-memory bandwidth is what the MMAs run short of); with `keep` also P_i and b_i,
// for the kept-gradient sum: P_i's tile columns col = (kh k + kw) * 64 + c stored column-quad
// major, [col / 4][n][col % 4], so that a warp's 32 rows n of one quad are 512 contiguous bytes.
// Roles (384 threads): warps 0, 2 and 3 TMA producers (stages round-robin), warp 1 MMA issuer,
// warps 4-11 bias sums and epilogue (two warps per TMEM lane quarter, each half the columns).
#include <algorithm>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tchalo {

constexpr int kThreads = 384;
constexpr int kEpiFirst = 4, kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kProducers = 3;                 // warps 0, 2, 3
constexpr int MAXST = 8;
constexpr int MAXG = 2;                       // MMAs per K step (filter-row groups of an example)
constexpr int CTL = 8192;
constexpr int SMEM_MAX = 232448 - 1024;       // dynamic shared memory (+ alignment slack)

struct Params {
  float* out;           // ||g_i||^2 [B]
  float* keep;          // or null: every example's gradient [B][k*k*16][p][4] (column quads)
  float* keep_b;        // and its bias [B, p]
  const __nv_bfloat16* Gr;   // output gradient, channels last [B, T, p] (the bias sums)
  unsigned* status;
  int B, p, k, kk, bias, T;
  int Wp, dil, pad;
  int ngu;              // MMAs per K step (filter-row pairs)
  int N, ncols, nbuf;   // MMA N (64 k), TMEM columns per example, TMEM buffers
  int nK;               // K pixels per example
  int spx, nk;          // K pixels per stage, stages per example
  int xrows, grows;     // rows per input / output-gradient box
  int xbytes, gbytes;   // bytes of the input box, of one 64-output G box
  int goff;             // offset of the G box in a stage (1024-aligned)
  int sbytes, nst;      // stage bytes, stages
  int ex_per_cta;
};

struct Ctl {
  uint64_t full[MAXST], empty[MAXST], accum[2], tfree[2][MAXG], drain;
  uint32_t tmem;
  int abort;
  float red[kEpiWarps];
  float redb[kEpiWarps][128];
};
static_assert(sizeof(Ctl) <= CTL, "control block");

__device__ __forceinline__ int floordiv(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
__device__ __forceinline__ int a_of(const Params& P, int kh) { return -(kh * P.dil - P.pad) * P.Wp; }

// An example's K pixels start at qs = -a(0); its output-gradient views read rows from a_lo =
// a(k-1) to a_hi = a(0) (+1 for the unused half of an odd row count), relative to the pixel.
__device__ __forceinline__ int k_first(const Params& P) { return -a_of(P, 0); }
__device__ __forceinline__ int a_lo(const Params& P) { return a_of(P, P.k - 1); }
// Group g: the filter rows of the A operand's halves (kh1 = -1: unused half) and the distance
// from the first half's view to the second (bytes).
__device__ __forceinline__ void group_rows(const Params& P, int g, int* kh0, int* kh1, int* lbo) {
  *kh0 = P.k - 1 - 2 * g;
  *kh1 = *kh0 - 1;
  *lbo = *kh1 >= 0 ? (a_of(P, *kh1) - a_of(P, *kh0)) * 128 : 128;
}
// First input row of stage u, first output-gradient row.
__device__ __forceinline__ int x_row(const Params& P, int u) { return floordiv(k_first(P) + u * P.spx - P.pad, P.Wp); }
__device__ __forceinline__ int g_row(const Params& P, int u) { return floordiv(k_first(P) + u * P.spx + a_lo(P), P.Wp); }

__device__ __forceinline__ void tma_load_4d(const CUtensorMap* map, uint64_t* bar, void* dst, int c, int x, int y,
                                            int n) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], [%2];"
      ::"r"(ptx::smem_u32(dst)), "l"(map), "r"(ptx::smem_u32(bar)), "r"(c), "r"(x), "r"(y), "r"(n)
      : "memory");
}

// Warps 0, 2 and 3 (pr = 0, 1, 2): stage k of the CTA's sequence (example k / nk, stage k % nk)
// when k % 3 == pr: the input box (xrows padded rows from column -pad) and the G box (grows
// output rows).  Boxes of this shape streamed at about 42 GB/s per SM from one issuing warp, 71
// from two and near 100 from three or more, hence the three.  The slot waits go by phase
// parity, sound while a slot's barrier is at most one phase behind: a producer's previous stage
// k - 3 was loaded after stage k - 3 - nst was consumed, which keeps it so for nst >= 3 (the
// planner's minimum).
__device__ __forceinline__ void producer(const Params& P, const CUtensorMap* mX, const CUtensorMap* mG,
                                         uint8_t* smem, Ctl* c, int e0, int e1, int pr) {
  volatile int* abort = &c->abort;
  const int total = (e1 - e0) * P.nk;
  int last = -1;
  for (int k = pr; k < total; k += kProducers) {
    const int s = k % P.nst;
    const bool w = k < P.nst || ptx::mbar_wait(&c->empty[s], ((k / P.nst) & 1) ^ 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) break;
    if (ptx::elect_one()) {
      const int e = e0 + k / P.nk, u = k % P.nk;
      uint8_t* st = smem + s * P.sbytes;
      ptx::mbar_arrive_expect_tx(&c->full[s], (uint32_t)(P.xbytes + P.gbytes));
      tma_load_4d(mX, &c->full[s], st, 0, -P.pad, x_row(P, u), e);
      tma_load_4d(mG, &c->full[s], st + P.goff, 0, -P.pad, g_row(P, u), e);
    }
    __syncwarp();
    last = k;
  }
  if (*abort && (threadIdx.x & 31) == 0)
    for (int q = max(pr, last - P.nst + 1); q <= last; ++q)
      if (q % kProducers == pr) ptx::mbar_wait_drain(&c->full[q % P.nst], (q / P.nst) & 1);
}

// Warp 1: per example, every stage's K steps: B = the input views (all kw), one MMA per
// filter-row pair, a stage's K steps group by group.  Each group's TMEM is released on its own
// (tfree[b][g]), so the next example's first MMAs into group 0 start while the epilogue still
// drains group 1 (with one 384-column buffer the whole drain would otherwise idle the tensor
// pipe).  The stage's tile offsets advance without divisions and the descriptors by one K step
// (2048 bytes) at a time: the issuing thread's work between MMAs is a few adds.
__device__ __forceinline__ void mma_issuer(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0, int e1) {
  volatile int* abort = &c->abort;
  const uint32_t idesc = ptx::idesc_bf16_f32(128, P.N, 1, 1);
  const uint64_t dhi = ptx::sdesc_sw128(0, 0, 1024);   // version, swizzle, SBO
  uint64_t lbo_bits[MAXG];                             // the A halves' distance, descriptor bits
  int adelta[MAXG];                                    // view of the first half - a_lo (pixels)
#pragma unroll
  for (int g = 0; g < MAXG; ++g) {
    int kh0, kh1, lbo;
    group_rows(P, g < P.ngu ? g : 0, &kh0, &kh1, &lbo);
    lbo_bits[g] = (uint64_t)(((uint32_t)lbo >> 4) & 0x3FFFu) << 16;
    adelta[g] = a_of(P, kh0) - a_lo(P);
  }
  const uint64_t bbits = dhi | ((uint64_t)(((uint32_t)(P.dil * 128) >> 4) & 0x3FFFu) << 16);
  const int sr = P.spx % P.Wp;   // a stage's offsets advance by spx pixels: whole rows and sr
  int s = 0, ph = 0;
  bool live = true;
  for (int x = 0; x < e1 - e0 && live; ++x) {
    const int b = x % P.nbuf;
    const uint32_t dbase = tmem + b * P.ncols;
    // pixel offsets of the stage's first K pixel in its input tile (view b(0)) and in its
    // output-gradient tile (view a_lo): the remainders of x_row and g_row
    int rx = k_first(P) - P.pad - x_row(P, 0) * P.Wp;
    int rg = k_first(P) + a_lo(P) - g_row(P, 0) * P.Wp;
    for (int u = 0; u < P.nk; ++u) {
      const bool w = ptx::mbar_wait(&c->full[s], ph, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      const uint32_t st = ptx::smem_u32(smem + s * P.sbytes);
      const int nkq = (min(P.spx, P.nK - u * P.spx) + 15) >> 4;
      const uint64_t db0 = bbits | (uint64_t)(((st + (uint32_t)rx * 128) >> 4) & 0x3FFFu);
#pragma unroll
      for (int g = 0; g < MAXG; ++g) {
        if (g >= P.ngu) break;
        if (u == 0) {   // the group's TMEM columns, free once the epilogue has read example x - nbuf's
          if (x >= P.nbuf) {
            const bool w2 = ptx::mbar_wait(&c->tfree[b][g], ((x / P.nbuf) & 1) ^ 1, abort, P.status);
            if (!__all_sync(0xffffffffu, w2)) { live = false; break; }
          }
          ptx::tc_fence_after();
        }
        if (ptx::elect_one()) {
          uint64_t da = dhi | lbo_bits[g] | (uint64_t)(((st + P.goff + (uint32_t)(rg + adelta[g]) * 128) >> 4) & 0x3FFFu);
          uint64_t db = db0;
          for (int kq = 0; kq < nkq; ++kq) {
            ptx::umma_bf16(dbase + g * P.N, da, db, idesc, (u | kq) != 0);
            da += 2048 >> 4;
            db += 2048 >> 4;
          }
        }
        __syncwarp();
      }
      if (!live) break;
      if (ptx::elect_one()) ptx::umma_commit(&c->empty[s]);
      __syncwarp();
      rx += sr;
      if (rx >= P.Wp) rx -= P.Wp;
      rg += sr;
      if (rg >= P.Wp) rg -= P.Wp;
      if (++s == P.nst) {
        s = 0;
        ph ^= 1;
      }
    }
    if (live) {
      if (ptx::elect_one()) ptx::umma_commit(&c->accum[b]);
      __syncwarp();
    }
  }
}

// Warps 4-11, per example: first the bias sums from the output gradient in global memory, then
// the example's TMEM group by group: lane m of group g is half m / 64 (filter row kh0 or kh1),
// output m % 64; its columns kw * 64 + c, the two warps of a lane quarter taking one half of
// them each, all their loads in flight before one wait, the group released before its squares
// and stores.
__device__ __forceinline__ void epilogue(const Params& P, Ctl* c, uint32_t tmem, int e0, int e1) {
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, colhalf = (warp - kEpiFirst) >> 2;
  const int et = threadIdx.x - 32 * kEpiFirst;   // 0 .. kEpiThreads - 1
  const int m = quarter * 32 + lane;             // TMEM lane
  const int nch = P.p >> 3;                      // 16-byte chunks (8 outputs) of a G row
  int ncp = 1;                                   // ... rounded up to a power of two
  while (ncp < nch) ncp <<= 1;
  const int chunk = et & (ncp - 1), phase = et / ncp, nphase = kEpiThreads / ncp;
  const int nl = P.k;                            // 32-column loads per warp and group (N / 2 / 32)
  bool ok = true;
  for (int x = 0; x < e1 - e0; ++x) {
    const int b = x % P.nbuf, e = e0 + x;
    const bool duty = P.bias;
    float bs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) bs[i] = 0.f;
    if (duty && chunk < nch) {   // rows t = phase, phase + nphase, ... of G_i, outputs 8 chunk ..
      const uint4* gp = reinterpret_cast<const uint4*>(P.Gr + (size_t)e * P.T * P.p) + chunk;
      for (int t = phase; t < P.T; t += nphase) {
        const uint4 v = __ldg(gp + (size_t)t * nch);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          bs[2 * i] += __uint_as_float(w4[i] << 16);
          bs[2 * i + 1] += __uint_as_float(w4[i] & 0xFFFF0000u);
        }
      }
    }
    float ss = 0.f;
    if (ok) {
      const bool w = ptx::mbar_wait(&c->accum[b], (x / P.nbuf) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) ok = false;
    }
    if (ok) {
      ptx::tc_fence_after();
      for (int g = 0; g < P.ngu; ++g) {
        int kh0, kh1, lbo;
        group_rows(P, g, &kh0, &kh1, &lbo);
        const int kh = m >> 6 ? kh1 : kh0;
        const int n = m & 63;
        const bool valid = kh >= 0 && n < P.p;
        const int cbase = colhalf * 32 * nl;     // first column of this warp's half
        const uint32_t base = tmem + b * P.ncols + g * P.N + cbase + ((uint32_t)(quarter * 32) << 16);
        float v[3][32];
#pragma unroll
        for (int i = 0; i < 3; ++i)
          if (i < nl) ptx::tmem_ld32(base + 32 * i, v[i]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();   // the group's columns are read: the next example's MMAs may start
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c->tfree[b][g]);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            if (i < nl) {
#pragma unroll
              for (int q = 0; q < 32; ++q) ss = fmaf(v[i][q], v[i][q], ss);
              if (P.keep) {   // 32 consecutive columns (tap * 64 + c) of row n: 8 quads
                const int c0 = cbase + 32 * i;
                const int quad0 = (kh * P.k + (c0 >> 6)) * 16 + ((c0 & 63) >> 2);
                float4* kp = reinterpret_cast<float4*>(P.keep) + ((size_t)e * P.kk * 16 + quad0) * P.p + n;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  kp[(size_t)q * P.p] = make_float4(v[i][4 * q], v[i][4 * q + 1], v[i][4 * q + 2], v[i][4 * q + 3]);
              }
            }
          }
        }
      }
    }
    if (duty) {   // b_i: the phases' sums (lanes chunk, chunk + ncp, ... of a warp, then the warps)
      for (int o = ncp; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) bs[i] += __shfl_xor_sync(0xffffffffu, bs[i], o);
      if (lane < ncp && lane < nch)
#pragma unroll
        for (int i = 0; i < 8; ++i) c->redb[warp - kEpiFirst][chunk * 8 + i] = bs[i];
      asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
      const int n = et;
      if (n < P.p) {
        float bn = 0.f;
#pragma unroll
        for (int w = 0; w < kEpiWarps; ++w) bn += c->redb[w][n];
        ss = fmaf(bn, bn, ss);
        if (P.keep_b && ok) P.keep_b[(size_t)e * P.p + n] = bn;
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) c->red[warp - kEpiFirst] = ss;
    asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");
    if (et == 0) {
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kEpiWarps; ++w) total += c->red[w];
      if (ok && !*abort) P.out[e] = total;
    }
    asm volatile("bar.sync 2, %0;" ::"r"(kEpiThreads) : "memory");   // red, redb reused
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_halo_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapG, Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* c = reinterpret_cast<Ctl*>(smem + P.nst * P.sbytes);
  const int warp = threadIdx.x >> 5;
  const int e0 = blockIdx.x * P.ex_per_cta;
  const int e1 = min(P.B, e0 + P.ex_per_cta);

  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nst; ++s) {
      ptx::mbar_init(&c->full[s], 1);
      ptx::mbar_init(&c->empty[s], 1);   // the MMAs' commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&c->accum[b], 1);
      for (int g = 0; g < MAXG; ++g) ptx::mbar_init(&c->tfree[b][g], kEpiWarps);
    }
    ptx::mbar_init(&c->drain, 1);
    c->abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mapX);
    ptx::prefetch_tensormap(&mapG);
  }
  if (warp == 1) ptx::tmem_alloc(&c->tmem, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c->tmem;
  pdl_trigger();   // the next kernel in the stream may start launching
  pdl_wait();      // the previous kernel has completed; its writes are visible

  if (warp >= kEpiFirst) epilogue(P, c, tmem, e0, e1);
  else if (warp == 1) mma_issuer(P, smem, c, tmem, e0, e1);
  else producer(P, &mapX, &mapG, smem, c, e0, e1, warp == 0 ? 0 : warp - 1);

  ptx::tc_fence_before();
  __syncthreads();
  if (*(volatile int*)&c->abort && threadIdx.x == 32) {
    ptx::umma_commit(&c->drain);   // arrives once every MMA issued so far has completed
    ptx::mbar_wait_drain(&c->drain, 0);
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace tchalo
}  // namespace dpk

namespace dph {
using namespace dpk;

static int cdiv_h(long a, long b) { return (int)((a + b - 1) / b); }
static int fdiv_h(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
static size_t al256_h(size_t n) { return (n + 255) & ~size_t(255); }

struct HaloPlan {
  int Wp, kk, ngu, N, ncols, nbuf, nK, spx, nk, xrows, grows, xbytes, gbytes, goff, sbytes, nst, ctas, eps;
};

// Rows a box must hold over every stage: the input box covers the stage's K pixels shifted by
// b(0) .. b(k-1), the output-gradient box shifted by a_lo .. a_hi (each K step reads 16 pixels
// from its own start, so the last pixel read is the stage's last + shift).
static void box_rows(const Geom& g, int Wp, int spx, int nk, int qs, int a_lo, int a_hi, int* xr, int* gr) {
  const int b_lo = -g.pad, b_hi = (g.k - 1) * g.dil - g.pad;
  for (int u = 0; u < nk; ++u) {
    const int q0 = qs + u * spx, q1 = q0 + spx - 1;
    *xr = std::max(*xr, fdiv_h(q1 + b_hi, Wp) - fdiv_h(q0 + b_lo, Wp) + 1);
    *gr = std::max(*gr, fdiv_h(q1 + a_hi, Wp) - fdiv_h(q0 + a_lo, Wp) + 1);
  }
}

static bool halo_plan(const Geom& g, HaloPlan* h) {
  if (!g.conv || g.Z != 1 || g.kz != 1 || g.kh != g.k || g.padh != g.pad || g.stride != 1) return false;
  if (g.Cin != 64 || g.Hout != g.H || g.Wout != g.W || g.p % 8 || g.p > 64 || g.T < 1) return false;
  // k = 1 or 3 (N = 64 k <= 256), "same" padding (the centre row's view is a = 0)
  if ((g.k != 1 && g.k != 3) || g.pad * 2 != g.dil * (g.k - 1)) return false;
  h->Wp = g.W + 2 * g.pad;
  if (h->Wp > 256) return false;
  h->kk = g.k * g.k;
  h->N = 64 * g.k;
  h->ngu = (g.k + 1) / 2;
  h->nK = (g.Hout + (g.k - 1) * g.dil) * h->Wp;
  h->ncols = h->ngu * h->N;
  h->nbuf = 2 * h->ncols <= 512 ? 2 : 1;
  const int a0 = g.pad * h->Wp, aZ = -((g.k - 1) * g.dil - g.pad) * h->Wp;   // a(0), a(k-1)
  // Stages of spx K pixels: the widest (fewest halo rows per pixel) that keeps at least four
  // stages in flight, else 64 pixels with three.
  for (int spx : {256, 192, 128, 64}) {
    const int nk = cdiv_h(h->nK, spx);
    int xr = 0, gr = 0;
    box_rows(g, h->Wp, spx, nk, -a0, aZ, a0 + (g.k & 1), &xr, &gr);
    if (xr > 256 || gr > 256) continue;
    const int xbytes = xr * h->Wp * 128, gbytes = gr * h->Wp * 128;
    const int goff = (xbytes + 1023) / 1024 * 1024;   // swizzled boxes start on 1024-byte boundaries
    const int sbytes = goff + (gbytes + 1023) / 1024 * 1024;
    const int nst = std::min<int>(tchalo::MAXST, (tchalo::SMEM_MAX - tchalo::CTL) / sbytes);
    if (nst < (spx == 64 ? 3 : 4)) continue;
    h->spx = spx;
    h->nk = nk;
    h->xrows = xr;
    h->grows = gr;
    h->xbytes = xbytes;
    h->gbytes = gbytes;
    h->goff = goff;
    h->sbytes = sbytes;
    h->nst = nst;
    h->eps = cdiv_h(g.B, std::min(g.B, 152));
    h->ctas = cdiv_h(g.B, h->eps);
    return true;
  }
  return false;
}

bool tc_halo_supported(const Geom& g) {
  HaloPlan h;
  return halo_plan(g, &h) && (double)g.B * g.H * g.W * g.Cin < 4e9;
}

// Workspace: the NHWC copy of a channels-first input (front, as the im2col kernels keep it)
// and the output gradient's channels-last rows (channels-first G).
static size_t halo_xbytes(const Geom& g) { return g.nhwc ? 0 : al256_h((size_t)g.B * g.H * g.W * g.Cin * 2); }
static size_t halo_gbytes(const Geom& g) { return g.nhwc ? 0 : al256_h((size_t)g.B * g.T * g.p * 2); }

size_t tc_halo_ws_bytes(const Geom& g) {
  HaloPlan h;
  if (!halo_plan(g, &h)) return 0;
  return std::max<size_t>(halo_xbytes(g) + halo_gbytes(g), 256);
}

cudaError_t launch_tc_halo_norm(const Geom& g, const void* A, const void* G, float* out, void* ws, unsigned* status,
                                cudaStream_t s, float* keep, float* keep_b) {
  HaloPlan h;
  if (!halo_plan(g, &h) || !ws) return cudaErrorInvalidValue;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const void* Xh = A;
  const void* Gr = G;
  cudaError_t e = cudaSuccess;
  if (!g.nhwc) {
    Xh = w;
    Gr = w + halo_xbytes(g);
    // NCHW -> NHWC, [p, T] -> [T, p]: one launch
    e = launch_transpose_rows2(g.B, g.H * g.W, g.Cin, A, w, g.T, g.p, G, w + halo_xbytes(g), s);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mX, mG;
  {   // input [B, H, W, 64]: boxes of 64 channels x Wp columns x xrows rows
    const uint64_t d[4] = {(uint64_t)g.Cin, (uint64_t)g.W, (uint64_t)g.H, (uint64_t)g.B};
    const uint64_t st[3] = {(uint64_t)g.Cin * 2, (uint64_t)g.W * g.Cin * 2, (uint64_t)g.H * g.W * g.Cin * 2};
    const uint32_t box[4] = {64, (uint32_t)h.Wp, (uint32_t)h.xrows, 1};
    if (!encode_tmap_bf16(&mX, Xh, 4, d, st, box)) return cudaErrorInvalidValue;
  }
  {   // output gradient [B, Hout, Wout, p]: boxes of 64 outputs (zero fill past p) x Wp columns x grows rows
    const uint64_t d[4] = {(uint64_t)g.p, (uint64_t)g.Wout, (uint64_t)g.Hout, (uint64_t)g.B};
    const uint64_t st[3] = {(uint64_t)g.p * 2, (uint64_t)g.Wout * g.p * 2, (uint64_t)g.T * g.p * 2};
    const uint32_t box[4] = {64, (uint32_t)h.Wp, (uint32_t)h.grows, 1};
    if (!encode_tmap_bf16(&mG, Gr, 4, d, st, box)) return cudaErrorInvalidValue;
  }
  tchalo::Params P = {};
  P.out = out;
  P.keep = keep;
  P.keep_b = g.has_bias ? keep_b : nullptr;
  P.Gr = static_cast<const __nv_bfloat16*>(Gr);
  P.status = status;
  P.B = g.B;
  P.p = g.p;
  P.k = g.k;
  P.kk = h.kk;
  P.bias = g.has_bias;
  P.T = g.T;
  P.Wp = h.Wp;
  P.dil = g.dil;
  P.pad = g.pad;
  P.ngu = h.ngu;
  P.N = h.N;
  P.ncols = h.ncols;
  P.nbuf = h.nbuf;
  P.nK = h.nK;
  P.spx = h.spx;
  P.nk = h.nk;
  P.xrows = h.xrows;
  P.grows = h.grows;
  P.xbytes = h.xbytes;
  P.gbytes = h.gbytes;
  P.goff = h.goff;
  P.sbytes = h.sbytes;
  P.nst = h.nst;
  P.ex_per_cta = h.eps;
  const int smem = 1024 + h.nst * h.sbytes + tchalo::CTL;
  int dev = 0;
  cudaGetDevice(&dev);
  static int attr_set[64] = {};
  if (dev >= 0 && dev < 64 && attr_set[dev] < smem) {
    e = cudaFuncSetAttribute(tchalo::tc_halo_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = smem;
  }
  return launch_pdl(tchalo::tc_halo_kernel, dim3(h.ctas), dim3(tchalo::kThreads), (size_t)smem, s, mX, mG, P);
}

}  // namespace dph
