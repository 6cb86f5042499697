// Conv layers with few unfolded columns on the tensor cores, the unfold formed in shared
// memory by the CTA itself.
//
// The per-example gradient of a conv layer is P_i = F^{-1}(G_i)^T U(a_i) ([MixGhost]
// section 3.1, eq. 3.1): the output gradient G_i [p, T] against the unfolded input U(a_i)
// [T, D].  When D plus one column for the bias fits in 64 -- the first layer of an image
// network, whose input has a few channels (3x3 over RGB: D = 27) -- the layer's traffic is
// dominated by G_i, and U(a_i) is cheap to form on chip: each CTA keeps the example's input
// (a few KB) in shared memory and six warps write U(a_i)^T 64 pixels at a time, in the
// K-major 128-byte-swizzled layout the tensor core reads, next to the TMA-loaded block of
// G_i.  Neither unfolded rows nor a transposed output gradient reach global memory, so the
// layer costs one read of G and of the input.
//   norm mode: ||P_i||^2 (plus ||b_i||^2) per example -- the instantiated norm of
//              [MixGhost] section 3; with `keep` the kernel also stores P_i [p, D] (the weight
//              layout [p, Cin, kh, kw]) and b_i for the kept-gradient clipped sum.
//   sum mode:  sum_i c_i P_i folded in fp32 registers (the clip factor of [FastClip]
//              section 5 applied in fp32) over the CTA's examples; the example splits are
//              summed in a fixed order afterwards.
//   bias:      row D of U(a_i)^T is constant one on the T pixels, so column D of the product
//              is b_i = sum_t G_i[:, t] ([MixGhost] eq. 2.4's bias term), in fp32 like the rest.
// One CTA per (128-output tile, example split); per example one MMA chain of M = 128 (the
// outputs; rows past p read zeros), N = D + bias rounded up to 16, K = the example's pixels,
// into one of four TMEM buffers.
// Roles (384 threads): warp 0 loads the examples' inputs (TMA, one box per example, or 16-byte
// vectors scattered to channels-first rows), warp 1
// issues the MMAs, warps 2, 3, 8-11 (the builders) take the 64-pixel chunks in turn: each
// copies its chunk's G block into the ring with cp.async and forms U^T next to it while the
// copies land (a stream of 128-byte rows through the SM's one TMA queue was measured to move
// only ~16 GB/s per SM here; a single copying warp, with the copies' completion counted on the
// chunk barrier, reached less than copies spread over the six builders), warps 4-7 are the
// epilogue (one TMEM lane quarter each, one output row per thread).
#include <algorithm>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tcunf {

constexpr int BM = 128;                       // outputs per CTA (the MMA's M)
constexpr int NMAX = 64;                      // unfolded columns + bias, rounded up to 16
// Stage ring: per 64-pixel chunk the G block (128 outputs x 64 pixels, 16 KB; 8 KB when
// p <= 64: the MMA's rows 64-127 then read whatever follows, and land in TMEM lanes the
// epilogue never reads) and the U^T block (Np rows of 128 B), as many stages as fit.
constexpr int RING = 172032;                  // bytes of the stage ring
constexpr int MAXST = 16;
constexpr int XMAXE = 8192;                   // input elements per example held on chip
constexpr int XBUF = ((XMAXE + 32) * 2 + 1023) / 1024 * 1024;   // + slack for the 32-byte windows;
                                                              // 1024-aligned TMA destinations
constexpr int NBUF = 4;                       // TMEM buffers, 64 columns apart
constexpr int kThreads = 384;
constexpr int kBuilders = 6;                  // warps 2, 3, 8, 9, 10, 11
constexpr int kBT = 32 * kBuilders;
constexpr int kEpiFirst = 4, kEpiWarps = 4;
constexpr int CTL = 2048;
constexpr int SMEM = 1024 + RING + 2 * XBUF + CTL;
static_assert(SMEM <= 232448, "shared memory per CTA");

struct Params {
  const __nv_bfloat16* X;   // the layer input, one example contiguous: [Cin, H, W] or [H, W, Cin]
  const __nv_bfloat16* G;   // the output gradient (for the L2 prefetch)
  const float* factors;     // sum mode
  float* out;               // norm: ||g_i||^2 [B] (one output tile) or partials [tiles, B]
  float* part;              // sum: [splits, p, D] partials, or dW itself with one split
  float* part_b;            // sum with bias: [splits, p], or db itself with one split
  float* keep;              // norm mode, or null: every example's gradient [B, p, D]
  float* keep_b;            // and its bias [B, p]
  unsigned* status;
  int B, T, p, D, Np, bias;
  int Cin, H, W, Hout, Wout, k, kh, stride, pad, padh, dil;
  int nhwc;                 // input and output gradient channels last (the input is staged
                            // channels first on chip all the same)
  int XP;                   // channels first: padded row pitch of the input on chip (elements)
  int xelems;               // Cin * H * W
  int xvec;                 // the builders move the input in 16-byte vectors
  int xtma;                 // channels first, W % 8 == 0: one TMA box per example lands the
                            // input in its padded rows (the pads are the box's zero fill)
  int xrows;                // Cin * H
  int fast;                 // stride 1, Wout % 8 == 0, pad <= 8, channels first: 8-pixel windows
  int nk;                   // 64-pixel chunks per example
  int ex_per_split;
  int grows;                // G rows per output tile (min(p, 128))
  int accumulate;           // sum mode with one split: add to dW / db
  int nst, sbytes, ubase;   // stages in the ring, bytes per stage, offset of the U^T block
};

struct Ctl {
  uint64_t full[MAXST], empty[MAXST], accum[NBUF], tfree[NBUF], drain;
  uint64_t xfull[2], xempty[2];         // the input buffers (TMA-loaded inputs)
  uint32_t tmem;
  int abort;
  float red[2][kEpiWarps];
  int coff[NMAX], dh[NMAX], dw[NMAX];   // per unfolded column: input offset of its channel, tap shifts
};
static_assert(sizeof(Ctl) <= CTL, "control block");

// Warp 1: per example one accumulation chain into TMEM buffer x % NBUF.
__device__ __forceinline__ void mma_issuer(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0, int e1) {
  volatile int* abort = &c->abort;
  const uint32_t idesc = ptx::idesc_bf16_f32(BM, P.Np, P.nhwc ? 1 : 0, 0);
  // A: K-major 128 rows of 128 B (K step of 16 pixels = 32 B), or channels last MN-major:
  // two boxes of 64 pixel rows x 64 outputs, 8 KB apart (K step 2048 B).  B: U^T K-major.
  const int a_kstep = P.nhwc ? 2048 : 32;
  int k = 0;
  bool live = true;
  for (int e = e0; e < e1 && live; ++e) {
    const int x = e - e0, b = x % NBUF;
    if (x >= NBUF) {
      const bool w = ptx::mbar_wait(&c->tfree[b], ((x / NBUF) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) break;
    }
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem + b * 64;
    for (int u = 0; u < P.nk; ++u, ++k) {
      const int s = k % P.nst;
      const bool w = ptx::mbar_wait(&c->full[s], (k / P.nst) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      ptx::tc_fence_after();
      const uint32_t a = ptx::smem_u32(smem + s * P.sbytes);
      const uint64_t da = P.nhwc ? ptx::sdesc_sw128(a, 8192, 1024) : ptx::sdesc_sw128(a, 16, 1024);
      const uint64_t du = ptx::sdesc_sw128(a + P.ubase, 16, 1024);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::umma_bf16(d_tmem, ptx::sdesc_add(da, kk * a_kstep), ptx::sdesc_add(du, kk * 32), idesc,
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

// On-chip input position of element (channel offset coff = c*H*XP, row h, column w): channels
// first in padded rows (8 zeros either side), whatever the input's layout in memory.
__device__ __forceinline__ int xpos(const Params& P, int coff, int h, int w) { return coff + h * P.XP + 8 + w; }

// On-chip position of element q of one example's input as it lies in memory.
__device__ __forceinline__ int xdst(const Params& P, int q) {
  if (!P.nhwc) return (q / P.W) * P.XP + 8 + q % P.W;
  const int px = q / P.Cin, c = q - px * P.Cin;   // channels last: [H, W, Cin]
  return (c * P.H + px / P.W) * P.XP + 8 + px % P.W;
}

// The example's input into an on-chip buffer element by element (interior only: the pads
// stay zero), when it does not come in 16-byte vectors.
__device__ __forceinline__ void load_x_scalar(const Params& P, int e, int bt, __nv_bfloat16* xs) {
  const __nv_bfloat16* src = P.X + (size_t)e * P.xelems;
  for (int q = bt; q < P.xelems; q += kBT) xs[xdst(P, q)] = src[q];
}

// One 16-byte unit of U^T, element by element: column n, pixels t0 .. t0+7 of the example
// (any stride, dilation or width; the window path of build_chunk covers stride 1).
__device__ __forceinline__ uint4 build_unit(const Params& P, const Ctl* c, const __nv_bfloat16* xs, int n, int t0) {
  const int coff = c->coff[n];
  if (coff == -2 || t0 >= P.T) return make_uint4(0u, 0u, 0u, 0u);       // padding column / past T
  if (coff == -1) {                                                       // the bias column: ones on T
    if (t0 + 8 <= P.T) return make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __float2bfloat16_rn(t0 + j < P.T ? 1.f : 0.f);
    return *reinterpret_cast<const uint4*>(o);
  }
  __align__(16) __nv_bfloat16 o[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int t = t0 + j;
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (t < P.T) {
      const int ho = t / P.Wout, wo = t - ho * P.Wout;
      const int h = ho * P.stride + c->dh[n], w = wo * P.stride + c->dw[n];
      if (h >= 0 && h < P.H && w >= 0 && w < P.W) v = xs[xpos(P, coff, h, w)];
    }
    o[j] = v;
  }
  return *reinterpret_cast<const uint4*>(o);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Elements r .. r+7 of the 16 held in w0, w1 (r < 8): a word select and a funnel shift by
// half a word, without branches.
__device__ __forceinline__ uint4 extract8(const uint4& w0, const uint4& w1, int r) {
  const int q = r >> 1;
  const uint32_t sh = (uint32_t)(r & 1) * 16;
  const uint32_t c0 = w0.x, c1 = w0.y, c2 = w0.z, c3 = w0.w, c4 = w1.x, c5 = w1.y, c6 = w1.z, c7 = w1.w;
  const uint32_t s0 = q == 0 ? c0 : q == 1 ? c1 : q == 2 ? c2 : c3;
  const uint32_t s1 = q == 0 ? c1 : q == 1 ? c2 : q == 2 ? c3 : c4;
  const uint32_t s2 = q == 0 ? c2 : q == 1 ? c3 : q == 2 ? c4 : c5;
  const uint32_t s3 = q == 0 ? c3 : q == 1 ? c4 : q == 2 ? c5 : c6;
  const uint32_t s4 = q == 0 ? c4 : q == 1 ? c5 : q == 2 ? c6 : c7;
  return make_uint4(__funnelshift_r(s0, s1, sh), __funnelshift_r(s1, s2, sh), __funnelshift_r(s2, s3, sh),
                    __funnelshift_r(s3, s4, sh));
}

// 16-byte global -> shared copy in flight until cp.async.wait_all; `bytes` 0 writes zeros
// (and reads nothing).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// One warp's copies of chunk u's G block into the ring (128-byte swizzled rows, as the MMA's
// A operand reads them).  Channels first: rows = outputs m0.., 8 pixels per copy, pixels past
// T zero.  Channels last: rows = pixels, 8 outputs per copy, two 64-output boxes 8 KB apart,
// pixels past T and outputs past p zero.  Rows of outputs past p are not written: the MMA's
// products there land in TMEM lanes the epilogue does not read.
__device__ __forceinline__ void copy_g(const Params& P, uint32_t a, int e, int u, int m0, int lane) {
  const int t0 = u * 64;
  if (!P.nhwc) {
    const __nv_bfloat16* g = P.G + ((size_t)e * P.p + m0) * P.T;
    const int rows = min(P.grows, P.p - m0);
    for (int q = lane; q < rows * 8; q += 32) {
      const int r = q >> 3, j = q & 7, t = t0 + j * 8;
      const bool in = t < P.T;
      cp_async16(a + r * 128 + ((j ^ (r & 7)) << 4), g + (size_t)r * P.T + (in ? t : 0), in ? 16u : 0u);
    }
  } else {
    const int nbox = m0 + 64 < P.p ? 2 : 1;
    const __nv_bfloat16* g = P.G + (size_t)e * P.T * P.p;
    for (int q = lane; q < nbox * 512; q += 32) {
      const int jb = q >> 9, r = (q >> 3) & 63, j = q & 7;
      const int t = t0 + r, ch = m0 + jb * 64 + j * 8;
      const bool in = t < P.T && ch < P.p;
      cp_async16(a + jb * 8192 + r * 128 + ((j ^ (r & 7)) << 4), g + (in ? (size_t)t * P.p + ch : 0),
                 in ? 16u : 0u);
    }
  }
}

// Warp 0 (TMA inputs): example x's input into buffer x & 1 as soon as the builders have
// released example x - 2.
__device__ __forceinline__ void producer(const Params& P, const CUtensorMap* mX, uint8_t* xbuf, Ctl* c, int e0,
                                         int e1) {
  volatile int* abort = &c->abort;
  int x = 0;
  for (; x < e1 - e0; ++x) {
    const int b = x & 1;
    const bool w = x < 2 || ptx::mbar_wait(&c->xempty[b], ((x >> 1) & 1) ^ 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) break;
    if (ptx::elect_one()) {
      ptx::mbar_arrive_expect_tx(&c->xfull[b], (uint32_t)P.xrows * P.XP * 2);
      ptx::tma_load_3d(mX, &c->xfull[b], xbuf + b * XBUF, -8, 0, e0 + x);   // x = -8: the left pad
    }
    __syncwarp();
  }
  // loads still in flight after an abort land before the CTA ends
  if (*abort && (threadIdx.x & 31) == 0)
    for (int q = max(0, x - 2); q < x; ++q) ptx::mbar_wait_drain(&c->xfull[q & 1], (q >> 1) & 1);
}

// Warp 0 when the input arrives in 16-byte vectors but not by TMA (channels last, or rows not
// a multiple of 8 wide): example x's input into buffer x & 1, each vector's elements to their
// channels' padded rows, as soon as the builders have released example x - 2; one arrival on
// xfull once the warp's stores are done.  (The builders meeting at a barrier per example to
// copy it themselves left most of them waiting on the slowest: VGG-11's first layer with
// channels-last inputs ran 84 us against 56 channels first.)
__device__ __forceinline__ void stager(const Params& P, __nv_bfloat16* xbuf0, __nv_bfloat16* xbuf1, Ctl* c, int e0,
                                       int e1) {
  volatile int* abort = &c->abort;
  const int lane = threadIdx.x & 31;
  const int nv = P.xelems >> 3, wv = P.W >> 3;
  for (int x = 0; x < e1 - e0; ++x) {
    const int b = x & 1;
    const bool w = x < 2 || ptx::mbar_wait(&c->xempty[b], ((x >> 1) & 1) ^ 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) break;
    __nv_bfloat16* xs = b ? xbuf1 : xbuf0;
    const uint4* src = reinterpret_cast<const uint4*>(P.X + (size_t)(e0 + x) * P.xelems);
    for (int q0 = 0; q0 < nv; q0 += 128) {   // four vectors in flight per lane
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = q0 + j * 32 + lane;
        if (q < nv) v[j] = __ldg(src + q);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int q = q0 + j * 32 + lane;
        if (q >= nv) continue;
        if (!P.nhwc) {
          *reinterpret_cast<uint4*>(xs + (q / wv) * P.XP + 8 + (q % wv) * 8) = v[j];
        } else {
          const __nv_bfloat16* e8 = reinterpret_cast<const __nv_bfloat16*>(&v[j]);
#pragma unroll
          for (int k = 0; k < 8; ++k) xs[xdst(P, q * 8 + k)] = e8[k];
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&c->xfull[b]);
  }
}

// Per-lane unfold metadata for the fast path: this lane's column n = 4 i + lane / 8 (i < Np/4)
// reads input position ubase[i] + h * XP + wo with h = ho + udh[i] (ubase = -1: the bias
// column's ones, -2: a zero column).
struct UnitMeta {
  int ubase[NMAX / 4], udh[NMAX / 4];
};

__device__ __forceinline__ void unit_meta(const Params& P, const Ctl* c, int lane, UnitMeta& m) {
  const int nsub = lane >> 3, nu = P.Np >> 2;
#pragma unroll
  for (int i = 0; i < NMAX / 4; ++i) {
    const int n = i * 4 + nsub;
    const int co = i < nu ? c->coff[n] : -2;
    m.ubase[i] = co >= 0 ? co + 8 + c->dw[n] : co;
    m.udh[i] = i < nu ? c->dh[n] : 0;
  }
}

// One warp forms chunk u (64 pixels) of U^T: lane = (column group lane / 8, 8-pixel group
// lane % 8).  Fast inputs: each 16-byte unit is an 8-element window of a padded input row
// (two aligned loads and extract8), four units' loads in flight at once; otherwise per
// element (build_unit).
__device__ __forceinline__ void build_chunk(const Params& P, const Ctl* c, const UnitMeta& um,
                                            const __nv_bfloat16* xs, uint32_t us, int u, int lane) {
  const int tc = lane & 7, nsub = lane >> 3;
  const int t0 = u * 64 + tc * 8;
  const int nu = P.Np >> 2;
  if (!P.fast) {
    for (int i = 0; i < nu; ++i) {
      const int n = i * 4 + nsub;
      sts128(us + n * 128 + ((tc ^ (n & 7)) << 4), build_unit(P, c, xs, n, t0));
    }
    return;
  }
  const uint32_t xa = ptx::smem_u32(xs);
  const bool in_t = t0 < P.T;
  const int ho = t0 / P.Wout, wo = t0 - ho * P.Wout;
#pragma unroll
  for (int i0 = 0; i0 < NMAX / 4; i0 += 4) {
    if (i0 >= nu) break;
    uint4 w0[4], w1[4];
    int rr[4], kind[4];   // 0 zeros, 1 input window, 2 the bias column's ones
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int base = um.ubase[i0 + j];
      const int h = ho + um.udh[i0 + j];
      int kd = 0, r = 0;
      w0[j] = make_uint4(0u, 0u, 0u, 0u);
      w1[j] = w0[j];
      if (in_t && base >= 0 && h >= 0 && h < P.H) {
        const int pos = base + h * P.XP + wo;
        const uint32_t ad = xa + (uint32_t)(pos & ~7) * 2;
        w0[j] = lds128(ad);
        w1[j] = lds128(ad + 16);
        r = pos & 7;
        kd = 1;
      } else if (in_t && base == -1) {
        kd = 2;
      }
      rr[j] = r;
      kind[j] = kd;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = (i0 + j) * 4 + nsub;
      const uint4 v = kind[j] == 1   ? extract8(w0[j], w1[j], rr[j])
                      : kind[j] == 2 ? make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u)
                                     : make_uint4(0u, 0u, 0u, 0u);
      sts128(us + n * 128 + ((tc ^ (n & 7)) << 4), v);
    }
  }
}

// Warps 2, 3, 8-11 (builder bw): chunks k with k % 6 == bw, in order.  Per chunk: the G copies
// go out, U^T is formed while they land, then the copies are waited for and everything is
// made visible to the tensor core before the builder's one arrival on the chunk's full
// barrier.  (Issuing a chunk's copies one chunk of the builder ahead measured slower: the
// builder then waits for a ring slot six chunks earlier.)  The input of example x sits in
// buffer x & 1: inputs that warp 0 lands (by TMA or vector copies) are waited for (xfull) and
// released per builder (xempty); otherwise the builders copy it element by element and meet at
// a barrier before using it.  Every builder walks every example (also after an abort, when it
// skips the work) so that the barrier and the release counts stay complete.
__device__ __forceinline__ void builders(const Params& P, uint8_t* smem, __nv_bfloat16* xbuf0,
                                         __nv_bfloat16* xbuf1, Ctl* c, int e0, int e1, int m0, int bw) {
  volatile int* abort = &c->abort;
  const int lane = threadIdx.x & 31, bt = bw * 32 + lane;
  UnitMeta um;
  unit_meta(P, c, lane, um);
  const bool xbar = P.xtma || P.xvec;   // the input arrives through xfull / xempty (TMA or warp 0)
  for (int e = e0; e < e1; ++e) {
    const int x = e - e0;
    __nv_bfloat16* xs = (x & 1) ? xbuf1 : xbuf0;
    bool live = true;
    if (xbar) {
      const bool w = ptx::mbar_wait(&c->xfull[x & 1], (x >> 1) & 1, abort, P.status);
      live = __all_sync(0xffffffffu, w);
    } else {
      load_x_scalar(P, e, bt, xs);
      asm volatile("bar.sync 3, %0;" ::"r"(kBT) : "memory");
    }
    for (int u = 0; u < P.nk && live; ++u) {
      const int k = x * P.nk + u;
      if (k % kBuilders != bw) continue;
      const int s = k % P.nst;
      const bool w = k < P.nst || ptx::mbar_wait(&c->empty[s], ((k / P.nst) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      const uint32_t st = ptx::smem_u32(smem + s * P.sbytes);
      copy_g(P, st, e, u, m0, lane);
      build_chunk(P, c, um, xs, st + P.ubase, u, lane);
      asm volatile("cp.async.wait_all;" ::: "memory");
      ptx::fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c->full[s]);
    }
    if (xbar) {
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c->xempty[x & 1]);
    }
  }
}

// Warps 4-7: one output row per thread, the example's Np columns from TMEM.
template <bool kNorm>
__device__ __forceinline__ void epilogue(const Params& P, Ctl* c, uint32_t tmem, int e0, int e1, int m0) {
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int m = m0 + quarter * 32 + lane;
  const bool row = m < P.p;
  float acc[kNorm ? 1 : NMAX];
  if constexpr (!kNorm) {
#pragma unroll
    for (int j = 0; j < NMAX; ++j) acc[j] = 0.f;
  }
  bool ok = true;
  for (int e = e0; e < e1; ++e) {
    const int x = e - e0, b = x % NBUF;
    float ss = 0.f;
    if (ok) {
      const bool w = ptx::mbar_wait(&c->accum[b], (x / NBUF) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) ok = false;
    }
    if (ok) {
      ptx::tc_fence_after();
      float vv[NMAX / 16][16];
      const uint32_t base = tmem + b * 64 + ((uint32_t)(quarter * 32) << 16);
      // all 64 columns of the buffer (those past Np hold stale values and are never used)
#pragma unroll
      for (int ch = 0; ch < NMAX / 16; ++ch) ptx::tmem_ld16(base + ch * 16, vv[ch]);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c->tfree[b]);
      if constexpr (kNorm) {
        if (row) {
          float* kp = P.keep ? P.keep + ((size_t)e * P.p + m) * P.D : nullptr;
#pragma unroll
          for (int ch = 0; ch < NMAX / 16; ++ch) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = ch * 16 + jj;
              const float x2 = vv[ch][jj];
              if (j < P.D || (P.bias && j == P.D)) ss = fmaf(x2, x2, ss);
              if (kp && j < P.D) kp[j] = x2;
              if (P.keep_b && P.bias && j == P.D) P.keep_b[(size_t)e * P.p + m] = x2;
            }
          }
        }
      } else {
        const float cf = __ldg(P.factors + e);
#pragma unroll
        for (int ch = 0; ch < NMAX / 16; ++ch)
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) acc[ch * 16 + jj] = fmaf(cf, vv[ch][jj], acc[ch * 16 + jj]);
      }
    }
    if constexpr (kNorm) {
      ss = warp_sum(ss);
      if (lane == 0) c->red[x & 1][quarter] = ss;
      asm volatile("bar.sync 2, %0;" ::"r"(32 * kEpiWarps) : "memory");
      if (threadIdx.x == 32 * kEpiFirst && !*abort) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kEpiWarps; ++w) t += c->red[x & 1][w];
        P.out[(size_t)blockIdx.x * P.B + e] = t;
      }
    }
  }
  if constexpr (!kNorm) {
    if (!ok || *abort || !row) return;
    // with one split the partial is the sum itself (added to dW / db on request)
    const bool direct = gridDim.z == 1;
    float* pw = P.part + ((size_t)blockIdx.z * P.p + m) * P.D;
    const bool add = direct && P.accumulate;
    float* pb = P.bias && P.part_b ? P.part_b + (size_t)blockIdx.z * P.p + m : nullptr;
#pragma unroll
    for (int ch = 0; ch < NMAX / 16; ++ch)
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = ch * 16 + jj;
        const float a = acc[j];
        if (j < P.D) pw[j] = add ? pw[j] + a : a;
        if (pb && j == P.D) *pb = add ? *pb + a : a;
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
    ptx::tmem_dealloc(tmem, 256);
  }
}

template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
tc_unfold_kernel(const __grid_constant__ CUtensorMap mapX, Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __nv_bfloat16* xbuf0 = reinterpret_cast<__nv_bfloat16*>(smem + RING);
  __nv_bfloat16* xbuf1 = reinterpret_cast<__nv_bfloat16*>(smem + RING + XBUF);
  Ctl* c = reinterpret_cast<Ctl*>(smem + RING + 2 * XBUF);
  const int warp = threadIdx.x >> 5;
  const int m0 = blockIdx.x * BM;
  const int e0 = blockIdx.z * P.ex_per_split;
  const int e1 = min(P.B, e0 + P.ex_per_split);

  // The input buffers' pads (channels first, inputs the builders copy): zero, never written.
  for (int q = threadIdx.x; q < 2 * XBUF / 16; q += blockDim.x)
    reinterpret_cast<uint4*>(smem + RING)[q] = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  if (threadIdx.x < NMAX) {   // column n = (c*kh + ih)*k + iw of the unfold; -1 the bias, -2 padding
    const int n = threadIdx.x, kk = P.kh * P.k;
    if (n < P.D) {
      const int ch = n / kk, r = n - ch * kk, ih = r / P.k, iw = r - ih * P.k;
      c->coff[n] = ch * P.H * P.XP;
      c->dh[n] = ih * P.dil - P.padh;
      c->dw[n] = iw * P.dil - P.pad;
    } else {
      c->coff[n] = (n == P.D && P.bias) ? -1 : -2;
      c->dh[n] = 0;
      c->dw[n] = 0;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.nst; ++s) {
      ptx::mbar_init(&c->full[s], 1);     // the chunk's builder
      ptx::mbar_init(&c->empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      ptx::mbar_init(&c->accum[b], 1);
      ptx::mbar_init(&c->tfree[b], kEpiWarps);
    }
    ptx::mbar_init(&c->drain, 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&c->xfull[b], 1);
      ptx::mbar_init(&c->xempty[b], kBuilders);
    }
    c->abort = 0;
    ptx::fence_mbar_init();
    if (P.xtma) ptx::prefetch_tensormap(&mapX);
  }
  if (warp == 1) ptx::tmem_alloc(&c->tmem, 256);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c->tmem;
  pdl_trigger();   // the next kernel in the stream may start launching
  pdl_wait();      // the previous kernel has completed; its writes are visible

  if (warp >= kEpiFirst && warp < kEpiFirst + kEpiWarps) {
    epilogue<kNorm>(P, c, tmem, e0, e1, m0);
  } else if (warp == 0) {
    if (P.xtma) producer(P, &mapX, smem + RING, c, e0, e1);
    else if (P.xvec) stager(P, xbuf0, xbuf1, c, e0, e1);
  } else if (warp == 1) {
    mma_issuer(P, smem, c, tmem, e0, e1);
  } else {
    const int bw = warp < kEpiFirst ? warp - 2 : warp - kEpiFirst - kEpiWarps + 2;   // 0..5
    builders(P, smem, xbuf0, xbuf1, c, e0, e1, m0, bw);
  }
  finish(c, tmem);
}

}  // namespace tcunf
}  // namespace dpk

namespace dph {
using namespace dpk;

static int cdiv_u(long a, long b) { return (int)((a + b - 1) / b); }
static size_t al256_u(size_t n) { return (n + 255) & ~size_t(255); }

static int unfold_np(const Geom& g) { return (g.D + (g.has_bias ? 1 : 0) + 15) / 16 * 16; }
static int unfold_xp(const Geom& g) { return (g.W + 7) / 8 * 8 + 16; }

bool tc_unfold_supported(const Geom& g) {
  if (!g.conv || g.Z != 1 || g.kz != 1 || g.B < 1 || g.p < 1 || g.T < 1) return false;
  if (unfold_np(g) > tcunf::NMAX) return false;
  if (g.nhwc ? g.p % 8 != 0 : g.T % 8 != 0) return false;   // 16-byte TMA row strides of G
  const long xe = (long)g.Cin * g.H * unfold_xp(g);   // the input on chip, channels first, padded rows
  return xe <= tcunf::XMAXE;
}

static int unfold_splits(const Geom& g) {
  const int tm = cdiv_u(g.p, tcunf::BM);
  const long want = std::max<long>(1, std::min<long>(g.B, 152 / tm));
  return cdiv_u(g.B, cdiv_u(g.B, want));
}

size_t tc_unfold_ws_bytes(const Geom& g, bool norm) {
  const int tm = cdiv_u(g.p, tcunf::BM), splits = unfold_splits(g);
  if (norm) return tm > 1 ? al256_u((size_t)tm * g.B * 4) : 0;
  return splits > 1 ? al256_u((size_t)splits * g.p * g.D * 4) + al256_u((size_t)splits * g.p * 4) : 0;
}

// The input of one example as one TMA box of its Cin*H rows, XP wide from column -8, so
// that the box's zero fill forms the padded rows (channels first, W % 8 == 0, aligned input).
static bool unfold_xmap(const Geom& g, const void* A, const tcunf::Params& P, CUtensorMap* mX) {
  *mX = CUtensorMap{};
  if (!P.xtma) return true;
  const uint64_t dx[3] = {(uint64_t)g.W, (uint64_t)g.Cin * g.H, (uint64_t)g.B};
  const uint64_t sx[2] = {(uint64_t)g.W * 2, (uint64_t)g.Cin * g.H * g.W * 2};
  const uint32_t box[3] = {(uint32_t)P.XP, (uint32_t)P.xrows, 1};
  return encode_tmap_bf16(mX, A, 3, dx, sx, box, false);
}

static tcunf::Params unfold_params(const Geom& g, const void* A, unsigned* status) {
  tcunf::Params P = {};
  P.X = static_cast<const __nv_bfloat16*>(A);
  P.grows = std::min(g.p, tcunf::BM);
  P.status = status;
  P.B = g.B;
  P.T = g.T;
  P.p = g.p;
  P.D = g.D;
  P.Np = unfold_np(g);
  P.bias = g.has_bias;
  P.Cin = g.Cin;
  P.H = g.H;
  P.W = g.W;
  P.Hout = g.Hout;
  P.Wout = g.Wout;
  P.k = g.k;
  P.kh = g.kh;
  P.stride = g.stride;
  P.pad = g.pad;
  P.padh = g.padh;
  P.dil = g.dil;
  P.nhwc = g.nhwc;
  P.XP = unfold_xp(g);
  P.xelems = g.Cin * g.H * g.W;
  const bool al = (reinterpret_cast<uintptr_t>(A) & 15u) == 0;
  P.xvec = al && P.xelems % 8 == 0 && (g.nhwc || g.W % 8 == 0);
  P.fast = g.stride == 1 && g.Wout % 8 == 0 && g.pad <= 8 && g.padh <= 8;
  P.xrows = g.Cin * g.H;
  P.xtma = al && !g.nhwc && g.W % 8 == 0 && P.XP <= 256 && P.xrows <= 256;
  P.nk = cdiv_u(g.T, 64);
  // the ring: G blocks of 8 KB when p <= 64 (the MMA's rows 64-127 read past them, inside the
  // ring), else 16 KB, then the U^T block; the last stage's reads end inside the ring
  P.ubase = g.p <= 64 ? 8192 : 16384;
  P.sbytes = (P.ubase + P.Np * 128 + 1023) / 1024 * 1024;
  const int tail = std::max(P.sbytes, 16384);
  P.nst = std::min(tcunf::MAXST, (tcunf::RING - tail) / P.sbytes + 1);
  const int splits = unfold_splits(g);
  P.ex_per_split = cdiv_u(g.B, splits);
  return P;
}

template <bool kNorm>
static cudaError_t unfold_launch(const Geom& g, const CUtensorMap& mX, const tcunf::Params& P, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcunf::tc_unfold_kernel<kNorm>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tcunf::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(cdiv_u(g.p, tcunf::BM), 1, cdiv_u(g.B, P.ex_per_split));
  launch_plain(tcunf::tc_unfold_kernel<kNorm>, grid, tcunf::kThreads, tcunf::SMEM, s, mX, P);
  return cudaGetLastError();
}

cudaError_t launch_tc_unfold_norm(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                  unsigned* status, cudaStream_t s, float* keep, float* keep_b) {
  if (!tc_unfold_supported(g)) return cudaErrorInvalidValue;
  CUtensorMap mX;
  tcunf::Params P = unfold_params(g, A, status);
  P.G = static_cast<const __nv_bfloat16*>(G);
  if (!unfold_xmap(g, A, P, &mX)) return cudaErrorInvalidValue;
  const int tm = cdiv_u(g.p, tcunf::BM);
  if (tm > 1 && !ws) return cudaErrorInvalidValue;
  P.out = tm > 1 ? static_cast<float*>(ws) : out;
  P.keep = keep;
  P.keep_b = g.has_bias ? keep_b : nullptr;
  cudaError_t e = unfold_launch<true>(g, mX, P, s);
  if (e != cudaSuccess || tm == 1) return e;
  return launch_reduce_splits(static_cast<float*>(ws), tm, (size_t)g.B, out, 0, s);
}

cudaError_t launch_tc_unfold_sum(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                                 float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s,
                                 NoiseArgs* nz) {
  if (!tc_unfold_supported(g)) return cudaErrorInvalidValue;
  CUtensorMap mX;
  tcunf::Params P = unfold_params(g, A, status);
  P.G = static_cast<const __nv_bfloat16*>(G);
  if (!unfold_xmap(g, A, P, &mX)) return cudaErrorInvalidValue;
  const int splits = cdiv_u(g.B, P.ex_per_split);
  if (splits > 1 && !ws) return cudaErrorInvalidValue;
  float* part_w = static_cast<float*>(ws);
  float* part_b = splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                                        al256_u((size_t)splits * g.p * g.D * 4))
                             : nullptr;
  P.factors = factors;
  P.part = splits > 1 ? part_w : dW;
  P.part_b = db ? (splits > 1 ? part_b : db) : nullptr;
  P.accumulate = accumulate;
  cudaError_t e = unfold_launch<false>(g, mX, P, s);
  if (e != cudaSuccess || splits == 1) return e;
  const size_t nw = (size_t)g.p * g.D;
  return launch_reduce_splits2(SplitSeg{part_w, nw, nw, dW}, SplitSeg{part_b, (size_t)g.p, db ? (size_t)g.p : 0, db},
                               splits, accumulate, s, nz);
}

}  // namespace dph
