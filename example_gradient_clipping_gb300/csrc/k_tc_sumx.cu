// Clipped sum with the clip factor applied per example in fp32, on the tensor cores.
//
//   dW = sum_i c_i P_i,  P_i = G_i^T A_i  (the per-example gradient of [MixGhost] eq. 2.4),
//   db = sum_i c_i sum_t G_i[t, :]
//
// The reweighted contraction of [FastClip] section 5 written per example: the tensor
// cores form P_i for one 128 x 256 output tile in TMEM (one buffer per example,
// double-buffered), and eight epilogue warps fold it into register accumulators
// with D += c_i * P_i.  No operand is rescaled or re-rounded, and no CUDA-core work
// sits between a TMA load and the MMA that consumes it.  Rows of example i are loaded
// with 3D TMA boxes [1, rows, 64] (rows past T read as zero): full 64-row stages,
// then 16-row stages for the remainder.  A column tile narrower than 256 (the layer's
// last, or a narrow layer) loads only the boxes it needs and runs its MMAs at that width
// (a multiple of 16).  In CTAs of the first column tile the
// epilogue warps also sum the G rows from shared memory for the bias.  Examples are
// split across the CTAs of a thread-block cluster (up to 4 per output tile): after
// the main loop each CTA stages its fp32 partial tile in its own shared memory, and
// after a cluster barrier each CTA adds one slice of rows from every peer over
// distributed shared memory, in a fixed order, so the result is deterministic and
// needs no global workspace.  When clusters of 4 cannot cover the GPU (few output
// tiles), the examples are split over the grid instead: each CTA writes its partial
// tile to the workspace and a second kernel sums the partials in split order.
//   warpgroup 0: warps 0 and 2 TMA producers (alternate stages: one issuing thread
//                streams only ~48 B/clk into an SM, two reach ~96), warp 1 MMA
//                issuer, warp 3 reduces the bias across the cluster (64 registers
//                each after setmaxnreg.dec)
//   warpgroups 1-2: eight epilogue warps, two per TMEM lane quarter, 128 columns
//                each (216 registers after setmaxnreg.inc: 128 accumulators); in
//                CTAs of the first column tile they also sum the G rows of every
//                stage for the bias (they idle between examples otherwise)
// Register budget: 128 x 64 + 256 x 216 = 63488 <= 64512 = 384 threads x 168 at launch.
//
// Norm mode (kNorm): the same per-example products serve the instantiated norm of
// [MixGhost] section 3 (per-sample gradients formed, then their Frobenius norm):
// the epilogue adds up P_i^2 over the tile instead of folding c_i P_i, plus the
// squared bias gradient ||sum_t G_i[t, :]||^2 over the tile's outputs in the first
// column tile, and writes one partial per (tile, example); a fixed-order reduction
// over the tiles gives ||g_i||^2.  No cluster: the examples are split over the grid.
// With `keep`, the epilogue also stores P_i and the bias gradient of every example for
// the kept-gradient clipped sum.
#include <algorithm>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tcsumx {

#ifndef DPCLIP_SUMX_FR
#define DPCLIP_SUMX_FR 64
#endif
#ifndef DPCLIP_SUMX_STAGES
#define DPCLIP_SUMX_STAGES 4
#endif
constexpr int BM = 128, BN = 256, STAGES = DPCLIP_SUMX_STAGES;
constexpr int FR = DPCLIP_SUMX_FR;           // rows of a full stage (a multiple of 16)
constexpr int BOX = FR * 64 * 2;             // FR rows x 128 B
constexpr int STAGE = 6 * BOX;               // G: 2 boxes, A: 4 boxes
constexpr int kEpiWarps = 8;
constexpr int kBiasWarps = 1;                // warp 3: joins the workers' barriers
constexpr int kThreads = 384;                // 3 warpgroups
constexpr int kEpiFirst = 4;                 // first epilogue warp
constexpr int kSyncThreads = 32 * (kBiasWarps + kEpiWarps);   // warps 3-11, named barrier 1
constexpr int kLeader = 96;                  // first worker thread (warp 3, lane 0)
constexpr int SMEM = STAGES * STAGE + 1024 + 512;

constexpr int PSTR = BN + 4;                 // staged partial row stride (floats)
constexpr int PART_BYTES = BM * PSTR * 4;    // staged weight partial, then 128 bias floats
static_assert(PART_BYTES + BM * 4 <= STAGES * STAGE, "staging fits in the stage buffers");
static_assert(STAGES % 2 == 0, "each slot is filled by one of the two producers");

struct Params {
  const float* factors;
  float* dW;
  float* db;          // null: no bias
  unsigned* status;
  int B, T, p, d;
  int ex_per_split, splits, accumulate;   // splits = cluster size along z
  int nfull, n16;     // per example: 64-row stages, then 16-row stages
  float* part;        // norm mode: [tiles, B] per-tile partial squared norms
  int norm_bias;      // norm mode: the layer has a bias
  int gsplit;         // examples split over the grid (no cluster): CTA z writes its partial
                      // tile to dW + z*p*d (db + z*p), reduced afterwards in z order
  float* keep;        // norm mode, or null: every example's gradient [B, p, d] and bias [B, p]
  float* keep_b;
  int early;          // A and G are the caller's inputs: loads may start before pdl_wait
  // Sum mode, bias: with bias_nt == 1 the CTAs of the first column tile sum the G rows of
  // every example; with bias_nt > 1 column tile j < bias_nt sums those of the examples x
  // (counted from the split's first) with x % bias_nt == j, and writes its partial bias to
  // bias_part [bias_nt, p] (summed over the tiles afterwards, in order)
  int bias_nt;
  float* bias_part;
};

// Does this CTA sum the G rows of example x (counted from its split's first) for the bias?
__device__ __forceinline__ bool bias_example(const Params& P, int x) {
  if (!P.db) return false;
  return P.bias_nt == 1 ? blockIdx.y == 0 : (int)blockIdx.y == x % P.bias_nt;
}

// Shared-memory control block after the stages.
struct Ctl {
  uint64_t full[STAGES], empty[STAGES], bfree[STAGES], accum[2], tfree[2], drain;
  uint32_t tmem;
  int abort;
  int flags[2];       // [1] go / no-go after the main loops
  float red[2][8];    // norm mode: per-warp partials of the last two examples
};

__device__ __forceinline__ void sync_workers() {
  asm volatile("bar.sync 1, %0;" ::"r"(kSyncThreads) : "memory");
}

// One CTA-wide go/no-go after the main loops (the branches that follow hold barriers).
__device__ __forceinline__ bool finish_decision(Ctl* c) {
  sync_workers();
  if (threadIdx.x == kLeader) c->flags[1] = *(volatile int*)&c->abort ? 0 : 1;
  sync_workers();
  return c->flags[1] != 0;
}

// The MMA width of column tile n0: the layer's remaining columns rounded up to 16 (at most
// BN), so narrow layers load and multiply only their own columns.
// kTrim false (every column tile full: D % 256 == 0) keeps the full-width code paths.
template <bool kTrim>
__device__ __forceinline__ int tile_n(const Params& P, int n0) {
  if constexpr (!kTrim) return BN;
  else return min(BN, (P.d - n0 + 15) & ~15);
}

// Warps 0 and 2 (all lanes): TMA producers; producer `pr` loads the stages k with
// k % 2 == pr (the two G boxes and the A boxes the tile's width needs).
template <bool kNorm, bool kTrim>
__device__ __forceinline__ void producer(const Params& P, const CUtensorMap* mG64, const CUtensorMap* mA64,
                                         const CUtensorMap* mG16, const CUtensorMap* mA16, uint8_t* smem,
                                         Ctl* c, int e0, int e1, int m0, int n0, int pr) {
  volatile int* abort = &c->abort;
  const int ns = P.nfull + P.n16;
  const int na = (tile_n<kTrim>(P, n0) + 63) / 64;      // A boxes per stage
  int k = 0, issued = 0;
  bool live = true;
  int last = -1;
  // sum mode: per slot, whether its last stage had its G rows summed for the bias (the
  // slot is then also released by the epilogue warps, on bfree) and the parity of the
  // slot's such rounds so far
  uint32_t pend = 0, par = 0;
  for (int e = e0; e < e1 && live; ++e) {
    const bool bias_e = !kNorm && bias_example(P, e - e0);
    for (int u = 0; u < ns; ++u, ++k) {
      if ((k & 1) != pr) continue;
      const int s = k % STAGES;
      bool w = ptx::mbar_wait(&c->empty[s], ((k / STAGES) & 1) ^ 1, abort, P.status);
      if (!kNorm && ((pend >> s) & 1u)) {
        w = w && ptx::mbar_wait(&c->bfree[s], (par >> s) & 1u, abort, P.status);
        par ^= 1u << s;
        pend &= ~(1u << s);
      }
      if (bias_e) pend |= 1u << s;
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      const bool big = u < P.nfull;
      const int y = big ? u * FR : P.nfull * FR + (u - P.nfull) * 16;
      const CUtensorMap* mg = big ? mG64 : mG16;
      const CUtensorMap* ma = big ? mA64 : mA16;
      uint8_t* st = smem + s * STAGE;
      if (ptx::elect_one()) {
        ptx::mbar_arrive_expect_tx(&c->full[s], (big ? FR : 16) * 128 * (2 + na));
        ptx::tma_load_3d(mg, &c->full[s], st, m0, y, e);
        ptx::tma_load_3d(mg, &c->full[s], st + BOX, m0 + 64, y, e);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < na) ptx::tma_load_3d(ma, &c->full[s], st + (2 + j) * BOX, n0 + 64 * j, y, e);
      }
      __syncwarp();
      ++issued;
      last = k;
    }
  }
  if (*abort && (threadIdx.x & 31) == 0) {   // let this producer's copies in flight land
    for (int q = max(0, last - STAGES + 1); q <= last; ++q)
      if ((q & 1) == pr) ptx::mbar_wait_drain(&c->full[q % STAGES], (q / STAGES) & 1);
  }
  (void)issued;
}

#ifndef DPCLIP_SUMX_PREFETCH
#define DPCLIP_SUMX_PREFETCH 2
#endif
// Examples ahead of the producers whose rows warp 3 prefetches into L2.
constexpr int kPrefetch = DPCLIP_SUMX_PREFETCH;

// TMA prefetch of one box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}

// Warp 3 (sum mode): L2 prefetch of the rows kPrefetch examples ahead of the producers,
// so that their loads find the rows in L2 instead of waiting for HBM (the CTAs that share
// a box request it at about the same time, and each waited for the first one's miss).
// The CTAs of the first column tile prefetch their G columns, those of the first row tile
// their A columns, so every byte is prefetched once.  Warp 3 follows the producers by
// waiting for the first stage of each example to land.
template <bool kTrim>
__device__ __forceinline__ void prefetcher(const Params& P, const CUtensorMap* mG64, const CUtensorMap* mA64,
                                           const CUtensorMap* mG16, const CUtensorMap* mA16, Ctl* c, int e0,
                                           int e1, int m0, int n0) {
  const bool pg = blockIdx.y == 0, pa = blockIdx.x == 0;
  if (!pg && !pa) return;
  volatile int* abort = &c->abort;
  const int ns = P.nfull + P.n16;
  const int na = (tile_n<kTrim>(P, n0) + 63) / 64;
  auto fetch = [&](int e) {
    if (ptx::elect_one()) {
      for (int u = 0; u < ns; ++u) {
        const bool big = u < P.nfull;
        const int y = big ? u * FR : P.nfull * FR + (u - P.nfull) * 16;
        if (pg) {
          tma_prefetch_3d(big ? mG64 : mG16, m0, y, e);
          tma_prefetch_3d(big ? mG64 : mG16, m0 + 64, y, e);
        }
        if (pa)
          for (int j = 0; j < na; ++j) tma_prefetch_3d(big ? mA64 : mA16, n0 + 64 * j, y, e);
      }
    }
    __syncwarp();
  };
  for (int e = e0; e < min(e1, e0 + kPrefetch); ++e) fetch(e);
  for (int e = e0; e + kPrefetch < e1; ++e) {
    const int k = (e - e0) * ns;
    const bool w = ptx::mbar_wait(&c->full[k % STAGES], (k / STAGES) & 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) return;
    fetch(e + kPrefetch);
  }
}

// Warp 1 (all lanes): MMA issuer.  Descriptors are built once per stage from the
// stage base; the elected lane issues the MMAs and the commits.
template <bool kTrim>
__device__ __forceinline__ void mma_issuer(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0,
                                           int e1) {
  volatile int* abort = &c->abort;
  const int ns = P.nfull + P.n16;
  const uint32_t idesc = ptx::idesc_bf16_f32(BM, tile_n<kTrim>(P, blockIdx.y * BN), 1, 1);
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
    for (int u = 0; u < ns; ++u, ++k) {
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait(&c->full[s], (k / STAGES) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      // no tcgen05 fence here: the TMA data is ordered by the mbarrier (both async proxy),
      // and a per-stage fence was measured to stall the MMA pipe
      const uint32_t g = ptx::smem_u32(smem + s * STAGE);
      // 16 rows per MMA = two 8-row groups of 1024 B; 64-column chunks are BOX apart
      const uint64_t da = ptx::sdesc_sw128(g, BOX, 1024);
      const uint64_t dbd = ptx::sdesc_sw128(g + 2 * BOX, BOX, 1024);
      if (ptx::elect_one()) {
        if (u < P.nfull) {
#pragma unroll
          for (int kk = 0; kk < FR / 16; ++kk)
            ptx::umma_bf16(d_tmem, ptx::sdesc_add(da, kk * 2048), ptx::sdesc_add(dbd, kk * 2048), idesc,
                           (u | kk) != 0);
        } else {
          ptx::umma_bf16(d_tmem, da, dbd, idesc, u != 0);
        }
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

// t[0..7] += the eight bf16 values of v.
__device__ __forceinline__ void add_bf16x8(const uint4& v, float* t) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    t[2 * q] += f.x;
    t[2 * q + 1] += f.y;
  }
}

// Norm mode, warps 4-11: per example, sum of P_e^2 over the tile (plus the squared
// bias sums in the first column tile) -> part[tile, e].  Every epilogue warp passes
// one barrier per example, also after an abort, so none waits for a warp that left.
template <bool kTrim>
__device__ __forceinline__ void epilogue_norm(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem,
                                              int e0, int e1, bool do_bias) {
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = (warp - kEpiFirst) >> 2;
  const int et = threadIdx.x - 32 * kEpiFirst;
  const int bbox = et >> 7, bq = (et >> 4) & 7, bj = et & 15;
  const int ns = P.nfull + P.n16;
  const size_t tile = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
  const int ncol = tile_n<kTrim>(P, blockIdx.y * BN) - half * 128;   // this warp's columns with products
  bool ok = true;
  int k = 0;
  for (int e = e0; e < e1; ++e) {
    const int x = e - e0, b = x & 1;
    float ss = 0.f;
    if (ok && do_bias) {
      float bt[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) bt[q] = 0.f;
      for (int u = 0; u < ns; ++u, ++k) {
        const int s = k % STAGES;
        const bool w = ptx::mbar_wait(&c->full[s], (k / STAGES) & 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        const uint8_t* gt = smem + s * STAGE + bbox * BOX + bj * 128 + ((bq ^ (bj & 7)) << 4);
        if (u < P.nfull) {
          uint4 v[FR / 16];
#pragma unroll
          for (int h = 0; h < FR / 16; ++h) v[h] = *reinterpret_cast<const uint4*>(gt + h * 16 * 128);
#pragma unroll
          for (int h = 0; h < FR / 16; ++h) add_bf16x8(v[h], bt);
        } else {
          add_bf16x8(*reinterpret_cast<const uint4*>(gt), bt);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c->empty[s]);
      }
      // the 16 lanes of a half-warp share 8 output columns: total them, square them once
      float bsq = 0.f;
      const int mb = blockIdx.x * BM + bbox * 64 + bq * 8;   // this group's first output
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float v = bt[q];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        bsq = fmaf(v, v, bsq);
        if (P.keep_b && bj == 0 && mb + q < P.p) P.keep_b[(size_t)e * P.p + mb + q] = v;
      }
      if (bj == 0) ss = bsq;
    }
    if (ok) {
      const bool w = ptx::mbar_wait(&c->accum[b], (x >> 1) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) ok = false;
    }
    if (ok) {
      ptx::tc_fence_after();
      const uint32_t base = tmem + b * 256 + half * 128 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
      for (int ch = 0; ch < 8; ch += 2) {
        if (kTrim && ch * 16 >= ncol) break;       // (warp-uniform; widths are multiples of 16)
        float v0[16], v1[16];
        ptx::tmem_ld16(base + ch * 16, v0);
        ptx::tmem_ld16(base + ch * 16 + 16, v1);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) ss = fmaf(v0[j], v0[j], ss);
        if (!kTrim || (ch + 1) * 16 < ncol) {
#pragma unroll
          for (int j = 0; j < 16; ++j) ss = fmaf(v1[j], v1[j], ss);
        }
        const int m = blockIdx.x * BM + quarter * 32 + lane;
        const int n = blockIdx.y * BN + half * 128 + ch * 16;   // d % 8 == 0: whole float4s
        if (P.keep && m < P.p) {
          float* dst = P.keep + ((size_t)e * P.p + m) * P.d + n;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (n + 4 * j < P.d)
              *reinterpret_cast<float4*>(dst + 4 * j) = make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
            if (n + 16 + 4 * j < P.d)
              *reinterpret_cast<float4*>(dst + 16 + 4 * j) =
                  make_float4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&c->tfree[b]);
    }
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
  finish_decision(c);
}

// Warps 4-11: drain P_e from TMEM into fp32 register accumulators, D += c_e * P_e.
template <bool kTrim>
__device__ __forceinline__ void epilogue(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0,
                                         int e1, int m0, int n0, bool do_bias) {
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
  const int half = (warp - kEpiFirst) >> 2;      // columns 128*half .. +127
  // bias: thread -> (box, 16-byte chunk, row phase); the 16 threads sharing a column
  // group are the lanes of one half-warp
  const int et = threadIdx.x - 32 * kEpiFirst;   // 0..255
  const int bbox = et >> 7, bq = (et >> 4) & 7, bj = et & 15;
  const int ns = P.nfull + P.n16;
  const int ncol = tile_n<kTrim>(P, n0) - half * 128;   // this warp's columns with products (past them:
                                                  // stale TMEM, accumulated but never stored)
  float bacc[8], btmp[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) bacc[q] = btmp[q] = 0.f;
  float acc[128];
#pragma unroll
  for (int j = 0; j < 128; ++j) acc[j] = 0.f;
  bool ok = true;
  for (int e = e0; e < e1 && ok; ++e) {
    const int x = e - e0, b = x & 1;
    const bool bias_e = bias_example(P, x);
    if (bias_e) {
      for (int u = 0; u < ns; ++u) {
        const int k = x * ns + u, s = k % STAGES;
        const bool w = ptx::mbar_wait(&c->full[s], (k / STAGES) & 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        // 128-byte swizzle: chunk q of row r sits at chunk q ^ (r % 8)
        const uint8_t* gt = smem + s * STAGE + bbox * BOX + bj * 128 + ((bq ^ (bj & 7)) << 4);
        if (u < P.nfull) {
          uint4 v[FR / 16];
#pragma unroll
          for (int h = 0; h < FR / 16; ++h) v[h] = *reinterpret_cast<const uint4*>(gt + h * 16 * 128);
#pragma unroll
          for (int h = 0; h < FR / 16; ++h) add_bf16x8(v[h], btmp);
        } else {
          add_bf16x8(*reinterpret_cast<const uint4*>(gt), btmp);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c->bfree[s]);
      }
      if (!ok) break;
    }
    const bool w = ptx::mbar_wait(&c->accum[b], (x >> 1) & 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
    ptx::tc_fence_after();
    const float cf = __ldg(P.factors + e);
    const uint32_t base = tmem + b * 256 + half * 128 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
    for (int ch = 0; ch < 8; ch += 4) {
      if (kTrim && ch * 16 >= ncol) break;         // (warp-uniform)
      float v[4][16];                              // four loads in flight per wait
#pragma unroll
      for (int u = 0; u < 4; ++u) ptx::tmem_ld16(base + (ch + u) * 16, v[u]);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[(ch + u) * 16 + j] = fmaf(cf, v[u][j], acc[(ch + u) * 16 + j]);
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&c->tfree[b]);
    if (bias_e) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        bacc[q] = fmaf(cf, btmp[q], bacc[q]);
        btmp[q] = 0.f;
      }
    }
  }
  if (do_bias) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float v = bacc[q];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      bacc[q] = v;
    }
  }
  const bool good = finish_decision(c);
  if (!good) return;
  if (do_bias && bj == 0) {
    float* partb = reinterpret_cast<float*>(smem + PART_BYTES);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = bbox * 64 + bq * 8 + q;
      if (P.splits > 1) partb[j] = bacc[q];   // staged for the cluster reduction
      else if (P.bias_nt > 1 && m0 + j < P.p) P.bias_part[(size_t)blockIdx.y * P.p + m0 + j] = bacc[q];
      else if (P.gsplit && m0 + j < P.p) P.db[(size_t)blockIdx.z * P.p + m0 + j] = bacc[q];
      else if (m0 + j < P.p) P.db[m0 + j] = bacc[q] + (P.accumulate ? P.db[m0 + j] : 0.f);
    }
  }
  // stage the tile in shared memory (the stage buffers are idle: every load was consumed
  // and every MMA completed before the last accum wait)
  const int row = quarter * 32 + lane;
  {
    float* part = reinterpret_cast<float*>(smem) + row * PSTR + half * 128;
#pragma unroll
    for (int j = 0; j < 128; j += 4)
      *reinterpret_cast<float4*>(part + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
  }
  if (P.splits > 1) return;      // the cluster reduction reads the staged partials
  // this CTA owns the tile (one split), or its grid split's partial of it: whole rows
  // from shared memory, 64 threads per 1 KB row, so the stores coalesce
  asm volatile("bar.sync 2, %0;" ::"r"(32 * kEpiWarps) : "memory");
  const int et2 = threadIdx.x - 32 * kEpiFirst;
  const bool vec = (P.d & 3) == 0;
  const int accum = P.gsplit ? 0 : P.accumulate;
  float* base_out = P.dW + (P.gsplit ? (size_t)blockIdx.z * P.p * P.d : 0);
  const float* stg = reinterpret_cast<const float*>(smem);
  for (int item = et2; item < BM * (BN / 4); item += 32 * kEpiWarps) {
    const int r = item / (BN / 4), c4 = item % (BN / 4);
    const int m = m0 + r, n = n0 + c4 * 4;
    if (m >= P.p) continue;
    float4 o = *reinterpret_cast<const float4*>(stg + r * PSTR + c4 * 4);
    float* out = base_out + (size_t)m * P.d + n;
    if (vec && n + 4 <= P.d) {
      if (accum) {
        const float4 old = *reinterpret_cast<const float4*>(out);
        o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
      }
      *reinterpret_cast<float4*>(out) = o;
    } else {
      const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (n + q < P.d) out[q] = ov[q] + (accum ? out[q] : 0.f);
    }
  }
}

// After the cluster barrier: this CTA adds rows [r0, r1) of every peer's staged
// partial (fixed peer order) and writes them; warps 2-3 do the same for the bias.
__device__ __forceinline__ void cluster_reduce(const Params& P, uint8_t* smem, int m0, int n0, bool do_bias) {
  const int S = P.splits;
  const uint32_t rank = ptx::cluster_rank();
  const int warp = threadIdx.x >> 5;
  if (warp >= kEpiFirst) {
    const int t = threadIdx.x - 32 * kEpiFirst;     // 0..255
    const int rows_per = (BM + S - 1) / S;
    const int r0 = min(BM, (int)rank * rows_per), r1 = min(BM, r0 + rows_per);
    const uint32_t base = ptx::smem_u32(smem);
    const bool vec = (P.d & 3) == 0;
    const int items = (r1 - r0) * (BN / 4);
    for (int it0 = t; it0 < items; it0 += 512) {
      // two output float4s per pass, all peers' loads in flight together
      float4 v[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int item = it0 + h * 256;
        if (item >= items) continue;
        const int row = r0 + item / (BN / 4), c4 = item % (BN / 4);
        const uint32_t off = base + (uint32_t)(row * PSTR + c4 * 4) * 4u;
#pragma unroll
        for (int sp = 0; sp < 8; ++sp)
          if (sp < S) v[h][sp] = ptx::ld_cluster_v4(ptx::map_rank(off, sp));
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int item = it0 + h * 256;
        if (item >= items) continue;
        const int row = r0 + item / (BN / 4), c4 = item % (BN / 4);
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sp = 0; sp < 8; ++sp)
          if (sp < S) { sum.x += v[h][sp].x; sum.y += v[h][sp].y; sum.z += v[h][sp].z; sum.w += v[h][sp].w; }
        const int m = m0 + row, n = n0 + c4 * 4;
        if (m >= P.p) continue;
        float* out = P.dW + (size_t)m * P.d + n;
        if (vec && n + 4 <= P.d) {
          if (P.accumulate) {
            const float4 old = *reinterpret_cast<const float4*>(out);
            sum.x += old.x; sum.y += old.y; sum.z += old.z; sum.w += old.w;
          }
          *reinterpret_cast<float4*>(out) = sum;
        } else {
          const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (n + q < P.d) out[q] = sv[q] + (P.accumulate ? out[q] : 0.f);
        }
      }
    }
  } else if (warp == 3 && do_bias) {
    const int t = threadIdx.x - 96;                  // 0..31
    const int cols_per = (BM + S - 1) / S;
    const int c0 = min(BM, (int)rank * cols_per), c1 = min(BM, c0 + cols_per);
    const uint32_t base = ptx::smem_u32(smem + PART_BYTES);
    for (int j = c0 + t; j < c1; j += 32) {
      float sum = 0.f;
      for (int sp = 0; sp < S; ++sp) sum += ptx::ld_cluster_f32(ptx::map_rank(base + 4u * j, sp));
      const int col = m0 + j;
      if (col >= P.p) continue;
      if (P.bias_nt > 1) P.bias_part[(size_t)blockIdx.y * P.p + col] = sum;
      else P.db[col] = sum + (P.accumulate ? P.db[col] : 0.f);
    }
  }
}

// Common tail, executed by every warp inside its own role branch (so each runs under
// its warpgroup's register budget): cluster reduction of the split partials, drain
// after an abort, TMEM release.  Every thread of every CTA passes the same barriers.
__device__ __forceinline__ void finish(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int m0, int n0,
                                       bool do_bias) {
  ptx::tc_fence_before();
  __syncthreads();
  if (P.splits > 1) {
    ptx::cluster_sync();                               // all partials staged
    if (c->flags[1]) cluster_reduce(P, smem, m0, n0, do_bias);
    ptx::cluster_sync();                               // peers are done reading
  }
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

template <bool kNorm, bool kTrim>
__global__ void __launch_bounds__(kThreads, 1)
tc_sumx_kernel(const __grid_constant__ CUtensorMap mapG64, const __grid_constant__ CUtensorMap mapA64,
               const __grid_constant__ CUtensorMap mapG16, const __grid_constant__ CUtensorMap mapA16,
               Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* c = reinterpret_cast<Ctl*>(smem + STAGES * STAGE);

  const int warp = threadIdx.x >> 5;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int e0 = blockIdx.z * P.ex_per_split;
  const int e1 = min(P.B, e0 + P.ex_per_split);
  // this CTA sums G rows for the bias (norm mode: the first column tile, every example;
  // sum mode: see bias_example)
  const bool do_bias = kNorm ? (P.norm_bias != 0 && blockIdx.y == 0)
                             : (P.db != nullptr && (int)blockIdx.y < P.bias_nt);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&c->full[s], 1);
      // norm mode: the MMA commit plus the eight epilogue warps when they sum G rows;
      // sum mode: the MMA commit, and bfree the eight warps for the stages they sum
      ptx::mbar_init(&c->empty[s], kNorm && do_bias ? 1 + kEpiWarps : 1);
      ptx::mbar_init(&c->bfree[s], kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&c->accum[b], 1);
      ptx::mbar_init(&c->tfree[b], kEpiWarps);
    }
    ptx::mbar_init(&c->drain, 1);
    c->abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mapG64);
    ptx::prefetch_tensormap(&mapA64);
    ptx::prefetch_tensormap(&mapG16);
    ptx::prefetch_tensormap(&mapA16);
  }
  if (warp == 1) ptx::tmem_alloc(&c->tmem, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c->tmem;
  pdl_trigger();   // the next kernel in the stream may start launching
  // With P.early, A and G (the caller's inputs, which no library kernel writes) are loaded
  // and multiplied before the previous kernel in the stream has completed: the factors,
  // the outputs and the workspace are touched after pdl_wait, which every warp passes
  // before its first such access.  Otherwise every warp waits here.
  if (!P.early) pdl_wait();

  if (warp >= kEpiFirst) {
    pdl_wait();
    ptx::regs_inc<216>();
    if constexpr (kNorm)
      epilogue_norm<kTrim>(P, smem, c, tmem, e0, e1, do_bias);
    else
      epilogue<kTrim>(P, smem, c, tmem, e0, e1, m0, n0, do_bias);
    finish(P, smem, c, tmem, m0, n0, do_bias);
  } else {
    ptx::regs_dec<64>();
    if (warp == 0 || warp == 2) {
      producer<kNorm, kTrim>(P, &mapG64, &mapA64, &mapG16, &mapA16, smem, c, e0, e1, m0, n0, warp >> 1);
    } else if (warp == 1) {
      mma_issuer<kTrim>(P, smem, c, tmem, e0, e1);
    } else {
      if (!kNorm && kPrefetch > 0) prefetcher<kTrim>(P, &mapG64, &mapA64, &mapG16, &mapA16, c, e0, e1, m0, n0);
      pdl_wait();
      finish_decision(c);        // warp 3 joins the workers' barrier
    }
    pdl_wait();
    finish(P, smem, c, tmem, m0, n0, do_bias);
  }
}

}  // namespace tcsumx
}  // namespace dpk

namespace dph {
using namespace dpk;

static int cdiv_x(long a, long b) { return (int)((a + b - 1) / b); }

// Clusters of `size` CTAs of this kernel that the current device runs at once (one
// CTA per SM; a cluster must fit in one GPC, so large clusters strand SMs).
static int active_clusters(int size) {
  static int cache[64][9] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || size < 1 || size > 8) return 0;
  if (!cache[dev][size]) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, size);
    cfg.blockDim = dim3(tcsumx::kThreads);
    cfg.dynamicSmemBytes = tcsumx::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = size;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, tcsumx::tc_sumx_kernel<false, false>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152 / size;   // planning fallback: the full SM count
    }
    cache[dev][size] = n;
  }
  return cache[dev][size];
}

// Clusters larger than 4 CTAs were measured to start over ~20 us on GB300 (18
// clusters of 8), against ~0.1 us for clusters of 2.
constexpr long kMaxCluster = 4;

// Examples are split over a cluster of S <= kMaxCluster CTAs per output tile: the
// largest S whose clusters for every tile run in one wave (at least 1).  The planning-only
// variant (no device) assumes 152 SMs in clusters of any size.
static void tc_sumx_split(const Geom& g, int* splits, int* ex_per_split, bool query_device) {
  const long tiles = (long)cdiv_x(g.p, tcsumx::BM) * cdiv_x(g.D, tcsumx::BN);
  long s = 1;
  for (long c = std::min<long>(kMaxCluster, g.B); c >= 2; --c) {
    const long fit = query_device ? (long)active_clusters((int)c) : 152 / c;
    if (tiles <= fit) { s = c; break; }
  }
  const int eps = cdiv_x(g.B, s);
  *ex_per_split = eps;
  *splits = cdiv_x(g.B, eps);
}

// When clusters of <= 4 CTAs per tile cannot give the GPU ~120 CTAs, the examples are
// split over the grid instead (no cluster): about one CTA per SM, each writing a
// partial tile to the workspace, summed in split order by a second kernel.
static int tc_sumx_grid_splits(const Geom& g) {
  const long tiles = (long)cdiv_x(g.p, tcsumx::BM) * cdiv_x(g.D, tcsumx::BN);
  if (tiles * kMaxCluster >= 120) return 0;
  const long s = std::min<long>(g.B, 152 / tiles);
  if (s <= kMaxCluster) return 0;
  const int eps = cdiv_x(g.B, s);
  return cdiv_x(g.B, eps);
}

bool tc_sumx_supported(const Geom& g) {
  return !g.conv && (g.p % 8 == 0) && (g.D % 8 == 0) && g.p >= 8 && g.D >= 8 && g.T >= 64;
}

// Column tiles that share the bias (Params::bias_nt).  The CTAs that sum G rows for the
// bias read 16 KB more of shared memory per stage than the others, and shared-memory
// bandwidth is what bounds this kernel (about a quarter more time on the ViT-Base MLP
// layers when one column tile summed every example), so with examples split over
// clusters and enough of them (B >= 256: at least 64 per CTA) every column tile sums its
// share, at the cost of a reduction of bias_nt partial vectors after the kernel.
static int tc_sumx_bias_nt(const Geom& g) {
  const int ntn = cdiv_x(g.D, tcsumx::BN);
  return (g.has_bias && !tc_sumx_grid_splits(g) && ntn > 1 && g.B >= 256) ? ntn : 1;
}

size_t tc_sumx_ws_bytes(const Geom& g) {
  const int gs = tc_sumx_grid_splits(g);
  if (gs) return (size_t)gs * ((size_t)g.p * g.D + g.p) * sizeof(float);
  const int bnt = tc_sumx_bias_nt(g);
  return bnt > 1 ? (size_t)bnt * g.p * sizeof(float) : 0;
}

cudaError_t launch_tc_sumx(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                           float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s, NoiseArgs* nz,
                           bool early) {
  CUtensorMap mg64, ma64, mg16, ma16;
  const uint64_t dg[3] = {(uint64_t)g.p, (uint64_t)g.T, (uint64_t)g.B};
  const uint64_t sg[2] = {(uint64_t)g.p * 2, (uint64_t)g.T * g.p * 2};
  const uint64_t da[3] = {(uint64_t)g.D, (uint64_t)g.T, (uint64_t)g.B};
  const uint64_t sa[2] = {(uint64_t)g.D * 2, (uint64_t)g.T * g.D * 2};
  const uint32_t box64[3] = {64, (uint32_t)tcsumx::FR, 1}, box16[3] = {64, 16, 1};
  if (!encode_tmap_bf16(&mg64, G, 3, dg, sg, box64) || !encode_tmap_bf16(&ma64, A, 3, da, sa, box64) ||
      !encode_tmap_bf16(&mg16, G, 3, dg, sg, box16) || !encode_tmap_bf16(&ma16, A, 3, da, sa, box16))
    return cudaErrorInvalidValue;
  int splits, eps;
  const int gsplits = tc_sumx_grid_splits(g);
  if (gsplits && !ws) return cudaErrorInvalidValue;
  if (gsplits) {
    eps = cdiv_x(g.B, gsplits);
    splits = 1;
  } else {
    tc_sumx_split(g, &splits, &eps, true);
  }
  float* part_w = static_cast<float*>(ws);
  float* part_b = (gsplits && db) ? part_w + (size_t)gsplits * g.p * g.D : nullptr;
  tcsumx::Params P = {};
  P.factors = factors;
  P.dW = gsplits ? part_w : dW;
  P.db = gsplits ? part_b : db;
  P.status = status;
  P.B = g.B;
  P.T = g.T;
  P.p = g.p;
  P.d = g.D;
  P.ex_per_split = eps;
  P.splits = splits;
  P.accumulate = accumulate;
  P.gsplit = gsplits ? 1 : 0;
  const int bias_nt = db ? tc_sumx_bias_nt(g) : 1;
  if (bias_nt > 1 && !ws) return cudaErrorInvalidValue;
  P.bias_nt = bias_nt;
  P.bias_part = bias_nt > 1 ? static_cast<float*>(ws) : nullptr;
  P.early = early ? 1 : 0;
  int nfull = g.T / tcsumx::FR, rem = g.T - tcsumx::FR * nfull;
  int n16 = (rem + 15) / 16;
  if (n16 > tcsumx::FR / 16 - 1) { nfull += 1; n16 = 0; }
  P.nfull = nfull;
  P.n16 = n16;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcsumx::tc_sumx_kernel<false, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, tcsumx::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tcsumx::tc_sumx_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tcsumx::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cdiv_x(g.p, tcsumx::BM), cdiv_x(g.D, tcsumx::BN), gsplits ? gsplits : splits);
  cfg.blockDim = dim3(tcsumx::kThreads);
  cfg.dynamicSmemBytes = tcsumx::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = splits;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  cudaError_t e = g.D % tcsumx::BN
                      ? cudaLaunchKernelEx(&cfg, tcsumx::tc_sumx_kernel<false, true>, mg64, ma64, mg16, ma16, P)
                      : cudaLaunchKernelEx(&cfg, tcsumx::tc_sumx_kernel<false, false>, mg64, ma64, mg16, ma16, P);
  count_launch();
  if (e == cudaSuccess && bias_nt > 1) {   // the column tiles' partial biases, in order
    e = launch_reduce_splits(P.bias_part, bias_nt, (size_t)g.p, db, accumulate, s, nz, nz ? nz->off_b : 0);
    if (nz && nz->on) nz->applied_b = 1;
  }
  if (e != cudaSuccess || !gsplits) return e;
  const size_t nw = (size_t)g.p * g.D;
  return launch_reduce_splits2(SplitSeg{part_w, nw, nw, dW}, SplitSeg{part_b, (size_t)g.p, db ? (size_t)g.p : 0, db},
                               gsplits, accumulate, s, nz);
}

// Instantiated norm on the tensor cores: per-tile partials [tiles, B] in the workspace,
// then a fixed-order sum over the tiles.  The examples are split over the grid so the
// CTAs cover the SMs about once.
size_t tc_inst_ws_bytes(const Geom& g) {
  const size_t tiles = (size_t)cdiv_x(g.p, tcsumx::BM) * cdiv_x(g.D, tcsumx::BN);
  return tiles * (size_t)g.B * sizeof(float);
}

cudaError_t launch_tc_inst(const Geom& g, const void* A, const void* G, float* out, float* ws,
                           unsigned* status, cudaStream_t s, float* keep, float* keep_b, bool early) {
  CUtensorMap mg64, ma64, mg16, ma16;
  const uint64_t dg[3] = {(uint64_t)g.p, (uint64_t)g.T, (uint64_t)g.B};
  const uint64_t sg[2] = {(uint64_t)g.p * 2, (uint64_t)g.T * g.p * 2};
  const uint64_t da[3] = {(uint64_t)g.D, (uint64_t)g.T, (uint64_t)g.B};
  const uint64_t sa[2] = {(uint64_t)g.D * 2, (uint64_t)g.T * g.D * 2};
  const uint32_t box64[3] = {64, (uint32_t)tcsumx::FR, 1}, box16[3] = {64, 16, 1};
  if (!encode_tmap_bf16(&mg64, G, 3, dg, sg, box64) || !encode_tmap_bf16(&ma64, A, 3, da, sa, box64) ||
      !encode_tmap_bf16(&mg16, G, 3, dg, sg, box16) || !encode_tmap_bf16(&ma16, A, 3, da, sa, box16))
    return cudaErrorInvalidValue;
  const int tm = cdiv_x(g.p, tcsumx::BM), tn = cdiv_x(g.D, tcsumx::BN);
  const long tiles = (long)tm * tn;
  long chunks = std::max<long>(1, std::min<long>(g.B, 152 / tiles));
  const int eps = cdiv_x(g.B, chunks);
  chunks = cdiv_x(g.B, eps);
  tcsumx::Params P = {};
  P.early = early ? 1 : 0;
  P.status = status;
  P.B = g.B;
  P.T = g.T;
  P.p = g.p;
  P.d = g.D;
  P.ex_per_split = eps;
  P.splits = 1;
  int nfull = g.T / tcsumx::FR, rem = g.T - tcsumx::FR * nfull;
  int n16 = (rem + 15) / 16;
  if (n16 > tcsumx::FR / 16 - 1) { nfull += 1; n16 = 0; }
  P.nfull = nfull;
  P.n16 = n16;
  P.part = ws;
  P.norm_bias = g.has_bias;
  P.keep = keep;
  P.keep_b = g.has_bias ? keep_b : nullptr;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcsumx::tc_sumx_kernel<true, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, tcsumx::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tcsumx::tc_sumx_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tcsumx::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dim3 grid(tm, tn, (unsigned)chunks);
  if (g.D % tcsumx::BN)
    launch_pdl(tcsumx::tc_sumx_kernel<true, true>, grid, tcsumx::kThreads, tcsumx::SMEM, s, mg64, ma64, mg16, ma16, P);
  else
    launch_pdl(tcsumx::tc_sumx_kernel<true, false>, grid, tcsumx::kThreads, tcsumx::SMEM, s, mg64, ma64, mg16, ma16,
               P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_reduce_splits(ws, (int)tiles, (size_t)g.B, out, 0, s);
}

}  // namespace dph
