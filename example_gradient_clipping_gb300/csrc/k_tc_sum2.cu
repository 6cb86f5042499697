// Clipped sum with the clip factor applied per example in fp32, on CTA pairs.
//
//   dW = sum_i c_i P_i,  P_i = G_i^T A_i  (the per-example gradient of [MixGhost] eq. 2.4),
//   db = sum_i c_i sum_t G_i[t, :]
//
// The same per-example reweighted contraction as the single-CTA kernel (k_tc_sumx.cu),
// with one 256 x 256 output tile per cluster of two CTAs on two SMs: the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256), whose rows [128r, 128r+128) come from CTA r's
// slice of G (its 128 outputs) and whose columns come half from each CTA's slice of A.
// Each SM therefore receives 32 KB per 64-row stage for a 128 x 256 product instead of
// 48 KB (TMA delivery into the SM, not the tensor cores, bounds the single-CTA kernel).
// Measured on GB300 it is nevertheless 1.4-1.5x slower than the single-CTA kernel on the
// sequence (768 x 768) and ViT MLP (768 x 3072) layers: its stages land every ~0.85 us
// instead of ~0.47 us, and ncu counts 1.4x the L2 sector requests for 2/3 of the bytes
// delivered (the single-CTA kernel's CTAs that share an operand box request it in step,
// ~1.5 bytes delivered per byte requested).  The library takes it only when pinned
// (DPCLIP_SUM_KERNEL=pair).
//
// Synchronisation of the pair:
//   full[s]   (each CTA)   its own TMA bytes of stage s
//   pfull[s]  (even CTA)   the odd CTA's stage s has landed (warp 1 of the odd CTA waits
//                          on its own full[s] and arrives here remotely)
//   empty[s]  (each CTA)   stage s consumed: the even CTA's MMA commit is multicast to
//                          both CTAs (plus, in the first column tile, the eight epilogue
//                          warps that sum the G rows for the bias)
//   accum[b]  (each CTA)   TMEM buffer b holds P_e: multicast commit
//   tfree[b]  (even CTA)   both CTAs' epilogues drained buffer b (16 warp arrivals)
// Waits on the barriers that other-CTA arrivals complete (pfull, tfree, and empty / accum,
// which the multicast commits complete) poll without suspending the thread.
// Cluster barriers after the barrier set-up and before the TMEM release keep every remote
// arrival and every MMA read of the peer's shared memory inside both CTAs' lifetimes.
// Examples are split over the grid: with several splits each CTA writes a partial tile,
// summed afterwards in split order; with one split it writes (or adds to) dW directly.
//   warps 0, 2: TMA producers (alternate stages); warp 1: MMA issuer (even CTA) or
//   forwarder (odd CTA); warp 3: joins the workers' barrier; warps 4-11: epilogue.
#include <algorithm>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tcsum2 {

constexpr int BM = 128, BN = 256, STAGES = 6;
constexpr int BOX = 64 * 64 * 2;             // 64 rows x 128 B
constexpr int STAGE = 4 * BOX;               // G: 2 boxes (this CTA's 128 outputs), A: 2 boxes
constexpr int kEpiWarps = 8;
constexpr int kThreads = 384;
constexpr int kEpiFirst = 4;
constexpr int kSyncThreads = 32 * (1 + kEpiWarps);   // warps 3-11, named barrier 1
constexpr int kLeader = 96;
constexpr int SMEM = STAGES * STAGE + 1024 + 512;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(2 * BM, BN, 1, 1);
constexpr int PSTR = BN + 4;
constexpr int PART_BYTES = BM * PSTR * 4;
static_assert(PART_BYTES <= STAGES * STAGE, "staging fits in the stage buffers");

struct Params {
  const float* factors;
  float* dW;
  float* db;          // null: no bias
  unsigned* status;
  int B, T, p, d;
  int ex_per_split, accumulate;
  int nfull, n16;     // per example: 64-row stages, then 16-row stages
  int gsplit;         // several grid splits: CTA z writes its partial tile to dW + z*p*d
                      // (db + z*p), summed afterwards in z order
};

struct Ctl {
  uint64_t full[STAGES], pfull[STAGES], empty[STAGES], accum[2], tfree[2], drain;
  uint32_t tmem;
  int abort;
  int flags[2];
};

__device__ __forceinline__ void sync_workers() {
  asm volatile("bar.sync 1, %0;" ::"r"(kSyncThreads) : "memory");
}

__device__ __forceinline__ bool finish_decision(Ctl* c) {
  sync_workers();
  if (threadIdx.x == kLeader) c->flags[1] = *(volatile int*)&c->abort ? 0 : 1;
  sync_workers();
  return c->flags[1] != 0;
}

// Warps 0 and 2: stage k (k % 2 == pr) = this CTA's 128 outputs of G and its half of the
// pair's A columns, rows [y, y + 64) (or 16) of example e.
__device__ __forceinline__ void producer(const Params& P, const CUtensorMap* mG64, const CUtensorMap* mA64,
                                         const CUtensorMap* mG16, const CUtensorMap* mA16, uint8_t* smem,
                                         Ctl* c, int e0, int e1, int m0, int na, int pr) {
  volatile int* abort = &c->abort;
  const int ns = P.nfull + P.n16;
  int k = 0, last = -1;
  bool live = true;
  for (int e = e0; e < e1 && live; ++e) {
    for (int u = 0; u < ns; ++u, ++k) {
      if ((k & 1) != pr) continue;
      const int s = k % STAGES;
      const bool w = ptx::mbar_wait_cluster(&c->empty[s], ((k / STAGES) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      const bool big = u < P.nfull;
      const int y = big ? u * 64 : P.nfull * 64 + (u - P.nfull) * 16;
      const CUtensorMap* mg = big ? mG64 : mG16;
      const CUtensorMap* ma = big ? mA64 : mA16;
      uint8_t* st = smem + s * STAGE;
      if (ptx::elect_one()) {
        ptx::mbar_arrive_expect_tx(&c->full[s], (big ? 64 : 16) * 128 * 4);
        ptx::tma_load_3d(mg, &c->full[s], st, m0, y, e);
        ptx::tma_load_3d(mg, &c->full[s], st + BOX, m0 + 64, y, e);
        ptx::tma_load_3d(ma, &c->full[s], st + 2 * BOX, na, y, e);
        ptx::tma_load_3d(ma, &c->full[s], st + 3 * BOX, na + 64, y, e);
      }
      __syncwarp();
      last = k;
    }
  }
  if (*abort && (threadIdx.x & 31) == 0) {   // let this producer's copies in flight land
    for (int q = max(0, last - STAGES + 1); q <= last; ++q)
      if ((q & 1) == pr) ptx::mbar_wait_drain(&c->full[q % STAGES], (q / STAGES) & 1);
  }
}

// Warp 1 of the odd CTA: tell the even CTA when each of this CTA's stages has landed.
__device__ __forceinline__ void forwarder(const Params& P, Ctl* c, int e0, int e1) {
  volatile int* abort = &c->abort;
  const int total = (e1 - e0) * (P.nfull + P.n16);
  for (int k = 0; k < total; ++k) {
    const int s = k % STAGES;
    const bool w = ptx::mbar_wait_cluster(&c->full[s], (k / STAGES) & 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) break;
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive_rank(&c->pfull[s], 0);
    __syncwarp();
  }
}

// Warp 1 of the even CTA: the pair MMAs.  Per example, P_e into TMEM buffer e % 2 of both
// CTAs once both epilogues released it.
__device__ __forceinline__ void mma_issuer(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0,
                                           int e1) {
  volatile int* abort = &c->abort;
  const int ns = P.nfull + P.n16;
  int k = 0;
  bool live = true;
  for (int e = e0; e < e1 && live; ++e) {
    const int x = e - e0, b = x & 1;
    if (x >= 2) {
      const bool w = ptx::mbar_wait_cluster(&c->tfree[b], ((x >> 1) & 1) ^ 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) break;
    }
    ptx::tc_fence_after();
    const uint32_t d_tmem = tmem + b * 256;
    for (int u = 0; u < ns; ++u, ++k) {
      const int s = k % STAGES;
      bool w = ptx::mbar_wait_cluster(&c->full[s], (k / STAGES) & 1, abort, P.status);
      w = w && ptx::mbar_wait_cluster(&c->pfull[s], (k / STAGES) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      const uint32_t g = ptx::smem_u32(smem + s * STAGE);
      // MN-major, 128-byte swizzle: 64-column chunks are BOX apart, 16 rows per MMA = 2 KB
      const uint64_t da = ptx::sdesc_sw128(g, BOX, 1024);
      const uint64_t dbd = ptx::sdesc_sw128(g + 2 * BOX, BOX, 1024);
      if (ptx::elect_one()) {
        if (u < P.nfull) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::umma_pair_bf16(d_tmem, ptx::sdesc_add(da, kk * 2048), ptx::sdesc_add(dbd, kk * 2048), kIdesc,
                                (u | kk) != 0);
        } else {
          ptx::umma_pair_bf16(d_tmem, da, dbd, kIdesc, u != 0);
        }
        ptx::umma_pair_commit_mc(&c->empty[s], 3);
      }
      __syncwarp();
    }
    if (live) {
      if (ptx::elect_one()) ptx::umma_pair_commit_mc(&c->accum[b], 3);
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

// Warps 4-11 of both CTAs: drain P_e from this CTA's TMEM into fp32 registers,
// D += c_e * P_e; in the first column tile also sum the G rows of every stage for the bias.
__device__ __forceinline__ void epilogue(const Params& P, uint8_t* smem, Ctl* c, uint32_t tmem, int e0,
                                         int e1, int m0, int n0, bool do_bias, uint32_t rank) {
  volatile int* abort = &c->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
  const int half = (warp - kEpiFirst) >> 2;      // columns 128*half .. +127
  const int et = threadIdx.x - 32 * kEpiFirst;   // 0..255
  const int bbox = et >> 7, bq = (et >> 4) & 7, bj = et & 15;
  const int ns = P.nfull + P.n16;
  float bacc[8], btmp[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) bacc[q] = btmp[q] = 0.f;
  float acc[128];
#pragma unroll
  for (int j = 0; j < 128; ++j) acc[j] = 0.f;
  bool ok = true;
  int k = 0;
  for (int e = e0; e < e1 && ok; ++e) {
    const int x = e - e0, b = x & 1;
    if (do_bias) {
      for (int u = 0; u < ns; ++u, ++k) {
        const int s = k % STAGES;
        const bool w = ptx::mbar_wait_cluster(&c->full[s], (k / STAGES) & 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        // 128-byte swizzle: chunk q of row r sits at chunk q ^ (r % 8)
        const uint8_t* gt = smem + s * STAGE + bbox * BOX + bj * 128 + ((bq ^ (bj & 7)) << 4);
        if (u < P.nfull) {
          uint4 v[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) v[h] = *reinterpret_cast<const uint4*>(gt + h * 16 * 128);
#pragma unroll
          for (int h = 0; h < 4; ++h) add_bf16x8(v[h], btmp);
        } else {
          add_bf16x8(*reinterpret_cast<const uint4*>(gt), btmp);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c->empty[s]);
      }
      if (!ok) break;
    }
    const bool w = ptx::mbar_wait_cluster(&c->accum[b], (x >> 1) & 1, abort, P.status);
    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
    ptx::tc_fence_after();
    const float cf = __ldg(P.factors + e);
    const uint32_t base = tmem + b * 256 + half * 128 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
    for (int ch = 0; ch < 8; ch += 4) {
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
    if (lane == 0) {
      if (rank == 0) ptx::mbar_arrive(&c->tfree[b]);
      else ptx::mbar_arrive_rank(&c->tfree[b], 0);
    }
    if (do_bias) {
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
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = bbox * 64 + bq * 8 + q;
      if (m0 + j >= P.p) continue;
      if (P.gsplit) P.db[(size_t)blockIdx.z * P.p + m0 + j] = bacc[q];
      else P.db[m0 + j] = bacc[q] + (P.accumulate ? P.db[m0 + j] : 0.f);
    }
  }
  // stage the tile in shared memory (every load was consumed and every MMA completed
  // before the last accum wait), then whole rows out, 64 threads per 1 KB row
  const int row = quarter * 32 + lane;
  {
    float* part = reinterpret_cast<float*>(smem) + row * PSTR + half * 128;
#pragma unroll
    for (int j = 0; j < 128; j += 4)
      *reinterpret_cast<float4*>(part + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
  }
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

// Common tail, inside each role branch: the even CTA drains its MMAs after an abort;
// a cluster barrier (every thread of both CTAs) precedes the pair TMEM release.
__device__ __forceinline__ void finish(Ctl* c, uint32_t tmem, uint32_t rank) {
  ptx::tc_fence_before();
  __syncthreads();
  if (*(volatile int*)&c->abort && rank == 0 && threadIdx.x == 32) {
    ptx::umma_pair_commit(&c->drain);   // arrives once every pair MMA issued so far has completed
    ptx::mbar_wait_drain(&c->drain, 0);
  }
  __syncthreads();
  ptx::cluster_sync();
  if ((threadIdx.x >> 5) == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_sum2_kernel(const __grid_constant__ CUtensorMap mapG64, const __grid_constant__ CUtensorMap mapA64,
               const __grid_constant__ CUtensorMap mapG16, const __grid_constant__ CUtensorMap mapA16,
               Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* c = reinterpret_cast<Ctl*>(smem + STAGES * STAGE);

  const int warp = threadIdx.x >> 5;
  const uint32_t rank = ptx::cluster_rank();              // cluster (2, 1, 1)
  const int m0 = (int)(blockIdx.x >> 1) * (2 * BM) + (int)rank * BM;   // this CTA's outputs
  const int n0 = blockIdx.y * BN;                          // the pair's columns
  const int na = n0 + (int)rank * (BN / 2);                // this CTA's half of them (A)
  const int e0 = blockIdx.z * P.ex_per_split;
  const int e1 = min(P.B, e0 + P.ex_per_split);
  const bool do_bias = P.db != nullptr && blockIdx.y == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&c->full[s], 1);
      ptx::mbar_init(&c->pfull[s], 1);
      ptx::mbar_init(&c->empty[s], do_bias ? 1 + kEpiWarps : 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&c->accum[b], 1);
      ptx::mbar_init(&c->tfree[b], 2 * kEpiWarps);
    }
    ptx::mbar_init(&c->drain, 1);
    c->abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mapG64);
    ptx::prefetch_tensormap(&mapA64);
    ptx::prefetch_tensormap(&mapG16);
    ptx::prefetch_tensormap(&mapA16);
  }
  ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrival or multicast commit
  if (warp == 1) ptx::tmem_alloc_pair(&c->tmem, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = c->tmem;
  pdl_trigger();   // the next kernel in the stream may start launching
  pdl_wait();      // the previous kernel has completed; its writes are visible

  if (warp >= kEpiFirst) {
    ptx::regs_inc<216>();
    epilogue(P, smem, c, tmem, e0, e1, m0, n0, do_bias, rank);
    finish(c, tmem, rank);
  } else {
    ptx::regs_dec<64>();
    if (warp == 0 || warp == 2) {
      producer(P, &mapG64, &mapA64, &mapG16, &mapA16, smem, c, e0, e1, m0, na, warp >> 1);
    } else if (warp == 1) {
      if (rank == 0) mma_issuer(P, smem, c, tmem, e0, e1);
      else forwarder(P, c, e0, e1);
    } else {
      finish_decision(c);        // warp 3 joins the workers' barrier
    }
    finish(c, tmem, rank);
  }
}

}  // namespace tcsum2
}  // namespace dpk

namespace dph {
using namespace dpk;

static int cdiv_p(long a, long b) { return (int)((a + b - 1) / b); }

bool tc_sum2_supported(const Geom& g) {
  return !g.conv && (g.p % 8 == 0) && (g.D % 8 == 0) && g.p > 128 && g.D > 128 && g.T >= 64;
}

// Examples split over the grid so the pairs cover the SMs about once.
static int tc_sum2_splits(const Geom& g) {
  const long ctas = 2L * cdiv_p(g.p, 2 * tcsum2::BM) * cdiv_p(g.D, tcsum2::BN);
  const long s = std::max<long>(1, std::min<long>(g.B, 152 / ctas));
  const int eps = cdiv_p(g.B, s);
  return cdiv_p(g.B, eps);
}

size_t tc_sum2_ws_bytes(const Geom& g) {
  const int s = tc_sum2_splits(g);
  return s > 1 ? (size_t)s * ((size_t)g.p * g.D + g.p) * sizeof(float) : 0;
}

cudaError_t launch_tc_sum2(const Geom& g, const void* A, const void* G, const float* factors, float* dW,
                           float* db, int accumulate, void* ws, unsigned* status, cudaStream_t s) {
  CUtensorMap mg64, ma64, mg16, ma16;
  const uint64_t dg[3] = {(uint64_t)g.p, (uint64_t)g.T, (uint64_t)g.B};
  const uint64_t sg[2] = {(uint64_t)g.p * 2, (uint64_t)g.T * g.p * 2};
  const uint64_t da[3] = {(uint64_t)g.D, (uint64_t)g.T, (uint64_t)g.B};
  const uint64_t sa[2] = {(uint64_t)g.D * 2, (uint64_t)g.T * g.D * 2};
  const uint32_t box64[3] = {64, 64, 1}, box16[3] = {64, 16, 1};
  if (!encode_tmap_bf16(&mg64, G, 3, dg, sg, box64) || !encode_tmap_bf16(&ma64, A, 3, da, sa, box64) ||
      !encode_tmap_bf16(&mg16, G, 3, dg, sg, box16) || !encode_tmap_bf16(&ma16, A, 3, da, sa, box16))
    return cudaErrorInvalidValue;
  const int splits = tc_sum2_splits(g);
  if (splits > 1 && !ws) return cudaErrorInvalidValue;
  const int eps = cdiv_p(g.B, splits);
  float* part_w = static_cast<float*>(ws);
  float* part_b = (splits > 1 && db) ? part_w + (size_t)splits * g.p * g.D : nullptr;
  tcsum2::Params P = {};
  P.factors = factors;
  P.dW = splits > 1 ? part_w : dW;
  P.db = splits > 1 ? part_b : db;
  P.status = status;
  P.B = g.B;
  P.T = g.T;
  P.p = g.p;
  P.d = g.D;
  P.ex_per_split = eps;
  P.accumulate = accumulate;
  P.gsplit = splits > 1 ? 1 : 0;
  int nfull = g.T / 64, rem = g.T - 64 * nfull;
  int n16 = (rem + 15) / 16;
  if (n16 > 3) { nfull += 1; n16 = 0; }
  P.nfull = nfull;
  P.n16 = n16;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcsum2::tc_sum2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tcsum2::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * cdiv_p(g.p, 2 * tcsum2::BM), cdiv_p(g.D, tcsum2::BN), splits);
  cfg.blockDim = dim3(tcsum2::kThreads);
  cfg.dynamicSmemBytes = tcsum2::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, tcsum2::tc_sum2_kernel, mg64, ma64, mg16, ma16, P);
  count_launch();
  if (e != cudaSuccess || splits <= 1) return e;
  const size_t nw = (size_t)g.p * g.D;
  return launch_reduce_splits2(SplitSeg{part_w, nw, nw, dW}, SplitSeg{part_b, (size_t)g.p, db ? (size_t)g.p : 0, db},
                               splits, accumulate, s);
}

}  // namespace dph
