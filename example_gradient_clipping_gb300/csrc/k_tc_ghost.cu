// Ghost norm on the 5th-generation tensor cores ([MixGhost] eq. 2.7, Appendix C.3):
//
//   s_i = sum_{t,s} (A_i A_i^T)_{ts} (G_i G_i^T)_{ts} + has_bias * sum_{t,s} (G_i G_i^T)_{ts}
//
// The second term is ||sum_t g_t||^2, the bias gradient's squared norm.  One CTA per
// example.  Rows are cut into 128-row blocks; for each block pair (tb <= sb) both
// Gram tiles are accumulated in TMEM (two 128-column fp32 tiles), then read back
// to form the Hadamard sum, weighted 2 off the diagonal (both Grams are symmetric).
// TMEM holds two such pairs, so the epilogue of one pair overlaps the MMAs of the
// next.  Operands are K-major (rows of A and G are contiguous), loaded by 3D TMA
// boxes [1, 128 rows, 64 columns] whose rows past T read as zero, into a ring of
// eight 16 KB slots: a diagonal block pair takes one slot per K step (the tile is
// both operands), an off-diagonal pair two.
//   warps 0 and 6: TMA producers (alternate slots: one issuing thread streams only
//   ~48 B/clk into an SM); warp 1: MMA issuer; warps 2-5: epilogue.
// Dual mode (two row blocks, 128 < T <= 256): the Grams of the wider operand X (A or G)
// are formed first, all three block pairs at once from the two row blocks loaded per K
// step (TMEM columns 0..383), then the narrower operand Y pair by pair into columns
// 384..511; after each Y pair the epilogue forms that pair's Hadamard sum.  The wider
// operand's rows are loaded once instead of once per pair.  The second row block holds
// T - 128 rows: (linear layers) its loads cover only r1 = T - 128 rounded up to 16 rows and
// the MMAs that take it as B run at N = r1, so the Gram tiles with block 1 on the B side have
// r1 written columns and the (1, 1) tiles r1 rows with data (the rest of block 1's slot is
// stale); the epilogue reads only those (the entries it skips are zero in the full tiles).
// Dual-mode CTAs are persistent (at most one per SM, examples blockIdx.x + n * gridDim.x): the
// producers stream the next example's tiles while the current one's last pairs are reduced,
// and its X Grams start once the epilogue has read the previous example's last Y pair.
// Packed mode (2T <= 128): one CTA takes ept = 128 / T examples whose rows are
// consecutive in memory (2D boxes over the flattened rows), so one Gram tile holds
// every example's Gram as a diagonal block; the epilogue adds only entries (r, s) of
// the same example, row by row, then sums each example's T rows in a fixed order.
// K splits (single row block or packed, fewer CTAs than SMs): the A-Gram is linear in its
// K chunks, so CTA y of a cluster of ksplit forms the A-Gram over its share of the unfolded
// columns, the whole G-Gram, and its part of the Hadamard sum (rank 0 adds the bias term);
// the parts go to rank 0's shared memory and rank 0 sums them in rank order after a
// cluster barrier (no second kernel).
#include <algorithm>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace dpk {
namespace tcghost {

constexpr int BT = 128, BK = 64, STAGES = 8;
constexpr int TILE = BT * BK * 2;   // 16 KB
constexpr int STAGE = TILE;         // one tile per slot
constexpr int kThreads = 224;
constexpr int MAXSPLIT = 8;         // K splits: one cluster (portable size)
constexpr int SMEM = STAGES * STAGE + 1024 + 2048 + MAXSPLIT * BT * 4 + 64;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(BT, BT, 0, 0);

struct Params {
  float* out;
  unsigned* status;
  int T, d, p, has_bias;
  int B, ept;          // packed mode: examples per CTA (0: one CTA per example)
  // conv layers: mapA is a TMA im2col map over an NHWC copy of the input, and K
  // chunk q of the unfolded rows is channel block q / (k*k), filter tap q % (k*k)
  int conv, Wout, k, stride, pad, dil;
  int early;           // A and G are the caller's inputs: loads may start before pdl_wait
  int ksplit;          // splits of the A-Gram's K chunks (grid y, one cluster of ksplit CTAs)
  int r1;              // dual mode: rows loaded for the second row block (16 .. 128, a multiple of 16)
};

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Load K chunk kk (64 unfolded columns) of the 128 rows that start at row t0 of
// example e: a tiled box, or for conv layers an im2col block of one filter tap.
__device__ __forceinline__ void load_a_rows(const Params& P, const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int kk, int t0, int e, bool flat_rows) {
  if (P.conv) {
    const int taps = P.k * P.k, cc = kk / taps, tap = kk - cc * taps;
    const int kh = tap / P.k, kw = tap - kh * P.k;
    const int ho = t0 / P.Wout, wo = t0 - ho * P.Wout;
    ptx::tma_load_im2col_4d(map, bar, dst, cc * 64, wo * P.stride - P.pad, ho * P.stride - P.pad, e,
                            (uint16_t)(kw * P.dil), (uint16_t)(kh * P.dil));
  } else if (flat_rows) {
    ptx::tma_load_2d(map, bar, dst, kk * BK, e * P.T + t0);
  } else {
    ptx::tma_load_3d(map, bar, dst, kk * BK, t0, e);
  }
}

__device__ __forceinline__ void pair_of(int j, int nb, int& tb, int& sb) {
  tb = 0;
  while (j >= nb - tb) { j -= nb - tb; ++tb; }
  sb = tb + j;
}

__global__ void __launch_bounds__(kThreads, 1)
tc_ghost_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapG,
                const __grid_constant__ CUtensorMap mapA1, const __grid_constant__ CUtensorMap mapG1, Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;       // [2]
  uint64_t* tfree = accum + 2;            // [2]
  uint64_t* drainb = tfree + 2;           // MMAs in flight at an abort
  uint64_t* ydone = drainb + 1;           // dual mode: a Y pair's Gram (and all X Grams) complete
  uint64_t* yfree = ydone + 1;            // dual mode: the epilogue has read the Y Gram
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(yfree + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 2);   // [8] (dual mode: [2][8])
  float* rowbuf = red + 8;                                 // packed mode: [2][BT] per-row sums
  float* csum = rowbuf + 2 * BT;                           // K splits (rank 0): [split][example]
  uint32_t* cabort = reinterpret_cast<uint32_t*>(csum + MAXSPLIT * BT);   // [split] aborted

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x;
  const bool packed = P.ept > 0;
  const int nb = packed ? 1 : (P.T + BT - 1) / BT;
  const int npairs = nb * (nb + 1) / 2;
  const int kA = (P.d + BK - 1) / BK, kG = (P.p + BK - 1) / BK;
  const bool dual = !packed && nb == 2;
  const bool x_is_g = kG >= kA;                 // dual: the wider operand goes first
  const int kX = x_is_g ? kG : kA, kY = x_is_g ? kA : kG;
  // this split's A chunks [ka0, ka1) (all of them without K splits)
  const int split = blockIdx.y;   // = the cluster rank with K splits
  const int ka0 = (int)((long)kA * split / P.ksplit), ka1 = (int)((long)kA * (split + 1) / P.ksplit);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&accum[b], 1);
      ptx::mbar_init(&tfree[b], 4);
    }
    ptx::mbar_init(drainb, 1);
    ptx::mbar_init(ydone, 1);
    ptx::mbar_init(yfree, 4);
    *abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&mapA);
    ptx::prefetch_tensormap(&mapG);
    if (P.r1 < BT) {
      ptx::prefetch_tensormap(&mapA1);
      ptx::prefetch_tensormap(&mapG1);
    }
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();   // the next kernel in the stream may start launching
  // With P.early, A and G (the caller's inputs, which no library kernel writes) are loaded
  // and multiplied before the previous kernel in the stream has completed; the epilogue
  // warps pass pdl_wait before they write.  Otherwise every warp waits here.
  if (!P.early) pdl_wait();

  if (warp == 0 || warp == 6) {
    // TMA producers (whole warp; the elected lane issues); producer pr loads slots k % 2 == pr
    const int pr = warp == 6 ? 1 : 0;
    int k = 0, issued = 0, last = -1;
    bool live = true;
    // dual mode: the CTA's examples one after another (ex = blockIdx.x, += gridDim.x)
    for (int ex = i; dual && ex < P.B && live; ex += gridDim.x) {
      // X: both row blocks per K step; then Y: pairs (0,0), (0,1), (1,1)
      const int nunits = 2 * kX + 4 * kY;
      for (int u = 0; u < nunits && live; ++u, ++k) {
        if ((k & 1) != pr) continue;
        const int s = k % STAGES;
        const bool w = ptx::mbar_wait(&empty[s], ((k / STAGES) & 1) ^ 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { live = false; break; }
        bool is_a;
        int kk, blk;
        if (u < 2 * kX) {
          kk = u >> 1;
          blk = u & 1;
          is_a = !x_is_g;
        } else {
          const int v = u - 2 * kX;       // pair 0: kY units, pair 1: 2 kY, pair 2: kY
          if (v < kY) { kk = v; blk = 0; }
          else if (v < 3 * kY) { kk = (v - kY) >> 1; blk = (v - kY) & 1; }
          else { kk = v - 3 * kY; blk = 1; }
          is_a = x_is_g;
        }
        if (ptx::elect_one()) {
          // block 1: its r1 rows (maps with r1-row boxes) unless it takes whole tiles
          const bool cut = blk == 1 && P.r1 < BT;
          ptx::mbar_arrive_expect_tx(&full[s], cut ? (uint32_t)P.r1 * BK * 2 : (uint32_t)TILE);
          if (is_a)
            load_a_rows(P, cut ? &mapA1 : &mapA, &full[s], smem + s * STAGE, kk, blk * BT, ex, false);
          else
            ptx::tma_load_3d(cut ? &mapG1 : &mapG, &full[s], smem + s * STAGE, kk * BK, blk * BT, ex);
        }
        __syncwarp();
        ++issued;
        last = k;
      }
    }
    for (int j = 0; j < npairs && live && !dual; ++j) {
      int tb, sb;
      pair_of(j, nb, tb, sb);
      const bool diag = tb == sb;
      for (int ph = 0; ph < 2 && live; ++ph) {
        const CUtensorMap* map = ph == 0 ? &mapA : &mapG;
        const int k_lo = ph == 0 ? ka0 : 0, k_hi = ph == 0 ? ka1 : kG;
        for (int kk = k_lo; kk < k_hi; ++kk) {
          for (int h = 0; h < (diag ? 1 : 2); ++h, ++k) {
            if ((k & 1) != pr) continue;
            const int s = k % STAGES;
            const bool w = ptx::mbar_wait(&empty[s], ((k / STAGES) & 1) ^ 1, abort, P.status);
            if (!__all_sync(0xffffffffu, w)) { live = false; break; }
            if (ptx::elect_one()) {
              ptx::mbar_arrive_expect_tx(&full[s], TILE);
              const int e = packed ? i * P.ept : i, t0 = packed ? 0 : (h ? sb : tb) * BT;
              if (ph == 0)
                load_a_rows(P, map, &full[s], smem + s * STAGE, kk, t0, e, packed);
              else if (packed)
                ptx::tma_load_2d(map, &full[s], smem + s * STAGE, kk * BK, e * P.T);
              else
                ptx::tma_load_3d(map, &full[s], smem + s * STAGE, kk * BK, t0, e);
            }
            __syncwarp();
            ++issued;
            last = k;
          }
          if (!live) break;
        }
      }
    }
    if (*abort && lane == 0) {   // let this producer's copies in flight land
      for (int q = max(0, last - STAGES + 1); q <= last; ++q)
        if ((q & 1) == pr) ptx::mbar_wait_drain(&full[q % STAGES], (q / STAGES) & 1);
    }
    (void)issued;
  } else if (warp == 1) {
    // MMA issuer (whole warp; the elected lane issues)
    int k = 0;
    bool live = true;
    const uint32_t idesc1 = ptx::idesc_bf16_f32(BT, P.r1, 0, 0);   // B = row block 1: N = r1
    int qq = 0;                                                     // Y pairs issued so far
    for (int ex = i; dual && ex < P.B && live; ex += gridDim.x) {
      // a later example's Grams overwrite TMEM once the epilogue has read the last Y pair
      if (qq > 0) {
        const bool w = ptx::mbar_wait(yfree, (qq - 1) & 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { live = false; break; }
      }
      ptx::tc_fence_after();
      // X Grams: (X0,X0) -> cols 0, (X0,X1) -> 128, (X1,X1) -> 256
      for (int kk = 0; kk < kX && live; ++kk, k += 2) {
        const int s0 = k % STAGES, s1 = (k + 1) % STAGES;
        bool w = ptx::mbar_wait(&full[s0], (k / STAGES) & 1, abort, P.status);
        w = w && ptx::mbar_wait(&full[s1], ((k + 1) / STAGES) & 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { live = false; break; }
        const uint64_t d0 = ptx::sdesc_sw128(ptx::smem_u32(smem + s0 * STAGE), 16, 1024);
        const uint64_t d1 = ptx::sdesc_sw128(ptx::smem_u32(smem + s1 * STAGE), 16, 1024);
        if (ptx::elect_one()) {
#pragma unroll
          for (int u = 0; u < BK / 16; ++u) {
            const uint64_t a0 = ptx::sdesc_add(d0, u * 32), a1 = ptx::sdesc_add(d1, u * 32);
            ptx::umma_bf16(tmem, a0, a0, kIdesc, (kk | u) != 0);
            ptx::umma_bf16(tmem + 128, a0, a1, idesc1, (kk | u) != 0);
            ptx::umma_bf16(tmem + 256, a1, a1, idesc1, (kk | u) != 0);
          }
          ptx::umma_commit(&empty[s0]);
          ptx::umma_commit(&empty[s1]);
        }
        __syncwarp();
      }
      // Y Gram of each pair into cols 384, after the epilogue read the previous one
      for (int q = 0; q < 3 && live; ++q, ++qq) {
        if (q > 0) {
          const bool w = ptx::mbar_wait(yfree, (qq - 1) & 1, abort, P.status);
          if (!__all_sync(0xffffffffu, w)) { live = false; break; }
          ptx::tc_fence_after();
        }
        const bool diag = q != 1;
        for (int kk = 0; kk < kY; ++kk) {
          const int s0 = k % STAGES, s1 = (k + 1) % STAGES;
          bool w = ptx::mbar_wait(&full[s0], (k / STAGES) & 1, abort, P.status);
          if (!diag) w = w && ptx::mbar_wait(&full[s1], ((k + 1) / STAGES) & 1, abort, P.status);
          if (!__all_sync(0xffffffffu, w)) { live = false; break; }
          const uint64_t da = ptx::sdesc_sw128(ptx::smem_u32(smem + s0 * STAGE), 16, 1024);
          const uint64_t db = diag ? da : ptx::sdesc_sw128(ptx::smem_u32(smem + s1 * STAGE), 16, 1024);
          if (ptx::elect_one()) {
#pragma unroll
            for (int u = 0; u < BK / 16; ++u)
              ptx::umma_bf16(tmem + 384, ptx::sdesc_add(da, u * 32), ptx::sdesc_add(db, u * 32),
                             q == 0 ? kIdesc : idesc1, (kk | u) != 0);
            ptx::umma_commit(&empty[s0]);
            if (!diag) ptx::umma_commit(&empty[s1]);
          }
          __syncwarp();
          k += diag ? 1 : 2;
        }
        if (live) {
          if (ptx::elect_one()) ptx::umma_commit(ydone);
          __syncwarp();
        }
      }
    }
    for (int j = 0; j < npairs && live && !dual; ++j) {
      int tb, sb;
      pair_of(j, nb, tb, sb);
      const bool diag = tb == sb;
      const int b = j & 1;
      if (j >= 2) {
        const bool w = ptx::mbar_wait(&tfree[b], ((j >> 1) & 1) ^ 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) break;
      }
      ptx::tc_fence_after();
      for (int ph = 0; ph < 2 && live; ++ph) {
        const int k_lo = ph == 0 ? ka0 : 0, k_hi = ph == 0 ? ka1 : kG;
        const uint32_t d_tmem = tmem + b * 256 + ph * 128;
        for (int kk = k_lo; kk < k_hi; ++kk) {
          const int s0 = k % STAGES, s1 = (k + 1) % STAGES;
          bool w = ptx::mbar_wait(&full[s0], (k / STAGES) & 1, abort, P.status);
          if (!diag) w = w && ptx::mbar_wait(&full[s1], ((k + 1) / STAGES) & 1, abort, P.status);
          if (!__all_sync(0xffffffffu, w)) { live = false; break; }
          // (no tcgen05 fence per K step: the mbarrier orders the TMA data)
          // K-major, 128-byte swizzle: 16 columns = 32 bytes along the swizzled row
          const uint64_t da = ptx::sdesc_sw128(ptx::smem_u32(smem + s0 * STAGE), 16, 1024);
          const uint64_t db = diag ? da : ptx::sdesc_sw128(ptx::smem_u32(smem + s1 * STAGE), 16, 1024);
          if (ptx::elect_one()) {
#pragma unroll
            for (int u = 0; u < BK / 16; ++u)
              ptx::umma_bf16(d_tmem, ptx::sdesc_add(da, u * 32), ptx::sdesc_add(db, u * 32), kIdesc,
                             (kk != k_lo) || u != 0);
            ptx::umma_commit(&empty[s0]);
            if (!diag) ptx::umma_commit(&empty[s1]);
          }
          __syncwarp();
          k += diag ? 1 : 2;
        }
      }
      if (live) {
        if (ptx::elect_one()) ptx::umma_commit(&accum[b]);
        __syncwarp();
      }
    }
  } else if (warp < 6) {
    // ---- epilogue warps: lane quarter (warp & 3) of both Gram tiles ----
    pdl_wait();
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;          // TMEM lane = tile row
    // packed: columns [c_lo, c_hi) are this row's example block
    const int c_lo = packed ? row / P.T * P.T : 0, c_hi = packed ? c_lo + P.T : BT;
    float H = 0.f, S = 0.f;
    bool ok = true;
    // dual mode: the CTA's examples one after another; every epilogue warp passes the
    // per-example barrier once per example, so after a failed wait it only skips the work
    int qq = 0, el = 0;                                  // Y pairs read, examples done
    for (int ex = i; dual && ex < P.B; ex += gridDim.x, ++el) {
      H = 0.f;
      S = 0.f;
      for (int q = 0; q < 3; ++q, ++qq) {
        if (!ok) continue;
        const bool w = ptx::mbar_wait(ydone, qq & 1, abort, P.status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; continue; }
        ptx::tc_fence_after();
        float h = 0.f, sg = 0.f;
        const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
        const uint32_t bx = tmem + q * 128 + lanes, by = tmem + 384 + lanes;
        // columns the pair's MMAs wrote; rows of block 1 past r1 hold no data
        const int cmax = q == 0 ? BT : P.r1;
        const bool rok = q != 2 || row < P.r1;
#pragma unroll 1
        for (int c = 0; c < BT / 32 && c * 32 < cmax; ++c) {
          float vx[32], vy[32];
          ptx::tmem_ld32(bx + c * 32, vx);
          ptx::tmem_ld32(by + c * 32, vy);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (rok && c * 32 + e < cmax) {
              h = fmaf(vx[e], vy[e], h);
              sg += x_is_g ? vx[e] : vy[e];
            }
          }
        }
        const float wgt = q == 1 ? 2.f : 1.f;
        H = fmaf(wgt, h, H);
        S = fmaf(wgt, sg, S);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(yfree);
      }
      // the example's norm: the four warps' sums (two buffers: a warp may reach the next
      // example's writes while thread 64 still reads this one's)
      H = warp_sum(H);
      S = warp_sum(S);
      float* rb = red + (el & 1) * 8;
      if (lane == 0) {
        rb[(warp - 2) * 2] = H;
        rb[(warp - 2) * 2 + 1] = S;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps only
      if (threadIdx.x == 64 && ok && !*abort) {
        float h = 0.f, sv = 0.f;
        for (int q = 0; q < 4; ++q) { h += rb[2 * q]; sv += rb[2 * q + 1]; }
        P.out[ex] = h + (P.has_bias ? sv : 0.f);
      }
    }
    for (int j = 0; j < npairs && !dual; ++j) {
      int tb, sb;
      pair_of(j, nb, tb, sb);
      const int b = j & 1;
      const bool w = ptx::mbar_wait(&accum[b], (j >> 1) & 1, abort, P.status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      ptx::tc_fence_after();
      float h = 0.f, sg = 0.f;
      const uint32_t base = tmem + b * 256 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BT / 32; ++c) {
        float va[32], vg[32];
        ptx::tmem_ld32(base + c * 32, va);
        ptx::tmem_ld32(base + 128 + c * 32, vg);
        ptx::tmem_wait_ld();
        if (packed) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = c * 32 + e;
            const bool in = col >= c_lo && col < c_hi;
            h = fmaf(in ? va[e] : 0.f, vg[e], h);
            sg += in ? vg[e] : 0.f;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            h = fmaf(va[e], vg[e], h);
            sg += vg[e];
          }
        }
      }
      const float wgt = (tb == sb) ? 1.f : 2.f;
      H = fmaf(wgt, h, H);
      S = fmaf(wgt, sg, S);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tfree[b]);
    }
    if (packed) {
      rowbuf[row] = H;
      rowbuf[BT + row] = S;
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps only
      const int e = threadIdx.x - 64, ex = i * P.ept + e;
      if (e < P.ept && ex < P.B && ok && !*abort) {
        float h = 0.f, sg = 0.f;
        for (int r = e * P.T; r < (e + 1) * P.T; ++r) { h += rowbuf[r]; sg += rowbuf[BT + r]; }
        const float v = h + (P.has_bias && split == 0 ? sg : 0.f);
        if (P.ksplit > 1) st_cluster_f32(ptx::map_rank(ptx::smem_u32(csum + split * BT + e), 0), v);
        else P.out[ex] = v;
      }
    } else if (!dual) {
      H = warp_sum(H);
      S = warp_sum(S);
      if (lane == 0) {
        red[(warp - 2) * 2] = H;
        red[(warp - 2) * 2 + 1] = S;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps only
      if (threadIdx.x == 64 && ok && !*abort) {
        float h = 0.f, s = 0.f;
        for (int q = 0; q < 4; ++q) { h += red[2 * q]; s += red[2 * q + 1]; }
        const float v = h + (P.has_bias && split == 0 ? s : 0.f);
        if (P.ksplit > 1) st_cluster_f32(ptx::map_rank(ptx::smem_u32(csum + split * BT), 0), v);
        else P.out[i] = v;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (*abort && threadIdx.x == 32) {
    ptx::umma_commit(drainb);   // arrives once every MMA issued so far has completed
    ptx::mbar_wait_drain(drainb, 0);
  }
  if (P.ksplit > 1) {
    // every CTA's parts (and abort flag) are in rank 0's shared memory after the barrier;
    // rank 0 adds them in rank order
    if (threadIdx.x == 0) st_cluster_u32(ptx::map_rank(ptx::smem_u32(cabort + split), 0), *abort ? 1u : 0u);
    ptx::cluster_sync();
    if (split == 0) {
      bool bad = false;
      for (int r = 0; r < P.ksplit; ++r) bad |= cabort[r] != 0;
      const int ne = packed ? P.ept : 1;
      const int e = threadIdx.x - 64;
      if (!bad && e >= 0 && e < ne) {
        const int ex = packed ? i * P.ept + e : i;
        if (ex < P.B) {
          float v = 0.f;
          for (int r = 0; r < P.ksplit; ++r) v += csum[r * BT + e];
          P.out[ex] = v;
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace tcghost
}  // namespace dpk

namespace dph {
using namespace dpk;

bool tc_ghost_supported(const Geom& g) {
  return !g.conv && (g.d % 8 == 0) && (g.p % 8 == 0) && g.T >= 2 && g.T <= 512;
}

static int ghost_ept(const Geom& g) { return 2 * g.T <= tcghost::BT ? tcghost::BT / g.T : 0; }

// K splits of the A-Gram when the examples give fewer CTAs than SMs (not in dual mode).
static int ghost_ksplit(const Geom& g) {
  const int ept = ghost_ept(g);
  const int nb = (g.T + tcghost::BT - 1) / tcghost::BT;
  if (!ept && nb == 2) return 1;
  const long ctas = ept ? (g.B + ept - 1) / ept : g.B;
  const int kA = (g.D + tcghost::BK - 1) / tcghost::BK;
  return (int)std::max<long>(1, std::min<long>(std::min(kA, tcghost::MAXSPLIT), 152 / std::max<long>(1, ctas)));
}

size_t tc_ghost_ws_bytes(const Geom&) { return 0; }

static cudaError_t run_ghost(const Geom& g, const CUtensorMap& ma, const CUtensorMap& mg, const CUtensorMap& ma1,
                             const CUtensorMap& mg1, tcghost::Params P, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcghost::tc_ghost_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, tcghost::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  P.ksplit = ghost_ksplit(g);
  // two row blocks: persistent CTAs, one per SM at most (the kernel loops over examples)
  const bool dual = !P.ept && (g.T + tcghost::BT - 1) / tcghost::BT == 2;
  const dim3 grid(P.ept ? (g.B + P.ept - 1) / P.ept : dual ? std::min(g.B, 152) : g.B, P.ksplit);
  if (P.ksplit == 1) {
    launch_pdl(tcghost::tc_ghost_kernel, grid, tcghost::kThreads, tcghost::SMEM, s, ma, mg, ma1, mg1, P);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(tcghost::kThreads);
  cfg.dynamicSmemBytes = tcghost::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = P.ksplit;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, tcghost::tc_ghost_kernel, ma, mg, ma1, mg1, P);
  count_launch();
  return e;
}

// Conv layers with Cin % 64 == 0: the A-Gram reads the unfolded rows through TMA im2col
// loads (128 pixels x 64 channels per filter tap) from an NHWC copy of the input; the
// G-Gram reads the output gradient in its row layout [B, T, p].  Workspace: the NHWC
// copy, then the row layout of G.
bool tc_ghost_conv_supported(const Geom& g) {
  if (g.kh != g.k || g.padh != g.pad || g.Z != 1 || g.kz != 1) return false;   // square 2D kernels (TMA im2col)
  return g.conv && g.Cin % 64 == 0 && g.p % 8 == 0 && g.T >= 2 && g.T <= 512 && g.stride <= 8 &&
         g.pad <= 127 && g.dil * (g.k - 1) - g.pad <= 128 && (double)g.B * g.H * g.W * g.Cin < 4e9;
}

static size_t al256g(size_t n) { return (n + 255) & ~size_t(255); }

size_t tc_ghost_conv_ws_bytes(const Geom& g) {
  return al256g((size_t)g.B * g.H * g.W * g.Cin * 2) + al256g((size_t)g.B * g.T * g.p * 2);
}

cudaError_t launch_tc_ghost_conv(const Geom& g, const void* A, const void* G, float* out, void* ws,
                                 unsigned* status, cudaStream_t s) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  void* Xh = w;
  void* Gt = w + al256g((size_t)g.B * g.H * g.W * g.Cin * 2);
  if (g.nhwc) {          // channels last: the inputs are the NHWC source and the rows already
    Xh = const_cast<void*>(A);
    Gt = const_cast<void*>(G);
  } else {
    // NCHW -> NHWC and [p, T] -> [T, p], in one launch where both take the tiled kernel
    const cudaError_t e = launch_transpose_rows2(g.B, g.H * g.W, g.Cin, A, Xh, g.T, g.p, G, Gt, s);
    if (e != cudaSuccess) return e;
  }
  const int ept = ghost_ept(g);
  CUtensorMap ma, mg;
  if (!encode_im2col_bf16(&ma, Xh, g, tcghost::BT)) return cudaErrorInvalidValue;
  if (ept) {
    const uint64_t dg[2] = {(uint64_t)g.p, (uint64_t)g.B * g.T}, sg[1] = {(uint64_t)g.p * 2};
    const uint32_t box[2] = {tcghost::BK, tcghost::BT};
    if (!encode_tmap_bf16(&mg, Gt, 2, dg, sg, box)) return cudaErrorInvalidValue;
  } else {
    const uint64_t dg[3] = {(uint64_t)g.p, (uint64_t)g.T, (uint64_t)g.B};
    const uint64_t sg[2] = {(uint64_t)g.p * 2, (uint64_t)g.T * g.p * 2};
    const uint32_t box[3] = {tcghost::BK, tcghost::BT, 1};
    if (!encode_tmap_bf16(&mg, Gt, 3, dg, sg, box)) return cudaErrorInvalidValue;
  }
  tcghost::Params P{out, status, g.T, g.D, g.p, g.has_bias, g.B, ept, 1, g.Wout, g.k, g.stride, g.pad, g.dil, 0, 1,
                    tcghost::BT};
  return run_ghost(g, ma, mg, ma, mg, P, s);
}

cudaError_t launch_tc_ghost(const Geom& g, const void* A, const void* G, float* out, float* /*ws*/,
                            unsigned* status, cudaStream_t s, bool early) {
  CUtensorMap ma, mg, ma1, mg1;
  int r1 = tcghost::BT;
  const int ept = ghost_ept(g);
  if (ept) {   // flattened rows [B*T, width]
    const uint64_t da[2] = {(uint64_t)g.d, (uint64_t)g.B * g.T}, sa[1] = {(uint64_t)g.d * 2};
    const uint64_t dg[2] = {(uint64_t)g.p, (uint64_t)g.B * g.T}, sg[1] = {(uint64_t)g.p * 2};
    const uint32_t box[2] = {tcghost::BK, tcghost::BT};
    if (!encode_tmap_bf16(&ma, A, 2, da, sa, box) || !encode_tmap_bf16(&mg, G, 2, dg, sg, box))
      return cudaErrorInvalidValue;
  } else {
    const uint64_t da[3] = {(uint64_t)g.d, (uint64_t)g.T, (uint64_t)g.B};
    const uint64_t sa[2] = {(uint64_t)g.d * 2, (uint64_t)g.T * g.d * 2};
    const uint64_t dg[3] = {(uint64_t)g.p, (uint64_t)g.T, (uint64_t)g.B};
    const uint64_t sg[2] = {(uint64_t)g.p * 2, (uint64_t)g.T * g.p * 2};
    const uint32_t box[3] = {tcghost::BK, tcghost::BT, 1};
    if (!encode_tmap_bf16(&ma, A, 3, da, sa, box) || !encode_tmap_bf16(&mg, G, 3, dg, sg, box))
      return cudaErrorInvalidValue;
    // two row blocks: the second one's T - 128 rows, rounded up to 16, in boxes of their own
    if (g.T > tcghost::BT && g.T <= 2 * tcghost::BT) r1 = std::min(tcghost::BT, (g.T - tcghost::BT + 15) / 16 * 16);
    if (r1 < tcghost::BT) {
      const uint32_t box1[3] = {tcghost::BK, (uint32_t)r1, 1};
      if (!encode_tmap_bf16(&ma1, A, 3, da, sa, box1) || !encode_tmap_bf16(&mg1, G, 3, dg, sg, box1))
        return cudaErrorInvalidValue;
    }
  }
  tcghost::Params P{out, status, g.T, g.d, g.p, g.has_bias, g.B, ept, 0, 0, 0, 0, 0, 0, early ? 1 : 0, 1, r1};
  return r1 < tcghost::BT ? run_ghost(g, ma, mg, ma1, mg1, P, s) : run_ghost(g, ma, mg, ma, mg, P, s);
}

}  // namespace dph
