// C ABI of libdpclip: argument validation, the layerwise plan, workspace sizing and
// launches.  No allocation happens on any of these paths.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "common.cuh"
#include "tc.cuh"

using dpk::Geom;

namespace {

thread_local std::string g_last_error;

dp_status fail(dp_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dp_status ok() { return DP_OK; }

dp_status cuda_fail(cudaError_t e, const char* where) {
  return fail(DP_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Device status word, one per device (the address is looked up per device).
__device__ unsigned int g_status_word;

unsigned* status_ptr() {
  static unsigned* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned*>(p);
  }
  return cache[dev];
}

// Validate a descriptor and resolve the per-example contraction geometry.
dp_status make_geom(const dp_layer_desc* d, Geom* g) {
  if (!d) return fail(DP_ERR_INVALID_ARG, "desc is NULL");
  if (d->dtype != DP_BF16 && d->dtype != DP_FP32)
    return fail(DP_ERR_INVALID_ARG, "dtype %d is not DP_BF16 or DP_FP32", d->dtype);
  if (d->B <= 0 || d->p <= 0) return fail(DP_ERR_INVALID_ARG, "B=%d and p=%d must be > 0", d->B, d->p);
  std::memset(g, 0, sizeof(*g));
  g->B = d->B;
  g->p = d->p;
  g->has_bias = d->has_bias ? 1 : 0;
  if (d->kind != DP_LINEAR && d->layout != DP_NCHW && d->layout != DP_NHWC)
    return fail(DP_ERR_INVALID_ARG, "layout %d is not DP_NCHW or DP_NHWC", d->layout);
  g->nhwc = d->kind != DP_LINEAR && d->layout == DP_NHWC;
  if (d->kind == DP_LINEAR) {
    if (d->T <= 0 || d->d <= 0)
      return fail(DP_ERR_INVALID_ARG, "linear layer needs T=%d > 0 and d=%d > 0", d->T, d->d);
    g->conv = 0;
    g->T = d->T;
    g->d = g->D = d->d;
  } else if (d->kind == DP_CONV2D) {
    if (d->Cin <= 0 || d->H <= 0 || d->W <= 0 || d->k <= 0 || d->stride <= 0 || d->pad < 0 ||
        d->dil <= 0)
      return fail(DP_ERR_INVALID_ARG, "conv2d needs Cin, H, W, k, stride, dil > 0 and pad >= 0");
    const long Ho = ((long)d->H + 2L * d->pad - (long)d->dil * (d->k - 1) - 1) / d->stride + 1;
    const long Wo = ((long)d->W + 2L * d->pad - (long)d->dil * (d->k - 1) - 1) / d->stride + 1;
    if (Ho <= 0 || Wo <= 0) return fail(DP_ERR_INVALID_ARG, "conv2d output is empty");
    g->conv = 1;
    g->Cin = d->Cin; g->H = d->H; g->W = d->W; g->k = d->k;
    g->stride = d->stride; g->pad = d->pad; g->dil = d->dil;
    g->kh = d->k; g->padh = d->pad;
    g->Z = 1; g->Zout = 1; g->kz = 1; g->padz = 0;
    g->Hout = (int)Ho; g->Wout = (int)Wo;
    g->T = (int)(Ho * Wo);
    g->D = d->Cin * d->k * d->k;
    g->d = g->D;
  } else if (d->kind == DP_CONV3D) {
    if (d->Cin <= 0 || d->Z <= 0 || d->H <= 0 || d->W <= 0 || d->k <= 0 || d->stride <= 0 || d->pad < 0 ||
        d->dil <= 0)
      return fail(DP_ERR_INVALID_ARG, "conv3d needs Cin, Z, H, W, k, stride, dil > 0 and pad >= 0");
    auto out = [&](int n) { return ((long)n + 2L * d->pad - (long)d->dil * (d->k - 1) - 1) / d->stride + 1; };
    const long Zo = out(d->Z), Ho = out(d->H), Wo = out(d->W);
    if (Zo <= 0 || Ho <= 0 || Wo <= 0) return fail(DP_ERR_INVALID_ARG, "conv3d output is empty");
    if ((double)Zo * Ho * Wo > 2e9 || (double)d->Cin * d->k * d->k * d->k > 2e9)
      return fail(DP_ERR_UNSUPPORTED, "conv3d layer too large for 32-bit indexing");
    g->conv = 1;
    g->Cin = d->Cin; g->H = d->H; g->W = d->W; g->k = d->k;
    g->stride = d->stride; g->pad = d->pad; g->dil = d->dil;
    g->kh = d->k; g->padh = d->pad;
    g->Z = d->Z; g->Zout = (int)Zo; g->kz = d->k; g->padz = d->pad;
    g->Hout = (int)Ho; g->Wout = (int)Wo;
    g->T = (int)(Zo * Ho * Wo);
    g->D = d->Cin * d->k * d->k * d->k;
    g->d = g->D;
  } else if (d->kind == DP_CONV1D) {
    // one input row [Cin, W], a 1 x k kernel: stride, padding and dilation along W only
    if (d->Cin <= 0 || d->W <= 0 || d->k <= 0 || d->stride <= 0 || d->pad < 0 || d->dil <= 0)
      return fail(DP_ERR_INVALID_ARG, "conv1d needs Cin, W, k, stride, dil > 0 and pad >= 0");
    const long Wo = ((long)d->W + 2L * d->pad - (long)d->dil * (d->k - 1) - 1) / d->stride + 1;
    if (Wo <= 0) return fail(DP_ERR_INVALID_ARG, "conv1d output is empty");
    g->conv = 1;
    g->Cin = d->Cin; g->H = 1; g->W = d->W; g->k = d->k;
    g->stride = d->stride; g->pad = d->pad; g->dil = d->dil;
    g->kh = 1; g->padh = 0;
    g->Z = 1; g->Zout = 1; g->kz = 1; g->padz = 0;
    g->Hout = 1; g->Wout = (int)Wo;
    g->T = (int)Wo;
    g->D = d->Cin * d->k;
    g->d = g->D;
  } else {
    return fail(DP_ERR_INVALID_ARG, "kind %d is not DP_LINEAR, DP_CONV2D, DP_CONV1D or DP_CONV3D", d->kind);
  }
  // element counts must fit the kernels' 32-bit per-example and 64-bit global indexing
  if ((double)g->T * g->D > 2e9 || (double)g->T * g->p > 2e9 || (double)g->p * g->D > 2e9)
    return fail(DP_ERR_UNSUPPORTED, "layer too large for one example's 32-bit indexing");
  return DP_OK;
}

// Layerwise decision ([MixGhost] section 4, eq. 4.1): ghost norm iff its space 2T^2
// is below the instantiation space p*D; ties instantiate; one row -> closed form.
int resolve_mode(const Geom& g, int requested) {
  if (requested == DP_NORM_T1) return DP_NORM_T1;
  const double T = g.T, p = g.p, D = g.D;
  if (requested == DP_NORM_AUTO) {
    if (g.T == 1 && !g.conv) return DP_NORM_T1;
    // space priority: the ghost norm's 2T^2 against the instantiated gradient's p*D
    return 2.0 * T * T < p * D ? DP_NORM_GHOST : DP_NORM_INSTANTIATE;
  }
  if (requested == DP_NORM_AUTO_TIME) {
    if (g.T == 1 && !g.conv) return DP_NORM_T1;
    // speed priority: Gram products and Hadamard sum against the gradient and its square
    const double ghost = 2.0 * T * T * D + 2.0 * T * T * p + 2.0 * T * T;
    const double inst = 2.0 * T * p * D + 2.0 * p * D;
    return ghost < inst ? DP_NORM_GHOST : DP_NORM_INSTANTIATE;
  }
  return requested;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Conv layers in bf16 whose output count p is a multiple of 8 (16-byte TMA rows) run
// the linear tensor-core kernels on their row layout, written into the front of the
// workspace: U [B, T, Dp] then Gt [B, T, p], Dp = D rounded up to 8 with zero
// columns.  Zero columns leave the norms unchanged; a clipped sum over Dp columns
// goes to a padded buffer in the workspace and its first D columns to dW.
Geom rows_geom(const Geom& g) {
  Geom r = g;
  r.conv = 0;
  r.nhwc = 0;
  r.D = r.d = dph::conv_rows_width(g);
  return r;
}
bool rows_layout_ok(const Geom& g) { return !g.conv || g.p % 8 == 0; }
size_t rows_bytes(const Geom& g) {
  if (!g.conv) return 0;
  const size_t Dp = dph::conv_rows_width(g);
  return align256((size_t)g.B * g.T * Dp * 2) + align256((size_t)g.B * g.T * g.p * 2);
}
// Padded clipped-sum output (weights then bias) when Dp != D.
size_t padded_out_bytes(const Geom& g) {
  if (!g.conv || dph::conv_rows_width(g) == g.D) return 0;
  return align256((size_t)g.p * dph::conv_rows_width(g) * 4) + align256((size_t)g.p * 4);
}

// Clipped-sum kernel: 0 SIMT, 1 row-scaled tensor-core GEMM, 2 per-example tensor-core
// accumulation (single CTA), 3 per-example conv kernel with TMA im2col loads, 4 the
// row-scaled GEMM with im2col loads, 5 the one-row outer-product sum, 7 the on-chip unfold
// kernel of narrow conv layers.  The per-example
// kernels split the examples over clusters or the grid; the row-scaled GEMM splits the
// batch rows over the whole grid.
struct Plan {
  int kernel;
  bool rows;    // conv layer through its row layout
  Geom lg;      // the geometry the kernel sees
};

bool tc_inputs(const Geom& g, int dtype, const void* A, const void* G, const void* ws) {
  if (dtype != DP_BF16 || !aligned16(A) || !aligned16(G) || !rows_layout_ok(g)) return false;
  return !g.conv || aligned16(ws);
}

// DPCLIP_SUM_KERNEL=rows|example pins the tensor-core clipped-sum kernel where the
// shape allows it (all compute the same sum; used by the tests and for tuning).
int pinned_sum_kernel() {
  const char* v = std::getenv("DPCLIP_SUM_KERNEL");
  if (!v) return 0;
  if (!std::strcmp(v, "rows")) return 1;
  if (!std::strcmp(v, "example")) return 2;
  return 0;
}

int sum_kernel_for(const Geom& lg) {
  const int pin = pinned_sum_kernel();
  if (pin == 2 && dph::tc_sumx_supported(lg)) return 2;
  if (pin == 1 && dph::tc_sum_supported(lg)) return 1;
  const long tiles = (long)((lg.p + 127) / 128) * ((lg.D + 255) / 256);
  if (dph::tc_sumx_supported(lg) && tiles * std::min(4, lg.B) >= 64) return 2;
  if (dph::tc_sum_supported(lg)) return 1;
  if (dph::tc_sumx_supported(lg)) return 2;
  return 0;
}

// DPCLIP_CONV=rows keeps conv layers on their written-out row layout, DPCLIP_CONV=im2col on
// the im2col kernels where the shifted-tile kernel would take them (tests, tuning);
// otherwise conv layers the TMA kernels take use them.
bool conv_rows_pinned() {
  const char* v = std::getenv("DPCLIP_CONV");
  return v && !std::strcmp(v, "rows");
}
bool conv_im2col_pinned() {
  const char* v = std::getenv("DPCLIP_CONV");
  return v && !std::strcmp(v, "im2col");
}

bool im2col_inputs(const Geom& g, int dtype, const void* A, const void* G, const void* ws) {
  return g.conv && dtype == DP_BF16 && aligned16(A) && aligned16(G) && aligned16(ws) && !conv_rows_pinned();
}
bool use_tc_conv(const Geom& g, int dtype, const void* A, const void* G, const void* ws) {
  return im2col_inputs(g, dtype, A, G, ws) && dph::tc_conv_supported(g);
}
// Stride-1 "same" 1x1 / 3x3 conv layers, 64 input channels, at most 64 outputs: the filter
// rows and columns as shifted views of one output-gradient tile and one input tile.
bool use_tc_halo(const Geom& g, int dtype, const void* A, const void* G, const void* ws) {
  return im2col_inputs(g, dtype, A, G, ws) && !conv_im2col_pinned() && dph::tc_halo_supported(g);
}
// Conv layers with at most 64 unfolded columns (plus bias) form their unfold on chip and
// read G as it lies (DPCLIP_CONV=rows keeps them on the written-out row layout).
bool use_tc_unfold(const Geom& g, int dtype, const void* G) {
  return g.conv && dtype == DP_BF16 && aligned16(G) && !conv_rows_pinned() && dph::tc_unfold_supported(g);
}

// Conv clipped sums with im2col loads: per-example TMEM products (fp32 scaling) when an
// example has at least 128 rows, else the row-scaled GEMM (many examples per stage).
// One-row linear layers whose outer-product sum is small (or fp32) take the FFMA kernel.
bool use_t1_sum(const Geom& g, int dtype) {
  return !g.conv && g.T == 1 && (dtype == DP_FP32 || (double)g.p * g.d * g.B < (double)(1 << 28));
}

Plan sum_plan(const Geom& g, int dtype, const void* A, const void* G, const void* ws) {
  Plan pl{0, false, g};
  if (use_t1_sum(g, dtype)) return Plan{5, false, g};
  if (!pinned_sum_kernel() && use_tc_unfold(g, dtype, G)) return Plan{7, false, g};
  if (!pinned_sum_kernel() && im2col_inputs(g, dtype, A, G, ws)) {
    if (g.T >= 128 && dph::tc_conv_supported(g)) return Plan{3, false, g};
    if (dph::tc_sum_conv_supported(g)) return Plan{4, false, g};
  }
  if (!tc_inputs(g, dtype, A, G, ws)) return pl;
  const Geom lg = g.conv ? rows_geom(g) : g;
  const int k = sum_kernel_for(lg);
  if (k) pl = Plan{k, g.conv != 0, lg};
  return pl;
}

enum { NK_T1, NK_SIMT_GHOST, NK_SIMT_INST, NK_TC_GHOST, NK_TC_INST, NK_TC_CONV, NK_TC_GHOST_CONV, NK_TC_UNFOLD,
       NK_TC_HALO };

Plan norm_plan(const Geom& g, int mode, int dtype, const void* A, const void* G, const void* ws) {
  if (mode == DP_NORM_T1) return Plan{NK_T1, false, g};
  if (mode == DP_NORM_INSTANTIATE && use_tc_unfold(g, dtype, G)) return Plan{NK_TC_UNFOLD, false, g};
  if (mode == DP_NORM_INSTANTIATE && use_tc_halo(g, dtype, A, G, ws)) return Plan{NK_TC_HALO, false, g};
  if (mode == DP_NORM_INSTANTIATE && use_tc_conv(g, dtype, A, G, ws)) return Plan{NK_TC_CONV, false, g};
  if (mode == DP_NORM_GHOST && im2col_inputs(g, dtype, A, G, ws) && dph::tc_ghost_conv_supported(g))
    return Plan{NK_TC_GHOST_CONV, false, g};
  const Plan simt{mode == DP_NORM_GHOST ? NK_SIMT_GHOST : NK_SIMT_INST, false, g};
  if (!tc_inputs(g, dtype, A, G, ws)) return simt;
  const Geom lg = g.conv ? rows_geom(g) : g;
  if (mode == DP_NORM_GHOST && dph::tc_ghost_supported(lg)) return Plan{NK_TC_GHOST, g.conv != 0, lg};
  if (mode == DP_NORM_INSTANTIATE && dph::tc_sumx_supported(lg)) return Plan{NK_TC_INST, g.conv != 0, lg};
  return simt;
}

size_t simt_sum_bytes(const Geom& g) {
  return dph::simt_sum_splits(g) * ((size_t)g.p * g.D + g.p) * sizeof(float);
}

// Workspace a call needs on the path it takes (row layout first, then the kernel's own).
size_t sum_ws_bytes(const Geom& g, const Plan& pl) {
  const Geom& lg = pl.lg;
  // a conv layer's row-scaled GEMM reads pre-scaled rows; its bias is summed separately
  const size_t inner = pl.kernel == 7   ? dph::tc_unfold_ws_bytes(g, false)
                       : pl.kernel == 5 ? dph::t1_sum_ws_bytes(g)
                       : pl.kernel == 4 ? dph::tc_sum_conv_ws_bytes(g)
                       : pl.kernel == 3 ? dph::tc_conv_ws_bytes(g, false)
                       : pl.kernel == 2 ? dph::tc_sumx_ws_bytes(lg)
                       : pl.kernel == 1 ? align256(dph::tc_sum_ws_bytes(lg)) +
                                              (pl.rows ? dph::scaled_rows_bias_bytes(g.B, g.T, g.p) : 0)
                                        : simt_sum_bytes(g);
  return (pl.rows ? rows_bytes(g) + padded_out_bytes(g) : 0) + inner;
}

size_t norm_ws_bytes(const Geom& g, const Plan& pl) {
  size_t inner = 0;
  switch (pl.kernel) {
    case NK_T1: inner = 0; break;
    case NK_SIMT_GHOST: inner = dph::simt_ghost_ws_floats(g) * sizeof(float); break;
    case NK_SIMT_INST: inner = dph::simt_inst_ws_floats(g) * sizeof(float); break;
    case NK_TC_GHOST: inner = dph::tc_ghost_ws_bytes(pl.lg); break;
    case NK_TC_INST: inner = dph::tc_inst_ws_bytes(pl.lg); break;
    case NK_TC_CONV: inner = dph::tc_conv_ws_bytes(g, true); break;
    case NK_TC_GHOST_CONV: inner = dph::tc_ghost_conv_ws_bytes(g); break;
    case NK_TC_UNFOLD: inner = dph::tc_unfold_ws_bytes(g, true); break;
    case NK_TC_HALO: inner = dph::tc_halo_ws_bytes(g); break;
  }
  return (pl.rows ? rows_bytes(g) : 0) + inner;
}

// Kept per-example gradients: the instantiating tensor-core norm kernels store g_i and b_i;
// the layout (conv tile column order, or [p, D] / [p, Dp] rows) follows from the plan, which
// for aligned bf16 inputs depends on the geometry alone.
static const char kAlignedProbe[16] __attribute__((aligned(16))) = {};

bool keep_plan(int dtype, const Geom& g, const void* A, const void* G, const void* ws, Plan* pl) {
  if (dtype != DP_BF16 || g.T == 1) return false;
  *pl = norm_plan(g, DP_NORM_INSTANTIATE, dtype, A, G, ws);
  return pl->kernel == NK_TC_CONV || pl->kernel == NK_TC_INST || pl->kernel == NK_TC_UNFOLD ||
         pl->kernel == NK_TC_HALO;
}
bool keep_plan(int dtype, const Geom& g, Plan* pl) {
  return keep_plan(dtype, g, kAlignedProbe, kAlignedProbe, kAlignedProbe, pl);
}
// Columns of each kept gradient (conv tile columns or the on-chip unfold's weight layout = D;
// rows of a padded conv layer = Dp).
int kept_width(const Geom& g, const Plan& pl) {
  return pl.kernel == NK_TC_CONV || pl.kernel == NK_TC_UNFOLD || pl.kernel == NK_TC_HALO ? g.D : pl.lg.D;
}
size_t kept_sum_need(const Geom& g, const Plan& pl) {
  return dph::kept_sum_ws_bytes(g.B, g.p, kept_width(g, pl)) + (pl.rows ? padded_out_bytes(g) : 0);
}

// The size dp_workspace_size reports covers every path a call with `desc` can take
// (the choice also depends on the dtype and the alignment of the pointers).
size_t max_ws_bytes(const Geom& g, int mode) {
  static const char kAligned[16] __attribute__((aligned(16))) = {};
  const void* al = kAligned;
  const void* mis = kAligned + 1;
  size_t n = 0;
  for (int dt : {DP_BF16, DP_FP32})
    for (const void* ptr : {al, mis}) {
      n = std::max(n, norm_ws_bytes(g, norm_plan(g, mode, dt, ptr, ptr, ptr)));
      n = std::max(n, sum_ws_bytes(g, sum_plan(g, dt, ptr, ptr, ptr)));
    }
  // either tensor-core sum kernel may be pinned, and conv layers may be kept on rows
  if (dph::tc_conv_supported(g))
    n = std::max(n, std::max(dph::tc_conv_ws_bytes(g, true), dph::tc_conv_ws_bytes(g, false)));
  if (dph::tc_sum_conv_supported(g)) n = std::max(n, dph::tc_sum_conv_ws_bytes(g));
  if (mode == DP_NORM_GHOST && dph::tc_ghost_conv_supported(g)) n = std::max(n, dph::tc_ghost_conv_ws_bytes(g));
  if (g.conv && rows_layout_ok(g) && mode == DP_NORM_GHOST && dph::tc_ghost_supported(rows_geom(g)))
    n = std::max(n, rows_bytes(g) + dph::tc_ghost_ws_bytes(rows_geom(g)));
  if (rows_layout_ok(g)) {
    if (g.conv) {
      const Geom lg = rows_geom(g);
      if (mode == DP_NORM_INSTANTIATE && dph::tc_sumx_supported(lg))
        n = std::max(n, rows_bytes(g) + dph::tc_inst_ws_bytes(lg));
    }
    const Geom lg = g.conv ? rows_geom(g) : g;
    const size_t pre = rows_bytes(g) + padded_out_bytes(g);
    if (dph::tc_sum_supported(lg))
      n = std::max(n, pre + align256(dph::tc_sum_ws_bytes(lg)) +
                          (g.conv ? dph::scaled_rows_bias_bytes(g.B, g.T, g.p) : 0));
    if (dph::tc_sumx_supported(lg)) n = std::max(n, pre + dph::tc_sumx_ws_bytes(lg));
  }
  Plan kp;
  if (keep_plan(DP_BF16, g, &kp)) n = std::max(n, std::max(norm_ws_bytes(g, kp), kept_sum_need(g, kp)));
  return n;
}

// Launch the row layout of a conv layer into the workspace; returns the pointers.
cudaError_t prepare_rows(const Geom& g, const Plan& pl, const void*& A, const void*& G, void*& ws,
                         cudaStream_t stream, const float* scale = nullptr, float* db = nullptr,
                         int accumulate = 0, float* bias_part = nullptr, dph::NoiseArgs* nz = nullptr) {
  if (!pl.rows) return cudaSuccess;
  uint8_t* base = static_cast<uint8_t*>(ws);
  void* U = base;
  void* Gt = base + align256((size_t)g.B * g.T * dph::conv_rows_width(g) * 2);
  cudaError_t e = dph::launch_conv_rows(g, A, G, U, Gt, stream, scale, db, accumulate, bias_part, nz);
  A = U;
  if (!g.nhwc || scale) G = Gt;     // channels-last output gradients are the rows already
  ws = base + rows_bytes(g);
  return e;
}


std::atomic<unsigned long long> g_launches{0};

}  // namespace

namespace dph {
void count_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// For entry points defined in other translation units.
dp_status geom_from_desc(const dp_layer_desc* d, Geom* g) { return make_geom(d, g); }
dp_status set_error(dp_status st, const char* msg) { return fail(st, "%s", msg); }
}  // namespace dph

extern "C" {

unsigned long long dp_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }


int dp_abi_version(void) { return DPCLIP_ABI_VERSION; }

const char* dp_last_error(void) { return g_last_error.c_str(); }

dp_status dp_plan(const dp_layer_desc* desc, int requested, int* chosen_mode, int* rows_T,
                  int* width_D) {
  Geom g;
  dp_status st = make_geom(desc, &g);
  if (st != DP_OK) return st;
  if (requested < DP_NORM_AUTO || requested > DP_NORM_AUTO_TIME)
    return fail(DP_ERR_INVALID_ARG, "norm mode %d unknown", requested);
  if (requested == DP_NORM_T1 && (g.T != 1 || g.conv))
    return fail(DP_ERR_INVALID_ARG, "DP_NORM_T1 needs a linear layer with T == 1 (T=%d)", g.T);
  if (chosen_mode) *chosen_mode = resolve_mode(g, requested);
  if (rows_T) *rows_T = g.T;
  if (width_D) *width_D = g.D;
  return ok();
}

size_t dp_workspace_size(const dp_layer_desc* desc, int mode) {
  Geom g;
  if (make_geom(desc, &g) != DP_OK) return 0;
  if (mode < DP_NORM_AUTO || mode > DP_NORM_AUTO_TIME) return 0;
  if (mode == DP_NORM_T1 && (g.T != 1 || g.conv)) return 0;
  return max_ws_bytes(g, resolve_mode(g, mode));
}

dp_status dp_layer_sqnorms(const dp_layer_desc* desc, const void* A, const void* G, int mode,
                           float* sqnorm_out, int* chosen_mode_out, void* workspace,
                           size_t ws_bytes, cudaStream_t stream) {
  int chosen = 0;
  dp_status st = dp_plan(desc, mode, &chosen, nullptr, nullptr);
  if (st != DP_OK) return st;
  if (!A || !G || !sqnorm_out) return fail(DP_ERR_INVALID_ARG, "A, G and sqnorm_out must be non-NULL");
  Geom g;
  make_geom(desc, &g);
  const Plan pl = norm_plan(g, chosen, desc->dtype, A, G, workspace);
  const size_t need = norm_ws_bytes(g, pl);
  if (need && (!workspace || ws_bytes < need))
    return fail(DP_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need,
                workspace ? ws_bytes : (size_t)0);
  void* wsp = workspace;
  cudaError_t e = prepare_rows(g, pl, A, G, wsp, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_layer_sqnorms row layout");
  float* ws = static_cast<float*>(wsp);
  switch (pl.kernel) {
    case NK_T1: e = dph::launch_t1_norm(g, desc->dtype, A, G, sqnorm_out, stream); break;
    // linear layers read the caller's A and G, which may start before the previous kernel ends
    case NK_TC_GHOST:
      e = dph::launch_tc_ghost(pl.lg, A, G, sqnorm_out, ws, status_ptr(), stream, !pl.rows);
      break;
    case NK_TC_INST:
      e = dph::launch_tc_inst(pl.lg, A, G, sqnorm_out, ws, status_ptr(), stream, nullptr, nullptr, !pl.rows);
      break;
    case NK_TC_CONV: e = dph::launch_tc_conv_norm(g, A, G, sqnorm_out, ws, status_ptr(), stream); break;
    case NK_TC_GHOST_CONV: e = dph::launch_tc_ghost_conv(g, A, G, sqnorm_out, ws, status_ptr(), stream); break;
    case NK_TC_UNFOLD: e = dph::launch_tc_unfold_norm(g, A, G, sqnorm_out, ws, status_ptr(), stream); break;
    case NK_TC_HALO: e = dph::launch_tc_halo_norm(g, A, G, sqnorm_out, ws, status_ptr(), stream); break;
    case NK_SIMT_GHOST: e = dph::launch_simt_ghost(g, desc->dtype, A, G, sqnorm_out, ws, stream); break;
    case NK_SIMT_INST: e = dph::launch_simt_inst(g, desc->dtype, A, G, sqnorm_out, ws, stream); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "dp_layer_sqnorms launch");
  if (chosen_mode_out) *chosen_mode_out = chosen;
  return ok();
}

dp_status dp_clip_factors(const float* sqnorms, int B, int L, int per_layer, const float* C,
                          float* factors_out, cudaStream_t stream) {
  if (!sqnorms || !factors_out || !C) return fail(DP_ERR_INVALID_ARG, "NULL pointer argument");
  if (B <= 0 || L <= 0) return fail(DP_ERR_INVALID_ARG, "B=%d and L=%d must be > 0", B, L);
  if (per_layer && L > 64)
    return fail(DP_ERR_UNSUPPORTED, "per-layer clipping supports up to 64 layers per call (L=%d)", L);
  const int nC = per_layer ? L : 1;
  for (int l = 0; l < nC; ++l)
    if (!(C[l] > 0.f) || !std::isfinite(C[l]))
      return fail(DP_ERR_INVALID_ARG, "bound C[%d]=%g must be finite and > 0", l, (double)C[l]);
  unsigned* st = status_ptr();
  if (!st) return fail(DP_ERR_CUDA, "cannot resolve the device status word");
  cudaError_t e = dph::launch_clip_factors(sqnorms, B, L, per_layer, C, factors_out, st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_clip_factors launch");
  return ok();
}

// Whether a dp_layer_sqnorms call in `norm_mode` leaves the NHWC copy of a conv layer's
// input at the front of its workspace (the im2col ghost and instantiation kernels do).
static bool norm_leaves_nhwc(const Geom& g, int norm_mode, int dtype, const void* A, const void* G, const void* ws) {
  if (!g.conv || g.nhwc || norm_mode < DP_NORM_AUTO || norm_mode > DP_NORM_AUTO_TIME || norm_mode == DP_NORM_T1)
    return false;   // (channels-last inputs need no copy to share)
  const Plan npl = norm_plan(g, resolve_mode(g, norm_mode), dtype, A, G, ws);
  return npl.kernel == NK_TC_GHOST_CONV || npl.kernel == NK_TC_CONV || npl.kernel == NK_TC_HALO;
}

// The noise of a fused call: the scale and divisor as dp_add_noise forms them.
static dp_status noise_args(const dp_noise_desc* nd, const Geom& g, dph::NoiseArgs* nz) {
  *nz = dph::NoiseArgs{};
  if (!nd) return fail(DP_ERR_INVALID_ARG, "noise descriptor is NULL");
  if (nd->B <= 0) return fail(DP_ERR_INVALID_ARG, "B=%d must be > 0", nd->B);
  if (!(nd->sigma >= 0.f) || !std::isfinite(nd->sigma) || !(nd->C >= 0.f) || !std::isfinite(nd->C))
    return fail(DP_ERR_INVALID_ARG, "sigma=%g and C=%g must be finite and >= 0", (double)nd->sigma, (double)nd->C);
  const uint64_t n = (uint64_t)g.p * g.D + (uint64_t)g.p;
  if (nd->offset + n < nd->offset) return fail(DP_ERR_INVALID_ARG, "offset + p*D + p overflows");
  nz->on = 1;
  nz->sc = (float)((double)nd->sigma * (double)nd->C);
  nz->invB = (float)(1.0 / (double)nd->B);
  nz->seed = nd->seed;
  nz->seed_dev = nd->seed_dev;
  nz->off_a = nd->offset;
  nz->off_b = nd->offset + (uint64_t)g.p * g.D;
  return DP_OK;
}

// The noise pass over dW and db when no kernel of the sum fused it.
static cudaError_t finish_noise(const Geom& g, float* dW, float* db, const dph::NoiseArgs* nz, cudaStream_t s) {
  if (!nz || !nz->on) return cudaSuccess;
  const size_t nw = (size_t)g.p * g.D;
  const bool w = !nz->applied_a, b = db && !nz->applied_b;
  if (w && b && db == dW + nw)
    return dph::launch_add_noise(dW, nw + g.p, nz->sc, nz->invB, nz->seed, nz->off_a, nz->seed_dev, s);
  cudaError_t e = w ? dph::launch_add_noise(dW, nw, nz->sc, nz->invB, nz->seed, nz->off_a, nz->seed_dev, s)
                    : cudaSuccess;
  if (e == cudaSuccess && b) e = dph::launch_add_noise(db, g.p, nz->sc, nz->invB, nz->seed, nz->off_b, nz->seed_dev, s);
  return e;
}

static dp_status clipped_sum_impl(const dp_layer_desc* desc, const void* A, const void* G, const float* factors,
                                  float* dW, float* db, int accumulate, void* workspace, size_t ws_bytes,
                                  cudaStream_t stream, int reuse_norm_mode, const dp_noise_desc* noise) {
  Geom g;
  dp_status st = make_geom(desc, &g);
  if (st != DP_OK) return st;
  if (!A || !G || !factors || !dW) return fail(DP_ERR_INVALID_ARG, "A, G, factors and dW must be non-NULL");
  if (db && !g.has_bias) return fail(DP_ERR_INVALID_ARG, "db given for a layer without bias");
  dph::NoiseArgs nzv;
  dph::NoiseArgs* nz = nullptr;
  if (noise) {
    if ((st = noise_args(noise, g, &nzv)) != DP_OK) return st;
    nz = &nzv;
  }
  const Plan pl = sum_plan(g, desc->dtype, A, G, workspace);
  const size_t need = sum_ws_bytes(g, pl);
  if (need && (!workspace || ws_bytes < need))
    return fail(DP_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need,
                workspace ? ws_bytes : (size_t)0);
  void* wsp = workspace;
  // conv rows for the row-scaled GEMM: the transpose writes bf16(c_i G_i^T) directly and
  // sums the bias on the way (its partials sit after the GEMM's in the workspace)
  const bool prescale = pl.rows && pl.kernel == 1;
  float* bias_part = prescale ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + rows_bytes(g) +
                                                         padded_out_bytes(g) +
                                                         align256(dph::tc_sum_ws_bytes(pl.lg)))
                              : nullptr;
  cudaError_t e = prepare_rows(g, pl, A, G, wsp, stream, prescale ? factors : nullptr, prescale ? db : nullptr,
                               accumulate, bias_part, prescale ? nz : nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "dp_clipped_sum row layout");
  // padded columns: the kernel writes a padded buffer, then its first D columns go out
  const bool padded = pl.rows && padded_out_bytes(g) != 0;
  float* kdW = dW;
  float* kdb = db;
  int kacc = accumulate;
  if (padded) {
    kdW = static_cast<float*>(wsp);
    kdb = db ? kdW + align256((size_t)g.p * pl.lg.D * 4) / 4 : nullptr;
    kacc = 0;
    wsp = static_cast<uint8_t*>(wsp) + padded_out_bytes(g);
  }
  if (pl.kernel == 7)
    e = dph::launch_tc_unfold_sum(g, A, G, factors, dW, db, accumulate, wsp, status_ptr(), stream, nz);
  else if (pl.kernel == 5)
    e = dph::launch_t1_sum(g, desc->dtype, A, G, factors, dW, db, accumulate, static_cast<float*>(wsp), stream, nz);
  else if (pl.kernel == 4 || pl.kernel == 3) {
    const bool xh = reuse_norm_mode >= 0 && norm_leaves_nhwc(g, reuse_norm_mode, desc->dtype, A, G, workspace);
    if (pl.kernel == 4)
      e = dph::launch_tc_sum_conv(g, A, G, factors, dW, db, accumulate, wsp, status_ptr(), stream, xh, nz);
    else
      e = dph::launch_tc_conv_sum(g, A, G, factors, dW, db, accumulate, wsp, status_ptr(), stream, xh, nz);
  }
  else if (pl.kernel == 2)   // (a padded output gets its noise after the compaction below)
    e = dph::launch_tc_sumx(pl.lg, A, G, factors, kdW, kdb, kacc, wsp, status_ptr(), stream, padded ? nullptr : nz,
                            !pl.rows);
  else if (prescale) {
    e = dph::launch_tc_sum_prescaled(pl.lg, A, G, kdW, kacc, static_cast<float*>(wsp), status_ptr(), stream,
                                     padded ? nullptr : nz);
    kdb = nullptr;   // the bias went straight to db
  } else if (pl.kernel == 1)
    e = dph::launch_tc_sum(pl.lg, A, G, factors, kdW, kdb, kacc, static_cast<float*>(wsp), status_ptr(),
                           stream, padded ? nullptr : nz);
  else
    e = dph::launch_simt_clipped_sum(g, desc->dtype, A, G, factors, dW, db, accumulate,
                                     static_cast<float*>(wsp), (int)dph::simt_sum_splits(g), stream);
  if (e == cudaSuccess && padded) {
    e = dph::launch_compact_cols(kdW, g.p, g.D, pl.lg.D, dW, accumulate, stream);
    if (e == cudaSuccess && kdb) e = dph::launch_compact_cols(kdb, 1, g.p, g.p, db, accumulate, stream);
  }
  if (e == cudaSuccess) e = finish_noise(g, dW, db, nz, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_clipped_sum launch");
  return ok();
}

size_t dp_grads_size(const dp_layer_desc* desc) {
  Geom g;
  if (make_geom(desc, &g) != DP_OK) return 0;
  Plan pl;
  if (!keep_plan(desc->dtype, g, &pl)) return 0;
  const size_t w = (size_t)g.B * g.p * kept_width(g, pl);
  return (w + (g.has_bias ? (size_t)g.B * g.p : 0)) * sizeof(float);
}

dp_status dp_layer_sqnorms_keep(const dp_layer_desc* desc, const void* A, const void* G, float* sqnorm_out,
                                float* grads, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  Geom g;
  dp_status st = make_geom(desc, &g);
  if (st != DP_OK) return st;
  if (!A || !G || !sqnorm_out || !grads)
    return fail(DP_ERR_INVALID_ARG, "A, G, sqnorm_out and grads must be non-NULL");
  if (!aligned16(grads)) return fail(DP_ERR_INVALID_ARG, "grads must be 16-byte aligned");
  Plan pl;
  if (!keep_plan(desc->dtype, g, A, G, workspace, &pl))
    return fail(DP_ERR_UNSUPPORTED,
                "this layer's instantiated norm does not run on a kernel that keeps per-example gradients "
                "(bf16 with 16-byte aligned A, G and workspace, tensor-core shapes)");
  const size_t need = norm_ws_bytes(g, pl);
  if (need && (!workspace || ws_bytes < need))
    return fail(DP_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need,
                workspace ? ws_bytes : (size_t)0);
  void* wsp = workspace;
  cudaError_t e = prepare_rows(g, pl, A, G, wsp, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_layer_sqnorms_keep row layout");
  float* keep_b = g.has_bias ? grads + (size_t)g.B * g.p * kept_width(g, pl) : nullptr;
  if (pl.kernel == NK_TC_CONV)
    e = dph::launch_tc_conv_norm(g, A, G, sqnorm_out, wsp, status_ptr(), stream, grads, keep_b);
  else if (pl.kernel == NK_TC_UNFOLD)
    e = dph::launch_tc_unfold_norm(g, A, G, sqnorm_out, wsp, status_ptr(), stream, grads, keep_b);
  else if (pl.kernel == NK_TC_HALO)
    e = dph::launch_tc_halo_norm(g, A, G, sqnorm_out, wsp, status_ptr(), stream, grads, keep_b);
  else
    e = dph::launch_tc_inst(pl.lg, A, G, sqnorm_out, static_cast<float*>(wsp), status_ptr(), stream, grads, keep_b,
                            !pl.rows);
  if (e != cudaSuccess) return cuda_fail(e, "dp_layer_sqnorms_keep launch");
  return ok();
}

static dp_status kept_sum_impl(const dp_layer_desc* desc, const float* grads, const float* factors, float* dW,
                               float* db, int accumulate, void* workspace, size_t ws_bytes, cudaStream_t stream,
                               const dp_noise_desc* noise) {
  Geom g;
  dp_status st = make_geom(desc, &g);
  if (st != DP_OK) return st;
  if (!grads || !factors || !dW) return fail(DP_ERR_INVALID_ARG, "grads, factors and dW must be non-NULL");
  if (db && !g.has_bias) return fail(DP_ERR_INVALID_ARG, "db given for a layer without bias");
  dph::NoiseArgs nzv;
  dph::NoiseArgs* nz = nullptr;
  if (noise) {
    if ((st = noise_args(noise, g, &nzv)) != DP_OK) return st;
    nz = &nzv;
  }
  Plan pl;
  if (!keep_plan(desc->dtype, g, &pl))
    return fail(DP_ERR_UNSUPPORTED, "this layer keeps no per-example gradients (see dp_grads_size)");
  const size_t need = kept_sum_need(g, pl);
  if (!workspace || ws_bytes < need)
    return fail(DP_ERR_INVALID_ARG, "workspace of %zu bytes needed, %zu given", need,
                workspace ? ws_bytes : (size_t)0);
  const int width = kept_width(g, pl);
  const float* keep_b = g.has_bias ? grads + (size_t)g.B * g.p * width : nullptr;
  const int conv_kk = pl.kernel == NK_TC_CONV || pl.kernel == NK_TC_HALO ? g.k * g.k : 0;
  const bool padded = pl.rows && padded_out_bytes(g) != 0;
  float* kdW = dW;
  float* kdb = db;
  void* wsp = workspace;
  if (padded) {     // rows of a conv layer whose unfolded width was padded: compact afterwards
    kdW = static_cast<float*>(wsp);
    kdb = db ? kdW + align256((size_t)g.p * width * 4) / 4 : nullptr;
    wsp = static_cast<uint8_t*>(wsp) + padded_out_bytes(g);
  }
  cudaError_t e = dph::launch_kept_sum(g.B, g.p, width, conv_kk, grads, keep_b, factors, kdW, kdb,
                                       padded ? 0 : accumulate, stream, pl.kernel == NK_TC_HALO,
                                       padded ? nullptr : nz, wsp);   // (a padded sum: its noise after compaction)
  if (e == cudaSuccess && padded) {
    e = dph::launch_compact_cols(kdW, g.p, g.D, width, dW, accumulate, stream);
    if (e == cudaSuccess && kdb) e = dph::launch_compact_cols(kdb, 1, g.p, g.p, db, accumulate, stream);
  }
  if (e == cudaSuccess) e = finish_noise(g, dW, db, nz, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_clipped_sum_kept launch");
  return ok();
}

dp_status dp_clipped_sum_kept(const dp_layer_desc* desc, const float* grads, const float* factors, float* dW,
                              float* db, int accumulate, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return kept_sum_impl(desc, grads, factors, dW, db, accumulate, workspace, ws_bytes, stream, nullptr);
}

dp_status dp_clipped_sum_kept_noised(const dp_layer_desc* desc, const float* grads, const float* factors, float* dW,
                                     float* db, int accumulate, const dp_noise_desc* noise, void* workspace,
                                     size_t ws_bytes, cudaStream_t stream) {
  if (!noise) return fail(DP_ERR_INVALID_ARG, "noise descriptor is NULL");
  return kept_sum_impl(desc, grads, factors, dW, db, accumulate, workspace, ws_bytes, stream, noise);
}

dp_status dp_clipped_sum(const dp_layer_desc* desc, const void* A, const void* G, const float* factors, float* dW,
                         float* db, int accumulate, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return clipped_sum_impl(desc, A, G, factors, dW, db, accumulate, workspace, ws_bytes, stream, -1, nullptr);
}

dp_status dp_clipped_sum_noised(const dp_layer_desc* desc, int norm_mode, const void* A, const void* G,
                                const float* factors, float* dW, float* db, int accumulate,
                                const dp_noise_desc* noise, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (norm_mode < -1 || norm_mode > DP_NORM_AUTO_TIME) return fail(DP_ERR_INVALID_ARG, "norm mode %d unknown", norm_mode);
  if (!noise) return fail(DP_ERR_INVALID_ARG, "noise descriptor is NULL");
  return clipped_sum_impl(desc, A, G, factors, dW, db, accumulate, workspace, ws_bytes, stream, norm_mode, noise);
}

dp_status dp_clipped_sum_reuse(const dp_layer_desc* desc, int norm_mode, const void* A, const void* G,
                               const float* factors, float* dW, float* db, int accumulate, void* workspace,
                               size_t ws_bytes, cudaStream_t stream) {
  if (norm_mode < DP_NORM_AUTO || norm_mode > DP_NORM_AUTO_TIME)
    return fail(DP_ERR_INVALID_ARG, "norm mode %d unknown", norm_mode);
  return clipped_sum_impl(desc, A, G, factors, dW, db, accumulate, workspace, ws_bytes, stream, norm_mode, nullptr);
}

int dp_layout_reused(const dp_layer_desc* desc, int norm_mode) {
  Geom g;
  if (make_geom(desc, &g) != DP_OK) return 0;
  static const char al[16] __attribute__((aligned(16))) = {};
  if (!norm_leaves_nhwc(g, norm_mode, desc->dtype, al, al, al)) return 0;
  const Plan spl = sum_plan(g, desc->dtype, al, al, al);
  return (spl.kernel == 4 || spl.kernel == 3) ? 1 : 0;
}

static dp_status add_noise_impl(float* grad, size_t n, float sigma, float C, int B, uint64_t seed,
                                const unsigned long long* seed_dev, uint64_t offset, cudaStream_t stream) {
  if (n == 0) return ok();
  if (!grad) return fail(DP_ERR_INVALID_ARG, "grad is NULL");
  if (B <= 0) return fail(DP_ERR_INVALID_ARG, "B=%d must be > 0", B);
  if (!(sigma >= 0.f) || !std::isfinite(sigma) || !(C >= 0.f) || !std::isfinite(C))
    return fail(DP_ERR_INVALID_ARG, "sigma=%g and C=%g must be finite and >= 0", (double)sigma, (double)C);
  if (offset + n < offset) return fail(DP_ERR_INVALID_ARG, "offset + n overflows");
  const float sc = (float)((double)sigma * (double)C);
  const float invB = (float)(1.0 / (double)B);
  cudaError_t e = dph::launch_add_noise(grad, n, sc, invB, seed, offset, seed_dev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_add_noise launch");
  return ok();
}

dp_status dp_add_noise(float* grad, size_t n, float sigma, float C, int B, uint64_t seed,
                       uint64_t offset, cudaStream_t stream) {
  return add_noise_impl(grad, n, sigma, C, B, seed, nullptr, offset, stream);
}

dp_status dp_add_noise_devseed(float* grad, size_t n, float sigma, float C, int B,
                               const unsigned long long* seed_dev, uint64_t offset,
                               cudaStream_t stream) {
  if (!seed_dev && n) return fail(DP_ERR_INVALID_ARG, "seed_dev is NULL");
  return add_noise_impl(grad, n, sigma, C, B, 0, seed_dev, offset, stream);
}

dp_status dp_add_noise_blocks(float* grad, const dp_noise_block* blocks, int nblocks, float sigma, int B,
                              uint64_t seed, const unsigned long long* seed_dev, cudaStream_t stream) {
  if (!grad || !blocks) return fail(DP_ERR_INVALID_ARG, "grad and blocks must be non-NULL");
  if (nblocks < 1 || nblocks > dpk::kMaxNoiseBlocks)
    return fail(DP_ERR_INVALID_ARG, "nblocks=%d must be in 1..%d", nblocks, dpk::kMaxNoiseBlocks);
  if (B <= 0) return fail(DP_ERR_INVALID_ARG, "B=%d must be > 0", B);
  if (!(sigma >= 0.f) || !std::isfinite(sigma))
    return fail(DP_ERR_INVALID_ARG, "sigma=%g must be finite and >= 0", (double)sigma);
  dpk::NoiseBlocks nb{};
  nb.count = nblocks;
  uint64_t end = 0;
  for (int b = 0; b < nblocks; ++b) {
    const dp_noise_block& k = blocks[b];
    if (!(k.C >= 0.f) || !std::isfinite(k.C)) return fail(DP_ERR_INVALID_ARG, "block %d: C=%g", b, (double)k.C);
    if (k.offset + k.n < k.offset) return fail(DP_ERR_INVALID_ARG, "block %d: offset + n overflows", b);
    if (b && k.offset < end) return fail(DP_ERR_INVALID_ARG, "block %d overlaps or precedes block %d", b, b - 1);
    end = k.offset + k.n;
    nb.off[b] = k.offset;
    nb.n[b] = k.n;
    nb.sc[b] = (float)((double)sigma * (double)k.C);
    nb.qcum[b + 1] = nb.qcum[b] + (k.n ? ((k.offset + k.n + 3) >> 2) - (k.offset >> 2) : 0);
  }
  const float invB = (float)(1.0 / (double)B);
  cudaError_t e = dph::launch_add_noise_blocks(grad, nb, invB, seed, seed_dev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_add_noise_blocks launch");
  return ok();
}

dp_status dp_adaptive_bound(const float* sqnorms, int B, float C_l2, float alpha, float beta,
                            float sigma_l2, uint64_t seed, int layer, float* out,
                            cudaStream_t stream) {
  if (!sqnorms || !out) return fail(DP_ERR_INVALID_ARG, "sqnorms and out must be non-NULL");
  if (B <= 0 || layer < 0) return fail(DP_ERR_INVALID_ARG, "B=%d must be > 0 and layer=%d >= 0", B, layer);
  if (!(C_l2 > 0.f) || !std::isfinite(alpha) || !std::isfinite(beta) || !(sigma_l2 >= 0.f))
    return fail(DP_ERR_INVALID_ARG, "C_l2 > 0, finite alpha and beta, sigma_l2 >= 0 required");
  unsigned* st = status_ptr();
  if (!st) return fail(DP_ERR_CUDA, "dp_adaptive_bound: no device status word on the current device");
  cudaError_t e = dph::launch_adaptive_bound(sqnorms, B, 1, &C_l2, alpha, beta, sigma_l2, seed, nullptr, layer,
                                             out, st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_adaptive_bound launch");
  return ok();
}

dp_status dp_adaptive_bounds(const float* sqnorms, int B, int layer0, int L, const float* C_l2, float alpha,
                             float beta, float sigma_l2, uint64_t seed, const unsigned long long* seed_dev,
                             float* out, cudaStream_t stream) {
  if (!sqnorms || !out || !C_l2) return fail(DP_ERR_INVALID_ARG, "sqnorms, C_l2 and out must be non-NULL");
  if (B <= 0 || layer0 < 0 || L < 1 || L > 64)
    return fail(DP_ERR_INVALID_ARG, "B=%d must be > 0, layer0=%d >= 0 and 1 <= L=%d <= 64", B, layer0, L);
  for (int l = 0; l < L; ++l)
    if (!(C_l2[l] > 0.f) || !std::isfinite(C_l2[l]))
      return fail(DP_ERR_INVALID_ARG, "C_l2[%d] must be finite and > 0", l);
  if (!std::isfinite(alpha) || !std::isfinite(beta) || !(sigma_l2 >= 0.f))
    return fail(DP_ERR_INVALID_ARG, "finite alpha and beta, sigma_l2 >= 0 required");
  unsigned* st = status_ptr();
  if (!st) return fail(DP_ERR_CUDA, "dp_adaptive_bounds: no device status word on the current device");
  cudaError_t e = dph::launch_adaptive_bound(sqnorms, B, L, C_l2, alpha, beta, sigma_l2, seed, seed_dev, layer0, out,
                                             st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_adaptive_bounds launch");
  return ok();
}

dp_status dp_selftest_wait_timeout(unsigned long long* waited_ns, cudaStream_t stream) {
  unsigned* st = status_ptr();
  if (!st) return fail(DP_ERR_CUDA, "cannot resolve the device status word");
  const cudaError_t e = dph::launch_selftest_wait(st, waited_ns, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_selftest_wait_timeout launch");
  return ok();
}

dp_status dp_check_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "dp_check_status sync");
  unsigned* st = status_ptr();
  if (!st) return fail(DP_ERR_CUDA, "cannot resolve the device status word");
  unsigned v = 0;
  e = cudaMemcpy(&v, st, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "dp_check_status read");
  if (v) {
    const unsigned zero = 0;
    e = cudaMemcpy(st, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "dp_check_status clear");
  }
  if (v & dpk::kStatusTimeout) return fail(DP_ERR_TIMEOUT, "a bounded device wait gave up");
  if (v & dpk::kStatusNonfinite) return fail(DP_ERR_NONFINITE, "a per-example norm was not finite");
  return ok();
}

}  // extern "C"
