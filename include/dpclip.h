/*
 * dpclip.h -- C ABI of libdpclip, DP-SGD per-example gradient clipping on GB300 (sm_103a).
 *
 * The library computes, for captured layer activations A and output gradients G,
 * the per-example gradient norms (ghost norm or per-example instantiation, chosen
 * layer by layer), the clip factors, the clipped sum sum_i c_i G_i^T A_i with its
 * bias gradient, and the Gaussian noise with the 1/B scale.  Pages (by title):
 *   [FastClip]   "Scaling up Differentially Private Deep Learning with Fast
 *                Per-Example Gradient Clipping"
 *   [ThreeTools] "Three Tools for Practical Differential Privacy"
 *   [MixGhost]   "Scalable and Efficient Training of Large Convolutional Neural
 *                Networks with Differential Privacy"
 *
 * Conventions for every call:
 *  - Pointers named A, G, sqnorms, factors, dW, db, grad, workspace are DEVICE
 *    pointers; the caller owns every buffer and the library never allocates on
 *    these paths (workspace is caller-provided, sized by dp_workspace_size).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream) unless noted.
 *    Arguments are validated on the host before anything is launched; a bad
 *    argument returns DP_ERR_INVALID_ARG (or DP_ERR_UNSUPPORTED) and launches
 *    nothing.  dp_last_error() then holds a message (per calling thread).
 *  - Device-side conditions (a non-finite norm) set a device status word that
 *    dp_check_status() returns and clears.
 *  - Stream order: the library's kernels use programmatic dependent launch.  Each
 *    waits for the previous kernel in the stream before it reads what that kernel
 *    wrote, except that the tensor-core kernels of linear layers may start loading
 *    A and G while the previous kernel still runs, if that kernel lets its dependents
 *    launch early (the library's own kernels do; kernels that do not use programmatic
 *    launch, such as PyTorch's and cuBLAS's, complete first).  So A and G must be
 *    complete before the previous such kernel in the stream starts: never written by
 *    a kernel that itself triggers programmatic launch right before the call.  The
 *    library never writes A or G.
 *  - Layouts (row-major, contiguous, PyTorch conventions):
 *      linear: A [B, T, d], G [B, T, p]; weight gradient [p, d]
 *      conv2d: A [B, Cin, H, W] (NCHW), G [B, p, Hout, Wout]; weight gradient
 *              [p, Cin, k, k]; T = Hout*Wout, D = Cin*k*k.
 *    bf16 inputs are accumulated in fp32; every output is fp32.
 */
#ifndef DPCLIP_H
#define DPCLIP_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DPCLIP_ABI_VERSION 3

typedef enum {
  DP_OK = 0,
  DP_ERR_INVALID_ARG = 1,   /* bad pointer, size, mode or descriptor */
  DP_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement */
  DP_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  DP_ERR_NONFINITE = 4,     /* a norm was inf/NaN: that example's factor was set to 0 */
  DP_ERR_TIMEOUT = 5        /* a bounded device wait gave up */
} dp_status;

typedef enum { DP_BF16 = 0, DP_FP32 = 1 } dp_dtype;
typedef enum { DP_LINEAR = 0, DP_CONV2D = 1, DP_CONV1D = 2, DP_CONV3D = 3 } dp_kind;
/* Memory layout of a conv layer's A and G: channels first (PyTorch's default, NCHW) or
 * channels last (NHWC: A [B, H, W, Cin], G [B, Hout, Wout, p]; conv1d [B, L, C], conv3d
 * [B, Z, H, W, C]; PyTorch's channels_last memory format).  Channels-last inputs feed the
 * TMA im2col loads and the row layout directly, without the layout copies. */
typedef enum { DP_NCHW = 0, DP_NHWC = 1 } dp_layout;

/* How the per-example norm is formed ([MixGhost] section 4, the layerwise decision). */
typedef enum {
  DP_NORM_AUTO = 0,          /* ghost iff 2T^2 < p*D (ties instantiate); T == 1 -> closed form */
  DP_NORM_GHOST = 1,         /* Gram identity: sum_{t,s} (a_t.a_s)(g_t.g_s) */
  DP_NORM_INSTANTIATE = 2,   /* g_i = G_i^T U(A_i) formed on chip, squared and summed */
  DP_NORM_T1 = 3,            /* one row: ||a||^2 ||g||^2 (reported; also accepted when T == 1) */
  DP_NORM_AUTO_TIME = 4      /* speed priority ([MixGhost] section 4 with its Table 1 / Appendix C
                                counts): ghost iff 2T^2 (D + p) + 2T^2 < 2TpD + 2pD (ties
                                instantiate); T == 1 -> closed form.  Resolved, never reported. */
} dp_norm_mode;

/* One layer.  Linear uses B, T, d, p; conv2d uses B, Cin, H, W, p, k, stride, pad, dil
 * (square kernel; Hout = (H + 2 pad - dil (k-1) - 1)/stride + 1, likewise Wout); conv1d
 * uses B, Cin, W (the length), p, k, stride, pad, dil (A [B, Cin, W], G [B, p, Wout],
 * weight gradient [p, Cin, k]; H is ignored); conv3d adds the input depth Z (A [B, Cin,
 * Z, H, W], G [B, p, Zout, Hout, Wout], a cubic kernel, weight gradient [p, Cin, k, k, k]). */
typedef struct {
  int kind;      /* dp_kind */
  int dtype;     /* dp_dtype of A and G */
  int B;         /* examples */
  int T, d, p;   /* linear: rows per example, in features; p = out features / channels */
  int Cin, H, W, k, stride, pad, dil;
  int has_bias;  /* 1: the bias gradient joins the norm and the sum */
  int Z;         /* conv3d: input depth (ignored otherwise) */
  int layout;    /* conv layers: dp_layout of A and G (ignored for linear layers) */
} dp_layer_desc;

/* ABI version (DPCLIP_ABI_VERSION).  Host only. */
int dp_abi_version(void);

/* Number of kernels this library has launched in the process so far (all devices and
 * streams).  Host only; for accounting launches in a timed region. */
unsigned long long dp_launch_count(void);

/* Message for the last non-DP_OK status returned on this thread ("" if none). Host only. */
const char* dp_last_error(void);

/* Host-only planner: validates `desc`, resolves `requested` (DP_NORM_AUTO applies the
 * layerwise rule of [MixGhost] eq. 4.1 -- the smaller of the ghost space 2T^2 and the
 * instantiation space p*D, Appendix F; DP_NORM_AUTO_TIME compares the time counts
 * instead) and reports the rows T and width D of the
 * per-example contraction.  Any output pointer may be NULL.  Needs no GPU. */
dp_status dp_plan(const dp_layer_desc* desc, int requested, int* chosen_mode, int* rows_T,
                  int* width_D);

/* Bytes of workspace dp_layer_sqnorms / dp_clipped_sum need for `desc` (0 if invalid).
 * `mode` is the requested norm mode for dp_layer_sqnorms; the clipped sum's need is
 * included.  Host only. */
size_t dp_workspace_size(const dp_layer_desc* desc, int mode);

/* Per-example squared gradient norm of one layer:
 *   sqnorm_out[i] = ||dL_i/dW||_F^2 + has_bias * ||dL_i/db||^2,   i < B   (fp32, device)
 * dL_i/dW = G_i^T A_i (linear, [MixGhost] eq. 2.4) or F^{-1}(G_i)^T U(A_i) (conv,
 * eq. 2.6); formed by the ghost norm (eq. 2.7: sum_{t,s} (U U^T)_{ts} (G G^T)_{ts}),
 * by instantiation on chip, or by the one-row closed form ||a||^2 ||g||^2
 * ([FastClip] eq. 6), per `mode`.  chosen_mode_out (host int, may be NULL) receives
 * the mode used.  workspace: device, >= dp_workspace_size(desc, mode) bytes. */
dp_status dp_layer_sqnorms(const dp_layer_desc* desc, const void* A, const void* G, int mode,
                           float* sqnorm_out, int* chosen_mode_out, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/* dp_layer_sqnorms without a workspace argument, for callers that cannot allocate
 * device memory: code that runs inside another framework's hook or callback and has
 * no handle on that framework's allocator, so it must not call cudaMalloc behind its
 * back (cudaMalloc and cudaFree synchronize the device and the memory escapes the
 * framework's accounting), or a latency-bound loop that cannot afford that device-wide
 * synchronization.  The pages have no counterpart: it changes where the scratch lives,
 * not what is computed.
 * Same arguments and results as dp_layer_sqnorms, minus the workspace.  The ghost and
 * instantiation kernels keep their partial sums in a 4 MiB array the library owns
 * (one per GPU that loads the library, held until the process exits); a layer whose
 * partials need more returns DP_ERR_UNSUPPORTED and launches nothing.  Allocates
 * nothing.  The first call on a device looks up that array's address with the device
 * current (make it before any stream capture) and keeps it for the life of the process:
 * after a cudaDeviceReset (or any reset of the device's primary context) the kept
 * address is stale, so do not call this entry point again in a process that reset the
 * device.  Every call shares the array: calls that overlap on the GPU (other streams,
 * other threads) race and give wrong norms; serialize them.  Each call writes every
 * partial it reads, so what an earlier call left in the array does not matter. */
dp_status dp_layer_sqnorms_noalloc(const dp_layer_desc* desc, const void* A, const void* G,
                                   int mode, float* sqnorm_out, int* chosen_mode_out,
                                   cudaStream_t stream);

/* Clip factors ([FastClip] section 2, clip_c; [MixGhost] Appendix C, min(R/||g||, 1)).
 * sqnorms: device fp32 [L, B] (row l = one layer's sqnorm_out).
 * per_layer = 0 (flat): n_i = sqrt(sum_l sqnorms[l,i]); factors_out[i] = 1 if n_i <= C[0]
 *   else C[0]/n_i; factors_out is [B].
 * per_layer = 1 ([ThreeTools] section 2): factors_out[l,i] from n_{l,i} and C[l]; [L, B].
 * C: HOST array of 1 (flat) or L (per-layer) bounds, each > 0.
 * A non-finite n gives factor 0 and sets DP_ERR_NONFINITE in the device status. */
dp_status dp_clip_factors(const float* sqnorms, int B, int L, int per_layer, const float* C,
                          float* factors_out, cudaStream_t stream);

/* Clipped sum of one layer, as one reweighted contraction ([FastClip] section 5, the
 * reweighted loss; [MixGhost] section 3.2, the second back-propagation):
 *   dW[j, m] (+)= sum_i factors[i] * (dL_i/dW)[j, m]        fp32 [p, D], device
 *   db[j]    (+)= sum_i factors[i] * sum_t G_i[t, j]        fp32 [p], device (NULL: skipped)
 * factors: device fp32 [B] (a row of dp_clip_factors' output).  accumulate = 0 writes,
 * 1 adds to the existing dW/db (gradient accumulation over micro-batches).
 * An example whose norm overflowed but whose inputs are finite gets factor 0 from
 * dp_clip_factors and adds nothing.  An example whose A or G hold inf or NaN (factor 0,
 * DP_ERR_NONFINITE raised by dp_clip_factors) still meets the contraction: exactly the
 * outputs it reaches through a non-finite value become NaN (0 * inf: row j of dW and db[j]
 * for a non-finite G_i[t, j], column m of dW for a non-finite A_i[t, m]); every other entry
 * is the sum over the remaining examples.  A caller that sees the status discards the step.
 * workspace: device, >= dp_workspace_size(desc, 0) bytes. */
dp_status dp_clipped_sum(const dp_layer_desc* desc, const void* A, const void* G,
                         const float* factors, float* dW, float* db, int accumulate,
                         void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Gaussian mechanism and average ([FastClip] section 2; [MixGhost] eq. 2.1):
 *   grad[j] = (grad[j] + sigma * C * z_{offset + j}) / B,   j < n   (fp32, device, in place)
 * z_e is the standard normal of element e of Philox4x32-10 (Salmon et al., SC'11)
 * stream 0 under `seed`, through Box-Muller:
 *   counter (e/4 low, e/4 high, 0, 0), key (seed low, seed high); u_k = (x_k>>9 + 1/2)/2^23;
 *   z0,z1 = sqrt(-2 ln u0)(cos, sin)(2 pi u1); z2,z3 likewise from u2,u3; e takes z_{e mod 4}.
 * The words are exact; z is evaluated in fp32 (the angle's sine and cosine by the hardware
 * approximations) within 1e-5 |z| + 4e-6 of the exact transform.
 * Use offset = the first index of this buffer in the flat parameter vector so that
 * every parameter draws its own normal. */
dp_status dp_add_noise(float* grad, size_t n, float sigma, float C, int B, uint64_t seed,
                       uint64_t offset, cudaStream_t stream);

/* dp_add_noise with the seed read from device memory (*seed_dev, a 64-bit value) when
 * the kernel runs, so that a captured CUDA graph draws fresh noise on every replay
 * after the caller updates *seed_dev.  Same noise definition as dp_add_noise. */
dp_status dp_add_noise_devseed(float* grad, size_t n, float sigma, float C, int B,
                               const unsigned long long* seed_dev, uint64_t offset,
                               cudaStream_t stream);

/* The noise pass of dp_add_noise over several blocks of one flat gradient in one launch,
 * each block with its own bound (per-layer clipping, [ThreeTools] section 2):
 *   grad[o_b + j] = (grad[o_b + j] + sigma * C_b * z_{o_b + j}) / B,   j < n_b,
 * with z as dp_add_noise defines it and o_b the block's flat index (grad points to the flat
 * vector's element 0).  Bit-identical to one dp_add_noise call per block.  blocks: host
 * array of 1..64 blocks in increasing offset order, not overlapping (DP_ERR_INVALID_ARG
 * otherwise, or for B <= 0 or a negative or non-finite sigma or C_b).  seed_dev non-NULL: the
 * seed is read from device memory when the kernel runs, seed is then ignored. */
typedef struct {
  uint64_t offset;   /* flat index of the block's first element */
  uint64_t n;        /* elements */
  float C;           /* the block's bound */
} dp_noise_block;
dp_status dp_add_noise_blocks(float* grad, const dp_noise_block* blocks, int nblocks, float sigma, int B,
                              uint64_t seed, const unsigned long long* seed_dev, cudaStream_t stream);

/* Adaptive clipping bound of one layer ([ThreeTools] section 3):
 *   C_next = alpha/B * (sum_i min(sqrt(sqnorms[i]), C_l2) + sigma_l2 * C_l2 * z),
 *   C_l2_next = beta * C_next,
 * z = element `layer` of noise stream 1 (counter word 2 = 1) under `seed`.
 * sqnorms: device fp32 [B].  out: device fp32 [2] = {C_next, C_l2_next}.
 * A non-finite norm sets DP_ERR_NONFINITE in the device status word (read it with
 * dp_check_status) and enters the sum as the bound C_l2 (min(inf, C_l2)). */
dp_status dp_adaptive_bound(const float* sqnorms, int B, float C_l2, float alpha, float beta,
                            float sigma_l2, uint64_t seed, int layer, float* out,
                            cudaStream_t stream);

/* dp_adaptive_bound of layers layer0 .. layer0 + L - 1 in one launch (1 <= L <= 64,
 * [ThreeTools] section 3): the k-th of them reads sqnorms[k*B .. k*B + B - 1] (device fp32
 * [L, B]) and its bound C_l2[k] (host array of L, each finite and > 0) and writes
 * out[2k] = C_next, out[2k + 1] = C_l2_next (device fp32 [L, 2]); its z is element
 * layer0 + k of noise stream 1 under the seed.  Equal, bit for bit, to L dp_adaptive_bound
 * calls with layer = layer0 + k.  seed_dev non-NULL: the seed is read from device memory (a
 * 64-bit value) when the kernel runs, seed is then ignored (for a captured step replayed
 * with a new seed).  DP_ERR_INVALID_ARG for NULL pointers, B <= 0, layer0 < 0, L out of
 * range or bad bounds; a non-finite norm as in dp_adaptive_bound. */
dp_status dp_adaptive_bounds(const float* sqnorms, int B, int layer0, int L, const float* C_l2, float alpha,
                             float beta, float sigma_l2, uint64_t seed, const unsigned long long* seed_dev,
                             float* out, cudaStream_t stream);

/* ---- A layout shared by a layer's norm and sum calls ---------------------------------
 * Conv layers on the im2col kernels work on an NHWC copy of the input, which both the norm
 * and the sum call write at the front of the workspace.  dp_clipped_sum_reuse is
 * dp_clipped_sum for a call whose `workspace` is the one this layer's dp_layer_sqnorms call
 * (with `norm_mode`, the same desc, A and G) used, untouched since: it reads that copy
 * instead of writing it again.  Results are undefined if anything else wrote the workspace
 * in between.  dp_layout_reused reports, for aligned bf16 inputs, 1 when the copy is
 * reused and 0 when the call is plain dp_clipped_sum.  Host only. */
dp_status dp_clipped_sum_reuse(const dp_layer_desc* desc, int norm_mode, const void* A, const void* G,
                               const float* factors, float* dW, float* db, int accumulate, void* workspace,
                               size_t ws_bytes, cudaStream_t stream);
int dp_layout_reused(const dp_layer_desc* desc, int norm_mode);

/* ---- Kept per-example gradients (instantiated layers) --------------------------------
 * Where a layer's norm is formed by instantiation ([MixGhost] section 3, the FastGradClip
 * side of the mixed clipping), the instantiating kernel can also store every example's
 * gradient g_i and bias gradient b_i; the clipped sum is then the weighted gradient
 * sum_i c_i g_i of the stored gradients, as in the Opacus approach of [MixGhost] section 2
 * (2pD flop per example, Appendix C.5; one read) instead of a second contraction over the
 * T rows (2TpD).  It trades B*(p*D + p)*4 bytes of device memory for that time, and pays
 * off when T is large (a few hundred rows and up).
 *
 * dp_grads_size: bytes of the `grads` buffer for `desc` (fp32, an internal layout), or 0
 * when the layer's instantiated norm does not run on a kernel that keeps gradients (it
 * needs bf16 inputs and the tensor-core shapes; T == 1 layers are excluded).  Host only.
 *
 * dp_layer_sqnorms_keep: the instantiated norm of dp_layer_sqnorms (sqnorm_out [B], as with
 * DP_NORM_INSTANTIATE) that also writes every example's gradient into `grads` (device,
 * 16-byte aligned, dp_grads_size bytes, caller-owned).  A, G and the workspace must be
 * 16-byte aligned; otherwise DP_ERR_UNSUPPORTED and nothing is launched.  Workspace as
 * dp_workspace_size(desc, DP_NORM_INSTANTIATE).
 *
 * dp_clipped_sum_kept: dW (+)= sum_i factors[i] g_i, db (+)= sum_i factors[i] b_i from a
 * `grads` buffer that dp_layer_sqnorms_keep filled for the same `desc`; same output layout,
 * accumulate flag and determinism as dp_clipped_sum.  Workspace as dp_workspace_size. */
size_t dp_grads_size(const dp_layer_desc* desc);
dp_status dp_layer_sqnorms_keep(const dp_layer_desc* desc, const void* A, const void* G, float* sqnorm_out,
                                float* grads, void* workspace, size_t ws_bytes, cudaStream_t stream);
dp_status dp_clipped_sum_kept(const dp_layer_desc* desc, const float* grads, const float* factors, float* dW,
                              float* db, int accumulate, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ---- The clipped sum and the noise in one call ---------------------------------------
 * The Gaussian mechanism and average of dp_add_noise applied to this layer's blocks of the
 * flat gradient right after its clipped sum:
 *   dW[j] = (S_W[j] + sigma * C * z_{offset + j}) / B,       j < p*D
 *   db[j] = (S_b[j] + sigma * C * z_{offset + p*D + j}) / B, j < p
 * S = the clipped sum of dp_clipped_sum (norm_mode = -1), of dp_clipped_sum_reuse
 * (norm_mode >= 0: the layout reuse described above) or of dp_clipped_sum_kept, plus the
 * old contents of dW/db when accumulate = 1; z as dp_add_noise defines it, `offset` = the
 * index of dW[0] in the flat parameter vector (db[0] follows at offset + p*D).  Where the sum
 * ends in a reduction of example splits, that pass adds the noise (one pass over the
 * gradient less); otherwise the noise pass follows in the same call.  Either way the
 * result is bit-identical to the sum call followed by dp_add_noise on the same blocks.
 * seed_dev non-NULL: the seed is read from device memory when the kernels run (as
 * dp_add_noise_devseed), seed is then ignored.  Arguments, workspace and errors otherwise
 * as the sum call; DP_ERR_INVALID_ARG for B <= 0 or a negative or non-finite sigma or C. */
typedef struct {
  float sigma, C;                       /* the noise standard deviation is sigma * C */
  int B;                                /* the divisor (the logical batch size) */
  uint64_t seed;                        /* Philox key */
  const unsigned long long* seed_dev;   /* device, or NULL */
  uint64_t offset;                      /* flat index of dW[0] */
} dp_noise_desc;
dp_status dp_clipped_sum_noised(const dp_layer_desc* desc, int norm_mode, const void* A, const void* G,
                                const float* factors, float* dW, float* db, int accumulate,
                                const dp_noise_desc* noise, void* workspace, size_t ws_bytes,
                                cudaStream_t stream);
dp_status dp_clipped_sum_kept_noised(const dp_layer_desc* desc, const float* grads, const float* factors,
                                     float* dW, float* db, int accumulate, const dp_noise_desc* noise,
                                     void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Synchronizes `stream`, returns the device status word (DP_OK, DP_ERR_NONFINITE or
 * DP_ERR_TIMEOUT) raised since the last check, and clears it. */
dp_status dp_check_status(cudaStream_t stream);

/* Diagnostic of the device-side failure path.  Launches (asynchronously, on `stream`)
 * one kernel that allocates tensor memory and waits on an mbarrier nothing arrives on:
 * the bounded wait gives up after the device wait limit (2 s), raises DP_ERR_TIMEOUT in
 * the device status word (read it with dp_check_status), and the kernel releases its
 * tensor memory as the tensor-core kernels do after a timeout and returns; the context
 * stays usable.  If `waited_ns` (device, one value) is non-NULL it receives the time the
 * kernel spent from the start of the wait to the release, in ns.  Returns DP_ERR_CUDA if
 * the launch fails. */
dp_status dp_selftest_wait_timeout(unsigned long long* waited_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DPCLIP_H */
