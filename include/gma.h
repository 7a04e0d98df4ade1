/*
 * gma.h -- C ABI of libgma.so: the forward pass of Gaussian Mixture Attention (GMA) on an
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (page "Attention par Mélange Gaussien (GMA)", gist.science/fr/paper/2606.18283):
 *
 *   Méthodologie §1 "Routage Latent Probabiliste": each routing vector x (a row of Q_X or K_X)
 *     is mapped to its GMM posterior responsibilities gamma_k = p(z = k | x) over K learned
 *     diagonal Gaussians with means mu_k, variances Sigma_k and priors pi_k.
 *   Méthodologie §3 "Variantes et Entraînement": variances through softplus, priors through
 *     softmax.  Here  sigma^2 = softplus(raw_var) + var_floor  and  pi = softmax(prior_logits).
 *   Méthodologie §2 "Routage de Mémoire Latente": keys write a K-slot memory
 *     V~ = Gamma_K^T V and a normaliser Z = Gamma_K^T 1; queries read it through the page's
 *     displayed equation  O = Gamma_Q V~ / (Gamma_Q Z + eps).
 *   Méthodologie §3: the causal variant replaces V~ and Z by prefix sums, so that row i of O
 *     depends only on keys j <= i (inclusive).
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, row-major and contiguous, in DEVICE memory of the current CUDA
 *     device, 16-byte aligned:
 *       Q_X, K_X      [B][H][N][d_r]    dtype (bf16 or fp32)
 *       V             [B][H][N][d_v]    dtype
 *       O             [B][H][N][d_v]    dtype (fp32 if GMA_FLAG_OUT_F32)
 *       gamma         [B][H][N][K]      dtype (fp32 if GMA_FLAG_OUT_F32)
 *       mu, raw_var   [H][K][d_r]       fp32   (one GMM per head, shared by queries, keys and
 *                                               the whole batch)
 *       prior_logits  [H][K]            fp32
 *   - The caller owns and allocates every buffer, including the workspace (size from
 *     gma_workspace_size).  The library never allocates, frees or synchronises inside these
 *     calls: all work is enqueued on `stream` (NULL = the legacy default stream) and the call
 *     returns without waiting for it.
 *   - The workspace needs no initialisation: the library clears what it must on `stream`.
 *     Calls that share one workspace must be ordered on the GPU (same stream, or events).
 *   - Argument and shape errors return before anything is enqueued.  A failed kernel launch
 *     returns GMA_ERR_CUDA.  Conditions found on the device (parameters outside the range the
 *     tensor-core path can represent, a bounded wait that timed out) are recorded in the
 *     workspace's error word and reported by gma_check_workspace; the library never traps.
 *   - Supported sizes: B, H, N >= 1; d_r, d_v in {16, 32, 64, 128}; 1 <= K <= 1024;
 *     B*H*N*max(d_r, d_v, K) < 2^31.  Inputs must be finite and |x| < 256 for bf16 inputs.
 */
#ifndef GMA_H
#define GMA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t. */
typedef struct CUstream_st *gma_stream_t;

typedef enum {
    GMA_OK = 0,
    GMA_ERR_INVALID_ARG = 1,       /* null or misaligned pointer, non-positive size, bad eps  */
    GMA_ERR_UNSUPPORTED_SHAPE = 2, /* d_r, d_v or K outside the supported set               */
    GMA_ERR_RANGE = 3,             /* device: a reparametrised parameter exceeds fp16 range  */
    GMA_ERR_WORKSPACE = 4,         /* workspace null, misaligned or smaller than required    */
    GMA_ERR_CUDA = 5,              /* a CUDA runtime call or kernel launch failed            */
    GMA_ERR_TIMEOUT = 6,           /* device: a bounded wait gave up                         */
    GMA_ERR_NO_DEVICE = 7          /* no usable sm_103 device is current                     */
} gma_status_t;

typedef enum { GMA_F32 = 0, GMA_BF16 = 1 } gma_dtype_t;

/* Bits of gma_shape_t.flags. */
#define GMA_FLAG_SIMT 0x1u     /* force the fp32 CUDA-core kernels (the path fp32 inputs take) */
#define GMA_FLAG_OUT_F32 0x2u  /* write O (or gamma) as fp32 even for bf16 inputs              */
#define GMA_FLAG_RECOMPUTE_KEYS 0x4u /* causal, tensor-core path: recompute the key
                                      * responsibilities in the output pass instead of keeping
                                      * them in the workspace (smaller workspace, slower)     */
#define GMA_FLAG_SINGLE_PASS 0x8u /* causal, tensor-core path: the fused variant (page's
                                   * Méthodologie §2-§3): one kernel launch after the parameter
                                   * kernel, the responsibilities never written to memory.
                                   * Each CTA sweeps its segment's keys for the segment's own
                                   * memory, exchanges memories with the preceding segments of
                                   * its slice through the workspace (decoupled look-back, every
                                   * wait bounded), then runs the output sweep.  Needs K <= 128
                                   * and a shape the tensor-core family covers: otherwise the
                                   * call returns GMA_ERR_UNSUPPORTED_SHAPE.  Other entry points
                                   * ignore it.                                              */
#define GMA_FLAG_TEST_WITHHOLD 0x80000000u
/* For tests of the device-side timeout path only; never set it in production.  The call's
 * bounded waits give up after about a millisecond instead of a second, and the tensor-core
 * causal and bidirectional key passes withhold one row-phase hand-off (the signal that the
 * first chunk's [x^2, x] tile is built), so the waits on it run out: every role of the kernel
 * leaves its loop, tensor memory is released, and gma_check_workspace then reports
 * GMA_ERR_TIMEOUT.  With GMA_FLAG_SINGLE_PASS only the first segment of each slice withholds
 * it; the other segments learn of its failure through the look-back and stop.  The output of
 * such a call is undefined; the next call without the flag on the same stream runs normally. */

typedef struct {
    int B, H, N;     /* batch, heads, sequence length                                       */
    int d_r;         /* routing dimension (columns of Q_X and K_X)                          */
    int K;           /* number of Gaussian components                                       */
    int d_v;         /* value dimension                                                     */
    int dtype;       /* gma_dtype_t of Q_X, K_X, V and the output                           */
    float eps;       /* added to every query row's normaliser Gamma_Q Z; eps >= 0           */
    float var_floor; /* sigma^2 = softplus(raw_var) + var_floor; var_floor >= 0             */
    unsigned flags;  /* GMA_FLAG_* bits                                                     */
} gma_shape_t;

/* Variants for gma_workspace_size. */
#define GMA_VARIANT_RESPONSIBILITIES 0
#define GMA_VARIANT_BIDIRECTIONAL 1
#define GMA_VARIANT_CAUSAL 2
#define GMA_VARIANT_DECODE 3
#define GMA_VARIANT_USAGE 4
#define GMA_VARIANT_BACKWARD 5

/* Bytes of device workspace one call of `variant` with `shape` needs (0 for an invalid shape).
 * The workspace must be 256-byte aligned.  Its first 256 bytes hold the error word that
 * gma_check_workspace reads.  For the causal variant on the tensor-core path (bf16, no
 * GMA_FLAG_SIMT) it includes the key responsibilities of every token, B*H*N*Kp bf16 values
 * (Kp = 64 for K <= 64, else 128), unless GMA_FLAG_RECOMPUTE_KEYS or GMA_FLAG_SINGLE_PASS is
 * set; with GMA_FLAG_SINGLE_PASS it holds instead a segment counter, one flag per segment and the
 * segments' inclusive prefix memories (the call zeroes the counter and flags).  With K > 128 on the
 * tensor-core path (components in tiles of 128) it also holds every routing row's log-sum-exp
 * over all components (fp32) and, for the forward passes, fp32 partial sums of the queries'
 * numerators and normalisers (B*H*N*(d_v + 1) floats). */
size_t gma_workspace_size(const gma_shape_t *shape, int variant);

/* Posterior responsibilities (Méthodologie §1):
 *   gamma[b][h][i][k] = p(z = k | X[b][h][i]) under head h's GMM.
 * X [B][H][N][d_r] dtype; gamma [B][H][N][K] dtype (fp32 with GMA_FLAG_OUT_F32).
 * shape->d_v and shape->eps are ignored. */
gma_status_t gma_responsibilities(const gma_shape_t *shape, const void *X, const float *mu,
                                  const float *raw_var, const float *prior_logits, void *gamma,
                                  void *workspace, size_t workspace_bytes, gma_stream_t stream);

/* Bidirectional GMA (Méthodologie §2):
 *   V~ = Gamma_K^T V,  Z = Gamma_K^T 1,  O = Gamma_Q V~ / (Gamma_Q Z + eps)
 * per (b, h) slice, over the whole sequence. */
gma_status_t gma_forward_bidirectional(const gma_shape_t *shape, const void *QX, const void *KX,
                                       const void *V, const float *mu, const float *raw_var,
                                       const float *prior_logits, void *O, void *workspace,
                                       size_t workspace_bytes, gma_stream_t stream);

/* Causal GMA (Méthodologie §3): as above with V~ and Z replaced by inclusive prefix sums,
 *   O_i = gamma_Q,i (sum_{j<=i} gamma_K,j^T v_j) / (gamma_Q,i . sum_{j<=i} gamma_K,j + eps).
 * Repeated calls on the same inputs give the same bits, except with GMA_FLAG_SINGLE_PASS: its
 * segments add their predecessors' memories in the order they find them published, so the
 * rounding can differ from call to call. */
gma_status_t gma_forward_causal(const gma_shape_t *shape, const void *QX, const void *KX,
                                const void *V, const float *mu, const float *raw_var,
                                const float *prior_logits, void *O, void *workspace,
                                size_t workspace_bytes, gma_stream_t stream);

/* One autoregressive decode step of causal GMA (Méthodologie §3: the prefix memory V~ and its
 * normaliser Z grow by one token, which then reads them), for every (b, h) slice at once:
 *   gamma_K = p(z | kx),   S[k][c] += gamma_K[k] v[c] (c < d_v),   S[k][d_v] += gamma_K[k],
 *   gamma_Q = p(z | qx),   o[c] = (gamma_Q . S[:, c]) / (gamma_Q . S[:, d_v] + eps).
 * shape->N must be 1 (one new token per slice).  qx, kx [B][H][d_r] and v [B][H][d_v] in
 * shape->dtype; state [B][H][K][d_v + 1] fp32, caller-owned, read and updated in place (all zeros
 * for an empty prefix; after N steps it equals the causal forward's memory after N tokens);
 * o [B][H][d_v] in shape->dtype (fp32 with GMA_FLAG_OUT_F32).  fp32 arithmetic on the CUDA cores
 * for every shape; the workspace is gma_workspace_size(shape, GMA_VARIANT_DECODE) bytes. */
gma_status_t gma_decode_step(const gma_shape_t *shape, const void *qx, const void *kx, const void *v,
                             const float *mu, const float *raw_var, const float *prior_logits,
                             float *state, void *o, void *workspace, size_t workspace_bytes,
                             gma_stream_t stream);

/* Backward pass (Méthodologie §3: end-to-end training by backpropagation through the softmax
 * posteriors and the ratio): the gradients of sum(dO * O) for the bidirectional (causal = 0) or
 * causal (causal = 1) forward pass with the same arguments.
 *   dO, and the outputs dQX, dKX [B][H][N][d_r], dV [B][H][N][d_v]: dtype (bf16 or fp32);
 *   dmu, draw_var [H][K][d_r] and dprior_logits [H][K]: fp32, summed over the batch.
 * Every step runs in fp32 on the CUDA cores (the forward's own preparation, then the reverse
 * passes over 64-token segments); gma_kernel_family(shape, GMA_VARIANT_BACKWARD) is 0.  The
 * workspace is gma_workspace_size(shape, GMA_VARIANT_BACKWARD) bytes: fp32 responsibilities and
 * their gradients for every token (4 B*H*N*K floats) and the segment memories.  Outputs are
 * written, not accumulated; results repeat exactly from call to call. */
gma_status_t gma_backward(const gma_shape_t *shape, int causal, const void *QX, const void *KX, const void *V,
                          const float *mu, const float *raw_var, const float *prior_logits, const void *dO,
                          void *dQX, void *dKX, void *dV, float *dmu, float *draw_var, float *dprior_logits,
                          void *workspace, size_t workspace_bytes, gma_stream_t stream);

/* Component-usage diagnostics of the responsibilities of X (Résultats et Performance,
 * interpretability: components used, usage entropy, hard assignments), per head h:
 *   assign [B][H][N] int32  argmax_k gamma_{b,h,i,k}, the lowest k on ties
 *   counts [H][K] int32     tokens assigned to each component (over the batch and the sequence)
 *   mass [H][K] fp32        sum over tokens of gamma_{.,h,.,k}
 *   used [H] int32          components with a non-zero count
 *   entropy [H] fp32        -sum_k p_k ln p_k / ln K with p = counts / (B N); 0 when K = 1
 * X [B][H][N][d_r] dtype; gamma is computed by the family gma_kernel_family(shape,
 * GMA_VARIANT_RESPONSIBILITIES) names (tensor-core logits for bf16 inputs it covers, so a token
 * whose two largest responsibilities nearly tie may be assigned either way), kept in fp32 in the
 * workspace, gma_workspace_size(shape, GMA_VARIANT_USAGE) bytes.  shape->d_v and eps are
 * ignored.  Every output is caller-owned device memory, 16-byte aligned; counts are overwritten. */
gma_status_t gma_usage(const gma_shape_t *shape, const void *X, const float *mu, const float *raw_var,
                       const float *prior_logits, int32_t *assign, int32_t *counts, float *mass,
                       int32_t *used, float *entropy, void *workspace, size_t workspace_bytes,
                       gma_stream_t stream);

/* Cross-attention: bidirectional GMA with a separate key set (Méthodologie §2; the page's
 * Conclusion names cross-attention as future work).  shape->N = N_q queries per slice; n_k keys:
 *   QX [B][H][N_q][d_r], KX [B][H][n_k][d_r], V [B][H][n_k][d_v] (dtype), O [B][H][N_q][d_v];
 *   V~ = Gamma_K^T V, Z = Gamma_K^T 1 over the n_k keys,  O = Gamma_Q V~ / (Gamma_Q Z + eps).
 * The kernel family is that of gma_kernel_family(shape, GMA_VARIANT_BIDIRECTIONAL); the workspace
 * is gma_workspace_size_cross(shape, n_k) bytes (0 for an invalid shape or n_k < 1).  With
 * n_k == shape->N this computes what gma_forward_bidirectional computes. */
size_t gma_workspace_size_cross(const gma_shape_t *shape, int n_k);
gma_status_t gma_forward_cross(const gma_shape_t *shape, int n_k, const void *QX, const void *KX,
                               const void *V, const float *mu, const float *raw_var,
                               const float *prior_logits, void *O, void *workspace,
                               size_t workspace_bytes, gma_stream_t stream);

/* Causal GMA for callers that cannot allocate device memory.  The page has no counterpart to
 * this entry point: it exists for callers such as allocator or memory-pool callbacks, plugins
 * whose host application owns every device allocation, or loops that must not call cudaMalloc
 * after start-up, which can pass inputs and outputs but no workspace.
 *   - Computes exactly what gma_forward_causal computes, with the same arguments minus the
 *     workspace, which comes from a fixed array of GMA_NOALLOC_SCRATCH_BYTES inside the library's
 *     device image.  Every GPU that loads libgma.so holds that array until the process exits.
 *   - If gma_workspace_size(shape, GMA_VARIANT_CAUSAL) exceeds GMA_NOALLOC_SCRATCH_BYTES, the
 *     call runs as if GMA_FLAG_RECOMPUTE_KEYS were set; if that workspace exceeds it too, the
 *     call returns GMA_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device (with that device current) looks up the array's device
 *     address; make that first call before any stream capture.  The address is looked up again
 *     when the current CUDA context changes (after cudaDeviceReset, for instance): make the
 *     first call after such a change outside stream capture too.  No call allocates or frees
 *     memory (no cudaMalloc, cudaFree or allocating library routine).
 *   - All calls on a device share the one array, which keeps the last call's contents; the call
 *     clears what must start at zero.  Calls that overlap on the GPU (other streams, other host
 *     threads) race on the array: order them on one stream or with events.
 *   - Argument, shape and launch errors are returned as usual.  Conditions found on the device
 *     (a parameter outside the range the tensor-core path holds, a bounded wait that timed out)
 *     are recorded in the array's header; gma_noalloc_check reports them. */
#define GMA_NOALLOC_SCRATCH_BYTES (32u << 20)
gma_status_t gma_forward_causal_noalloc(const gma_shape_t *shape, const void *QX, const void *KX,
                                        const void *V, const float *mu, const float *raw_var,
                                        const float *prior_logits, void *O, gma_stream_t stream);

/* gma_check_workspace for the array behind gma_forward_causal_noalloc on the current device:
 * waits for `stream`, then returns the condition the device recorded during the last no-alloc
 * call on this device (GMA_OK if none), or GMA_ERR_CUDA if the stream reported an error.  Like
 * the entry point itself, it allocates nothing. */
gma_status_t gma_noalloc_check(gma_stream_t stream);

/* Waits for `stream`, then returns the condition the device recorded in `workspace` during the
 * last call that used it (GMA_OK if none), or GMA_ERR_CUDA if the stream reported an error. */
gma_status_t gma_check_workspace(const void *workspace, gma_stream_t stream);

/* Which kernel family a call with this shape and variant runs: 0 = fp32 CUDA-core kernels,
 * 1 = tcgen05 tensor-core kernels, -1 = the shape is invalid.  The tensor-core family takes bf16
 * inputs with d_r <= 64 and d_v <= 128 (a multiple of 16) for every K up to 1024; fp32 inputs,
 * d_r = 128 and GMA_FLAG_SIMT take the CUDA cores.  The decode step (N == 1) and the backward
 * pass always run on the CUDA cores. */
int gma_kernel_family(const gma_shape_t *shape, int variant);

/* Static description of a status code. */
const char *gma_status_string(gma_status_t status);

/* Launch timing, for benchmarks.  gma_timing_enable(capacity > 0) creates `capacity` pairs of
 * CUDA events (call it outside stream capture); from then on every kernel launch of the library
 * is bracketed by an event pair recorded on its stream.  gma_timing_enable(0) turns it off.
 * gma_timing_read waits for the recorded launches and copies up to `cap` (kernel id, ms) pairs,
 * oldest first, into caller-owned host arrays, then clears the record; it returns the number
 * copied, or -1 on a CUDA error.  Launches beyond `capacity` are not recorded.
 * gma_kernel_name maps a kernel id to a static string. */
gma_status_t gma_timing_enable(int capacity);
int gma_timing_read(int *kernel_ids, float *ms, int cap);
const char *gma_kernel_name(int kernel_id);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int gma_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GMA_H */
