// gma_internal.cuh -- definitions shared by the CUDA translation units of libgma.so.
//
// Nothing here is part of the public ABI (that is include/gma.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gma.h"

namespace gma {

// ------------------------------------------------------------------ workspace header
// The first 256 bytes of every workspace.  `error` holds the first device-side condition that a
// kernel recorded (a gma_status_t), `detail` a kernel-specific code for diagnostics.
// reserved[0] != 0 asks the bounded waits for their short limit (GMA_FLAG_TEST_WITHHOLD).
struct WsHeader {
    unsigned error;
    unsigned detail;
    unsigned reserved[62];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

__device__ __forceinline__ void record_error(WsHeader *hdr, unsigned code, unsigned detail)
{
    if (atomicCAS(&hdr->error, 0u, code) == 0u) hdr->detail = detail;
}

// ------------------------------------------------------------------ element access
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v)
{
    return __bfloat162float(v);
}

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

// ------------------------------------------------------------------ host-side helpers
static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A linear allocator over a caller-provided workspace: offsets only, no allocation.
struct Carve {
    size_t off = sizeof(WsHeader);
    size_t take(size_t bytes)
    {
        size_t at = align_up(off, 256);
        off = at + bytes;
        return at;
    }
    size_t total() const { return align_up(off, 256); }
};

inline bool valid_dim(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// ------------------------------------------------------------------ optional launch timing
// When enabled through gma_timing_enable, every kernel launch of the library is bracketed by a
// pair of CUDA events recorded on the launching stream; gma_timing_read returns the durations.
// Kernel ids name the launch sites (kernel_name gives the string).
enum KernelId {
    KID_SIMT_PARAMS = 1, KID_SIMT_RESP, KID_SIMT_STATE, KID_SIMT_SCAN, KID_SIMT_OUT, KID_SIMT_SMALL,
    KID_TC_PARAMS = 16, KID_TC_RESP, KID_TC_BIDIR_WRITE, KID_TC_BIDIR_READ, KID_TC_CAUSAL_AGG,
    KID_TC_CAUSAL_SCAN, KID_TC_CAUSAL_OUT, KID_TC_LSE, KID_TC_DIVIDE, KID_TC_CAUSAL_FUSED, KID_DECODE = 32, KID_DECODE_PARAMS, KID_USAGE_ROWS, KID_USAGE_MASS, KID_USAGE_STATS, KID_BWD_NUMDEN,
    KID_BWD_DQ, KID_BWD_SCAN, KID_BWD_DK, KID_BWD_DX, KID_BWD_PARAMS, KID_BWD_PFINAL, KID_COUNT
};
const char *kernel_name(int id);
void timing_begin(cudaStream_t st, int kernel_id);
void timing_end(cudaStream_t st);

// Launch with programmatic stream serialisation: the kernel may start once the kernel ahead of
// it in the stream has let it (griddepcontrol.launch_dependents) or finished; it must execute
// griddepcontrol.wait before it reads anything that kernel writes.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

// --------------------------------------------------------------- fp32 CUDA-core kernel family
size_t simt_workspace_size(const gma_shape_t &s, int variant);
gma_status_t simt_responsibilities(const gma_shape_t &s, const void *X, const float *mu,
                                   const float *raw, const float *logits, void *gamma, void *ws,
                                   cudaStream_t st);
// s.N queries and n_k keys per slice (n_k == s.N but for cross-attention, which is bidirectional).
gma_status_t simt_forward(const gma_shape_t &s, bool causal, int n_k, const void *QX, const void *KX,
                          const void *V, const float *mu, const float *raw, const float *logits,
                          void *O, void *ws, cudaStream_t st);
size_t simt_workspace_size_cross(const gma_shape_t &s, int n_k);
// The read phase's inputs (fp32 CUDA cores, direct form): per-head 1/sigma^2 [H][K][d_r] followed by
// mu^T, (1/sigma^2)^T, (1/sigma)^T and (-mu/sigma)^T [H][d_r][K] (iv holds 5 H K d_r floats), and
// constants [H][K]; Gamma_Q, Gamma_K [B*H*N][K]; segment memories [B*H][ceil(N/64)][K][d_v+1],
// scanned (causal: exclusive prefix per 64-token segment; bidirectional: the total in segment 0).
gma_status_t simt_prepare(const gma_shape_t &s, bool causal, const void *QX, const void *KX, const void *V,
                          const float *mu, const float *raw, const float *logits, float *iv, float *cst, float *gq,
                          float *gk, float *agg, cudaStream_t st);

// --------------------------------------------------------------- backward pass
size_t backward_workspace_size(const gma_shape_t &s);
gma_status_t backward(const gma_shape_t &s, bool causal, const void *QX, const void *KX, const void *V,
                      const float *mu, const float *raw, const float *logits, const void *dO, void *dQX, void *dKX,
                      void *dV, float *dmu, float *draw, float *dlogits, void *ws, cudaStream_t st);

// --------------------------------------------------------------- decode step
size_t decode_workspace_size(const gma_shape_t &s);
gma_status_t decode_step(const gma_shape_t &s, const void *qx, const void *kx, const void *v, const float *mu,
                         const float *raw, const float *logits, float *state, void *o, void *ws, cudaStream_t st);

// --------------------------------------------------------------- usage diagnostics
size_t usage_workspace_size(const gma_shape_t &s);
gma_status_t usage(const gma_shape_t &s, const void *X, const float *mu, const float *raw, const float *logits,
                   int *assign, int *counts, float *mass, int *used, float *entropy, void *ws, cudaStream_t st);

// --------------------------------------------------------------- tcgen05 kernel family
bool tc_supported(const gma_shape_t &s, int variant);
size_t tc_workspace_size(const gma_shape_t &s, int variant);
gma_status_t tc_responsibilities(const gma_shape_t &s, const void *X, const float *mu,
                                 const float *raw, const float *logits, void *gamma, void *ws,
                                 cudaStream_t st);
gma_status_t tc_forward(const gma_shape_t &s, bool causal, int n_k, const void *QX, const void *KX,
                        const void *V, const float *mu, const float *raw, const float *logits,
                        void *O, void *ws, cudaStream_t st);
size_t tc_workspace_size_cross(const gma_shape_t &s, int n_k);
// Usage diagnostics fused into the tensor-core responsibilities pass: per row the argmax, the
// per-head histogram (atomic adds into counts, zeroed by the caller), and per-CTA sums of the
// responsibilities mass_part [B*H*tc_usage_blocks(s)][K] (CTA = slice * blocks + block).
int tc_usage_blocks(const gma_shape_t &s);
gma_status_t tc_usage(const gma_shape_t &s, const void *X, const float *mu, const float *raw, const float *logits,
                      int *assign, int *counts, float *mass_part, void *ws, cudaStream_t st);

}  // namespace gma

// Launch helper: timing brackets plus the launch-error check.
#define GMA_LAUNCH(kid, st, ...)                                                              \
    do {                                                                                      \
        ::gma::timing_begin((st), (kid));                                                     \
        __VA_ARGS__;                                                                          \
        ::gma::timing_end((st));                                                              \
        if (cudaPeekAtLastError() != cudaSuccess) return GMA_ERR_CUDA;                        \
    } while (0)
