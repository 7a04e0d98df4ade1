// gma_api.cu -- the extern "C" entry points of libgma.so (declared in include/gma.h):
// argument validation, workspace sizing and the choice of kernel family.
#include <stddef.h>
#include <string.h>

#include "gma_internal.cuh"

using namespace gma;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Validates what every call needs; `variant` selects which sizes matter.
gma_status_t validate_shape(const gma_shape_t *s, int variant)
{
    if (!s) return GMA_ERR_INVALID_ARG;
    if (s->B < 1 || s->H < 1 || s->N < 1 || s->K < 1) return GMA_ERR_INVALID_ARG;
    if (s->dtype != GMA_F32 && s->dtype != GMA_BF16) return GMA_ERR_INVALID_ARG;
    if (!(s->var_floor >= 0.f) || !(s->eps >= 0.f)) return GMA_ERR_INVALID_ARG;
    if (s->flags & ~(GMA_FLAG_SIMT | GMA_FLAG_OUT_F32 | GMA_FLAG_RECOMPUTE_KEYS | GMA_FLAG_SINGLE_PASS |
                     GMA_FLAG_TEST_WITHHOLD))
        return GMA_ERR_INVALID_ARG;
    if (!valid_dim(s->d_r) || s->K > 1024) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (variant != GMA_VARIANT_RESPONSIBILITIES && !valid_dim(s->d_v))
        return GMA_ERR_UNSUPPORTED_SHAPE;
    const long long rows = (long long)s->B * s->H * s->N;
    long long widest = s->d_r > s->K ? s->d_r : s->K;
    if (variant != GMA_VARIANT_RESPONSIBILITIES && s->d_v > widest) widest = s->d_v;
    if (rows * widest >= (1ll << 31)) return GMA_ERR_UNSUPPORTED_SHAPE;
    return GMA_OK;
}

// 1 = tcgen05 tensor-core family (bf16 inputs it covers), 0 = fp32 CUDA-core family.
int family_of(const gma_shape_t &s, int variant) { return tc_supported(s, variant) ? 1 : 0; }

// The single-launch causal variant exists in the tensor-core family only.
bool single_pass_unsupported(const gma_shape_t &s, int variant)
{
    return variant == GMA_VARIANT_CAUSAL && (s.flags & GMA_FLAG_SINGLE_PASS) && family_of(s, variant) != 1;
}

gma_status_t check_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_NO_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return GMA_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return GMA_ERR_NO_DEVICE;
    return GMA_OK;
}

// The word a test-of-timeouts call puts in the header (static storage: the copy reads it after
// the call has returned).
const unsigned kShortWaits = 1u;

gma_status_t begin_call_sized(size_t need, void *ws, size_t ws_bytes, cudaStream_t st, unsigned flags = 0)
{
    if (!ws || ((uintptr_t)ws & 255u)) return GMA_ERR_WORKSPACE;
    if (need == 0 || ws_bytes < need) return GMA_ERR_WORKSPACE;
    gma_status_t d = check_device();
    if (d != GMA_OK) return d;
    if (cudaMemsetAsync(ws, 0, sizeof(WsHeader), st) != cudaSuccess) return GMA_ERR_CUDA;
    if ((flags & GMA_FLAG_TEST_WITHHOLD) &&
        cudaMemcpyAsync((char *)ws + offsetof(WsHeader, reserved), &kShortWaits, sizeof(kShortWaits),
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
        return GMA_ERR_CUDA;
    return GMA_OK;
}

gma_status_t begin_call(const gma_shape_t *s, int variant, void *ws, size_t ws_bytes, cudaStream_t st)
{
    return begin_call_sized(gma_workspace_size(s, variant), ws, ws_bytes, st, s->flags);
}

// The key side of a cross-attention call: the query shape with N = n_k.
gma_status_t validate_cross(const gma_shape_t *s, int n_k, gma_shape_t *sk)
{
    gma_status_t r = validate_shape(s, GMA_VARIANT_BIDIRECTIONAL);
    if (r != GMA_OK) return r;
    if (n_k < 1) return GMA_ERR_INVALID_ARG;
    *sk = *s;
    sk->N = n_k;
    return validate_shape(sk, GMA_VARIANT_BIDIRECTIONAL);
}

gma_status_t forward_common(bool causal, const gma_shape_t *s, const void *QX, const void *KX,
                            const void *V, const float *mu, const float *raw,
                            const float *logits, void *O, void *ws, size_t ws_bytes,
                            gma_stream_t stream)
{
    const int variant = causal ? GMA_VARIANT_CAUSAL : GMA_VARIANT_BIDIRECTIONAL;
    gma_status_t r = validate_shape(s, variant);
    if (r != GMA_OK) return r;
    if (single_pass_unsupported(*s, variant)) return GMA_ERR_UNSUPPORTED_SHAPE;
    const void *ptrs[] = {QX, KX, V, mu, raw, logits, O};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GMA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    r = begin_call(s, variant, ws, ws_bytes, st);
    if (r != GMA_OK) return r;
    if (family_of(*s, variant) == 1)
        return tc_forward(*s, causal, s->N, QX, KX, V, mu, raw, logits, O, ws, st);
    return simt_forward(*s, causal, s->N, QX, KX, V, mu, raw, logits, O, ws, st);
}

}  // namespace

extern "C" {

size_t gma_workspace_size(const gma_shape_t *s, int variant)
{
    if (variant == GMA_VARIANT_DECODE) {
        if (validate_shape(s, GMA_VARIANT_CAUSAL) != GMA_OK || s->N != 1) return 0;
        return decode_workspace_size(*s);
    }
    if (variant == GMA_VARIANT_USAGE) {
        if (validate_shape(s, GMA_VARIANT_RESPONSIBILITIES) != GMA_OK) return 0;
        return usage_workspace_size(*s);
    }
    if (variant == GMA_VARIANT_BACKWARD) {
        if (validate_shape(s, GMA_VARIANT_CAUSAL) != GMA_OK) return 0;
        return backward_workspace_size(*s);
    }
    if (variant < GMA_VARIANT_RESPONSIBILITIES || variant > GMA_VARIANT_CAUSAL) return 0;
    if (validate_shape(s, variant) != GMA_OK || single_pass_unsupported(*s, variant)) return 0;
    return family_of(*s, variant) == 1 ? tc_workspace_size(*s, variant)
                                       : simt_workspace_size(*s, variant);
}

int gma_kernel_family(const gma_shape_t *s, int variant)
{
    if (variant == GMA_VARIANT_DECODE)
        return (validate_shape(s, GMA_VARIANT_CAUSAL) == GMA_OK && s->N == 1) ? 0 : -1;
    if (variant == GMA_VARIANT_USAGE) variant = GMA_VARIANT_RESPONSIBILITIES;
    if (variant == GMA_VARIANT_BACKWARD) return validate_shape(s, GMA_VARIANT_CAUSAL) == GMA_OK ? 0 : -1;
    if (variant < GMA_VARIANT_RESPONSIBILITIES || variant > GMA_VARIANT_CAUSAL) return -1;
    if (validate_shape(s, variant) != GMA_OK || single_pass_unsupported(*s, variant)) return -1;
    return family_of(*s, variant);
}

gma_status_t gma_responsibilities(const gma_shape_t *s, const void *X, const float *mu,
                                  const float *raw, const float *logits, void *gamma, void *ws,
                                  size_t ws_bytes, gma_stream_t stream)
{
    gma_status_t r = validate_shape(s, GMA_VARIANT_RESPONSIBILITIES);
    if (r != GMA_OK) return r;
    const void *ptrs[] = {X, mu, raw, logits, gamma};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GMA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    r = begin_call(s, GMA_VARIANT_RESPONSIBILITIES, ws, ws_bytes, st);
    if (r != GMA_OK) return r;
    if (family_of(*s, GMA_VARIANT_RESPONSIBILITIES) == 1)
        return tc_responsibilities(*s, X, mu, raw, logits, gamma, ws, st);
    return simt_responsibilities(*s, X, mu, raw, logits, gamma, ws, st);
}

gma_status_t gma_forward_bidirectional(const gma_shape_t *s, const void *QX, const void *KX,
                                       const void *V, const float *mu, const float *raw,
                                       const float *logits, void *O, void *ws, size_t ws_bytes,
                                       gma_stream_t stream)
{
    return forward_common(false, s, QX, KX, V, mu, raw, logits, O, ws, ws_bytes, stream);
}

gma_status_t gma_forward_causal(const gma_shape_t *s, const void *QX, const void *KX,
                                const void *V, const float *mu, const float *raw,
                                const float *logits, void *O, void *ws, size_t ws_bytes,
                                gma_stream_t stream)
{
    return forward_common(true, s, QX, KX, V, mu, raw, logits, O, ws, ws_bytes, stream);
}

size_t gma_workspace_size_cross(const gma_shape_t *s, int n_k)
{
    gma_shape_t sk;
    if (validate_cross(s, n_k, &sk) != GMA_OK) return 0;
    return family_of(*s, GMA_VARIANT_BIDIRECTIONAL) == 1 ? tc_workspace_size_cross(*s, n_k)
                                                         : simt_workspace_size_cross(*s, n_k);
}

gma_status_t gma_forward_cross(const gma_shape_t *s, int n_k, const void *QX, const void *KX, const void *V,
                               const float *mu, const float *raw, const float *logits, void *O, void *ws,
                               size_t ws_bytes, gma_stream_t stream)
{
    gma_shape_t sk;
    gma_status_t r = validate_cross(s, n_k, &sk);
    if (r != GMA_OK) return r;
    const void *ptrs[] = {QX, KX, V, mu, raw, logits, O};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GMA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    r = begin_call_sized(gma_workspace_size_cross(s, n_k), ws, ws_bytes, st);
    if (r != GMA_OK) return r;
    if (family_of(*s, GMA_VARIANT_BIDIRECTIONAL) == 1)
        return tc_forward(*s, false, n_k, QX, KX, V, mu, raw, logits, O, ws, st);
    return simt_forward(*s, false, n_k, QX, KX, V, mu, raw, logits, O, ws, st);
}

gma_status_t gma_backward(const gma_shape_t *s, int causal, const void *QX, const void *KX, const void *V,
                          const float *mu, const float *raw, const float *logits, const void *dO, void *dQX, void *dKX,
                          void *dV, float *dmu, float *draw, float *dlogits, void *ws, size_t ws_bytes,
                          gma_stream_t stream)
{
    gma_status_t r = validate_shape(s, GMA_VARIANT_CAUSAL);
    if (r != GMA_OK) return r;
    if (causal != 0 && causal != 1) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {QX, KX, V, mu, raw, logits, dO, dQX, dKX, dV, dmu, draw, dlogits};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GMA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    r = begin_call(s, GMA_VARIANT_BACKWARD, ws, ws_bytes, st);
    if (r != GMA_OK) return r;
    return backward(*s, causal != 0, QX, KX, V, mu, raw, logits, dO, dQX, dKX, dV, dmu, draw, dlogits, ws, st);
}

gma_status_t gma_usage(const gma_shape_t *s, const void *X, const float *mu, const float *raw, const float *logits,
                       int32_t *assign, int32_t *counts, float *mass, int32_t *used, float *entropy, void *ws,
                       size_t ws_bytes, gma_stream_t stream)
{
    gma_status_t r = validate_shape(s, GMA_VARIANT_RESPONSIBILITIES);
    if (r != GMA_OK) return r;
    const void *ptrs[] = {X, mu, raw, logits, assign, counts, mass, used, entropy};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GMA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    r = begin_call(s, GMA_VARIANT_USAGE, ws, ws_bytes, st);
    if (r != GMA_OK) return r;
    return usage(*s, X, mu, raw, logits, assign, counts, mass, used, entropy, ws, st);
}

gma_status_t gma_decode_step(const gma_shape_t *s, const void *qx, const void *kx, const void *v,
                             const float *mu, const float *raw, const float *logits, float *state,
                             void *o, void *ws, size_t ws_bytes, gma_stream_t stream)
{
    gma_status_t r = validate_shape(s, GMA_VARIANT_CAUSAL);
    if (r != GMA_OK) return r;
    if (s->N != 1) return GMA_ERR_INVALID_ARG;
    const void *ptrs[] = {qx, kx, v, mu, raw, logits, state, o};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GMA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    r = begin_call(s, GMA_VARIANT_DECODE, ws, ws_bytes, st);
    if (r != GMA_OK) return r;
    return decode_step(*s, qx, kx, v, mu, raw, logits, state, o, ws, st);
}

gma_status_t gma_check_workspace(const void *ws, gma_stream_t stream)
{
    if (!ws || ((uintptr_t)ws & 255u)) return GMA_ERR_WORKSPACE;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GMA_ERR_CUDA;
    WsHeader h;
    if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return GMA_ERR_CUDA;
    return (gma_status_t)h.error;
}

const char *gma_status_string(gma_status_t s)
{
    switch (s) {
    case GMA_OK: return "ok";
    case GMA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or flag)";
    case GMA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (d_r, d_v in {16,32,64,128}; 1 <= K <= 1024)";
    case GMA_ERR_RANGE: return "a reparametrised GMM parameter exceeds the range the tensor-core path holds";
    case GMA_ERR_WORKSPACE: return "workspace null, not 256-byte aligned, or too small";
    case GMA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case GMA_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case GMA_ERR_NO_DEVICE: return "no sm_103 CUDA device is current";
    }
    return "unknown status";
}

int gma_version(void) { return 100; }

}  // extern "C"
