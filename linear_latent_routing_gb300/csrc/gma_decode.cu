// gma_decode.cu -- one autoregressive decode step of causal GMA (gma_decode_step).
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §3: the causal variant keeps the latent memory V~ and its normaliser Z as prefix
// sums, so a new token costs O(K d_v): its key and value join the prefix, then its query reads it.
// Per (batch, head) slice:
//   gamma_K = p(z | k_x),  S[k][c] += gamma_K[k] v[c] (c < d_v),  S[k][d_v] += gamma_K[k]
//   gamma_Q = p(z | q_x),  o[c] = (gamma_Q . S[:, c]) / (gamma_Q . S[:, d_v] + eps)
// with the posterior of §1 in its direct form (x - mu)^2 / sigma^2, in fp32 on the CUDA cores.
//
// The step is bound by reading and writing the state, K (d_v + 1) fp32 per slice.  One CTA per
// slice: thread 0 starts bulk copies (cp.async.bulk) of the slice's state, in chunks of about
// 16 KB, into a ring of shared-memory stages before anything else, so the loads are in flight
// while the CTA computes the two rows of responsibilities; each chunk is then updated and read
// in shared memory and written back with a bulk store.  For K not a multiple of 4 (rows would
// not start on 16-byte boundaries) the threads copy the chunks themselves.
//
// Logits are summed with error-free transformations (Knuth's TwoSum; Ogita, Rump and Oishi,
// "Accurate sum and dot product", SIAM J. Sci. Comput. 2005): each logit is kept as an unrounded
// pair (A, B), and the softmax subtracts the maximum from A before adding B, so a logit of
// magnitude ~100 does not lose its last digits to the fp32 rounding of the sum.
#include "gma_internal.cuh"
#include "tc_ptx.cuh"

#include <cuda_bf16.h>

namespace gma {
namespace {

using namespace tc;

constexpr int DT = 256;     // threads per CTA
constexpr int NS = 4;       // stages in the state ring

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float &d, float x) { d = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 &d, float x) { d = __float2bfloat16_rn(x); }

// s + e = a + b exactly (TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ float block_max(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int w = 1; w < DT / 32; ++w) m = fmaxf(m, red[w]);
    return m;
}

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < DT / 32; ++w) s += red[w];
    return s;
}

// Rows of state per chunk: about 16 KB per chunk, a multiple of 4 rows.
template <int DV> __host__ __device__ constexpr int chunk_rows() { return 4096 / DV; }

struct DecodeSmem {
    int ring, lq_a, lq_b, lk_a, lk_b, xq, xk, vv, red, part, bars, flag, total;
};

__host__ __device__ inline DecodeSmem decode_smem(int DV, int K, int d_r)
{
    DecodeSmem L;
    const int ne = DV + 1;
    int o = 0;
    auto take = [&](int bytes) { int at = o; o += (bytes + 15) & ~15; return at; };
    L.ring = take(NS * (4096 / DV) * ne * 4);
    L.lq_a = take(4 * K);
    L.lq_b = take(4 * K);
    L.lk_a = take(4 * K);
    L.lk_b = take(4 * K);
    L.xq = take(4 * d_r);
    L.xk = take(4 * d_r);
    L.vv = take(4 * DV);
    L.red = take(4 * 32);
    L.part = take(4 * DT);
    L.bars = take(8 * NS);
    L.flag = take(16);
    L.total = o;
    return L;
}

// Logit pair (A, B) of rows k_x and q_x for component k of head h: the sum of
// (x_d - mu_kd)^2 / sigma^2_kd is s + e exactly up to the products' rounding;
// A = -s/2 (exact), B = c_k - e/2 with c_k = log pi_k - 1/2 sum_d log sigma^2_kd.
// DL lanes cover one row, 4 dimensions each.
__device__ __forceinline__ void logit_pairs(const float *__restrict__ mu, const float *__restrict__ iv,
                                            const float *__restrict__ cst, const float *xq, const float *xk,
                                            float *lq_a, float *lq_b, float *lk_a, float *lk_b, int h, int K,
                                            int d_r)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int DL = d_r >> 2, RW = 32 / DL;
    const int dl = lane % DL, rsub = lane / DL;
    const float4 q4 = *reinterpret_cast<const float4 *>(xq + 4 * dl);
    const float4 k4 = *reinterpret_cast<const float4 *>(xk + 4 * dl);
    const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
    for (int base = warp * RW; base < K; base += (DT / 32) * RW) {
        const int k = base + rsub;
        const int kk = k < K ? k : K - 1;
        const size_t off = ((size_t)h * K + kk) * d_r + 4 * dl;
        const float4 m4 = __ldg(reinterpret_cast<const float4 *>(mu + off));
        const float4 w4 = __ldg(reinterpret_cast<const float4 *>(iv + off));
        const float mv[4] = {m4.x, m4.y, m4.z, m4.w}, wv[4] = {w4.x, w4.y, w4.z, w4.w};
        float sq = 0.f, eq = 0.f, sk = 0.f, ek = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float dq = qv[j] - mv[j], dk = kv[j] - mv[j];
            float s, e;
            two_sum(sq, __fmul_rn(__fmul_rn(dq, dq), wv[j]), s, e);
            sq = s;
            eq += e;
            two_sum(sk, __fmul_rn(__fmul_rn(dk, dk), wv[j]), s, e);
            sk = s;
            ek += e;
        }
        for (int o = DL >> 1; o > 0; o >>= 1) {
            const float sq2 = __shfl_xor_sync(0xffffffffu, sq, o), eq2 = __shfl_xor_sync(0xffffffffu, eq, o);
            const float sk2 = __shfl_xor_sync(0xffffffffu, sk, o), ek2 = __shfl_xor_sync(0xffffffffu, ek, o);
            float s, e;
            two_sum(sq, sq2, s, e);
            sq = s;
            eq = eq + eq2 + e;
            two_sum(sk, sk2, s, e);
            sk = s;
            ek = ek + ek2 + e;
        }
        if (dl == 0 && k < K) {
            const float c0 = __ldg(cst + (size_t)h * K + k);
            lq_a[k] = -0.5f * sq;
            lq_b[k] = c0 - 0.5f * eq;
            lk_a[k] = -0.5f * sk;
            lk_b[k] = c0 - 0.5f * ek;
        }
    }
}

// In place: a[k] <- softmax_k(a[k] + b[k]), with the maximum taken from a before b is added.
__device__ __forceinline__ void softmax_pairs(float *a, float *b, int K, float *red)
{
    float m = -INFINITY;
    for (int k = threadIdx.x; k < K; k += DT) m = fmaxf(m, a[k] + b[k]);
    m = block_max(m, red);
    float s = 0.f;
    for (int k = threadIdx.x; k < K; k += DT) {
        const float e = expf((a[k] - m) + b[k]);
        a[k] = e;
        s += e;
    }
    s = block_sum(s, red);
    const float inv = 1.f / s;
    for (int k = threadIdx.x; k < K; k += DT) a[k] *= inv;
}

template <int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(DT) decode_kernel(const Tin *__restrict__ qx, const Tin *__restrict__ kx,
                                                    const Tin *__restrict__ v, const float *__restrict__ mu,
                                                    const float *__restrict__ inv_var,
                                                    const float *__restrict__ cst, float *__restrict__ state,
                                                    Tout *__restrict__ o, WsHeader *hdr, int H, int d_r, int K,
                                                    float eps)
{
    constexpr int NE = DV + 1, KC = chunk_rows<DV>(), G = DT / DV;
    extern __shared__ __align__(128) unsigned char smem[];
    const DecodeSmem L = decode_smem(DV, K, d_r);
    float *ring = reinterpret_cast<float *>(smem + L.ring);
    float *lq_a = reinterpret_cast<float *>(smem + L.lq_a), *lq_b = reinterpret_cast<float *>(smem + L.lq_b);
    float *lk_a = reinterpret_cast<float *>(smem + L.lk_a), *lk_b = reinterpret_cast<float *>(smem + L.lk_b);
    float *xq = reinterpret_cast<float *>(smem + L.xq), *xk = reinterpret_cast<float *>(smem + L.xk);
    float *vv = reinterpret_cast<float *>(smem + L.vv), *red = reinterpret_cast<float *>(smem + L.red);
    float *part = reinterpret_cast<float *>(smem + L.part);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.flag);

    const int bh = blockIdx.x, h = bh % H, t = threadIdx.x;
    const bool bulk = (K & 3) == 0;
    const int nch = (K + KC - 1) / KC;
    float *S = state + (size_t)bh * K * NE;
    auto chunk_bytes = [&](int c) { return (uint32_t)(min(KC, K - c * KC) * NE * 4); };

    if (t == 0) {
        *abort = 0;
        if (bulk) {
            for (int s = 0; s < NS; ++s) mbar_init(full + s, 1);
            fence_mbar_init();
            for (int c = 0; c < nch && c < NS; ++c) {
                mbar_arrive_expect_tx(full + c, chunk_bytes(c));
                bulk_g2s(ring + c * KC * NE, S + (size_t)c * KC * NE, chunk_bytes(c), full + c);
            }
        }
    }
    for (int d = t; d < d_r; d += DT) {
        xq[d] = to_f(qx[(size_t)bh * d_r + d]);
        xk[d] = to_f(kx[(size_t)bh * d_r + d]);
    }
    for (int c = t; c < DV; c += DT) vv[c] = to_f(v[(size_t)bh * DV + c]);
    __syncthreads();
    logit_pairs(mu, inv_var, cst, xq, xk, lq_a, lq_b, lk_a, lk_b, h, K, d_r);
    __syncthreads();
    softmax_pairs(lq_a, lq_b, K, red);
    softmax_pairs(lk_a, lk_b, K, red);
    __syncthreads();
    const float *gq = lq_a, *gk = lk_a;

    // the state, chunk by chunk: add this token's key row, read with its query row
    const int col = t % DV, grp = t / DV;
    const float add = vv[col];
    float acc = 0.f, zacc = 0.f;
    int failed_at = -1;
    for (int c = 0; c < nch; ++c) {
        const int s = bulk ? c % NS : 0;
        float *st = ring + s * KC * NE;
        const int rows = min(KC, K - c * KC), k0 = c * KC;
        if (bulk) {
            const bool ok = mbar_wait_abortable(full + s, (c / NS) & 1, hdr, 100, abort);
            if (__syncthreads_or(!ok)) {
                failed_at = c;
                break;
            }
        } else {
            for (int i = t; i < rows * NE; i += DT) st[i] = S[(size_t)k0 * NE + i];
            __syncthreads();
        }
        for (int r = grp; r < rows; r += G) {
            const float x = fmaf(gk[k0 + r], add, st[r * NE + col]);
            st[r * NE + col] = x;
            acc = fmaf(gq[k0 + r], x, acc);
        }
        for (int r = t; r < rows; r += DT) {
            const float z = gk[k0 + r] + st[r * NE + DV];
            st[r * NE + DV] = z;
            zacc = fmaf(gq[k0 + r], z, zacc);
        }
        if (bulk) {
            fence_proxy_async_smem();
            __syncthreads();
            if (t == 0) {
                bulk_s2g(S + (size_t)k0 * NE, st, chunk_bytes(c));
                bulk_commit_group();
                const int nxt = c - 1 + NS;   // refill the stage stored one chunk ago
                if (c >= 1 && nxt < nch) {
                    bulk_wait_read_but1();
                    const int sp = (c - 1) % NS;
                    mbar_arrive_expect_tx(full + sp, chunk_bytes(nxt));
                    bulk_g2s(ring + sp * KC * NE, S + (size_t)nxt * KC * NE, chunk_bytes(nxt), full + sp);
                }
            }
        } else {
            __syncthreads();
            for (int i = t; i < rows * NE; i += DT) S[(size_t)k0 * NE + i] = st[i];
            __syncthreads();
        }
    }
    if (bulk && t == 0) {
        if (failed_at >= 0) {
            // loads issued but not consumed (chunks failed_at .. issued - 1, one per stage):
            // wait for them, bounded, so no copy lands in shared memory after the CTA exits
            const int issued = min(nch, failed_at == 0 ? NS : NS + failed_at - 1);
            for (int j = failed_at; j < issued; ++j) (void)mbar_wait(full + j % NS, (j / NS) & 1, hdr, 101);
        }
        bulk_wait_all();
    }
    if (failed_at >= 0) return;
    // reduce the row groups' partial readouts, then normalise
    part[t] = acc;
    const float den = block_sum(zacc, red);
    __syncthreads();
    if (t < DV) {
        float num = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) num += part[g * DV + t];
        from_f(o[(size_t)bh * DV + t], num / (den + eps));
    }
}

template <int DV>
gma_status_t launch_dv(const gma_shape_t &s, const void *qx, const void *kx, const void *v, const float *mu,
                       const float *iv, const float *cst, float *state, void *o, WsHeader *hdr, cudaStream_t st)
{
    const int BH = s.B * s.H;
    const size_t smem = (size_t)decode_smem(DV, s.K, s.d_r).total;
    const bool out32 = (s.flags & GMA_FLAG_OUT_F32) || s.dtype == GMA_F32;
    if (s.dtype == GMA_F32) {
        auto k = decode_kernel<DV, float, float>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_DECODE, st,
                   (k<<<BH, DT, smem, st>>>((const float *)qx, (const float *)kx, (const float *)v, mu, iv, cst,
                                            state, (float *)o, hdr, s.H, s.d_r, s.K, s.eps)));
    } else if (out32) {
        auto k = decode_kernel<DV, __nv_bfloat16, float>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_DECODE, st,
                   (k<<<BH, DT, smem, st>>>((const __nv_bfloat16 *)qx, (const __nv_bfloat16 *)kx,
                                            (const __nv_bfloat16 *)v, mu, iv, cst, state, (float *)o, hdr, s.H,
                                            s.d_r, s.K, s.eps)));
    } else {
        auto k = decode_kernel<DV, __nv_bfloat16, __nv_bfloat16>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_DECODE, st,
                   (k<<<BH, DT, smem, st>>>((const __nv_bfloat16 *)qx, (const __nv_bfloat16 *)kx,
                                            (const __nv_bfloat16 *)v, mu, iv, cst, state, (__nv_bfloat16 *)o, hdr,
                                            s.H, s.d_r, s.K, s.eps)));
    }
    return GMA_OK;
}

}  // namespace

size_t decode_workspace_size(const gma_shape_t &s)
{
    Carve c;
    c.take(sizeof(float) * (size_t)s.H * s.K * s.d_r);   // 1 / sigma^2
    c.take(sizeof(float) * (size_t)s.H * s.K);           // log pi - 1/2 sum log sigma^2
    return c.total();
}

gma_status_t decode_step(const gma_shape_t &s, const void *qx, const void *kx, const void *v, const float *mu,
                         const float *raw, const float *logits, float *state, void *o, void *ws, cudaStream_t st)
{
    Carve c;
    float *iv = (float *)((char *)ws + c.take(sizeof(float) * (size_t)s.H * s.K * s.d_r));
    float *cst = (float *)((char *)ws + c.take(sizeof(float) * (size_t)s.H * s.K));
    gma_status_t r = simt_params(s, raw, logits, iv, cst, st);
    if (r != GMA_OK) return r;
    WsHeader *hdr = (WsHeader *)ws;
    switch (s.d_v) {
    case 16: return launch_dv<16>(s, qx, kx, v, mu, iv, cst, state, o, hdr, st);
    case 32: return launch_dv<32>(s, qx, kx, v, mu, iv, cst, state, o, hdr, st);
    case 64: return launch_dv<64>(s, qx, kx, v, mu, iv, cst, state, o, hdr, st);
    case 128: return launch_dv<128>(s, qx, kx, v, mu, iv, cst, state, o, hdr, st);
    }
    return GMA_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace gma
