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
// The step is bound by reading and writing the state, K (d_v + 1) fp32 per slice.  The main
// kernel is persistent (one CTA per SM, each taking every gridDim-th slice) and warp-specialised:
//   warp 0      streams the state of its slices, chunk after chunk (about 16 KB each), with bulk
//               copies (cp.async.bulk) into a ring of ~11 shared-memory stages, across slice
//               boundaries, so the next slices' loads are in flight while this one is worked on;
//   warps 1-4   compute the next slice's two rows of responsibilities into one of two buffers;
//   warps 5-12  add the key row to each chunk, read it with the query row, and write the chunk
//               back with a bulk store; a stage is refilled once its store has read it.
// For K not a multiple of 4 (rows would not start on 16-byte boundaries) a plain kernel, one CTA
// per slice whose threads copy the chunks themselves, takes the step.
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

constexpr int PT = 256;           // plain kernel: threads per CTA
constexpr int NLW = 8;            // persistent kernel: responsibility warps
constexpr int NSW = 4;            // persistent kernel: state warps
constexpr int ST = NSW * 32;      // state threads
constexpr int LT = NLW * 32;      // responsibility threads
constexpr int WT = 32 * (1 + NLW + NSW);
constexpr int BAR_STATE = 1, BAR_LOGIT = 2;   // named barriers (0 is __syncthreads)
constexpr int SMEM_BUDGET = 220 * 1024;
constexpr int MAX_STAGES = 16;
constexpr int PAR_SMEM_MAX = 8192;   // components x dimensions whose parameters are staged in shared memory

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

// Barrier over `n` threads (id 0: the whole CTA) that returns whether any of them passed true.
__device__ __forceinline__ bool bar_any(int id, int n, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(id), "r"(n)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ void group_sync(int id, int n)
{
    if (id == 0)
        __syncthreads();
    else
        named_bar_sync(id, n);
}

// Sum of one value per thread over a group of n threads (whole warps, group-local thread
// index gt) synchronised by barrier `id`; red holds n / 32 floats.
__device__ __forceinline__ float group_sum(float v, float *red, int gt, int n, int id)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    group_sync(id, n);
    if ((gt & 31) == 0) red[gt >> 5] = v;
    group_sync(id, n);
    float s = 0.f;
    for (int w = 0; w < n / 32; ++w) s += red[w];
    return s;
}

// Rows of state per chunk: about 32 KB per chunk, a multiple of 4 rows.
template <int DV> __host__ __device__ constexpr int chunk_rows() { return 8192 / DV; }
__host__ __device__ inline int chunk_rows_rt(int DV) { return 8192 / DV; }

// Logit pairs (A, B) of rows q_x and k_x for component k of head h:
//   sum_d (x_d - mu_kd)^2 / sigma^2_kd = s + e,  A = -s/2 (exact),  B = c_k - e/2,
// with c_k = log pi_k - 1/2 sum_d log sigma^2_kd.  Terms are accumulated four at a time with
// fused multiply-adds (the partial of four terms is small, so its rounding is too), and the
// partials are added to (s, e) with TwoSum, which keeps the rounding of the large running sum in
// e: the error of s + e is that of the four-term partials, not of a magnitude-~100 sum.
// The parameters come interleaved and transposed, mw[h][d][k] = (mu_kd, 1 / sigma^2_kd).  P
// adjacent lanes share one component, each summing d_r / P dimensions of both rows from
// coalesced 8-byte loads (issued in batches before the first of a batch is used), and their
// partial sums are merged, still exactly, by shuffles.
__device__ __forceinline__ void add_pair(float &s, float &e, float b)
{
    float t, r;
    two_sum(s, b, t, r);
    s = t;
    e += r;
}

__device__ __forceinline__ void merge_pair(float &s, float &e, int o)
{
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o), e2 = __shfl_xor_sync(0xffffffffu, e, o);
    float t, r;
    two_sum(s, s2, t, r);
    s = t;
    e = e + e2 + r;
}

// Lanes per component: up to 4, while every lane keeps at least `ud` dimensions.
__host__ __device__ inline int logit_parts(int K, int n, int d_r, int ud)
{
    int P = K * 4 <= n ? 4 : (K * 2 <= n ? 2 : 1);
    while (P > 1 && d_r / P < ud) P >>= 1;
    return P;
}

// Sums for item `it` (component it / P, dimensions (it % P) d_r / P onward) of both rows,
// merged over the P lanes of the component; every lane of the warp must call it.  `base` points
// at head h's parameters (rows ldk components apart), in global memory (GLOBAL) or a
// shared-memory copy.
template <bool GLOBAL>
__device__ __forceinline__ void item_sums(const float2 *base, int ldk, const float *xq, const float *xk, int K,
                                          int d_r, int P, int it, float &sq, float &eq, float &sk, float &ek)
{
    constexpr int UD = GLOBAL ? 16 : 8;   // loads in flight per batch (d_r >= 16 is a multiple)
    const int nd = d_r / P;               // a multiple of UD
    const int k = min(it / P, K - 1), d_lo = (it % P) * nd;
    sq = eq = sk = ek = 0.f;
    for (int d0 = d_lo; d0 < d_lo + nd; d0 += UD) {
        const float2 *pp = base + (size_t)d0 * ldk + k;
        float2 pr[UD];
#pragma unroll
        for (int u = 0; u < UD; ++u) pr[u] = GLOBAL ? __ldg(pp + (size_t)u * ldk) : pp[(size_t)u * ldk];
#pragma unroll
        for (int u4 = 0; u4 < UD; u4 += 4) {
            const float4 q4 = *reinterpret_cast<const float4 *>(xq + d0 + u4);
            const float4 k4 = *reinterpret_cast<const float4 *>(xk + d0 + u4);
            const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
            float bq = 0.f, bk = 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 p = pr[u4 + u];
                const float dq = qv[u] - p.x, dk = kv[u] - p.x;
                bq = fmaf(__fmul_rn(dq, dq), p.y, bq);
                bk = fmaf(__fmul_rn(dk, dk), p.y, bk);
            }
            add_pair(sq, eq, bq);
            add_pair(sk, ek, bk);
        }
    }
    for (int o = 1; o < P; o <<= 1) {
        merge_pair(sq, eq, o);
        merge_pair(sk, ek, o);
    }
}

template <bool GLOBAL>
__device__ __forceinline__ void logit_pairs(const float2 *base, int ldk, const float *cst, const float *xq,
                                            const float *xk, float *lq_a, float *lq_b, float *lk_a, float *lk_b,
                                            int K, int d_r, int gt, int n)
{
    const int P = logit_parts(K, n, d_r, GLOBAL ? 16 : 8);
    const int items = K * P, lane = gt & 31;
    // every lane of a warp runs the same iterations (the shuffles need all 32)
    for (int it0 = gt - lane; it0 < items; it0 += n) {
        const int it = it0 + lane;
        float sq, eq, sk, ek;
        item_sums<GLOBAL>(base, ldk, xq, xk, K, d_r, P, it, sq, eq, sk, ek);
        if (it < items && it % P == 0) {
            const int k = it / P;
            const float c = cst[k];
            lq_a[k] = -0.5f * sq;
            lq_b[k] = c - 0.5f * eq;
            lk_a[k] = -0.5f * sk;
            lk_b[k] = c - 0.5f * ek;
        }
    }
}

// Reparametrised parameters in the layout the decode kernels read:
//   mw[h][d][k] = (mu_kd, 1 / (softplus(raw_kd) + floor)),
//   cst[h][k]   = log pi_k - 1/2 sum_d log sigma^2_kd,  log pi = log softmax of the prior logits.
// Grid H x ceil(K / PK): one warp per component reads its row (lanes along d, all loads issued
// at once) and a block writes its PK components transposed through shared memory.  The decode
// kernel that follows is allowed to start at once (it waits for this grid before reading).
constexpr int PP = 256, PK = PP / 32;
__global__ void __launch_bounds__(PP) decode_params_kernel(const float *__restrict__ mu, const float *__restrict__ raw,
                                                           const float *__restrict__ logits, float2 *__restrict__ mw,
                                                           float *__restrict__ cst, int K, int d_r, float floor_)
{
    grid_dependency_launch();
    __shared__ float2 tile[128][PK + 1];
    const int h = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = blockIdx.y * PK + warp;
    const int kk = k < K ? k : K - 1;
    const float *rk = raw + ((size_t)h * K + kk) * d_r;
    const float *mk = mu + ((size_t)h * K + kk) * d_r;
    const float *lh = logits + (size_t)h * K;
    float rv[4], mv[4];   // d_r <= 128
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int d = lane + 32 * u;
        rv[u] = d < d_r ? rk[d] : 0.f;
        mv[u] = d < d_r ? mk[d] : 0.f;
    }
    float m = -INFINITY;
    for (int j = lane; j < K; j += 32) m = fmaxf(m, lh[j]);
    float logdet = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int d = lane + 32 * u;
        if (d < d_r) {
            const float r = rv[u];
            const float var = fmaxf(r, 0.f) + log1pf(expf(-fabsf(r))) + floor_;
            tile[d][warp] = make_float2(mv[u], 1.0f / var);
            logdet += logf(var);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        logdet += __shfl_xor_sync(0xffffffffu, logdet, o);
    }
    float se = 0.f;
    for (int j = lane; j < K; j += 32) se += expf(lh[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
    if (lane == 0 && k < K) cst[(size_t)h * K + k] = (lh[k] - (m + logf(se))) - 0.5f * logdet;
    __syncthreads();
    // transposed write: thread -> (d, component) with the PK components of a row consecutive
    for (int q = threadIdx.x; q < d_r * PK; q += PP) {
        const int d = q / PK, kl = q - d * PK, kw = blockIdx.y * PK + kl;
        if (kw < K) mw[((size_t)h * d_r + d) * K + kw] = tile[d][kl];
    }
}

// In place over a group of n threads, for both rows at once: a[k] <- softmax_k(a[k] + b[k]),
// with the maximum taken before b is added to the difference.  red holds 2 n / 32 floats.
__device__ __forceinline__ void softmax_pairs2(float *qa, const float *qb, float *ka, const float *kb, int K,
                                               float *red, int gt, int n, int id)
{
    const int nw = n / 32;
    float mq = -INFINITY, mk = -INFINITY;
    for (int k = gt; k < K; k += n) {
        mq = fmaxf(mq, qa[k] + qb[k]);
        mk = fmaxf(mk, ka[k] + kb[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    }
    group_sync(id, n);
    if ((gt & 31) == 0) {
        red[gt >> 5] = mq;
        red[nw + (gt >> 5)] = mk;
    }
    group_sync(id, n);
    mq = red[0];
    mk = red[nw];
    for (int w = 1; w < nw; ++w) {
        mq = fmaxf(mq, red[w]);
        mk = fmaxf(mk, red[nw + w]);
    }
    float sq = 0.f, sk = 0.f;
    for (int k = gt; k < K; k += n) {
        const float eq = expf((qa[k] - mq) + qb[k]), ek = expf((ka[k] - mk) + kb[k]);
        qa[k] = eq;
        ka[k] = ek;
        sq += eq;
        sk += ek;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    group_sync(id, n);
    if ((gt & 31) == 0) {
        red[gt >> 5] = sq;
        red[nw + (gt >> 5)] = sk;
    }
    group_sync(id, n);
    sq = 0.f;
    sk = 0.f;
    for (int w = 0; w < nw; ++w) {
        sq += red[w];
        sk += red[nw + w];
    }
    const float iq = 1.f / sq, ik = 1.f / sk;
    for (int k = gt; k < K; k += n) {
        qa[k] *= iq;
        ka[k] *= ik;
    }
}

// Both rows' responsibilities over a group of n threads (barrier `id`): gq[k] = p(z = k | q_x),
// gk[k] = p(z = k | k_x).  When every component's P lanes fit in the group at once, each lane
// keeps its logit pair in registers and the softmax needs two barriers; otherwise the pairs go
// through shared memory (ga, gb) and softmax_pairs2.  red holds 4 n / 32 floats.  The caller
// synchronises the group before reading gq, gk.
template <bool GLOBAL>
__device__ __forceinline__ void responsibilities(const float2 *base, int ldk, const float *cst, const float *xq,
                                                 const float *xk, float *gq, float *qb, float *gk, float *kb,
                                                 float *red, int K, int d_r, int gt, int n, int id)
{
    const int P = logit_parts(K, n, d_r, GLOBAL ? 16 : 8);
    if (K * P > n) {
        logit_pairs<GLOBAL>(base, ldk, cst, xq, xk, gq, qb, gk, kb, K, d_r, gt, n);
        group_sync(id, n);
        softmax_pairs2(gq, qb, gk, kb, K, red, gt, n, id);
        return;
    }
    const int nw = n / 32, lane = gt & 31, w = gt >> 5, items = K * P;
    const bool own = gt < items && gt % P == 0;
    float sq = 0.f, eq = 0.f, sk = 0.f, ek = 0.f;
    if (gt - lane < items) item_sums<GLOBAL>(base, ldk, xq, xk, K, d_r, P, gt, sq, eq, sk, ek);
    const int k = min(gt / P, K - 1);
    const float c = own ? cst[k] : 0.f;
    const float aq = -0.5f * sq, bq = c - 0.5f * eq, ak = -0.5f * sk, bk = c - 0.5f * ek;
    float mq = own ? aq + bq : -INFINITY, mk = own ? ak + bk : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    }
    if (lane == 0) {
        red[w] = mq;
        red[nw + w] = mk;
    }
    group_sync(id, n);
    mq = red[0];
    mk = red[nw];
    for (int q = 1; q < nw; ++q) {
        mq = fmaxf(mq, red[q]);
        mk = fmaxf(mk, red[nw + q]);
    }
    const float xq_ = own ? expf((aq - mq) + bq) : 0.f, xk_ = own ? expf((ak - mk) + bk) : 0.f;
    float s_q = xq_, s_k = xk_;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s_q += __shfl_xor_sync(0xffffffffu, s_q, o);
        s_k += __shfl_xor_sync(0xffffffffu, s_k, o);
    }
    if (lane == 0) {
        red[2 * nw + w] = s_q;
        red[3 * nw + w] = s_k;
    }
    group_sync(id, n);
    s_q = 0.f;
    s_k = 0.f;
    for (int q = 0; q < nw; ++q) {
        s_q += red[2 * nw + q];
        s_k += red[3 * nw + q];
    }
    if (own) {
        gq[k] = xq_ * (1.f / s_q);
        gk[k] = xk_ * (1.f / s_k);
    }
}

// One chunk's rows for this thread's column: S[r][col] += gk[r] add, acc += gq[r] S[r][col]; rows
// r = grp, grp + G, ...; U rows' loads are issued before they are used, and two accumulators
// halve the dependent chain.  With G == 1 the rows are consecutive and gk, gq (16-byte aligned
// there) are read four at a time.
template <int NE, int G>
__device__ __forceinline__ void update_rows(float *st, const float *gk, const float *gq, int rows, int grp, int col,
                                            float add, float &acc)
{
    constexpr int U = 8;
    float acc2 = 0.f;
    int r = grp;
    for (; r + (U - 1) * G < rows; r += U * G) {
        float x[U], a[U], b[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = st[(r + u * G) * NE + col];
        if (G == 1) {
#pragma unroll
            for (int u = 0; u < U; u += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(gk + r + u);
                const float4 b4 = *reinterpret_cast<const float4 *>(gq + r + u);
                a[u] = a4.x, a[u + 1] = a4.y, a[u + 2] = a4.z, a[u + 3] = a4.w;
                b[u] = b4.x, b[u + 1] = b4.y, b[u + 2] = b4.z, b[u + 3] = b4.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                a[u] = gk[r + u * G];
                b[u] = gq[r + u * G];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            x[u] = fmaf(a[u], add, x[u]);
            st[(r + u * G) * NE + col] = x[u];
        }
#pragma unroll
        for (int u = 0; u < U; u += 2) {
            acc = fmaf(b[u], x[u], acc);
            acc2 = fmaf(b[u + 1], x[u + 1], acc2);
        }
    }
    for (; r < rows; r += G) {
        const float x = fmaf(gk[r], add, st[r * NE + col]);
        st[r * NE + col] = x;
        acc = fmaf(gq[r], x, acc);
    }
    acc += acc2;
}

// ---------------------------------------------------------------- persistent kernel
struct PSmem {
    int ring, nstage, gbuf, gslot, part, red_s, red_l, bars, flag, par, total;
};

// Per responsibility slot: qa, qb, ka, kb [K] | xq, xk [d_r] | v [DV]  (floats).
__host__ __device__ inline int gslot_floats(int DV, int K, int d_r) { return 4 * K + 2 * d_r + DV; }

__host__ __device__ inline PSmem persist_smem(int DV, int K, int d_r)
{
    PSmem L;
    const int chunk = chunk_rows_rt(DV) * (DV + 1) * 4;
    int o = 0;
    auto take = [&](int bytes) { int at = o; o += (bytes + 15) & ~15; return at; };
    L.gslot = (gslot_floats(DV, K, d_r) * 4 + 15) & ~15;
    L.gbuf = take(2 * L.gslot);
    L.part = take(4 * ST);
    L.red_s = take(4 * 32);
    L.red_l = take(4 * 4 * (LT / 32));
    L.bars = take(8 * (2 * MAX_STAGES + 4));
    L.flag = take(16);
    // a copy of one head's parameters, (mu, 1 / sigma^2) [d_r][K], when K d_r <= PAR_SMEM_MAX
    L.par = K * d_r <= PAR_SMEM_MAX ? take(8 * K * d_r) : -1;
    L.ring = (o + 127) & ~127;
    int ns = (SMEM_BUDGET - L.ring) / chunk;
    L.nstage = ns < MAX_STAGES ? ns : MAX_STAGES;
    L.total = L.ring + L.nstage * chunk;
    return L;
}

template <int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(WT, 1) decode_persistent_kernel(
    const Tin *__restrict__ qx, const Tin *__restrict__ kx, const Tin *__restrict__ v, const float2 *__restrict__ mw,
    const float *__restrict__ cst, float *__restrict__ state, Tout *__restrict__ o, WsHeader *hdr, int BH, int H,
    int d_r, int K, float eps)
{
    constexpr int NE = DV + 1, KC = chunk_rows<DV>(), G = ST / DV;
    // slices in head-major order (sigma = h B + b), a contiguous range per CTA, so a CTA meets
    // at most a few heads and keeps one head's parameters in shared memory while it can
    extern __shared__ __align__(128) unsigned char smem[];
    const PSmem L = persist_smem(DV, K, d_r);
    const int NS = L.nstage;
    float *ring = reinterpret_cast<float *>(smem + L.ring);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *done = full + MAX_STAGES, *gfull = full + 2 * MAX_STAGES, *gempty = gfull + 2;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.flag);
    auto slot = [&](int j) { return reinterpret_cast<float *>(smem + L.gbuf + j * L.gslot); };

    const int nch = (K + KC - 1) / KC;
    const int B = BH / H;
    const int lo = (int)((long long)blockIdx.x * BH / gridDim.x);
    const int nsl = (int)((long long)(blockIdx.x + 1) * BH / gridDim.x) - lo;
    auto slice_of = [&](int i) {
        const int sg = lo + i;
        return (sg % B) * H + sg / B;
    };
    auto chunk_bytes = [&](int c) { return (uint32_t)(min(KC, K - c * KC) * NE * 4); };
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        *abort = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(done + s, ST);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(gfull + j, 1);
            mbar_init(gempty + j, 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    int issued = 0;   // thread 0: chunks whose loads it started
    if (warp == 0) {
        // ------------------------------------------------ producer: loads and stores of the state
        // Chunk n of this CTA's stream is chunk n % nch of its slice n / nch, in stage n % NS.
        if (threadIdx.x == 0) {
            const int N = nsl * nch;
            auto gaddr = [&](int n) {
                return state + (size_t)slice_of(n / nch) * K * NE + (size_t)(n % nch) * KC * NE;
            };
            for (; issued < N && issued < NS; ++issued) {
                mbar_arrive_expect_tx(full + issued, chunk_bytes(issued % nch));
                bulk_g2s(ring + (size_t)issued * KC * NE, gaddr(issued), chunk_bytes(issued % nch), full + issued);
            }
            for (int n = 0; n < N; ++n) {
                const int s = n % NS;
                float *st = ring + (size_t)s * KC * NE;
                if (!mbar_wait_abortable(done + s, (n / NS) & 1, hdr, 110, abort)) break;
                bulk_s2g(gaddr(n), st, chunk_bytes(n % nch));
                bulk_commit_group();
                if (issued < N) {   // issued == n + NS: refill this stage once its store has read it
                    bulk_wait_read();
                    mbar_arrive_expect_tx(full + s, chunk_bytes(issued % nch));
                    bulk_g2s(st, gaddr(issued), chunk_bytes(issued % nch), full + s);
                    ++issued;
                }
            }
            bulk_wait_read();   // the stores have read their source; they complete on their own
        }
    } else if (warp <= NLW) {
        // ------------------------------------------------ responsibilities of the next slices
        const int lt = threadIdx.x - 32;
        float *red = reinterpret_cast<float *>(smem + L.red_l);
        float2 *par = L.par >= 0 ? reinterpret_cast<float2 *>(smem + L.par) : nullptr;
        // this thread's element of the next slice's q_x, k_x and v rows, loaded one slice ahead
        // and converted only when used, so the loads stay in flight meanwhile
        Tin nq{}, nk{}, nv{};
        auto fetch = [&](int i) {
            const int bh = slice_of(i);
            if (lt < d_r) {
                nq = qx[(size_t)bh * d_r + lt];
                nk = kx[(size_t)bh * d_r + lt];
            }
            if (lt < DV) nv = v[(size_t)bh * DV + lt];
        };
        if (nsl > 0) fetch(0);
        int cur_h = -1;
        for (int i = 0; i < nsl; ++i) {
            const int j = i & 1;
            bool ok = true;
            if (i >= 2) ok = mbar_wait_abortable(gempty + j, ((i >> 1) - 1) & 1, hdr, 112, abort);
            if (bar_any(BAR_LOGIT, LT, !ok)) break;
            const int bh = slice_of(i), h = bh % H;
            float *g = slot(j);
            float *qa = g, *qb = g + K, *ka = g + 2 * K, *kb = g + 3 * K;
            float *xq = g + 4 * K, *xk = xq + d_r, *vv = xk + d_r;
            if (lt < d_r) {
                xq[lt] = to_f(nq);
                xk[lt] = to_f(nk);
            }
            if (lt < DV) vv[lt] = to_f(nv);
            if (i + 1 < nsl) fetch(i + 1);
            if (i == 0) grid_dependency_wait();   // the parameters come from the kernel before
            if (par && h != cur_h) {
                // a new head: its parameters into shared memory (every reader of the old ones
                // has passed the barrier above); all of a thread's loads are issued at once
                const uint4 *src = reinterpret_cast<const uint4 *>(mw + (size_t)h * d_r * K);
                uint4 *dst = reinterpret_cast<uint4 *>(par);
                const int n16 = K * d_r / 2;
#pragma unroll 16
                for (int q = lt; q < n16; q += LT) dst[q] = __ldg(src + q);
                cur_h = h;
            }
            named_bar_sync(BAR_LOGIT, LT);
            if (par)
                responsibilities<false>(par, K, cst + (size_t)h * K, xq, xk, qa, qb, ka, kb, red, K, d_r, lt, LT,
                                        BAR_LOGIT);
            else
                responsibilities<true>(mw + (size_t)h * d_r * K, K, cst + (size_t)h * K, xq, xk, qa, qb, ka, kb, red,
                                       K, d_r, lt, LT, BAR_LOGIT);
            named_bar_sync(BAR_LOGIT, LT);
            if (lt == 0) mbar_arrive(gfull + j);
        }
    } else {
        // ------------------------------------------------ state: update, read, write back
        const int t = threadIdx.x - 32 * (1 + NLW);
        const int col = t % DV, grp = t / DV;
        float *part = reinterpret_cast<float *>(smem + L.part);
        float *red = reinterpret_cast<float *>(smem + L.red_s);
        int n = 0;
        bool failed = false;
        for (int i = 0; i < nsl && !failed; ++i) {
            const int j = i & 1;
            const bool okg = mbar_wait_abortable(gfull + j, (i >> 1) & 1, hdr, 113, abort);
            if (bar_any(BAR_STATE, ST, !okg)) break;
            const int bh = slice_of(i);
            const float *g = slot(j);
            const float *gq = g, *gk = g + 2 * K;
            const float add = g[4 * K + 2 * d_r + col];
            float acc = 0.f, zacc = 0.f;
            for (int c = 0; c < nch; ++c, ++n) {
                const int s = n % NS;
                float *st = ring + (size_t)s * KC * NE;
                const bool ok = mbar_wait_abortable(full + s, (n / NS) & 1, hdr, 114, abort);
                if (bar_any(BAR_STATE, ST, !ok)) {
                    failed = true;
                    break;
                }
                const int rows = min(KC, K - c * KC), k0 = c * KC;
                update_rows<NE, G>(st, gk + k0, gq + k0, rows, grp, col, add, acc);
                for (int r = t; r < rows; r += ST) {
                    const float z = gk[k0 + r] + st[r * NE + DV];
                    st[r * NE + DV] = z;
                    zacc = fmaf(gq[k0 + r], z, zacc);
                }
                fence_proxy_async_smem();   // this thread's writes, before the producer's bulk store
                mbar_arrive(done + s);
            }
            if (failed) break;
            if (G > 1) part[t] = acc;
            // (its barriers also mean every state thread is done with slot j: it is free again;
            // part[] and red[] are next written after the next slice's chunk barriers)
            const float den = group_sum(zacc, red, t, ST, BAR_STATE);
            if (t == 0) mbar_arrive(gempty + j);
            if (t < DV) {
                float num = acc;
#pragma unroll
                for (int q = 1; q < G; ++q) num += part[q * DV + t];
                from_f(o[(size_t)bh * DV + t], num / (den + eps));
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort) {
        // after a timeout some loads may not have been consumed: wait for each stage's last
        // one (bounded) so no copy lands in shared memory after the CTA has exited
        for (int s = 0; s < NS && s < issued; ++s) {
            const int last = s + ((issued - 1 - s) / NS) * NS;
            (void)mbar_wait(full + s, (last / NS) & 1, hdr, 111);
        }
    }
}

// ---------------------------------------------------------------- plain kernel (K % 4 != 0)
template <int DV, typename Tin, typename Tout>
__global__ void __launch_bounds__(PT) decode_plain_kernel(const Tin *__restrict__ qx, const Tin *__restrict__ kx,
                                                          const Tin *__restrict__ v, const float2 *__restrict__ mw,
                                                          const float *__restrict__ cst, float *__restrict__ state,
                                                          Tout *__restrict__ o, int H, int d_r, int K, float eps)
{
    constexpr int NE = DV + 1, KC = chunk_rows<DV>(), G = PT / DV;
    extern __shared__ __align__(128) unsigned char smem[];
    float *st = reinterpret_cast<float *>(smem);
    float *qa = st + KC * NE, *qb = qa + K, *ka = qb + K, *kb = ka + K;
    float *xq = kb + K, *xk = xq + d_r, *vv = xk + d_r, *red = vv + DV, *part = red + 32;
    const int bh = blockIdx.x, h = bh % H, t = threadIdx.x;
    for (int d = t; d < d_r; d += PT) {
        xq[d] = to_f(qx[(size_t)bh * d_r + d]);
        xk[d] = to_f(kx[(size_t)bh * d_r + d]);
    }
    for (int c = t; c < DV; c += PT) vv[c] = to_f(v[(size_t)bh * DV + c]);
    grid_dependency_wait();   // the parameters come from the kernel before
    __syncthreads();
    responsibilities<true>(mw + (size_t)h * d_r * K, K, cst + (size_t)h * K, xq, xk, qa, qb, ka, kb, red, K, d_r,
                           t, PT, 0);
    __syncthreads();
    const int col = t % DV, grp = t / DV;
    const float add = vv[col];
    float acc = 0.f, zacc = 0.f;
    float *S = state + (size_t)bh * K * NE;
    for (int k0 = 0; k0 < K; k0 += KC) {
        const int rows = min(KC, K - k0);
        for (int i = t; i < rows * NE; i += PT) st[i] = S[(size_t)k0 * NE + i];
        __syncthreads();
        update_rows<NE, G>(st, ka + k0, qa + k0, rows, grp, col, add, acc);
        for (int r = t; r < rows; r += PT) {
            const float z = ka[k0 + r] + st[r * NE + DV];
            st[r * NE + DV] = z;
            zacc = fmaf(qa[k0 + r], z, zacc);
        }
        __syncthreads();
        for (int i = t; i < rows * NE; i += PT) S[(size_t)k0 * NE + i] = st[i];
        __syncthreads();
    }
    part[t] = acc;
    const float den = group_sum(zacc, red, t, PT, 0);
    if (t < DV) {
        float num = 0.f;
#pragma unroll
        for (int q = 0; q < G; ++q) num += part[q * DV + t];
        from_f(o[(size_t)bh * DV + t], num / (den + eps));
    }
}

inline size_t plain_smem(int DV, int K, int d_r)
{
    return 4 * ((size_t)chunk_rows_rt(DV) * (DV + 1) + 4 * K + 2 * d_r + DV + 32 + PT);
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

struct DecodeArgs {
    const void *qx, *kx, *v;
    const float *mu, *raw, *logits;
    float *state;
    void *o;
    const float2 *mw;   // reparametrised parameters (global path)
    const float *cst;
    WsHeader *hdr;
};

inline bool persistent_path(const gma_shape_t &s) { return (s.K & 3) == 0; }

template <int DV, typename Tin, typename Tout>
gma_status_t launch_typed(const gma_shape_t &s, const DecodeArgs &a, cudaStream_t st)
{
    const int BH = s.B * s.H;
    cudaError_t e = cudaSuccess;
    if (persistent_path(s)) {
        const PSmem L = persist_smem(DV, s.K, s.d_r);
        if (L.nstage < 2) return GMA_ERR_UNSUPPORTED_SHAPE;
        const int sms = sm_count();
        if (sms <= 0) return GMA_ERR_CUDA;
        const int grid = BH < sms ? BH : sms;
        auto k = decode_persistent_kernel<DV, Tin, Tout>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_DECODE, st,
                   (e = launch_pdl(k, dim3(grid), dim3(WT), (size_t)L.total, st, (const Tin *)a.qx, (const Tin *)a.kx,
                                   (const Tin *)a.v, a.mw, a.cst, a.state, (Tout *)a.o, a.hdr, BH, s.H, s.d_r, s.K,
                                   s.eps)));
    } else {
        const size_t smem = plain_smem(DV, s.K, s.d_r);
        auto k = decode_plain_kernel<DV, Tin, Tout>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_DECODE, st,
                   (e = launch_pdl(k, dim3(BH), dim3(PT), smem, st, (const Tin *)a.qx, (const Tin *)a.kx,
                                   (const Tin *)a.v, a.mw, a.cst, a.state, (Tout *)a.o, s.H, s.d_r, s.K, s.eps)));
    }
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template <int DV>
gma_status_t launch_dv(const gma_shape_t &s, const DecodeArgs &a, cudaStream_t st)
{
    if (s.dtype == GMA_F32) return launch_typed<DV, float, float>(s, a, st);
    if (s.flags & GMA_FLAG_OUT_F32) return launch_typed<DV, __nv_bfloat16, float>(s, a, st);
    return launch_typed<DV, __nv_bfloat16, __nv_bfloat16>(s, a, st);
}

}  // namespace

size_t decode_workspace_size(const gma_shape_t &s)
{
    Carve c;
    c.take(sizeof(float2) * (size_t)s.H * s.K * s.d_r);   // (mu, 1 / sigma^2), [H][d_r][K]
    c.take(sizeof(float) * (size_t)s.H * s.K);            // log pi - 1/2 sum log sigma^2
    return c.total();
}

gma_status_t decode_step(const gma_shape_t &s, const void *qx, const void *kx, const void *v, const float *mu,
                         const float *raw, const float *logits, float *state, void *o, void *ws, cudaStream_t st)
{
    Carve c;
    DecodeArgs a;
    a.qx = qx;
    a.kx = kx;
    a.v = v;
    a.mu = mu;
    a.raw = raw;
    a.logits = logits;
    a.state = state;
    a.o = o;
    a.mw = (const float2 *)((char *)ws + c.take(sizeof(float2) * (size_t)s.H * s.K * s.d_r));
    a.cst = (const float *)((char *)ws + c.take(sizeof(float) * (size_t)s.H * s.K));
    a.hdr = (WsHeader *)ws;
    GMA_LAUNCH(KID_DECODE_PARAMS, st,
                   (decode_params_kernel<<<dim3((unsigned)s.H, (unsigned)((s.K + PK - 1) / PK)), PP, 0, st>>>(
                       mu, raw, logits, (float2 *)a.mw, (float *)a.cst, s.K, s.d_r, s.var_floor)));
    switch (s.d_v) {
    case 16: return launch_dv<16>(s, a, st);
    case 32: return launch_dv<32>(s, a, st);
    case 64: return launch_dv<64>(s, a, st);
    case 128: return launch_dv<128>(s, a, st);
    }
    return GMA_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace gma
