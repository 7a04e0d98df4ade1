// gma_simt.cu -- the fp32 CUDA-core kernel family of libgma.so.
//
// Every step in fp32 on the CUDA cores, with the Gaussian log-density in its direct form
// (x - mu)^2 / sigma^2.  This is the path fp32 inputs take (tensor cores cannot hold fp32's
// precision), the path GMA_FLAG_SIMT selects, and the correctness anchor for the tcgen05 family.
//
// Method (page "Attention par Mélange Gaussien (GMA)", gist.science/fr/paper/2606.18283,
// Méthodologie §1-§3): responsibilities by the GMM posterior; write phase
// V~ = Gamma_K^T V, Z = Gamma_K^T 1; read phase O = Gamma_Q V~ / (Gamma_Q Z + eps); causal
// variant by inclusive prefix sums.
//
// Structure: Gamma_Q and Gamma_K are materialised in the workspace (fp32); keys are cut into
// segments of SEG tokens whose partial memories [V~ | Z] are summed (bidirectional) or
// exclusive-prefix-scanned (causal); each query segment then reads its memory and, for the
// causal variant, adds the masked in-segment affinity (Gamma_Q Gamma_K^T restricted to j <= i).
#include "gma_internal.cuh"
#include "simt_tile.cuh"
#include "tc_ptx.cuh"

namespace gma {
namespace {

using tc::grid_dependency_launch;
using tc::grid_dependency_wait;

// Every kernel of this family starts by waiting for the grid before it (programmatic dependent
// launch; nothing is read or written before) and lets the next one be scheduled, so that the
// launch latencies of a call's kernels overlap.
__device__ __forceinline__ void chain_enter()
{
    grid_dependency_wait();
    grid_dependency_launch();
}

constexpr int SEG = 64;        // tokens per segment
constexpr int KT = 32;         // component tile for the staged dot products
constexpr int THREADS = 256;
constexpr int PARAM_THREADS = 64;   // two component rows per block: the fp64 log-determinants spread over the SMs

// ---------------------------------------------------------------- reparametrisation
// Per head h: inv_var[h][k][d] = 1 / (softplus(raw) + floor);
//             cst[h][k]        = log pi_k - 1/2 sum_d log sigma^2_kd,  log pi = log softmax.
// One warp per component row (grid H x ceil(K / 2)); every warp first reduces its head's
// prior logits to their log-sum-exp (K <= 1024: at most 32 values per lane).
// The block at inv_var also receives the transposes the responsibilities stage from, [H][d_r][K]
// each, after the H K d_r values of inv_var: mu^T, (1 / sigma^2)^T, (1 / sigma)^T and
// (-mu / sigma)^T (the callers' workspace holds all five).
__global__ void simt_params_kernel(const float *__restrict__ raw, const float *__restrict__ logits,
                                   const float *__restrict__ mu, float *__restrict__ inv_var,
                                   float *__restrict__ cst, int K, int d_r, float floor_)
{
    chain_enter();
    const int h = blockIdx.x, lane = threadIdx.x & 31;
    const int k = blockIdx.y * (PARAM_THREADS / 32) + (threadIdx.x >> 5);
    const float *lh = logits + (size_t)h * K;
    const int kr = k < K ? k : K - 1;
    const float *rk = raw + ((size_t)h * K + kr) * d_r;
    float rv[4];   // d_r <= 128: this lane's raw variances, loaded before the reductions
#pragma unroll
    for (int i = 0; i < 4; ++i) rv[i] = lane + 32 * i < d_r ? rk[lane + 32 * i] : 0.f;
    float m = -INFINITY;
    for (int j = lane; j < K; j += 32) m = fmaxf(m, lh[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int j = lane; j < K; j += 32) s += expf(lh[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (k >= K) return;
    const float lse = m + logf(s);
    float *ik = inv_var + ((size_t)h * K + k) * d_r;
    // the log-determinant is summed in double (once per component per call), so that the
    // constant carries only its final fp32 rounding into the logits
    double logdet = 0.0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int d = lane + 32 * i;
        if (d < d_r) {
            const float r = rv[i];
            const float var = fmaxf(r, 0.f) + log1pf(expf(-fabsf(r))) + floor_;
            ik[d] = 1.0f / var;
            const size_t HKD = (size_t)gridDim.x * K * d_r, tr = ((size_t)h * d_r + d) * K + k;
            const float m = mu[((size_t)h * K + k) * d_r + d], sd = 1.0f / sqrtf(var);
            inv_var[HKD + tr] = m;
            inv_var[2 * HKD + tr] = 1.0f / var;
            inv_var[3 * HKD + tr] = sd;
            inv_var[4 * HKD + tr] = -sd * m;
            logdet += log((double)var);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) logdet += __shfl_xor_sync(0xffffffffu, logdet, o);
    if (lane == 0) cst[(size_t)h * K + k] = (float)(((double)lh[k] - (double)lse) - 0.5 * logdet);
}

// ---------------------------------------------------------------- responsibilities
// (IVG: the inverse variances iv_k are in global memory, read through the read-only cache; else
// in shared memory.)
// The rows of mu and 1/sigma^2 are read four floats at a time (16-byte aligned: the API checks the
// parameter pointers, d_r is a multiple of 4 and the workspace is 256-byte aligned); the sums run
// over d in order.
template <bool IVG>
__device__ __forceinline__ float4 iv4(const float *iv_k, int d)
{
    return IVG ? __ldg(reinterpret_cast<const float4 *>(iv_k + d)) : *reinterpret_cast<const float4 *>(iv_k + d);
}

template <int DR, bool IVG = true>
__device__ __forceinline__ float logit_direct(const float (&x)[DR], const float *__restrict__ mu_k,
                                              const float *iv_k, float c_k)
{
    float q = 0.f;
#pragma unroll
    for (int d = 0; d < DR; d += 4) {
        const float4 m = __ldg(reinterpret_cast<const float4 *>(mu_k + d));
        const float4 w = iv4<IVG>(iv_k, d);
        const float t0 = x[d] - m.x, t1 = x[d + 1] - m.y, t2 = x[d + 2] - m.z, t3 = x[d + 3] - m.w;
        q = fmaf(t0 * t0, w.x, q);
        q = fmaf(t1 * t1, w.y, q);
        q = fmaf(t2 * t2, w.z, q);
        q = fmaf(t3 * t3, w.w, q);
    }
    return fmaf(-0.5f, q, c_k);
}

// hi + lo += b, exactly: Knuth's TwoSum gives the rounding error of hi + b, which joins lo.
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float b)
{
    const float s = hi + b;
    const float bb = s - hi;
    const float e = (hi - (s - bb)) + (b - bb);
    hi = s;
    lo += e;
}

// The same logit as an unevaluated sum hi + lo, for fp32 inputs.  A logit of a few hundred
// summed in fp32 one term at a time keeps only ~1e-5 of absolute accuracy, which the 1e-5
// tolerance of fp32 outputs cannot afford at d_r = 128.  Here the quadratic form is summed in
// four-term FMA partials (each small, so rounded finely), and their running total starting from
// c_k is kept as a TwoSum pair (Knuth, TAOCP vol. 2, 4.2.2; the "accurate sum" of Ogita, Rump
// and Oishi, 2005).  Differences of nearby logits, hi_k - hi_j + (lo_k - lo_j), then carry the
// accuracy of the four-term partials instead of that of a number of size |L|.
template <int DR, bool IVG = true>
__device__ __forceinline__ float2 logit_direct_pair(const float (&x)[DR], const float *__restrict__ mu_k,
                                                    const float *iv_k, float c_k)
{
    float hi = c_k, lo = 0.f;
#pragma unroll
    for (int d0 = 0; d0 < DR; d0 += 4) {
        const float4 m = __ldg(reinterpret_cast<const float4 *>(mu_k + d0));
        const float4 w = iv4<IVG>(iv_k, d0);
        const float t0 = x[d0] - m.x, t1 = x[d0 + 1] - m.y, t2 = x[d0 + 2] - m.z, t3 = x[d0 + 3] - m.w;
        float p = 0.f;
        p = fmaf(t0 * t0, w.x, p);
        p = fmaf(t1 * t1, w.y, p);
        p = fmaf(t2 * t2, w.z, p);
        p = fmaf(t3 * t3, w.w, p);
        two_sum_acc(hi, lo, -0.5f * p);   // (the factor is a power of two: exact)
    }
    return make_float2(hi, lo);
}

// The routing vectors of one 64-row segment of one (b, h) slice per block of 256 threads: a 16 x 16
// grid in which each thread forms the logits of 4 rows x 4 components of a 64-component tile, from
// x^T and two parameter transposes staged in shared memory (per dimension one 16-byte load of
// each).  Each logit is summed over d in order.  fp32 inputs: exactly as logit_direct_pair does,
// (x - mu)^2 / sigma^2 in four-term partials into a TwoSum pair.  bf16 inputs: u^2 with
// u = x / sigma - mu / sigma, two FMAs per term.  The softmax over K: the row's maximum and sum are reduced
// over the 16 threads that hold it; above 64 components a first sweep keeps a running maximum and
// sum per row, and a second recomputes the logits and writes gamma_k = exp(L_k - max) / sum.
// fp32 inputs take the logits as TwoSum pairs: the maximum is taken over the high parts and
// exp((hi_k - m) + lo_k) is evaluated with the subtraction first.
constexpr int RT = 64;    // components per tile
constexpr int RLD = 68;   // row stride of the transposed tiles (a multiple of 4, not of 8)

template <int DR>
__host__ __device__ constexpr int resp_smem_floats() { return 3 * DR * RLD + RT; }

// blockIdx.y picks the side: routing vectors X0 (N0 per slice) into gamma0, or X1 (N1) into gamma1.
template <int DR, typename Tin, typename Tout>
__global__ void __launch_bounds__(THREADS, sizeof(Tin) == 4 ? 2 : 4) simt_resp_kernel(const Tin *__restrict__ X0, const Tin *__restrict__ X1,
                                                              const float *__restrict__ mu,
                                                              const float *__restrict__ inv_var,
                                                              const float *__restrict__ cst, Tout *__restrict__ gamma0,
                                                              Tout *__restrict__ gamma1, int B, int H, int N0, int N1,
                                                              int K)
{
    chain_enter();
    const int N = blockIdx.y ? N1 : N0, nseg = (N + SEG - 1) / SEG;
    if ((int)blockIdx.x >= B * H * nseg) return;
    const Tin *X = blockIdx.y ? X1 : X0;
    Tout *gamma = blockIdx.y ? gamma1 : gamma0;
    constexpr bool PRECISE = sizeof(Tin) == 4;
    extern __shared__ __align__(16) float smr[];
    float *xT = smr;                 // [DR][RLD] x^T
    float *mT = xT + DR * RLD;       // [DR][RLD] mu^T of the tile
    float *wT = mT + DR * RLD;       // [DR][RLD] (1 / sigma^2)^T of the tile
    float *cs = wT + DR * RLD;       // [RT]      log pi_k - 1/2 sum_d log sigma^2_kd
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg, h = bh % H;
    const int n = min(SEG, N - seg * SEG);
    const long long row0 = (long long)bh * N + seg * SEG;
    const int t = threadIdx.x, tx = t & 15, r0 = (t >> 4) * 4;
    // staged pair: mu^T and (1 / sigma^2)^T for fp32 inputs; (-mu / sigma)^T and (1 / sigma)^T for
    // bf16 inputs, whose terms are then u = x / sigma - mu / sigma (one FMA) and u^2 (one more)
    const size_t HKD = (size_t)H * K * DR;
    const float *muTh = inv_var + (PRECISE ? 1 : 4) * HKD + (size_t)h * DR * K;
    const float *ivTh = inv_var + (PRECISE ? 2 : 3) * HKD + (size_t)h * DR * K;
    const float *ch = cst + (size_t)h * K;
#pragma unroll 8
    for (int e = t; e < SEG * DR; e += THREADS) {
        const int r = e / DR, d = e % DR;
        xT[d * RLD + r] = r < n ? to_f32(X[(row0 + r) * DR + d]) : 0.f;
    }
    // logits of the tile starting at k0 into hi (and lo); -inf beyond K
    float hi[4][4], lo[4][4];
    auto logits = [&](int k0) {
        const int kn = min(RT, K - k0);
        __syncthreads();
#pragma unroll 8
        for (int e = t; e < RT * DR; e += THREADS) {   // rows of the transposes: coalesced, conflict-free
            const int d = e / RT, kk = e % RT;
            const bool ok = kk < kn;
            mT[d * RLD + kk] = ok ? muTh[(size_t)d * K + k0 + kk] : 0.f;
            wT[d * RLD + kk] = ok ? ivTh[(size_t)d * K + k0 + kk] : 0.f;
        }
        if (t < RT) cs[t] = t < kn ? ch[k0 + t] : 0.f;
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                hi[r][c] = PRECISE ? cs[4 * tx + c] : 0.f;
                lo[r][c] = 0.f;
            }
        if constexpr (PRECISE) {
            for (int d0 = 0; d0 < DR; d0 += 4) {
                float p[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) p[r][c] = 0.f;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int d = d0 + u;
                    const float4 a = *reinterpret_cast<const float4 *>(xT + d * RLD + r0);
                    const float4 m = *reinterpret_cast<const float4 *>(mT + d * RLD + 4 * tx);
                    const float4 w = *reinterpret_cast<const float4 *>(wT + d * RLD + 4 * tx);
                    const float av[4] = {a.x, a.y, a.z, a.w}, mv[4] = {m.x, m.y, m.z, m.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float q = av[r] - mv[c];
                            p[r][c] = fmaf(q * q, wv[c], p[r][c]);
                        }
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) two_sum_acc(hi[r][c], lo[r][c], -0.5f * p[r][c]);
            }
        } else {
#pragma unroll 4
            for (int d = 0; d < DR; ++d) {
                const float4 a = *reinterpret_cast<const float4 *>(xT + d * RLD + r0);
                const float4 m = *reinterpret_cast<const float4 *>(mT + d * RLD + 4 * tx);
                const float4 w = *reinterpret_cast<const float4 *>(wT + d * RLD + 4 * tx);
                const float av[4] = {a.x, a.y, a.z, a.w}, mv[4] = {m.x, m.y, m.z, m.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float u = fmaf(av[r], wv[c], mv[c]);   // (x - mu) / sigma
                        hi[r][c] = fmaf(u, u, hi[r][c]);
                    }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) hi[r][c] = fmaf(-0.5f, hi[r][c], cs[4 * tx + c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (4 * tx + c >= kn)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    hi[r][c] = -INFINITY;
                    lo[r][c] = 0.f;
                }
    };
    auto rmax16 = [](float v) {
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        return v;
    };
    auto rsum16 = [](float v) {
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    };
    float m[4], ssum[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        m[r] = -INFINITY;
        ssum[r] = 0.f;
    }
    for (int k0 = 0; k0 < K; k0 += RT) {
        logits(k0);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float tm = rmax16(fmaxf(fmaxf(hi[r][0], hi[r][1]), fmaxf(hi[r][2], hi[r][3])));
            const float nm = fmaxf(m[r], tm);
            float e = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) e += expf((hi[r][c] - nm) + lo[r][c]);
            ssum[r] = ssum[r] * expf(m[r] - nm) + rsum16(e);
            m[r] = nm;
        }
    }
    for (int k0 = 0; k0 < K; k0 += RT) {
        if (K > RT) logits(k0);   // (one tile: its logits are still in registers)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float inv = 1.f / ssum[r];
            if (r0 + r < n)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int k = k0 + 4 * tx + c;
                    if (k < K) gamma[(row0 + r0 + r) * K + k] = from_f32<Tout>(expf((hi[r][c] - m[r]) + lo[r][c]) * inv);
                }
        }
    }
}

// ---------------------------------------------------------------- write phase, per segment
// agg[bh][seg][k][c] = sum_{j in seg} gamma_K[j][k] * [v_j | 1][c],  c in [0, d_v], for one tile of
// 64 components (blockIdx.y): a register-tiled product over the staged Gamma_K tile and value rows
// (simt_tile.cuh), summed over j in order.
template <int DV, typename Tin>
__global__ void __launch_bounds__(THREADS, 2) simt_state_kernel(const float *__restrict__ gk, const Tin *__restrict__ V,
                                                            float *__restrict__ agg, int N, int K, int nseg)
{
    chain_enter();
    __shared__ __align__(16) float sg[SEG * 64];   // Gamma_K tile [j][k]
    __shared__ __align__(16) float sv[SEG * DV];   // value rows [j][c]
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg, k0 = blockIdx.y * 64;
    const int j0 = seg * SEG, jn = min(SEG, N - j0), kn = min(64, K - k0);
    const long long row0 = (long long)bh * N + j0;
    tile::stage<64>(sg, 64, gk + row0 * K + k0, K, jn, kn);
    tile::stage<DV>(sv, DV, V + row0 * DV, DV, jn, DV);
    __syncthreads();
    float acc[4][DV / 16];
    tile::zero<DV>(acc);
    tile::mac<DV>(acc, sg, 64, sv, DV, SEG);   // rows k, columns c
    float *out = agg + ((size_t)bh * nseg + seg) * K * (DV + 1);
    const int r0 = tile::orow();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int k = k0 + r0 + r;
        if (k < K)
#pragma unroll
            for (int c = 0; c < DV / 16; ++c) out[(size_t)k * (DV + 1) + tile::ocol<DV>(c)] = acc[r][c];
    }
    {   // Z: four threads per component (t / 4), rows t % 4, t % 4 + 4, ... then two shuffles
        const int t = threadIdx.x, k = t >> 2;
        float z = 0.f;
#pragma unroll 4
        for (int jj = t & 3; jj < SEG; jj += 4) z += sg[jj * 64 + k];
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        if ((t & 3) == 0 && k < kn) out[(size_t)(k0 + k) * (DV + 1) + DV] = z;
    }
}

// Causal: replace each segment's partial by the exclusive prefix over earlier segments.
// Bidirectional: write the total over all segments into segment 0's slot.  One thread per V4
// consecutive elements of the K x (d_v + 1) memory (16-byte accesses when K (d_v + 1) is a multiple
// of 4); the loads of 16 segments are issued before their sums.
template <int V4>
__global__ void simt_scan_kernel(float *__restrict__ agg, long long total, int nseg, int KD,
                                 int causal)
{
    chain_enter();
    typedef typename std::conditional<V4 == 4, float4, float>::type vec;
    const long long idx = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * V4;
    if (idx >= total) return;
    const long long bh = idx / KD, e = idx % KD;
    vec *base = reinterpret_cast<vec *>(agg + bh * nseg * KD + e);
    const size_t step = (size_t)KD / V4;
    vec run = tile::vzero<vec>();
    for (int s0 = 0; s0 < nseg; s0 += 16) {
        vec a[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) a[u] = s0 + u < nseg ? base[(size_t)(s0 + u) * step] : tile::vzero<vec>();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (s0 + u >= nseg) break;
            if (causal) base[(size_t)(s0 + u) * step] = run;
            run = tile::vadd(run, a[u]);
        }
    }
    if (!causal) base[0] = run;
}

// ---------------------------------------------------------------- read phase, per segment
// O_i = (gamma_Q,i S + sum_{j<=i in seg} P_ij v_j) / (gamma_Q,i Z + sum_{j<=i in seg} P_ij + eps)
// with P = Gamma_Q Gamma_K^T on the segment (causal only) and [S | Z] the segment's memory.
// agg_nseg: segments per slice in agg (the key side's; equal to nseg but for cross-attention).
template <typename Tin, typename Tout>
__global__ void simt_out_kernel(const float *__restrict__ gq, const float *__restrict__ gk,
                                const Tin *__restrict__ V, const float *__restrict__ agg,
                                Tout *__restrict__ O, int N, int K, int d_v, int nseg, int agg_nseg,
                                float eps, int causal)
{
    chain_enter();
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int i0 = seg * SEG, in = min(SEG, N - i0);
    const int DV1 = d_v + 1;
    const float *S = agg + ((size_t)bh * agg_nseg + (causal ? seg : 0)) * K * DV1;
    const float *gqs = gq + ((size_t)bh * N + i0) * K;
    const float *gks = gk + ((size_t)bh * N + i0) * K;
    __shared__ float P[SEG][SEG + 1];
    __shared__ float sq[SEG][KT + 1];
    __shared__ float sk[SEG][KT + 1];
    __shared__ float den[SEG];

    if (causal) {
        float acc[SEG * SEG / THREADS];
#pragma unroll
        for (int r = 0; r < SEG * SEG / THREADS; ++r) acc[r] = 0.f;
        for (int k0 = 0; k0 < K; k0 += KT) {
            const int kn = min(KT, K - k0);
            for (int e = threadIdx.x; e < SEG * KT; e += blockDim.x) {
                const int i = e / KT, kk = e % KT;
                const bool ok = i < in && kk < kn;
                sq[i][kk] = ok ? gqs[(size_t)i * K + k0 + kk] : 0.f;
                sk[i][kk] = ok ? gks[(size_t)i * K + k0 + kk] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < SEG * SEG / THREADS; ++r) {
                const int e = threadIdx.x + r * THREADS;
                const int i = e / SEG, j = e % SEG;
                float a = acc[r];
                for (int kk = 0; kk < KT; ++kk) a = fmaf(sq[i][kk], sk[j][kk], a);
                acc[r] = a;
            }
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < SEG * SEG / THREADS; ++r) {
            const int e = threadIdx.x + r * THREADS;
            const int i = e / SEG, j = e % SEG;
            P[i][j] = (j <= i && i < in) ? acc[r] : 0.f;
        }
        __syncthreads();
    }
    // denominators first (column d_v of the memory), then numerators
    for (int i = threadIdx.x; i < in; i += blockDim.x) {
        float d = 0.f;
        for (int k = 0; k < K; ++k) d = fmaf(gqs[(size_t)i * K + k], S[(size_t)k * DV1 + d_v], d);
        if (causal)
            for (int j = 0; j <= i; ++j) d += P[i][j];
        den[i] = d + eps;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < in * d_v; e += blockDim.x) {
        const int i = e / d_v, c = e % d_v;
        float n = 0.f;
        for (int k = 0; k < K; ++k) n = fmaf(gqs[(size_t)i * K + k], S[(size_t)k * DV1 + c], n);
        if (causal)
            for (int j = 0; j <= i; ++j)
                n = fmaf(P[i][j], to_f32(V[((size_t)bh * N + i0 + j) * d_v + c]), n);
        O[((size_t)bh * N + i0 + i) * d_v + c] = from_f32<Tout>(n / den[i]);
    }
}

// ---------------------------------------------------------------- one launch for short slices
// Bidirectional and cross-attention calls whose slices are short: one CTA per (b, h) slice runs
// every step above in shared memory, with the same arithmetic in the same order -- the head's
// parameters (as simt_params_kernel), Gamma_Q and Gamma_K (as simt_resp_kernel), the memory
// summed per SEG-token segment and the segments then added in order (as simt_state_kernel and
// simt_scan_kernel), and the read (as simt_out_kernel) -- in one launch instead of five.
// Shared memory (floats): 1/sigma^2 [K][DR], constants [K], Gamma_Q [N][K], Gamma_K [NK][K],
// the value rows [NK][d_v], per-segment memories [nseg][K][d_v + 1], [S | Z] [K][d_v + 1],
// normalisers [N].
template <int DR>
constexpr int small_threads() { return DR <= 32 ? 1024 : DR == 64 ? 512 : 256; }   // (registers: x[DR])

template <int DR, typename Tin, typename Tout>
__global__ void __launch_bounds__(small_threads<DR>()) simt_small_kernel(
    const Tin *__restrict__ QX, const Tin *__restrict__ KX, const Tin *__restrict__ V, const float *__restrict__ mu,
    const float *__restrict__ raw, const float *__restrict__ logits, Tout *__restrict__ O, int H, int N, int NK, int K,
    int d_v, float floor_, float eps)
{
    chain_enter();
    constexpr bool PRECISE = sizeof(Tin) == 4;
    constexpr int NT = small_threads<DR>();
    extern __shared__ float sm[];
    const int bh = blockIdx.x, h = bh % H, DV1 = d_v + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nseg = (NK + SEG - 1) / SEG;
    float *iv = sm;
    float *cs = iv + (size_t)K * DR;
    float *gq = cs + K;
    float *gk = gq + (size_t)N * K;
    float *vs = gk + (size_t)NK * K;
    float *part = vs + (size_t)NK * d_v;
    float *S = part + (size_t)nseg * K * DV1;
    float *den = S + (size_t)K * DV1;

    // the slice's value rows, by coalesced loads (used after the responsibilities)
    const Tin *Vs = V + (size_t)bh * NK * d_v;
    for (int e = threadIdx.x; e < NK * d_v; e += NT) vs[e] = to_f32(Vs[e]);
    // the head's parameters: one warp per component
    const float *lh = logits + (size_t)h * K;
    for (int k = warp; k < K; k += NT / 32) {
        const float *rk = raw + ((size_t)h * K + k) * DR;
        float rv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rv[i] = lane + 32 * i < DR ? rk[lane + 32 * i] : 0.f;
        float m = -INFINITY;
        for (int j = lane; j < K; j += 32) m = fmaxf(m, lh[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
        for (int j = lane; j < K; j += 32) sum += expf(lh[j] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float lse = m + logf(sum);
        double logdet = 0.0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int d = lane + 32 * i;
            if (d < DR) {
                const float r = rv[i];
                const float var = fmaxf(r, 0.f) + log1pf(expf(-fabsf(r))) + floor_;
                iv[k * DR + d] = 1.0f / var;
                logdet += log((double)var);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) logdet += __shfl_xor_sync(0xffffffffu, logdet, o);
        if (lane == 0) cs[k] = (float)(((double)lh[k] - (double)lse) - 0.5 * logdet);
    }
    __syncthreads();

    // Gamma_Q and Gamma_K: one thread per routing vector
    const float *muh = mu + (size_t)h * K * DR;
    for (int r = threadIdx.x; r < N + NK; r += NT) {
        const bool q = r < N;
        const int row = q ? r : r - N;
        const Tin *xr = q ? QX + ((size_t)bh * N + row) * DR : KX + ((size_t)bh * NK + row) * DR;
        float x[DR];
#pragma unroll
        for (int d = 0; d < DR; ++d) x[d] = to_f32(xr[d]);
        auto logit = [&](int k) -> float2 {
            if (PRECISE) return logit_direct_pair<DR, false>(x, muh + (size_t)k * DR, iv + k * DR, cs[k]);
            return make_float2(logit_direct<DR, false>(x, muh + (size_t)k * DR, iv + k * DR, cs[k]), 0.f);
        };
        float m = -INFINITY, sum = 0.f;
        for (int k = 0; k < K; ++k) {
            const float2 L = logit(k);
            if (L.x > m) {
                sum = sum * expf(m - L.x) + expf(L.y);
                m = L.x;
            } else {
                sum += expf((L.x - m) + L.y);
            }
        }
        const float inv = 1.f / sum;
        float *g = (q ? gq : gk) + (size_t)row * K;
        for (int k = 0; k < K; ++k) {
            const float2 L = logit(k);
            g[k] = expf((L.x - m) + L.y) * inv;
        }
    }
    __syncthreads();

    // [S | Z]: each segment's sum (as the segment pass), then the segments added in order
    for (int e = threadIdx.x; e < nseg * K * DV1; e += NT) {
        const int sg = e / (K * DV1), o = e % (K * DV1), kk = o / DV1, c = o % DV1;
        const int j0 = sg * SEG, jn = min(SEG, NK - j0);
        float acc = 0.f;
        if (c < d_v) {
            for (int j = 0; j < jn; ++j) acc = fmaf(gk[(size_t)(j0 + j) * K + kk], vs[(size_t)(j0 + j) * d_v + c], acc);
        } else {
            for (int j = 0; j < jn; ++j) acc += gk[(size_t)(j0 + j) * K + kk];
        }
        part[e] = acc;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < K * DV1; e += NT) {
        float run = 0.f;
        for (int sg = 0; sg < nseg; ++sg) run += part[(size_t)sg * K * DV1 + e];
        S[e] = run;
    }
    __syncthreads();

    // the read: normalisers, then numerators
    for (int i = threadIdx.x; i < N; i += NT) {
        float d = 0.f;
        for (int k = 0; k < K; ++k) d = fmaf(gq[(size_t)i * K + k], S[(size_t)k * DV1 + d_v], d);
        den[i] = d + eps;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < N * d_v; e += NT) {
        const int i = e / d_v, c = e % d_v;
        float n = 0.f;
        for (int k = 0; k < K; ++k) n = fmaf(gq[(size_t)i * K + k], S[(size_t)k * DV1 + c], n);
        O[((size_t)bh * N + i) * d_v + c] = from_f32<Tout>(n / den[i]);
    }
}

// Shared memory of simt_small_kernel (0: the shape takes the five launches).
size_t small_smem_bytes(const gma_shape_t &s, bool causal, int n_k)
{
    if (causal || s.N > 512 || n_k > 512) return 0;
    const size_t dv1 = (size_t)s.d_v + 1, nseg = (size_t)(n_k + SEG - 1) / SEG;
    const size_t f = (size_t)s.K * s.d_r + s.K + (size_t)s.N * s.K + (size_t)n_k * s.K + (size_t)n_k * s.d_v +
                     nseg * s.K * dv1 + (size_t)s.K * dv1 + s.N;
    return f * 4 <= 160 * 1024 ? f * 4 : 0;
}

// ---------------------------------------------------------------- host side
struct SimtLayout {
    size_t inv_var, cst, gq, gk, agg, total;
    int nseg;
};

// n_k: keys per slice (s.N but for cross-attention); L.nseg splits the keys.
SimtLayout simt_layout(const gma_shape_t &s, int variant, int n_k)
{
    SimtLayout L{};
    Carve c;
    const size_t rows = (size_t)s.B * s.H * s.N;
    const size_t rows_k = (size_t)s.B * s.H * n_k;
    L.inv_var = c.take(5 * sizeof(float) * (size_t)s.H * s.K * s.d_r);   // 1/sigma^2 and four transposes
    L.cst = c.take(sizeof(float) * (size_t)s.H * s.K);
    L.nseg = (n_k + SEG - 1) / SEG;
    if (variant != GMA_VARIANT_RESPONSIBILITIES) {
        L.gq = c.take(sizeof(float) * rows * s.K);
        L.gk = c.take(sizeof(float) * rows_k * s.K);
        L.agg = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * s.K * (s.d_v + 1));
    }
    L.total = c.total();
    return L;
}

SimtLayout simt_layout(const gma_shape_t &s, int variant) { return simt_layout(s, variant, s.N); }

// A launch of this family's kernels: programmatic dependent launch (see chain_enter).
template <typename... P, typename... A>
gma_status_t launch_chained(int kid, cudaStream_t st, void (*k)(P...), dim3 g, dim3 b, A... args)
{
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(kid, st, (e = launch_pdl(k, g, b, 0, st, args...)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

// Responsibilities of X0 (N0 rows per slice) into g0 and, when X1 is given, of X1 (N1) into g1, in
// one launch.
template <int DR, typename Tin, typename Tout>
gma_status_t launch_resp_dr(const Tin *X0, const Tin *X1, const float *mu, const float *iv, const float *cst, Tout *g0,
                            Tout *g1, int B, int H, int N0, int N1, int K, cudaStream_t st)
{
    const int nseg = (max(N0, X1 ? N1 : 0) + SEG - 1) / SEG;
    const int smem = (int)sizeof(float) * resp_smem_floats<DR>();
    if (cudaFuncSetAttribute(simt_resp_kernel<DR, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return GMA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_SIMT_RESP, st,
               (e = launch_pdl(simt_resp_kernel<DR, Tin, Tout>, dim3((unsigned)(B * H * nseg), X1 ? 2u : 1u),
                               dim3(THREADS), (size_t)smem, st, X0, X1, mu, iv, cst, g0, g1, B, H, N0, N1, K)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template <typename Tin, typename Tout>
gma_status_t launch_resp(int d_r, const Tin *X0, const Tin *X1, const float *mu, const float *iv, const float *cst,
                         Tout *g0, Tout *g1, int B, int H, int N0, int N1, int K, cudaStream_t st)
{
    switch (d_r) {
    case 16: return launch_resp_dr<16, Tin, Tout>(X0, X1, mu, iv, cst, g0, g1, B, H, N0, N1, K, st);
    case 32: return launch_resp_dr<32, Tin, Tout>(X0, X1, mu, iv, cst, g0, g1, B, H, N0, N1, K, st);
    case 64: return launch_resp_dr<64, Tin, Tout>(X0, X1, mu, iv, cst, g0, g1, B, H, N0, N1, K, st);
    case 128: return launch_resp_dr<128, Tin, Tout>(X0, X1, mu, iv, cst, g0, g1, B, H, N0, N1, K, st);
    default: return GMA_ERR_UNSUPPORTED_SHAPE;
    }
}

// Everything the read phase needs: the parameters, Gamma_Q and Gamma_K (fp32), and the segment
// memories [S | Z] scanned (causal: exclusive prefix per segment; bidirectional: the total in
// segment 0).  s.N queries and n_k keys per slice; nseg splits the keys into SEG-token segments.
template <typename Tin>
gma_status_t prepare_typed(const gma_shape_t &s, bool causal, int n_k, const Tin *QX, const Tin *KX,
                           const Tin *V, const float *mu, const float *raw, const float *logits, float *iv,
                           float *cst, float *gq, float *gk, float *agg, int nseg, cudaStream_t st)
{
    gma_status_t r = launch_chained(KID_SIMT_PARAMS, st, simt_params_kernel, dim3((unsigned)s.H, (unsigned)((s.K + PARAM_THREADS / 32 - 1) / (PARAM_THREADS / 32))),
                                    dim3(PARAM_THREADS), raw, logits, mu, iv, cst, s.K, s.d_r, s.var_floor);
    if (r != GMA_OK) return r;
    r = launch_resp<Tin, float>(s.d_r, QX, KX, mu, iv, cst, gq, gk, s.B, s.H, s.N, n_k, s.K, st);
    if (r != GMA_OK) return r;
    const int BH = s.B * s.H;
    dim3 gs((unsigned)(BH * nseg), (unsigned)((s.K + 63) / 64));
    switch (s.d_v) {
    case 16: r = launch_chained(KID_SIMT_STATE, st, simt_state_kernel<16, Tin>, gs, dim3(THREADS), gk, V, agg, n_k, s.K, nseg); break;
    case 32: r = launch_chained(KID_SIMT_STATE, st, simt_state_kernel<32, Tin>, gs, dim3(THREADS), gk, V, agg, n_k, s.K, nseg); break;
    case 64: r = launch_chained(KID_SIMT_STATE, st, simt_state_kernel<64, Tin>, gs, dim3(THREADS), gk, V, agg, n_k, s.K, nseg); break;
    case 128: r = launch_chained(KID_SIMT_STATE, st, simt_state_kernel<128, Tin>, gs, dim3(THREADS), gk, V, agg, n_k, s.K, nseg); break;
    default: return GMA_ERR_UNSUPPORTED_SHAPE;
    }
    if (r != GMA_OK) return r;
    const int KD = s.K * (s.d_v + 1);
    const long long tot = (long long)BH * KD;
    if (KD % 4 == 0)
        return launch_chained(KID_SIMT_SCAN, st, simt_scan_kernel<4>, dim3((unsigned)((tot / 4 + 255) / 256)), dim3(256),
                              agg, tot, nseg, KD, causal ? 1 : 0);
    return launch_chained(KID_SIMT_SCAN, st, simt_scan_kernel<1>, dim3((unsigned)((tot + 255) / 256)), dim3(256), agg,
                          tot, nseg, KD, causal ? 1 : 0);
}

// The one-launch path for short bidirectional slices (simt_small_kernel).
template <typename Tin, typename Tout>
gma_status_t launch_small(const gma_shape_t &s, int n_k, const Tin *QX, const Tin *KX, const Tin *V, const float *mu,
                          const float *raw, const float *logits, Tout *O, size_t smem, cudaStream_t st)
{
    const dim3 g((unsigned)(s.B * s.H));
    cudaError_t e = cudaSuccess;
    switch (s.d_r) {
    case 16:
        if (cudaFuncSetAttribute(simt_small_kernel<16, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_SIMT_SMALL, st, (e = launch_pdl(simt_small_kernel<16, Tin, Tout>, g, dim3(small_threads<16>()), smem, st, QX, KX, V, mu, raw, logits, O, s.H, s.N, n_k, s.K, s.d_v, s.var_floor, s.eps))); break;
    case 32:
        if (cudaFuncSetAttribute(simt_small_kernel<32, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_SIMT_SMALL, st, (e = launch_pdl(simt_small_kernel<32, Tin, Tout>, g, dim3(small_threads<32>()), smem, st, QX, KX, V, mu, raw, logits, O, s.H, s.N, n_k, s.K, s.d_v, s.var_floor, s.eps))); break;
    case 64:
        if (cudaFuncSetAttribute(simt_small_kernel<64, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_SIMT_SMALL, st, (e = launch_pdl(simt_small_kernel<64, Tin, Tout>, g, dim3(small_threads<64>()), smem, st, QX, KX, V, mu, raw, logits, O, s.H, s.N, n_k, s.K, s.d_v, s.var_floor, s.eps))); break;
    case 128:
        if (cudaFuncSetAttribute(simt_small_kernel<128, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GMA_ERR_CUDA;
        GMA_LAUNCH(KID_SIMT_SMALL, st, (e = launch_pdl(simt_small_kernel<128, Tin, Tout>, g, dim3(small_threads<128>()), smem, st, QX, KX, V, mu, raw, logits, O, s.H, s.N, n_k, s.K, s.d_v, s.var_floor, s.eps))); break;
    default: return GMA_ERR_UNSUPPORTED_SHAPE;
    }
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

// s.N queries and n_k keys per slice (n_k == s.N for the causal variant).
template <typename Tin, typename Tout>
gma_status_t forward_typed(const gma_shape_t &s, bool causal, int n_k, const Tin *QX, const Tin *KX,
                           const Tin *V, const float *mu, const float *raw, const float *logits,
                           Tout *O, char *ws, cudaStream_t st)
{
    const size_t small = small_smem_bytes(s, causal, n_k);
    if (small) return launch_small<Tin, Tout>(s, n_k, QX, KX, V, mu, raw, logits, O, small, st);
    const SimtLayout L = simt_layout(s, causal ? GMA_VARIANT_CAUSAL : GMA_VARIANT_BIDIRECTIONAL, n_k);
    float *iv = (float *)(ws + L.inv_var), *cst = (float *)(ws + L.cst);
    float *gq = (float *)(ws + L.gq), *gk = (float *)(ws + L.gk), *agg = (float *)(ws + L.agg);
    gma_status_t r = prepare_typed<Tin>(s, causal, n_k, QX, KX, V, mu, raw, logits, iv, cst, gq, gk, agg, L.nseg, st);
    if (r != GMA_OK) return r;
    const int BH = s.B * s.H;
    const int nseg_q = (s.N + SEG - 1) / SEG;
    return launch_chained(KID_SIMT_OUT, st, simt_out_kernel<Tin, Tout>, dim3((unsigned)(BH * nseg_q)), dim3(THREADS), gq,
                          gk, V, agg, O, s.N, s.K, s.d_v, nseg_q, L.nseg, s.eps, causal ? 1 : 0);
}


}  // namespace

gma_status_t simt_prepare(const gma_shape_t &s, bool causal, const void *QX, const void *KX, const void *V,
                          const float *mu, const float *raw, const float *logits, float *iv, float *cst, float *gq,
                          float *gk, float *agg, cudaStream_t st)
{
    const int nseg = (s.N + SEG - 1) / SEG;
    if (s.dtype == GMA_F32)
        return prepare_typed<float>(s, causal, s.N, (const float *)QX, (const float *)KX, (const float *)V, mu, raw,
                                    logits, iv, cst, gq, gk, agg, nseg, st);
    typedef __nv_bfloat16 bf;
    return prepare_typed<bf>(s, causal, s.N, (const bf *)QX, (const bf *)KX, (const bf *)V, mu, raw, logits, iv, cst,
                             gq, gk, agg, nseg, st);
}

size_t simt_workspace_size(const gma_shape_t &s, int variant) { return simt_layout(s, variant).total; }

size_t simt_workspace_size_cross(const gma_shape_t &s, int n_k)
{
    return simt_layout(s, GMA_VARIANT_BIDIRECTIONAL, n_k).total;
}

gma_status_t simt_responsibilities(const gma_shape_t &s, const void *X, const float *mu,
                                   const float *raw, const float *logits, void *gamma, void *ws,
                                   cudaStream_t st)
{
    const SimtLayout L = simt_layout(s, GMA_VARIANT_RESPONSIBILITIES);
    char *w = (char *)ws;
    float *iv = (float *)(w + L.inv_var), *cst = (float *)(w + L.cst);
    const gma_status_t r = launch_chained(KID_SIMT_PARAMS, st, simt_params_kernel,
                                          dim3((unsigned)s.H, (unsigned)((s.K + PARAM_THREADS / 32 - 1) / (PARAM_THREADS / 32))), dim3(PARAM_THREADS), raw,
                                          logits, mu, iv, cst, s.K, s.d_r, s.var_floor);
    if (r != GMA_OK) return r;
    const bool out32 = (s.flags & GMA_FLAG_OUT_F32) || s.dtype == GMA_F32;
    if (s.dtype == GMA_F32)
        return launch_resp<float, float>(s.d_r, (const float *)X, (const float *)nullptr, mu, iv, cst, (float *)gamma, (float *)nullptr, s.B, s.H, s.N, 0, s.K, st);
    if (out32)
        return launch_resp<__nv_bfloat16, float>(s.d_r, (const __nv_bfloat16 *)X, (const __nv_bfloat16 *)nullptr, mu, iv, cst, (float *)gamma, (float *)nullptr, s.B, s.H, s.N, 0, s.K, st);
    return launch_resp<__nv_bfloat16, __nv_bfloat16>(s.d_r, (const __nv_bfloat16 *)X, (const __nv_bfloat16 *)nullptr, mu, iv, cst, (__nv_bfloat16 *)gamma, (__nv_bfloat16 *)nullptr, s.B, s.H, s.N, 0, s.K, st);
}

gma_status_t simt_forward(const gma_shape_t &s, bool causal, int n_k, const void *QX, const void *KX,
                          const void *V, const float *mu, const float *raw, const float *logits,
                          void *O, void *ws, cudaStream_t st)
{
    char *w = (char *)ws;
    if (s.dtype == GMA_F32)
        return forward_typed<float, float>(s, causal, n_k, (const float *)QX, (const float *)KX,
                                           (const float *)V, mu, raw, logits, (float *)O, w, st);
    typedef __nv_bfloat16 bf;
    if (s.flags & GMA_FLAG_OUT_F32)
        return forward_typed<bf, float>(s, causal, n_k, (const bf *)QX, (const bf *)KX, (const bf *)V,
                                        mu, raw, logits, (float *)O, w, st);
    return forward_typed<bf, bf>(s, causal, n_k, (const bf *)QX, (const bf *)KX, (const bf *)V, mu,
                                 raw, logits, (bf *)O, w, st);
}

}  // namespace gma
