// gma_tc.cu -- the tcgen05 tensor-core kernel family of libgma.so (bf16 inputs, sm_103a).
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §1 (posterior responsibilities), §2 (write phase V~ = Gamma_K^T V, Z = Gamma_K^T 1;
// read phase O = Gamma_Q V~ / (Gamma_Q Z + eps)), §3 (causal variant by prefix sums; softplus
// variances and softmax priors).
//
// GB300 design.
//  * The diagonal-Gaussian log-density is expanded into one dense contraction per token:
//      log2e * L_k = [x^2 , x] . [-w_k/2 ; mu_k w_k] * log2e + c_k,   w = 1/sigma^2,
//    an M=128 x N=K x K=2 d_r tcgen05.mma (fp16 operands, fp32 accumulators in TMEM).  The
//    softmax over K runs on the CUDA cores straight out of TMEM (one thread per token row).
//  * Gamma stays on chip (shared memory, bf16).  Write, read and the causal chunk products are
//    tcgen05.mma with bf16 operands and fp32 accumulation.  The normaliser rides along as an
//    extra block of ones next to V (16 extra MMA columns), so Z and Gamma_Q Z come out of the
//    same MMAs as V~ and Gamma_Q V~.
//  * Causal: the sequence is cut into chunks of C = 128 tokens.  Per chunk
//      O_c = (Gamma_Q,c S_{c-1} + tril(Gamma_Q,c Gamma_K,c^T) [V_c, 1])  (numerator | normaliser)
//      S_c = S_{c-1} + Gamma_K,c^T [V_c, 1]
//    with the running memory S (K x (d_v+16), fp32) in TMEM.  Chunks are grouped into segments
//    handled by different CTAs; a first kernel writes each segment's memory, a scan turns them
//    into exclusive prefixes, and the chunked kernel starts each segment from its prefix.
//  * Gamma_Q is kept unnormalised (row maximum 1); with row sum s_i the read is
//      O_i = num_i / (den_i + eps * s_i),
//    which equals the page's O_i exactly.
//
// Shared-memory operand layouts (all written either by TMA or by the CUDA cores with the same
// address swizzle the tensor cores read):
//  * K-major, 128-byte swizzle: rows of 64 two-byte elements (128 B), 8-row groups of 1 KB,
//    64-element column blocks ("atoms") stacked after each other; chunk q of row r lives at
//    16 * ((q % 8) ^ (r % 8)).  Used for [x^2, x], the Gaussian table, Gamma_Q, Gamma_K, P.
//  * MN-major, 32-byte swizzle: blocks of 16 columns x rows, 32 B per row; the two 16-byte
//    halves of row r are swapped when bit 2 of r is set.  Used for [V | 1] and the memory S.
#include <cuda.h>
#include <mutex>

#include <cstring>

#include "tc_common.cuh"

namespace gma {
namespace tck {

using namespace tc;

// Shared-memory plan of one CTA.  Regions are 1 KB aligned.
struct Smem {
    uint32_t bimg, abuf, gk, gq, ve, sp, cst, bars, tslot, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ Smem(int DR, int kn16, int d_v, bool need_k, bool need_q, bool need_sp)
    {
        const int ka = DR * 2 < 64 ? 64 : DR * 2;
        const uint32_t tile_bytes = (uint32_t)(ka / 64) * 128u;   // per row of a K-major tile
        uint32_t o = 0;
        bimg = o; o = al(o + tile_bytes * (uint32_t)kn16 + 32u * (uint32_t)kn16);
        abuf = o; o = al(o + tile_bytes * (uint32_t)C);
        gk = o; if (need_k) o = al(o + 2u * C * 128u);
        gq = o; if (need_q) o = al(o + 2u * C * 128u);
        ve = o; if (need_k) o = al(o + (uint32_t)(d_v + 16) * C * 2u);
        sp = o; if (need_sp) o = al(o + (uint32_t)(d_v + 16) * KMAX * 2u);
        cst = o; o += KMAX * 4;
        bars = o; o += 8 * 8;
        tslot = o; o += 16;
        total = o;
    }
};

struct Bars {
    uint64_t *bimg, *v, *mma, *mma2;
};

// Issues the logits MMA  L[tmem d] = A[abuf] * B[bimg]^T  (M = 128 tokens, N = kn16, K = ka).
template <int DR>
__device__ __forceinline__ void issue_logits(uint32_t d, uint32_t abuf, uint32_t bimg, int kn16)
{
    constexpr int KA = DR * 2 < 64 ? 64 : DR * 2;
    const uint32_t id = idesc_f16(128, (uint32_t)kn16, 0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < KA / 16; ++s) mma_f16(d, kdesc(abuf, s, C), kdesc(bimg, s, kn16), id, s > 0);
}


__device__ __forceinline__ void sync_tc()
{
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Everything written to shared memory by the CUDA cores becomes visible to the tensor cores.
__device__ __forceinline__ void publish_smem()
{
    fence_proxy_async_smem();
    sync_tc();
}

// Common CTA prologue: barriers, TMEM, Gaussian table and constants.
__device__ __forceinline__ void cta_setup(uint8_t *smem, const Smem &L, Bars &bars, uint32_t ncols,
                                          const Args &a, int h, uint32_t &tmem)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + L.bars);
    bars.bimg = b;
    bars.v = b + 1;
    bars.mma = b + 2;
    bars.mma2 = b + 3;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.tslot);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(b + i, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) tmem_alloc(tslot, ncols);
    float *cst = reinterpret_cast<float *>(smem + L.cst);
    for (int k = threadIdx.x; k < KMAX; k += THREADS)
        cst[k] = k < a.kn16 ? a.cst[(size_t)h * (a.bimg_head / a.bimg_bytes) * a.kn16 + a.tile * a.kn16 + k] : NEG_BIG;
    sync_tc();
    tmem = *tslot;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bars.bimg, (uint32_t)a.bimg_bytes);
        bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars.bimg);
    }
}

__device__ __forceinline__ void cta_teardown(uint32_t tmem, uint32_t ncols)
{
    sync_tc();
    if (threadIdx.x < 32) tmem_dealloc(tmem, ncols);
}

// All threads wait; returns false on every thread if any of them timed out.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t &phase, WsHeader *hdr, unsigned where)
{
    const bool ok = mbar_wait(bar, phase, hdr, where);
    phase ^= 1u;
    return !__syncthreads_or(!ok);
}


// ================================================================== kernels

// Per head h (grid.x) and group of 8 components (grid.y): the Gaussian table (main part
// log2e * [-w/2 ; mu w] as fp16, K-major SW128, kn16 rows; const part (c_hi, c_lo) with
// c_hi + c_lo = c_k = log2e * (log pi_k - 1/2 sum_d (mu^2 w + log sigma^2)), K-major SW32) and
// the fp32 constants cst[h][k] = c_k.  w = 1 / (softplus(raw) + floor), log pi = log softmax.
// Padded components (k >= K) get zero rows.  Values beyond fp16 range are reported as
// GMA_ERR_RANGE.  Each component is handled by 16 consecutive threads (grid.y: groups of 8
// components), one 16-byte feature chunk at a time; their partial sums meet through warp shuffles.
__global__ void __launch_bounds__(THREADS) tc_params_kernel(const float *__restrict__ mu,
                                                            const float *__restrict__ raw,
                                                            const float *__restrict__ logits,
                                                            uint8_t *__restrict__ bimg,
                                                            float *__restrict__ cst, int K, int kn16,
                                                            int d_r, int bimg_bytes, int main_bytes,
                                                            int ntile, float floor_, WsHeader *hdr)
{
    // With more than 128 components (ntile > 1) the head's image is ntile complete images of 128
    // rows each (kn16 = 128): component n sits in tile n / 128, row n % 128.
    grid_dependency_launch();   // the segment pass may start; it waits for this grid before reading
    const int h = blockIdx.x;
    const int ka = d_r * 2 < 64 ? 64 : d_r * 2;
    const float *lh = logits + (size_t)h * K;
    // log-sum-exp of the head's prior logits (K <= 1024: up to eight per thread), by warp
    // shuffles and one exchange between the four warps
    __shared__ float red[2][THREADS / 32];
    float m = -INFINITY;
    for (int j = threadIdx.x; j < K; j += THREADS) m = fmaxf(m, lh[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[0][threadIdx.x >> 5] = m;
    __syncthreads();
    m = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
    float sum = 0.f;
    for (int j = threadIdx.x; j < K; j += THREADS) sum += expf(lh[j] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((threadIdx.x & 31) == 0) red[1][threadIdx.x >> 5] = sum;
    __syncthreads();
    const float lse = m + logf((red[1][0] + red[1][1]) + (red[1][2] + red[1][3]));
    const int n = blockIdx.y * 8 + (threadIdx.x >> 4);    // component
    uint8_t *img = bimg + (size_t)h * ntile * bimg_bytes + (size_t)(n / kn16) * bimg_bytes;
    const int nr = n % kn16;                               // its row in its tile's image
    const int sub = threadIdx.x & 15;
    const bool in_table = n < kn16 * ntile;
    const bool real = n < K;
    float acc = 0.f;
    bool range_ok = true;
    if (in_table) {
        for (int q = sub; q < ka / 8; q += 16) {
            // this chunk's raw variances and means, all loaded before any is used
            float rr[8], mm[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int f = q * 8 + j;
                const int d = f < d_r ? f : f - d_r;
                const bool ld = real && f < 2 * d_r;
                rr[j] = ld ? raw[((size_t)h * K + n) * d_r + d] : 0.f;
                mm[j] = ld ? mu[((size_t)h * K + n) * d_r + d] : 0.f;
            }
            uint16_t hv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int f = q * 8 + j;
                float val = 0.f;
                if (real && f < 2 * d_r) {
                    const float r = rr[j];
                    const float var = fmaxf(r, 0.f) + log1pf(expf(-fabsf(r))) + floor_;
                    const float w = 1.0f / var;
                    const float mv = mm[j];
                    if (f < d_r) {
                        val = -0.5f * w * LOG2E;
                        acc += mv * mv * w + logf(var);
                    } else {
                        val = mv * w * LOG2E;
                    }
                    if (!(fabsf(val) < 65504.f)) range_ok = false;
                }
                __half hh = __float2half_rn(val);
                hv[j] = *reinterpret_cast<uint16_t *>(&hh);
            }
            uint4 v;
            v.x = hv[0] | ((uint32_t)hv[1] << 16);
            v.y = hv[2] | ((uint32_t)hv[3] << 16);
            v.z = hv[4] | ((uint32_t)hv[5] << 16);
            v.w = hv[6] | ((uint32_t)hv[7] << 16);
            *reinterpret_cast<uint4 *>(img + sw128(nr, q, kn16)) = v;
        }
    }
    // sum the 16 partial sums of this component (lanes 16g .. 16g+15 of the warp)
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    acc += __shfl_xor_sync(0xffffffffu, acc, 8);
    if (in_table && sub == 0) {
        const float c = real ? ((lh[n] - lse) - 0.5f * acc) * LOG2E : 0.f;
        if (!(fabsf(c) < 65504.f)) range_ok = false;
        const __half hi = __float2half_rn(c);
        const __half lo = __float2half_rn(c - __half2float(hi));
        uint4 half0 = make_uint4(0, 0, 0, 0);
        half0.x = (uint32_t)(*reinterpret_cast<const uint16_t *>(&hi)) |
                  ((uint32_t)(*reinterpret_cast<const uint16_t *>(&lo)) << 16);
        uint8_t *row = img + main_bytes + nr * 32;
        const int flip = (nr >> 2) & 1;
        *reinterpret_cast<uint4 *>(row + (flip << 4)) = half0;
        *reinterpret_cast<uint4 *>(row + ((flip ^ 1) << 4)) = make_uint4(0, 0, 0, 0);
        cst[(size_t)h * kn16 * ntile + n] = real ? c : NEG_BIG;
    }
    if (!range_ok) record_error(hdr, GMA_ERR_RANGE, 1u);
}

// Causal: exclusive prefix of the segment memories within each slice (in place).
// Bidirectional: the total over all segments, written to segment 0.
// One thread per float of one slice's memory; consecutive threads take consecutive floats (each
// load instruction of a warp reads 128 contiguous bytes).  All of a thread's segments (NB at a
// time, NB chosen from the segment count) are loaded before any result is stored, so the loads
// are in flight together.
template <int NB>
// KD: floats per segment memory (the stride); KDu: the leading floats that carry components
// (kn16 rows; the rows beyond are zero in every segment and stay so).
__global__ void __launch_bounds__(256) tc_scan_kernel(float *__restrict__ agg, long long total, int nseg,
                                                      int KD, int KDu, int causal)
{
    grid_dependency_wait();     // the segment memories come from the kernel before
    grid_dependency_launch();
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const long long bh = idx / KDu, e = idx % KDu;
    float *base = agg + bh * nseg * KD + e;
    float run = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += NB) {
        float v[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) v[u] = s0 + u < nseg ? __ldcg(base + (size_t)(s0 + u) * KD) : 0.f;
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            if (causal && s0 + u < nseg) base[(size_t)(s0 + u) * KD] = run;
            run += v[u];
        }
    }
    if (!causal) base[0] = run;
}


// The responsibilities kernel stages its output rows ([C][33] floats) in the [x^2, x] buffer when
// that buffer (ka / 64 x 128 B x C) holds them: d_r >= 64.
__host__ __device__ constexpr bool resp_stage_in_a(int d_r) { return (d_r * 2 < 64 ? 64 : d_r * 2) / 64 * 128 * C >= C * 33 * 4; }

// Responsibilities only: gamma rows (normalised) straight from registers to global memory.
template <int DR>
__global__ void __launch_bounds__(THREADS, 1) tc_resp_kernel(const Args a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Smem L(DR, a.kn16, 16, false, false, false);
    const int ntile = a.nseg;
    const int bh = blockIdx.x / ntile, grp = blockIdx.x % ntile, h = bh % a.H;
    const int t = threadIdx.x, warp = t >> 5;
    const int tok0 = grp * a.cps * C;
    const int tok_end = min(a.N, tok0 + a.cps * C);
    Bars bars;
    uint32_t tmem;
    uint32_t ph_b = 0, ph_m = 0;
    cta_setup(smem, L, bars, 128, a, h, tmem);
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t sb = smem_u32(smem);
    float *cst = reinterpret_cast<float *>(smem + L.cst);
    // the staging tile [C][33]: in the [x^2, x] buffer when that is large enough (it is free between
    // the logits MMA and the next tile's build), else after the layout
    constexpr bool STAGE_IN_A = resp_stage_in_a(DR);
    uint8_t *extra = smem + ((L.total + 127u) & ~127u);
    float *stage = reinterpret_cast<float *>(STAGE_IN_A ? smem + L.abuf : extra);
    // usage diagnostics: histogram and column sums of this CTA's rows, and the column sums' partials
    const bool usage = a.assign != nullptr;
    const bool tiled = a.lse_q != nullptr;   // more than 128 components: this launch does one tile
    int *hist = reinterpret_cast<int *>(STAGE_IN_A ? extra : extra + (size_t)C * 33 * 4);
    float *msum = reinterpret_cast<float *>(hist + KMAX);
    float *cpart = msum + KMAX;   // [4][32]
    if (usage) {
        for (int k = t; k < KMAX; k += THREADS) {
            hist[k] = 0;
            msum[k] = 0.f;
        }
        __syncthreads();
    }
    bool ok = wait_all(bars.bimg, ph_b, a.hdr, 40);
    uint4 x[DR / 8];
    if (ok) load_x<DR>(a.QX, (long long)bh * a.N + tok0 + t, tok0 + t < tok_end, x);
    const int kc = (a.K + 31) >> 5;
    for (int base = tok0; ok && base < tok_end; base += C) {
        const bool valid = base + t < tok_end;
        build_a<DR>(smem + L.abuf, t, x);
        publish_smem();
        if (t == 0) {
            issue_logits<DR>(tmem, sb + L.abuf, sb + L.bimg, a.kn16);
            mma_commit(bars.mma);
        }
        // (components in tiles: the row's log2-sum-exp over all components)
        const float lse = (tiled && valid) ? a.lse_q[(long long)bh * a.N + base + t] : 0.f;
        if (!(ok = wait_all(bars.mma, ph_m, a.hdr, 41))) break;
        const int nb = base + C;
        load_x<DR>(a.QX, (long long)bh * a.N + nb + t, nb + t < tok_end, x);
        // softmax over the row in three passes over TMEM, 32 components at a time (the maximum,
        // with the logits plus their constants stored back; the sum, with the exponentials stored
        // back; then the normalised values), so no thread holds the whole row in registers; with
        // components in tiles, one pass: gamma = exp2(L - lse)
        float m = tiled ? lse : NEG_BIG;
        int arg = 0;   // the first component of largest responsibility
        float inv = 1.f;
        if (!tiled) {
            // (the logits with their constants go back into TMEM for the next pass)
#pragma unroll 1
            for (int c = 0; c < kc; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
                if (c * 32 + 32 <= a.K) {   // (a whole group: no bound tests)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float l = __uint_as_float(r[j]) + cst[c * 32 + j];
                        r[j] = __float_as_uint(l);
                        if (l > m) {
                            m = l;
                            arg = c * 32 + j;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float l = __uint_as_float(r[j]) + cst[c * 32 + j];
                        r[j] = __float_as_uint(l);
                        if (c * 32 + j < a.K && l > m) {
                            m = l;
                            arg = c * 32 + j;
                        }
                    }
                }
                tmem_st16(tmem + lane_off + c * 32, *reinterpret_cast<const uint32_t(*)[16]>(r));
                tmem_st16(tmem + lane_off + c * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(r + 16));
            }
            tmem_st_wait();
            if (usage && valid) {
                a.assign[(long long)bh * a.N + base + t] = arg;
                atomicAdd(&hist[arg], 1);
            }
            // the exponentials go back into the logits' columns, so the last pass only scales them
            float s = 0.f;
#pragma unroll 1
            for (int c = 0; c < kc; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_off + c * 32, r);
                tmem_ld_wait();
                if (c * 32 + 32 <= a.K) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float e = ex2(__uint_as_float(r[j]) - m);
                        s += e;
                        r[j] = __float_as_uint(e);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float e = c * 32 + j < a.K ? ex2(__uint_as_float(r[j]) - m) : 0.f;
                        s += e;
                        r[j] = __float_as_uint(e);
                    }
                }
                tmem_st16(tmem + lane_off + c * 32, *reinterpret_cast<const uint32_t(*)[16]>(r));
                tmem_st16(tmem + lane_off + c * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(r + 16));
            }
            tmem_st_wait();
            inv = 1.0f / s;
        }
        // the tile's rows leave through shared memory, 32 components at a time, so that a warp's
        // global stores cover whole row segments (one thread per row would scatter them)
        const long long row0 = (long long)bh * a.N + base;
        const int nrows = min(C, tok_end - base);
#pragma unroll 1
        for (int c = 0; c < kc; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + c * 32, r);
            tmem_ld_wait();
            if (!tiled && c * 32 + 32 <= a.K) {   // (the stored exponentials of a whole group)
#pragma unroll
                for (int j = 0; j < 32; ++j) stage[t * 33 + j] = __uint_as_float(r[j]) * inv;
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int k = c * 32 + j;
                    stage[t * 33 + j] = k >= a.K ? 0.f
                                       : tiled ? ex2(__uint_as_float(r[j]) + cst[k] - m) * inv
                                               : __uint_as_float(r[j]) * inv;   // (the stored exponential)
                }
            }
            __syncthreads();
            const int ncol = min(32, a.K - c * 32);
            if (usage) {
                // column sums of the tile's rows: each warp a quarter of the rows (q, q + 4, ...),
                // one column per lane (conflict-free), then the four partials in order
                const int j = t & 31, q = t >> 5;
                float cs = 0.f;
#pragma unroll 8
                for (int rr = q; rr < nrows; rr += 4) cs += stage[rr * 33 + j];
                cpart[q * 32 + j] = cs;
                __syncthreads();
                if (t < 32) msum[c * 32 + t] += (cpart[t] + cpart[32 + t]) + (cpart[64 + t] + cpart[96 + t]);
            } else {
                for (int e = t; e < nrows * 32; e += THREADS) {
                    const int rr = e >> 5, j = e & 31;
                    if (j < ncol) {
                        const long long at = (row0 + rr) * a.kall + a.tile * KMAX + c * 32 + j;
                        if (a.out_f32)
                            ((float *)a.gamma)[at] = stage[rr * 33 + j];
                        else
                            ((bf16 *)a.gamma)[at] = __float2bfloat16_rn(stage[rr * 33 + j]);
                    }
                }
            }
            __syncthreads();
        }
        sync_tc();
    }
    if (usage) {
        __syncthreads();
        for (int k = t; k < a.K; k += THREADS) {
            if (hist[k] && !tiled) atomicAdd(&a.counts[(size_t)h * a.K + k], hist[k]);
            a.mass_part[(size_t)blockIdx.x * a.kall + a.tile * KMAX + k] = msum[k];
        }
    }
    cta_teardown(tmem, 128);
}

// ================================================================== host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    });
    return fn;
}

// 3-D map over V [BH][N][d_v] bf16: dims {d_v, N, BH}, box {16, 128, 1}, 32-byte swizzle.
bool make_vmap(CUtensorMap *m, const void *V, int BH, int N, int d_v)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_v, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d_v * 2, (cuuint64_t)N * d_v * 2};
    cuuint32_t box[3] = {16, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same tensor with boxes of 64 columns and the 128-byte swizzle (d_v a multiple of 64): the
// MN-major operand atoms that the tensor cores read most efficiently.
bool make_vmap128(CUtensorMap *m, const void *V, int BH, int N, int d_v)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || d_v % 64 != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_v, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d_v * 2, (cuuint64_t)N * d_v * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(V), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int kn16, ne, ka, bimg_bytes, bimg_main_bytes;
    int ntile;                  // component tiles of 128 (1 when K <= 128)
    size_t off_lse_q, off_lse_k, off_part, off_pden;
    int nseg, cps;              // forward: segments per slice and chunks per segment
    int kg;                     // causal: components per stored key-responsibility row (64 or 128)
    size_t off_bimg, off_cst, off_agg, off_gam, total;
    size_t off_flags, off_incl; // single-launch causal: ticket and flags, inclusive prefixes
};

constexpr int kSms = 152;   // GB300

uint32_t keysmall_smem(int d_r, int K, int d_v);   // gma_tc_keysmall.cu

// The bidirectional key pass runs two CTAs per SM (gma_tc_keysmall.cu) where the shape allows.
uint32_t smem_for(uint32_t need, uint32_t tmem_cols);

// Dynamic shared memory of the responsibilities kernel (layout, staging tile unless it lives in the
// [x^2, x] buffer, histogram, column sums and their partials), and its CTAs per SM (at most four:
// 128 TMEM columns each).
uint32_t resp_smem(int d_r, int kn16)
{
    const uint32_t base = (Smem(d_r, kn16, 16, false, false, false).total + 127u) & ~127u;
    const uint32_t extra = (resp_stage_in_a(d_r) ? 0u : (uint32_t)C * 33u * 4u) + KMAX * 8u + 4u * 32u * 4u;
    return smem_for(base + extra + 1024u, 128);
}

int resp_ctas_per_sm(int d_r, int kn16)
{
    const int n = (int)(228u * 1024u / resp_smem(d_r, kn16));
    return n < 1 ? 1 : n > 4 ? 4 : n;
}

bool key_pass_small(const gma_shape_t &s, int variant)
{
    return variant == GMA_VARIANT_BIDIRECTIONAL && s.K <= 64 && keysmall_smem(s.d_r, s.K, s.d_v) != 0;
}

// `s` describes the keys; n_q is the number of queries per slice (cross-attention), s.N if < 0.
// per_sm: CTAs per SM the split is planned for (0: that of the variant's key pass).
Plan make_plan(const gma_shape_t &s, int variant, int per_sm = 0, int n_q = -1)
{
    if (n_q < 0) n_q = s.N;
    if (per_sm <= 0) per_sm = key_pass_small(s, variant) ? 2 : 1;
    Plan p{};
    p.ntile = s.K > KMAX ? (s.K + KMAX - 1) / KMAX : 1;
    p.kn16 = p.ntile > 1 ? KMAX : (s.K + 15) / 16 * 16;
    p.ne = s.d_v + 16;
    p.ka = s.d_r * 2 < 64 ? 64 : s.d_r * 2;
    p.bimg_main_bytes = p.ka / 64 * 128 * p.kn16;
    p.bimg_bytes = p.bimg_main_bytes + 32 * p.kn16;
    const int BH = s.B * s.H;
    const int nchunks = (s.N + C - 1) / C;
    // Segments per slice: one CTA per segment, per_sm CTAs per SM at a time.  Time model: waves
    // of CTAs x (set-up + chunks per segment), with the set-up (operand tables, start memory, the
    // first chunk's loads) worth about 0.6 chunk; the cheapest split wins (the larger one on a
    // tie).
    if (variant == GMA_VARIANT_RESPONSIBILITIES) {
        // as many CTAs as fit on the SMs at once (128 TMEM columns each, shared memory): one wave
        int n = resp_ctas_per_sm(s.d_r, p.kn16) * kSms / BH;
        if (n > nchunks) n = nchunks;
        if (n < 1) n = 1;
        p.cps = (nchunks + n - 1) / n;
        p.nseg = (nchunks + p.cps - 1) / p.cps;
    } else {
        // (The single-launch causal kernel takes the same split.  Its second sweep re-reads each
        // segment's key rows and values; segments short enough for those of all CTAs in flight to
        // stay in L2 were measured slower: the look-back and the per-segment set-up cost more.)
        // (bidirectional shapes whose key pass runs two CTAs per SM: a set-up of 2 chunks, which
        // gives one segment per slice at the classification-shaped workload; measured 184 -> 160 µs
        // per step against the 0.6 of the other passes, the read pass included)
        const double setup = key_pass_small(s, variant) ? 2.0 : 0.6;
        double best = 1e30;
        int best_n = 1;
        const int top = nchunks < 2048 ? nchunks : 2048;
        for (int n = 1; n <= top; ++n) {
            const int cps = (nchunks + n - 1) / n;
            const int segs = (nchunks + cps - 1) / cps;
            const long long ctas = (long long)BH * segs;
            const long long waves = (ctas + (long long)per_sm * kSms - 1) / ((long long)per_sm * kSms);
            const double cost = (double)waves * (setup + cps);
            if (cost <= best) {
                best = cost;
                best_n = segs;
            }
        }
        p.cps = (nchunks + best_n - 1) / best_n;
        p.nseg = (nchunks + p.cps - 1) / p.cps;
    }
    Carve c;
    p.off_bimg = c.take((size_t)s.H * p.ntile * p.bimg_bytes);
    p.off_cst = c.take(sizeof(float) * (size_t)s.H * p.ntile * p.kn16);
    if (variant != GMA_VARIANT_RESPONSIBILITIES)
        p.off_agg = c.take(sizeof(float) * (size_t)BH * p.nseg * KMAX * p.ne);
    if (variant == GMA_VARIANT_CAUSAL && (s.flags & GMA_FLAG_SINGLE_PASS)) {
        // the single-launch kernel: segment tickets and flags; agg holds the segments' own memories
        p.off_flags = c.take(sizeof(int) * (1 + (size_t)BH * p.nseg));
        p.off_incl = c.take(sizeof(float) * (size_t)BH * p.nseg * KMAX * p.ne);
    } else if (variant == GMA_VARIANT_CAUSAL && !(s.flags & GMA_FLAG_RECOMPUTE_KEYS)) {
        // Gamma_K of every token, written by the segment pass and read by the output pass
        p.kg = p.kn16 <= 64 ? 64 : 128;
        p.off_gam = c.take((size_t)2 * BH * s.N * p.kg);
    }
    if (p.ntile > 1 && variant == GMA_VARIANT_RESPONSIBILITIES)   // the rows' log2-sum-exp
        p.off_lse_q = c.take(sizeof(float) * (size_t)BH * s.N);
    if (p.ntile > 1 && (variant == GMA_VARIANT_CAUSAL || variant == GMA_VARIANT_BIDIRECTIONAL)) {
        // components in tiles: every query and key row's log2-sum-exp, and the partial sums of the
        // queries' numerators and normalisers
        p.off_lse_q = c.take(sizeof(float) * (size_t)BH * n_q);
        p.off_lse_k = c.take(sizeof(float) * (size_t)BH * s.N);
        p.off_part = c.take(sizeof(float) * (size_t)BH * n_q * s.d_v);
        p.off_pden = c.take(sizeof(float) * (size_t)BH * n_q);
    }
    p.total = c.total();
    return p;
}

Args make_args(const gma_shape_t &s, const Plan &p, char *ws)
{
    Args a{};
    a.bimg = (const uint8_t *)(ws + p.off_bimg);
    a.cst = (const float *)(ws + p.off_cst);
    a.agg = p.off_agg ? (float *)(ws + p.off_agg) : nullptr;
    a.hdr = (WsHeader *)ws;
    a.H = s.H;
    a.N = s.N;
    a.K = s.K;
    a.kn16 = p.kn16;
    a.d_v = s.d_v;
    a.ne = p.ne;
    a.nseg = p.nseg;
    a.cps = p.cps;
    a.agg_nseg = p.nseg;
    a.bimg_bytes = p.bimg_bytes;
    a.bimg_main_bytes = p.bimg_main_bytes;
    a.bimg_head = p.bimg_bytes * p.ntile;
    a.tile = 0;
    a.kall = s.K;
    a.lse_q = p.off_lse_q ? (const float *)(ws + p.off_lse_q) : nullptr;
    a.lse_k = p.off_lse_k ? (const float *)(ws + p.off_lse_k) : nullptr;
    a.part = p.off_part ? (float *)(ws + p.off_part) : nullptr;
    a.pden = p.off_pden ? (float *)(ws + p.off_pden) : nullptr;
    a.pmode = 0;
    a.eps = s.eps;
    a.out_f32 = (s.flags & GMA_FLAG_OUT_F32) ? 1 : 0;
    a.gam = p.off_gam ? (bf16 *)(ws + p.off_gam) : nullptr;
    a.kg = p.kg;
    a.test_withhold = (s.flags & GMA_FLAG_TEST_WITHHOLD) ? 1 : 0;
    return a;
}

// Dynamic shared memory for a kernel that allocates `tmem_cols` TMEM columns: at least enough
// that no more CTAs fit on one SM (228 KB of shared memory) than its 512 columns can serve,
// so no CTA ever waits inside tcgen05.alloc for a co-resident CTA.
bool make_xmap(CUtensorMap *m, const void *X, int BH, int N, int d_r)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_r, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d_r * 2, (cuuint64_t)N * d_r * 2};
    cuuint32_t box[3] = {(cuuint32_t)d_r, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = d_r == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : d_r == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(X), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Key responsibilities [BH][N][kg] bf16: boxes of 64 components x 128 tokens, 128-byte swizzle
// (the K-major operand layout of the kernels' Gamma_K tile).
bool make_gmap(CUtensorMap *m, const void *G, int BH, int N, int kg)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kg, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kg * 2, (cuuint64_t)N * kg * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)C, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(G), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_available() { return encode_fn() != nullptr; }

uint32_t smem_for(uint32_t need, uint32_t tmem_cols)
{
    const uint32_t per_sm = 228u * 1024u;
    const uint32_t ctas = 512u / tmem_cols;              // CTAs the TMEM can hold at once
    const uint32_t floor_ = per_sm / (ctas + 1) + 1024u; // one more would not fit
    return need > floor_ ? need : floor_;
}


gma_status_t launch_params(const gma_shape_t &s, const Plan &p, char *ws, const float *mu,
                           const float *raw, const float *logits, cudaStream_t st)
{
    GMA_LAUNCH(KID_TC_PARAMS, st,
               (tc_params_kernel<<<dim3(s.H, p.ntile * p.kn16 / 8), THREADS, 0, st>>>(mu, raw, logits, (uint8_t *)(ws + p.off_bimg),
                                                          (float *)(ws + p.off_cst), s.K, p.kn16, s.d_r,
                                                          p.bimg_bytes, p.bimg_main_bytes, p.ntile, s.var_floor, (WsHeader *)ws)));
    return GMA_OK;
}

template <int DR>   // gma_tc_keysmall.cu
gma_status_t launch_keysmall(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap, int nblocks,
                             cudaStream_t st);

template <int DR>   // gma_tc_causal.cu
gma_status_t launch_causal_fused(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap,
                                 const CUtensorMap &qmap, int *ticket_flags, float *incl, int nblocks, cudaStream_t st);

// `s` describes the keys (s.N keys); `pq` splits the queries, of which there are n_q (the same
// as s.N but for cross-attention, which is bidirectional).
template <int DR>
gma_status_t forward_dr(const gma_shape_t &s, bool causal, const void *QX, const void *KX,
                        const void *V, void *O, char *ws, const Plan &p, const Plan &pq, int n_q,
                        cudaStream_t st)
{
    Args a = make_args(s, p, ws);
    a.QX = (const bf16 *)QX;
    a.KX = (const bf16 *)KX;
    a.O = O;
    const int BH = s.B * s.H;
    CUtensorMap vmap, gmap;
    if (!make_vmap(&vmap, V, BH, s.N, s.d_v)) return GMA_ERR_CUDA;
    memset(&gmap, 0, sizeof(gmap));
    if (a.gam && !make_gmap(&gmap, a.gam, BH, s.N, p.kg)) return GMA_ERR_CUDA;
    CUtensorMap kmap;
    if (!make_xmap(&kmap, a.KX, BH, s.N, DR)) return GMA_ERR_CUDA;
    if (causal && p.off_flags) {
        // one launch: segment memories by look-back (ticket and flags zeroed by the caller)
        CUtensorMap qmap;
        if (!make_xmap(&qmap, a.QX, BH, s.N, DR)) return GMA_ERR_CUDA;
        return launch_causal_fused<DR>(a, vmap, kmap, qmap, (int *)(ws + p.off_flags), (float *)(ws + p.off_incl),
                                       BH * p.nseg, st);
    }
    {
        const gma_status_t r = !causal && key_pass_small(s, GMA_VARIANT_BIDIRECTIONAL)
                                   ? launch_keysmall<DR>(a, vmap, kmap, BH * p.nseg, st)
                                   : launch_segmem_pipelined<DR>(a, vmap, kmap, gmap, BH * p.nseg, st);
        if (r != GMA_OK) return r;
    }
    const int KD = KMAX * p.ne, KDu = p.kn16 * p.ne;
    const long long tot = (long long)BH * KDu;
    if (causal || p.nseg > 1) {   // (a bidirectional slice of one segment already holds its total)
        const unsigned nb = (unsigned)((tot + 255) / 256);
        const int cz = causal ? 1 : 0;
        cudaError_t e = cudaSuccess;
        if (p.nseg <= 4)
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<4>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, cz)));
        else if (p.nseg <= 8)
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<8>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, cz)));
        else if (p.nseg <= 20)
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<20>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, cz)));
        else
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<40>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, cz)));
        if (e != cudaSuccess) return GMA_ERR_CUDA;
    }
    if (causal && p.ntile > 1) return GMA_ERR_UNSUPPORTED_SHAPE;   // (tiled_causal_dr handles those)
    if (causal) {
        CUtensorMap qmap;
        if (!make_xmap(&qmap, a.QX, BH, s.N, DR)) return GMA_ERR_CUDA;
        if (a.gam) {
            // Gamma_K was stored by the segment pass; value tiles with the 128-byte swizzle where
            // d_v allows
            CUtensorMap vmap_o = vmap;
            Args ao = a;
            if (s.d_v % 64 == 0) {
                if (!make_vmap128(&vmap_o, V, BH, s.N, s.d_v)) return GMA_ERR_CUDA;
                ao.v128 = 1;
            }
            const gma_status_t r = launch_causal_gamma<DR>(ao, vmap_o, qmap, gmap, BH * p.nseg, st);
            if (r != GMA_OK) return r;
        } else {
            const gma_status_t r = launch_causal_pipelined<DR>(a, vmap, kmap, qmap, BH * p.nseg, st);
            if (r != GMA_OK) return r;
        }
    } else {
        // the query side: its own length and split, reading the key side's total memory
        Args aq = a;
        aq.N = n_q;
        aq.nseg = pq.nseg;
        aq.cps = pq.cps;
        aq.agg_nseg = p.nseg;
        CUtensorMap qmap, omap;
        if (!make_xmap(&qmap, aq.QX, BH, n_q, DR)) return GMA_ERR_CUDA;
        // bf16 output rows of 64-column multiples leave through TMA stores (boxes of 64 x 128); an
        // output the tensor map cannot describe keeps the threads' own stores
        const bool o_tma = !aq.out_f32 && s.d_v % 64 == 0 && make_vmap128(&omap, aq.O, BH, n_q, s.d_v);
        const gma_status_t r = launch_bidir_read2<DR>(aq, qmap, o_tma ? &omap : nullptr, BH * pq.nseg, st);
        if (r != GMA_OK) return r;
    }
    return GMA_OK;
}

// Components in tiles: O = numerator / normaliser, both summed over the tiles in part / pden
// (one thread per sixteen output values, four 16-byte streaming loads in flight each).
__global__ void __launch_bounds__(256) tc_divide_kernel(const float *__restrict__ part, const float *__restrict__ pden,
                                                        void *__restrict__ O, long long rows, int d_v, int out_f32)
{
    grid_dependency_wait();   // the partial sums come from the passes before
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // group of sixteen values
    const int per_row = d_v / 16;
    if (i >= rows * per_row) return;
    const float inv = 1.0f / pden[i / per_row];
    const float4 *src = reinterpret_cast<const float4 *>(part) + 4 * i;
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldcs(src + j);
    if (out_f32) {
        float4 *dst = reinterpret_cast<float4 *>(O) + 4 * i;
#pragma unroll
        for (int j = 0; j < 4; ++j) __stcs(dst + j, make_float4(v[j].x * inv, v[j].y * inv, v[j].z * inv, v[j].w * inv));
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(O) + 2 * i;
#pragma unroll
        for (int j = 0; j < 2; ++j)
            __stcs(dst + j, make_uint4(pack_bf16(v[2 * j].x * inv, v[2 * j].y * inv),
                                       pack_bf16(v[2 * j].z * inv, v[2 * j].w * inv),
                                       pack_bf16(v[2 * j + 1].x * inv, v[2 * j + 1].y * inv),
                                       pack_bf16(v[2 * j + 1].z * inv, v[2 * j + 1].w * inv)));
    }
}

// Causal, more than 128 components: the log2-sum-exp of every query and key row over all
// components first; then per tile of 128 components the segment pass (Gamma_K of the tile as
// exp2(L - lse)), the scan, and the output pass, which adds the tile's numerators and normalisers
// to the partial sums and, after the last tile, divides and writes O.  Exact: the numerator and
// the normaliser of the page's read are sums over the components, and so are their tiles' parts.
template <int DR>
gma_status_t tiled_causal_dr(const gma_shape_t &s, const void *QX, const void *KX, const void *V, void *O, char *ws,
                             const Plan &p, cudaStream_t st)
{
    Args a = make_args(s, p, ws);
    a.QX = (const bf16 *)QX;
    a.KX = (const bf16 *)KX;
    a.O = O;
    const int BH = s.B * s.H;
    CUtensorMap vmap, gmap, kmap, qmap, vmap_o;
    if (!make_vmap(&vmap, V, BH, s.N, s.d_v)) return GMA_ERR_CUDA;
    if (!make_gmap(&gmap, a.gam, BH, s.N, p.kg)) return GMA_ERR_CUDA;
    if (!make_xmap(&kmap, a.KX, BH, s.N, DR)) return GMA_ERR_CUDA;
    if (!make_xmap(&qmap, a.QX, BH, s.N, DR)) return GMA_ERR_CUDA;
    vmap_o = vmap;
    if (s.d_v % 64 == 0) {
        if (!make_vmap128(&vmap_o, V, BH, s.N, s.d_v)) return GMA_ERR_CUDA;
    }
    gma_status_t r = launch_lse<DR>(a, a.QX, a.KX, (float *)a.lse_q, (float *)a.lse_k, s.K, BH, st);
    if (r != GMA_OK) return r;
    const int KD = KMAX * p.ne, KDu = KMAX * p.ne;
    const long long tot = (long long)BH * KDu;
    const unsigned nb = (unsigned)((tot + 255) / 256);
    for (int t = 0; t < p.ntile; ++t) {
        Args at = a;
        at.tile = t;
        at.K = s.K - KMAX * t < KMAX ? s.K - KMAX * t : KMAX;
        if ((r = launch_segmem_pipelined<DR>(at, vmap, kmap, gmap, BH * p.nseg, st)) != GMA_OK) return r;
        cudaError_t e = cudaSuccess;
        if (p.nseg <= 4)
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<4>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 1)));
        else if (p.nseg <= 8)
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<8>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 1)));
        else if (p.nseg <= 20)
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<20>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 1)));
        else
            GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<40>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 1)));
        if (e != cudaSuccess) return GMA_ERR_CUDA;
        at.pmode = t == 0 ? 1 : 2;
        at.v128 = s.d_v % 64 == 0 ? 1 : 0;
        if ((r = launch_causal_gamma<DR>(at, vmap_o, qmap, gmap, BH * p.nseg, st)) != GMA_OK) return r;
    }
    const long long groups = (long long)BH * s.N * (s.d_v / 16);
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_DIVIDE, st,
               (e = launch_pdl(tc_divide_kernel, dim3((unsigned)((groups + 255) / 256)), dim3(256), 0, st,
                               (const float *)a.part, (const float *)a.pden, O, (long long)BH * s.N, s.d_v,
                               a.out_f32)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

// Responsibilities (or the usage diagnostics' pass over them).  More than 128 components: every
// row's log2-sum-exp (and, for the diagnostics, its argmax and the counts) first, then one
// launch per tile of 128 components writing that tile's columns of gamma (or of the mass sums).
// Bidirectional (and cross-attention: n_q queries, sk.N keys), more than 128 components: the
// rows' log2-sum-exp first; per tile of 128 components the key pass (Gamma_K = exp2(L - lse)),
// the sum of the segment memories, and the read pass adding the tile's numerators and
// normalisers to the partial sums; then the divide.
template <int DR>
gma_status_t tiled_bidir_dr(const gma_shape_t &sk, const void *QX, const void *KX, const void *V, void *O, char *ws,
                            const Plan &p, const Plan &pq, int n_q, cudaStream_t st)
{
    Args a = make_args(sk, p, ws);
    a.QX = (const bf16 *)QX;
    a.KX = (const bf16 *)KX;
    a.O = O;
    const int BH = sk.B * sk.H;
    CUtensorMap vmap, gmap, kmap, qmap;
    memset(&gmap, 0, sizeof(gmap));
    if (!make_vmap(&vmap, V, BH, sk.N, sk.d_v)) return GMA_ERR_CUDA;
    if (!make_xmap(&kmap, a.KX, BH, sk.N, DR)) return GMA_ERR_CUDA;
    if (!make_xmap(&qmap, a.QX, BH, n_q, DR)) return GMA_ERR_CUDA;
    Args al = a;   // the pre-pass: queries (n_q per slice) then keys (sk.N per slice)
    al.N = n_q;
    gma_status_t r = launch_lse<DR>(al, a.QX, a.KX, (float *)a.lse_q, (float *)a.lse_k, sk.K, BH, st, nullptr,
                                    nullptr, sk.N);
    if (r != GMA_OK) return r;
    const int KD = KMAX * p.ne, KDu = KMAX * p.ne;
    const long long tot = (long long)BH * KDu;
    const unsigned nb = (unsigned)((tot + 255) / 256);
    for (int t = 0; t < p.ntile; ++t) {
        Args at = a;
        at.tile = t;
        at.K = sk.K - KMAX * t < KMAX ? sk.K - KMAX * t : KMAX;
        if ((r = launch_segmem_pipelined<DR>(at, vmap, kmap, gmap, BH * p.nseg, st)) != GMA_OK) return r;
        if (p.nseg > 1) {   // (a slice of one segment already holds its total)
            cudaError_t e = cudaSuccess;
            if (p.nseg <= 4)
                GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<4>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 0)));
            else if (p.nseg <= 8)
                GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<8>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 0)));
            else if (p.nseg <= 20)
                GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<20>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 0)));
            else
                GMA_LAUNCH(KID_TC_CAUSAL_SCAN, st, (e = launch_pdl(tc_scan_kernel<40>, dim3(nb), dim3(256), 0, st, a.agg, tot, p.nseg, KD, KDu, 0)));
            if (e != cudaSuccess) return GMA_ERR_CUDA;
        }
        Args aq = at;
        aq.N = n_q;
        aq.nseg = pq.nseg;
        aq.cps = pq.cps;
        aq.agg_nseg = p.nseg;
        aq.pmode = t == 0 ? 1 : 2;
        if ((r = launch_bidir_read2<DR>(aq, qmap, nullptr, BH * pq.nseg, st)) != GMA_OK) return r;
    }
    const long long groups = (long long)BH * n_q * (sk.d_v / 16);
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_DIVIDE, st,
               (e = launch_pdl(tc_divide_kernel, dim3((unsigned)((groups + 255) / 256)), dim3(256), 0, st,
                               (const float *)a.part, (const float *)a.pden, O, (long long)BH * n_q, sk.d_v,
                               a.out_f32)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template <int DR>
gma_status_t resp_dr(const gma_shape_t &s, const void *X, void *gamma, char *ws, const Plan &p,
                     cudaStream_t st, int *assign = nullptr, int *counts = nullptr, float *mass_part = nullptr)
{
    Args a = make_args(s, p, ws);
    a.QX = (const bf16 *)X;
    a.gamma = gamma;
    a.assign = assign;
    a.counts = counts;
    a.mass_part = mass_part;
    const uint32_t sm = resp_smem(DR, p.kn16);
    if (!set_smem(tc_resp_kernel<DR>, sm)) return GMA_ERR_CUDA;
    if (p.ntile > 1) {
        float *lse = (float *)(ws + p.off_lse_q);
        const gma_status_t r = launch_lse<DR>(a, a.QX, nullptr, lse, nullptr, s.K, s.B * s.H, st, assign, counts);
        if (r != GMA_OK) return r;
        a.lse_q = lse;
    }
    for (int t = 0; t < p.ntile; ++t) {
        Args at = a;
        at.tile = t;
        at.K = s.K - KMAX * t < KMAX ? s.K - KMAX * t : KMAX;
        GMA_LAUNCH(KID_TC_RESP, st, (tc_resp_kernel<DR><<<s.B * s.H * p.nseg, THREADS, sm, st>>>(at)));
    }
    return GMA_OK;
}

}  // namespace tck

// ------------------------------------------------------------------ family entry points
bool tc_supported(const gma_shape_t &s, int variant)
{
    if (s.dtype != GMA_BF16 || (s.flags & GMA_FLAG_SIMT)) return false;
    if (!(s.d_r == 16 || s.d_r == 32 || s.d_r == 64)) return false;
    // more than 128 components: in tiles of 128 (the causal path only with stored key
    // responsibilities)
    if (s.K > tck::KMAX && variant == GMA_VARIANT_CAUSAL && (s.flags & (GMA_FLAG_RECOMPUTE_KEYS | GMA_FLAG_SINGLE_PASS)))
        return false;
    // value tiles move in 16-column TMA boxes, and the numerator and memory hold d_v <= 128
    // TMEM columns each
    if (s.d_v % 16 != 0 || s.d_v > 128) return false;
    (void)variant;
    return tck::encode_fn() != nullptr;
}

size_t tc_workspace_size(const gma_shape_t &s, int variant) { return tck::make_plan(s, variant).total; }

gma_status_t tc_responsibilities(const gma_shape_t &s, const void *X, const float *mu,
                                 const float *raw, const float *logits, void *gamma, void *ws,
                                 cudaStream_t st)
{
    const tck::Plan p = tck::make_plan(s, GMA_VARIANT_RESPONSIBILITIES);
    char *w = (char *)ws;
    gma_status_t r = tck::launch_params(s, p, w, mu, raw, logits, st);
    if (r != GMA_OK) return r;
    switch (s.d_r) {
    case 16: return tck::resp_dr<16>(s, X, gamma, w, p, st);
    case 32: return tck::resp_dr<32>(s, X, gamma, w, p, st);
    case 64: return tck::resp_dr<64>(s, X, gamma, w, p, st);
    }
    return GMA_ERR_UNSUPPORTED_SHAPE;
}

int tc_usage_blocks(const gma_shape_t &s)
{
    const tck::Plan p = tck::make_plan(s, GMA_VARIANT_RESPONSIBILITIES);
    return p.nseg;
}

gma_status_t tc_usage(const gma_shape_t &s, const void *X, const float *mu, const float *raw, const float *logits,
                      int *assign, int *counts, float *mass_part, void *ws, cudaStream_t st)
{
    const tck::Plan p = tck::make_plan(s, GMA_VARIANT_RESPONSIBILITIES);
    char *w = (char *)ws;
    gma_status_t r = tck::launch_params(s, p, w, mu, raw, logits, st);
    if (r != GMA_OK) return r;
    switch (s.d_r) {
    case 16: return tck::resp_dr<16>(s, X, nullptr, w, p, st, assign, counts, mass_part);
    case 32: return tck::resp_dr<32>(s, X, nullptr, w, p, st, assign, counts, mass_part);
    case 64: return tck::resp_dr<64>(s, X, nullptr, w, p, st, assign, counts, mass_part);
    }
    return GMA_ERR_UNSUPPORTED_SHAPE;
}

size_t tc_workspace_size_cross(const gma_shape_t &s, int n_k)
{
    gma_shape_t sk = s;
    sk.N = n_k;
    return tck::make_plan(sk, GMA_VARIANT_BIDIRECTIONAL, 0, s.N).total;
}

namespace tck {
int bidir_read2_ctas_per_sm(int d_r, int kn16, int d_v);   // gma_tc_bidir.cu
}

gma_status_t tc_forward(const gma_shape_t &s, bool causal, int n_k, const void *QX, const void *KX,
                        const void *V, const float *mu, const float *raw, const float *logits,
                        void *O, void *ws, cudaStream_t st)
{
    gma_shape_t sk = s;   // the key side
    sk.N = n_k;
    const int variant = causal ? GMA_VARIANT_CAUSAL : GMA_VARIANT_BIDIRECTIONAL;
    const tck::Plan p = tck::make_plan(sk, variant, 0, s.N);
    // the bidirectional read pass runs two CTAs per SM on shapes small enough for that; its split
    // is planned for it (it only sets the query segments: the workspace follows the key plan)
    const tck::Plan pq = causal ? p
                                : tck::make_plan(s, variant, tck::bidir_read2_ctas_per_sm(s.d_r, p.kn16, s.d_v));
    char *w = (char *)ws;
    if (p.off_flags &&   // the single-launch kernel's ticket and flags start at zero
        cudaMemsetAsync(w + p.off_flags, 0, sizeof(int) * (1 + (size_t)s.B * s.H * p.nseg), st) != cudaSuccess)
        return GMA_ERR_CUDA;
    gma_status_t r = tck::launch_params(s, p, w, mu, raw, logits, st);
    if (r != GMA_OK) return r;
    if (p.ntile > 1 && causal) {
        switch (s.d_r) {
        case 16: return tck::tiled_causal_dr<16>(s, QX, KX, V, O, w, p, st);
        case 32: return tck::tiled_causal_dr<32>(s, QX, KX, V, O, w, p, st);
        case 64: return tck::tiled_causal_dr<64>(s, QX, KX, V, O, w, p, st);
        }
        return GMA_ERR_UNSUPPORTED_SHAPE;
    }
    if (p.ntile > 1) {
        switch (s.d_r) {
        case 16: return tck::tiled_bidir_dr<16>(sk, QX, KX, V, O, w, p, pq, s.N, st);
        case 32: return tck::tiled_bidir_dr<32>(sk, QX, KX, V, O, w, p, pq, s.N, st);
        case 64: return tck::tiled_bidir_dr<64>(sk, QX, KX, V, O, w, p, pq, s.N, st);
        }
        return GMA_ERR_UNSUPPORTED_SHAPE;
    }
    switch (s.d_r) {
    case 16: return tck::forward_dr<16>(sk, causal, QX, KX, V, O, w, p, pq, s.N, st);
    case 32: return tck::forward_dr<32>(sk, causal, QX, KX, V, O, w, p, pq, s.N, st);
    case 64: return tck::forward_dr<64>(sk, causal, QX, KX, V, O, w, p, pq, s.N, st);
    }
    return GMA_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace gma
