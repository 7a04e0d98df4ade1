// gma_usage.cu -- component-usage diagnostics of the responsibilities (gma_usage).
//
// Page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283), Résultats et
// Performance (interpretability): how many of the K components the responsibilities use, the
// entropy of that usage, and the hard assignments of tokens to components.  Per head h:
//   assign[b][h][i] = argmax_k gamma_{b,h,i,k}   (the lowest k on ties)
//   counts[h][k]    = #{(b, i) : assign[b][h][i] = k}
//   mass[h][k]      = sum_{b,i} gamma_{b,h,i,k}
//   used[h]         = #{k : counts[h][k] > 0}
//   entropy[h]      = -sum_k p_k ln p_k / ln K,  p = counts[h] / (B N)   (0 for K = 1)
//
// Steps, tensor-core family: the responsibilities pass itself keeps each row's argmax, a shared-
// memory histogram and the column sums of its tiles (no responsibilities reach HBM).  CUDA-core
// family: the responsibilities (fp32) into the workspace, then one pass over them (a warp per
// token row: argmax by shuffles, a shared-memory histogram per block, per-block partial masses).
// Both: a fixed-order reduction of the partial masses; per-head used count and entropy.  Counts are integer sums, so the order of the atomic
// additions does not matter; the masses are summed in a fixed order, so results repeat exactly.
#include "gma_internal.cuh"

namespace gma {
namespace {

constexpr int UT = 256;      // threads per block
constexpr int UROWS = 64;    // token rows per block (8 warps x 8 rows)

// Rows [r0, r0 + UROWS) of slice bh; KPL = components per lane (K <= 32 KPL).
template <int KPL>
__global__ void __launch_bounds__(UT) usage_rows_kernel(const float *__restrict__ gamma, int *__restrict__ assign,
                                                        int *__restrict__ counts, float *__restrict__ part, int H,
                                                        int N, int K, int nblk)
{
    __shared__ int hist[1024];
    __shared__ float wm[UT / 32][1024];
    const int bh = blockIdx.x / nblk, blk = blockIdx.x % nblk, h = bh % H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int k = threadIdx.x; k < K; k += UT) hist[k] = 0;
    __syncthreads();
    float m[KPL];
#pragma unroll
    for (int j = 0; j < KPL; ++j) m[j] = 0.f;
    const int r0 = blk * UROWS;
    for (int rr = warp; rr < UROWS; rr += UT / 32) {
        const int i = r0 + rr;
        if (i >= N) break;
        const float *g = gamma + ((size_t)bh * N + i) * K;
        float best = -1.f;
        int arg = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < KPL; ++j) {
            const int k = lane + 32 * j;
            if (k < K) {
                const float x = g[k];
                m[j] += x;
                if (x > best) {   // k grows with j: the first maximum of this lane is kept
                    best = x;
                    arg = k;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
            if (ob > best || (ob == best && oa < arg)) {
                best = ob;
                arg = oa;
            }
        }
        if (lane == 0) {
            assign[(size_t)bh * N + i] = arg;
            atomicAdd(&hist[arg], 1);
        }
    }
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
        const int k = lane + 32 * j;
        if (k < K) wm[warp][k] = m[j];
    }
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += UT) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < UT / 32; ++w) s += wm[w][k];
        part[(size_t)blockIdx.x * K + k] = s;
        if (hist[k]) atomicAdd(&counts[(size_t)h * K + k], hist[k]);
    }
}

// mass[h][k] = sum of the per-block partials of head h in a fixed order: block (h, 32
// components), warp w takes parts w, w + 8, ... (part q = block q % nblk of slice b = q / nblk),
// four running sums per lane, then the eight warps' sums in order.
__global__ void __launch_bounds__(UT) usage_mass_kernel(const float *__restrict__ part, float *__restrict__ mass,
                                                        int B, int H, int K, int nblk)
{
    __shared__ float ws[UT / 32][32];
    const int h = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = blockIdx.x * 32 + lane;
    const int kk = k < K ? k : K - 1;
    const int np = B * nblk;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    auto at = [&](int q) {
        const int b = q / nblk, blk = q - b * nblk;
        return __ldg(part + ((size_t)(b * H + h) * nblk + blk) * K + kk);
    };
    int q = warp;
    for (; q + 3 * (UT / 32) < np; q += 4 * (UT / 32)) {
        s0 += at(q);
        s1 += at(q + UT / 32);
        s2 += at(q + 2 * (UT / 32));
        s3 += at(q + 3 * (UT / 32));
    }
    for (; q < np; q += UT / 32) s0 += at(q);
    ws[warp][lane] = (s0 + s1) + (s2 + s3);
    __syncthreads();
    if (warp == 0 && k < K) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < UT / 32; ++w) s += ws[w][lane];
        mass[(size_t)h * K + k] = s;
    }
}

// One warp per head: components used and the normalised entropy of the counts.
__global__ void usage_stats_kernel(const int *__restrict__ counts, int *__restrict__ used,
                                   float *__restrict__ entropy, int H, int K, long long tokens)
{
    const int h = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (h >= H) return;
    int u = 0;
    float e = 0.f;
    const float inv = 1.f / (float)tokens;
    for (int k = lane; k < K; k += 32) {
        const int c = counts[(size_t)h * K + k];
        if (c > 0) {
            ++u;
            const float p = (float)c * inv;
            e -= p * logf(p);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        u += __shfl_xor_sync(0xffffffffu, u, o);
        e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if (lane == 0) {
        used[h] = u;
        entropy[h] = K > 1 ? e / logf((float)K) : 0.f;
    }
}

struct UsageLayout {
    size_t gamma, part, total;
    int nblk;
    bool fused;       // tensor-core family: diagnostics in the responsibilities pass itself
    gma_shape_t rs;   // the responsibilities call: fp32 output
};

UsageLayout usage_layout(const gma_shape_t &s)
{
    UsageLayout L{};
    L.rs = s;
    L.rs.flags |= GMA_FLAG_OUT_F32;
    L.fused = tc_supported(L.rs, GMA_VARIANT_RESPONSIBILITIES);
    L.nblk = L.fused ? tc_usage_blocks(L.rs) : (s.N + UROWS - 1) / UROWS;
    // the responsibilities' own workspace first, so its header is this call's header
    const size_t resp = L.fused ? tc_workspace_size(L.rs, GMA_VARIANT_RESPONSIBILITIES)
                                : simt_workspace_size(L.rs, GMA_VARIANT_RESPONSIBILITIES);
    size_t off = (resp + 255) & ~(size_t)255;
    L.gamma = off;
    if (!L.fused)   // the CUDA-core family writes the responsibilities, then a pass reads them
        off += ((size_t)s.B * s.H * s.N * s.K * sizeof(float) + 255) & ~(size_t)255;
    L.part = off;
    off += ((size_t)s.B * s.H * L.nblk * s.K * sizeof(float) + 255) & ~(size_t)255;
    L.total = off;
    return L;
}

template <int KPL>
gma_status_t launch_rows(const float *gamma, int *assign, int *counts, float *part, const gma_shape_t &s, int nblk,
                         cudaStream_t st)
{
    GMA_LAUNCH(KID_USAGE_ROWS, st,
               (usage_rows_kernel<KPL><<<(unsigned)(s.B * s.H * nblk), UT, 0, st>>>(gamma, assign, counts, part, s.H,
                                                                                    s.N, s.K, nblk)));
    return GMA_OK;
}

}  // namespace

size_t usage_workspace_size(const gma_shape_t &s) { return usage_layout(s).total; }

gma_status_t usage(const gma_shape_t &s, const void *X, const float *mu, const float *raw, const float *logits,
                   int *assign, int *counts, float *mass, int *used, float *entropy, void *ws, cudaStream_t st)
{
    const UsageLayout L = usage_layout(s);
    char *w = (char *)ws;
    float *gamma = (float *)(w + L.gamma);
    float *part = (float *)(w + L.part);
    if (cudaMemsetAsync(counts, 0, sizeof(int) * (size_t)s.H * s.K, st) != cudaSuccess) return GMA_ERR_CUDA;
    gma_status_t r = GMA_OK;
    const int kpl = (s.K + 31) / 32;
    if (L.fused)
        r = tc_usage(L.rs, X, mu, raw, logits, assign, counts, part, ws, st);
    else if ((r = simt_responsibilities(L.rs, X, mu, raw, logits, gamma, ws, st)) != GMA_OK)
        return r;
    else if (kpl <= 1) r = launch_rows<1>(gamma, assign, counts, part, s, L.nblk, st);
    else if (kpl <= 2) r = launch_rows<2>(gamma, assign, counts, part, s, L.nblk, st);
    else if (kpl <= 4) r = launch_rows<4>(gamma, assign, counts, part, s, L.nblk, st);
    else if (kpl <= 8) r = launch_rows<8>(gamma, assign, counts, part, s, L.nblk, st);
    else if (kpl <= 16) r = launch_rows<16>(gamma, assign, counts, part, s, L.nblk, st);
    else r = launch_rows<32>(gamma, assign, counts, part, s, L.nblk, st);
    if (r != GMA_OK) return r;
    GMA_LAUNCH(KID_USAGE_MASS, st,
               (usage_mass_kernel<<<dim3((unsigned)((s.K + 31) / 32), (unsigned)s.H), UT, 0, st>>>(
                   part, mass, s.B, s.H, s.K, L.nblk)));
    GMA_LAUNCH(KID_USAGE_STATS, st,
               (usage_stats_kernel<<<(unsigned)((s.H + 7) / 8), 256, 0, st>>>(counts, used, entropy, s.H, s.K,
                                                                             (long long)s.B * s.N)));
    return GMA_OK;
}

}  // namespace gma
