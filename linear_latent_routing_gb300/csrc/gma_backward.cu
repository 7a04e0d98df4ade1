// gma_backward.cu -- the backward pass of GMA (gma_backward), fp32 on the CUDA cores.
//
// Page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283), Méthodologie
// §3: the model trains end to end by backpropagation through the softmax posteriors and the
// ratio; the page's analysis section notes that the gradients are modulated by the
// responsibilities.  For one (b, h) slice with [S | Z] the key memory (inclusive prefix for the
// causal variant), num = Gamma_Q S, den = Gamma_Q Z + eps, O = num / den, and dO given:
//   dnum = dO / den,  dden = -(dO . num) / den^2                       (per query row)
//   dGamma_Q[i] = [dnum_i | dden_i] [S_i | Z_i]^T                     (S_i: the row's memory)
//   D_j = sum_{i sees j} Gamma_Q[i]^T [dnum_i | dden_i]                 (suffix sums, causal)
//   d[v_j | 1] = Gamma_K[j] D_j,  dGamma_K[j] = D_j [v_j | 1]^T
//   dL = Gamma * (dGamma - <Gamma, dGamma>)                            (softmax over components)
//   dx_d = -sum_k dL_k (x_d - mu_kd) / s_kd;  dmu, d(raw), d(prior logits) summed over rows.
// Structure: the forward's own preparation (parameters, Gamma_Q, Gamma_K, 64-token segment
// memories, scanned), then per 64-token segment the in-segment (causal) terms explicitly and the
// carried memory D or S for the rest, exactly as the forward read phase splits its work; the
// parameter gradients are summed per row chunk and then in a fixed order, so results repeat.
#include "gma_internal.cuh"
#include "tc_ptx.cuh"

namespace gma {
namespace {

// Every kernel of this file starts by waiting for the grid before it (programmatic dependent
// launch; nothing is read or written before) and lets the next one be scheduled, so that the
// launch latencies of the backward pass's kernels overlap.
__device__ __forceinline__ void chain_enter()
{
    tc::grid_dependency_wait();
    tc::grid_dependency_launch();
}

template <typename... P, typename... A>
gma_status_t launch_chained(int kid, cudaStream_t st, void (*k)(P...), dim3 g, dim3 b, size_t smem, A... args)
{
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(kid, st, (e = launch_pdl(k, g, b, smem, st, args...)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

constexpr int SEG = 64;        // tokens per segment (the forward preparation's split)
constexpr int KT = 32;         // component tile
constexpr int BT = 256;        // threads per block

// Dynamic shared memory per segment kernel: P [SEG][SEG+1] and a tile area.
__host__ __device__ inline int seg_smem_floats(int d_v)
{
    const int dv1 = d_v + 1;
    const int tile = 2 * SEG * (KT + 1) > SEG * (dv1 + 1) * 2 ? 2 * SEG * (KT + 1) : SEG * (dv1 + 1) * 2;
    return SEG * (SEG + 1) + tile + SEG;
}

// P[i][j] = Gamma_A[i] . Gamma_B[j] over the segment rows (i from rows a0.., j from b0..), via
// K tiles in shared memory; only entries with (upper ? j >= i : j <= i) are kept (both < n).
__device__ void seg_gram(const float *__restrict__ ga, const float *__restrict__ gb, int K, int n, bool upper,
                         float (*P)[SEG + 1], float (*sa)[KT + 1], float (*sb)[KT + 1])
{
    constexpr int PER = SEG * SEG / BT;
    float acc[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) acc[r] = 0.f;
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        for (int e = threadIdx.x; e < SEG * KT; e += BT) {
            const int i = e / KT, kk = e % KT;
            const bool ok = i < n && kk < kn;
            sa[i][kk] = ok ? ga[(size_t)i * K + k0 + kk] : 0.f;
            sb[i][kk] = ok ? gb[(size_t)i * K + k0 + kk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < PER; ++r) {
            const int e = threadIdx.x + r * BT;
            const int i = e / SEG, j = e % SEG;
            float a = acc[r];
            for (int kk = 0; kk < KT; ++kk) a = fmaf(sa[i][kk], sb[j][kk], a);
            acc[r] = a;
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int e = threadIdx.x + r * BT;
        const int i = e / SEG, j = e % SEG;
        const bool keep = i < n && j < n && (upper ? j >= i : j <= i);
        P[i][j] = keep ? acc[r] : 0.f;
    }
    __syncthreads();
}

// dnd[row] = [dnum | dden] for the query rows of one segment.
template <typename Tin>
__global__ void __launch_bounds__(BT) bwd_numden_kernel(const float *__restrict__ gq, const float *__restrict__ gk,
                                                        const Tin *__restrict__ V, const float *__restrict__ agg,
                                                        const Tin *__restrict__ dO, float *__restrict__ dnd, int N,
                                                        int K, int d_v, int nseg, float eps, int causal)
{
    chain_enter();
    extern __shared__ float sm[];
    const int dv1 = d_v + 1;
    float(*P)[SEG + 1] = reinterpret_cast<float(*)[SEG + 1]>(sm);
    float *tile = sm + SEG * (SEG + 1);
    float *den = tile + (seg_smem_floats(d_v) - SEG * (SEG + 1) - SEG);
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int i0 = seg * SEG, n = min(SEG, N - i0);
    const float *S = agg + ((size_t)bh * nseg + (causal ? seg : 0)) * K * dv1;
    const float *gqs = gq + ((size_t)bh * N + i0) * K;
    const float *gks = gk + ((size_t)bh * N + i0) * K;
    if (causal)
        seg_gram(gqs, gks, K, n, false, P, reinterpret_cast<float(*)[KT + 1]>(tile),
                 reinterpret_cast<float(*)[KT + 1]>(tile + SEG * (KT + 1)));
    // nd[i][c]: numerator (c < d_v) and denominator without eps (c = d_v)
    float *nd = tile;
    for (int e = threadIdx.x; e < n * dv1; e += BT) {
        const int i = e / dv1, c = e % dv1;
        float a = 0.f;
        for (int k = 0; k < K; ++k) a = fmaf(gqs[(size_t)i * K + k], S[(size_t)k * dv1 + c], a);
        if (causal)
            for (int j = 0; j <= i; ++j)
                a = fmaf(P[i][j], c < d_v ? to_f32(V[((size_t)bh * N + i0 + j) * d_v + c]) : 1.f, a);
        nd[i * dv1 + c] = a;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += BT) {
        const float dn = nd[i * dv1 + d_v] + eps;
        float dot = 0.f;
        for (int c = 0; c < d_v; ++c) dot = fmaf(to_f32(dO[((size_t)bh * N + i0 + i) * d_v + c]), nd[i * dv1 + c], dot);
        den[i] = dn;
        nd[i * dv1 + d_v] = -dot / (dn * dn);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n * dv1; e += BT) {
        const int i = e / dv1, c = e % dv1;
        const float v = c < d_v ? to_f32(dO[((size_t)bh * N + i0 + i) * d_v + c]) / den[i] : nd[i * dv1 + d_v];
        dnd[((size_t)bh * N + i0 + i) * dv1 + c] = v;
    }
}

// dGamma_Q for the query rows of one segment:
//   dgq[i][k] = dnd_i . [S | Z][k] + sum_{j <= i in segment} (dnd_i . [v_j | 1]) Gamma_K[j][k].
template <typename Tin>
__global__ void __launch_bounds__(BT) bwd_dgq_kernel(const float *__restrict__ gk, const Tin *__restrict__ V,
                                                     const float *__restrict__ agg, const float *__restrict__ dnd,
                                                     float *__restrict__ dgq, int N, int K, int d_v, int nseg,
                                                     int causal)
{
    chain_enter();
    extern __shared__ float sm[];
    const int dv1 = d_v + 1;
    float(*A)[SEG + 1] = reinterpret_cast<float(*)[SEG + 1]>(sm);
    float *rows = sm + SEG * (SEG + 1);          // dnd rows [SEG][dv1]
    float *vrows = rows + SEG * dv1;             // [v | 1] rows [SEG][dv1]
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int i0 = seg * SEG, n = min(SEG, N - i0);
    const float *S = agg + ((size_t)bh * nseg + (causal ? seg : 0)) * K * dv1;
    for (int e = threadIdx.x; e < SEG * dv1; e += BT) {
        const int i = e / dv1, c = e % dv1;
        rows[e] = i < n ? dnd[((size_t)bh * N + i0 + i) * dv1 + c] : 0.f;
        vrows[e] = i < n ? (c < d_v ? to_f32(V[((size_t)bh * N + i0 + i) * d_v + c]) : 1.f) : 0.f;
    }
    __syncthreads();
    if (causal) {
        for (int e = threadIdx.x; e < SEG * SEG; e += BT) {
            const int i = e / SEG, j = e % SEG;
            float a = 0.f;
            if (j <= i && i < n)
                for (int c = 0; c < dv1; ++c) a = fmaf(rows[i * dv1 + c], vrows[j * dv1 + c], a);
            A[i][j] = a;
        }
        __syncthreads();
    }
    const float *gks = gk + ((size_t)bh * N + i0) * K;
    for (int e = threadIdx.x; e < n * K; e += BT) {
        const int i = e / K, k = e % K;
        float a = 0.f;
        for (int c = 0; c < dv1; ++c) a = fmaf(rows[i * dv1 + c], S[(size_t)k * dv1 + c], a);
        if (causal)
            for (int j = 0; j <= i; ++j) a = fmaf(A[i][j], gks[(size_t)j * K + k], a);
        dgq[((size_t)bh * N + i0 + i) * K + k] = a;
    }
}

// Segment partials G[bh][seg][k][c] = sum_{i in segment} Gamma_Q[i][k] dnd[i][c].
__global__ void __launch_bounds__(BT) bwd_seg_kernel(const float *__restrict__ gq, const float *__restrict__ dnd,
                                                     float *__restrict__ dagg, int N, int K, int d_v, int nseg)
{
    chain_enter();
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int k0 = blockIdx.y * KT;
    const int j0 = seg * SEG, jn = min(SEG, N - j0);
    const int kn = min(KT, K - k0);
    const int dv1 = d_v + 1;
    __shared__ float sg[SEG][KT + 1];
    __shared__ float sv[SEG][129 + 1];
    for (int e = threadIdx.x; e < SEG * KT; e += BT) {
        const int j = e / KT, kk = e % KT;
        sg[j][kk] = (j < jn && kk < kn) ? gq[((size_t)bh * N + j0 + j) * K + k0 + kk] : 0.f;
    }
    for (int e = threadIdx.x; e < SEG * dv1; e += BT) {
        const int j = e / dv1, c = e % dv1;
        sv[j][c] = j < jn ? dnd[((size_t)bh * N + j0 + j) * dv1 + c] : 0.f;
    }
    __syncthreads();
    float *out = dagg + ((size_t)bh * nseg + seg) * K * dv1;
    for (int e = threadIdx.x; e < kn * dv1; e += BT) {
        const int kk = e / dv1, c = e % dv1;
        float acc = 0.f;
        for (int j = 0; j < jn; ++j) acc = fmaf(sg[j][kk], sv[j][c], acc);
        out[(size_t)(k0 + kk) * dv1 + c] = acc;
    }
}

// Causal: each segment's partial becomes the exclusive suffix over later segments (what the
// keys of the segment see from queries after it).  Bidirectional: the total into segment 0.
__global__ void bwd_scan_kernel(float *__restrict__ dagg, long long total, int nseg, int KD, int causal)
{
    chain_enter();
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const long long bh = idx / KD, e = idx % KD;
    float *base = dagg + bh * nseg * KD + e;
    float run = 0.f;
    for (int s = nseg - 1; s >= 0; --s) {
        const float a = base[(size_t)s * KD];
        if (causal) base[(size_t)s * KD] = run;
        run += a;
    }
    if (!causal) base[0] = run;
}

// The key rows of one segment: with D the carried memory (exclusive suffix or total),
//   d[v_j | 1] = Gamma_K[j] D + sum_{i >= j in segment} (Gamma_K[j] . Gamma_Q[i]) dnd_i
//   dgk[j][k]  = [v_j | 1] . D[k] + sum_{i >= j in segment} ([v_j | 1] . dnd_i) Gamma_Q[i][k]
template <typename Tin>
__global__ void __launch_bounds__(BT) bwd_dk_kernel(const float *__restrict__ gq, const float *__restrict__ gk,
                                                    const Tin *__restrict__ V, const float *__restrict__ dagg,
                                                    const float *__restrict__ dnd, float *__restrict__ dgk,
                                                    Tin *__restrict__ dV, int N, int K, int d_v, int nseg,
                                                    int causal)
{
    chain_enter();
    extern __shared__ float sm[];
    const int dv1 = d_v + 1;
    float(*P)[SEG + 1] = reinterpret_cast<float(*)[SEG + 1]>(sm);
    float *tile = sm + SEG * (SEG + 1);
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int j0 = seg * SEG, n = min(SEG, N - j0);
    const float *D = dagg + ((size_t)bh * nseg + (causal ? seg : 0)) * K * dv1;
    const float *gqs = gq + ((size_t)bh * N + j0) * K;
    const float *gks = gk + ((size_t)bh * N + j0) * K;
    // P[j][i] = Gamma_K[j] . Gamma_Q[i] for i >= j
    if (causal)
        seg_gram(gks, gqs, K, n, true, P, reinterpret_cast<float(*)[KT + 1]>(tile),
                 reinterpret_cast<float(*)[KT + 1]>(tile + SEG * (KT + 1)));
    float *rows = tile;                      // dnd rows [SEG][dv1]
    float *vrows = rows + SEG * dv1;         // [v | 1] rows
    for (int e = threadIdx.x; e < SEG * dv1; e += BT) {
        const int i = e / dv1, c = e % dv1;
        rows[e] = i < n ? dnd[((size_t)bh * N + j0 + i) * dv1 + c] : 0.f;
        vrows[e] = i < n ? (c < d_v ? to_f32(V[((size_t)bh * N + j0 + i) * d_v + c]) : 1.f) : 0.f;
    }
    __syncthreads();
    // dV (columns c < d_v of d[v | 1])
    for (int e = threadIdx.x; e < n * d_v; e += BT) {
        const int j = e / d_v, c = e % d_v;
        float a = 0.f;
        for (int k = 0; k < K; ++k) a = fmaf(gks[(size_t)j * K + k], D[(size_t)k * dv1 + c], a);
        if (causal)
            for (int i = j; i < n; ++i) a = fmaf(P[j][i], rows[i * dv1 + c], a);
        dV[((size_t)bh * N + j0 + j) * d_v + c] = from_f32<Tin>(a);
    }
    __syncthreads();
    // A[j][i] = [v_j | 1] . dnd_i for i >= j, into P's storage
    if (causal) {
        for (int e = threadIdx.x; e < SEG * SEG; e += BT) {
            const int j = e / SEG, i = e % SEG;
            float a = 0.f;
            if (i >= j && i < n)
                for (int c = 0; c < dv1; ++c) a = fmaf(vrows[j * dv1 + c], rows[i * dv1 + c], a);
            P[j][i] = a;
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < n * K; e += BT) {
        const int j = e / K, k = e % K;
        float a = 0.f;
        for (int c = 0; c < dv1; ++c) a = fmaf(vrows[j * dv1 + c], D[(size_t)k * dv1 + c], a);
        if (causal)
            for (int i = j; i < n; ++i) a = fmaf(P[j][i], gqs[(size_t)i * K + k], a);
        dgk[((size_t)bh * N + j0 + j) * K + k] = a;
    }
}

// dL = Gamma * (dGamma - <Gamma, dGamma>) in place over dg, one warp per row.
__global__ void __launch_bounds__(BT) bwd_softmax_kernel(const float *__restrict__ g, float *__restrict__ dg,
                                                         long long rows, int K)
{
    chain_enter();
    const long long r = (long long)blockIdx.x * (BT / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float *gr = g + r * K;
    float *dr = dg + r * K;
    float dot = 0.f;
    for (int k = lane; k < K; k += 32) dot = fmaf(gr[k], dr[k], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    for (int k = lane; k < K; k += 32) dr[k] = gr[k] * (dr[k] - dot);
}

// dx_d = -sum_k dL_k (x_d - mu_kd) / s_kd, one thread per row.
template <int DR, typename Tin>
__global__ void __launch_bounds__(BT) bwd_dx_kernel(const Tin *__restrict__ X, const float *__restrict__ dL,
                                                    const float *__restrict__ mu, const float *__restrict__ iv,
                                                    Tin *__restrict__ dX, int H, int N, int K, long long rows)
{
    chain_enter();
    const long long r = (long long)blockIdx.x * BT + threadIdx.x;
    if (r >= rows) return;
    const int h = (int)((r / N) % H);
    float x[DR], dx[DR];
#pragma unroll
    for (int d = 0; d < DR; ++d) {
        x[d] = to_f32(X[r * DR + d]);
        dx[d] = 0.f;
    }
    const float *muh = mu + (size_t)h * K * DR, *ivh = iv + (size_t)h * K * DR;
    const float *dl = dL + r * K;
    for (int k = 0; k < K; ++k) {
        const float a = dl[k];
#pragma unroll
        for (int d = 0; d < DR; ++d) dx[d] = fmaf(-a * __ldg(ivh + (size_t)k * DR + d), x[d] - __ldg(muh + (size_t)k * DR + d), dx[d]);
    }
#pragma unroll
    for (int d = 0; d < DR; ++d) dX[r * DR + d] = from_f32<Tin>(dx[d]);
}

// Per-chunk partial sums of the parameter gradients of head h over its rows (query rows, then
// key rows), for 32 components (lanes) x 32 dimensions (or d_r < 32):
//   pmu[h][c][k][d] = sum dL_k w_kd (x_d - mu_kd),
//   ps [h][c][k][d] = sum dL_k (w_kd^2 (x_d - mu_kd)^2 - w_kd) / 2,
//   pl [h][c][k]    = sum dL_k (from the first dimension block only).
template <typename Tin>
__global__ void __launch_bounds__(BT) bwd_param_partial_kernel(const Tin *__restrict__ QX, const Tin *__restrict__ KX,
                                                               const float *__restrict__ dLq,
                                                               const float *__restrict__ dLk,
                                                               const float *__restrict__ mu,
                                                               const float *__restrict__ iv, float *__restrict__ pmu,
                                                               float *__restrict__ ps, float *__restrict__ pl, int B,
                                                               int H, int N, int K, int d_r, int kchunks, int R)
{
    chain_enter();
    __shared__ float red[BT / 32][32][33];
    const int h = blockIdx.x, kc = blockIdx.y % kchunks, dc = blockIdx.y / kchunks, ch = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = kc * 32 + lane, d0 = dc * 32, dn = min(32, d_r - d0);
    const bool kv = k < K;
    const int kk = kv ? k : K - 1;
    float m[32], w[32], amu[32], as[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        const bool ok = u < dn;
        m[u] = ok ? mu[((size_t)h * K + kk) * d_r + d0 + u] : 0.f;
        w[u] = ok ? iv[((size_t)h * K + kk) * d_r + d0 + u] : 0.f;
        amu[u] = 0.f;
        as[u] = 0.f;
    }
    float al = 0.f;
    const long long per = (long long)B * N, rows = 2 * per;
    const long long lo = rows * ch / R, hi = rows * (ch + 1) / R;
    for (long long q = lo + warp; q < hi; q += BT / 32) {
        const int side = q >= per;
        const long long rem = side ? q - per : q;
        const int b = (int)(rem / N), n = (int)(rem % N);
        const long long row = ((long long)b * H + h) * N + n;
        const Tin *X = side ? KX : QX;
        const float a = kv ? (side ? dLk : dLq)[row * K + k] : 0.f;
        al += a;
        const float xl = lane < dn ? to_f32(X[row * d_r + d0 + lane]) : 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const float xd = __shfl_sync(0xffffffffu, xl, u);
            const float diff = xd - m[u], wd = w[u] * diff;
            amu[u] = fmaf(a, wd, amu[u]);
            as[u] = fmaf(a, 0.5f * (wd * wd - w[u]), as[u]);
        }
    }
    for (int pass = 0; pass < 2; ++pass) {
        const float *acc = pass == 0 ? amu : as;
#pragma unroll
        for (int u = 0; u < 32; ++u) red[warp][lane][u] = acc[u];
        __syncthreads();
        // thread t sums (component t / 32... ) in warp order
        for (int e = threadIdx.x; e < 32 * 32; e += BT) {
            const int l = e / 32, u = e % 32;
            float s = 0.f;
#pragma unroll
            for (int wv = 0; wv < BT / 32; ++wv) s += red[wv][l][u];
            const int kk2 = kc * 32 + l;
            if (kk2 < K && u < dn) {
                float *dst = pass == 0 ? pmu : ps;
                dst[(((size_t)h * R + ch) * K + kk2) * d_r + d0 + u] = s;
            }
        }
        __syncthreads();
    }
    if (dc == 0) {
        red[warp][lane][0] = al;
        __syncthreads();
        if (warp == 0) {
            float s = 0.f;
#pragma unroll
            for (int wv = 0; wv < BT / 32; ++wv) s += red[wv][lane][0];
            if (kv) pl[((size_t)h * R + ch) * K + k] = s;
        }
    }
}

// dmu, d(raw) = ds * sigmoid(raw), d(logits) = dlogpi - pi * sum(dlogpi): the chunks in order.
__global__ void __launch_bounds__(BT) bwd_param_final_kernel(const float *__restrict__ pmu, const float *__restrict__ ps,
                                                             const float *__restrict__ pl, const float *__restrict__ raw,
                                                             const float *__restrict__ logits, float *__restrict__ dmu,
                                                             float *__restrict__ draw, float *__restrict__ dlogits,
                                                             int K, int d_r, int R)
{
    chain_enter();
    __shared__ float red[BT / 32][2];
    const int h = blockIdx.x;
    const int KD = K * d_r;
    for (int e = threadIdx.x; e < KD; e += BT) {
        float a = 0.f, b = 0.f;
        for (int c = 0; c < R; ++c) {
            a += pmu[((size_t)h * R + c) * KD + e];
            b += ps[((size_t)h * R + c) * KD + e];
        }
        const float r = raw[(size_t)h * KD + e];
        dmu[(size_t)h * KD + e] = a;
        draw[(size_t)h * KD + e] = b / (1.f + expf(-r));
    }
    // prior logits: pi = softmax(logits); dlogits = dlogpi - pi * sum_k dlogpi
    const float *lh = logits + (size_t)h * K;
    float m = -INFINITY, tl = 0.f;
    for (int k = threadIdx.x; k < K; k += BT) m = fmaxf(m, lh[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5][0] = m;
    __syncthreads();
    m = red[0][0];
    for (int wv = 1; wv < BT / 32; ++wv) m = fmaxf(m, red[wv][0]);
    float se = 0.f;
    for (int k = threadIdx.x; k < K; k += BT) {
        se += expf(lh[k] - m);
        float a = 0.f;
        for (int c = 0; c < R; ++c) a += pl[((size_t)h * R + c) * K + k];
        tl += a;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        se += __shfl_xor_sync(0xffffffffu, se, o);
        tl += __shfl_xor_sync(0xffffffffu, tl, o);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        red[threadIdx.x >> 5][0] = se;
        red[threadIdx.x >> 5][1] = tl;
    }
    __syncthreads();
    se = 0.f;
    tl = 0.f;
    for (int wv = 0; wv < BT / 32; ++wv) {
        se += red[wv][0];
        tl += red[wv][1];
    }
    for (int k = threadIdx.x; k < K; k += BT) {
        float a = 0.f;
        for (int c = 0; c < R; ++c) a += pl[((size_t)h * R + c) * K + k];
        const float pi = expf(lh[k] - m) / se;
        dlogits[(size_t)h * K + k] = a - pi * tl;
    }
}

struct BwdLayout {
    size_t iv, cst, gq, gk, agg, dnd, dagg, dgq, dgk, pmu, ps, pl, total;
    int nseg, R, kchunks, dchunks;
};

BwdLayout bwd_layout(const gma_shape_t &s)
{
    BwdLayout L{};
    Carve c;
    const size_t T = (size_t)s.B * s.H * s.N;
    const int dv1 = s.d_v + 1;
    L.nseg = (s.N + SEG - 1) / SEG;
    L.kchunks = (s.K + 31) / 32;
    L.dchunks = (s.d_r + 31) / 32;
    const long long rows = 2ll * s.B * s.N;
    int R = (int)((2 * 152 + s.H * L.kchunks * L.dchunks - 1) / (s.H * L.kchunks * L.dchunks));
    if (R < 1) R = 1;
    if (R > 64) R = 64;
    if (R > rows / 64 + 1) R = (int)(rows / 64 + 1);
    L.R = R;
    L.iv = c.take(sizeof(float) * (size_t)s.H * s.K * s.d_r);
    L.cst = c.take(sizeof(float) * (size_t)s.H * s.K);
    L.gq = c.take(sizeof(float) * T * s.K);
    L.gk = c.take(sizeof(float) * T * s.K);
    L.agg = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * s.K * dv1);
    L.dnd = c.take(sizeof(float) * T * dv1);
    L.dagg = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * s.K * dv1);
    L.dgq = c.take(sizeof(float) * T * s.K);
    L.dgk = c.take(sizeof(float) * T * s.K);
    L.pmu = c.take(sizeof(float) * (size_t)s.H * R * s.K * s.d_r);
    L.ps = c.take(sizeof(float) * (size_t)s.H * R * s.K * s.d_r);
    L.pl = c.take(sizeof(float) * (size_t)s.H * R * s.K);
    L.total = c.total();
    return L;
}

template <typename Tin>
gma_status_t launch_dx(int d_r, const Tin *X, const float *dL, const float *mu, const float *iv, Tin *dX, int H, int N,
                       int K, long long rows, cudaStream_t st)
{
    const unsigned blocks = (unsigned)((rows + BT - 1) / BT);
    gma_status_t rr = GMA_OK;
    switch (d_r) {
    case 16: if ((rr = launch_chained(KID_BWD_DX, st, bwd_dx_kernel<16, Tin>, dim3(blocks), dim3(BT), 0, X, dL, mu, iv, dX, H, N, K, rows)) != GMA_OK) return rr; break;
    case 32: if ((rr = launch_chained(KID_BWD_DX, st, bwd_dx_kernel<32, Tin>, dim3(blocks), dim3(BT), 0, X, dL, mu, iv, dX, H, N, K, rows)) != GMA_OK) return rr; break;
    case 64: if ((rr = launch_chained(KID_BWD_DX, st, bwd_dx_kernel<64, Tin>, dim3(blocks), dim3(BT), 0, X, dL, mu, iv, dX, H, N, K, rows)) != GMA_OK) return rr; break;
    case 128: if ((rr = launch_chained(KID_BWD_DX, st, bwd_dx_kernel<128, Tin>, dim3(blocks), dim3(BT), 0, X, dL, mu, iv, dX, H, N, K, rows)) != GMA_OK) return rr; break;
    default: return GMA_ERR_UNSUPPORTED_SHAPE;
    }
    return GMA_OK;
}

template <typename Tin>
gma_status_t backward_typed(const gma_shape_t &s, bool causal, const Tin *QX, const Tin *KX, const Tin *V,
                            const float *mu, const float *raw, const float *logits, const Tin *dO, Tin *dQX, Tin *dKX,
                            Tin *dV, float *dmu, float *draw, float *dlogits, char *ws, cudaStream_t st)
{
    const BwdLayout L = bwd_layout(s);
    float *iv = (float *)(ws + L.iv), *cst = (float *)(ws + L.cst);
    float *gq = (float *)(ws + L.gq), *gk = (float *)(ws + L.gk), *agg = (float *)(ws + L.agg);
    float *dnd = (float *)(ws + L.dnd), *dagg = (float *)(ws + L.dagg);
    float *dgq = (float *)(ws + L.dgq), *dgk = (float *)(ws + L.dgk);
    float *pmu = (float *)(ws + L.pmu), *ps = (float *)(ws + L.ps), *pl = (float *)(ws + L.pl);
    gma_status_t r = simt_prepare(s, causal, QX, KX, V, mu, raw, logits, iv, cst, gq, gk, agg, st);
    if (r != GMA_OK) return r;
    gma_status_t rr = GMA_OK;
    const int BH = s.B * s.H, cz = causal ? 1 : 0;
    const unsigned nblk = (unsigned)(BH * L.nseg);
    const size_t smem = sizeof(float) * (size_t)seg_smem_floats(s.d_v);
    if (cudaFuncSetAttribute(bwd_numden_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dgq_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dk_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GMA_ERR_CUDA;
    if ((rr = launch_chained(KID_BWD_NUMDEN, st, bwd_numden_kernel<Tin>, dim3(nblk), dim3(BT), smem, gq, gk, V, agg, dO, dnd, s.N, s.K, s.d_v, L.nseg, s.eps, cz)) != GMA_OK) return rr;
    if ((rr = launch_chained(KID_BWD_DQ, st, bwd_dgq_kernel<Tin>, dim3(nblk), dim3(BT), smem, gk, V, agg, dnd, dgq, s.N, s.K, s.d_v, L.nseg, cz)) != GMA_OK) return rr;
    dim3 gs(nblk, (unsigned)((s.K + KT - 1) / KT));
    if ((rr = launch_chained(KID_BWD_SEG, st, bwd_seg_kernel, dim3(gs), dim3(BT), 0, gq, dnd, dagg, s.N, s.K, s.d_v, L.nseg)) != GMA_OK) return rr;
    const int KD = s.K * (s.d_v + 1);
    const long long tot = (long long)BH * KD;
    if ((rr = launch_chained(KID_BWD_SCAN, st, bwd_scan_kernel, dim3((unsigned)((tot + 255) / 256)), dim3(256), 0, dagg, tot, L.nseg, KD, cz)) != GMA_OK) return rr;
    if ((rr = launch_chained(KID_BWD_DK, st, bwd_dk_kernel<Tin>, dim3(nblk), dim3(BT), smem, gq, gk, V, dagg, dnd, dgk, dV, s.N, s.K, s.d_v, L.nseg, cz)) != GMA_OK) return rr;
    const long long T = (long long)BH * s.N;
    if ((rr = launch_chained(KID_BWD_SOFTMAX, st, bwd_softmax_kernel, dim3((unsigned)((T + 7) / 8)), dim3(BT), 0, gq, dgq, T, s.K)) != GMA_OK) return rr;
    if ((rr = launch_chained(KID_BWD_SOFTMAX, st, bwd_softmax_kernel, dim3((unsigned)((T + 7) / 8)), dim3(BT), 0, gk, dgk, T, s.K)) != GMA_OK) return rr;
    r = launch_dx<Tin>(s.d_r, QX, dgq, mu, iv, dQX, s.H, s.N, s.K, T, st);
    if (r != GMA_OK) return r;
    r = launch_dx<Tin>(s.d_r, KX, dgk, mu, iv, dKX, s.H, s.N, s.K, T, st);
    if (r != GMA_OK) return r;
    dim3 gp((unsigned)s.H, (unsigned)(L.kchunks * L.dchunks), (unsigned)L.R);
    if ((rr = launch_chained(KID_BWD_PARAMS, st, bwd_param_partial_kernel<Tin>, dim3(gp), dim3(BT), 0, QX, KX, dgq, dgk, mu, iv, pmu, ps, pl, s.B, s.H, s.N, s.K, s.d_r, L.kchunks, L.R)) != GMA_OK) return rr;
    if ((rr = launch_chained(KID_BWD_PFINAL, st, bwd_param_final_kernel, dim3((unsigned)s.H), dim3(BT), 0, pmu, ps, pl, raw, logits, dmu, draw, dlogits, s.K, s.d_r, L.R)) != GMA_OK) return rr;
    return GMA_OK;
}

}  // namespace

size_t backward_workspace_size(const gma_shape_t &s) { return bwd_layout(s).total; }

gma_status_t backward(const gma_shape_t &s, bool causal, const void *QX, const void *KX, const void *V,
                      const float *mu, const float *raw, const float *logits, const void *dO, void *dQX, void *dKX,
                      void *dV, float *dmu, float *draw, float *dlogits, void *ws, cudaStream_t st)
{
    char *w = (char *)ws;
    if (s.dtype == GMA_F32)
        return backward_typed<float>(s, causal, (const float *)QX, (const float *)KX, (const float *)V, mu, raw, logits,
                                     (const float *)dO, (float *)dQX, (float *)dKX, (float *)dV, dmu, draw, dlogits, w,
                                     st);
    typedef __nv_bfloat16 bf;
    return backward_typed<bf>(s, causal, (const bf *)QX, (const bf *)KX, (const bf *)V, mu, raw, logits, (const bf *)dO,
                              (bf *)dQX, (bf *)dKX, (bf *)dV, dmu, draw, dlogits, w, st);
}

}  // namespace gma
