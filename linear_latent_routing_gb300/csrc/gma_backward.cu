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
// carried memory D or S for the rest, exactly as the forward read phase splits its work.
//
// Every contraction is a register-tiled product over shared-memory tiles (simt_tile.cuh).  Each is
// formed in the orientation its consumer reads (P^T where the next product contracts over keys,
// for instance); the query side's in-segment P^T and A^T tiles are also stored, and the key side
// stages them back (transposed into shared memory) instead of forming them again.  All sums run
// in a fixed order (no atomics): repeated calls give identical bits.
#include "gma_internal.cuh"
#include "simt_tile.cuh"
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

constexpr int SEG = 64;   // tokens per segment (the forward preparation's split)
constexpr int KT = 64;    // components per tile
using namespace tile;

// ---------------------------------------------------------------- query side, per segment
// num = Gamma_Q S + tril(P) V and den = Gamma_Q Z + tril(P) 1 + eps for the query rows of one
// segment (P = Gamma_Q Gamma_K^T on the segment, causal only; [S | Z] the segment's memory), then
//   dnd[i] = [dO_i / den_i | -(dO_i . num_i) / den_i^2]
// and the segment's partial G[k][c] = sum_i Gamma_Q[i][k] dnd[i][c], whose suffix sums over later
// segments are what the keys of a segment receive from the queries after it.
template <int DV>
__host__ __device__ constexpr int numden_smem_floats() { return 2 * KT * LT + KT * DV + KT + 2 * SEG; }

template <int DV, typename Tin>
__global__ void __launch_bounds__(BT, DV == 64 ? 4 : 2) bwd_numden_kernel(const float *__restrict__ gq, const float *__restrict__ gk,
                                                        const Tin *__restrict__ V, const float *__restrict__ agg,
                                                        const Tin *__restrict__ dO, float *__restrict__ dnd,
                                                        float *__restrict__ dagg, float *__restrict__ Pg, int N, int K,
                                                        int nseg, float eps, int causal)
{
    chain_enter();
    extern __shared__ __align__(16) float sm[];
    constexpr int DV1 = DV + 1, NC = DV / 16;
    float *gqT = sm;                 // [KT][LT] Gamma_Q^T tile; later Gamma_Q tiles [SEG][KT]
    float *gkT = gqT + KT * LT;      // [KT][LT] Gamma_K^T tile; later P^T [SEG][LT]
    float *sS = gkT + KT * LT;       // [KT][DV] S tile; later the value rows, then the dnum rows
    float *zS = sS + KT * DV;        // [KT]     Z of the tile
    float *den = zS + KT;            // [SEG]
    float *dd = den + SEG;           // [SEG]    dden
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int i0 = seg * SEG, n = min(SEG, N - i0);
    const long long row0 = (long long)bh * N + i0;
    const float *S = agg + ((size_t)bh * nseg + (causal ? seg : 0)) * K * DV1;
    const int t = threadIdx.x, r0 = orow();
    float accP[4][4], accN[4][NC];
    zero<64>(accP);
    zero<DV>(accN);
    float dpart = 0.f;
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        stage_t<KT>(gqT, LT, gq + row0 * K + k0, K, n, kn);
        if (causal) stage_t<KT>(gkT, LT, gk + row0 * K + k0, K, n, kn);
        stage<DV>(sS, DV, S + (size_t)k0 * DV1, DV1, kn, DV);
        if (t < KT) zS[t] = t < kn ? S[(size_t)(k0 + t) * DV1 + DV] : 0.f;
        __syncthreads();
        if (causal) mac<64>(accP, gkT, LT, gqT, LT, KT);   // P^T: rows j, columns i
        mac<DV>(accN, gqT, LT, sS, DV, KT);                // rows i, columns c
        if (t < SEG) {
            float a = 0.f;
            for (int k = 0; k < KT; ++k) a = fmaf(gqT[k * LT + t], zS[k], a);
            dpart += a;
        }
    }
    __syncthreads();
    if (causal) {
        // P^T[j][i], kept for i >= j; also stored for the key-side kernel (row j: 64 floats)
        float *Pt = Pg + (size_t)blockIdx.x * SEG * SEG;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = r0 + r;
            float4 v;
            v.x = ocol<64>(0) >= j ? accP[r][0] : 0.f;
            v.y = ocol<64>(1) >= j ? accP[r][1] : 0.f;
            v.z = ocol<64>(2) >= j ? accP[r][2] : 0.f;
            v.w = ocol<64>(3) >= j ? accP[r][3] : 0.f;
            *reinterpret_cast<float4 *>(gkT + j * LT + ocol<64>(0)) = v;
            *reinterpret_cast<float4 *>(Pt + j * SEG + ocol<64>(0)) = v;
        }
        stage<DV>(sS, DV, V + row0 * DV, DV, n, DV);
        __syncthreads();
        mac_range<DV>(accN, gkT, LT, sS, DV, 0, r0 + 4);   // (P^T[j][i] = 0 for j > i)
        if (t < SEG) {
            float a = 0.f;
            for (int j = 0; j < SEG; ++j) a += gkT[j * LT + t];
            dpart += a;
        }
    }
    if (t < SEG) den[t] = dpart + eps;
    __syncthreads();
    // dnum over num, then dden (the rows' dot products summed over the 16 threads of each row)
    float dot[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = r0 + r;
        const float dn = den[i];
        dot[r] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float o = i < n ? to_f32(dO[(row0 + i) * DV + ocol<DV>(c)]) : 0.f;
            dot[r] = fmaf(o, accN[r][c], dot[r]);
            accN[r][c] = o / dn;
        }
    }
    row_sums(dot);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = r0 + r;
        const float dn = den[i];
        const float ddi = i < n ? -dot[r] / (dn * dn) : 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            if (i < n) dnd[(row0 + i) * DV1 + ocol<DV>(c)] = accN[r][c];
            sS[i * DV + ocol<DV>(c)] = accN[r][c];
        }
        if (tile_tx() == 0) {
            if (i < n) dnd[(row0 + i) * DV1 + DV] = ddi;
            dd[i] = ddi;
        }
    }
    // G, one component tile at a time
    float *G = dagg + ((size_t)bh * nseg + seg) * K * DV1;
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        stage<KT>(gqT, KT, gq + row0 * K + k0, K, n, kn);
        __syncthreads();
        float accG[4][NC];
        zero<DV>(accG);
        mac<DV>(accG, gqT, KT, sS, DV, SEG);   // rows k, columns c
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int k = k0 + r0 + r;
            if (k < K)
#pragma unroll
                for (int c = 0; c < NC; ++c) G[(size_t)k * DV1 + ocol<DV>(c)] = accG[r][c];
        }
        if (t < kn) {
            float a = 0.f;
            for (int i = 0; i < SEG; ++i) a = fmaf(gqT[i * KT + t], dd[i], a);
            G[(size_t)(k0 + t) * DV1 + DV] = a;
        }
    }
}

// dGamma_Q[i][k] = dnd_i . [S | Z][k] + sum_{j <= i in segment} A[i][j] Gamma_K[j][k] for the query
// rows of one segment, with A[i][j] = dnd_i . [v_j | 1] (causal only), and the row's
// <Gamma_Q, dGamma_Q> for the softmax step.
template <int DV>
__host__ __device__ constexpr int dgq_smem_floats() { return 2 * DV * LT + SEG * LT + SEG * KT + KT + SEG; }

template <int DV, typename Tin>
__global__ void __launch_bounds__(BT, DV == 64 ? 3 : 2) bwd_dgq_kernel(const float *__restrict__ gq, const float *__restrict__ gk,
                                                     const Tin *__restrict__ V, const float *__restrict__ agg,
                                                     const float *__restrict__ dnd, float *__restrict__ dgq,
                                                     float *__restrict__ dotq, float *__restrict__ Ag, int N, int K,
                                                     int nseg, int causal)
{
    chain_enter();
    extern __shared__ __align__(16) float sm[];
    constexpr int DV1 = DV + 1;
    float *dnT = sm;                 // [DV][LT]  dnum^T
    float *VT = dnT + DV * LT;       // [DV][LT]  V^T; later the S^T tiles
    float *AT = VT + DV * LT;        // [SEG][LT] A^T
    float *gK = AT + SEG * LT;       // [SEG][KT] Gamma_K tile
    float *zS = gK + SEG * KT;       // [KT]
    float *dd = zS + KT;             // [SEG]
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int i0 = seg * SEG, n = min(SEG, N - i0);
    const long long row0 = (long long)bh * N + i0;
    const float *S = agg + ((size_t)bh * nseg + (causal ? seg : 0)) * K * DV1;
    const int t = threadIdx.x, r0 = orow();
    stage_t<DV>(dnT, LT, dnd + row0 * DV1, DV1, n, DV);
    if (t < SEG) dd[t] = t < n ? dnd[(row0 + t) * DV1 + DV] : 0.f;
    if (causal) {
        stage_t<DV>(VT, LT, V + row0 * DV, DV, n, DV);
        __syncthreads();
        float accA[4][4];
        zero<64>(accA);
        mac<64>(accA, VT, LT, dnT, LT, DV);   // rows j, columns i: v_j . dnum_i
        // also stored for the key-side kernel (row j: 64 floats)
        float *At = Ag + (size_t)blockIdx.x * SEG * SEG;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = r0 + r;
            float a[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = ocol<64>(c);
                a[c] = i >= j ? accA[r][c] + dd[i] : 0.f;
            }
            const float4 v = make_float4(a[0], a[1], a[2], a[3]);
            *reinterpret_cast<float4 *>(AT + j * LT + ocol<64>(0)) = v;
            *reinterpret_cast<float4 *>(At + j * SEG + ocol<64>(0)) = v;
        }
    }
    const bool one = K <= KT;
    float dot[4] = {0.f, 0.f, 0.f, 0.f}, gsv[4][4], acc[4][4];
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        stage_t<DV>(VT, LT, S + (size_t)k0 * DV1, DV1, kn, DV);   // S^T: [c][k]
        if (t < KT) zS[t] = t < kn ? S[(size_t)(k0 + t) * DV1 + DV] : 0.f;
        if (causal) stage<KT>(gK, KT, gk + row0 * K + k0, K, n, kn);
        __syncthreads();
        zero<64>(acc);
        mac<64>(acc, dnT, LT, VT, LT, DV);                  // rows i, columns k
        if (causal) mac_range<64>(acc, AT, LT, gK, KT, 0, r0 + 4);   // (A^T[j][i] = 0 for j > i)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = r0 + r;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int kk = ocol<64>(c), k = k0 + kk;
                const float v = fmaf(dd[i], zS[kk], acc[r][c]);
                gsv[r][c] = i < n && k < K ? gq[(row0 + i) * K + k] : 0.f;
                dot[r] = fmaf(gsv[r][c], v, dot[r]);
                acc[r][c] = v;
                if (!one && i < n && k < K) dgq[(row0 + i) * K + k] = v;
            }
        }
    }
    row_sums(dot);
    // one tile: the row's dGamma is all here, so dL = Gamma (dGamma - <Gamma, dGamma>) is written
    // in its place; otherwise the kernel through the responsibilities forms it from dot
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = r0 + r;
        if (one) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int k = ocol<64>(c);
                if (i < n && k < K) dgq[(row0 + i) * K + k] = gsv[r][c] * (acc[r][c] - dot[r]);
            }
        } else if (tile_tx() == 0 && i < n) {
            dotq[row0 + i] = dot[r];
        }
    }
}

// Causal: each segment's partial becomes the exclusive suffix over later segments (what the
// keys of the segment see from queries after it).  Bidirectional: the total into segment 0.
// One thread per V4 consecutive elements of the K x (d_v + 1) memory (V4 = 4 with 16-byte accesses
// when K (d_v + 1) is a multiple of 4, else 1); the loads of 16 segments are issued before their
// sums, so a thread waits once per 16 segments.
template <int V4>
__global__ void __launch_bounds__(BT) bwd_scan_kernel(float *__restrict__ dagg, long long total, int nseg, int KD,
                                                      int causal)
{
    chain_enter();
    typedef typename std::conditional<V4 == 4, float4, float>::type vec;
    const long long idx = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * V4;
    if (idx >= total) return;
    const long long bh = idx / KD, e = idx % KD;
    vec *base = reinterpret_cast<vec *>(dagg + bh * nseg * KD + e);
    const size_t step = (size_t)KD / V4;
    vec run = vzero<vec>();
    for (int s1 = nseg; s1 > 0; s1 -= 16) {
        vec a[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) a[u] = s1 - 1 - u >= 0 ? base[(size_t)(s1 - 1 - u) * step] : vzero<vec>();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (s1 - 1 - u < 0) break;
            if (causal) base[(size_t)(s1 - 1 - u) * step] = run;
            run = vadd(run, a[u]);
        }
    }
    if (!causal) base[0] = run;
}

// The key rows of one segment, with D the carried memory (exclusive suffix or total):
//   dV[j] = Gamma_K[j] D + sum_{i >= j in segment} P[i][j] dnum_i      (the first d_v columns
//                                                                      of d[v_j | 1])
//   dGamma_K[j][k] = [v_j | 1] . D[k] + sum_{i >= j in segment} A[i][j] Gamma_Q[i][k]
// (P = Gamma_Q Gamma_K^T and A[i][j] = dnd_i . [v_j | 1], causal only: the query-side kernels'
// tiles, stored transposed per segment and read back here), and the row's <Gamma_K, dGamma_K>.
template <int DV>
__host__ __device__ constexpr int dk_smem_floats() { return 2 * KT * LT + 2 * DV * LT + KT; }

template <int DV, typename Tin>
__global__ void __launch_bounds__(BT, DV == 64 ? 3 : 2) bwd_dk_kernel(const float *__restrict__ gq, const float *__restrict__ gk,
                                                    const Tin *__restrict__ V, const float *__restrict__ dagg,
                                                    const float *__restrict__ dnd, const float *__restrict__ Pg,
                                                    const float *__restrict__ Ag, float *__restrict__ dgk,
                                                    float *__restrict__ dotk, Tin *__restrict__ dV, int N, int K,
                                                    int nseg, int causal)
{
    chain_enter();
    extern __shared__ __align__(16) float sm[];
    constexpr int DV1 = DV + 1, NC = DV / 16;
    float *gqT = sm;                 // [SEG][LT] P, then A
    float *gkT = gqT + KT * LT;      // [KT][LT] Gamma_K^T tile; later Gamma_Q tiles [SEG][KT]
    float *VT = gkT + KT * LT;       // [DV][LT] V^T; before it, the D tiles [KT][DV], then the dnum rows
    float *DT = VT + DV * LT;        // [DV][LT] D^T tiles
    float *zD = DT + DV * LT;        // [KT]
    float *sD = VT;
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg;
    const int j0 = seg * SEG, n = min(SEG, N - j0);
    const long long row0 = (long long)bh * N + j0;
    const float *D = dagg + ((size_t)bh * nseg + (causal ? seg : 0)) * K * DV1;
    const int t = threadIdx.x, r0 = orow();
    // dV
    float accV[4][NC];
    zero<DV>(accV);
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        stage_t<KT>(gkT, LT, gk + row0 * K + k0, K, n, kn);
        stage<DV>(sD, DV, D + (size_t)k0 * DV1, DV1, kn, DV);
        __syncthreads();
        mac<DV>(accV, gkT, LT, sD, DV, KT);                // rows j, columns c
    }
    __syncthreads();
    if (causal) {
        // P[i][j] from the query-side kernel's P^T tile
        stage_t<SEG>(gqT, LT, Pg + (size_t)blockIdx.x * SEG * SEG, SEG, SEG, SEG);
        stage<DV>(sD, DV, dnd + row0 * DV1, DV1, n, DV);
        __syncthreads();
        mac_range<DV>(accV, gqT, LT, sD, DV, r0, SEG);   // sum_{i >= j} P[i][j] dnum_i
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int j = r0 + r;
        if (j < n)
#pragma unroll
            for (int c = 0; c < NC; ++c) dV[(row0 + j) * DV + ocol<DV>(c)] = from_f32<Tin>(accV[r][c]);
    }
    // dGamma_K
    __syncthreads();
    stage_t<DV>(VT, LT, V + row0 * DV, DV, n, DV);
    // A[i][j] from the query-side kernel's A^T tile
    if (causal) stage_t<SEG>(gqT, LT, Ag + (size_t)blockIdx.x * SEG * SEG, SEG, SEG, SEG);
    const bool one = K <= KT;
    float dot[4] = {0.f, 0.f, 0.f, 0.f}, gsv[4][4], acc[4][4];
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        stage_t<DV>(DT, LT, D + (size_t)k0 * DV1, DV1, kn, DV);   // D^T: [c][k]
        if (t < KT) zD[t] = t < kn ? D[(size_t)(k0 + t) * DV1 + DV] : 0.f;
        if (causal) stage<KT>(gkT, KT, gq + row0 * K + k0, K, n, kn);
        __syncthreads();
        zero<64>(acc);
        mac<64>(acc, VT, LT, DT, LT, DV);                 // rows j, columns k
        if (causal) mac_range<64>(acc, gqT, LT, gkT, KT, r0, SEG);   // (A[i][j] = 0 for i < j)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = r0 + r;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int kk = ocol<64>(c), k = k0 + kk;
                const float v = acc[r][c] + zD[kk];
                gsv[r][c] = j < n && k < K ? gk[(row0 + j) * K + k] : 0.f;
                dot[r] = fmaf(gsv[r][c], v, dot[r]);
                acc[r][c] = v;
                if (!one && j < n && k < K) dgk[(row0 + j) * K + k] = v;
            }
        }
    }
    row_sums(dot);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int j = r0 + r;
        if (one) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int k = ocol<64>(c);
                if (j < n && k < K) dgk[(row0 + j) * K + k] = gsv[r][c] * (acc[r][c] - dot[r]);
            }
        } else if (tile_tx() == 0 && j < n) {
            dotk[row0 + j] = dot[r];
        }
    }
}

// ---------------------------------------------------------------- through the responsibilities
// The rows of one segment of one side (blockIdx.y: 0 queries, 1 keys):
//   dL = Gamma (dGamma - <Gamma, dGamma>)     (written back over dGamma for the parameters; with
//                                             one component tile the kernels before formed it)
//   dx_d = sum_k dL_k (w_kd mu_kd - w_kd x_d)  (w = 1 / sigma^2)
// The contraction over k runs as the products above, with the factor w_kd mu_kd - w_kd x_d formed
// per step from the thread's own x (two FMAs per term).
template <int DR>
__host__ __device__ constexpr int dx_smem_floats() { return KT * LT + 2 * KT * DR + SEG; }

template <int DR, typename Tin>
__global__ void __launch_bounds__(BT, DR <= 64 ? 3 : 2) bwd_dx_kernel(const Tin *__restrict__ QX, const Tin *__restrict__ KX,
                                                    const float *__restrict__ gq, const float *__restrict__ gk,
                                                    float *__restrict__ dgq, float *__restrict__ dgk,
                                                    const float *__restrict__ dotq, const float *__restrict__ dotk,
                                                    const float *__restrict__ mu, const float *__restrict__ iv,
                                                    Tin *__restrict__ dQX, Tin *__restrict__ dKX, int H, int N, int K,
                                                    int nseg)
{
    chain_enter();
    extern __shared__ __align__(16) float sm[];
    constexpr int NC = DR / 16;
    float *dLT = sm;                 // [KT][LT] dL^T tile
    float *sW = dLT + KT * LT;       // [KT][DR] w
    float *sWM = sW + KT * DR;       // [KT][DR] w mu
    float *sdot = sWM + KT * DR;     // [SEG]
    const int side = blockIdx.y;
    const Tin *X = side ? KX : QX;
    const float *g = side ? gk : gq;
    float *dg = side ? dgk : dgq;
    Tin *dX = side ? dKX : dQX;
    const int bh = blockIdx.x / nseg, seg = blockIdx.x % nseg, h = bh % H;
    const int i0 = seg * SEG, n = min(SEG, N - i0);
    const long long row0 = (long long)bh * N + i0;
    const int t = threadIdx.x, r0 = orow();
    const bool one = K <= KT;   // (one component tile: dGamma already holds dL)
    if (t < SEG) sdot[t] = t < n && !one ? (side ? dotk : dotq)[row0 + t] : 0.f;
    float x[4][NC], acc[4][NC];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            x[r][c] = r0 + r < n ? to_f32(X[(row0 + r0 + r) * DR + ocol<DR>(c)]) : 0.f;
            acc[r][c] = 0.f;
        }
    const float *muh = mu + (size_t)h * K * DR, *ivh = iv + (size_t)h * K * DR;
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        // the tile's Gamma and dGamma first (8 of each per thread in flight), then dL; a thread
        // keeps component kk and takes rows rb, rb + 4, ...
        constexpr int PER = SEG * KT / BT;
        const int kk = t % KT, rb = t / KT;
        const bool kok = kk < kn;
        const long long o0 = (row0 + rb) * K + k0 + kk;
#pragma unroll
        for (int h0 = 0; h0 < PER; h0 += PER / 2) {   // (two halves: fewer registers held)
            float gv[PER / 2], dv[PER / 2];
#pragma unroll
            for (int u = 0; u < PER / 2; ++u) {
                const int rr = rb + 4 * (h0 + u);
                const bool ok = kok && rr < n;
                gv[u] = ok && !one ? g[o0 + (long long)(h0 + u) * 4 * K] : 0.f;
                dv[u] = ok ? dg[o0 + (long long)(h0 + u) * 4 * K] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < PER / 2; ++u) {
                const int rr = rb + 4 * (h0 + u);
                const float v = one ? dv[u] : gv[u] * (dv[u] - sdot[rr]);
                if (!one && kok && rr < n) dg[o0 + (long long)(h0 + u) * 4 * K] = v;
                dLT[kk * LT + rr] = v;
            }
        }
        stage<DR>(sW, DR, ivh + (size_t)k0 * DR, DR, kn, DR);
        stage<DR>(sWM, DR, muh + (size_t)k0 * DR, DR, kn, DR);
        __syncthreads();
        for (int e = t; e < KT * DR; e += BT) sWM[e] *= sW[e];   // w mu
        __syncthreads();
#pragma unroll 2
        for (int q = 0; q < KT; ++q) {
            const float4 a = *reinterpret_cast<const float4 *>(dLT + q * LT + r0);
            float w[NC], wm[NC];
            ld_cols<DR>(w, sW + q * DR);
            ld_cols<DR>(wm, sWM + q * DR);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                acc[0][c] = fmaf(a.x, fmaf(-w[c], x[0][c], wm[c]), acc[0][c]);
                acc[1][c] = fmaf(a.y, fmaf(-w[c], x[1][c], wm[c]), acc[1][c]);
                acc[2][c] = fmaf(a.z, fmaf(-w[c], x[2][c], wm[c]), acc[2][c]);
                acc[3][c] = fmaf(a.w, fmaf(-w[c], x[3][c], wm[c]), acc[3][c]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
        if (r0 + r < n)
#pragma unroll
            for (int c = 0; c < NC; ++c) dX[(row0 + r0 + r) * DR + ocol<DR>(c)] = from_f32<Tin>(acc[r][c]);
}

// ---------------------------------------------------------------- parameter gradients
// Partial sums of head h over a range of 64-row blocks (query rows, then key rows; block b is side
// b / (B nseg), batch row (b / nseg) % B, segment b % nseg) for the components of one tile:
//   m1[h][ch][k][d] = sum dL_k x_d,  m2[h][ch][k][d] = sum dL_k x_d^2,  pl[h][ch][k] = sum dL_k,
// two FMAs per term (x^2 formed once per row and column); the final kernel turns them into
// sum dL_k (x_d - mu_kd) = m1 - mu pl and sum dL_k (x_d - mu_kd)^2 = m2 - 2 mu m1 + mu^2 pl.
template <int DR>
__host__ __device__ constexpr int param_smem_floats() { return SEG * KT + SEG * DR; }

template <int DR, typename Tin>
__global__ void __launch_bounds__(BT, 2) bwd_param_partial_kernel(const Tin *__restrict__ QX, const Tin *__restrict__ KX,
                                                                  const float *__restrict__ dLq,
                                                                  const float *__restrict__ dLk,
                                                                  float *__restrict__ m1, float *__restrict__ m2,
                                                                  float *__restrict__ pl, int B, int H, int N, int K,
                                                                  int nseg, int R)
{
    chain_enter();
    extern __shared__ __align__(16) float sm[];
    constexpr int NC = DR / 16;
    float *sL = sm;                  // [SEG][KT] dL rows
    float *sX = sL + SEG * KT;       // [SEG][DR] x rows
    const int h = blockIdx.x, k0 = blockIdx.y * KT, ch = blockIdx.z;
    const int kn = min(KT, K - k0);
    const int t = threadIdx.x, r0 = orow();
    float a1[4][NC], a2[4][NC];
    zero<DR>(a1);
    zero<DR>(a2);
    float al = 0.f;
    const int nb = 2 * B * nseg;
    const int lo = (int)((long long)nb * ch / R), hi = (int)((long long)nb * (ch + 1) / R);
    // block b's dL and x rows; the loads of block b + 1 are issued before block b's products
    Staged<KT> nL;
    Staged<DR> nX;
    auto load = [&](int b) {
        const int side = b / (B * nseg), bb = (b / nseg) % B, seg = b % nseg;
        const int n = min(SEG, N - seg * SEG);
        const long long row0 = ((long long)bb * H + h) * N + seg * SEG;
        stage_load<KT>(nL, (side ? dLk : dLq) + row0 * K + k0, K, n, kn);
        stage_load<DR>(nX, (side ? KX : QX) + row0 * DR, DR, n, DR);
    };
    constexpr bool PREFETCH = DR <= 64;   // (at d_r = 128 the accumulators leave no registers for it)
    if (PREFETCH && lo < hi) load(lo);
    for (int b = lo; b < hi; ++b) {
        __syncthreads();
        if (!PREFETCH) load(b);
        stage_store<KT>(sL, KT, nL);
        stage_store<DR>(sX, DR, nX);
        __syncthreads();
        if (PREFETCH && b + 1 < hi) load(b + 1);
#pragma unroll 4
        for (int q = 0; q < SEG; ++q) {
            const float4 a = *reinterpret_cast<const float4 *>(sL + q * KT + r0);
            float xv[NC];
            ld_cols<DR>(xv, sX + q * DR);
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const float x2 = xv[c] * xv[c];
                a1[0][c] = fmaf(a.x, xv[c], a1[0][c]);
                a1[1][c] = fmaf(a.y, xv[c], a1[1][c]);
                a1[2][c] = fmaf(a.z, xv[c], a1[2][c]);
                a1[3][c] = fmaf(a.w, xv[c], a1[3][c]);
                a2[0][c] = fmaf(a.x, x2, a2[0][c]);
                a2[1][c] = fmaf(a.y, x2, a2[1][c]);
                a2[2][c] = fmaf(a.z, x2, a2[2][c]);
                a2[3][c] = fmaf(a.w, x2, a2[3][c]);
            }
        }
        if (t < KT)
            for (int q = 0; q < SEG; ++q) al += sL[q * KT + t];
    }
    const size_t base = ((size_t)h * R + ch) * K;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int k = k0 + r0 + r;
        if (r0 + r < kn)
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                m1[(base + k) * DR + ocol<DR>(c)] = a1[r][c];
                m2[(base + k) * DR + ocol<DR>(c)] = a2[r][c];
            }
    }
    if (t < kn) pl[base + k0 + t] = al;
}

// Over the chunks in order, a1 = sum dL_k x_d, a2 = sum dL_k x_d^2, c = sum dL_k; then
//   dmu = w (a1 - mu c),  d(raw) = (w^2 (a2 - 2 mu a1 + mu^2 c) - w c) / 2 * sigmoid(raw);
// the last block row (blockIdx.y == gridDim.y - 1) takes d(logits) = dlogpi - pi * sum(dlogpi) per
// head instead.  Eight chunks' loads are issued at a time.
__global__ void __launch_bounds__(BT) bwd_param_final_kernel(const float *__restrict__ m1, const float *__restrict__ m2,
                                                             const float *__restrict__ pl, const float *__restrict__ iv,
                                                             const float *__restrict__ mu, const float *__restrict__ raw,
                                                             const float *__restrict__ logits, float *__restrict__ dmu,
                                                             float *__restrict__ draw, float *__restrict__ dlogits,
                                                             int K, int d_r, int R)
{
    chain_enter();
    __shared__ float red[BT / 32][2];
    __shared__ float sl[1024];   // dlogpi per component (K <= 1024)
    const int h = blockIdx.x;
    const int KD = K * d_r;
    if (blockIdx.y + 1 < gridDim.y) {
        const int e = blockIdx.y * BT + threadIdx.x;
        if (e >= KD) return;
        const int k = e / d_r;
        float a = 0.f, b = 0.f, c = 0.f;
        for (int c0 = 0; c0 < R; c0 += 8) {
            float va[8], vb[8], vc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool ok = c0 + u < R;
                const size_t ch = (size_t)h * R + c0 + u;
                va[u] = ok ? m1[ch * KD + e] : 0.f;
                vb[u] = ok ? m2[ch * KD + e] : 0.f;
                vc[u] = ok ? pl[ch * K + k] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                a += va[u];
                b += vb[u];
                c += vc[u];
            }
        }
        const float w = iv[(size_t)h * KD + e], m = mu[(size_t)h * KD + e], r = raw[(size_t)h * KD + e];
        const float s1 = fmaf(-m, c, a);                       // sum dL (x - mu)
        const float s2 = fmaf(m, fmaf(m, c, -2.f * a), b);     // sum dL (x - mu)^2
        dmu[(size_t)h * KD + e] = w * s1;
        draw[(size_t)h * KD + e] = 0.5f * (w * w * s2 - w * c) / (1.f + expf(-r));
        return;
    }
    // prior logits: pi = softmax(logits); dlogits = dlogpi - pi * sum_k dlogpi
    const float *lh = logits + (size_t)h * K;
    float m = -INFINITY, tl = 0.f;
    for (int k = threadIdx.x; k < K; k += BT) {
        m = fmaxf(m, lh[k]);
        float a = 0.f;
        for (int c0 = 0; c0 < R; c0 += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = c0 + u < R ? pl[((size_t)h * R + c0 + u) * K + k] : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) a += v[u];
        }
        sl[k] = a;
        tl += a;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        tl += __shfl_xor_sync(0xffffffffu, tl, o);
    }
    if ((threadIdx.x & 31) == 0) {
        red[threadIdx.x >> 5][0] = m;
        red[threadIdx.x >> 5][1] = tl;
    }
    __syncthreads();
    m = red[0][0];
    tl = 0.f;
    for (int wv = 0; wv < BT / 32; ++wv) {
        m = fmaxf(m, red[wv][0]);
        tl += red[wv][1];
    }
    float se = 0.f;
    for (int k = threadIdx.x; k < K; k += BT) se += expf(lh[k] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5][0] = se;
    __syncthreads();
    se = 0.f;
    for (int wv = 0; wv < BT / 32; ++wv) se += red[wv][0];
    for (int k = threadIdx.x; k < K; k += BT) {
        const float pi = expf(lh[k] - m) / se;
        dlogits[(size_t)h * K + k] = sl[k] - pi * tl;
    }
}

struct BwdLayout {
    size_t iv, cst, gq, gk, agg, dnd, dagg, dgq, dgk, dotq, dotk, pt, at, m1, m2, pl, total;
    int nseg, R, ktiles;
};

BwdLayout bwd_layout(const gma_shape_t &s)
{
    BwdLayout L{};
    Carve c;
    const size_t T = (size_t)s.B * s.H * s.N;
    const int dv1 = s.d_v + 1;
    L.nseg = (s.N + SEG - 1) / SEG;
    L.ktiles = (s.K + KT - 1) / KT;
    // parameter partials: one wave of two blocks per SM, at most one chunk per 64-row block
    const int nb = 2 * s.B * L.nseg;
    int R = 2 * 152 / (s.H * L.ktiles);
    if (R > nb) R = nb;
    if (R < 1) R = 1;
    L.R = R;
    L.iv = c.take(5 * sizeof(float) * (size_t)s.H * s.K * s.d_r);   // 1/sigma^2 and four transposes
    L.cst = c.take(sizeof(float) * (size_t)s.H * s.K);
    L.gq = c.take(sizeof(float) * T * s.K);
    L.gk = c.take(sizeof(float) * T * s.K);
    L.agg = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * s.K * dv1);
    L.dnd = c.take(sizeof(float) * T * dv1);
    L.dagg = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * s.K * dv1);
    L.dgq = c.take(sizeof(float) * T * s.K);
    L.dgk = c.take(sizeof(float) * T * s.K);
    L.dotq = c.take(sizeof(float) * T);
    L.dotk = c.take(sizeof(float) * T);
    L.pt = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * SEG * SEG);   // P^T per segment
    L.at = c.take(sizeof(float) * (size_t)s.B * s.H * L.nseg * SEG * SEG);   // A^T per segment
    L.m1 = c.take(sizeof(float) * (size_t)s.H * R * s.K * s.d_r);
    L.m2 = c.take(sizeof(float) * (size_t)s.H * R * s.K * s.d_r);
    L.pl = c.take(sizeof(float) * (size_t)s.H * R * s.K);
    L.total = c.total();
    return L;
}

template <typename... P>
bool set_smem(void (*k)(P...), int floats)
{
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, floats * (int)sizeof(float)) ==
           cudaSuccess;
}

// The segment kernels for one value width.
template <int DV, typename Tin>
gma_status_t launch_segments(const gma_shape_t &s, const BwdLayout &L, bool causal, const Tin *V, const Tin *dO,
                             Tin *dV, char *ws, cudaStream_t st)
{
    float *gq = (float *)(ws + L.gq), *gk = (float *)(ws + L.gk), *agg = (float *)(ws + L.agg);
    float *dnd = (float *)(ws + L.dnd), *dagg = (float *)(ws + L.dagg);
    float *dgq = (float *)(ws + L.dgq), *dgk = (float *)(ws + L.dgk);
    float *dotq = (float *)(ws + L.dotq), *dotk = (float *)(ws + L.dotk);
    float *pt = (float *)(ws + L.pt), *at = (float *)(ws + L.at);
    const int BH = s.B * s.H, cz = causal ? 1 : 0;
    const dim3 grid((unsigned)(BH * L.nseg));
    if (!set_smem(bwd_numden_kernel<DV, Tin>, numden_smem_floats<DV>()) ||
        !set_smem(bwd_dgq_kernel<DV, Tin>, dgq_smem_floats<DV>()) ||
        !set_smem(bwd_dk_kernel<DV, Tin>, dk_smem_floats<DV>()))
        return GMA_ERR_CUDA;
    gma_status_t r = GMA_OK;
    if ((r = launch_chained(KID_BWD_NUMDEN, st, bwd_numden_kernel<DV, Tin>, grid, dim3(BT),
                            sizeof(float) * numden_smem_floats<DV>(), (const float *)gq, (const float *)gk, V,
                            (const float *)agg, dO, dnd, dagg, pt, s.N, s.K, L.nseg, s.eps, cz)) != GMA_OK)
        return r;
    if ((r = launch_chained(KID_BWD_DQ, st, bwd_dgq_kernel<DV, Tin>, grid, dim3(BT),
                            sizeof(float) * dgq_smem_floats<DV>(), (const float *)gq, (const float *)gk, V,
                            (const float *)agg, (const float *)dnd, dgq, dotq, at, s.N, s.K, L.nseg, cz)) != GMA_OK)
        return r;
    const int KD = s.K * (s.d_v + 1);
    const long long tot = (long long)BH * KD;
    if (KD % 4 == 0)
        r = launch_chained(KID_BWD_SCAN, st, bwd_scan_kernel<4>, dim3((unsigned)((tot / 4 + BT - 1) / BT)), dim3(BT), 0,
                           dagg, tot, L.nseg, KD, cz);
    else
        r = launch_chained(KID_BWD_SCAN, st, bwd_scan_kernel<1>, dim3((unsigned)((tot + BT - 1) / BT)), dim3(BT), 0,
                           dagg, tot, L.nseg, KD, cz);
    if (r != GMA_OK) return r;
    return launch_chained(KID_BWD_DK, st, bwd_dk_kernel<DV, Tin>, grid, dim3(BT), sizeof(float) * dk_smem_floats<DV>(),
                          (const float *)gq, (const float *)gk, V, (const float *)dagg, (const float *)dnd,
                          (const float *)pt, (const float *)at, dgk, dotk, dV, s.N, s.K, L.nseg, cz);
}

// The kernels through the responsibilities for one routing width.
template <int DR, typename Tin>
gma_status_t launch_rows(const gma_shape_t &s, const BwdLayout &L, const Tin *QX, const Tin *KX, const float *mu,
                         const float *raw, const float *logits, Tin *dQX, Tin *dKX, float *dmu, float *draw,
                         float *dlogits, char *ws, cudaStream_t st)
{
    const float *iv = (const float *)(ws + L.iv);
    const float *gq = (const float *)(ws + L.gq), *gk = (const float *)(ws + L.gk);
    float *dgq = (float *)(ws + L.dgq), *dgk = (float *)(ws + L.dgk);
    const float *dotq = (const float *)(ws + L.dotq), *dotk = (const float *)(ws + L.dotk);
    float *m1 = (float *)(ws + L.m1), *m2 = (float *)(ws + L.m2), *pl = (float *)(ws + L.pl);
    if (!set_smem(bwd_dx_kernel<DR, Tin>, dx_smem_floats<DR>()) ||
        !set_smem(bwd_param_partial_kernel<DR, Tin>, param_smem_floats<DR>()))
        return GMA_ERR_CUDA;
    gma_status_t r = GMA_OK;
    if ((r = launch_chained(KID_BWD_DX, st, bwd_dx_kernel<DR, Tin>, dim3((unsigned)(s.B * s.H * L.nseg), 2), dim3(BT),
                            sizeof(float) * dx_smem_floats<DR>(), QX, KX, gq, gk, dgq, dgk, dotq, dotk, mu, iv, dQX,
                            dKX, s.H, s.N, s.K, L.nseg)) != GMA_OK)
        return r;
    if ((r = launch_chained(KID_BWD_PARAMS, st, bwd_param_partial_kernel<DR, Tin>,
                            dim3((unsigned)s.H, (unsigned)L.ktiles, (unsigned)L.R), dim3(BT),
                            sizeof(float) * param_smem_floats<DR>(), QX, KX, (const float *)dgq, (const float *)dgk,
                            m1, m2, pl, s.B, s.H, s.N, s.K, L.nseg, L.R)) != GMA_OK)
        return r;
    const int KD = s.K * s.d_r;
    return launch_chained(KID_BWD_PFINAL, st, bwd_param_final_kernel, dim3((unsigned)s.H, (unsigned)((KD + BT - 1) / BT + 1)),
                          dim3(BT), 0, (const float *)m1, (const float *)m2, (const float *)pl, iv, mu, raw, logits, dmu,
                          draw, dlogits, s.K, s.d_r, L.R);
}

template <typename Tin>
gma_status_t backward_typed(const gma_shape_t &s, bool causal, const Tin *QX, const Tin *KX, const Tin *V,
                            const float *mu, const float *raw, const float *logits, const Tin *dO, Tin *dQX, Tin *dKX,
                            Tin *dV, float *dmu, float *draw, float *dlogits, char *ws, cudaStream_t st)
{
    const BwdLayout L = bwd_layout(s);
    gma_status_t r = simt_prepare(s, causal, QX, KX, V, mu, raw, logits, (float *)(ws + L.iv), (float *)(ws + L.cst),
                                  (float *)(ws + L.gq), (float *)(ws + L.gk), (float *)(ws + L.agg), st);
    if (r != GMA_OK) return r;
    switch (s.d_v) {
    case 16: r = launch_segments<16, Tin>(s, L, causal, V, dO, dV, ws, st); break;
    case 32: r = launch_segments<32, Tin>(s, L, causal, V, dO, dV, ws, st); break;
    case 64: r = launch_segments<64, Tin>(s, L, causal, V, dO, dV, ws, st); break;
    case 128: r = launch_segments<128, Tin>(s, L, causal, V, dO, dV, ws, st); break;
    default: return GMA_ERR_UNSUPPORTED_SHAPE;
    }
    if (r != GMA_OK) return r;
    switch (s.d_r) {
    case 16: return launch_rows<16, Tin>(s, L, QX, KX, mu, raw, logits, dQX, dKX, dmu, draw, dlogits, ws, st);
    case 32: return launch_rows<32, Tin>(s, L, QX, KX, mu, raw, logits, dQX, dKX, dmu, draw, dlogits, ws, st);
    case 64: return launch_rows<64, Tin>(s, L, QX, KX, mu, raw, logits, dQX, dKX, dmu, draw, dlogits, ws, st);
    case 128: return launch_rows<128, Tin>(s, L, QX, KX, mu, raw, logits, dQX, dKX, dmu, draw, dlogits, ws, st);
    default: return GMA_ERR_UNSUPPORTED_SHAPE;
    }
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
