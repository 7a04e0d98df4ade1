// gma_tc_causal_g.cu -- the chunked causal GMA kernel fed with stored key responsibilities
// (tcgen05, sm_103a), warp-specialised.
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §3 (causal variant: prefix sums of the latent memory and its normaliser) on top
// of §1 (posterior responsibilities) and §2 (write and read phases).
//
// The segment pass has already computed Gamma_K of every token (bf16, normalised) and stored it
// in the workspace; this pass reads it back by TMA instead of recomputing it.  One CTA handles
// one segment of one (batch, head) slice from the segment's exclusive prefix memory S_start, in
// chunks of C = 128 tokens.  With E_Q = exp2 of the query logits minus their row maximum (row
// sums s_i, kept unnormalised):
//   [P | O_num] = E_Q [Gamma_K^T | S_{c-1}]          (tensor cores, one N = 128 + d_v chain)
//   O_num += tril(P) V_c                             (tensor cores)
//   den    = E_Q . Z_{c-1} + sum_{j<=i} P_ij         (CUDA cores, fp32)
//   O      = O_num / (den + eps * s)
//   S_c^T  = S_{c-1}^T + V_c^T Gamma_K               (tensor cores, fp32 in TMEM)
//   Z_c    = Z_{c-1} + column sums of Gamma_K        (CUDA cores, fp32)
// The running memory is kept transposed (TMEM lane = value column, columns = components), so
// that its bf16 copy is written row by row as K-major rows next to Gamma_K's in one operand tile
// [Gamma_K ; S^T] (128 + d_v rows): P and the inter-chunk read E_Q S_{c-1} come out of the same
// MMA chain.  Value tiles are held 128 columns wide (zeros beyond d_v), so that V^T is an M = 128
// operand for every d_v.
//
// Warp roles (448 threads):
//   warps 0-3   mask side:  E_Q of the upper half of the components (see below), then the causal
//                           mask of P (bf16, back into TMEM as the A operand of tril(P) V) and
//                           the complete normaliser;
//   warps 4-7   query side: [x^2, x] of the queries (in place in the TMA-filled A tile), E_Q of
//                           the lower half of the components, their row sums and E_Q . Z_{c-1};
//   warps 8-11  state/out:  the starting memory, Z_c, the bf16 operand copy of S_c^T, and the
//                           output rows;
//   warp 12     control:    every tcgen05.mma, each as soon as its inputs are complete;
//   warp 13     loader:     every TMA load (query rows, Gamma_K and value tiles), each as soon
//                           as its buffer is free, so that no load waits behind an MMA issue.
// Tensor memory (512 columns): [0,128) query logits, then E_Q; [128,256) P; [256,384) output
// numerator; [384,512) the running memory S^T.  The next chunk's query logits are computed while
// the current chunk is masked, so the query exponentials are the only long step between chunks;
// two warps share each row of them: each takes the maximum of one half of the components'
// logits, the two half-row maxima are exchanged, and each exponentiates its half.  E_Q of 32-column group g (of kc groups, h = ceil(kc / 2) in the lower half) is
// packed into 16 columns at 16 g (g < h) or 16 h + 16 g (g >= h), after both halves have read
// all of their logits.
// Every wait is bounded; a timeout records GMA_ERR_TIMEOUT and makes all roles leave their loops.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

constexpr int GTHREADS = 448;
enum GBar {
    G_BIMG, G_V0, G_V1, G_XQ, G_GT,                             // TMA (transaction counts)
    G_AQ, G_XM, G_GQ0, G_GQ1, G_PS0, G_PS1, G_ZP, G_SP, G_OF,   // 128 threads (XM, GQ: 256)
    G_ZB0, G_ZB1,                                               // 128 threads
    G_LQ, G_P, G_PQ, G_S, G_PV0, G_PV1,                         // tcgen05.commit
    G_NBAR
};
// Barriers completed once per chunk but waited on by a role that could in principle fall a
// chunk behind come in pairs by chunk parity (GQ, PS, PV): each completes once per two chunks.
constexpr uint32_t R_LQ = 0, R_P = 128, R_O = 256, R_S = 384;

struct GSmem {
    uint32_t bimg, ax, abq, gk, ve0, ve1, zbuf, zpart, xmax, dsq, dsm, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ GSmem(int DR, int kn16, int d_v)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        const uint32_t tile = ka / 64u * 128u;
        uint32_t o = 0;
        bimg = o; o = al(o + tile * (uint32_t)kn16 + 32u * (uint32_t)kn16);
        ax = o; o = al(o + (uint32_t)C * 32u);
        abq = o; o = al(o + (uint32_t)C * DR * 4u);   // queries [x^2 | x]
        gk = o; o = al(o + 2u * (uint32_t)(C + d_v) * 128u);   // [Gamma_K (TMA) ; S^T], two atoms
        ve0 = o; o = al(o + (uint32_t)KMAX * C * 2u);   // value tiles by chunk parity, 128 columns
        ve1 = o; o = al(o + (uint32_t)KMAX * C * 2u);
        zbuf = o; o += 2u * KMAX * 4u;         // Z_{c-1} by chunk parity
        zpart = o; o += 2u * 8u * KMAX * 4u;   // partial column sums by chunk parity
        xmax = o; o += 4u * C * 4u;            // half-row maxima per half, by chunk parity
        dsq = o; o += 2u * C * 8u;             // query side's (row sum, E_Q . Z), by chunk parity
        dsm = o; o += 2u * C * 8u;             // (row sum, normaliser) per query row, by chunk parity
        bars = o; o += G_NBAR * 8u;
        misc = o; o += 16u;
        total = o;
    }
};

// TMA of the Gamma_K rows [tok, tok + 128) of slice bh: kg / 64 boxes of 64 components, each
// the 128-byte-swizzled K-major layout of one 64-component atom of the [Gamma_K ; S^T] tile
// (nb = 128 + d_v rows per atom; Gamma_K takes the first 128).
__device__ __forceinline__ void load_g_tile(uint8_t *gk, const CUtensorMap *map, uint64_t *bar, int kg, int nb, int tok,
                                            int bh)
{
    mbar_arrive_expect_tx(bar, (uint32_t)(C * kg * 2));
    for (int hf = 0; hf < kg / 64; ++hf)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(gk + hf * nb * 128)),
            "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(64 * hf), "r"(tok), "r"(bh)
            : "memory");
}

// Query rows: the maximum of this row's logits over the 32-column groups [g0, g1) and the columns
// below K (one group per wait: holding two groups at once would not fit the register budget).
__device__ __forceinline__ float query_max_half(uint32_t tl, int K, int g0, int g1)
{
    float m[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) m[u] = NEG_BIG;
#pragma unroll 1
    for (int c = g0; c < g1; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if ((c + 1) * 32 <= K || 32 * c + j < K) m[j & 7] = fmaxf(m[j & 7], __uint_as_float(r[j]));
    }
    return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

// Four consecutive floats of shared memory, read in program order with respect to the other
// inline-assembly statements (so that the loads of one group are not hoisted above the previous
// group's tensor-memory store, which would keep both groups' values live at once).
__device__ __forceinline__ float4 lds4_ordered(const float *p)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// Query rows: unnormalised E_Q = exp2(L - m) of one 32-column group c held in r, zero beyond K,
// back into TMEM at tl as bf16 pairs (group c at column 16 c + (c >= h ? 16 h : 0)); adds the
// group's sum and its dot product with z = Z_{c-1} to *srow and *den.
__device__ __forceinline__ void query_exp_group(uint32_t tl, int K, int c, int h, float m, uint32_t (&r)[32],
                                                const float *z, float &srow, float &den)
{
    srow += chunk_exp(r, c, K, m);
    float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 zz = lds4_ordered(z + 32 * c + 4 * q);
        d4[0] = fmaf(__uint_as_float(r[4 * q]), zz.x, d4[0]);
        d4[1] = fmaf(__uint_as_float(r[4 * q + 1]), zz.y, d4[1]);
        d4[2] = fmaf(__uint_as_float(r[4 * q + 2]), zz.z, d4[2]);
        d4[3] = fmaf(__uint_as_float(r[4 * q + 3]), zz.w, d4[3]);
    }
    den += (d4[0] + d4[1]) + (d4[2] + d4[3]);
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    tmem_st16(tl + 16 * c + (c >= h ? 16 * h : 0), w);   // E_Q (bf16 pairs)
}

// Mask side: row i of P (fp32 in TMEM at tl) masked to columns j <= i, written back as bf16
// pairs in place; returns the sum of the kept fp32 values.
__device__ __forceinline__ float mask_row(uint32_t tl, int i)
{
    float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int col = 32 * c + 2 * j;
            const float p0 = col <= i ? __uint_as_float(r[2 * j]) : 0.f;
            const float p1 = col + 1 <= i ? __uint_as_float(r[2 * j + 1]) : 0.f;
            d4[j & 3] += p0 + p1;
            w[j] = pack_bf16(p0, p1);
        }
        tmem_st16(tl + 16 * c, w);
    }
    tmem_st_wait();
    return (d4[0] + d4[1]) + (d4[2] + d4[3]);
}

// State side: row n of the running memory S^T (the 128 component columns of TMEM lane n at tl)
// as bf16 into row 128 + n of the [Gamma_K ; S^T] tile gk (nb rows per atom).  Every lane loads
// (the loads are warp-collective); only rows n < d_v are written.
__device__ __forceinline__ void state_rows_t(uint32_t tl, uint8_t *gk, int nb, int n, bool write)
{
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        if (write) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = 8 * q;
                *reinterpret_cast<uint4 *>(gk + sw128(C + n, 4 * c + q, nb)) =
                    make_uint4(pk2(r[e], r[e + 1], 1.f), pk2(r[e + 2], r[e + 3], 1.f), pk2(r[e + 4], r[e + 5], 1.f),
                               pk2(r[e + 6], r[e + 7], 1.f));
            }
        }
    }
}

// State side: this thread's share of the column sums of the Gamma_K tile: components 8q..8q+7
// over the rows g, g+8, ..., g+120 (t = 16 g + q), into zp[g][8q .. 8q+7].
__device__ __forceinline__ void colsum_rows(const uint8_t *gk, int nb, float *zp, int t)
{
    const int q = t & 15, g = t >> 4;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int u = 0; u < C / 8; ++u) {
        const uint4 v = *reinterpret_cast<const uint4 *>(gk + sw128(g + 8 * u, q, nb));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[2 * e] += __uint_as_float(w[e] << 16);
            acc[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
        }
    }
    float4 *o = reinterpret_cast<float4 *>(zp + g * KMAX + 8 * q);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// Output side: output row orow = (d_v numerator columns of TMEM at tl) * inv, bf16 or fp32.
__device__ __forceinline__ void out_row(uint32_t tl, int d_v, float inv, bool valid, void *O, long long orow,
                                        int out_f32)
{
#pragma unroll 1
    for (int c = 0; c < (d_v + 31) / 32; ++c) {   // 32 columns per wait
        uint32_t r[32];
        if (d_v == 16) {
            tmem_ld16(tl, *reinterpret_cast<uint32_t(*)[16]>(r));
        } else {
            tmem_ld32(tl + 32 * c, r);
        }
        tmem_ld_wait();
        if (!valid) continue;
        const int col0 = 32 * c;
        const int ncol = d_v - col0 < 32 ? d_v - col0 : 32;
        if (out_f32) {
            float4 *o4 = reinterpret_cast<float4 *>((float *)O + orow * d_v + col0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (4 * q < ncol)
                    o4[q] = make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                                        __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv);
        } else {
            uint4 *o4 = reinterpret_cast<uint4 *>((bf16 *)O + orow * d_v + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (8 * q < ncol)
                    o4[q] = make_uint4(pk2(r[8 * q], r[8 * q + 1], inv), pk2(r[8 * q + 2], r[8 * q + 3], inv),
                                       pk2(r[8 * q + 4], r[8 * q + 5], inv), pk2(r[8 * q + 6], r[8 * q + 7], inv));
        }
    }
}

}  // namespace

template <int DR>
__global__ void __launch_bounds__(GTHREADS, 1) tc_causal_gamma_kernel(const Args a,
                                                                      const __grid_constant__ CUtensorMap vmap,
                                                                      const __grid_constant__ CUtensorMap qmap,
                                                                      const __grid_constant__ CUtensorMap gmap)
{
    // (no wait here: the set-up and the first loads of Q_X and V, which no kernel writes, overlap
    // the kernel before; the threads that read its results wait below)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const GSmem L(DR, a.kn16, a.d_v);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.misc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.misc + 4);
    float *zbuf = reinterpret_cast<float *>(smem + L.zbuf);
    float *zpart = reinterpret_cast<float *>(smem + L.zpart);
    float *xmax = reinterpret_cast<float *>(smem + L.xmax);
    float2 *dsq = reinterpret_cast<float2 *>(smem + L.dsq);
    float2 *dsm = reinterpret_cast<float2 *>(smem + L.dsm);
    const int bh = blockIdx.x / a.nseg, seg = blockIdx.x % a.nseg, h = bh % a.H;
    const int t = threadIdx.x, warp = t >> 5;
    const int tok0 = seg * a.cps * C;
    const int tok_end = min(a.N, tok0 + a.cps * C);
    const int nch = (tok_end - tok0 + C - 1) / C;
    const int d_v = a.d_v;
    // 32-column groups of E_Q: as many as the table's rows need (with components in tiles, the
    // last tile's E_Q beyond its K components is written as zeros, not left over from the logits)
    const int kc = (a.kn16 + 31) >> 5;
    const int nb = C + d_v;                         // rows of the [Gamma_K ; S^T] operand tile
    constexpr uint32_t XT = (uint32_t)C * DR * 2;   // bytes of one [x] tile (the TMA destination)

    // ---------------------------------------------------------------- set-up (all threads)
    if (warp == 12) {
        if (t == 384) {
            static const uint32_t counts[G_NBAR] = {1,   1,   1,   1,   1,   128, 256, 256, 256, 128,
                                                    128, 128, 128, 128, 128, 128, 1,   1,   1,   1,
                                                    1,   1};
            for (int i = 0; i < G_NBAR; ++i) mbar_init(bars + i, counts[i]);
            *abort = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(tslot, 512);
    } else if (warp < 4) {
        // [Gamma_K ; S^T] tile (with 64 stored components the second atom's Gamma_K rows are never
        // loaded) and both value tiles (their blocks beyond d_v are never loaded): zeros
        for (uint32_t o = t * 16; o < 2u * (uint32_t)(C + d_v) * 128u; o += 128 * 16)
            *reinterpret_cast<uint4 *>(smem + L.gk + o) = make_uint4(0, 0, 0, 0);
        for (uint32_t o = t * 16; o < (uint32_t)KMAX * C * 2u; o += 128 * 16) {
            *reinterpret_cast<uint4 *>(smem + L.ve0 + o) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(smem + L.ve1 + o) = make_uint4(0, 0, 0, 0);
        }
    } else if (warp < 8) {
        // constant A operand of the logits: (1, 1, 0, ...) in every row, K-major SW32
        const int i = t - 128;
        const uint32_t one2 = 0x3C003C00u;   // fp16 pair (1, 1)
        const int flip = (i >> 2) & 1;
        *reinterpret_cast<uint4 *>(smem + L.ax + i * 32 + (flip << 4)) = make_uint4(one2, 0, 0, 0);
        *reinterpret_cast<uint4 *>(smem + L.ax + i * 32 + ((flip ^ 1) << 4)) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);

    const int hq = (kc + 1) >> 1;   // 32-column groups of E_Q taken by the query side

    if (warp == 12) {
        // ============================================================ control warp: tcgen05.mma
        if (t == 384) {
            const uint32_t id_pq = idesc_f16(128, (uint32_t)nb, 1, 1, 0, 0);
            const uint32_t id_o = idesc_f16(128, (uint32_t)d_v, 1, 1, 0, 1);
            const uint32_t id_s = idesc_f16(128, (uint32_t)a.kn16, 1, 1, 1, 1);
            const int ksteps = a.kn16 / 16;
            auto eq_col = [&](int s) -> uint32_t { return (uint32_t)(8 * s + (s >= 2 * hq ? 16 * hq : 0)); };
            auto ve = [&](int c) -> uint32_t { return (c & 1) ? L.ve1 : L.ve0; };
            // value tile of chunk c, k-step s (16 tokens), as an MN-major operand
            auto vdesc = [&](int c, int s) -> uint64_t {
                return a.v128 ? mn128desc(sb + ve(c), s, C) : mn32desc(sb + ve(c), s, C);
            };
            int last_pv = -1;
            bool ok = mbar_wait_abortable(bars + G_BIMG, 0, a.hdr, 100, abort);
            const uint32_t bimg = sb + L.bimg, bconst = sb + L.bimg + (uint32_t)a.bimg_main_bytes;
            // query logits of chunk cq
            auto query_logits = [&](int cq) -> bool {
                if (!mbar_wait_abortable(bars + G_AQ, cq & 1, a.hdr, 101, abort)) return false;
                tc_fence_after();
                issue_logits_x<DR>(tmem + R_LQ, sb + L.abq, bimg, bconst, sb + L.ax, a.kn16);
                mma_commit(bars + G_LQ);
                return true;
            };
            // S^T += V^T Gamma_K of chunk cc (M = 128 value columns, zeros beyond d_v)
            auto update = [&](int cc) {
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s)
                    mma_f16(tmem + R_S, vdesc(cc, s), mn128desc(sb + L.gk, s, nb), id_s, 1u);
                mma_commit(bars + G_S);
            };
            if (ok && nch > 0) ok = query_logits(0);
            for (int c = 0; ok && c < nch; ++c) {
                const uint32_t ph = c & 1;
                // the S update goes first if its operands are already there (it needs no query)
                bool s_done = false;
                if (mbar_test_wait(bars + G_GT, ph) && mbar_test_wait(bars + G_V0 + ph, (c >> 1) & 1) &&
                    mbar_test_wait(bars + G_SP, ph)) {
                    update(c);
                    s_done = true;
                }
                // [P | O] = E_Q [Gamma_K^T | S_{c-1}]: E_Q and Gamma_K ready, S_{c-1}^T read out
                // into its rows of the tile, R_P free (tril(P_{c-1}) V done) and R_O read out
                if (!(ok = mbar_wait_abortable(bars + G_GQ0 + ph, (c >> 1) & 1, a.hdr, 103, abort))) break;
                if (!(ok = mbar_wait_abortable(bars + G_GT, ph, a.hdr, 104, abort))) break;
                if (c > 0 && !(ok = mbar_wait_abortable(bars + G_PV0 + ((c - 1) & 1), ((c - 1) >> 1) & 1, a.hdr,
                                                        106, abort)))
                    break;
                if (!(ok = mbar_wait_abortable(bars + G_SP, ph, a.hdr, 105, abort))) break;
                if (c > 0 && !(ok = mbar_wait_abortable(bars + G_OF, (c - 1) & 1, a.hdr, 107, abort))) break;
                tc_fence_after();
                for (int s = 0; s < ksteps; ++s)
                    mma_f16_tmem_a(tmem + R_P, tmem + R_LQ + eq_col(s), kdesc(sb + L.gk, s, nb), id_pq, s > 0);
                mma_commit(bars + G_P);
                mma_commit(bars + G_PQ);
                if (!s_done) {
                    if (!(ok = mbar_wait_abortable(bars + G_V0 + ph, (c >> 1) & 1, a.hdr, 108, abort))) break;
                    update(c);
                }
                // the next chunk's query logits once E_Q is consumed (they run while P is masked)
                if (c + 1 < nch) {
                    if (!(ok = mbar_wait_abortable(bars + G_PQ, ph, a.hdr, 109, abort))) break;
                    if (!(ok = query_logits(c + 1))) break;
                }
                // intra-chunk: O += tril(P) V
                if (!(ok = mbar_wait_abortable(bars + G_PS0 + ph, (c >> 1) & 1, a.hdr, 110, abort))) break;
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s)
                    mma_f16_tmem_a(tmem + R_O, tmem + R_P + 8 * s, vdesc(c, s), id_o, 1u);
                mma_commit(bars + G_PV0 + ph);
                last_pv = c;
            }
            // drain: MMAs complete in issue order, so the last commit covers them all
            if (last_pv >= 0) mbar_wait(bars + G_PV0 + (last_pv & 1), (last_pv >> 1) & 1, a.hdr, 114);
        }
    } else if (warp == 13) {
        // ============================================================ loader warp: every TMA load
        if (t == 416) {
            // TMA loads in flight: the chunk index of the last one issued per buffer (each buffer's
            // barrier completes one phase per load, and a load is issued only after the previous
            // one into that buffer was consumed)
            int last_v0 = -1, last_v1 = -1, last_xq = -1, last_gt = -1;
            bool ok = true;
            auto load_v = [&](int c) {
                uint8_t *dst = smem + ((c & 1) ? L.ve1 : L.ve0);
                if (a.v128)
                    load_v_chunk128(dst, &vmap, bars + G_V0 + (c & 1), d_v, tok0 + c * C, bh);
                else
                    load_v_chunk(dst, &vmap, bars + G_V0 + (c & 1), d_v, tok0 + c * C, bh);
                if (c & 1) last_v1 = c; else last_v0 = c;
            };
            // the query rows of chunk cq, once the logits of chunk cq - 1 are done with the A tile
            auto stage_queries = [&](int cq) -> bool {
                if (!mbar_wait_abortable(bars + G_LQ, (cq - 1) & 1, a.hdr, 102, abort)) return false;
                load_x_tile(smem + L.abq + XT, &qmap, bars + G_XQ, DR, tok0 + cq * C, bh);
                last_xq = cq;
                return true;
            };
            if (nch > 0) {
                load_x_tile(smem + L.abq + XT, &qmap, bars + G_XQ, DR, tok0, bh);
                last_xq = 0;
                load_v(0);
            }
            if (nch > 1) load_v(1);
            // Gamma_K and the tables come from the kernels before (the scan is the last of them)
            grid_dependency_wait();
            mbar_arrive_expect_tx(bars + G_BIMG, (uint32_t)a.bimg_bytes);
            bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars + G_BIMG);
            if (nch > 0) {
                load_g_tile(smem + L.gk, &gmap, bars + G_GT, a.kg, nb, tok0, bh);
                last_gt = 0;
            }
            if (nch > 1) ok = stage_queries(1);
            for (int c = 0; ok && c < nch; ++c) {
                const uint32_t ph = c & 1;
                // the value buffer of chunk c - 1 is free once tril(P_{c-1}) V has read it
                if (c > 0 && c + 1 < nch) {
                    if (!(ok = mbar_wait_abortable(bars + G_PV0 + ((c - 1) & 1), ((c - 1) >> 1) & 1, a.hdr, 116,
                                                   abort)))
                        break;
                    load_v(c + 1);
                }
                // Gamma_K of chunk c + 1 once P, the S update and the column sums have read chunk c's
                if (c + 1 < nch) {
                    if (!(ok = mbar_wait_abortable(bars + G_PQ, ph, a.hdr, 117, abort))) break;
                    if (!(ok = mbar_wait_abortable(bars + G_S, ph, a.hdr, 111, abort))) break;
                    if (!(ok = mbar_wait_abortable(bars + G_ZP, ph, a.hdr, 112, abort))) break;
                    load_g_tile(smem + L.gk, &gmap, bars + G_GT, a.kg, nb, tok0 + (c + 1) * C, bh);
                    last_gt = c + 1;
                }
                if (c + 2 < nch && !(ok = stage_queries(c + 2))) break;
            }
            // TMA loads still in flight (only after a timeout) complete before shared memory is
            // released
            if (last_v0 >= 0) mbar_wait(bars + G_V0, (last_v0 >> 1) & 1, a.hdr, 115);
            if (last_v1 >= 0) mbar_wait(bars + G_V1, (last_v1 >> 1) & 1, a.hdr, 115);
            if (last_xq >= 0) mbar_wait(bars + G_XQ, last_xq & 1, a.hdr, 115);
            if (last_gt >= 0) mbar_wait(bars + G_GT, last_gt & 1, a.hdr, 115);
        }
    } else if (warp < 8) {
        // ============================================================ query rows: mask side
        // (warps 0-3, upper component groups) and query side (warps 4-7, lower groups)
        const bool qs = warp >= 4;
        const int i = t & 127;
        const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int g0 = qs ? 0 : hq, g1 = qs ? hq : kc;
        uint8_t *abq = smem + L.abq;
        if (qs && nch > 0 && mbar_wait_abortable(bars + G_XQ, 0, a.hdr, 130, abort)) {
            build_inplace<DR>(abq, i);
            fence_proxy_async_smem();
            mbar_arrive(bars + G_AQ);
        }
        if (a.lse_q) grid_dependency_wait();   // (the rows' log2-sum-exp come from the kernels before)
        for (int c = 0; c < nch; ++c) {
            const uint32_t ph = c & 1;
            const bool valid = tok0 + c * C + i < tok_end;
            // (components in tiles: the row's log2-sum-exp over all components, read ahead; E_Q is
            // then the row's normalised responsibilities and needs no maximum)
            const float lse = (a.lse_q && valid) ? a.lse_q[(long long)bh * a.N + tok0 + c * C + i] : 0.f;
            // E_Q: the row maximum from both halves, then each half's exponentials
            if (!mbar_wait_abortable(bars + G_LQ, ph, a.hdr, 131, abort)) break;
            tc_fence_after();
            float m;
            if (a.lse_q) {
                m = valid ? lse : __int_as_float(0x7f800000);
            } else {
                const float mh = query_max_half(lane + R_LQ, a.K, g0, g1);
                xmax[(qs ? 0 : 2 * C) + ph * C + i] = mh;
                tc_fence_before();
                mbar_arrive(bars + G_XM);
                if (!mbar_spin_wait(bars + G_XM, ph, a.hdr, 134, abort)) break;
                tc_fence_after();
                m = valid ? fmaxf(mh, xmax[(qs ? 2 * C : 0) + ph * C + i]) : __int_as_float(0x7f800000);
            }
            // Z_{c-1} (published by the state side as soon as Gamma_K's column sums give it)
            if (!mbar_wait_abortable(bars + G_ZB0 + ph, (c >> 1) & 1, a.hdr, 132, abort)) break;
            // E_Q of this half, one group per wait: a row past the end of the sequence has
            // m = +inf, so all of its values are exp2(-inf) = 0; both halves have read all of
            // their logits before either writes (the maxima were exchanged in between)
            float2 part = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int gq = g0; gq < g1; ++gq) {
                uint32_t r[32];
                tmem_ld32(lane + R_LQ + 32 * gq, r);
                tmem_ld_wait();
                query_exp_group(lane + R_LQ, a.K, gq, hq, m, r, zbuf + ph * KMAX, part.x, part.y);
            }
            tmem_st_wait();
            if (qs) dsq[ph * C + i] = part;
            tc_fence_before();
            mbar_arrive(bars + G_GQ0 + ph);
            if (qs) {
                // the next chunk's queries, while P, the inter-chunk read and the mask run
                if (c + 1 < nch) {
                    if (!mbar_wait_abortable(bars + G_XQ, (c + 1) & 1, a.hdr, 133, abort)) break;
                    build_inplace<DR>(abq, i);
                    fence_proxy_async_smem();
                    mbar_arrive(bars + G_AQ);
                }
            } else {
                // causal mask of P; P (bf16 pairs) back into TMEM as the A operand of tril(P) V
                if (!mbar_wait_abortable(bars + G_P, ph, a.hdr, 120, abort)) break;
                if (!mbar_wait_abortable(bars + G_GQ0 + ph, (c >> 1) & 1, a.hdr, 121, abort)) break;   // dsq
                tc_fence_after();
                const float intra = mask_row(lane + R_P, i);
                const float2 q = dsq[ph * C + i];
                dsm[ph * C + i] = make_float2(q.x + part.x, q.y + part.y + intra);
                tc_fence_before();
                mbar_arrive(bars + G_PS0 + ph);
            }
        }
    } else {
        // ============================================================ state and output side
        // t - 256: the TMEM lane, which is value column n of S^T and token row of the output; also
        // component k of the running normaliser Z
        const int k = t - 256, n = t - 256;
        const uint32_t lane = tmem + ((uint32_t)((warp - 8) * 32) << 16);
        // starting memory: S_start^T to TMEM and as bf16 rows of the operand tile (column n of the
        // segment's memory, read component by component: consecutive lanes, consecutive floats)
        grid_dependency_wait();   // the segment's starting memory comes from the scan
        const float *seg_mem = a.agg + ((size_t)bh * a.nseg + seg) * KMAX * a.ne;
        const bool vrow = n < d_v;
#pragma unroll 1
        for (int b = 0; b < KMAX / 16; ++b) {
            uint32_t r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = vrow ? __float_as_uint(seg_mem[(size_t)(16 * b + j) * a.ne + n]) : 0u;
            tmem_st16(lane + R_S + 16 * b, r);
            if (vrow) {
                *reinterpret_cast<uint4 *>(smem + L.gk + sw128(C + n, 2 * b, nb)) =
                    make_uint4(pk2(r[0], r[1], 1.f), pk2(r[2], r[3], 1.f), pk2(r[4], r[5], 1.f), pk2(r[6], r[7], 1.f));
                *reinterpret_cast<uint4 *>(smem + L.gk + sw128(C + n, 2 * b + 1, nb)) = make_uint4(
                    pk2(r[8], r[9], 1.f), pk2(r[10], r[11], 1.f), pk2(r[12], r[13], 1.f), pk2(r[14], r[15], 1.f));
            }
        }
        const float *src = seg_mem + (size_t)k * a.ne;
        float zrun = src[d_v];
        zbuf[k] = zrun;
        mbar_arrive(bars + G_ZB0);   // Z_start, for chunk 0's normalisers
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bars + G_SP);   // phase 0: S_start ready
        // output of chunk cc (numerator complete, normaliser from the mask side)
        auto output = [&](int cc) -> bool {
            const uint32_t pc = cc & 1;
            if (!mbar_wait_abortable(bars + G_PS0 + pc, (cc >> 1) & 1, a.hdr, 140, abort)) return false;
            if (!mbar_wait_abortable(bars + G_PV0 + pc, (cc >> 1) & 1, a.hdr, 141, abort)) return false;
            tc_fence_after();
            const float2 sd = dsm[pc * C + k];
            const int row = tok0 + cc * C + k;
            if (a.pmode)
                tile_partial_row(lane + R_O, d_v, sd.y + a.eps * sd.x, row < tok_end, a.part, a.pden,
                                 (long long)bh * a.N + row, a.pmode);
            else
                out_row(lane + R_O, d_v, 1.0f / (sd.y + a.eps * sd.x), row < tok_end, a.O, (long long)bh * a.N + row,
                        a.out_f32);
            tc_fence_before();
            mbar_arrive(bars + G_OF);
            return true;
        };
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const uint32_t ph = c & 1;
            if (c > 0 && !(ok = output(c - 1))) break;
            // Z_c = Z_{c-1} + column sums of Gamma_K
            if (!(ok = mbar_wait_abortable(bars + G_GT, ph, a.hdr, 142, abort))) break;
            float *zp = zpart + ph * 8 * KMAX;
            colsum_rows(smem + L.gk, nb, zp, k);
            mbar_arrive(bars + G_ZP);
            if (!(ok = mbar_wait_abortable(bars + G_ZP, ph, a.hdr, 143, abort))) break;
            {
                float zs = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) zs += zp[g * KMAX + k];
                zrun += zs;
            }
            // Z_c for chunk c + 1's normalisers.  Its buffer last held Z_{c-2}, which chunk c - 1
            // read before its mask side finished (output(c - 1) above waited for that); the pair
            // of barriers by parity keeps a waiter from seeing a phase two ahead.
            zbuf[((c + 1) & 1) * KMAX + k] = zrun;
            mbar_arrive(bars + G_ZB0 + ((c + 1) & 1));
            // readout of S_c^T (after the update, and after the read of S_{c-1} that it overwrites)
            if (!(ok = mbar_wait_abortable(bars + G_S, ph, a.hdr, 144, abort))) break;
            if (!(ok = mbar_wait_abortable(bars + G_PQ, ph, a.hdr, 145, abort))) break;
            tc_fence_after();
            state_rows_t(lane + R_S, smem + L.gk, nb, n, vrow);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bars + G_SP);
        }
        if (ok && nch > 0) output(nch - 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 12) tmem_dealloc(tmem, 512);
}

// Shared memory the kernel needs (0 if the shape does not fit).
uint32_t causal_gamma_smem(int d_r, int kn16, int d_v)
{
    const uint32_t need = GSmem(d_r, kn16, d_v).total + 1024;
    return need <= 227u * 1024u ? smem_for(need, 512) : 0;
}

template <int DR>
gma_status_t launch_causal_gamma(const Args &a, const CUtensorMap &vmap, const CUtensorMap &qmap,
                                 const CUtensorMap &gmap, int nblocks, cudaStream_t st)
{
    const uint32_t sm = causal_gamma_smem(DR, a.kn16, a.d_v);
    if (sm == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (!set_smem(tc_causal_gamma_kernel<DR>, sm)) return GMA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_CAUSAL_OUT, st,
               (e = launch_pdl(tc_causal_gamma_kernel<DR>, dim3(nblocks), dim3(GTHREADS), sm, st, a, vmap, qmap, gmap)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template gma_status_t launch_causal_gamma<16>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_causal_gamma<32>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_causal_gamma<64>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, int, cudaStream_t);

}  // namespace tck
}  // namespace gma
