// gma_tc_lse.cu -- log-sum-exp of every routing row's logits over more than 128 components
// (tcgen05, sm_103a).
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §1: gamma_k = p(z = k | x) = exp(L_k) / sum_j exp(L_j), L_k = log pi_k N(x; mu_k,
// sigma_k^2).  With more than 128 components the logits of one row no longer fit one tensor-memory
// tile next to everything else a pass keeps there, so the passes take gamma tile by tile as
// exp2(L_k - lse), where lse = log2 sum_j exp2(L_j) over all components is computed here first
// (the table holds log2e-scaled logits, so everything is in the log2 domain).
//
// Both kernels work through the list of 128-row chunks of two row sets (the queries and the keys
// of a causal call), each CTA a contiguous share of it, so that consecutive chunks mostly share a
// head.  Two threads share each row, each with a share of the row's columns: each keeps a running
// maximum and sum, updated once per 64 of its columns (their maximum over eight independent
// chains, then their exponentials summed over four), and the two merge at the end of the chunk.
//
// Two tiles (129 to 256 components): tc_lse_resident_kernel, one CTA per SM, keeps a head's table
// in shared memory as one N = 256 operand and runs a pipeline over its chunks:
//   control warp:  one lane issues each chunk's logits (one MMA chain for both tiles) into one of
//                  two 256-column TMEM regions, as soon as the region is free and the chunk's
//                  [x^2, x] tile is built, and loads the table when the head changes;
//   reader warps:  eight: each loads its tile's 128 logits of a chunk, 64 at a time, frees the
//                  region, and updates its row's state; the lower half also builds the next
//                  chunk's [x^2, x] tile (two buffers) from rows loaded a chunk ahead, and merges
//                  the upper half's state at the end of each chunk.
// More tiles: tc_lse_stream_kernel, two CTAs per SM, streams the table images a pair of tiles at a
// time through one buffer, in the same N = 256 layout: per chunk, [x^2, x] is built once; per
// pair, one MMA chain fills the CTA's 256 TMEM columns, and the next pair's images load while the
// rows read them.  Two CTAs per SM overlap one another's waits (measured at 1024 components:
// 347 us, against 384 us streaming single tiles through two buffers, and 621 us for a pipelined
// CTA per SM streaming single tiles through four).
// Every wait is bounded, and a timeout stops all roles.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

// ------------------------------------------------------------------ streamed tables, in pairs
constexpr int STHREADS = 256;   // two threads per row of a 128-row chunk
constexpr int STREAM_CTAS = 2 * 152;   // two CTAs per GB300 SM (shared memory and 256 TMEM columns each)
enum SBar { S_TB, S_MMA, S_NBAR };

struct StreamSmem {
    uint32_t tab, abuf, ax, xch, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ StreamSmem(int DR, int bimg_bytes)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        uint32_t o = 0;
        tab = o; o = al(o + 2u * (uint32_t)bimg_bytes);   // a pair of tiles as one N = 256 operand
        abuf = o; o = al(o + ka / 64u * 128u * (uint32_t)C);
        ax = o; o = al(o + (uint32_t)C * 32u);
        xch = o; o += (uint32_t)C * 16u;   // the upper half's (max, sum, best logit, argmax) per row
        bars = o; o += S_NBAR * 8u;
        misc = o; o += 16u;
        total = o;
    }
};

// ------------------------------------------------------------------ resident tables, pipelined
constexpr int RTHREADS = 288;   // eight reader warps (two threads per row of a chunk), one control warp
constexpr int RESIDENT_CTAS = 152;   // one CTA per GB300 SM: two 256-column logits regions fill the TMEM
constexpr int NREG = 2;         // TMEM regions in the ring (one chunk's 256 logits each)
// TB: the table is loaded (transaction bytes); FULL: a region's logits are complete (MMA commit);
// FREE: every reader warp has loaded a region (8 arrivals); A: a chunk's [x^2, x] tile is built
// (4: the lower half's warps); XF / XE: the upper half's row states are in the exchange slot of a
// chunk parity / the lower half has read them (4 each); FIN: every MMA issued is done
enum LBar { L_TB, L_FIN, L_FULL0, L_FREE0 = L_FULL0 + NREG, L_A0 = L_FREE0 + NREG, L_A1, L_XF0, L_XF1, L_XE0, L_XE1,
            L_NBAR };

// The two tiles of a head's table as one N = 256 operand: each 64-column block of the [x^2, x]
// part holds tile 0's 128 rows, then tile 1's (so that one MMA chain covers both), and the constant
// part holds both tiles' rows in order.
struct ResidentSmem {
    uint32_t tab, ab0, ab1, ax, xch, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ ResidentSmem(int DR, int bimg_bytes)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        uint32_t o = 0;
        tab = o; o = al(o + 2u * (uint32_t)bimg_bytes);
        ab0 = o; o = al(o + ka / 64u * 128u * (uint32_t)C);   // [x^2, x] of even chunks
        ab1 = o; o = al(o + ka / 64u * 128u * (uint32_t)C);   // and of odd ones
        ax = o; o = al(o + (uint32_t)C * 32u);
        xch = o; o += 2u * (uint32_t)C * 16u;   // the upper half's (max, sum, best logit, argmax) per row, by chunk parity
        bars = o; o += L_NBAR * 8u;
        misc = o; o += 16u;
        total = o;
    }
};

// One thread's share of a tile: nv valid logits in ra then rb (NV: all 64 at compile time, or 0
// for a count known only at run time) update the running maximum m and sum s of exp2(L - m), and
// with want_arg the first column (index col0 + q) of largest logit.
template <int NV>
__device__ __forceinline__ void tile_update(const uint32_t (&ra)[32], const uint32_t (&rb)[32], int nv, float &m,
                                            float &s, float &best, int &arg, int col0, bool want_arg)
{
    auto val = [&](int q) { return __uint_as_float(q < 32 ? ra[q] : rb[q - 32]); };
    auto in = [&](int q) { return NV == 64 || q < nv; };
    float mx[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mx[u] = NEG_BIG;
#pragma unroll
    for (int q = 0; q < 64; ++q)
        if (in(q)) mx[q & 7] = fmaxf(mx[q & 7], val(q));
    const float tm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
    if (want_arg) {
#pragma unroll
        for (int q = 0; q < 64; ++q)
            if (in(q) && val(q) > best) {
                best = val(q);
                arg = col0 + q;
            }
    }
    const float mn = fmaxf(m, tm);
    float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 64; ++q)
        if (in(q)) sa[q & 3] += ex2(val(q) - mn);
    s = s * ex2(m - mn) + ((sa[0] + sa[1]) + (sa[2] + sa[3]));
    m = mn;
}

// The chunk list: every 128-row chunk of every slice of the first row set, then of the second.
struct ChunkInfo {
    const bf16 *X;
    float *out;
    int bh, tok0, n;   // slice, first row, rows per slice
};
struct ChunkList {
    const bf16 *rows0, *rows1;
    float *lse0, *lse1;
    long long side_chunks;   // chunks of the first set
    int cpn0, cpn1, N0, N1;  // chunks per slice and rows per slice of each set
    __device__ __forceinline__ ChunkInfo at(long long c) const
    {
        const bool side = c >= side_chunks;
        const long long cc = side ? c - side_chunks : c;
        const int cpn = side ? cpn1 : cpn0;
        return ChunkInfo{side ? rows1 : rows0, side ? lse1 : lse0, (int)(cc / cpn), (int)(cc % cpn) * C, side ? N1 : N0};
    }
};

// Row rt of chunk c's routing rows into x (zeros past the end of its slice).
template <int DR>
__device__ __forceinline__ void fetch_row(const ChunkList &cl, long long c, int rt, uint4 (&x)[DR / 8])
{
    const ChunkInfo ci = cl.at(c);
    load_x<DR>(ci.X, (long long)ci.bh * ci.n + ci.tok0 + rt, ci.tok0 + rt < ci.n, x);
}

// Tiles 2 j and 2 j + 1 (the second if there is one) of a head's table images (img) into tab as one
// N = 256 operand: each 64-column block of the [x^2, x] part holds the first tile's 128 rows, then
// the second's; the constant part holds both tiles' rows in order.  One thread; the bytes complete
// on bar.
__device__ __forceinline__ void load_table_pair(uint8_t *tab, const uint8_t *img, int bimg_bytes, int main_bytes,
                                                int ntile, int j, uint64_t *bar)
{
    constexpr int BLK = 128 * 128;   // one tile's 64-column block: 128 rows of 128 bytes
    const int nt = ntile - 2 * j < 2 ? ntile - 2 * j : 2;
    mbar_arrive_expect_tx(bar, (uint32_t)(nt * bimg_bytes));
    for (int t2 = 0; t2 < nt; ++t2) {
        const uint8_t *src = img + (size_t)(2 * j + t2) * bimg_bytes;
        for (int q = 0; q < main_bytes / BLK; ++q)
            bulk_g2s(tab + q * 2 * BLK + t2 * BLK, src + (size_t)q * BLK, (uint32_t)BLK, bar);
        bulk_g2s(tab + 2 * main_bytes + t2 * 128 * 32, src + main_bytes, 128u * 32u, bar);
    }
}

}  // namespace

// rows0 / rows1: the row sets (B*H slices of a.N and N1 rows of d_r bf16 each; rows1 may be null),
// lse0 / lse1 their outputs; the chunk list is every 128-row chunk of every slice of rows0, then
// of rows1.  With
// assign non-null (usage diagnostics of rows0) each row's argmax over all components (the lowest
// index on ties) is written there and counted into counts [H][K_all].
template <int DR>
__global__ void __launch_bounds__(STHREADS, 2) tc_lse_stream_kernel(const Args a, const bf16 *rows0, const bf16 *rows1,
                                                                    float *lse0, float *lse1, int K_all, int BH,
                                                                    int N1, int *assign, int *counts)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const StreamSmem L(DR, a.bimg_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.misc);
    volatile int *stop = reinterpret_cast<volatile int *>(smem + L.misc + 4);
    const int t = threadIdx.x, warp = t >> 5;
    const int rt = t & (C - 1), half = t >> 7;   // this thread's row of the chunk, and its tile of each pair
    const int ntile = (K_all + KMAX - 1) / KMAX, npair = (ntile + 1) / 2;
    const int cpn0 = (a.N + C - 1) / C, cpn1 = (N1 + C - 1) / C;   // chunks per slice of each set
    const long long side_chunks = (long long)BH * cpn0;
    if (t == 0) {
        for (int i = 0; i < S_NBAR; ++i) mbar_init(bars + i, 1);
        *stop = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    if (half == 0) {   // constant A operand of the logits: (1, 1, 0, ...) in every row, K-major SW32
        const uint32_t one2 = 0x3C003C00u;   // fp16 pair (1, 1)
        const int flip = (t >> 2) & 1;
        *reinterpret_cast<uint4 *>(smem + L.ax + t * 32 + (flip << 4)) = make_uint4(one2, 0, 0, 0);
        *reinterpret_cast<uint4 *>(smem + L.ax + t * 32 + ((flip ^ 1) << 4)) = make_uint4(0, 0, 0, 0);
    }
    // each CTA takes a contiguous range of the chunk list
    const int nsets = rows1 ? 2 : 1;
    const long long total = side_chunks + (nsets > 1 ? (long long)BH * cpn1 : 0ll);
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    const long long c_begin = (long long)blockIdx.x * per, c_end = min(total, c_begin + per);
    const int nloc = c_end > c_begin ? (int)(c_end - c_begin) : 0;
    const ChunkList cl{rows0, rows1, lse0, lse1, side_chunks, cpn0, cpn1, a.N, N1};
    uint4 x[DR / 8];   // lower half: this chunk's routing row, loaded during the chunk before
    if (half == 0 && nloc > 0) fetch_row<DR>(cl, c_begin, rt, x);
    grid_dependency_wait();   // the tables come from the parameter kernel
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);
    const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int main_bytes = a.bimg_main_bytes;
    // thread 0: the pair in the table buffer, and its load
    int res_h = -1, res_j = -1;
    bool pend = false;
    uint32_t ph_tb = 0;
    if (t == 0 && nloc > 0) {
        res_h = cl.at(c_begin).bh % a.H;
        res_j = 0;
        load_table_pair(smem + L.tab, a.bimg + (size_t)res_h * a.bimg_head, a.bimg_bytes, main_bytes, ntile, 0,
                        bars + S_TB);
        pend = true;
    }
    uint32_t ph_mma = 0;
    for (int lc = 0; lc < nloc; ++lc) {
        const ChunkInfo ci = cl.at(c_begin + lc);
        const int bh = ci.bh, nrow = ci.n, h = bh % a.H;
        const int row = ci.tok0 + rt;
        const bool valid = row < nrow;
        if (half == 0) build_a<DR>(smem + L.abuf, rt, x);   // (the MMAs of the chunk before are done)
        fence_proxy_async_smem();
        if (half == 0 && lc + 1 < nloc)   // the next chunk's row, in flight while this one is computed
            fetch_row<DR>(cl, c_begin + lc + 1, rt, x);
        tc_fence_before();
        __syncthreads();   // [x^2, x] built; the logits region read by every row
        tc_fence_after();
        float m = NEG_BIG, s = 0.f, best = NEG_BIG;
        int arg = 0;
        bool ok = true;
        for (int j = 0; j < npair; ++j) {
            if (t == 0) {   // this pair's logits, once its table is in
                if (pend) {
                    if (!mbar_wait(bars + S_TB, ph_tb, a.hdr, 60)) *stop = 1;
                    ph_tb ^= 1u;
                    pend = false;
                }
                if (!*stop) {
                    tc_fence_after();
                    issue_logits_c<DR>(tmem, sb + L.abuf, sb + L.tab, sb + L.tab + 2u * (uint32_t)main_bytes, sb + L.ax,
                                       2 * KMAX);
                    mma_commit(bars + S_MMA);
                }
            }
            __syncthreads();   // (thread 0's stop is seen by every thread)
            ok = !*stop && mbar_wait(bars + S_MMA, ph_mma, a.hdr, 61);
            ph_mma ^= 1u;
            if (__syncthreads_or(!ok)) break;
            tc_fence_after();
            if (t == 0) {   // the next step's pair, while the rows read this one (its MMA is done)
                const bool last = j + 1 == npair;
                if (!last || lc + 1 < nloc) {
                    const int hn = last ? cl.at(c_begin + lc + 1).bh % a.H : h, jn = last ? 0 : j + 1;
                    if (hn != res_h || jn != res_j) {
                        load_table_pair(smem + L.tab, a.bimg + (size_t)hn * a.bimg_head, a.bimg_bytes, main_bytes, ntile,
                                        jn, bars + S_TB);
                        pend = true;
                        res_h = hn;
                        res_j = jn;
                    }
                }
            }
            // this thread's tile of the pair (128 columns), 64 at a time
            const int kv = min(KMAX, K_all - KMAX * (2 * j + half));
            if (kv > 0) {
                for (int sub = 0; sub < 2; ++sub) {
                    uint32_t ra[32], rb[32];
                    const uint32_t col = 128u * half + 64u * sub;
                    tmem_ld32(lane + col, ra);   // (warp-uniform: every lane loads)
                    tmem_ld32(lane + col + 32u, rb);
                    tmem_ld_wait();
                    const int nv = min(64, max(0, kv - 64 * sub));
                    if (nv > 0) {
                        const int col0 = KMAX * (2 * j + half) + 64 * sub;
                        if (nv == 64)
                            tile_update<64>(ra, rb, 64, m, s, best, arg, col0, assign != nullptr);
                        else
                            tile_update<0>(ra, rb, nv, m, s, best, arg, col0, assign != nullptr);
                    }
                }
            }
            tc_fence_before();
            __syncthreads();   // the region read by every row before the next MMA writes it
            tc_fence_after();
        }
        if (!ok) break;
        // the upper half hands its row's state to the lower half (read before the lower half
        // reaches the next chunk's first barrier, so one slot per row suffices)
        float4 *xch = reinterpret_cast<float4 *>(smem + L.xch);
        if (half) xch[rt] = make_float4(m, s, best, __int_as_float(arg));
        __syncthreads();
        if (!half && valid) {
            const float4 o = xch[rt];
            const float mm = fmaxf(m, o.x);
            const float ss = s * ex2(m - mm) + o.y * ex2(o.x - mm);
            ci.out[(long long)bh * nrow + row] = mm + log2f(ss);
            if (assign) {   // the larger logit; on a tie the lower component index
                const int oarg = __float_as_int(o.w);
                if (o.z > best || (o.z == best && oarg < arg)) arg = oarg;
                assign[(long long)bh * nrow + row] = arg;
                atomicAdd(counts + (size_t)h * K_all + arg, 1);
            }
        }
    }
    // a table load still in flight (only after a stop, or prefetched past the last chunk: never)
    // completes before shared memory is released; every MMA issued has been waited for
    if (t == 0 && pend) mbar_wait(bars + S_TB, ph_tb, a.hdr, 62);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

template <int DR>
__global__ void __launch_bounds__(RTHREADS, 1) tc_lse_resident_kernel(const Args a, const bf16 *rows0, const bf16 *rows1,
                                                             float *lse0, float *lse1, int K_all, int BH,
                                                             int N1, int *assign, int *counts)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const ResidentSmem L(DR, a.bimg_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.misc);
    volatile int *stop = reinterpret_cast<volatile int *>(smem + L.misc + 4);
    const int t = threadIdx.x, warp = t >> 5, lid = t & 31;
    const int rt = t & (C - 1), half = (t >> 7) & 1;   // a reader's row of the chunk, and its half of the columns
    const int cpn0 = (a.N + C - 1) / C, cpn1 = (N1 + C - 1) / C;   // chunks per slice of each set
    const long long side_chunks = (long long)BH * cpn0;
    if (t == 0) {
        for (int i = 0; i < L_NBAR; ++i) {
            const uint32_t n = (i >= L_FREE0 && i < L_FREE0 + NREG) ? 8u : (i >= L_A0) ? 4u : 1u;
            mbar_init(bars + i, n);
        }
        *stop = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    if (t < C) {   // constant A operand of the logits: (1, 1, 0, ...) in every row, K-major SW32
        const uint32_t one2 = 0x3C003C00u;   // fp16 pair (1, 1)
        const int flip = (t >> 2) & 1;
        *reinterpret_cast<uint4 *>(smem + L.ax + t * 32 + (flip << 4)) = make_uint4(one2, 0, 0, 0);
        *reinterpret_cast<uint4 *>(smem + L.ax + t * 32 + ((flip ^ 1) << 4)) = make_uint4(0, 0, 0, 0);
    }
    // each CTA takes a contiguous range of the chunk list, so that consecutive chunks mostly share
    // a head: with two tiles, both table images then stay in shared memory from chunk to chunk
    const int nsets = rows1 ? 2 : 1;
    const long long total = side_chunks + (nsets > 1 ? (long long)BH * cpn1 : 0ll);
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    const long long c_begin = (long long)blockIdx.x * per, c_end = min(total, c_begin + per);
    const int nloc = c_end > c_begin ? (int)(c_end - c_begin) : 0;
    const ChunkList cl{rows0, rows1, lse0, lse1, side_chunks, cpn0, cpn1, a.N, N1};
    uint4 x[DR / 8];   // lower half: the row of the chunk whose [x^2, x] tile is built next
    if (warp < 4 && nloc > 0) fetch_row<DR>(cl, c_begin, rt, x);   // (the rows are inputs: no kernel before writes them)
    grid_dependency_wait();   // the tables come from the parameter kernel
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);
    const int main_bytes = a.bimg_main_bytes;

    if (warp == 8) {
        // ============================================================ control warp: MMAs, table
        if (lid == 0) {
            int res_h = -1;               // head whose table is in shared memory
            bool pend = false;            // its load not waited for yet
            uint32_t ph_tb = 0;
            bool ok = true, issued = false;
            // the table of chunk lc's head, unless it is there already (after the MMA of the chunk
            // before, the last to read the old one)
            auto load_table = [&](int lc) -> bool {
                const int h = cl.at(c_begin + lc).bh % a.H;
                if (h == res_h) return true;
                if (lc > 0 && !mbar_wait_abortable(bars + L_FULL0 + ((lc - 1) & 1), (uint32_t)(((lc - 1) >> 1) & 1),
                                                   a.hdr, 63, stop))
                    return false;
                load_table_pair(smem + L.tab, a.bimg + (size_t)h * a.bimg_head, a.bimg_bytes, main_bytes, 2, 0,
                                bars + L_TB);
                pend = true;
                res_h = h;
                return true;
            };
            for (int lc = 0; ok && lc < nloc; ++lc) {
                const int r = lc & 1;
                if (!(ok = load_table(lc))) break;
                if (pend) {
                    if (!(ok = mbar_wait_abortable(bars + L_TB, ph_tb, a.hdr, 60, stop))) break;
                    ph_tb ^= 1u;
                    pend = false;
                }
                if (!(ok = mbar_wait_abortable(bars + L_A0 + r, (uint32_t)((lc >> 1) & 1), a.hdr, 64, stop))) break;
                if (lc >= NREG &&
                    !(ok = mbar_wait_abortable(bars + L_FREE0 + r, (uint32_t)(((lc >> 1) - 1) & 1), a.hdr, 65, stop)))
                    break;
                tc_fence_after();
                issue_logits_c<DR>(tmem + 256u * r, sb + (r ? L.ab1 : L.ab0), sb + L.tab, sb + L.tab + 2u * (uint32_t)main_bytes,
                                   sb + L.ax, 2 * KMAX);
                mma_commit(bars + L_FULL0 + r);
                issued = true;
            }
            // the table load still in flight (only after a stop) completes before shared memory is
            // released, and every MMA issued before the tensor memory is
            if (pend) mbar_wait(bars + L_TB, ph_tb, a.hdr, 62);
            if (issued) {
                mma_commit(bars + L_FIN);
                mbar_wait(bars + L_FIN, 0, a.hdr, 68);
            }
        }
    } else {
        // ============================================================ readers
        const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        float4 *xch = reinterpret_cast<float4 *>(smem + L.xch);
        bool ok = true;
        if (half == 0 && nloc > 0) {   // the first chunk's [x^2, x] tile, and the next chunk's rows in flight
            build_a<DR>(smem + L.ab0, rt, x);
            fence_proxy_async_smem();
            __syncwarp();
            if (lid == 0) mbar_arrive(bars + L_A0);
            if (nloc > 1) fetch_row<DR>(cl, c_begin + 1, rt, x);
        }
        for (int lc = 0; ok && lc < nloc; ++lc) {
            const ChunkInfo ci = cl.at(c_begin + lc);
            const int bh = ci.bh, tok0 = ci.tok0, nrow = ci.n;
            float *out = ci.out;
            const int h = bh % a.H;
            const int row = tok0 + rt;
            const bool valid = row < nrow;
            const int r = lc & 1;
            if (half == 0 && lc + 1 < nloc) {
                // the next chunk's tile: its buffer was last read by the MMAs of chunk lc - 1, which
                // this thread has seen complete
                build_a<DR>(smem + (((lc + 1) & 1) ? L.ab1 : L.ab0), rt, x);
                fence_proxy_async_smem();
                __syncwarp();
                if (lid == 0) mbar_arrive(bars + L_A0 + ((lc + 1) & 1));
                if (lc + 2 < nloc) fetch_row<DR>(cl, c_begin + lc + 2, rt, x);
            }
            float m = NEG_BIG, s = 0.f, best = NEG_BIG;
            int arg = 0;
            if (!(ok = mbar_wait_abortable(bars + L_FULL0 + r, (uint32_t)((lc >> 1) & 1), a.hdr, 61, stop))) break;
            tc_fence_after();
            // this half's tile (128 columns of the region), 64 at a time; the region is freed once
            // both loads are in registers
            const int kv = min(KMAX, K_all - KMAX * half);   // valid components of the tile
            for (int sub = 0; sub < 2; ++sub) {
                uint32_t ra[32], rb[32];
                const uint32_t col = 256u * r + 128u * half + 64u * sub;
                tmem_ld32(lane + col, ra);
                tmem_ld32(lane + col + 32u, rb);
                tmem_ld_wait();
                if (sub == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lid == 0) mbar_arrive(bars + L_FREE0 + r);
                }
                const int nv = min(64, max(0, kv - 64 * sub));
                if (nv > 0) {
                    const int col0 = KMAX * half + 64 * sub;
                    if (nv == 64)
                        tile_update<64>(ra, rb, 64, m, s, best, arg, col0, assign != nullptr);
                    else
                        tile_update<0>(ra, rb, nv, m, s, best, arg, col0, assign != nullptr);
                }
            }
            // the upper half hands its row's state to the lower half through the slot of this
            // chunk's parity (free once the lower half has read it two chunks ago)
            const int p = lc & 1;
            if (half) {
                if (lc >= 2 && !(ok = mbar_wait_abortable(bars + L_XE0 + p, (uint32_t)(((lc >> 1) - 1) & 1), a.hdr, 66, stop)))
                    break;
                xch[p * C + rt] = make_float4(m, s, best, __int_as_float(arg));
                __syncwarp();
                if (lid == 0) mbar_arrive(bars + L_XF0 + p);
            } else {
                if (!(ok = mbar_wait_abortable(bars + L_XF0 + p, (uint32_t)((lc >> 1) & 1), a.hdr, 67, stop))) break;
                const float4 o = xch[p * C + rt];
                __syncwarp();
                if (lid == 0) mbar_arrive(bars + L_XE0 + p);
                if (valid) {
                    const float mm = fmaxf(m, o.x);
                    const float ss = s * ex2(m - mm) + o.y * ex2(o.x - mm);
                    out[(long long)bh * nrow + row] = mm + log2f(ss);
                    if (assign) {   // the larger logit; on a tie the lower component index
                        const int oarg = __float_as_int(o.w);
                        if (o.z > best || (o.z == best && oarg < arg)) arg = oarg;
                        assign[(long long)bh * nrow + row] = arg;
                        atomicAdd(counts + (size_t)h * K_all + arg, 1);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}


// Dynamic shared memory of each kernel (0 if it does not fit); the resident kernel's forces one
// CTA per SM (it allocates all 512 TMEM columns).
uint32_t lse_stream_smem(int d_r, int bimg_bytes)
{
    const uint32_t need = StreamSmem(d_r, bimg_bytes).total + 1024;
    return need <= 227u * 1024u ? smem_for(need, 256) : 0;
}

uint32_t lse_resident_smem(int d_r, int bimg_bytes)
{
    const uint32_t need = ResidentSmem(d_r, bimg_bytes).total + 1024;
    return need <= 227u * 1024u ? smem_for(need, 512) : 0;
}

template <int DR>
gma_status_t launch_lse(const Args &a, const bf16 *rows0, const bf16 *rows1, float *lse0, float *lse1, int K_all,
                        int BH, cudaStream_t st, int *assign, int *counts, int N1)
{
    if (N1 < 0) N1 = a.N;
    const long long chunks = (long long)BH * ((a.N + C - 1) / C) + (rows1 ? (long long)BH * ((N1 + C - 1) / C) : 0ll);
    const bool resident = (K_all + KMAX - 1) / KMAX == 2;
    const uint32_t sm = resident ? lse_resident_smem(DR, a.bimg_bytes) : lse_stream_smem(DR, a.bimg_bytes);
    if (sm == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    cudaError_t e = cudaSuccess;
    if (resident) {
        if (!set_smem(tc_lse_resident_kernel<DR>, sm)) return GMA_ERR_CUDA;
        const int grid = (int)(chunks < RESIDENT_CTAS ? chunks : RESIDENT_CTAS);
        GMA_LAUNCH(KID_TC_LSE, st,
                   (e = launch_pdl(tc_lse_resident_kernel<DR>, dim3(grid), dim3(RTHREADS), sm, st, a, rows0, rows1, lse0,
                                   lse1, K_all, BH, N1, assign, counts)));
    } else {
        if (!set_smem(tc_lse_stream_kernel<DR>, sm)) return GMA_ERR_CUDA;
        const int grid = (int)(chunks < STREAM_CTAS ? chunks : STREAM_CTAS);
        GMA_LAUNCH(KID_TC_LSE, st,
                   (e = launch_pdl(tc_lse_stream_kernel<DR>, dim3(grid), dim3(STHREADS), sm, st, a, rows0, rows1, lse0,
                                   lse1, K_all, BH, N1, assign, counts)));
    }
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template gma_status_t launch_lse<16>(const Args &, const bf16 *, const bf16 *, float *, float *, int, int, cudaStream_t,
                                     int *, int *, int);
template gma_status_t launch_lse<32>(const Args &, const bf16 *, const bf16 *, float *, float *, int, int, cudaStream_t,
                                     int *, int *, int);
template gma_status_t launch_lse<64>(const Args &, const bf16 *, const bf16 *, float *, float *, int, int, cudaStream_t,
                                     int *, int *, int);

}  // namespace tck
}  // namespace gma
