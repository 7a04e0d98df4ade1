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
// More tiles: tc_lse_stream_kernel, two CTAs per SM, streams the table images through two
// buffers, tile by tile; per chunk, [x^2, x] is built once, each tile's logits go into one of two
// TMEM regions, and the next tile's MMA is issued before the rows read the current one.  With
// eight tiles per chunk its two CTAs per SM keep more loads and MMAs in flight than a pipelined
// CTA streaming its tables through four buffers (measured at 1024 components: 384 us against
// 621 us; at 256 components the resident pipeline takes 103 us, this kernel 170 us).
// Every wait is bounded, and a timeout stops all roles.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

// ------------------------------------------------------------------ streamed tables
constexpr int STHREADS = 256;   // two threads per row of a 128-row chunk
constexpr int STREAM_CTAS = 2 * 152;   // two CTAs per GB300 SM (shared memory and 256 TMEM columns each)
enum SBar { S_TB0, S_TB1, S_MMA0, S_MMA1, S_NBAR };

struct StreamSmem {
    uint32_t tb0, tb1, abuf, ax, xch, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ StreamSmem(int DR, int bimg_bytes)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        uint32_t o = 0;
        tb0 = o; o = al(o + (uint32_t)bimg_bytes);
        tb1 = o; o = al(o + (uint32_t)bimg_bytes);
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
    const int rt = t & (C - 1), half = t >> 7;   // this thread's row of the chunk, and its half of the columns
    const int ntile = (K_all + KMAX - 1) / KMAX;
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
    grid_dependency_wait();   // the tables come from the parameter kernel
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);
    const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    // phases and pending loads of the two buffers, one bit each (ph_tb, pending: thread 0 alone)
    uint32_t ph_tb = 0, ph_mma = 0, pending = 0;
    const int main_bytes = a.bimg_main_bytes;

    // each CTA takes a contiguous range of the chunk list, so that consecutive chunks mostly share
    // a head: with two tiles, both table images then stay in shared memory from chunk to chunk
    const int nsets = rows1 ? 2 : 1;
    const long long total = side_chunks + (nsets > 1 ? (long long)BH * cpn1 : 0ll);
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    const long long c_begin = (long long)blockIdx.x * per, c_end = min(total, c_begin + per);
    // the chunk list: chunk c's slice, first token, rows per slice, rows and output
    auto chunk_at = [&](long long c, int &bh, int &tok0, int &n, const bf16 *&X, float *&out) {
        const int side = c >= side_chunks;
        const long long cc = side ? c - side_chunks : c;
        const int cpn = side ? cpn1 : cpn0;
        bh = (int)(cc / cpn);
        tok0 = (int)(cc % cpn) * C;
        n = side ? N1 : a.N;
        X = side ? rows1 : rows0;
        out = side ? lse1 : lse0;
    };
    int resident_h = -1;   // thread 0: the head whose two table images are in the buffers
    uint4 x[DR / 8];       // this chunk's routing row, loaded during the chunk before (lower half)
    if (c_begin < c_end && half == 0) {
        int bh0, tk0, n0;
        const bf16 *X0;
        float *o0;
        chunk_at(c_begin, bh0, tk0, n0, X0, o0);
        load_x<DR>(X0, (long long)bh0 * n0 + tk0 + rt, tk0 + rt < n0, x);
    }
    for (long long c = c_begin; c < c_end; ++c) {
        int bh, tok0, nrow;
        const bf16 *X;
        float *out;
        chunk_at(c, bh, tok0, nrow, X, out);
        const int h = bh % a.H;
        const int row = tok0 + rt;
        const bool valid = row < nrow;
        const uint8_t *img = a.bimg + (size_t)h * a.bimg_head;
        if (half == 0) build_a<DR>(smem + L.abuf, rt, x);
        fence_proxy_async_smem();
        if (c + 1 < c_end && half == 0) {   // the next chunk's row, in flight while this one is computed
            int bh1, tk1, n1;
            const bf16 *X1;
            float *o1;
            chunk_at(c + 1, bh1, tk1, n1, X1, o1);
            load_x<DR>(X1, (long long)bh1 * n1 + tk1 + rt, tk1 + rt < n1, x);
        }
        if (t == 0 && !(ntile <= 2 && h == resident_h)) {
            for (int j = 0; j < 2 && j < ntile; ++j) {
                mbar_arrive_expect_tx(bars + S_TB0 + j, (uint32_t)a.bimg_bytes);
                bulk_g2s(smem + (j ? L.tb1 : L.tb0), img + (size_t)j * a.bimg_bytes, (uint32_t)a.bimg_bytes,
                         bars + S_TB0 + j);
                pending |= 1u << j;
            }
            resident_h = ntile <= 2 ? h : -1;
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // thread 0: the logits of tile j, once its table is in
        auto issue = [&](int j) {
            const int b = j & 1;
            if ((pending >> b) & 1u) {   // (with two tiles and the same head as before, nothing was loaded)
                if (!mbar_wait(bars + S_TB0 + b, (ph_tb >> b) & 1u, a.hdr, 60)) {
                    *stop = 1;
                    return;
                }
                ph_tb ^= 1u << b;
                pending &= ~(1u << b);
            }
            tc_fence_after();
            const uint32_t tbuf = sb + (b ? L.tb1 : L.tb0);
            issue_logits_c<DR>(tmem + 128u * b, sb + L.abuf, tbuf, tbuf + (uint32_t)main_bytes, sb + L.ax, KMAX);
            mma_commit(bars + S_MMA0 + b);
        };
        if (t == 0) issue(0);
        float m = NEG_BIG, s = 0.f, best = NEG_BIG;
        int arg = 0;
        for (int j = 0; j < ntile; ++j) {
            const int b = j & 1;
            const bool ok = !*stop && mbar_wait(bars + S_MMA0 + b, (ph_mma >> b) & 1u, a.hdr, 61);
            ph_mma ^= 1u << b;
            if (__syncthreads_or(!ok)) break;
            tc_fence_after();
            if (t == 0) {
                if (j + 2 < ntile) {   // this buffer's table has been read by the MMA just completed
                    mbar_arrive_expect_tx(bars + S_TB0 + b, (uint32_t)a.bimg_bytes);
                    bulk_g2s(smem + (b ? L.tb1 : L.tb0), img + (size_t)(j + 2) * a.bimg_bytes, (uint32_t)a.bimg_bytes,
                             bars + S_TB0 + b);
                    pending |= 1u << b;
                }
                if (j + 1 < ntile) issue(j + 1);
            }
            // this half's 64 columns of the tile: their maximum, then the running maximum and sum
            const int nv = min(64, max(0, min(KMAX, K_all - KMAX * j) - 64 * half));
            uint32_t ra[32], rb[32];
            tmem_ld32(lane + 128u * b + 64u * half, ra);   // (every lane loads: warp-collective)
            tmem_ld32(lane + 128u * b + 64u * half + 32u, rb);
            tmem_ld_wait();
            if (nv > 0) {
                const int col0 = KMAX * j + 64 * half;
                if (nv == 64)
                    tile_update<64>(ra, rb, 64, m, s, best, arg, col0, assign != nullptr);
                else
                    tile_update<0>(ra, rb, nv, m, s, best, arg, col0, assign != nullptr);
            }
            tc_fence_before();
            __syncthreads();   // region b read by every row before the MMA of tile j + 2 writes it
            tc_fence_after();
        }
        if (*stop) break;
        // the upper half hands its row's state to the lower half (read before the lower half
        // reaches the next chunk's first barrier, so one slot per row suffices)
        float4 *xch = reinterpret_cast<float4 *>(smem + L.xch);
        if (half) xch[rt] = make_float4(m, s, best, __int_as_float(arg));
        __syncthreads();
        if (!half && valid) {
            const float4 o = xch[rt];
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
    // table loads still in flight (only after a stop) complete before shared memory is released;
    // an MMA that was issued has completed or been waited for by every thread
    if (t == 0)
        for (int b = 0; b < 2; ++b)
            if ((pending >> b) & 1u) mbar_wait(bars + S_TB0 + b, (ph_tb >> b) & 1u, a.hdr, 62);
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
#define LSE_FETCH_ROW(lc)                                                                                        \
    do {                                                                                                         \
        const ChunkInfo ci_ = cl.at(c_begin + (lc));                                                            \
        load_x<DR>(ci_.X, (long long)ci_.bh * ci_.n + ci_.tok0 + rt, ci_.tok0 + rt < ci_.n, x);                  \
    } while (0)
    if (warp < 4 && nloc > 0) LSE_FETCH_ROW(0);   // (the rows are inputs: no kernel before writes them)
    grid_dependency_wait();   // the tables come from the parameter kernel
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);
    const int main_bytes = a.bimg_main_bytes, blk = 128 * 128;   // (one tile's 64-column block: 16 KB)

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
                const uint8_t *img = a.bimg + (size_t)h * a.bimg_head;
                mbar_arrive_expect_tx(bars + L_TB, 2u * (uint32_t)a.bimg_bytes);
                for (int t2 = 0; t2 < 2; ++t2) {
                    const uint8_t *src = img + (size_t)t2 * a.bimg_bytes;
                    for (int q = 0; q < main_bytes / blk; ++q)
                        bulk_g2s(smem + L.tab + (uint32_t)(q * 2 * blk + t2 * blk), src + (size_t)q * blk, (uint32_t)blk,
                                 bars + L_TB);
                    bulk_g2s(smem + L.tab + (uint32_t)(2 * main_bytes + t2 * 128 * 32), src + main_bytes, 128u * 32u,
                             bars + L_TB);
                }
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
            if (nloc > 1) LSE_FETCH_ROW(1);
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
                if (lc + 2 < nloc) LSE_FETCH_ROW(lc + 2);
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
#undef LSE_FETCH_ROW
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
