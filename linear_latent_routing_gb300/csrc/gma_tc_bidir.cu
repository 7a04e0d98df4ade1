// gma_tc_bidir.cu -- the read phase of bidirectional GMA (tcgen05, sm_103a).
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §2, read phase: O = Gamma_Q V~ / (Gamma_Q Z + eps), with V~ = Gamma_K^T V and
// Z = Gamma_K^T 1 summed over the whole sequence (the segment pass and the scan leave the total
// of each (b, h) slice in its first segment's slot).
//
// With E_Q = exp2 of the query logits minus their row maximum (row sums s_i, kept unnormalised):
//   O_i = (E_Q V~)_i / (E_Q . Z + eps * s_i)
// the numerator by one tcgen05.mma chain (E_Q as the A operand from TMEM, V~ as bf16 from shared
// memory), the normaliser on the CUDA cores in fp32.
//
// Two groups of four warps take alternate chunks of 128 query tokens, each with its own TMEM
// columns (logits, then E_Q, and the numerator) and its own A tile, and each issues its own MMAs
// and TMA loads from one elected thread.  While one group exponentiates, the other's logits or
// numerator run on the tensor cores.  Every wait is bounded; a timeout records GMA_ERR_TIMEOUT
// and both groups leave their loops.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

constexpr int BTHREADS = 256;
// (B_F*: a group's output stage is free, its previous TMA store having read it; B_W*: the stage
// holds all 128 rows of the chunk)
enum BBar { B_BIMG, B_X0, B_X1, B_SP, B_A0, B_A1, B_E0, B_E1, B_L0, B_L1, B_O0, B_O1, B_F0, B_F1, B_W0, B_W1, B_NBAR };

struct BidirSmem {
    uint32_t bimg, ax, ab0, ab1, sp, os0, os1, z, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    // (the output stages, C rows of d_v bf16 per group, exist when d_v is a multiple of 64)
    __host__ __device__ BidirSmem(int DR, int kn16, int d_v)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        const uint32_t tile = ka / 64u * 128u;
        uint32_t o = 0;
        bimg = o; o = al(o + tile * (uint32_t)kn16 + 32u * (uint32_t)kn16);
        ax = o; o = al(o + (uint32_t)C * 32u);
        ab0 = o; o = al(o + (uint32_t)C * DR * 4u);   // group 0's [x^2 | x]
        ab1 = o; o = al(o + (uint32_t)C * DR * 4u);   // group 1's
        sp = o; o = al(o + (uint32_t)d_v * KMAX * 2u);
        const uint32_t ost = d_v % 64 == 0 ? (uint32_t)C * d_v * 2u : 0u;
        os0 = o; o = al(o + ost);
        os1 = o; o = al(o + ost);
        z = o; o += KMAX * 4u;
        bars = o; o += B_NBAR * 8u;
        misc = o; o += 16u;
        total = o;
    }
};

// Tensor-memory columns of one CTA: two groups, each with its logits (kn16 rounded up to 32) and
// numerator (d_v rounded up to 32), as a power of two of at least 32.  Small shapes fit in 256
// columns or fewer, so that two CTAs share an SM and one's latency hides behind the other's work.
__host__ __device__ inline uint32_t bidir_tmem_cols(int kn16, int d_v)
{
    const uint32_t need = 2u * ((uint32_t)((kn16 + 31) & ~31) + (uint32_t)((d_v + 31) & ~31));
    uint32_t cols = 32;
    while (cols < need) cols *= 2;
    return cols;
}

// Unnormalised E_Q of this row over all kc 32-column groups (zeros when not valid), back into
// TMEM at tl as bf16 pairs (group c at column 16 c); returns (row sum, dot product with z).
// With components in tiles (use_lse), E_Q = exp2(L - lse) with the row's log2-sum-exp over all
// components: the normalised responsibilities of this tile, no maximum needed.
__device__ __forceinline__ float2 exp_row(uint32_t tl, int K, int kc, bool valid, const float *z, bool use_lse,
                                          float lse)
{
    // a row past the end of the sequence exponentiates against +inf: all of its values are 0 (the
    // maximum is taken by every lane: its tensor-memory loads are warp-collective)
    const float mr = use_lse ? lse : row_max(tl, K, kc);
    const float m = valid ? mr : __int_as_float(0x7f800000);
    float srow = 0.f, den = 0.f;
#pragma unroll 1
    for (int c = 0; c < kc; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        srow += chunk_exp(r, c, K, m);
        float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            // read in program order, so that no group's z values are held ahead of its use
            float4 zz;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(zz.x), "=f"(zz.y), "=f"(zz.z), "=f"(zz.w)
                         : "r"(smem_u32(z + 32 * c + 4 * q)));
            d4[0] = fmaf(__uint_as_float(r[4 * q]), zz.x, d4[0]);
            d4[1] = fmaf(__uint_as_float(r[4 * q + 1]), zz.y, d4[1]);
            d4[2] = fmaf(__uint_as_float(r[4 * q + 2]), zz.z, d4[2]);
            d4[3] = fmaf(__uint_as_float(r[4 * q + 3]), zz.w, d4[3]);
        }
        den += (d4[0] + d4[1]) + (d4[2] + d4[3]);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        tmem_st16(tl + 16 * c, w);
    }
    tmem_st_wait();
    return make_float2(srow, den);
}

// Output row orow = (d_v numerator columns of TMEM at tl) * inv, bf16 or fp32.
__device__ __forceinline__ void store_row(uint32_t tl, int d_v, float inv, bool valid, void *O, long long orow,
                                          int out_f32)
{
#pragma unroll 1
    for (int c = 0; c < (d_v + 31) / 32; ++c) {
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

// The same row into the output stage os (rows of d_v bf16 in 64-column blocks with the 128-byte
// swizzle: the layout of the TMA boxes), zeros for rows past the end.
__device__ __forceinline__ void stage_row(uint32_t tl, int d_v, float inv, bool valid, uint8_t *os, int row)
{
    const float s = valid ? inv : 0.f;
#pragma unroll 1
    for (int c = 0; c < d_v / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4 *>(os + sw128(row, 4 * c + q, C)) =
                make_uint4(pk2(r[8 * q], r[8 * q + 1], s), pk2(r[8 * q + 2], r[8 * q + 3], s),
                           pk2(r[8 * q + 4], r[8 * q + 5], s), pk2(r[8 * q + 6], r[8 * q + 7], s));
    }
}

// MINB: CTAs per SM the register allocation is sized for (two for shapes whose tensor memory
// and shared memory let two CTAs share an SM, one otherwise).
template <int DR, int MINB>
__global__ void __launch_bounds__(BTHREADS, MINB) tc_bidir_read2_kernel(const Args a,
                                                                     const __grid_constant__ CUtensorMap qmap,
                                                                     const __grid_constant__ CUtensorMap omap)
{
    // (no wait here: the set-up and the first query rows, which no kernel writes, overlap the
    // kernel before; the threads that read its results wait below)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const BidirSmem L(DR, a.kn16, a.d_v);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.misc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.misc + 4);
    float *z = reinterpret_cast<float *>(smem + L.z);
    const int bh = blockIdx.x / a.nseg, seg = blockIdx.x % a.nseg, h = bh % a.H;
    const int t = threadIdx.x, warp = t >> 5;
    const int g = warp >> 2, i = t & 127;   // group, and row of the chunk / component row
    const int tok0 = seg * a.cps * C;
    const int tok_end = min(a.N, tok0 + a.cps * C);
    const int nch = (tok_end - tok0 + C - 1) / C;
    const int d_v = a.d_v;
    // 32-column groups of E_Q: as many as the table's rows need (with components in tiles, the last
    // tile's E_Q beyond its K components is written as zeros)
    const int kc = (a.kn16 + 31) >> 5;
    constexpr uint32_t XT = (uint32_t)C * DR * 2;
    const bool leader = i == 0;

    if (t == 0) {
        for (int b = 0; b < B_NBAR; ++b)
            mbar_init(bars + b, ((b >= B_SP && b <= B_E1) || b == B_W0 || b == B_W1) ? 128u : 1u);
        *abort = 0;
        fence_mbar_init();
    }
    const uint32_t ncols = bidir_tmem_cols(a.kn16, a.d_v);
    if (warp == 0) tmem_alloc(tslot, ncols);
    if (g == 1) {
        // constant A operand of the logits: (1, 1, 0, ...) in every row, K-major SW32
        const int flip = (i >> 2) & 1;
        *reinterpret_cast<uint4 *>(smem + L.ax + i * 32 + (flip << 4)) = make_uint4(0x3C003C00u, 0, 0, 0);
        *reinterpret_cast<uint4 *>(smem + L.ax + i * 32 + ((flip ^ 1) << 4)) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);
    // per group: the logits (E_Q in place) then the numerator, each rounded up to 32 columns
    const uint32_t lw = (uint32_t)((a.kn16 + 31) & ~31), ow = (uint32_t)((d_v + 31) & ~31);
    const uint32_t R_L = (uint32_t)g * (lw + ow), R_O = R_L + lw;
    const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint8_t *ab = smem + (g ? L.ab1 : L.ab0);
    uint64_t *bx = bars + B_X0 + g, *ba = bars + B_A0 + g, *be = bars + B_E0 + g;
    uint64_t *bl = bars + B_L0 + g, *bo = bars + B_O0 + g;
    int last_x = -1;   // leader: chunk of this group's TMA load still possibly in flight
    if (leader) {
        if (g < nch) {
            load_x_tile(ab + XT, &qmap, bx, DR, tok0 + g * C, bh);
            last_x = g;
        }
        if (t == 0) {
            grid_dependency_wait();   // the tables come from the kernels before
            mbar_arrive_expect_tx(bars + B_BIMG, (uint32_t)a.bimg_bytes);
            bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars + B_BIMG);
        }
    }
    // (components in tiles: the rows' log2-sum-exp, and the partial sums of the tiles before)
    if (a.lse_q && g == 1) grid_dependency_wait();
    if (g == 0) {
        grid_dependency_wait();   // the slice's total memory comes from the kernels before
        // the slice's total memory: V~ rows as the bf16 operand, Z into shared memory
        const float *src = a.agg + ((size_t)bh * a.agg_nseg * KMAX + i) * a.ne;
        for (int b = 0; b < d_v / 16; ++b) {
            const float4 *s4 = reinterpret_cast<const float4 *>(src + b * 16);
            uint32_t r[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = s4[q];
                r[4 * q] = __float_as_uint(f.x);
                r[4 * q + 1] = __float_as_uint(f.y);
                r[4 * q + 2] = __float_as_uint(f.z);
                r[4 * q + 3] = __float_as_uint(f.w);
            }
            *reinterpret_cast<uint4 *>(smem + L.sp + sw32(i, b, 0, KMAX)) =
                make_uint4(pk2(r[0], r[1], 1.f), pk2(r[2], r[3], 1.f), pk2(r[4], r[5], 1.f), pk2(r[6], r[7], 1.f));
            *reinterpret_cast<uint4 *>(smem + L.sp + sw32(i, b, 1, KMAX)) =
                make_uint4(pk2(r[8], r[9], 1.f), pk2(r[10], r[11], 1.f), pk2(r[12], r[13], 1.f), pk2(r[14], r[15], 1.f));
        }
        z[i] = src[d_v];
        fence_proxy_async_smem();
        mbar_arrive(bars + B_SP);
    }
    const uint32_t id_o = idesc_f16(128, (uint32_t)d_v, 1, 1, 0, 1);
    const int ksteps = a.kn16 / 16;
    bool ok = true;
    for (int c = g; ok && c < nch; c += 2) {
        const uint32_t n = (uint32_t)(c >> 1) & 1u;   // this group's barrier phase
        const int row = tok0 + c * C + i;
        const bool valid = row < tok_end;
        // [x^2, x] in place; the numerator columns of this group's previous chunk are read
        if (!(ok = mbar_wait_abortable(bx, n, a.hdr, 150, abort))) break;
        build_inplace<DR>(ab, i);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ba);
        if (leader) {
            if (c < 2 && !(ok = mbar_wait_abortable(bars + B_BIMG, 0, a.hdr, 151, abort))) break;
            if (!(ok = mbar_wait_abortable(ba, n, a.hdr, 152, abort))) break;
            tc_fence_after();
            issue_logits_x<DR>(tmem + R_L, sb + (g ? L.ab1 : L.ab0), sb + L.bimg,
                               sb + L.bimg + (uint32_t)a.bimg_main_bytes, sb + L.ax, a.kn16);
            mma_commit(bl);
        }
        // (components in tiles: the row's log2-sum-exp over all components, read ahead)
        const float lse_row = (a.lse_q && valid) ? a.lse_q[(long long)bh * a.N + row] : 0.f;
        if (!(ok = mbar_wait_abortable(bl, n, a.hdr, 153, abort))) break;
        if (leader && c + 2 < nch) {   // the A tile is read: this group's next rows
            load_x_tile(ab + XT, &qmap, bx, DR, tok0 + (c + 2) * C, bh);
            last_x = c + 2;
        }
        if (c < 2 && !(ok = mbar_wait_abortable(bars + B_SP, 0, a.hdr, 154, abort))) break;
        tc_fence_after();
        const float2 sd = exp_row(lane + R_L, a.K, kc, valid, z, a.lse_q != nullptr, lse_row);
        tc_fence_before();
        mbar_arrive(be);
        if (leader) {
            if (!(ok = mbar_wait_abortable(be, n, a.hdr, 155, abort))) break;
            tc_fence_after();
            for (int s = 0; s < ksteps; ++s)   // numerator = E_Q V~
                mma_f16_tmem_a(tmem + R_O, tmem + R_L + 8 * s, mn32desc(sb + L.sp, s, KMAX), id_o, s > 0);
            mma_commit(bo);
        }
        if (!(ok = mbar_wait_abortable(bo, n, a.hdr, 156, abort))) break;
        tc_fence_after();
        if (a.pmode) {
            tile_partial_row(lane + R_O, d_v, sd.y + a.eps * sd.x, valid, a.part, a.pden, (long long)bh * a.N + row,
                             a.pmode);
        } else if (a.o_tma) {
            // the group's stage is free once the TMA store of its previous chunk has read it (the
            // leader's own bulk group); then the rows go in, and the leader stores the box(es)
            uint8_t *os = smem + (g ? L.os1 : L.os0);
            if (leader && c >= 2) {
                bulk_wait_read();
                mbar_arrive(bars + B_F0 + g);
            }
            if (c >= 2 && !(ok = mbar_wait_abortable(bars + B_F0 + g, ((c >> 1) - 1) & 1, a.hdr, 159, abort))) break;
            stage_row(lane + R_O, d_v, 1.0f / (sd.y + a.eps * sd.x), valid, os, i);
            fence_proxy_async_smem();
            mbar_arrive(bars + B_W0 + g);
            if (leader) {
                if (!(ok = mbar_wait_abortable(bars + B_W0 + g, n, a.hdr, 160, abort))) break;
                for (int hb = 0; hb < d_v / 64; ++hb) tma_store_3d(&omap, os + hb * C * 128, 64 * hb, tok0 + c * C, bh);
                bulk_commit_group();
            }
        } else {
            store_row(lane + R_O, d_v, 1.0f / (sd.y + a.eps * sd.x), valid, a.O, (long long)bh * a.N + row,
                      a.out_f32);
        }
    }
    // the output stores have completed before the CTA (and its shared memory) is released
    if (a.o_tma && leader) bulk_wait_all();
    // a TMA load issued but not consumed (only after a timeout) completes before shared memory
    // is released
    if (leader && !ok && last_x >= 0) mbar_wait(bx, (uint32_t)(last_x >> 1) & 1u, a.hdr, 157);
    if (t == 0 && !ok) mbar_wait(bars + B_BIMG, 0, a.hdr, 158);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, ncols);
}

uint32_t bidir_read2_smem(int d_r, int kn16, int d_v)
{
    const uint32_t need = BidirSmem(d_r, kn16, d_v).total + 1024;
    return need <= 227u * 1024u ? smem_for(need, bidir_tmem_cols(kn16, d_v)) : 0;
}

int bidir_read2_ctas_per_sm(int d_r, int kn16, int d_v)
{
    const uint32_t cols = bidir_tmem_cols(kn16, d_v);
    const uint32_t sm = bidir_read2_smem(d_r, kn16, d_v);
    // two CTAs need the kernel within 128 registers a thread: it then spills 20-30 bytes at
    // d_r <= 32, a net gain (LRA-shaped workload: read pass 103 -> 93 us), but 40 bytes at
    // d_r = 64, a net loss (cross-attention workload: 37.5 -> 41.7 us)
    int n = (cols <= 256 && d_r <= 32) ? 2 : 1;
    if (sm == 0 || (uint32_t)n * sm > 228u * 1024u) n = 1;
    return n;
}

template <int DR, int MINB>
gma_status_t launch_bidir_read2_n(const Args &a, const CUtensorMap &qmap, const CUtensorMap &omap, int nblocks,
                                  uint32_t sm, cudaStream_t st)
{
    if (!set_smem(tc_bidir_read2_kernel<DR, MINB>, sm)) return GMA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_BIDIR_READ, st,
               (e = launch_pdl(tc_bidir_read2_kernel<DR, MINB>, dim3(nblocks), dim3(BTHREADS), sm, st, a, qmap, omap)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

// omap: the output's tensor map (bf16, 64-column boxes, 128-byte swizzle), or null for stores from
// the threads (fp32 output, d_v not a multiple of 64, or the tiles' partial sums).
template <int DR>
gma_status_t launch_bidir_read2(const Args &a, const CUtensorMap &qmap, const CUtensorMap *omap, int nblocks,
                                cudaStream_t st)
{
    const uint32_t sm = bidir_read2_smem(DR, a.kn16, a.d_v);
    if (sm == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    Args b = a;
    b.o_tma = omap && !a.out_f32 && !a.pmode && a.d_v % 64 == 0 ? 1 : 0;
    const CUtensorMap &om = b.o_tma ? *omap : qmap;   // (not read unless o_tma)
    return bidir_read2_ctas_per_sm(DR, a.kn16, a.d_v) == 2 ? launch_bidir_read2_n<DR, 2>(b, qmap, om, nblocks, sm, st)
                                                           : launch_bidir_read2_n<DR, 1>(b, qmap, om, nblocks, sm, st);
}

template gma_status_t launch_bidir_read2<16>(const Args &, const CUtensorMap &, const CUtensorMap *, int, cudaStream_t);
template gma_status_t launch_bidir_read2<32>(const Args &, const CUtensorMap &, const CUtensorMap *, int, cudaStream_t);
template gma_status_t launch_bidir_read2<64>(const Args &, const CUtensorMap &, const CUtensorMap *, int, cudaStream_t);

}  // namespace tck
}  // namespace gma
