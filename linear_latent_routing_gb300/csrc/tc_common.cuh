// tc_common.cuh -- definitions shared by the tcgen05 translation units of libgma.so: constants,
// kernel arguments, shared-memory operand layouts and their descriptors, the [x^2, x] builder and
// the TMA of value tiles.
//
// The Gaussian table of a head (written by tc_params_kernel) has two parts:
//   main:  kn16 rows (components) x ka columns, fp16, K-major 128-byte swizzle, holding
//          log2e * [-w/2 ; mu w] (w = 1/sigma^2), so that [x^2, x] . row = the x-dependent part of
//          log2e * log N(x; mu, sigma^2);
//   const: kn16 rows x 16 columns, fp16, K-major 32-byte swizzle, holding (c_hi, c_lo, 0, ...)
//          with c_hi + c_lo = log2e * (log pi - 1/2 sum_d (mu^2 w + log sigma^2)).
// Multiplied by a constant operand whose rows are (1, 1, 0, ...), the const part adds the
// per-component constant inside the same MMA, so the accumulator holds complete log2 logits.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "gma_internal.cuh"
#include "tc_ptx.cuh"

namespace gma {
namespace tck {

using namespace tc;

constexpr int C = 128;          // tokens per chunk (the MMA M dimension)
constexpr int THREADS = 128;    // one thread per TMEM lane / token row / component row
constexpr int KMAX = 128;       // components handled by this family
constexpr float LOG2E = 1.4426950408889634f;
constexpr float NEG_BIG = -1.0e30f;

typedef __nv_bfloat16 bf16;

struct Args {
    const bf16 *QX, *KX;
    void *O;                 // output (bf16 or fp32)
    void *gamma;             // responsibilities output (bf16 or fp32)
    int *assign;             // usage diagnostics (non-null: no gamma written): argmax per row,
    int *counts;             //   per-head histogram [H][K] (atomic adds), and per-CTA sums of
    float *mass_part;        //   the responsibilities [grid][K]
    const uint8_t *bimg;     // per-head Gaussian table image [H][bimg_bytes]: the [x^2, x] part
                             // (bimg_main_bytes), then the constant part (kn16 rows x 32 B)
    const float *cst;        // per-head log2-domain constants [H][kn16]
    float *agg;              // segment memories [BH][nseg][KMAX][ne] fp32
    WsHeader *hdr;
    int H, N, K, kn16, d_v, ne;
    int nseg, cps;           // segments per slice, chunks per segment
    int agg_nseg;            // segments per slice in agg (the key side's, for cross-attention)
    int bimg_bytes, bimg_main_bytes;
    float eps;
    int out_f32;
    bf16 *gam;               // causal: key responsibilities [BH][N][kg] (null: recomputed)
    int kg;
    int test_withhold;       // GMA_FLAG_TEST_WITHHOLD: the key pass withholds one hand-off
    int v128;                // value tiles in 64-column boxes with the 128-byte swizzle (d_v >= 64)
    int o_tma;               // bidirectional read: output rows staged in shared memory, written by
                             // TMA stores of 64-column boxes (bf16 output, d_v a multiple of 64)
    // More than 128 components: the components are cut into tiles of 128 and each pass works on
    // one tile (components [128 tile, 128 tile + K) of the head's K_all, K being the tile's count)
    // with every routing row's log2-sum-exp over all components precomputed (lse_q for the
    // queries, lse_k for the keys; null when K_all <= 128).  The causal output pass then adds
    // each tile's numerator and normaliser into part / pden (pmode 1: the first tile writes,
    // 2: a later tile adds; 0: one tile, O written directly); a last kernel divides the sums.
    int bimg_head;           // bytes of one head's table images (tiles x bimg_bytes)
    int tile;
    int kall;                // components in all (the row length of gamma and of the usage sums)
    const float *lse_q, *lse_k;
    float *part, *pden;
    int pmode;
};

// The Gaussian table image of head h for the tile a pass works on.
__device__ __forceinline__ const uint8_t *table_of(const Args &a, int h)
{
    return a.bimg + (size_t)h * a.bimg_head + (size_t)a.tile * a.bimg_bytes;
}

// ------------------------------------------------------------------ layout helpers
__device__ __forceinline__ uint32_t sw128(int row, int q, int rows)
{
    return (uint32_t)((q >> 3) * rows * 128 + row * 128 + (((q & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t sw32(int row, int blk, int half, int rows)
{
    return (uint32_t)(blk * rows * 32 + row * 32 + ((half ^ ((row >> 2) & 1)) << 4));
}

// K-major SW128 operand, k-step s (16 elements)
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int s, int rows)
{
    return smem_desc(base + (uint32_t)((s >> 2) * rows * 128 + (s & 3) * 32), 16, 1024, SW_128B);
}

// MN-major SW128 operand whose K dimension runs along rows (128 B each), k-step s.
__device__ __forceinline__ uint64_t mn128desc(uint32_t base, int s, int rows)
{
    return smem_desc(base + (uint32_t)(s * 16 * 128), (uint32_t)(rows * 128), 1024, SW_128B);
}

// K-major SW32 operand of one k-step (rows of 16 two-byte elements, 32 B each).
__device__ __forceinline__ uint64_t kdesc32(uint32_t base)
{
    return smem_desc(base, 16, 256, SW_32B);
}

// MN-major SW32 operand (blocks of 16 MN elements), k-step s.
__device__ __forceinline__ uint64_t mn32desc(uint32_t base, int s, int rows)
{
    return smem_desc(base + (uint32_t)(s * 16 * 32), (uint32_t)(rows * 32), 256, SW_32B);
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b)
{
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}


// Builds [x^2, x] (fp16, K-major SW128, ka columns) for token row `row` from its bf16 vector.
template <int DR>
__device__ __forceinline__ void build_a(uint8_t *abuf, int row, const uint4 (&x)[DR / 8])
{
    constexpr int KA = DR * 2 < 64 ? 64 : DR * 2;
#pragma unroll
    for (int q = 0; q < KA / 8; ++q) {
        uint4 v;
        if (q < DR / 8) {
            const bf16 *e = reinterpret_cast<const bf16 *>(&x[q]);
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __bfloat162float(e[j]);
            v.x = pack_f16(f[0] * f[0], f[1] * f[1]);
            v.y = pack_f16(f[2] * f[2], f[3] * f[3]);
            v.z = pack_f16(f[4] * f[4], f[5] * f[5]);
            v.w = pack_f16(f[6] * f[6], f[7] * f[7]);
        } else if (q < DR / 4) {
            const bf16 *e = reinterpret_cast<const bf16 *>(&x[q - DR / 8]);
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __bfloat162float(e[j]);
            v.x = pack_f16(f[0], f[1]);
            v.y = pack_f16(f[2], f[3]);
            v.z = pack_f16(f[4], f[5]);
            v.w = pack_f16(f[6], f[7]);
        } else {
            v = make_uint4(0, 0, 0, 0);
        }
        *reinterpret_cast<uint4 *>(abuf + sw128(row, q, C)) = v;
    }
}

// Byte offset of 16-byte chunk s of row r in a staged x tile (rows of DR bf16 = 2*DR bytes, TMA
// swizzle of the same width: 32, 64 or 128 bytes).
template <int DR>
__device__ __forceinline__ uint32_t xs_off(int r, int s)
{
    constexpr uint32_t M = DR == 64 ? 7u : DR == 32 ? 3u : 1u;
    const uint32_t o = (uint32_t)r * (DR * 2) + (uint32_t)s * 16u;
    return o ^ (((o >> 7) & M) << 4);
}

// build_a for token row `row` from the staged (TMA, swizzled) x tile xs: each 16-byte chunk of
// the row (8 bf16) gives one chunk of x^2 and one of x (fp16).
template <int DR>
__device__ __forceinline__ void build_a_s(uint8_t *abuf, int row, const uint8_t *xs)
{
    constexpr int KA = DR * 2 < 64 ? 64 : DR * 2;
#pragma unroll
    for (int q = 0; q < DR / 8; ++q) {
        const uint4 v = *reinterpret_cast<const uint4 *>(xs + xs_off<DR>(row, q));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t sq[4], li[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
            sq[j] = pack_f16(lo * lo, hi * hi);
            li[j] = pack_f16(lo, hi);
        }
        *reinterpret_cast<uint4 *>(abuf + sw128(row, q, C)) = make_uint4(sq[0], sq[1], sq[2], sq[3]);
        *reinterpret_cast<uint4 *>(abuf + sw128(row, DR / 8 + q, C)) = make_uint4(li[0], li[1], li[2], li[3]);
    }
#pragma unroll
    for (int q = DR / 4; q < KA / 8; ++q) *reinterpret_cast<uint4 *>(abuf + sw128(row, q, C)) = make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------------ [x^2, x] tile built in place
// The A operand of the logits as two K-major tiles of 128 rows x DR fp16 columns (rows of 2*DR
// bytes, swizzle of the same width): x^2 at ab, x at ab + 128 * 2 * DR.  TMA writes the bf16 rows
// into the x tile; the builder reads them, writes x^2 and rewrites x as fp16 in place.
template <int DR>
__device__ __forceinline__ void build_inplace(uint8_t *ab, int row)
{
    uint8_t *abx = ab + C * DR * 2;
#pragma unroll
    for (int q = 0; q < DR / 8; ++q) {
        const uint32_t o = xs_off<DR>(row, q);
        const uint4 v = *reinterpret_cast<const uint4 *>(abx + o);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t sq[4], li[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
            sq[j] = pack_f16(lo * lo, hi * hi);
            li[j] = pack_f16(lo, hi);
        }
        *reinterpret_cast<uint4 *>(ab + o) = make_uint4(sq[0], sq[1], sq[2], sq[3]);
        *reinterpret_cast<uint4 *>(abx + o) = make_uint4(li[0], li[1], li[2], li[3]);
    }
}

// Descriptor of k-step s (16 columns) of the in-place A tiles.
template <int DR>
__device__ __forceinline__ uint64_t abdesc(uint32_t ab, int s)
{
    constexpr int KPS = DR / 16;   // k-steps per tile
    constexpr uint32_t RB = DR * 2;
    return smem_desc(ab + (uint32_t)(s / KPS) * (uint32_t)C * RB + (uint32_t)(s % KPS) * 32u, 16, 8u * RB,
                     DR == 64 ? SW_128B : DR == 32 ? SW_64B : SW_32B);
}

// Logits of 128 tokens: [x^2, x] (in-place tiles at ab) times the head's table, plus the constant.
template <int DR>
__device__ __forceinline__ void issue_logits_x(uint32_t d, uint32_t ab, uint32_t bimg, uint32_t bconst, uint32_t ax,
                                               int kn16)
{
    const uint32_t id = idesc_f16(128, (uint32_t)kn16, 0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < DR / 8; ++s) mma_f16(d, abdesc<DR>(ab, s), kdesc(bimg, s, kn16), id, s > 0);
    mma_f16(d, kdesc32(ax), kdesc32(bconst), id, 1u);   // + per-component constant
}

// TMA of the x rows [tok, tok + 128) of slice bh (3-D map {DR, N, BH}, box {DR, 128, 1}; rows past
// the sequence read as zeros) into the staging tile xs.
__device__ __forceinline__ void load_x_tile(uint8_t *xs, const CUtensorMap *map, uint64_t *bar, int DR, int tok,
                                            int bh)
{
    mbar_arrive_expect_tx(bar, (uint32_t)(C * DR * 2));
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(xs)),
        "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(0), "r"(tok), "r"(bh)
        : "memory");
}

template <int DR>
__device__ __forceinline__ void load_x(const bf16 *X, long long row, bool valid, uint4 (&x)[DR / 8])
{
#pragma unroll
    for (int q = 0; q < DR / 8; ++q)
        x[q] = valid ? __ldg(reinterpret_cast<const uint4 *>(X + row * DR) + q) : make_uint4(0, 0, 0, 0);
}

// TMA of V rows [tok, tok + 128) of slice bh into the MN-major SW32 blocks of `ve`.
__device__ __forceinline__ void load_v_chunk(uint8_t *ve, const CUtensorMap *vmap, uint64_t *bar,
                                             int d_v, int tok, int bh)
{
    mbar_arrive_expect_tx(bar, (uint32_t)(C * d_v * 2));
    for (int b = 0; b < d_v / 16; ++b) {
        // 3-D map {d_v, N, BH}, box {16, 128, 1}
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(ve + b * C * 32)),
            "l"((uint64_t)vmap), "r"(smem_u32(bar)), "r"(b * 16), "r"(tok), "r"(bh)
            : "memory");
    }
}


// TMA of V rows [tok, tok + 128) of slice bh as d_v / 64 MN-major atoms of 64 columns with the
// 128-byte swizzle (3-D map {d_v, N, BH}, box {64, 128, 1}), atom b at ve + b * 16 KB.
__device__ __forceinline__ void load_v_chunk128(uint8_t *ve, const CUtensorMap *vmap, uint64_t *bar, int d_v, int tok,
                                                int bh)
{
    mbar_arrive_expect_tx(bar, (uint32_t)(C * d_v * 2));
    for (int b = 0; b < d_v / 64; ++b) {
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(ve + b * C * 128)),
            "l"((uint64_t)vmap), "r"(smem_u32(bar)), "r"(b * 64), "r"(tok), "r"(bh)
            : "memory");
    }
}

// ------------------------------------------------------------------ the pipelined causal kernel
uint32_t causal_pipelined_smem(int d_r, int kn16, int d_v);
template <int DR>
gma_status_t launch_causal_pipelined(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap,
                                     const CUtensorMap &qmap, int nblocks, cudaStream_t st);

uint32_t segmem_pipelined_smem(int d_r, int kn16, int d_v);
template <int DR>
gma_status_t launch_segmem_pipelined(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap,
                                     const CUtensorMap &gmap, int nblocks, cudaStream_t st);
uint32_t bidir_read2_smem(int d_r, int kn16, int d_v);
template <int DR>
gma_status_t launch_bidir_read2(const Args &a, const CUtensorMap &qmap, const CUtensorMap *omap, int nblocks,
                                cudaStream_t st);
uint32_t causal_gamma_smem(int d_r, int kn16, int d_v);
template <int DR>
gma_status_t launch_lse(const Args &a, const bf16 *rows0, const bf16 *rows1, float *lse0, float *lse1, int K_all,
                        int BH, cudaStream_t st, int *assign = nullptr, int *counts = nullptr, int N1 = -1);
template <int DR>
gma_status_t launch_causal_gamma(const Args &a, const CUtensorMap &vmap, const CUtensorMap &qmap,
                                 const CUtensorMap &gmap, int nblocks, cudaStream_t st);

// ------------------------------------------------------------------ host helpers (gma_tc.cu)
bool make_vmap(CUtensorMap *m, const void *V, int BH, int N, int d_v);
bool make_vmap128(CUtensorMap *m, const void *V, int BH, int N, int d_v);
bool make_xmap(CUtensorMap *m, const void *X, int BH, int N, int d_r);
bool make_gmap(CUtensorMap *m, const void *G, int BH, int N, int kg);
uint32_t smem_for(uint32_t need, uint32_t tmem_cols);
bool encode_available();

template <typename KernelT>
bool set_smem(KernelT kernel, uint32_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

}  // namespace tck
}  // namespace gma
