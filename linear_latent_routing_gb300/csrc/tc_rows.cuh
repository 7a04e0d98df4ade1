// tc_rows.cuh -- per-row softmax helpers and the logits MMA shared by the tcgen05 kernels that
// work one chunk of 128 tokens at a time (one thread per TMEM lane / token row).
#pragma once

#include "tc_common.cuh"

namespace gma {
namespace tck {
namespace {

// The row phases below run on one warp per SM sub-partition, so their speed is set by
// instruction latency: loads are issued together and reductions use independent accumulators.

// Row maximum over the first K fp32 columns of this thread's TMEM lane (kc = ceil(K/32) chunks
// of 32 columns, read two chunks per wait).
__device__ __forceinline__ float row_max(uint32_t taddr, int K, int kc)
{
    float m[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) m[u] = NEG_BIG;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < kc) {
            uint32_t ra[32];
            tmem_ld32(taddr + 32 * c, ra);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if ((c + 1) * 32 <= K || 32 * c + j < K) m[j & 7] = fmaxf(m[j & 7], __uint_as_float(ra[j]));
        }
    }
    return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

// exp2(L - m) of one chunk of 32 columns (0 beyond K), in place; returns the chunk's sum.
__device__ __forceinline__ float chunk_exp(uint32_t (&r)[32], int c, int K, float m)
{
    const bool full = (c + 1) * 32 <= K;
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float e = (full || 32 * c + j < K) ? ex2(__uint_as_float(r[j]) - m) : 0.f;
        r[j] = __float_as_uint(e);
        s[j & 3] += e;
    }
    return (s[0] + s[1]) + (s[2] + s[3]);
}

// Elementwise product of two bf16 pairs, rounded to nearest.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t pk2(uint32_t a, uint32_t b, float sc)
{
    return pack_bf16(__uint_as_float(a) * sc, __uint_as_float(b) * sc);
}

// Key side: Gamma_K row k = softmax of the TMEM logits at tl, normalised (zeros when not valid),
// as bf16 into the K-major SW128 tile gk; the exponentials of the row are held in registers as
// bf16 pairs until the row sum is known, so each tile element is written once.
__device__ __forceinline__ void key_softmax_reg(uint32_t tl, int K, int kc, bool valid, uint8_t *gk, int k)
{
    const float m = row_max(tl, K, kc);
    float sum = 0.f;
    uint32_t pk[64];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < kc) {
            uint32_t r[32];
            tmem_ld32(tl + 32 * c, r);
            tmem_ld_wait();
            sum += chunk_exp(r, c, K, m);
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[16 * c + j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        }
    }
    const float scf = valid ? 1.0f / sum : 0.f;
    const uint32_t sc2 = pack_bf16(scf, scf);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < kc) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t *e = pk + 16 * c + 4 * q;
                *reinterpret_cast<uint4 *>(gk + sw128(k, 4 * c + q, C)) =
                    make_uint4(mul_bf16x2(e[0], sc2), mul_bf16x2(e[1], sc2), mul_bf16x2(e[2], sc2), mul_bf16x2(e[3], sc2));
            }
        }
    }
}

// Output rows, components in tiles (more than 128 in all): this tile's numerator row (d_v columns
// of TMEM at tl) and its normaliser den_eps (the tile's E_Q . Z (+ masked P sums), plus eps times
// its E_Q row sum) go to the fp32 partial sums part [rows][d_v] and pden [rows]: the first tile
// (pmode 1) writes them, every later one adds to them with reductions in L2 (no value comes back,
// so nothing waits on the round trip); a last kernel divides.  Every lane loads (warp-collective).
__device__ __forceinline__ void tile_partial_row(uint32_t tl, int d_v, float den_eps, bool valid, float *part,
                                                 float *pden, long long orow, int pmode)
{
    float *pr = part + orow * d_v;
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
        float4 *p4 = reinterpret_cast<float4 *>(pr + col0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (4 * q >= ncol) continue;
            const float4 v = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                         __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            if (pmode == 1)
                p4[q] = v;
            else
                atomicAdd(p4 + q, v);   // (result unused: a reduction in L2)
        }
    }
    if (valid) {
        if (pmode == 1)
            pden[orow] = den_eps;
        else
            atomicAdd(pden + orow, den_eps);
    }
}

// Key side, components in tiles (more than 128 in all): Gamma_K row k of this tile is
// exp2(L - lse) with lse the row's log2-sum-exp over every component (zeros beyond the tile's K
// components and for rows past the sequence), as bf16 into the K-major SW128 tile gk.
__device__ __forceinline__ void key_gamma_lse(uint32_t tl, int K, int kc, bool valid, uint8_t *gk, int k, float lse)
{
    const float on = valid ? 1.f : 0.f;
#pragma unroll 1
    for (int c = 0; c < kc; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        const bool full = (c + 1) * 32 <= K;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int j = 8 * q + 2 * h;
                const float e0 = (full || 32 * c + j < K) ? ex2(__uint_as_float(r[j]) - lse) * on : 0.f;
                const float e1 = (full || 32 * c + j + 1 < K) ? ex2(__uint_as_float(r[j + 1]) - lse) * on : 0.f;
                w[h] = pack_bf16(e0, e1);
            }
            *reinterpret_cast<uint4 *>(gk + sw128(k, 4 * c + q, C)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int DR>
__device__ __forceinline__ void issue_logits_c(uint32_t d, uint32_t abuf, uint32_t bimg, uint32_t bconst,
                                               uint32_t ax, int kn16)
{
    constexpr int KA = DR * 2 < 64 ? 64 : DR * 2;
    const uint32_t id = idesc_f16(128, (uint32_t)kn16, 0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < KA / 16; ++s) mma_f16(d, kdesc(abuf, s, C), kdesc(bimg, s, kn16), id, s > 0);
    mma_f16(d, kdesc32(ax), kdesc32(bconst), id, 1u);   // + per-component constant
}

}  // namespace
}  // namespace tck
}  // namespace gma
