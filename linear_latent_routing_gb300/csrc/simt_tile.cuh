// simt_tile.cuh -- register-tiled fp32 products over shared-memory tiles, for the CUDA-core
// kernels (the backward pass and the fp32 family's segment memories).
//
// A block of BT = 256 threads forms a 16 x 16 grid; each thread holds 4 rows x (W / 16) columns of
// a 64-row output W columns wide (W = 16, 32, 64 or 128).  Both operands are staged in shared
// memory with the contracted index as their row, so that one step of a product is one 16-byte
// load of four rows of A, one or two loads of B and 4 W / 16 FMAs, summed in the order of the
// contracted index.
#pragma once
#include <type_traits>
#include "gma_internal.cuh"

namespace gma {
namespace tile {

constexpr int BT = 256;   // threads per block
constexpr int LT = 68;    // row stride of a transposed tile 64 wide (a multiple of 4 for 16-byte
                          // loads, not of 8, which spreads its column-wise writes over the banks)

// The 16 x 16 grid: thread (ty, tx) = (t / 16, t % 16) holds rows 4 ty .. 4 ty + 3 and columns of
// group tx; a warp covers 2 ty x 16 tx, so the 16 threads of a row are one half-warp.  (A layout
// of 8 ty x 4 tx per warp reads fewer shared-memory bytes per step but needs its row sums across
// warps; measured slower.)
__device__ __forceinline__ int tile_ty() { return threadIdx.x >> 4; }
__device__ __forceinline__ int tile_tx() { return threadIdx.x & 15; }

// The thread's first output row and its c-th output column in an output W columns wide: groups
// of four contiguous columns (two groups 64 apart at W = 128), narrower strips below 64.
__device__ __forceinline__ int orow() { return tile_ty() * 4; }
template <int W>
__device__ __forceinline__ int ocol(int c)
{
    const int tx = tile_tx();
    if constexpr (W == 128) return (c >> 2) * 64 + tx * 4 + (c & 3);
    else return tx * (W / 16) + c;
}

// The thread's W / 16 columns of one staged row.
template <int W>
__device__ __forceinline__ void ld_cols(float (&b)[W / 16], const float *row)
{
    const int tx = tile_tx();
    if constexpr (W == 16) {
        b[0] = row[tx];
    } else if constexpr (W == 32) {
        const float2 v = *reinterpret_cast<const float2 *>(row + 2 * tx);
        b[0] = v.x;
        b[1] = v.y;
    } else {
#pragma unroll
        for (int g = 0; g < W / 64; ++g) {
            const float4 v = *reinterpret_cast<const float4 *>(row + 64 * g + 4 * tx);
            b[4 * g] = v.x;
            b[4 * g + 1] = v.y;
            b[4 * g + 2] = v.z;
            b[4 * g + 3] = v.w;
        }
    }
}

// acc[r][c] += sum_{q0 <= q < q1} At[q][orow() + r] * Bt[q][ocol<W>(c)]: both operands in shared
// memory with the contracted index as their row (row strides lda, ldb floats, multiples of 4).  A
// thread whose rows see only part of a triangular operand passes that part's range.
template <int W>
__device__ __forceinline__ void mac_range(float (&acc)[4][W / 16], const float *At, int lda, const float *Bt,
                                          int ldb, int q0, int q1)
{
    const int r0 = orow();
#pragma unroll 4
    for (int q = q0; q < q1; ++q) {
        const float4 a = *reinterpret_cast<const float4 *>(At + q * lda + r0);
        float b[W / 16];
        ld_cols<W>(b, Bt + q * ldb);
#pragma unroll
        for (int c = 0; c < W / 16; ++c) {
            acc[0][c] = fmaf(a.x, b[c], acc[0][c]);
            acc[1][c] = fmaf(a.y, b[c], acc[1][c]);
            acc[2][c] = fmaf(a.z, b[c], acc[2][c]);
            acc[3][c] = fmaf(a.w, b[c], acc[3][c]);
        }
    }
}

// The whole contraction, q < nq.
template <int W>
__device__ __forceinline__ void mac(float (&acc)[4][W / 16], const float *At, int lda, const float *Bt, int ldb,
                                    int nq)
{
    mac_range<W>(acc, At, lda, Bt, ldb, 0, nq);
}

template <int W>
__device__ __forceinline__ void zero(float (&acc)[4][W / 16])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < W / 16; ++c) acc[r][c] = 0.f;
}

// dst[r][c] = src[r * sld + c] for r < 64, c < C (zero where r >= nr or c >= nc; those elements of
// src are not read); dst has row stride ld.  Lanes run along c: coalesced reads, conflict-free
// writes.  A thread keeps one column and steps its row by BT / C; the loop is unrolled, so that the
// thread's 64 C / BT loads are all in flight before the first store.
template <int C, typename T>
__device__ __forceinline__ void stage(float *dst, int ld, const T *src, long long sld, int nr, int nc)
{
    static_assert(BT % C == 0, "a thread keeps one column");
    constexpr int STEP = BT / C, PER = 64 / STEP;
    const int c = threadIdx.x % C, r0 = threadIdx.x / C;
    const T *p = src + (long long)r0 * sld + c;
    float v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) v[u] = (r0 + u * STEP < nr && c < nc) ? to_f32(p[(long long)u * STEP * sld]) : 0.f;
#pragma unroll
    for (int u = 0; u < PER; ++u) dst[(r0 + u * STEP) * ld + c] = v[u];
}

// stage in two halves, so that the loads of the next tile can be in flight during a product: the
// thread's elements into registers, then into shared memory.
template <int C>
struct Staged {
    static constexpr int PER = 64 * C / BT;
    float v[PER];
};

template <int C, typename T>
__device__ __forceinline__ void stage_load(Staged<C> &s, const T *src, long long sld, int nr, int nc)
{
    constexpr int STEP = BT / C;
    const int c = threadIdx.x % C, r0 = threadIdx.x / C;
    const T *p = src + (long long)r0 * sld + c;
#pragma unroll
    for (int u = 0; u < Staged<C>::PER; ++u)
        s.v[u] = (r0 + u * STEP < nr && c < nc) ? to_f32(p[(long long)u * STEP * sld]) : 0.f;
}

template <int C>
__device__ __forceinline__ void stage_store(float *dst, int ld, const Staged<C> &s)
{
    constexpr int STEP = BT / C;
    const int c = threadIdx.x % C, r0 = threadIdx.x / C;
#pragma unroll
    for (int u = 0; u < Staged<C>::PER; ++u) dst[(r0 + u * STEP) * ld + c] = s.v[u];
}

// The transpose: dst[c][r] = src[r * sld + c], dst with row stride ld.
template <int C, typename T>
__device__ __forceinline__ void stage_t(float *dst, int ld, const T *src, long long sld, int nr, int nc)
{
    static_assert(BT % C == 0, "a thread keeps one column");
    constexpr int STEP = BT / C, PER = 64 / STEP;
    const int c = threadIdx.x % C, r0 = threadIdx.x / C;
    const T *p = src + (long long)r0 * sld + c;
    float v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) v[u] = (r0 + u * STEP < nr && c < nc) ? to_f32(p[(long long)u * STEP * sld]) : 0.f;
#pragma unroll
    for (int u = 0; u < PER; ++u) dst[c * ld + r0 + u * STEP] = v[u];
}

// Zero and element-wise sum of a float or a float4 (the scans' vectors).
template <typename V>
__device__ __forceinline__ V vzero();
template <>
__device__ __forceinline__ float vzero<float>() { return 0.f; }
template <>
__device__ __forceinline__ float4 vzero<float4>() { return make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ float vadd(float a, float b) { return a + b; }
__device__ __forceinline__ float4 vadd(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }

// v[r] (the thread's partial for its row orow() + r) becomes the sum over the 16 threads of that row
// (a half-warp: shuffles over lanes xor 1, 2, 4, 8).
__device__ __forceinline__ void row_sums(float (&v)[4])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
}

}  // namespace tile
}  // namespace gma
