// gma_tc_causal.cu -- the chunked causal GMA kernel (tcgen05, sm_103a), warp-specialised.
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §3 (causal variant: the latent memory and its normaliser become prefix sums, so
// row i of O sees keys j <= i) on top of §1 (posterior responsibilities) and §2 (write phase,
// read phase O = Gamma_Q V~ / (Gamma_Q Z + eps)).
//
// One CTA handles one segment of one (batch, head) slice, starting from the segment's exclusive
// prefix memory S_start (V~ part and Z part), in chunks of C = 128 tokens.  With E_K = exp2 of the
// key logits minus their row maximum, r_j = 1 / (row sum of E_K) (so Gamma_K = diag(r) E_K), and
// E_Q the same for the queries (row sums s_i, kept unnormalised):
//   V'     = diag(r) V_c                             (value rows scaled in shared memory)
//   P      = E_Q E_K^T                               (tensor cores, fp32 in TMEM)
//   O_num  = E_Q S_{c-1} + tril(P) V'                (tensor cores)
//   den    = E_Q . Z_{c-1} + sum_{j<=i} P_ij r_j     (CUDA cores, fp32)
//   O      = O_num / (den + eps * s)
//   S_c    = S_{c-1} + E_K^T V'                      (tensor cores, fp32 in TMEM)
//   Z_c    = Z_{c-1} + E_K^T r                       (CUDA cores, fp32)
//
// Warp roles (416 threads):
//   warps 0-3   key side:   [x^2, x] of the keys (in place in the TMA-filled A tile), E_K into
//                           shared memory with r, the value rows scaled by r;
//   warps 4-7   query side: [x^2, x] of the queries, E_Q (bf16, back into TMEM as the A operand),
//                           its row sums and E_Q . Z, causal mask of P (bf16, back into TMEM);
//   warps 8-11  state/out:  the starting memory, Z_c, the bf16 operand copy of S_c, and the
//                           output rows (numerator from TMEM divided by the normaliser);
//   warp 12     control:    TMA of the routing rows and value tiles, and every tcgen05.mma,
//                           issued as soon as its operands are ready (mbarrier handshakes).
// Tensor memory (512 columns): [0,128) key logits, then P; [128,256) query logits, then E_Q;
// [256,384) output numerator; [384,512) the running memory S.
// Every wait is bounded; a timeout records GMA_ERR_TIMEOUT and makes all roles leave their loops.
//
// Single-launch variant (FUSED): the CTAs take their segments from a ticket counter (all slices'
// first segments, then their second ones, ...), and each computes its own segment memory before
// the sweep above:
//   sweep 1:  S_own = sum over the segment's chunks of E_K^T V' (tensor cores, TMEM [384,512)),
//             Z_own = sum of E_K^T r (CUDA cores), with two key-row and value buffers (the query
//             tile and the S operand tile are free until sweep 2);
//   look-back: S_own is published; the exclusive prefix S_start is summed backwards over the
//             published memories of the preceding segments of the slice, into TMEM [256,384),
//             until a segment whose inclusive prefix is published; S_start + S_own is then
//             published as this segment's inclusive prefix;
//   sweep 2:  the chunk loop above, from S_start held in TMEM.
// The key responsibilities never leave the chip; the memories pass through global memory (L2).
// A CTA only waits on segments with an earlier ticket, which are resident or finished, so the
// waits always end; they are bounded all the same, and a segment that fails publishes that, so
// that its successors stop waiting for it.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

constexpr int CTHREADS = 416;   // key side 0-3, query side 4-7, state/output 8-11, control 12
enum BarId {
    B_BIMG, B_V, B_XK, B_XQ,                                  // TMA (transaction counts)
    B_AK, B_AQ, B_GK, B_VS, B_GQ, B_PS, B_ZP, B_SP, B_OF,     // 128 threads of one role
    B_LK, B_LQ, B_S, B_PQ, B_PV,                              // tcgen05.commit
    NBAR
};
// Sweep 1 of the single-launch variant: key rows and value tiles of chunk c in buffer c & 1.
enum FBar {
    F_X0 = NBAR, F_X1, F_V0, F_V1,   // TMA (transaction counts)
    F_AK, F_GK, F_VS, F_ZP,          // 128 threads of one role
    F_LK0, F_LK1, F_S,               // tcgen05.commit
    F_END
};
constexpr uint32_t R_LK = 0, R_LQ = 128, R_O = 256, R_S = 384;
static_assert(KMAX == C, "the S operand tile doubles as a value buffer in sweep 1");

// Segment memories of the single-launch variant, exchanged between CTAs (global memory).
struct LookBack {
    int *ticket;    // one counter, zero before the launch: segments in start order
    int *flag;      // [BH][nseg]: 0 nothing yet, 1 own memory, 2 inclusive prefix, 3 failed
    float *own;     // [BH][nseg][KMAX][ne]: the segment's own memory (d_v columns, Z at d_v)
    float *incl;    // [BH][nseg][KMAX][ne]: the memory of the slice's segments up to this one
};

struct CausalSmem {
    uint32_t bimg, ax, abk, abq, gk, sp, ve, zbuf, zpart, rbuf, dsm, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ CausalSmem(int DR, int kn16, int d_v)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        const uint32_t tile = ka / 64u * 128u;
        uint32_t o = 0;
        bimg = o; o = al(o + tile * (uint32_t)kn16 + 32u * (uint32_t)kn16);
        ax = o; o = al(o + (uint32_t)C * 32u);
        abk = o; o = al(o + (uint32_t)C * DR * 4u);   // keys [x^2 | x]
        abq = o; o = al(o + (uint32_t)C * DR * 4u);   // queries [x^2 | x]
        gk = o; o = al(o + 2u * C * 128u);
        sp = o; o = al(o + (uint32_t)d_v * KMAX * 2u);
        ve = o; o = al(o + (uint32_t)d_v * C * 2u);
        zbuf = o; o += 2u * KMAX * 4u;        // Z_{c-1} by chunk parity
        zpart = o; o += 2u * 8u * KMAX * 4u;  // partial column sums by chunk parity
        rbuf = o; o += (uint32_t)C * 4u;      // r of the chunk's keys
        dsm = o; o += 2u * C * 8u;            // (row sum, normaliser) per query row, by chunk parity
        bars = o; o += F_END * 8u;
        misc = o; o += 16u;   // TMEM base, abort word, ticket, look-back broadcast
        total = o;
    }
};

// Key side: E_K row k = exp2(L - row max) (bf16; 0 beyond K) into the K-major SW128 tile gk;
// returns the row sum of the fp32 values.
__device__ __forceinline__ float key_exp(uint32_t tl, int K, int kc, uint8_t *gk, int k)
{
    const float m = row_max(tl, K, kc);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < kc) {
            uint32_t r[32];
            tmem_ld32(tl + 32 * c, r);
            tmem_ld_wait();
            sum += chunk_exp(r, c, K, m);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = 8 * q;
                *reinterpret_cast<uint4 *>(gk + sw128(k, 4 * c + q, C)) =
                    make_uint4(pk2(r[e], r[e + 1], 1.f), pk2(r[e + 2], r[e + 3], 1.f),
                               pk2(r[e + 4], r[e + 5], 1.f), pk2(r[e + 6], r[e + 7], 1.f));
            }
        }
    }
    return sum;
}

// Key side: value row k of the chunk (MN-major SW32 blocks of 16 columns) times r, in place.
__device__ __forceinline__ void scale_v_row(uint8_t *ve, int k, int d_v, float r)
{
    const uint32_t r2 = pack_bf16(r, r);
    for (int b = 0; b < d_v / 16; ++b) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint4 *p = reinterpret_cast<uint4 *>(ve + sw32(k, b, hf, C));
            const uint4 v = *p;
            *p = make_uint4(mul_bf16x2(v.x, r2), mul_bf16x2(v.y, r2), mul_bf16x2(v.z, r2), mul_bf16x2(v.w, r2));
        }
    }
}

// State side: row k of the running memory S (d_v fp32 columns of TMEM at tl) as bf16 into the
// MN-major SW32 operand tile sp.
__device__ __forceinline__ void state_readout(uint32_t tl, int d_v, uint8_t *sp, int k)
{
    for (int b0 = 0; b0 < d_v / 16; b0 += 4) {   // 64 columns per wait
        uint32_t ra[32], rb[32];
        if (d_v == 16) {
            uint32_t r16[16];
            tmem_ld16(tl, r16);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) ra[j] = r16[j];
        } else {
            tmem_ld32(tl + 16 * b0, ra);
            if (b0 + 2 < d_v / 16) tmem_ld32(tl + 16 * b0 + 32, rb);
            tmem_ld_wait();
        }
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            const int b = b0 + bb;
            if (b < d_v / 16) {
                uint32_t r[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) r[j] = bb < 2 ? ra[16 * bb + j] : rb[16 * (bb - 2) + j];
                const uint4 lo = make_uint4(pk2(r[0], r[1], 1.f), pk2(r[2], r[3], 1.f),
                                            pk2(r[4], r[5], 1.f), pk2(r[6], r[7], 1.f));
                const uint4 hi = make_uint4(pk2(r[8], r[9], 1.f), pk2(r[10], r[11], 1.f),
                                            pk2(r[12], r[13], 1.f), pk2(r[14], r[15], 1.f));
                *reinterpret_cast<uint4 *>(sp + sw32(k, b, 0, KMAX)) = lo;
                *reinterpret_cast<uint4 *>(sp + sw32(k, b, 1, KMAX)) = hi;
            }
        }
    }
}

// State side: this thread's share of Z_c - Z_{c-1} = E_K^T r: components 8q..8q+7 over the rows
// g, g+8, ..., g+120 of the chunk (t = 16 g + q), into zp[g][8q .. 8q+7].
__device__ __forceinline__ void colsum_part(const uint8_t *gk, const float *rb, float *zp, int t)
{
    const int q = t & 15, g = t >> 4;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int u = 0; u < C / 8; ++u) {
        const int j = g + 8 * u;
        const uint4 v = *reinterpret_cast<const uint4 *>(gk + sw128(j, q, C));
        const float r = rb[j];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(__uint_as_float(w[e] << 16), r, acc[2 * e]);
            acc[2 * e + 1] = fmaf(__uint_as_float(w[e] & 0xFFFF0000u), r, acc[2 * e + 1]);
        }
    }
    float4 *o = reinterpret_cast<float4 *>(zp + g * KMAX + 8 * q);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// Query side: unnormalised E_Q of this row (zeros when not valid) back into TMEM at tl as bf16
// pairs; returns (row sum of the fp32 values, E_Q . z) with z the fp32 normaliser Z_{c-1}.
__device__ __forceinline__ float2 query_softmax(uint32_t tl, int K, int kc, bool valid, const float *z)
{
    const float m = row_max(tl, K, kc);
    const float sc = valid ? 1.f : 0.f;
    const float4 *z4 = reinterpret_cast<const float4 *>(z);
    float srow = 0.f, den = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c < kc) {
            uint32_t r[32];
            tmem_ld32(tl + 32 * c, r);
            tmem_ld_wait();
            srow += chunk_exp(r, c, K, m);
            float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 zz = z4[8 * c + q];
                d4[0] = fmaf(__uint_as_float(r[4 * q]), zz.x, d4[0]);
                d4[1] = fmaf(__uint_as_float(r[4 * q + 1]), zz.y, d4[1]);
                d4[2] = fmaf(__uint_as_float(r[4 * q + 2]), zz.z, d4[2]);
                d4[3] = fmaf(__uint_as_float(r[4 * q + 3]), zz.w, d4[3]);
            }
            den += (d4[0] + d4[1]) + (d4[2] + d4[3]);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pk2(r[2 * j], r[2 * j + 1], sc);
            tmem_st16(tl + 16 * c, w);   // E_Q (bf16 pairs), in place
        }
    }
    tmem_st_wait();
    return make_float2(srow, den);
}

// Query side: row i of P (fp32 in TMEM at tl) masked to columns j <= i, written back as bf16
// pairs in place; returns sum_{j<=i} P_ij r_j.
__device__ __forceinline__ float causal_mask(uint32_t tl, int i, const float *rb)
{
    const float4 *r4 = reinterpret_cast<const float4 *>(rb);
    float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 rr = r4[8 * c + q];
            const int col = 32 * c + 4 * q;
            const float p0 = col <= i ? __uint_as_float(r[4 * q]) : 0.f;
            const float p1 = col + 1 <= i ? __uint_as_float(r[4 * q + 1]) : 0.f;
            const float p2 = col + 2 <= i ? __uint_as_float(r[4 * q + 2]) : 0.f;
            const float p3 = col + 3 <= i ? __uint_as_float(r[4 * q + 3]) : 0.f;
            d4[0] = fmaf(p0, rr.x, d4[0]);
            d4[1] = fmaf(p1, rr.y, d4[1]);
            d4[2] = fmaf(p2, rr.z, d4[2]);
            d4[3] = fmaf(p3, rr.w, d4[3]);
            w[2 * q] = pack_bf16(p0, p1);
            w[2 * q + 1] = pack_bf16(p2, p3);
        }
        tmem_st16(tl + 16 * c, w);
    }
    tmem_st_wait();
    return (d4[0] + d4[1]) + (d4[2] + d4[3]);
}

// Output side: output row orow = (d_v numerator columns of TMEM at tl) * inv, bf16 or fp32.
__device__ __forceinline__ void write_output(uint32_t tl, int d_v, float inv, bool valid, void *O,
                                          long long orow, int out_f32)
{
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

// ------------------------------------------------------------------ look-back (FUSED)
__device__ __forceinline__ int flag_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void flag_release(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A predecessor's flag once it is set (1 or 2), or 3 if it failed, this CTA is aborting, or the
// wait ran out (recorded as a timeout).
__device__ __forceinline__ int wait_flag(const int *p, WsHeader *hdr, volatile int *abort)
{
    int v = flag_acquire(p);
    if (v) return v;
    const long long t0 = clock64();
    while (true) {
        __nanosleep(100);
        v = flag_acquire(p);
        if (v) return v;
        if (*abort) return 3;
        if (wait_expired(clock64() - t0, hdr)) {
            record_error(hdr, GMA_ERR_TIMEOUT, 130);
            return 3;
        }
    }
}

// Row k of a memory, d_v fp32 columns of TMEM at tl plus its Z entry z, into the global row dst.
__device__ __forceinline__ void row_to_global(uint32_t tl, int d_v, float z, float *dst)
{
    for (int b = 0; b < d_v / 16; ++b) {
        uint32_t r[16];
        tmem_ld16(tl + 16 * b, r);
        tmem_ld_wait();
        float4 *o4 = reinterpret_cast<float4 *>(dst + 16 * b);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o4[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
    }
    dst[d_v] = z;
}

// TMEM row at tl (d_v fp32 columns) = (first ? 0 : itself) + the sum of the published rows k of
// the n segments in list (entry 2 j + 1: segment j's inclusive prefix, 2 j: its own memory; slot0
// = the slice's first segment); returns the sum of their Z entries.  The rows were published by
// other CTAs: read through L2, four segments' loads in flight at a time.
__device__ __forceinline__ float rows_add_list(uint32_t tl, int d_v, const int *list, int n, const LookBack &lb,
                                               size_t slot0, int k, int ne, bool first)
{
    for (int b = 0; b < d_v / 16; ++b) {
        uint32_t r[16];
        if (first) {
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = 0u;
        } else {
            tmem_ld16(tl + 16 * b, r);
            tmem_ld_wait();
        }
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = __uint_as_float(r[j]);
#pragma unroll 4
        for (int i = 0; i < n; ++i) {
            const int e = list[i];
            const float4 *s4 = reinterpret_cast<const float4 *>(
                ((e & 1) ? lb.incl : lb.own) + ((slot0 + (size_t)(e >> 1)) * KMAX + k) * ne + 16 * b);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = __ldcg(s4 + q);
                acc[4 * q] += f.x;
                acc[4 * q + 1] += f.y;
                acc[4 * q + 2] += f.z;
                acc[4 * q + 3] += f.w;
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(acc[j]);
        tmem_st16(tl + 16 * b, r);
    }
    tmem_st_wait();
    float z = 0.f;
    for (int i = 0; i < n; ++i) {
        const int e = list[i];
        z += __ldcg(((e & 1) ? lb.incl : lb.own) + ((slot0 + (size_t)(e >> 1)) * KMAX + k) * ne + d_v);
    }
    return z;
}

// TMEM row at tl (d_v fp32 columns) = 0.
__device__ __forceinline__ void row_zero(uint32_t tl, int d_v)
{
    uint32_t r[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = 0u;
    for (int b = 0; b < d_v / 16; ++b) tmem_st16(tl + 16 * b, r);
    tmem_st_wait();
}

// Global row dst = TMEM rows at ta + tb (d_v fp32 columns each) and Z entry z.
__device__ __forceinline__ void rows_sum_to_global(uint32_t ta, uint32_t tb, int d_v, float z, float *dst)
{
    for (int b = 0; b < d_v / 16; ++b) {
        uint32_t ra[16], rb[16];
        tmem_ld16(ta + 16 * b, ra);
        tmem_ld16(tb + 16 * b, rb);
        tmem_ld_wait();
        float4 *o4 = reinterpret_cast<float4 *>(dst + 16 * b);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o4[q] = make_float4(__uint_as_float(ra[4 * q]) + __uint_as_float(rb[4 * q]),
                                __uint_as_float(ra[4 * q + 1]) + __uint_as_float(rb[4 * q + 1]),
                                __uint_as_float(ra[4 * q + 2]) + __uint_as_float(rb[4 * q + 2]),
                                __uint_as_float(ra[4 * q + 3]) + __uint_as_float(rb[4 * q + 3]));
    }
    dst[d_v] = z;
}

}  // namespace

template <int DR, bool FUSED>
__global__ void __launch_bounds__(CTHREADS, 1) tc_causal_pipelined_kernel(const Args a,
                                                                          const __grid_constant__ CUtensorMap vmap,
                                                                          const __grid_constant__ CUtensorMap kmap,
                                                                          const __grid_constant__ CUtensorMap qmap,
                                                                          const LookBack lb)
{
    grid_dependency_wait();   // the scanned memories (or, FUSED, the parameter tables) come from the kernels before
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const CausalSmem L(DR, a.kn16, a.d_v);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.misc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.misc + 4);
    float *zbuf = reinterpret_cast<float *>(smem + L.zbuf);
    float *zpart = reinterpret_cast<float *>(smem + L.zpart);
    float *rbuf = reinterpret_cast<float *>(smem + L.rbuf);
    float2 *dsm = reinterpret_cast<float2 *>(smem + L.dsm);
    volatile int *tkslot = reinterpret_cast<volatile int *>(smem + L.misc + 8);
    volatile int *lbcast = reinterpret_cast<volatile int *>(smem + L.misc + 12);
    const int t = threadIdx.x, warp = t >> 5;
    const int d_v = a.d_v;
    const int kc = (a.K + 31) >> 5;
    constexpr uint32_t XT = (uint32_t)C * DR * 2;   // bytes of one [x] tile (the TMA destination)

    // ---------------------------------------------------------------- set-up (all threads)
    if (FUSED && t == 0) *tkslot = atomicAdd(lb.ticket, 1);
    if (warp == 12) {
        if (t == 384) {
            static const uint32_t counts[F_END] = {1,   1,   1,   1,   128, 128, 128, 128, 128,
                                                   128, 128, 128, 128, 1,   1,   1,   1,   1,
                                                   1,   1,   1,   1,   128, 128, 128, 128, 1, 1, 1};
            const int nb = FUSED ? (int)F_END : (int)NBAR;
            for (int i = 0; i < nb; ++i) mbar_init(bars + i, counts[i]);
            *abort = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(tslot, 512);
    } else if (warp < 4) {
        // E_K tile: components the exponentials never write must read as zero
        for (uint32_t o = t * 16; o < 2u * C * 128u; o += 128 * 16)
            *reinterpret_cast<uint4 *>(smem + L.gk + o) = make_uint4(0, 0, 0, 0);
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
    // the segment: by block index, or (FUSED) by ticket, segment-major (ticket = seg * BH + bh), so
    // that the segments running at once spread over all slices and each one's look-back meets an
    // inclusive prefix within a few steps
    const int nbh = (int)gridDim.x / a.nseg;
    const int tk = FUSED ? *tkslot : (int)blockIdx.x;
    const int bh = FUSED ? tk % nbh : tk / a.nseg, seg = FUSED ? tk / nbh : tk % a.nseg, h = bh % a.H;
    const int tok0 = seg * a.cps * C;
    const int tok_end = min(a.N, tok0 + a.cps * C);
    const int nch = (tok_end - tok0 + C - 1) / C;

    float zexcl = 0.f;   // FUSED, state side: the Z entry of this row of S_start
    if constexpr (FUSED) {
        // ============================================================ sweep 1 and look-back
        uint8_t *const xb0 = smem + L.abk, *const xb1 = smem + L.abq;   // key rows by chunk parity
        uint8_t *const vb0 = smem + L.ve, *const vb1 = smem + L.sp;     // value tiles by chunk parity
        if (warp == 12) {
            if (t == 384) {
                const uint32_t id_s = idesc_f16(128, (uint32_t)d_v, 1, 1, 1, 1);
                int last_s = -1, last_x[2] = {-1, -1};
                auto load = [&](int c) {
                    const int b = c & 1;
                    load_x_tile((b ? xb1 : xb0) + XT, &kmap, bars + F_X0 + b, DR, tok0 + c * C, bh);
                    load_v_chunk(b ? vb1 : vb0, &vmap, bars + F_V0 + b, d_v, tok0 + c * C, bh);
                    last_x[b] = c;
                };
                mbar_arrive_expect_tx(bars + B_BIMG, (uint32_t)a.bimg_bytes);
                bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars + B_BIMG);
                for (int c = 0; c < 2 && c < nch; ++c) load(c);
                bool ok = mbar_wait_abortable(bars + B_BIMG, 0, a.hdr, 100, abort);
                const uint32_t bimg = sb + L.bimg, bconst = sb + L.bimg + (uint32_t)a.bimg_main_bytes;
                // S_own += E_K^T V' of chunk j; the chunk's buffers then take chunk j + 2 (its key
                // rows were read by its logits, complete before its E_K was written)
                auto update = [&](int j) -> bool {
                    if (!mbar_wait_abortable(bars + F_GK, j & 1, a.hdr, 101, abort)) return false;
                    if (!mbar_wait_abortable(bars + F_VS, j & 1, a.hdr, 102, abort)) return false;
                    tc_fence_after();
                    const uint32_t vb = sb + ((j & 1) ? L.sp : L.ve);
                    for (int s = 0; s < C / 16; ++s)
                        mma_f16(tmem + R_S, mn128desc(sb + L.gk, s, C), mn32desc(vb, s, C), id_s,
                                (j > 0 || s > 0) ? 1u : 0u);
                    mma_commit(bars + F_S);
                    last_s = j;
                    if (j + 2 < nch) {
                        if (!mbar_wait_abortable(bars + F_S, j & 1, a.hdr, 103, abort)) return false;
                        load(j + 2);
                    }
                    return true;
                };
                for (int c = 0; ok && c < nch; ++c) {
                    const int b = c & 1;
                    if (!(ok = mbar_wait_abortable(bars + F_AK, c & 1, a.hdr, 104, abort))) break;
                    tc_fence_after();
                    issue_logits_x<DR>(tmem + (b ? R_LQ : R_LK), sb + (b ? L.abq : L.abk), bimg, bconst, sb + L.ax,
                                       a.kn16);
                    mma_commit(bars + F_LK0 + b);
                    if (c >= 1 && !(ok = update(c - 1))) break;
                }
                if (ok && nch > 0) ok = update(nch - 1);
                // drain: the last update, and loads still in flight (only after a timeout)
                if (last_s >= 0) mbar_wait(bars + F_S, last_s & 1, a.hdr, 105);
                for (int b = 0; b < 2; ++b)
                    if (last_x[b] >= 0) {
                        mbar_wait(bars + F_X0 + b, (last_x[b] >> 1) & 1, a.hdr, 106);
                        mbar_wait(bars + F_V0 + b, (last_x[b] >> 1) & 1, a.hdr, 106);
                    }
            }
        } else if (warp < 4) {
            // key side: [x^2, x], E_K and r, V' = diag(r) V
            const int k = t;
            const uint32_t lane = tmem + ((uint32_t)(warp * 32) << 16);
            for (int c = 0; c < nch; ++c) {
                const int b = c & 1;
                const uint32_t pb = (c >> 1) & 1;
                if (!mbar_wait_abortable(bars + F_X0 + b, pb, a.hdr, 110, abort)) break;
                build_inplace<DR>(b ? xb1 : xb0, k);
                fence_proxy_async_smem();
                // (a test of the timeout path withholds the first segment's first signal: that
                // segment's waits run out, and its successors learn of it by the look-back)
                if (!(a.test_withhold && seg == 0 && c == 0)) mbar_arrive(bars + F_AK);
                if (!mbar_wait_abortable(bars + F_LK0 + b, pb, a.hdr, 111, abort)) break;
                if (c >= 1) {
                    // E_K and r are free once the previous update and column sums have read them
                    if (!mbar_wait_abortable(bars + F_S, (c - 1) & 1, a.hdr, 112, abort)) break;
                    if (!mbar_wait_abortable(bars + F_ZP, (c - 1) & 1, a.hdr, 113, abort)) break;
                }
                tc_fence_after();
                const float sum = key_exp(lane + (b ? R_LQ : R_LK), a.K, kc, smem + L.gk, k);
                const float r = tok0 + c * C + k < tok_end ? 1.0f / sum : 0.f;
                rbuf[k] = r;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bars + F_GK);
                if (!mbar_wait_abortable(bars + F_V0 + b, pb, a.hdr, 114, abort)) break;
                scale_v_row(b ? vb1 : vb0, k, d_v, r);
                fence_proxy_async_smem();
                mbar_arrive(bars + F_VS);
            }
        } else if (warp >= 8) {
            // state side: Z_own, then the publication of S_own and the look-back
            const int k = t - 256;
            const uint32_t lane = tmem + ((uint32_t)((warp - 8) * 32) << 16);
            float zown = 0.f;
            bool ok = true;
            for (int c = 0; c < nch; ++c) {
                if (!(ok = mbar_wait_abortable(bars + F_GK, c & 1, a.hdr, 120, abort))) break;
                float *zp = zpart + (c & 1) * 8 * KMAX;
                colsum_part(smem + L.gk, rbuf, zp, k);
                mbar_arrive(bars + F_ZP);
                if (!(ok = mbar_wait_abortable(bars + F_ZP, c & 1, a.hdr, 121, abort))) break;
                float zs = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) zs += zp[g * KMAX + k];
                zown += zs;
            }
            if (ok) ok = nch > 0 && mbar_wait_abortable(bars + F_S, (nch - 1) & 1, a.hdr, 122, abort);
            if (!ok) *abort = 1;
            named_bar_sync(1, 128);   // (every state thread's abort is visible to thread 0)
            // one decision for the 128 threads (each broadcast: write, sync, read, sync)
            auto bcast = [&](int v) -> int {
                if (k == 0) *lbcast = v;
                named_bar_sync(1, 128);
                const int r = *lbcast;
                named_bar_sync(1, 128);
                return r;
            };
            ok = bcast(*abort ? 0 : 1) != 0;
            int *flags = lb.flag + (size_t)bh * a.nseg;
            const size_t row = ((size_t)bh * a.nseg + seg) * KMAX + k;
            if (ok) {
                tc_fence_after();
                if (seg > 0) {
                    row_to_global(lane + R_S, d_v, zown, lb.own + row * a.ne);
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (k == 0) flag_release(flags + seg, 1);
                    // S_start into TMEM [256,384): the predecessors' memories, backwards until an
                    // inclusive prefix (segment 0 always publishes one).  Thread 0 walks the flags
                    // and lists the segments (in zbuf, free until sweep 2); then every thread adds
                    // its rows of all of them.
                    int *list = reinterpret_cast<int *>(zbuf);
                    int j = seg - 1;
                    for (bool first = true; ok; first = false) {
                        int n = 0;
                        if (k == 0) {
                            for (int jj = j; jj >= 0 && n < 64; --jj) {
                                const int f = wait_flag(flags + jj, a.hdr, abort);
                                if (f != 1 && f != 2) {
                                    n = -1;
                                    break;
                                }
                                list[n++] = 2 * jj + (f == 2 ? 1 : 0);
                                if (f == 2) break;
                            }
                        }
                        n = bcast(n);
                        if (n <= 0) {
                            ok = false;
                            break;
                        }
                        const float z = rows_add_list(lane + R_O, d_v, list, n, lb, (size_t)bh * a.nseg, k, a.ne, first);
                        zexcl = first ? z : zexcl + z;
                        const int last = list[n - 1];
                        if (last & 1) break;   // an inclusive prefix: S_start is complete
                        named_bar_sync(1, 128);   // (every thread has read the list)
                        j = (last >> 1) - 1;
                        if (j < 0) ok = false;   // (cannot happen: segment 0 publishes its prefix)
                    }
                } else {
                    row_zero(lane + R_O, d_v);
                    zexcl = 0.f;
                }
                if (ok) {
                    rows_sum_to_global(lane + R_O, lane + R_S, d_v, zexcl + zown, lb.incl + row * a.ne);
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (k == 0) flag_release(flags + seg, 2);
                }
            }
            if (!ok) {
                *abort = 1;
                if (k == 0) flag_release(flags + seg, 3);   // the successors stop waiting for it
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (!FUSED || !*abort) {
    if (warp == 12) {
        // ============================================================ control warp
        if (t == 384) {
            const uint32_t id_p = idesc_f16(128, 128, 1, 1, 0, 0);
            const uint32_t id_o = idesc_f16(128, (uint32_t)d_v, 1, 1, 0, 1);
            const uint32_t id_s = idesc_f16(128, (uint32_t)d_v, 1, 1, 1, 1);
            const int ksteps = a.kn16 / 16;
            // TMA loads in flight: the chunk index of the last one issued per buffer (each buffer's
            // barrier completes one phase per load, and a load is issued only after the previous
            // one into that buffer was consumed)
            int last_v = -1, last_xk = -1, last_xq = -1;
            int last_pv = -1;
            bool ok = true;
            if (!FUSED) {   // (FUSED: loaded for sweep 1)
                mbar_arrive_expect_tx(bars + B_BIMG, (uint32_t)a.bimg_bytes);
                bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars + B_BIMG);
            }
            if (nch > 0) {
                load_x_tile(smem + L.abk + XT, &kmap, bars + B_XK, DR, tok0, bh);
                load_x_tile(smem + L.abq + XT, &qmap, bars + B_XQ, DR, tok0, bh);
                load_v_chunk(smem + L.ve, &vmap, bars + B_V, d_v, tok0, bh);
                last_xk = last_xq = last_v = 0;
            }
            ok = mbar_wait_abortable(bars + B_BIMG, 0, a.hdr, 50, abort);
            const uint32_t bimg = sb + L.bimg, bconst = sb + L.bimg + (uint32_t)a.bimg_main_bytes;
            const uint32_t ve = sb + L.ve;
            for (int c = 0; ok && c < nch; ++c) {
                const uint32_t ph = c & 1;
                const int nxt = tok0 + (c + 1) * C;
                if (c > 0) {
                    // the previous chunk's tril(P) V' is done with P (key logits region) and V'
                    if (!(ok = mbar_wait_abortable(bars + B_PV, (c - 1) & 1, a.hdr, 51, abort))) break;
                    load_v_chunk(smem + L.ve, &vmap, bars + B_V, d_v, tok0 + c * C, bh);
                    last_v = c;
                }
                // key logits
                if (!(ok = mbar_wait_abortable(bars + B_AK, ph, a.hdr, 52, abort))) break;
                tc_fence_after();
                issue_logits_x<DR>(tmem + R_LK, sb + L.abk, bimg, bconst, sb + L.ax, a.kn16);
                mma_commit(bars + B_LK);
                // query logits (the query side of the previous chunk is done with R_LQ)
                if (!(ok = mbar_wait_abortable(bars + B_AQ, ph, a.hdr, 53, abort))) break;
                if (c > 0 && !(ok = mbar_wait_abortable(bars + B_PQ, (c - 1) & 1, a.hdr, 54, abort))) break;
                tc_fence_after();
                issue_logits_x<DR>(tmem + R_LQ, sb + L.abq, bimg, bconst, sb + L.ax, a.kn16);
                mma_commit(bars + B_LQ);
                // the key A tile has been read: stage the next chunk's key rows
                if (!(ok = mbar_wait_abortable(bars + B_LK, ph, a.hdr, 62, abort))) break;
                if (c + 1 < nch) {
                    load_x_tile(smem + L.abk + XT, &kmap, bars + B_XK, DR, nxt, bh);
                    last_xk = c + 1;
                }
                // S update: E_K and V' ready, S_{c-1} read out
                if (!(ok = mbar_wait_abortable(bars + B_GK, ph, a.hdr, 55, abort))) break;
                if (!(ok = mbar_wait_abortable(bars + B_SP, ph, a.hdr, 58, abort))) break;
                if (!(ok = mbar_wait_abortable(bars + B_VS, ph, a.hdr, 59, abort))) break;
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s)   // S += E_K^T V'
                    mma_f16(tmem + R_S, mn128desc(sb + L.gk, s, C), mn32desc(ve, s, C), id_s, 1u);
                mma_commit(bars + B_S);
                // the query A tile has been read: stage the next chunk's query rows
                if (!(ok = mbar_wait_abortable(bars + B_LQ, ph, a.hdr, 63, abort))) break;
                if (c + 1 < nch) {
                    load_x_tile(smem + L.abq + XT, &qmap, bars + B_XQ, DR, nxt, bh);
                    last_xq = c + 1;
                }
                // P and the inter-chunk read (the output side is done with R_O)
                if (!(ok = mbar_wait_abortable(bars + B_GQ, ph, a.hdr, 60, abort))) break;
                if (c > 0 && !(ok = mbar_wait_abortable(bars + B_OF, (c - 1) & 1, a.hdr, 61, abort))) break;
                tc_fence_after();
                for (int s = 0; s < ksteps; ++s)   // P = E_Q E_K^T
                    mma_f16_tmem_a(tmem + R_LK, tmem + R_LQ + 8 * s, kdesc(sb + L.gk, s, C), id_p, s > 0);
                for (int s = 0; s < ksteps; ++s)   // O = E_Q S_{c-1}
                    mma_f16_tmem_a(tmem + R_O, tmem + R_LQ + 8 * s, mn32desc(sb + L.sp, s, KMAX), id_o, s > 0);
                mma_commit(bars + B_PQ);
                // intra-chunk: O += tril(P) V'
                if (!(ok = mbar_wait_abortable(bars + B_PS, ph, a.hdr, 56, abort))) break;
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s)
                    mma_f16_tmem_a(tmem + R_O, tmem + R_LK + 8 * s, mn32desc(ve, s, C), id_o, 1u);
                mma_commit(bars + B_PV);
                last_pv = c;
            }
            // drain: MMAs complete in issue order, so the last commit covers them all; TMA loads
            // still in flight (only after a timeout) complete before shared memory is released
            if (last_pv >= 0) mbar_wait(bars + B_PV, last_pv & 1, a.hdr, 57);
            if (last_v >= 0) mbar_wait(bars + B_V, last_v & 1, a.hdr, 58);
            if (last_xk >= 0) mbar_wait(bars + B_XK, last_xk & 1, a.hdr, 58);
            if (last_xq >= 0) mbar_wait(bars + B_XQ, last_xq & 1, a.hdr, 58);
        }
    } else if (warp < 4) {
        // ============================================================ key side
        const int k = t;   // TMEM lane and token row of the chunk
        const uint32_t lane = tmem + ((uint32_t)(warp * 32) << 16);
        uint8_t *abk = smem + L.abk;
        if (nch > 0 && mbar_wait_abortable(bars + B_XK, 0, a.hdr, 67, abort)) {
            build_inplace<DR>(abk, k);
            fence_proxy_async_smem();
            mbar_arrive(bars + B_AK);
        }
        for (int c = 0; c < nch; ++c) {
            const uint32_t ph = c & 1;
            const int base = tok0 + c * C;
            if (!mbar_wait_abortable(bars + B_LK, ph, a.hdr, 61, abort)) break;
            if (c > 0) {
                // the E_K tile and r are free once P, the S update and the column sums of the
                // previous chunk have read them
                if (!mbar_wait_abortable(bars + B_PQ, (c - 1) & 1, a.hdr, 63, abort)) break;
                if (!mbar_wait_abortable(bars + B_S, (c - 1) & 1, a.hdr, 62, abort)) break;
                if (!mbar_wait_abortable(bars + B_ZP, (c - 1) & 1, a.hdr, 64, abort)) break;
            }
            tc_fence_after();
            const float sum = key_exp(lane + R_LK, a.K, kc, smem + L.gk, k);
            const float r = base + k < tok_end ? 1.0f / sum : 0.f;
            rbuf[k] = r;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bars + B_GK);
            // V' = diag(r) V for this chunk
            if (!mbar_wait_abortable(bars + B_V, ph, a.hdr, 65, abort)) break;
            scale_v_row(smem + L.ve, k, d_v, r);
            fence_proxy_async_smem();
            mbar_arrive(bars + B_VS);
            // the next chunk's keys
            if (c + 1 < nch) {
                if (!mbar_wait_abortable(bars + B_XK, (c + 1) & 1, a.hdr, 67, abort)) break;
                build_inplace<DR>(abk, k);
                fence_proxy_async_smem();
                mbar_arrive(bars + B_AK);
            }
        }
    } else if (warp < 8) {
        // ============================================================ query side
        const int i = t - 128;
        const uint32_t lane = tmem + ((uint32_t)((warp - 4) * 32) << 16);
        uint8_t *abq = smem + L.abq;
        for (int c = 0; c < nch; ++c) {
            const uint32_t ph = c & 1;
            const int base = tok0 + c * C;
            const bool valid = base + i < tok_end;
            if (!mbar_wait_abortable(bars + B_XQ, ph, a.hdr, 75, abort)) break;
            build_inplace<DR>(abq, i);
            fence_proxy_async_smem();
            mbar_arrive(bars + B_AQ);
            if (!mbar_wait_abortable(bars + B_LQ, ph, a.hdr, 71, abort)) break;
            if (!mbar_wait_abortable(bars + B_SP, ph, a.hdr, 72, abort)) break;
            tc_fence_after();
            const float2 sd = query_softmax(lane + R_LQ, a.K, kc, valid, zbuf + ph * KMAX);
            tc_fence_before();
            mbar_arrive(bars + B_GQ);
            // causal mask of P; P (bf16 pairs) back into TMEM as the A operand of tril(P) V'
            if (!mbar_wait_abortable(bars + B_PQ, ph, a.hdr, 73, abort)) break;
            if (!mbar_wait_abortable(bars + B_GK, ph, a.hdr, 76, abort)) break;   // r of this chunk
            tc_fence_after();
            const float den = sd.y + causal_mask(lane + R_LK, i, rbuf);
            dsm[ph * C + i] = make_float2(sd.x, den);
            tc_fence_before();
            mbar_arrive(bars + B_PS);
        }
    } else {
        // ============================================================ state and output side
        const int k = t - 256;   // TMEM lane: component row of S, and token row of the output
        const uint32_t lane = tmem + ((uint32_t)((warp - 8) * 32) << 16);
        // starting memory (from the scan, or FUSED from the look-back in TMEM [256,384)): V~ part
        // to TMEM and as the bf16 operand, Z part to the running sum
        const float *src = a.agg + (((size_t)bh * a.nseg + seg) * KMAX + k) * a.ne;
        for (int b = 0; b < d_v / 16; ++b) {
            uint32_t r[16];
            if (FUSED) {
                tmem_ld16(lane + R_O + 16 * b, r);
                tmem_ld_wait();
            } else {
                const float4 *s4 = reinterpret_cast<const float4 *>(src + b * 16);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = s4[q];
                    r[4 * q] = __float_as_uint(f.x);
                    r[4 * q + 1] = __float_as_uint(f.y);
                    r[4 * q + 2] = __float_as_uint(f.z);
                    r[4 * q + 3] = __float_as_uint(f.w);
                }
            }
            tmem_st16(lane + R_S + 16 * b, r);
            const uint4 lo = make_uint4(pk2(r[0], r[1], 1.f), pk2(r[2], r[3], 1.f), pk2(r[4], r[5], 1.f), pk2(r[6], r[7], 1.f));
            const uint4 hi = make_uint4(pk2(r[8], r[9], 1.f), pk2(r[10], r[11], 1.f), pk2(r[12], r[13], 1.f), pk2(r[14], r[15], 1.f));
            *reinterpret_cast<uint4 *>(smem + L.sp + sw32(k, b, 0, KMAX)) = lo;
            *reinterpret_cast<uint4 *>(smem + L.sp + sw32(k, b, 1, KMAX)) = hi;
        }
        float zrun = FUSED ? zexcl : src[d_v];
        zbuf[k] = zrun;
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bars + B_SP);   // phase 0: S_start ready
        // output of chunk cc (numerator complete, normaliser from the query side)
        auto output = [&](int cc) -> bool {
            const uint32_t pc = cc & 1;
            if (!mbar_wait_abortable(bars + B_PS, pc, a.hdr, 77, abort)) return false;
            if (!mbar_wait_abortable(bars + B_PV, pc, a.hdr, 74, abort)) return false;
            tc_fence_after();
            const float2 sd = dsm[pc * C + k];
            const int row = tok0 + cc * C + k;
            write_output(lane + R_O, d_v, 1.0f / (sd.y + a.eps * sd.x), row < tok_end, a.O,
                         (long long)bh * a.N + row, a.out_f32);
            tc_fence_before();
            mbar_arrive(bars + B_OF);
            return true;
        };
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const uint32_t ph = c & 1;
            if (c > 0 && !(ok = output(c - 1))) break;
            // Z_c = Z_{c-1} + E_K^T r
            if (!(ok = mbar_wait_abortable(bars + B_GK, ph, a.hdr, 66, abort))) break;
            float *zp = zpart + ph * 8 * KMAX;
            colsum_part(smem + L.gk, rbuf, zp, k);
            mbar_arrive(bars + B_ZP);
            if (!(ok = mbar_wait_abortable(bars + B_ZP, ph, a.hdr, 68, abort))) break;
            {
                float zs = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) zs += zp[g * KMAX + k];
                zrun += zs;
            }
            // readout of S_c (after the update, and after the read of S_{c-1} that it overwrites)
            if (!(ok = mbar_wait_abortable(bars + B_S, ph, a.hdr, 69, abort))) break;
            if (!(ok = mbar_wait_abortable(bars + B_PQ, ph, a.hdr, 70, abort))) break;
            tc_fence_after();
            state_readout(lane + R_S, d_v, smem + L.sp, k);
            zbuf[((c + 1) & 1) * KMAX + k] = zrun;
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bars + B_SP);
        }
        if (ok && nch > 0) output(nch - 1);
    }
    }   // (sweep 2)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 12) tmem_dealloc(tmem, 512);
}

// Shared memory the pipelined causal kernel needs (0 if the shape does not fit).
uint32_t causal_pipelined_smem(int d_r, int kn16, int d_v)
{
    const uint32_t need = CausalSmem(d_r, kn16, d_v).total + 1024;
    return need <= 227u * 1024u ? smem_for(need, 512) : 0;
}

template <int DR>
gma_status_t launch_causal_pipelined(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap,
                                     const CUtensorMap &qmap, int nblocks, cudaStream_t st)
{
    const uint32_t sm = causal_pipelined_smem(DR, a.kn16, a.d_v);
    if (sm == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (!set_smem(tc_causal_pipelined_kernel<DR, false>, sm)) return GMA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_CAUSAL_OUT, st,
               (e = launch_pdl(tc_causal_pipelined_kernel<DR, false>, dim3(nblocks), dim3(CTHREADS), sm, st, a, vmap,
                               kmap, qmap, LookBack{})));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

// The single-launch causal kernel: one CTA per segment, nblocks = BH * nseg; ticket and flags
// (1 + BH * nseg ints) must be zero when it starts; a.agg takes the segments' own memories and
// incl their inclusive prefixes (BH * nseg * KMAX * ne floats each).
template <int DR>
gma_status_t launch_causal_fused(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap,
                                 const CUtensorMap &qmap, int *ticket_flags, float *incl, int nblocks, cudaStream_t st)
{
    const uint32_t sm = causal_pipelined_smem(DR, a.kn16, a.d_v);
    if (sm == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (!set_smem(tc_causal_pipelined_kernel<DR, true>, sm)) return GMA_ERR_CUDA;
    const LookBack lb{ticket_flags, ticket_flags + 1, a.agg, incl};
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_CAUSAL_FUSED, st,
               (e = launch_pdl(tc_causal_pipelined_kernel<DR, true>, dim3(nblocks), dim3(CTHREADS), sm, st, a, vmap,
                               kmap, qmap, lb)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template gma_status_t launch_causal_pipelined<16>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                                  const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_causal_pipelined<32>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                                  const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_causal_pipelined<64>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                                  const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_causal_fused<16>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, int *, float *, int, cudaStream_t);
template gma_status_t launch_causal_fused<32>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, int *, float *, int, cudaStream_t);
template gma_status_t launch_causal_fused<64>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                              const CUtensorMap &, int *, float *, int, cudaStream_t);

}  // namespace tck
}  // namespace gma
