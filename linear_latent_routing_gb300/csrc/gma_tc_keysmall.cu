// gma_tc_keysmall.cu -- the bidirectional key pass of the tcgen05 family (sm_103a) for small
// component counts: two CTAs per SM.
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §2, write phase: keys write the latent memory V~ = Gamma_K^T V and its normaliser
// Z = Gamma_K^T 1.  Over one segment of one (batch, head) slice, as the segment pass
// (gma_tc_segmem.cu) computes it:
//   agg[bh][seg][k][c] = sum_{j in segment} gamma_K[j][k] * [v_j | 1][c]   (fp32; c = d_v is Z).
// The memory update is transposed here:
//   S^T (TMEM: lane = column c of [V | 1], TMEM column = component k) += [V | 1]^T Gamma_K,
// so Gamma_K is the B operand (N = kn16 components) and its shared-memory tile holds kn16 columns
// (8 KB at K = 32, where an M operand would need all 128 rows, 32 KB).  [V | 1]^T is the M = 128
// operand: its rows beyond d_v + 16 read whatever follows the value tile in shared memory and
// land only in TMEM lanes that are never read.  With the smaller tiles and 128 or 256 TMEM
// columns, two CTAs share an SM, so one CTA's chunk latency overlaps the other's work.
//
// Roles (320 threads) and buffering follow the segment pass: two key groups of four warps take
// alternate chunks of 128 tokens ([x^2, x] from the TMA-staged key rows, which a group copies to
// registers and releases before converting them, at d_r <= 32; logits by tcgen05 into the chunk's own TMEM
// columns; softmax -> the group's Gamma_K tile); warp 8 issues the MMAs, warp 9 the TMA loads,
// each as soon as its buffer is free.  Every wait is bounded; a timeout records GMA_ERR_TIMEOUT and makes all
// roles leave their loops.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

constexpr int KTHREADS = 320;
enum KBar { K_BIMG, K_AK, K_LK0, K_LK1, K_GK0, K_GK1, K_SD0, K_SD1, K_V0, K_V1, K_XK, K_XF, K_FIN, K_NBAR };

struct SmallSmem {
    uint32_t ve0, ve1, abuf, xst, gk0, gk1, bimg, ax, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ SmallSmem(int DR, int kn16, int d_v)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        const uint32_t tile = ka / 64u * 128u;
        const uint32_t vbytes = (uint32_t)(d_v + 16) * C * 2u;   // value blocks + one block of ones
        uint32_t o = 0;
        ve0 = o; o = al(o + vbytes);
        ve1 = o; o = al(o + vbytes);
        abuf = o; o = al(o + tile * (uint32_t)C);
        xst = o; o = al(o + (uint32_t)C * DR * 2u);   // staged key rows (TMA, swizzled)
        gk0 = o; o = al(o + (uint32_t)kn16 * C * 2u);   // Gamma_K, MN-major blocks of 16 components
        gk1 = o; o = al(o + (uint32_t)kn16 * C * 2u);
        bimg = o; o = al(o + tile * (uint32_t)kn16 + 32u * (uint32_t)kn16);
        ax = o; o = al(o + (uint32_t)C * 32u);
        bars = o; o += K_NBAR * 8u;
        misc = o; o += 16u;
        // the M = 128 operand read from ve1 spans 128 columns: that span stays inside the CTA's
        // shared memory
        const uint32_t span = ve1 + 128u * C * 2u;
        total = o > span ? o : span;
    }
};

// TMEM columns of one CTA: two logits regions and the memory, 32 * kc columns each.
__host__ __device__ inline uint32_t small_tmem_cols(int K) { return (K + 31) / 32 * 96 <= 128 ? 128u : 256u; }

// Key side: Gamma_K row k = softmax of the TMEM logits at tl (K <= 64), normalised (zeros when
// not valid), as bf16 into the MN-major 32-byte-swizzled tile gk (blocks of 16 components, one
// 32-byte row per token), of which the first nblk blocks exist.
__device__ __forceinline__ void key_softmax_mn(uint32_t tl, int K, int kc, bool valid, uint8_t *gk, int k, int nblk)
{
    const float m = row_max(tl, K, kc);
    float sum = 0.f;
    uint32_t pk[32];   // component pairs (2i, 2i + 1)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        if (c < kc) {
            uint32_t r[32];
            tmem_ld32(tl + 32 * c, r);
            tmem_ld_wait();
            sum += chunk_exp(r, c, K, m);
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[16 * c + j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[16 * c + j] = 0u;
        }
    }
    const float scf = valid ? 1.0f / sum : 0.f;
    const uint32_t sc2 = pack_bf16(scf, scf);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (b < nblk) {
            const uint32_t *e = pk + 8 * b;
            *reinterpret_cast<uint4 *>(gk + sw32(k, b, 0, C)) =
                make_uint4(mul_bf16x2(e[0], sc2), mul_bf16x2(e[1], sc2), mul_bf16x2(e[2], sc2), mul_bf16x2(e[3], sc2));
            *reinterpret_cast<uint4 *>(gk + sw32(k, b, 1, C)) =
                make_uint4(mul_bf16x2(e[4], sc2), mul_bf16x2(e[5], sc2), mul_bf16x2(e[6], sc2), mul_bf16x2(e[7], sc2));
        }
    }
}

}  // namespace

template <int DR>
__global__ void __launch_bounds__(KTHREADS, 2) tc_key_memory_small_kernel(const Args a,
                                                                         const __grid_constant__ CUtensorMap vmap,
                                                                         const __grid_constant__ CUtensorMap kmap)
{
    // (no wait here: the set-up and the first loads of K_X and V, which no kernel writes, overlap
    // the kernel before; the loader waits before the tables, and every write follows that)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const SmallSmem L(DR, a.kn16, a.d_v);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L.misc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L.misc + 4);
    const int bh = blockIdx.x / a.nseg, seg = blockIdx.x % a.nseg, h = bh % a.H;
    const int t = threadIdx.x, warp = t >> 5;
    const int tok0 = seg * a.cps * C;
    const int tok_end = min(a.N, tok0 + a.cps * C);
    const int nch = (tok_end - tok0 + C - 1) / C;
    const int d_v = a.d_v, ne = a.ne;
    const int kc = (a.K + 31) >> 5;
    const uint32_t tcols = small_tmem_cols(a.K);
    const uint32_t R_L0 = 0, R_L1 = 32u * kc, R_S = 64u * kc;

    // ---------------------------------------------------------------- set-up
    if (warp == 8) {
        if (t == 256) {
            for (int i = 0; i < K_NBAR; ++i) mbar_init(bars + i, (i == K_AK || i == K_XF || i == K_GK0 || i == K_GK1) ? 128u : 1u);
            *abort = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(tslot, tcols);
    } else if (warp < 8) {
        // the ones blocks of [V | 1] and the constant operand (1, 1, 0, ...) of the logits
        const int u = t;   // 0..255
        const uint32_t one2 = 0x3F803F80u;   // bf16 pair (1, 1)
        const uint32_t o1 = (uint32_t)(d_v / 16) * C * 32;
        for (uint32_t o = u * 16; o < (uint32_t)C * 32; o += 256 * 16) {
            *reinterpret_cast<uint4 *>(smem + L.ve0 + o1 + o) = make_uint4(one2, one2, one2, one2);
            *reinterpret_cast<uint4 *>(smem + L.ve1 + o1 + o) = make_uint4(one2, one2, one2, one2);
        }
        if (u < C) {
            const int flip = (u >> 2) & 1;
            *reinterpret_cast<uint4 *>(smem + L.ax + u * 32 + (flip << 4)) = make_uint4(0x3C003C00u, 0, 0, 0);
            *reinterpret_cast<uint4 *>(smem + L.ax + u * 32 + ((flip ^ 1) << 4)) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = smem_u32(smem);
    // the next kernel may start now: this CTA holds its tensor memory, so a CTA of the next kernel
    // that allocates before it waits for this grid can never take the columns this one needs
    grid_dependency_launch();

    if (warp == 8) {
        // ============================================================ control warp: MMAs
        if (t == 256) {
            auto ve = [&](int c) { return (c & 1) ? L.ve1 : L.ve0; };
            auto gk = [&](int c) { return (c & 1) ? L.gk1 : L.gk0; };
            const uint32_t id_s = idesc_f16(128, (uint32_t)a.kn16, 1, 1, 1, 1);
            bool ok = mbar_wait_abortable(bars + K_BIMG, 0, a.hdr, 140, abort);
            int last_sd = -1;
            const uint32_t bimg = sb + L.bimg, bconst = sb + L.bimg + (uint32_t)a.bimg_main_bytes;
            // S^T update of chunk j: value tile and Gamma_K tile of buffer j & 1
            auto update = [&](int j) -> bool {
                const int g = j & 1, n = j >> 1;
                if (!mbar_wait_abortable(bars + K_GK0 + g, n & 1, a.hdr, 141, abort)) return false;
                if (!mbar_wait_abortable(bars + K_V0 + g, n & 1, a.hdr, 142, abort)) return false;
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s)
                    mma_f16(tmem + R_S, mn32desc(sb + ve(j), s, C), mn32desc(sb + gk(j), s, C), id_s,
                            (j > 0 || s > 0) ? 1u : 0u);
                mma_commit(bars + K_SD0 + g);
                last_sd = j;
                return true;
            };
            for (int c = 0; ok && c < nch; ++c) {
                const int g = c & 1;
                if (!(ok = mbar_wait_abortable(bars + K_AK, c & 1, a.hdr, 143, abort))) break;
                tc_fence_after();
                issue_logits_c<DR>(tmem + (g ? R_L1 : R_L0), sb + L.abuf, bimg, bconst, sb + L.ax, a.kn16);
                mma_commit(bars + K_LK0 + g);
                if (c >= 1 && !(ok = update(c - 1))) break;
            }
            if (ok && nch > 0) ok = update(nch - 1);
            // one more commit, on a barrier of its own: it completes once every MMA above has, an
            // unambiguous phase for the read-out of the memory and for releasing the tensor memory
            // (the last chunk's own barrier can lag two phases behind, which its parity cannot tell)
            mma_commit(bars + K_FIN);
            if (last_sd >= 0) mbar_wait(bars + K_FIN, 0, a.hdr, 144);
        }
    } else if (warp == 9) {
        // ============================================================ loader warp: TMA loads
        if (t == 288) {
            auto ve = [&](int c) { return (c & 1) ? L.ve1 : L.ve0; };
            bool ok = true;
            bool vpend0 = false, vpend1 = false;   // loads whose update has not been seen yet
            int vlast0 = -1, vlast1 = -1, last_xk = -1;
            auto load_v = [&](int c) {
                load_v_chunk(smem + ve(c), &vmap, bars + K_V0 + (c & 1), d_v, tok0 + c * C, bh);
                if (c & 1) { vpend1 = true; vlast1 = c; } else { vpend0 = true; vlast0 = c; }
            };
            for (int c = 0; c < 2 && c < nch; ++c) load_v(c);
            if (nch > 0) {
                load_x_tile(smem + L.xst, &kmap, bars + K_XK, DR, tok0, bh);
                last_xk = 0;
            }
            grid_dependency_wait();   // the parameter tables come from the kernel before
            mbar_arrive_expect_tx(bars + K_BIMG, (uint32_t)a.bimg_bytes);
            bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars + K_BIMG);
            // each load as soon as its buffer is free, whichever comes first: the key rows of chunk
            // nx once chunk nx - 1's were read, the values of chunk nv once the update of chunk
            // nv - 2 is done (neither test can see a phase ahead: each next phase needs a load this
            // loop has not issued yet); bounded like every wait
            int nx = 1, nv = 2;
            long long t0 = clock64();
            while (ok && (nx < nch || nv < nch)) {
                bool progress = false;
                if (nx < nch && mbar_test_wait(bars + K_XF, (nx - 1) & 1)) {
                    load_x_tile(smem + L.xst, &kmap, bars + K_XK, DR, tok0 + nx * C, bh);
                    last_xk = nx++;
                    progress = true;
                }
                if (nv < nch && mbar_test_wait(bars + K_SD0 + (nv & 1), ((nv - 2) >> 1) & 1)) {
                    if (nv & 1) vpend1 = false; else vpend0 = false;
                    load_v(nv++);
                    progress = true;
                }
                if (progress) {
                    t0 = clock64();
                } else if (*abort) {
                    ok = false;
                } else if (wait_expired(clock64() - t0, a.hdr)) {
                    record_error(a.hdr, GMA_ERR_TIMEOUT, 148);
                    *abort = 1;
                    ok = false;
                } else {
                    __nanosleep(32);
                }
            }
            // loads still in flight (only after a timeout) complete before shared memory is released
            if (last_xk >= 0) mbar_wait(bars + K_XK, last_xk & 1, a.hdr, 147);
            if (vpend0 && vlast0 >= 0) mbar_wait(bars + K_V0, (vlast0 >> 1) & 1, a.hdr, 147);
            if (vpend1 && vlast1 >= 0) mbar_wait(bars + K_V1, (vlast1 >> 1) & 1, a.hdr, 147);
        }
    } else {
        // ============================================================ key-side groups
        const int g = warp >> 2;            // group: chunks c with c % 2 == g
        const int k = t & 127;              // TMEM lane: token row; for the memory, column of [V | 1]
        const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        uint8_t *gk = smem + (g ? L.gk1 : L.gk0);
        const int nblk = a.kn16 / 16;
        for (int c = g; c < nch; c += 2) {
            const int n = c >> 1;
            const bool kvalid = tok0 + c * C + k < tok_end;
            // the [x^2, x] buffer is free once the previous chunk's logits are done
            if (c >= 1 && !mbar_wait_abortable(bars + K_LK0 + ((c - 1) & 1), ((c - 1) >> 1) & 1, a.hdr, 150, abort)) break;
            if (!mbar_wait_abortable(bars + K_XK, c & 1, a.hdr, 151, abort)) break;
            if constexpr (DR <= 32) {
                // the staged row into registers, the staging buffer released (the next chunk's
                // rows load during this chunk's conversion), then [x^2, x] into the A tile
                uint4 xr[DR / 8];
#pragma unroll
                for (int q = 0; q < DR / 8; ++q) xr[q] = *reinterpret_cast<const uint4 *>(smem + L.xst + xs_off<DR>(k, q));
                fence_proxy_async_smem();   // (these reads come before the next chunk's TMA overwrites the rows)
                mbar_arrive(bars + K_XF);
                build_a<DR>(smem + L.abuf, k, xr);
            } else {
                // (at d_r = 64 the row held in registers would spill under the two-CTA budget:
                // the tile is built from shared memory and the buffer released after)
                build_a_s<DR>(smem + L.abuf, k, smem + L.xst);
                fence_proxy_async_smem();
                mbar_arrive(bars + K_XF);
            }
            fence_proxy_async_smem();
            // (a test of the timeout path withholds the first chunk's signal: every wait on it
            // runs out, and all roles leave their loops)
            if (!(a.test_withhold && c == 0)) mbar_arrive(bars + K_AK);
            if (!mbar_wait_abortable(bars + K_LK0 + g, n & 1, a.hdr, 152, abort)) break;
            // this group's Gamma_K tile is free once the update two chunks back has read it
            if (c >= 2 && !mbar_wait_abortable(bars + K_SD0 + g, (n - 1) & 1, a.hdr, 153, abort)) break;
            tc_fence_after();
            key_softmax_mn(lane + (g ? R_L1 : R_L0), a.K, kc, kvalid, gk, k, nblk);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bars + K_GK0 + g);
        }
        // group 0 writes the segment's memory once the last update is done: lane k holds column
        // k of [V | 1] for every component; the rows between kn16 and 32 * kc (read as zeros by the
        // normaliser's dot product) are written as zeros
        if (g == 0 && !*abort) {
            float *dst = a.agg + ((size_t)bh * a.nseg + seg) * KMAX * ne;
            const bool ok = nch > 0 && mbar_wait_abortable(bars + K_FIN, 0, a.hdr, 154, abort);
            if (ok) {
                tc_fence_after();
                for (int b = 0; b < nblk; ++b) {
                    uint32_t r[16];
                    tmem_ld16(lane + R_S + 16 * b, r);
                    tmem_ld_wait();
                    if (k < ne) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) dst[(size_t)(16 * b + j) * ne + k] = __uint_as_float(r[j]);
                    }
                }
                if (k < ne)
                    for (int j = a.kn16; j < 32 * kc; ++j) dst[(size_t)j * ne + k] = 0.f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8) tmem_dealloc(tmem, tcols);
}

// Shared memory of the small key pass (0 if two CTAs of it do not fit on one SM, or the shape is
// outside it: K <= 64 and d_v + 16 <= 128 TMEM lanes).
uint32_t keysmall_smem(int d_r, int K, int d_v)
{
    if (K > 64 || d_v + 16 > 128) return 0;
    const int kn16 = (K + 15) / 16 * 16;
    const uint32_t need = SmallSmem(d_r, kn16, d_v).total + 1024;
    if (2u * need > 228u * 1024u - 2u * 1024u) return 0;
    return smem_for(need, small_tmem_cols(K));
}

template <int DR>
gma_status_t launch_keysmall(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap, int nblocks,
                             cudaStream_t st)
{
    const uint32_t sm = keysmall_smem(DR, a.K, a.d_v);
    if (sm == 0 || a.kn16 > 64) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (!set_smem(tc_key_memory_small_kernel<DR>, sm)) return GMA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_BIDIR_WRITE, st,
               (e = launch_pdl(tc_key_memory_small_kernel<DR>, dim3(nblocks), dim3(KTHREADS), sm, st, a, vmap, kmap)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template gma_status_t launch_keysmall<16>(const Args &, const CUtensorMap &, const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_keysmall<32>(const Args &, const CUtensorMap &, const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_keysmall<64>(const Args &, const CUtensorMap &, const CUtensorMap &, int, cudaStream_t);

}  // namespace tck
}  // namespace gma
