// gma_tc_segmem.cu -- segment memories for the tcgen05 family (sm_103a), warp-specialised.
//
// Method: page "Attention par Mélange Gaussien (GMA)" (gist.science/fr/paper/2606.18283),
// Méthodologie §2, write phase: keys write the latent memory V~ = Gamma_K^T V and its
// normaliser Z = Gamma_K^T 1.  Here over one segment of one (batch, head) slice:
//   agg[bh][seg][k][c] = sum_{j in segment} gamma_K[j][k] * [v_j | 1][c]   (fp32; c = d_v is Z).
// The bidirectional variant sums all segments of a slice; the causal variant scans them into
// exclusive prefixes, each the starting memory of the chunked kernel's segment.
//
// Warp roles (320 threads): two key-side groups of four warps take alternate chunks of 128
// tokens ([x^2, x] from the TMA-staged key rows, softmax -> Gamma_K in their own shared-memory
// tile); warp 9 issues the TMA loads of the key rows and value tiles, each as soon as its buffer
// is free (polling both, so neither kind of load waits behind the other); warp 8 issues the tcgen05.mma's (the logits into the chunk's own TMEM columns and
// S += Gamma_K^T [V | 1] into the running memory) and the stores of Gamma_K.  Logits, Gamma_K
// and value tiles are double buffered, so one group's softmax overlaps the other group's logits
// and memory update.
// Barriers are per buffer, so no waiter can fall two phases behind.  A key group copies its
// staged row into registers and releases the staging buffer before converting it, so that the
// next chunk's rows load meanwhile (the key rows' TMA and the [x^2, x] build are the chunk-to-
// chunk chain, measured); the softmax computes the exponentials again when it stores them
// instead of holding them, which leaves the registers for that copy.
// For the causal variant the kernel also stores each chunk's Gamma_K tile (bf16, normalised) to
// the workspace with a TMA store, so that the output pass reads it instead of recomputing it.
#include "tc_rows.cuh"

namespace gma {
namespace tck {

namespace {

constexpr int STHREADS = 320;
enum SBar { S_BIMG, S_AK, S_LK0, S_LK1, S_GK0, S_GK1, S_SD0, S_SD1, S_V0, S_V1, S_XK, S_XF, S_FIN, S_NBAR };
constexpr uint32_t SR_L0 = 0, SR_L1 = 128, SR_S = 256;

struct SegSmem {
    uint32_t bimg, ax, abuf, xst, gk0, gk1, ve0, ve1, bars, misc, total;
    __host__ __device__ static uint32_t al(uint32_t x) { return (x + 1023u) & ~1023u; }
    __host__ __device__ SegSmem(int DR, int kn16, int d_v)
    {
        const uint32_t ka = DR * 2 < 64 ? 64u : (uint32_t)DR * 2u;
        const uint32_t tile = ka / 64u * 128u;
        const uint32_t vbytes = (uint32_t)(d_v + 16) * C * 2u;   // value blocks + one block of ones
        uint32_t o = 0;
        bimg = o; o = al(o + tile * (uint32_t)kn16 + 32u * (uint32_t)kn16);
        ax = o; o = al(o + (uint32_t)C * 32u);
        abuf = o; o = al(o + tile * (uint32_t)C);
        xst = o; o = al(o + (uint32_t)C * DR * 2u);   // staged key rows (TMA, swizzled)
        gk0 = o; o = al(o + 2u * C * 128u);
        gk1 = o; o = al(o + 2u * C * 128u);
        ve0 = o; o = al(o + vbytes);
        ve1 = o; o = al(o + vbytes);
        bars = o; o += S_NBAR * 8u;
        misc = o; o += 16u;
        total = o;
    }
};

// Key side: Gamma_K row k = softmax of the TMEM logits at tl, normalised (zeros when not valid),
// as bf16 into the K-major SW128 tile gk: the maximum and the sum from the logits, then each
// chunk of 32 exponentials computed again and stored, instead of holding all of them in
// registers (the same values as key_softmax_reg, with fewer registers live).
__device__ __forceinline__ void key_softmax_lean(uint32_t tl, int K, int kc, bool valid, uint8_t *gk, int k)
{
    const float m = row_max(tl, K, kc);
    float sum = 0.f;
#pragma unroll 1
    for (int c = 0; c < kc; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        sum += chunk_exp(r, c, K, m);
    }
    const float scf = valid ? 1.0f / sum : 0.f;
    const uint32_t sc2 = pack_bf16(scf, scf);
#pragma unroll 1
    for (int c = 0; c < kc; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + 32 * c, r);
        tmem_ld_wait();
        chunk_exp(r, c, K, m);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t e[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                e[j] = mul_bf16x2(pack_bf16(__uint_as_float(r[8 * q + 2 * j]), __uint_as_float(r[8 * q + 2 * j + 1])), sc2);
            *reinterpret_cast<uint4 *>(gk + sw128(k, 4 * c + q, C)) = make_uint4(e[0], e[1], e[2], e[3]);
        }
    }
}

}  // namespace

template <int DR>
__global__ void __launch_bounds__(STHREADS, 1) tc_segment_memory_pipelined_kernel(const Args a,
                                                                                  const __grid_constant__ CUtensorMap vmap,
                                                                                  const __grid_constant__ CUtensorMap kmap,
                                                                                  const __grid_constant__ CUtensorMap gmap)
{
    // (no wait here: the set-up and the first loads of K_X and V, which no kernel writes, overlap
    // the kernel before; the threads that read its results wait below)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const SegSmem L(DR, a.kn16, a.d_v);
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

    // ---------------------------------------------------------------- set-up
    if (warp == 8) {
        if (t == 256) {
            for (int i = 0; i < S_NBAR; ++i) mbar_init(bars + i, (i == S_AK || i == S_XF || i == S_GK0 || i == S_GK1) ? 128u : 1u);
            *abort = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(tslot, 512);
    } else if (warp < 8) {
        // zero both Gamma_K tiles (components the softmax never writes), ones blocks of [V | 1],
        // and the constant operand (1, 1, 0, ...) of the logits
        const int u = t;   // 0..255
        for (uint32_t o = u * 16; o < 2u * C * 128u; o += 256 * 16) {
            *reinterpret_cast<uint4 *>(smem + L.gk0 + o) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(smem + L.gk1 + o) = make_uint4(0, 0, 0, 0);
        }
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
        // ============================================================ control warp: MMAs, stores
        if (t == 256) {
            auto ve = [&](int c) { return (c & 1) ? L.ve1 : L.ve0; };
            auto gk = [&](int c) { return (c & 1) ? L.gk1 : L.gk0; };
            const uint32_t id_s = idesc_f16(128, (uint32_t)ne, 1, 1, 1, 1);
            bool ok = mbar_wait_abortable(bars + S_BIMG, 0, a.hdr, 80, abort);
            int last_sd = -1;
            const uint32_t bimg = sb + L.bimg, bconst = sb + L.bimg + (uint32_t)a.bimg_main_bytes;
            // S update of chunk j: Gamma_K tile and value tile of buffer j & 1 (and the store of the
            // tile; its buffer is released with the update's commit once the store has read it)
            auto update = [&](int j) -> bool {
                const int g = j & 1, n = j >> 1;
                if (!mbar_wait_abortable(bars + S_GK0 + g, n & 1, a.hdr, 81, abort)) return false;
                if (!mbar_wait_abortable(bars + S_V0 + g, n & 1, a.hdr, 82, abort)) return false;
                if (a.gam) {
                    for (int h = 0; h < a.kg / 64; ++h)
                        tma_store_3d(&gmap, smem + gk(j) + h * C * 128, 64 * h, tok0 + j * C, bh);
                    bulk_commit_group();
                }
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s)
                    mma_f16(tmem + SR_S, mn128desc(sb + gk(j), s, C), mn32desc(sb + ve(j), s, C), id_s,
                            (j > 0 || s > 0) ? 1u : 0u);
                if (a.gam) bulk_wait_read();
                mma_commit(bars + S_SD0 + g);
                last_sd = j;
                return true;
            };
            for (int c = 0; ok && c < nch; ++c) {
                const int g = c & 1;
                if (!(ok = mbar_wait_abortable(bars + S_AK, c & 1, a.hdr, 83, abort))) break;
                tc_fence_after();
                issue_logits_c<DR>(tmem + (g ? SR_L1 : SR_L0), sb + L.abuf, bimg, bconst, sb + L.ax, a.kn16);
                mma_commit(bars + S_LK0 + g);
                if (c >= 1 && !(ok = update(c - 1))) break;
            }
            if (ok && nch > 0) ok = update(nch - 1);
            // one more commit, on a barrier of its own: it completes once every MMA above has, an
            // unambiguous phase for the read-out of the memory and for releasing the tensor memory
            // (the last chunk's own barrier can lag two phases behind, which its parity cannot tell)
            mma_commit(bars + S_FIN);
            if (last_sd >= 0) mbar_wait(bars + S_FIN, 0, a.hdr, 85);
            if (a.gam) bulk_wait_all();
        }
    } else if (warp == 9) {
        // ============================================================ loader warp: TMA loads
        if (t == 288) {
            auto ve = [&](int c) { return (c & 1) ? L.ve1 : L.ve0; };
            bool ok = true;
            bool vpend0 = false, vpend1 = false;   // loads whose update has not been seen yet
            int vlast0 = -1, vlast1 = -1, last_xk = -1;
            auto load_v = [&](int c) {
                load_v_chunk(smem + ve(c), &vmap, bars + S_V0 + (c & 1), d_v, tok0 + c * C, bh);
                if (c & 1) { vpend1 = true; vlast1 = c; } else { vpend0 = true; vlast0 = c; }
            };
            for (int c = 0; c < 2 && c < nch; ++c) load_v(c);
            if (nch > 0) {
                load_x_tile(smem + L.xst, &kmap, bars + S_XK, DR, tok0, bh);
                last_xk = 0;
            }
            // the parameter tables come from the kernel before: every MMA, and so every write of
            // this kernel (Gamma_K stores, segment memories), follows this wait
            grid_dependency_wait();
            mbar_arrive_expect_tx(bars + S_BIMG, (uint32_t)a.bimg_bytes);
            bulk_g2s(smem + L.bimg, table_of(a, h), (uint32_t)a.bimg_bytes, bars + S_BIMG);
            // each load as soon as its buffer is free, whichever comes first: the key rows of chunk
            // nx once chunk nx - 1's were read, the values of chunk nv once the update of chunk
            // nv - 2 is done (neither test can see a phase ahead: each next phase needs a load this
            // loop has not issued yet); bounded like every wait
            int nx = 1, nv = 2;
            long long t0 = clock64();
            while (ok && (nx < nch || nv < nch)) {
                bool progress = false;
                if (nx < nch && mbar_test_wait(bars + S_XF, (nx - 1) & 1)) {
                    load_x_tile(smem + L.xst, &kmap, bars + S_XK, DR, tok0 + nx * C, bh);
                    last_xk = nx++;
                    progress = true;
                }
                if (nv < nch && mbar_test_wait(bars + S_SD0 + (nv & 1), ((nv - 2) >> 1) & 1)) {
                    if (nv & 1) vpend1 = false; else vpend0 = false;
                    load_v(nv++);
                    progress = true;
                }
                if (progress) {
                    t0 = clock64();
                } else if (*abort) {
                    ok = false;
                } else if (wait_expired(clock64() - t0, a.hdr)) {
                    record_error(a.hdr, GMA_ERR_TIMEOUT, 88);
                    *abort = 1;
                    ok = false;
                } else {
                    __nanosleep(32);
                }
            }
            // loads still in flight (only after a timeout) complete before shared memory is released
            if (last_xk >= 0) mbar_wait(bars + S_XK, last_xk & 1, a.hdr, 86);
            if (vpend0 && vlast0 >= 0) mbar_wait(bars + S_V0, (vlast0 >> 1) & 1, a.hdr, 86);
            if (vpend1 && vlast1 >= 0) mbar_wait(bars + S_V1, (vlast1 >> 1) & 1, a.hdr, 86);
        }
    } else {
        // ============================================================ key-side groups
        const int g = warp >> 2;            // group: chunks c with c % 2 == g
        const int k = t & 127;              // TMEM lane, token row, component row
        const uint32_t lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        uint8_t *gk = smem + (g ? L.gk1 : L.gk0);
        if (a.lse_k) grid_dependency_wait();   // (the rows' log2-sum-exp come from the kernel before)
        for (int c = g; c < nch; c += 2) {
            const int n = c >> 1;
            const int base = tok0 + c * C;
            // the [x^2, x] buffer is free once the previous chunk's logits are done
            // (components in tiles: the row's log2-sum-exp over all components, read ahead)
            const bool kvalid = base + k < tok_end;
            const float lse = (a.lse_k && kvalid) ? a.lse_k[(long long)bh * a.N + base + k] : 0.f;
            if (c >= 1 && !mbar_wait_abortable(bars + S_LK0 + ((c - 1) & 1), ((c - 1) >> 1) & 1, a.hdr, 90, abort)) break;
            if (!mbar_wait_abortable(bars + S_XK, c & 1, a.hdr, 94, abort)) break;
            // the staged row into registers, the staging buffer released (the next chunk's rows
            // load during this chunk's conversion), then [x^2, x] into the A tile
            uint4 xr[DR / 8];
#pragma unroll
            for (int q = 0; q < DR / 8; ++q) xr[q] = *reinterpret_cast<const uint4 *>(smem + L.xst + xs_off<DR>(k, q));
            fence_proxy_async_smem();   // (these reads come before the next chunk's TMA overwrites the rows)
            mbar_arrive(bars + S_XF);
            build_a<DR>(smem + L.abuf, k, xr);
            fence_proxy_async_smem();
            // (a test of the timeout path withholds the first chunk's signal: every wait on it
            // runs out, and all roles leave their loops)
            if (!(a.test_withhold && c == 0)) mbar_arrive(bars + S_AK);
            if (!mbar_wait_abortable(bars + S_LK0 + g, n & 1, a.hdr, 91, abort)) break;
            if (c >= 2 && !mbar_wait_abortable(bars + S_SD0 + g, (n - 1) & 1, a.hdr, 92, abort)) break;
            tc_fence_after();
            if (a.lse_k)
                key_gamma_lse(lane + (g ? SR_L1 : SR_L0), a.K, kc, kvalid, gk, k, lse);
            else
                key_softmax_lean(lane + (g ? SR_L1 : SR_L0), a.K, kc, kvalid, gk, k);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bars + S_GK0 + g);
        }
        // group 0 writes the segment's memory once the last update is done
        if (g == 0 && !*abort) {
            float *dst = a.agg + (((size_t)bh * a.nseg + seg) * KMAX + k) * ne;
            bool ok = nch > 0 && mbar_wait_abortable(bars + S_FIN, 0, a.hdr, 93, abort);
            if (nch == 0) {
                for (int cc = 0; cc < ne; ++cc) dst[cc] = 0.f;
            } else if (ok) {
                tc_fence_after();
                for (int b = 0; b < ne / 16; ++b) {
                    uint32_t r[16];
                    tmem_ld16(lane + SR_S + 16 * b, r);
                    tmem_ld_wait();
                    float4 *o4 = reinterpret_cast<float4 *>(dst + 16 * b);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        o4[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 8) tmem_dealloc(tmem, 512);
}

uint32_t segmem_pipelined_smem(int d_r, int kn16, int d_v)
{
    const uint32_t need = SegSmem(d_r, kn16, d_v).total + 1024;
    return need <= 227u * 1024u ? smem_for(need, 512) : 0;
}

template <int DR>
gma_status_t launch_segmem_pipelined(const Args &a, const CUtensorMap &vmap, const CUtensorMap &kmap,
                                     const CUtensorMap &gmap, int nblocks, cudaStream_t st)
{
    const uint32_t sm = segmem_pipelined_smem(DR, a.kn16, a.d_v);
    if (sm == 0) return GMA_ERR_UNSUPPORTED_SHAPE;
    if (!set_smem(tc_segment_memory_pipelined_kernel<DR>, sm)) return GMA_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    GMA_LAUNCH(KID_TC_CAUSAL_AGG, st,
               (e = launch_pdl(tc_segment_memory_pipelined_kernel<DR>, dim3(nblocks), dim3(STHREADS), sm, st, a, vmap,
                               kmap, gmap)));
    return e == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

template gma_status_t launch_segmem_pipelined<16>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                                    const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_segmem_pipelined<32>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                                    const CUtensorMap &, int, cudaStream_t);
template gma_status_t launch_segmem_pipelined<64>(const Args &, const CUtensorMap &, const CUtensorMap &,
                                                    const CUtensorMap &, int, cudaStream_t);

}  // namespace tck
}  // namespace gma
