// gma_timing.cu -- optional per-launch timing with CUDA events (see gma_timing_enable).
#include <vector>

#include "gma_internal.cuh"

namespace gma {
namespace {

struct Rec {
    int kid;
    cudaEvent_t a, b;
};

struct Timing {
    bool on = false;
    std::vector<Rec> pool;   // events created once at enable time
    size_t used = 0;
    size_t dropped = 0;
    int pending_kid = 0;
};

Timing &T()
{
    static Timing t;
    return t;
}

}  // namespace

const char *kernel_name(int id)
{
    switch (id) {
    case KID_SIMT_PARAMS: return "simt_params";
    case KID_SIMT_RESP: return "simt_responsibilities";
    case KID_SIMT_STATE: return "simt_segment_memory";
    case KID_SIMT_SCAN: return "simt_segment_scan";
    case KID_SIMT_OUT: return "simt_read";
    case KID_SIMT_SMALL: return "simt_small_one_launch";
    case KID_TC_PARAMS: return "tc_params";
    case KID_TC_RESP: return "tc_responsibilities";
    case KID_TC_BIDIR_WRITE: return "tc_bidir_write";
    case KID_TC_BIDIR_READ: return "tc_bidir_read";
    case KID_TC_CAUSAL_AGG: return "tc_causal_segment_memory";
    case KID_TC_CAUSAL_SCAN: return "tc_causal_segment_scan";
    case KID_TC_CAUSAL_OUT: return "tc_causal_chunked";
    case KID_TC_LSE: return "tc_row_lse";
    case KID_TC_DIVIDE: return "tc_tile_divide";
    case KID_TC_CAUSAL_FUSED: return "tc_causal_single_launch";
    case KID_DECODE: return "decode_step";
    case KID_DECODE_PARAMS: return "decode_params";
    case KID_USAGE_ROWS: return "usage_rows";
    case KID_USAGE_MASS: return "usage_mass";
    case KID_USAGE_STATS: return "usage_stats";
    case KID_BWD_NUMDEN: return "bwd_numden";
    case KID_BWD_DQ: return "bwd_dgamma_q";
    case KID_BWD_SCAN: return "bwd_segment_scan";
    case KID_BWD_DK: return "bwd_dgamma_k_dv";
    case KID_BWD_DX: return "bwd_dx";
    case KID_BWD_PARAMS: return "bwd_param_partials";
    case KID_BWD_PFINAL: return "bwd_param_final";
    }
    return "unknown";
}

void timing_begin(cudaStream_t st, int kid)
{
    Timing &t = T();
    if (!t.on) return;
    if (t.used >= t.pool.size()) {
        ++t.dropped;
        t.pending_kid = -1;
        return;
    }
    t.pending_kid = kid;
    cudaEventRecord(t.pool[t.used].a, st);
}

void timing_end(cudaStream_t st)
{
    Timing &t = T();
    if (!t.on || t.pending_kid < 0) return;
    Rec &r = t.pool[t.used++];
    r.kid = t.pending_kid;
    cudaEventRecord(r.b, st);
}

}  // namespace gma

using namespace gma;

extern "C" {

// Enable (capacity > 0: number of launches to record) or disable (0) launch timing.  Creates
// or destroys the CUDA events; call it outside stream capture.  Returns GMA_OK or GMA_ERR_CUDA.
gma_status_t gma_timing_enable(int capacity)
{
    Timing &t = T();
    for (Rec &r : t.pool) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    t.pool.clear();
    t.used = t.dropped = 0;
    t.on = capacity > 0;
    for (int i = 0; i < capacity; ++i) {
        Rec r{0, nullptr, nullptr};
        if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) {
            t.on = false;
            return GMA_ERR_CUDA;
        }
        t.pool.push_back(r);
    }
    return GMA_OK;
}

// Copies up to `cap` recorded (kernel id, milliseconds) pairs, oldest first, waiting for each
// end event, then clears the record.  Returns the number copied (-1 on a CUDA error).
int gma_timing_read(int *kernel_ids, float *ms, int cap)
{
    Timing &t = T();
    int n = 0;
    for (size_t i = 0; i < t.used && n < cap; ++i) {
        if (cudaEventSynchronize(t.pool[i].b) != cudaSuccess) return -1;
        float v = 0.f;
        if (cudaEventElapsedTime(&v, t.pool[i].a, t.pool[i].b) != cudaSuccess) return -1;
        kernel_ids[n] = t.pool[i].kid;
        ms[n] = v;
        ++n;
    }
    t.used = 0;
    t.dropped = 0;
    return n;
}

// Name of a kernel id reported by gma_timing_read.
const char *gma_kernel_name(int kernel_id) { return kernel_name(kernel_id); }

}  // extern "C"
