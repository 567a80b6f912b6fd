// statekv_attend_scores_static: frame attention plus importance scores with
// no device allocation at all.
//
// Some callers cannot call cudaMalloc: their device memory belongs to
// another allocator (an inference server's memory pool, a framework that
// hosts this library as a plugin), or they must not risk the implicit
// device-wide synchronisation that cudaMalloc/cudaFree can cause in a
// latency-critical loop.  They cannot create a statekv handle, which
// allocates its state and scratch up front.  This entry point takes every
// input and output from the caller and keeps its only scratch -- the
// per-query-tile column sums of P that become the scores -- in a file-scope
// __device__ array of fixed size.
//
// The array lives in the module image: every GPU that loads this library
// holds kStaticScratchBytes of it until the process exits.  All calls on a
// device share it, so calls that overlap on the GPU (different streams, no
// ordering between them) race on it; serialise them.  The attention kernel
// writes every scratch element that the score reduction later reads, in the
// same call, so nothing has to be cleared between calls.
//
// In host code the array's name is only a host-side stand-in.  Its device
// address is taken with cudaGetSymbolAddress once per device, with that
// device current, on the first call made on it; make that first call before
// any stream capture.
#include <mutex>

#include "statekv_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;              // 16 MiB
constexpr size_t kStaticScratchFloats = kStaticScratchBytes / sizeof(float);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_colsum_scratch[kStaticScratchFloats];

struct StaticScratch {
    float* colsum = nullptr;
    bool ready = false;
};
StaticScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// A failed CUDA call: clear the runtime's last-error state (a refused launch,
// for instance, would otherwise be reported again by the next call that
// checks it, in this library or the caller's code) and report E_CUDA.
int cuda_fail() {
    cudaGetLastError();
    return STATEKV_E_CUDA;
}

// Device address of the static scratch for the current device.
int scratch_for_device(int dev, StaticScratch** out) {
    if (dev < 0 || dev >= kMaxDevices) return STATEKV_E_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    StaticScratch& s = g_scratch[dev];
    if (!s.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_colsum_scratch) != cudaSuccess) return cuda_fail();
        s.colsum = static_cast<float*>(p);
        s.ready = true;
    }
    *out = &s;
    return STATEKV_OK;
}

// s_j = (sum over query tiles of the column sums) / (G*T), fixed tile order.
__global__ void finish_scores_kernel(const float* colsum, float* scores, int units,
                                     int n_row_tiles, int m_pad, int m, float inv_rows) {
    const int u = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= units || j >= m) return;
    const float* cs = colsum + (int64_t)u * n_row_tiles * m_pad;
    float acc = 0.f;
    for (int t = 0; t < n_row_tiles; ++t) acc += cs[(int64_t)t * m_pad + j];
    scores[(int64_t)u * m + j] = acc * inv_rows;
}

}  // namespace

extern "C" int statekv_attend_scores_static(
    const void* q_rot, const void* pool_k, const void* pool_v, int32_t units, int32_t group,
    int32_t frame_tokens, int32_t head_dim, int32_t pool_rows, int32_t compressed,
    double logit_scale, int32_t dtype, void* o, float* scores, uint32_t* status,
    void* cuda_stream) {
    using namespace statekv;
    for (const void* p : {q_rot, pool_k, pool_v, static_cast<const void*>(o)})
        if (!p || reinterpret_cast<uintptr_t>(p) % 16) return STATEKV_E_INVALID_ARG;
    if (!scores || !status || reinterpret_cast<uintptr_t>(status) % 4) return STATEKV_E_INVALID_ARG;
    if (units < 1 || group < 1 || frame_tokens < 1 || compressed < 0 ||
        pool_rows < compressed + frame_tokens || !(logit_scale > 0.0))
        return STATEKV_E_INVALID_ARG;
    if (dtype != STATEKV_BF16 && dtype != STATEKV_F32) return STATEKV_E_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return STATEKV_E_UNSUPPORTED;
    const int64_t GT = (int64_t)group * frame_tokens;
    if (GT > 65536 || (int64_t)pool_rows > kMaxSlots) return STATEKV_E_UNSUPPORTED;
    const int row_tile = dtype == STATEKV_BF16 ? kTcRowTile : kSimtRowTile;
    const int64_t n_row_tiles = (GT + row_tile - 1) / row_tile;
    const int64_t m_pad = (pool_rows + 127) / 128 * 128;
    if ((int64_t)units * n_row_tiles * m_pad > (int64_t)kStaticScratchFloats)
        return STATEKV_E_CAPACITY;          // larger than the fixed 16 MiB scratch

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
    StaticScratch* sc = nullptr;
    int r = scratch_for_device(dev, &sc);
    if (r != STATEKV_OK) return r;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    // the status word reports this call only: a failure keeps the first
    // error it finds in a zero word, so a stale one would hide it
    if (cudaMemsetAsync(status, 0, kErrWords * sizeof(uint32_t), st) != cudaSuccess)
        return cuda_fail();

    AttnArgs a{};
    a.q_rot = q_rot; a.pool_k = pool_k; a.pool_v = pool_v; a.o = o;
    a.colsum = sc->colsum;
    a.err = status;
    a.U = units; a.GT = (int32_t)GT; a.T = frame_tokens; a.d = head_dim;
    a.slots = pool_rows; a.c = compressed; a.m_pad = (int32_t)m_pad;
    a.n_row_tiles = (int32_t)n_row_tiles;
    a.scale = (float)logit_scale;
    a.scale_log2 = (float)(logit_scale * 1.4426950408889634074);
    cudaError_t e;
    if (dtype == STATEKV_BF16) {
        TcMaps maps;
        if (!make_tc_maps(&maps, pool_k, pool_v, head_dim, pool_rows, units))
            return cuda_fail();
        e = launch_attention_tc(a, maps, st);
    } else {
        e = launch_attention_simt(a, st);
    }
    if (e != cudaSuccess) return cuda_fail();
    const int m = compressed + frame_tokens;
    dim3 grid((unsigned)((m + 255) / 256), (unsigned)units);
    finish_scores_kernel<<<grid, 256, 0, st>>>(sc->colsum, scores, units, (int)n_row_tiles,
                                                (int)m_pad, m, (float)(1.0 / (double)GT));
    return cudaGetLastError() == cudaSuccess ? STATEKV_OK : STATEKV_E_CUDA;
}
