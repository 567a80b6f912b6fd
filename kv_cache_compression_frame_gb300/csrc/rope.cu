// RoPE at virtual stream positions, with the detailed-state append fused in.
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"),
// 关键设计 3: every rotation angle uses the logical position L_n = nT (+ i) of
// the token in the stream, with one global scale alpha fixed for the whole
// run; 关键设计 1: the frame's K/V go to the detailed state D_n and join the
// candidate pool next to the compressed state.
//
// Two kernels:
//  * rope_table: cos/sin of p*omega_k for every position the detailed state
//    can hold, once per handle (the frames' and the decoded text's).  The
//    angle reaches ~1.3e5 rad at 512 frames, where an fp32 product p*omega
//    loses ~1e-2 rad, so the product and the reduction to [-pi, pi] are done
//    in fp64;
//  * rope: one pass over Q, K and V of all (stream, layer, head) rows.
//    Q' goes to scratch; K' and V go to the compressed pool after its c live
//    slots and to D rows [nT, nT+T) (text tokens being decoded: D only).
//    16-byte vector loads/stores, rows of d/2 + d/2 pairs handled by
//    d/(2*VEC) threads each.
#include "statekv_internal.cuh"
#include "sm100_ptx.cuh"

namespace statekv {
namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;

__global__ void rope_table_kernel(RopeTableArgs a) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)a.T * a.half;
    if (idx >= total) return;
    const int64_t i = idx / a.half;
    const int k = (int)(idx - i * a.half);
    double ang = (double)(a.p0 + i) * a.omega[k];
    double turns = rint(ang * (1.0 / kTwoPi));
    double r = fma(-turns, kTwoPi, ang);          // in [-pi, pi] (+ rounding)
    float s, c;
    sincosf((float)r, &s, &c);
    a.cs[i * a.half + rope_cs_index(k, a.half, a.vec)] = make_float2(c, s);
}

template <typename E> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const void* p, float (&x)[N]) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            float2 f = __bfloat1622float2(h[j]);
            x[2 * j] = f.x; x[2 * j + 1] = f.y;
        }
    }
    __device__ static uint4 pack(const float (&x)[N]) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int j = 0; j < N / 2; ++j) h[j] = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
        return u;
    }
};
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const void* p, float (&x)[N]) {
        float4 f = *reinterpret_cast<const float4*>(p);
        x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
    }
    __device__ static uint4 pack(const float (&x)[N]) {
        float4 f = make_float4(x[0], x[1], x[2], x[3]);
        return *reinterpret_cast<uint4*>(&f);
    }
};

// 6 CTAs (1536 threads) per SM, 40 registers a thread: each thread has one
// 32-byte chunk pair of inputs in flight, so occupancy sets the bytes in
// flight (5 CTAs at 48 registers: 15.4 us on the 2B stack, 6: 14.6 us; 8 at 32
// registers spills: 17.9 us; two chunk pairs per thread: 16.6 us)
template <typename E>
__global__ void __launch_bounds__(256, 6) rope_kernel(RopeArgs a) {
    constexpr int VEC = Vec<E>::N;
    // the attention kernel that follows may set itself up meanwhile; it
    // waits for this grid before it touches memory
    ptx::dep_trigger();
    const int half = a.d / 2;
    const int tpr = half / VEC;                      // threads per row (a power of two)
    // 32-bit index arithmetic (create bounds every row count below 2^31) and
    // a shift for tpr: 64-bit divisions by run-time values cost ~80
    // instructions each, more than the rest of the thread's work
    const uint32_t gid = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t row = gid >> (31 - __clz(tpr));
    const int j = (int)(gid & (uint32_t)(tpr - 1));
    const uint32_t rows_q = (uint32_t)a.rows_q, rows_kv = (uint32_t)a.rows_kv;
    if (row >= rows_q + 2u * rows_kv) return;
    const int k0 = j * VEC;

    const E* src;
    uint32_t src_row;
    int kind;                                        // 0 = Q, 1 = K, 2 = V
    if (row < rows_q) { kind = 0; src = (const E*)a.q; src_row = row; }
    else if (row < rows_q + rows_kv) { kind = 1; src = (const E*)a.k; src_row = row - rows_q; }
    else { kind = 2; src = (const E*)a.v; src_row = row - rows_q - rows_kv; }
    const uint32_t unit = src_row / (uint32_t)a.T;   // (stream, layer, head) of the row
    const int i = (int)(src_row - unit * (uint32_t)a.T);   // token index in the frame

    float x[VEC], y[VEC];
    const E* base = src + (int64_t)src_row * a.d;
    Vec<E>::load(base + k0, x);
    Vec<E>::load(base + half + k0, y);
    if (kind != 2) {
        // pairs 2p, 2p+1 of this thread: one 16-byte load (rope_cs_index)
        const float4* cs = reinterpret_cast<const float4*>(a.cs + (int64_t)i * half);
#pragma unroll
        for (int p = 0; p < VEC / 2; ++p) {
            const float4 t = cs[p * tpr + j];
            const int e = 2 * p;
            float xr = fmaf(x[e], t.x, -y[e] * t.y);
            float yr = fmaf(y[e], t.x, x[e] * t.y);
            x[e] = xr; y[e] = yr;
            xr = fmaf(x[e + 1], t.z, -y[e + 1] * t.w);
            yr = fmaf(y[e + 1], t.z, x[e + 1] * t.w);
            x[e + 1] = xr; y[e + 1] = yr;
        }
    }
    uint4 lo = Vec<E>::pack(x), hi = Vec<E>::pack(y);
    if (kind == 0) {
        E* dst = (E*)a.q_rot + (int64_t)src_row * a.d;
        *reinterpret_cast<uint4*>(dst + k0) = lo;
        *reinterpret_cast<uint4*>(dst + half + k0) = hi;
        return;
    }
    E* det = (E*)(kind == 1 ? a.det_k : a.det_v) + ((int64_t)unit * a.det_pitch + a.det_row0 + i) * a.d;
    *reinterpret_cast<uint4*>(det + k0) = lo;
    *reinterpret_cast<uint4*>(det + half + k0) = hi;
    if (a.pool_k) {                                  // text tokens go to D only
        // the previous frame's selection (possibly still running: this
        // kernel may start early, see launch_rope) reads the pool's frame
        // rows, which these stores replace
        ptx::dep_wait();
        E* pool = (E*)(kind == 1 ? a.pool_k : a.pool_v) + ((int64_t)unit * a.slots + a.c + i) * a.d;
        *reinterpret_cast<uint4*>(pool + k0) = lo;
        *reinterpret_cast<uint4*>(pool + half + k0) = hi;
    }
}

}  // namespace

cudaError_t launch_rope_table(const RopeTableArgs& a, cudaStream_t st) {
    const int64_t blocks = ((int64_t)a.T * a.half + 255) / 256;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    rope_table_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// early: the kernel may start while the previous kernel of the stream (the
// previous frame's selection, which triggers its dependents as soon as it
// has waited for the attention kernel before it) still runs.  Safe because
// that attention has then ended, so Q' (read by it) may be rewritten at
// once, and the pool rows the selection reads are written after
// dep_wait().  Inputs q, k, v were written before the selection was queued
// or by an operation between the two, which then orders them as usual.
cudaError_t launch_rope(const RopeArgs& a, int dtype, cudaStream_t st, bool early) {
    int vec = dtype == STATEKV_BF16 ? 8 : 4;
    int64_t threads = (a.rows_q + 2 * a.rows_kv) * (a.d / 2 / vec);
    int64_t blocks = (threads + 255) / 256;
    // the kernel's 32-bit thread index
    if (blocks * 256 > 0xffffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    if (dtype == STATEKV_BF16) return cudaLaunchKernelEx(&cfg, rope_kernel<__nv_bfloat16>, a);
    return cudaLaunchKernelEx(&cfg, rope_kernel<float>, a);
}

}  // namespace statekv
