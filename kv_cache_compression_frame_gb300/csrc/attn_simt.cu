// fp32 frame attention on CUDA cores, for fp32 storage.
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"),
// 关键设计 1: the frame's queries attend over [K̄_{n-1}; K_n] (compressed keys
// all visible, frame keys causal); 关键设计 2: the importance of key j is the
// attention it receives, so every tile also emits the column sums of the
// normalised probabilities P.
//
// Two sweeps over the key tiles of a 16-row query block:
//   sweep 1: running max / sum of exp -> per-row log-sum-exp;
//   sweep 2: P = exp(S - lse) (exact, final), O += P V, column sums of P.
// TF32 tensor cores would miss a 1e-5 relative tolerance, so this path stays
// on FFMA.  It is the small-shape path; bf16 storage uses the tcgen05 kernel.
#include "statekv_internal.cuh"

namespace statekv {
namespace {

constexpr int RB = kSimtRowTile;   // query rows per block
constexpr int KB = 32;             // keys per tile
constexpr int NT = 128;            // threads: 16 rows x 8 lanes

template <int D>
__global__ void __launch_bounds__(NT) attn_simt_kernel(AttnArgs a) {
    __shared__ float Qs[RB][D + 1];
    __shared__ float Ks[KB][D + 1];
    __shared__ float Vs[KB][D];
    __shared__ float Ps[RB][KB + 1];

    const int n_rb = a.n_row_tiles;
    const int u = blockIdx.x / n_rb;
    const int rb = blockIdx.x - u * n_rb;
    const int tid = threadIdx.x;
    const int r = tid >> 3;           // row within block
    const int sub = tid & 7;          // lane within the row group
    const int row = rb * RB + r;      // row within the unit (g*T + i)
    const bool valid = row < a.GT;
    const int i = valid ? row % a.T : 0;
    const int lim = valid ? a.c + i : -1;      // key kk visible iff kk <= lim

    // key range of the block
    const int r0 = rb * RB;
    const int r1 = min(r0 + RB, a.GT) - 1;
    int imax = (r0 / a.T == r1 / a.T) ? (r1 % a.T) : (a.T - 1);
    const int nkeys = a.c + imax + 1;
    const int ntiles = (nkeys + KB - 1) / KB;

    const float* q = (const float*)a.q_rot + ((int64_t)u * a.GT + r0) * D;
    for (int e = tid; e < RB * D; e += NT) {
        int rr = e / D;
        Qs[rr][e % D] = (r0 + rr < a.GT) ? q[e] : 0.f;
    }
    const float* pk = (const float*)a.pool_k + (int64_t)u * a.slots * D;
    const float* pv = (const float*)a.pool_v + (int64_t)u * a.slots * D;

    auto load_tile = [&](int t, bool with_v) {
        for (int e = tid; e < KB * D; e += NT) {
            int kr = e / D, dd = e % D;
            int kk = t * KB + kr;
            bool in = kk < a.c + a.T;
            Ks[kr][dd] = in ? pk[(int64_t)kk * D + dd] : 0.f;
            if (with_v) Vs[kr][dd] = in ? pv[(int64_t)kk * D + dd] : 0.f;
        }
    };
    auto scores = [&](int t, float (&s)[KB / 8]) {
#pragma unroll
        for (int e = 0; e < KB / 8; ++e) {
            int kr = sub + 8 * e;
            float acc = 0.f;
#pragma unroll 16
            for (int dd = 0; dd < D; ++dd) acc = fmaf(Qs[r][dd], Ks[kr][dd], acc);
            int kk = t * KB + kr;
            s[e] = (kk <= lim) ? acc * a.scale : -INFINITY;
        }
    };

    // ---------------- sweep 1: log-sum-exp per row
    float m = -INFINITY, l = 0.f;
    for (int t = 0; t < ntiles; ++t) {
        __syncthreads();
        load_tile(t, false);
        __syncthreads();
        float s[KB / 8];
        scores(t, s);
        float mx = s[0];
#pragma unroll
        for (int e = 1; e < KB / 8; ++e) mx = fmaxf(mx, s[e]);
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float mn = fmaxf(m, mx);
        if (mn != -INFINITY) {
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < KB / 8; ++e) sum += expf(s[e] - mn);
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            l = l * expf(m - mn) + sum;
            m = mn;
        }
    }
    const float lse = valid ? m + logf(l) : INFINITY;

    // ---------------- sweep 2: P, O = P V, column sums of P
    constexpr int DPT = D / 8;             // output columns per thread
    float o[DPT];
#pragma unroll
    for (int e = 0; e < DPT; ++e) o[e] = 0.f;
    float* colsum = a.colsum + ((int64_t)u * n_rb + rb) * a.m_pad;
    for (int t = 0; t < ntiles; ++t) {
        __syncthreads();
        load_tile(t, true);
        __syncthreads();
        float s[KB / 8];
        scores(t, s);
#pragma unroll
        for (int e = 0; e < KB / 8; ++e)
            Ps[r][sub + 8 * e] = (s[e] == -INFINITY) ? 0.f : expf(s[e] - lse);
        __syncthreads();
        if (tid < KB) {
            float cs = 0.f;
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) cs += Ps[rr][tid];
            colsum[t * KB + tid] = cs;
        }
#pragma unroll 4
        for (int kr = 0; kr < KB; ++kr) {
            float p = Ps[r][kr];
#pragma unroll
            for (int e = 0; e < DPT; ++e) o[e] = fmaf(p, Vs[kr][sub + 8 * e], o[e]);
        }
    }
    for (int kk = ntiles * KB + tid; kk < a.m_pad; kk += NT) colsum[kk] = 0.f;
    if (valid) {
        float* out = (float*)a.o + ((int64_t)u * a.GT + row) * D;
#pragma unroll
        for (int e = 0; e < DPT; ++e) out[sub + 8 * e] = o[e];
    }
}

}  // namespace

cudaError_t launch_attention_simt(const AttnArgs& a, cudaStream_t st) {
    dim3 grid((unsigned)(a.U * a.n_row_tiles));
    if (a.d == 64) attn_simt_kernel<64><<<grid, NT, 0, st>>>(a);
    else if (a.d == 128) attn_simt_kernel<128><<<grid, NT, 0, st>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace statekv
