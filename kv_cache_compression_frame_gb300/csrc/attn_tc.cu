// bf16 frame attention on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA), with the key column sums of P fused in.
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"):
//   关键设计 1 -- the frame's queries attend over [K̄_{n-1}; K_n]: every
//     compressed key is visible, frame keys are causal;
//   关键设计 2 -- key j's importance is the attention the frame's queries pay
//     to it, averaged over queries; this kernel emits, per 128-row query
//     tile, the column sums of the final normalised P;
//   整体框架 -- the per-frame cost O(T^2 + BT): the key loop covers only the
//     B compressed keys and the causally visible part of the frame.
//
// One CTA = one 128-row query tile of one (stream, layer, KV head).  Rows are
// (g, i) pairs of the G query heads that share the KV head, g-major.  Two
// sweeps over the 128-key tiles of the pool:
//   sweep 1: S = Q K^T (tcgen05, fp32 in TMEM) -> running row max / sum of
//            exp2 -> per-row log-sum-exp (kept in a register);
//   sweep 2: S again, P = exp2(S*scale - lse) (final, normalised), column
//            sums of fp32 P (warp reduce-scatter by shuffles, then across the
//            4 epilogue warps in shared memory), P -> bf16 -> shared memory
//            (K-major, 128B swizzle) -> O += P V on tcgen05 (V read MN-major).
// P is normalised by the global lse before PV, so O needs no rescaling.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer (one thread), warps 2..5 epilogue (TMEM lanes 32*(w%4)..+31).
// TMEM (512 columns): S double buffer at 0 and 128, O at 256.
// Every mbarrier wait is bounded; on timeout the CTA records
// STATEKV_E_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM, exits.
#include "statekv_internal.cuh"
#include "sm100_ptx.cuh"

namespace statekv {
namespace {

constexpr uint64_t kTimeoutNs = 1000000000ull;   // 1 s per wait

template <int D>
struct TcLayout {
    static constexpr int BM = 128, BN = 128;
    static constexpr int KCH = D / 64;                  // 128-byte chunks along d
    static constexpr int CHUNK = 128 * 128;             // [128 rows][64 bf16]
    static constexpr int Q_BYTES = KCH * CHUNK;
    static constexpr int KV_BYTES = KCH * CHUNK;
    static constexpr int P_BYTES = 2 * CHUNK;           // [128 rows][128 keys]
    static constexpr int NS = 2;                        // K/V pipeline stages
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
    static constexpr int OFF_P = OFF_V + NS * KV_BYTES;
    static constexpr int OFF_COL = OFF_P + P_BYTES;     // float [2][4][128]
    static constexpr int OFF_BAR = OFF_COL + 2 * 4 * 128 * 4;
    // barriers
    static constexpr int B_Q = 0;
    static constexpr int B_KV_FULL = 1;
    static constexpr int B_KV_EMPTY = B_KV_FULL + NS;
    static constexpr int B_S_FULL = B_KV_EMPTY + NS;
    static constexpr int B_S_EMPTY = B_S_FULL + 2;
    static constexpr int B_P_FULL = B_S_EMPTY + 2;
    static constexpr int B_P_EMPTY = B_P_FULL + 1;
    static constexpr int B_O_FULL = B_P_EMPTY + 1;
    static constexpr int B_DRAIN = B_O_FULL + 1;
    static constexpr int B_COL = B_DRAIN + 1;          // column-sum buffer ready [2]
    static constexpr int NBAR = B_COL + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_O = 256;
};

struct Sync {
    uint32_t bar0;                 // smem address of barrier 0
    volatile uint32_t* abort;      // CTA-wide abort flag (smem)
    uint32_t* err;

    __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }

    // Wait for the phase of the given parity; gives up on abort or timeout.
    __device__ bool wait(int i, uint32_t parity, uint32_t site) const {
        const uint32_t b = bar(i);
        if (ptx::mbar_test(b, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (ptx::mbar_test(b, parity)) return true;
            if (*abort) return false;
            if ((spin & 255u) == 0 && globaltimer_ns() - t0 > kTimeoutNs) {
                *abort = 1u;
                record_error(err, (uint32_t)STATEKV_E_TIMEOUT, site, (uint32_t)i);
                return false;
            }
        }
    }
    // Teardown wait: ignores the abort flag, still bounded.
    __device__ void drain(int i, uint32_t parity) const {
        const uint32_t b = bar(i);
        const uint64_t t0 = globaltimer_ns();
        while (!ptx::mbar_test(b, parity)) {
            if (globaltimer_ns() - t0 > kTimeoutNs) {
                record_error(err, (uint32_t)STATEKV_E_TIMEOUT, kSiteDrain, (uint32_t)i);
                return;
            }
        }
    }
};

// Column sums of a 32x32 block held one row per lane: after the call lane l
// holds the sum over the 32 lanes of column l.  Recursive halving: at each
// step a lane keeps half of its columns and adds its partner's copy of them.
__device__ __forceinline__ float warp_column_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            float send = up ? v[j] : v[j + w];
            float keep = up ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

template <int D>
__global__ void __launch_bounds__(192, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, AttnArgs a) {
    using L = TcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rt = a.n_row_tiles;
    const int u = blockIdx.x / n_rt;
    const int mt = blockIdx.x - u * n_rt;
    const int r0 = mt * L::BM;
    const int r1 = min(r0 + L::BM, a.GT) - 1;
    const bool one_head = (r0 / a.T) == (r1 / a.T);
    const int imax = one_head ? r1 % a.T : a.T - 1;
    const int imin = one_head ? r0 % a.T : 0;
    const int nkeys = a.c + imax + 1;                 // keys visible to some row
    const int nt = (nkeys + L::BN - 1) / L::BN;       // key tiles
    const int nfull = (a.c + imin + 1) / L::BN;       // tiles visible to every row

    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + L::OFF_MISC + 4);
    Sync sy{sbase + (uint32_t)L::OFF_BAR, abort_flag, a.err};

    if (threadIdx.x == 0) {
        ptx::mbar_init(sy.bar(L::B_Q), 1);
        for (int s = 0; s < L::NS; ++s) {
            ptx::mbar_init(sy.bar(L::B_KV_FULL + s), 1);
            ptx::mbar_init(sy.bar(L::B_KV_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(sy.bar(L::B_S_FULL + b), 1);
            ptx::mbar_init(sy.bar(L::B_S_EMPTY + b), 4);
        }
        ptx::mbar_init(sy.bar(L::B_P_FULL), 4);
        ptx::mbar_init(sy.bar(L::B_P_EMPTY), 1);
        ptx::mbar_init(sy.bar(L::B_O_FULL), 1);
        ptx::mbar_init(sy.bar(L::B_DRAIN), 1);
        ptx::mbar_init(sy.bar(L::B_COL), 4);
        ptx::mbar_init(sy.bar(L::B_COL + 1), 4);
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t sQ = sbase + L::OFF_Q;
    const uint32_t sK = sbase + L::OFF_K;
    const uint32_t sV = sbase + L::OFF_V;
    const uint32_t sP = sbase + L::OFF_P;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            ptx::mbar_arrive_expect_tx(sy.bar(L::B_Q), L::Q_BYTES);
            for (int kc = 0; kc < L::KCH; ++kc)
                ptx::tma_load_3d(sQ + kc * L::CHUNK, &tm_q, sy.bar(L::B_Q), kc * 64, r0, u);
            int issued_phase[L::NS];
            for (int s = 0; s < L::NS; ++s) issued_phase[s] = -1;
            int it = 0;
            for (int sweep = 0; sweep < 2; ++sweep) {
                const uint32_t bytes = L::KV_BYTES * (sweep ? 2 : 1);
                bool ok = true;
                for (int t = 0; t < nt; ++t, ++it) {
                    const int s = it % L::NS, js = it / L::NS;
                    if (!sy.wait(L::B_KV_EMPTY + s, (js & 1) ^ 1, kSiteKvEmpty)) { ok = false; break; }
                    const uint32_t fb = sy.bar(L::B_KV_FULL + s);
                    ptx::mbar_arrive_expect_tx(fb, bytes);
                    for (int kc = 0; kc < L::KCH; ++kc)
                        ptx::tma_load_3d(sK + s * L::KV_BYTES + kc * L::CHUNK, &tm_k, fb,
                                         kc * 64, t * L::BN, u);
                    if (sweep)
                        for (int kc = 0; kc < L::KCH; ++kc)
                            ptx::tma_load_3d(sV + s * L::KV_BYTES + kc * L::CHUNK, &tm_v, fb,
                                             kc * 64, t * L::BN, u);
                    issued_phase[s] = js & 1;
                }
                if (!ok) break;
            }
            // never leave a copy in flight into this CTA's shared memory
            sy.drain(L::B_Q, 0);
            for (int s = 0; s < L::NS; ++s)
                if (issued_phase[s] >= 0) sy.drain(L::B_KV_FULL + s, (uint32_t)issued_phase[s]);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, D, false, true);
            auto issue_qk = [&](uint32_t d_tmem, uint32_t k_stage) {
#pragma unroll
                for (int kc = 0; kc < L::KCH; ++kc)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        uint64_t ad = ptx::sdesc_sw128(sQ + kc * L::CHUNK + ks * 32, 16, 1024);
                        uint64_t bd = ptx::sdesc_sw128(k_stage + kc * L::CHUNK + ks * 32, 16, 1024);
                        ptx::umma_f16_ss(d_tmem, ad, bd, idesc_qk, (kc | ks) ? 1u : 0u);
                    }
            };
            auto issue_pv = [&](int tt) -> bool {
                if (!sy.wait(L::B_P_FULL, tt & 1, kSitePFull)) return false;
                ptx::tc_fence_after();
                const int sp = (nt + tt) % L::NS;
                const uint32_t v_stage = sV + sp * L::KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint64_t ad = ptx::sdesc_sw128(sP + (ks >> 2) * L::CHUNK + (ks & 3) * 32, 16, 1024);
                    // MN-major V: LBO = distance between 64-wide d chunks,
                    // SBO = distance between 8-key row groups
                    uint64_t bd = ptx::sdesc_sw128(v_stage + ks * 2048, L::CHUNK, 1024);
                    ptx::umma_f16_ss(tmem + L::TM_O, ad, bd, idesc_pv, (tt | ks) ? 1u : 0u);
                }
                ptx::umma_commit(sy.bar(L::B_P_EMPTY));
                ptx::umma_commit(sy.bar(L::B_KV_EMPTY + sp));
                return true;
            };
            bool ok = sy.wait(L::B_Q, 0, kSiteQFull);
            ptx::tc_fence_after();
            int it = 0;
            for (int t = 0; ok && t < nt; ++t, ++it) {            // sweep 1
                const int b = it & 1, jb = it >> 1, s = it % L::NS, js = it / L::NS;
                if (!sy.wait(L::B_S_EMPTY + b, (jb & 1) ^ 1, kSiteSEmpty)) { ok = false; break; }
                if (!sy.wait(L::B_KV_FULL + s, js & 1, kSiteKvFull)) { ok = false; break; }
                ptx::tc_fence_after();
                issue_qk(tmem + b * 128, sK + s * L::KV_BYTES);
                ptx::umma_commit(sy.bar(L::B_KV_EMPTY + s));
                ptx::umma_commit(sy.bar(L::B_S_FULL + b));
            }
            for (int t = 0; ok && t < nt; ++t, ++it) {            // sweep 2
                const int b = it & 1, jb = it >> 1, s = it % L::NS, js = it / L::NS;
                if (!sy.wait(L::B_S_EMPTY + b, (jb & 1) ^ 1, kSiteSEmpty)) { ok = false; break; }
                if (!sy.wait(L::B_KV_FULL + s, js & 1, kSiteKvFull)) { ok = false; break; }
                ptx::tc_fence_after();
                issue_qk(tmem + b * 128, sK + s * L::KV_BYTES);
                ptx::umma_commit(sy.bar(L::B_S_FULL + b));
                if (t > 0 && !issue_pv(t - 1)) { ok = false; break; }
            }
            if (ok && nt > 0 && issue_pv(nt - 1)) ptx::umma_commit(sy.bar(L::B_O_FULL));
            // all MMAs complete before TMEM is released
            ptx::umma_commit(sy.bar(L::B_DRAIN));
            sy.drain(L::B_DRAIN, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;                      // TMEM lane quarter
        const int row = q4 * 32 + lane;
        const int r_unit = r0 + row;
        const bool valid = r_unit < a.GT;
        const int lim = valid ? a.c + (r_unit % a.T) : -1;    // kk visible iff kk <= lim
        const uint32_t t_lane = tmem + ((uint32_t)(q4 * 32) << 16);
        float* colbuf = reinterpret_cast<float*>(base + L::OFF_COL);
        float* colsum = a.colsum + ((int64_t)u * n_rt + mt) * a.m_pad;
        const float sc = a.scale_log2;
        int it = 0;
        bool ok = true;

        // sweep 1: log-sum-exp (log2 domain)
        float mrun = -INFINITY, lrun = 0.f;
        for (int t = 0; t < nt; ++t, ++it) {
            const int b = it & 1, jb = it >> 1;
            if (!sy.wait(L::B_S_FULL + b, jb & 1, kSiteSFull)) { ok = false; break; }
            ptx::tc_fence_after();
            const bool full = t < nfull;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(t_lane + b * 128 + ch * 32, r);
                ptx::tmem_ld_wait();
                float x[32];
                float mx = -INFINITY;
                const int k0 = t * L::BN + ch * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float v = __uint_as_float(r[j]) * sc;
                    if (!full && k0 + j > lim) v = -INFINITY;
                    x[j] = v;
                    mx = fmaxf(mx, v);
                }
                const float mn = fmaxf(mrun, mx);
                if (mn != -INFINITY) {
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) sum += ptx::ex2_approx(x[j] - mn);
                    lrun = lrun * ptx::ex2_approx(mrun - mn) + sum;
                    mrun = mn;
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_S_EMPTY + b));
        }
        const float lse2 = (valid && lrun > 0.f) ? mrun + log2f(lrun) : INFINITY;

        // sweep 2: P, column sums, P -> shared memory for PV
        for (int t = 0; ok && t < nt; ++t, ++it) {
            const int b = it & 1, jb = it >> 1;
            if (!sy.wait(L::B_S_FULL + b, jb & 1, kSiteSFull)) { ok = false; break; }
            ptx::tc_fence_after();
            const bool full = t < nfull;
            uint32_t pk[4][16];
            float cval[4];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(t_lane + b * 128 + ch * 32, r);
                ptx::tmem_ld_wait();
                float p[32];
                const int k0 = t * L::BN + ch * 32;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float e = ptx::ex2_approx(fmaf(__uint_as_float(r[j]), sc, -lse2));
                    p[j] = (full || k0 + j <= lim) ? e : 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(p[2 * j], p[2 * j + 1]);
                    pk[ch][j] = *reinterpret_cast<uint32_t*>(&h);
                }
                cval[ch] = warp_column_sum32(p, lane);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_S_EMPTY + b));

            float* cb = colbuf + (t & 1) * 512 + q4 * 128;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) cb[ch * 32 + lane] = cval[ch];

            if (!sy.wait(L::B_P_EMPTY, (t & 1) ^ 1, kSitePEmpty)) { ok = false; break; }
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                const uint32_t chunk = sP + (ch >> 1) * L::CHUNK + row * 128;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t unit16 = (uint32_t)((ch & 1) * 4 + w);
                    const uint32_t addr = chunk + ((unit16 ^ (uint32_t)(row & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 :: "r"(addr), "r"(pk[ch][4 * w]), "r"(pk[ch][4 * w + 1]),
                                    "r"(pk[ch][4 * w + 2]), "r"(pk[ch][4 * w + 3]) : "memory");
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_P_FULL));

            // all four warps' partial column sums of this tile are in smem
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_COL + (t & 1)));
            if (!sy.wait(L::B_COL + (t & 1), (t >> 1) & 1, kSiteCol)) { ok = false; break; }
            const int e = q4 * 32 + lane;
            const float* cb0 = colbuf + (t & 1) * 512;
            colsum[t * L::BN + e] = cb0[e] + cb0[128 + e] + cb0[256 + e] + cb0[384 + e];
        }
        for (int kk = nt * L::BN + row; kk < a.m_pad; kk += 128) colsum[kk] = 0.f;

        // output rows
        if (ok && sy.wait(L::B_O_FULL, 0, kSiteOFull)) {
            ptx::tc_fence_after();
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o) + ((int64_t)u * a.GT + r_unit) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(t_lane + L::TM_O + ch * 32, r);
                ptx::tmem_ld_wait();
                if (valid) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * j]),
                                                                 __uint_as_float(r[2 * j + 1]));
                        w[j] = *reinterpret_cast<uint32_t*>(&h);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                }
            }
        }
        ptx::tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_tc(const AttnArgs& a, const CUtensorMap& q, const CUtensorMap& k,
                      const CUtensorMap& v, cudaStream_t st) {
    using L = TcLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    attn_tc_kernel<D><<<(unsigned)(a.U * a.n_row_tiles), 192, L::SMEM, st>>>(q, k, v, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_tc(const AttnArgs& a, const CUtensorMap& tm_q,
                                const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                cudaStream_t st) {
    if (a.d == 128) return launch_tc<128>(a, tm_q, tm_k, tm_v, st);
    if (a.d == 64) return launch_tc<64>(a, tm_q, tm_k, tm_v, st);
    return cudaErrorInvalidValue;
}

}  // namespace statekv
