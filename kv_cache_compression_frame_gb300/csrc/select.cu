// Score finish, Top-B selection and the in-place compressed-state update.
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"),
// 关键设计 2: the candidate pool U_n is the compressed state's tokens plus the
// frame's T tokens; each candidate j is scored by the mean attention the
// frame's queries paid to it, s_j; S̄_n = TopK({s_j}, B) forms C_n.
//
// One CTA per (stream, layer, KV head):
//   1. s_j = (sum over query-row tiles of the column sums of P) / (G*T), in a
//      fixed tile order (deterministic);
//   2. every candidate gets the 64-bit key (float bits of s_j) << 32 |
//      ~position: s_j >= 0, so the bit pattern orders like the value, and the
//      complemented position makes the lower position win a tie.  Keys are
//      distinct, so "keep the B largest keys" is exactly Top-B with the tie
//      rule;
//   3. an MSB-first radix select (8-bit digits from the highest bit where
//      keys differ; histograms shared by warp pairs) finds the E-th smallest
//      key, E = m - B;
//      keys at or below it are evicted;
//      (window policy, the sliding-window baseline: the key is the position,
//      so the B most recent tokens are kept);
//   4. slot reuse: the pool is [compressed slots 0..c) ; frame rows c..c+T).
//      Evicted slots below B ("holes") are refilled by surviving rows at or
//      above B ("movers"), paired in slot order; only those rows move
//      (<= T rows of K and V per unit instead of rewriting all B).
#include "statekv_internal.cuh"
#include "sm100_ptx.cuh"

namespace statekv {
namespace {

constexpr int kThreads = 1024;
constexpr int kHists = 16;                      // radix histograms, each shared by 2 warps

__device__ __forceinline__ uint64_t cand_key(float s, int32_t pos) {
    return ((uint64_t)__float_as_uint(s) << 32) | (uint64_t)(0xffffffffu - (uint32_t)pos);
}

__global__ void __launch_bounds__(kThreads) select_kernel(SelectArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint64_t* keys = reinterpret_cast<uint64_t*>(smem_raw);          // [slots]
    uint32_t* whist = reinterpret_cast<uint32_t*>(keys + a.slots);   // [kHists][256]
    uint32_t* kept_bits = whist + kHists * 256;                      // [ceil(slots/32)]
    // holes / movers [T] each reuse the key buffer once the keys are dead
    int32_t* holes = reinterpret_cast<int32_t*>(keys);
    int32_t* movers = holes + a.T;
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_tot[2][kThreads / 32];
    __shared__ uint64_t s_prefix, s_wand[kThreads / 32], s_wor[kThreads / 32];
    __shared__ uint32_t s_rank;
    __shared__ uint32_t s_unique;

    // launched while the attention kernel still runs (programmatic dependent
    // launch): its column partials and the pool are read only after it has
    // finished.  Then the next frame's RoPE kernel may start (it rewrites
    // Q', which the attention kernel read, and waits for this grid before
    // it writes the pool rows read here)
    ptx::dep_wait();
    ptx::dep_trigger();
    const int u = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int c = a.c, T = a.T, B = a.B;
    const int m = c + T;
    int32_t* pos = a.pos + (int64_t)u * a.slots;

    // ---- 1-2. scores, positions, keys.  A thread issues every load of its
    // KU keys (the partials of up to TU query tiles each, and the positions)
    // before it adds or stores anything: one memory round trip per KU keys
    // instead of one per tile (the position and score buffers may alias as
    // far as the compiler knows, which would otherwise serialise them too)
    const float* cs = a.colsum + (int64_t)u * a.n_row_tiles * a.m_pad;
    float* scores = a.scores + (int64_t)u * a.m_pad;
    int32_t* spos = a.score_pos + (int64_t)u * a.m_pad;
    constexpr int KU = 2, TU = 12;
    const int n_rt = a.n_row_tiles;
    uint64_t k_and = ~0ull, k_or = 0ull;
    for (int j0 = tid; j0 < m; j0 += KU * kThreads) {
        float sv[KU];
        int32_t pv[KU];
#pragma unroll
        for (int q = 0; q < KU; ++q) {
            const int j = j0 + q * kThreads;
            sv[q] = 0.f;
            pv[q] = 0;
            if (j < m) pv[q] = j < c ? pos[j] : a.pos_base + (j - c);
        }
        for (int t0 = 0; t0 < n_rt; t0 += TU) {
            float part[KU][TU];
#pragma unroll
            for (int q = 0; q < KU; ++q) {
                const int j = j0 + q * kThreads;
#pragma unroll
                for (int tt = 0; tt < TU; ++tt)
                    part[q][tt] = (j < m && t0 + tt < n_rt)
                                      ? __ldcg(cs + (int64_t)(t0 + tt) * a.m_pad + j) : 0.f;
            }
            // tile order: s_j has the same bits whatever the tiling above
#pragma unroll
            for (int q = 0; q < KU; ++q)
#pragma unroll
                for (int tt = 0; tt < TU; ++tt)
                    if (t0 + tt < n_rt) sv[q] += part[q][tt];
        }
#pragma unroll
        for (int q = 0; q < KU; ++q) {
            const int j = j0 + q * kThreads;
            if (j < m) {
                sv[q] *= a.inv_rows;
                scores[j] = sv[q];
                spos[j] = pv[q];
                if (m > B) {
                    const uint64_t k = a.window ? (uint64_t)(uint32_t)pv[q] << 32 : cand_key(sv[q], pv[q]);
                    keys[j] = k;
                    k_and &= k;
                    k_or |= k;
                }
            }
        }
    }
    if (m <= B) {                               // state not full: keep all
        for (int j = c + tid; j < m; j += kThreads) pos[j] = a.pos_base + (j - c);
        return;
    }

    // ---- 3. radix select of the E-th smallest key.  Bits every key shares
    // are skipped (the score's sign and exponent bits usually): the first
    // digit starts at the highest bit where keys differ.  Warps w and
    // w + kHists share a histogram, so few increments of different warps
    // collide on one address (with one histogram, every warp's increment
    // of the one bucket all keys share serialised).
    // AND and OR of all keys: per warp, then every warp folds the warps'
    // partials itself (no second barrier)
    auto and64 = [](uint64_t v) {
        return ((uint64_t)__reduce_and_sync(0xffffffffu, (uint32_t)(v >> 32)) << 32) |
               __reduce_and_sync(0xffffffffu, (uint32_t)v);
    };
    auto or64 = [](uint64_t v) {
        return ((uint64_t)__reduce_or_sync(0xffffffffu, (uint32_t)(v >> 32)) << 32) |
               __reduce_or_sync(0xffffffffu, (uint32_t)v);
    };
    {
        const uint64_t wa = and64(k_and), wo = or64(k_or);
        if (lane == 0) { s_wand[warp] = wa; s_wor[warp] = wo; }
    }
    for (int e = tid; e < kHists * 256; e += kThreads) whist[e] = 0u;
    __syncthreads();
    const uint64_t k_all_and = and64(s_wand[lane]), k_all_or = or64(s_wor[lane]);
    const uint64_t diff = k_all_and ^ k_all_or; // keys are distinct: diff != 0
    const int top = 63 - __clzll((long long)diff);
    uint64_t prefix = top < 63 ? (k_all_and & (~0ull << (top + 1))) : 0ull;
    uint32_t rank = (uint32_t)(m - B);          // E: the E-th smallest key is evicted last
    int hi = top;                               // highest bit of the current digit
    while (hi >= 0) {
        const int width = min(8, hi + 1);
        const int shift = hi + 1 - width;
        const uint32_t dmask = (1u << width) - 1u;
        uint32_t* wh = whist + (warp % kHists) * 256;
        for (int j0 = 0; j0 < m; j0 += kThreads) {
            const int j = j0 + tid;
            bool act = false;
            uint32_t dig = 0;
            if (j < m) {
                const uint64_t k = keys[j];
                act = hi == 63 || (k >> (hi + 1)) == (prefix >> (hi + 1));
                dig = (uint32_t)(k >> shift) & dmask;
            }
            // one shared atomic per key: with the common high bits skipped the
            // digits spread, and aggregating equal digits first (match_any)
            // cost more than the few same-address conflicts it saves
            if (act) atomicAdd(&wh[dig], 1u);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t acc = 0;
#pragma unroll
            for (int w = 0; w < kHists; ++w) acc += whist[w * 256 + tid];
            hist[tid] = acc;
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t h[8], run = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) { h[e] = hist[lane * 8 + e]; run += h[e]; }
            uint32_t incl = run;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t excl = incl - run;
            if (excl < rank && rank <= incl) {
                uint32_t below = excl;
                int b = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (below + h[e] >= rank) { b = e; break; }
                    below += h[e];
                }
                s_prefix = prefix | ((uint64_t)(lane * 8 + b) << shift);
                s_rank = rank - below;
                s_unique = h[b] == 1u ? 1u : 0u;
            }
        } else {
            // the histograms are read; clear them for the next digit
            for (int e = tid - 32; e < kHists * 256; e += kThreads - 32) whist[e] = 0u;
        }
        __syncthreads();
        prefix = s_prefix;
        rank = s_rank;
        if (s_unique) {
            // one key has this prefix: it is the E-th smallest; fetch it whole
            // and skip the remaining digits (usually the position digits)
            const uint64_t pre = s_prefix >> shift;
            __syncthreads();
            for (int j = tid; j < m; j += kThreads)
                if ((keys[j] >> shift) == pre) s_prefix = keys[j];
            __syncthreads();
            break;
        }
        hi -= width;
    }
    const uint64_t kappa = s_prefix;            // E-th smallest key: evict <= kappa

    // ---- 4. holes (slots < B evicted) and movers (slots >= B kept), slot
    // order: a kept-bit per candidate (coalesced key reads), then each thread
    // counts and lists the candidates of its contiguous chunk from the bits
    for (int j0 = 0; j0 < m; j0 += kThreads) {
        const int j = j0 + tid;
        const uint32_t bits = __ballot_sync(0xffffffffu, j < m && keys[j] > kappa);
        if (lane == 0 && j0 + warp * 32 < m) kept_bits[(j0 >> 5) + warp] = bits;
    }
    __syncthreads();                            // keys dead: holes / movers may overwrite them
    auto kept_at = [&](int j) -> bool { return (kept_bits[j >> 5] >> (j & 31)) & 1u; };
    const int per = (m + kThreads - 1) / kThreads;
    const int j0 = tid * per, j1 = min(j0 + per, m);
    uint32_t nh = 0, nm = 0;
    for (int j = j0; j < j1; ++j) {
        const bool kept = kept_at(j);
        nh += (j < B && !kept);
        nm += (j >= B && kept);
    }
    // block-wide exclusive scan of (nh, nm)
    uint32_t ih = nh, im = nm;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        uint32_t yh = __shfl_up_sync(0xffffffffu, ih, off);
        uint32_t ym = __shfl_up_sync(0xffffffffu, im, off);
        if (lane >= off) { ih += yh; im += ym; }
    }
    if (lane == 31) { warp_tot[0][warp] = ih; warp_tot[1][warp] = im; }
    __syncthreads();
    if (warp == 0) {
        uint32_t th = warp_tot[0][lane], tm = warp_tot[1][lane];
        uint32_t ph = th, pm = tm;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            uint32_t yh = __shfl_up_sync(0xffffffffu, ph, off);
            uint32_t ym = __shfl_up_sync(0xffffffffu, pm, off);
            if (lane >= off) { ph += yh; pm += ym; }
        }
        warp_tot[0][lane] = ph - th;
        warp_tot[1][lane] = pm - tm;
    }
    __syncthreads();
    uint32_t oh = warp_tot[0][warp] + ih - nh;
    uint32_t om = warp_tot[1][warp] + im - nm;
    for (int j = j0; j < j1; ++j) {
        const bool kept = kept_at(j);
        if (j < B && !kept) holes[oh++] = j;
        if (j >= B && kept) movers[om++] = j;
        // surviving frame rows that stay in place get their position
        if (kept && j >= c && j < B) pos[j] = a.pos_base + (j - c);
    }
    // the last thread's end offsets are the totals; every hole gets a mover
    __shared__ uint32_t s_pairs;
    if (tid == kThreads - 1) {
        s_pairs = min(oh, om);
        if (oh != om) record_error(a.err, (uint32_t)STATEKV_E_DEVICE, kSiteSelect, oh * 65536u + om);
    }
    __syncthreads();
    const uint32_t np = s_pairs;
    for (uint32_t r = tid; r < np; r += kThreads) pos[holes[r]] = a.pos_base + (movers[r] - c);

    // ---- row moves (K and V), 16-byte vectors.  Holes are slots < B and
    // movers slots >= B, so no row is both read and written: each thread
    // issues all its loads (up to 4 vectors of K and of V) before its stores,
    // one memory round trip instead of one per vector
    constexpr int MV = 4;
    const int vpr = a.row_bytes / 16;
    const int64_t unit_bytes = (int64_t)a.slots * a.row_bytes;
    uint4* pk = reinterpret_cast<uint4*>((char*)a.pool_k + u * unit_bytes);
    uint4* pv = reinterpret_cast<uint4*>((char*)a.pool_v + u * unit_bytes);
    const int64_t total = (int64_t)np * vpr;
    for (int64_t e0 = tid; e0 < total; e0 += MV * kThreads) {
        uint4 vk[MV], vv[MV];
        int64_t dst[MV];
#pragma unroll
        for (int q = 0; q < MV; ++q) {
            const int64_t e = e0 + (int64_t)q * kThreads;
            dst[q] = -1;
            if (e < total) {
                const int r = (int)(e / vpr), w = (int)(e - (int64_t)r * vpr);
                const int64_t src = (int64_t)movers[r] * vpr + w;
                dst[q] = (int64_t)holes[r] * vpr + w;
                vk[q] = pk[src];
                vv[q] = pv[src];
            }
        }
#pragma unroll
        for (int q = 0; q < MV; ++q)
            if (dst[q] >= 0) { pk[dst[q]] = vk[q]; pv[dst[q]] = vv[q]; }
    }
}

}  // namespace

size_t select_smem_bytes(int slots, int T) {
    (void)T;                                    // holes / movers live in the key buffer
    return (size_t)slots * sizeof(uint64_t) + (size_t)kHists * 256 * sizeof(uint32_t) +
           (size_t)(slots + 31) / 32 * sizeof(uint32_t);
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
    // a handle that never evicts never reaches the key buffer
    size_t smem = a.never_evicts ? 0 : select_smem_bytes(a.slots, a.T);
    cudaError_t e = cudaFuncSetAttribute(select_kernel,
        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.U);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_kernel, a);
}

}  // namespace statekv
