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
//   2. every candidate gets the 32-bit key "float bits of s_j": s_j >= 0, so
//      the bit pattern orders like the value;
//   3. an MSB-first radix select (11-bit digits from the highest bit where
//      keys differ) finds where the E = m - B smallest keys end; it stops as
//      soon as the boundary bucket is evicted whole.  Only if that leaves
//      keys of exactly equal score on both sides of the cut does a second
//      radix select over their positions pick the lower positions to keep
//      (the tie rule);
//      (window policy, the sliding-window baseline: the key is the position,
//      so the B most recent tokens are kept);
//   4. slot reuse: the pool is [compressed slots 0..c) ; frame rows c..c+T).
//      Evicted slots below B ("holes") are refilled by surviving rows at or
//      above B ("movers"), paired in slot order; only those rows move
//      (<= T rows of K and V per unit instead of rewriting all B).
// Every step is written for a full SM of warps (one 1024-thread CTA or two
// 512-thread ones: eight warps per sub-partition): per-thread work is kept to
// a few instructions per key (32-bit keys, warp ballots for the slot-ordered
// lists), since each one costs eight issue slots.
// With few units (one layer per launch: 2-8 units on 152 SMs) a unit is a
// cluster of C CTAs: CTA r finishes the scores of candidates
// [r*m/C, (r+1)*m/C) and stores their keys into every CTA's shared memory
// (distributed shared memory); after one cluster barrier each CTA holds all
// m keys and runs steps 3-4's cut and lists itself (the same inputs, so the
// same result everywhere), then moves its share of the rows.  Step 1, which
// reads all the partials, and the row moves are spread over C SMs.
#include <cstdlib>
#include <mutex>
#include <vector>

#include "statekv_internal.cuh"
#include "sm100_ptx.cuh"

namespace statekv {
namespace {

// CTA size: 1024 threads, or 512 (two CTAs per SM) when the units are more
// than the SMs, so that every unit's CTA starts at once
constexpr int kMaxWarps = 32;
constexpr int kDigit = 11;                      // radix digit width
constexpr int kBuckets = 1 << kDigit;
constexpr int kCopies = 4;                      // histogram copies: warp w counts into w % kCopies

// Where the R smallest of a set of 32-bit keys end: keys k with
// (k >> shift) < pre are among them, the cnt keys with (k >> shift) == pre
// are at the boundary (the r smallest of them are among them; all if
// r == cnt), larger keys are not.  shift = 32 compares nothing.
struct Cut {
    uint32_t shift, pre, r, cnt;
};
__device__ __forceinline__ uint32_t hi_bits(uint32_t k, uint32_t shift) {
    return (uint32_t)((uint64_t)k >> shift);
}

struct RadixScratch {
    uint32_t* hist;                             // [kCopies][kBuckets], zero on entry and exit
    uint32_t* comb;                             // [kBuckets] the copies' sum
    uint32_t* gtot;                             // [32] per 64-bucket group
    uint32_t* out;                              // [3] bucket, rank in it, its count
};

// The cut of the R smallest among the n active keys (1 <= R <= n; key_of(j,
// k) says whether candidate j is active and sets its key); k_and / k_or are
// the AND and OR of the active keys: their common high bits need no pass.
template <int NT, class KeyOf>
__device__ Cut radix_cut(const KeyOf& key_of, int m, uint32_t n, uint32_t R, uint32_t k_and,
                         uint32_t k_or, const RadixScratch& rs) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t diff = k_and ^ k_or;
    Cut q;
    q.shift = diff ? 32u - (uint32_t)__clz(diff) : 0u;
    q.pre = hi_bits(k_and, q.shift);
    q.r = R;
    q.cnt = n;
    while (q.shift > 0 && q.r != q.cnt) {
        const uint32_t w = min((uint32_t)kDigit, q.shift), sh = q.shift - w;
        const uint32_t dmask = (1u << w) - 1u;
        uint32_t* h = rs.hist + (warp % kCopies) * kBuckets;
        for (int j = tid; j < m; j += NT) {
            uint32_t k;
            if (key_of(j, k) && hi_bits(k, q.shift) == q.pre) atomicAdd(&h[(k >> sh) & dmask], 1u);
        }
        __syncthreads();
        // bucket totals, and per group of 64 buckets (32 groups, a warp each)
        for (int grp = warp; grp < 32; grp += NT / 32) {
            const int b0 = grp * 64 + lane, b1 = b0 + 32;
            uint32_t c0 = 0, c1 = 0;
#pragma unroll
            for (int cp = 0; cp < kCopies; ++cp) {
                c0 += rs.hist[cp * kBuckets + b0];
                c1 += rs.hist[cp * kBuckets + b1];
            }
            rs.comb[b0] = c0;
            rs.comb[b1] = c1;
            const uint32_t g = __reduce_add_sync(0xffffffffu, c0 + c1);
            if (lane == 0) rs.gtot[grp] = g;
        }
        __syncthreads();
        if (warp == 0) {
            // the group holding the r-th key, then its bucket (two per lane)
            const uint32_t g = rs.gtot[lane];
            uint32_t incl = g;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t excl = incl - g;
            const int gs = __ffs(__ballot_sync(0xffffffffu, excl < q.r && q.r <= incl)) - 1;
            const uint32_t base = __shfl_sync(0xffffffffu, excl, gs);
            const uint32_t x0 = rs.comb[gs * 64 + 2 * lane], x1 = rs.comb[gs * 64 + 2 * lane + 1];
            uint32_t inc2 = x0 + x1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, inc2, off);
                if (lane >= off) inc2 += y;
            }
            const uint32_t e0 = base + inc2 - x0 - x1;          // keys below bucket 2*lane
            if (e0 < q.r && q.r <= e0 + x0) {
                rs.out[0] = (uint32_t)(gs * 64 + 2 * lane);
                rs.out[1] = q.r - e0;
                rs.out[2] = x0;
            } else if (e0 + x0 < q.r && q.r <= e0 + x0 + x1) {
                rs.out[0] = (uint32_t)(gs * 64 + 2 * lane + 1);
                rs.out[1] = q.r - e0 - x0;
                rs.out[2] = x1;
            }
        } else {
            // the copies are summed into comb: clear them for the next digit
            uint4* hv = reinterpret_cast<uint4*>(rs.hist);
            for (int e = tid - 32; e < kCopies * kBuckets / 4; e += NT - 32)
                hv[e] = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncthreads();
        q.pre = (q.pre << w) | rs.out[0];
        q.r = rs.out[1];
        q.cnt = rs.out[2];
        q.shift = sh;
    }
    return q;
}

// CL: a unit may be a cluster of a.cluster CTAs (the few-unit launch); the
// one-CTA-per-unit launch is compiled without the cluster steps.
template <int NT, bool CL>
__global__ void __launch_bounds__(NT, 1024 / NT) select_kernel(SelectArgs a) {
    constexpr int NW = NT / 32;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int nchunk = (a.slots + 31) / 32;
    uint32_t* vals = reinterpret_cast<uint32_t*>(smem_raw);          // [slots] keys
    uint32_t* hist = vals + nchunk * 32;                             // [kCopies][kBuckets]
    uint32_t* comb = hist + kCopies * kBuckets;                      // [kBuckets]
    uint32_t* hmask = comb + kBuckets;                               // [nchunk] hole bits
    uint32_t* mmask = hmask + nchunk;                                // [nchunk] mover bits
    // holes / movers (at most min(B, T) each) reuse the key buffer once the
    // eviction bits are taken
    int32_t* holes = reinterpret_cast<int32_t*>(vals);
    int32_t* movers = holes + min(a.B, a.T);
    __shared__ uint32_t gtot[32], rout[3];
    __shared__ uint32_t s_and[kMaxWarps], s_or[kMaxWarps];
    __shared__ uint32_t c_and[8], c_or[8];          // per CTA of the unit's cluster
    __shared__ uint32_t wtot[2][kMaxWarps];
    __shared__ uint32_t s_pairs;

    // launched while the attention kernel still runs (programmatic dependent
    // launch): its column partials and the pool are read only after it has
    // finished.  Then the next frame's RoPE kernel may start (it rewrites
    // Q', which the attention kernel read, and waits for this grid before
    // it writes the pool rows read here)
    // a cluster's CTAs store keys into each other's shared memory: each
    // first has to know the others have started (arrive here, wait below)
    const bool cl_bar = CL && a.cluster > 1 && a.c + a.T > a.B;
    if (cl_bar) ptx::cluster_arrive_relaxed();
    ptx::dep_wait();
    ptx::dep_trigger();
    const int C = CL ? a.cluster : 1;
    const int rank = CL && C > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int u = (int)blockIdx.x / C;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int c = a.c, T = a.T, B = a.B;
    const int m = c + T;
    // this CTA's candidates [j_lo, j_hi): groups of 4 (16-byte aligned)
    const int g4 = (m + 3) / 4;
    const int j_lo = 4 * (rank * g4 / C), j_hi = min(m, 4 * ((rank + 1) * g4 / C));
    int32_t* pos = a.pos + (int64_t)u * a.slots;
    if (m > B) {                                // the histograms start at zero
        uint4* hv = reinterpret_cast<uint4*>(hist);
        for (int e = tid; e < kCopies * kBuckets / 4; e += NT) hv[e] = make_uint4(0u, 0u, 0u, 0u);
    }

    // ---- 1-2. scores, positions, keys.  A thread issues every load of its
    // KU keys (the partials of up to TU query tiles each, and the positions)
    // before it adds or stores anything: one memory round trip per KU keys
    // instead of one per tile (the position and score buffers may alias as
    // far as the compiler knows, which would otherwise serialise them too)
    const float* cs = a.colsum + (int64_t)u * a.n_row_tiles * a.m_pad;
    float* scores = a.scores + (int64_t)u * a.m_pad;
    int32_t* spos = a.score_pos + (int64_t)u * a.m_pad;
    // each thread takes 4 consecutive candidates (16-byte loads of each
    // tile's partials: the whole unit's partials are in flight at once)
    constexpr int TU = 12;
    const int n_rt = a.n_row_tiles;
    uint32_t k_and = ~0u, k_or = 0u;
    const uint32_t vals_s = ptx::smem_u32(vals);
    if (cl_bar) ptx::cluster_wait();
    for (int j0 = j_lo + 4 * tid; j0 < j_hi; j0 += 4 * NT) {
        float sv[4] = {0.f, 0.f, 0.f, 0.f};
        int32_t pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = j0 + e;
            pv[e] = j < c ? pos[min(j, j_hi - 1)] : a.pos_base + (j - c);
        }
        for (int t0 = 0; t0 < n_rt; t0 += TU) {
            float4 part[TU];
#pragma unroll
            for (int tt = 0; tt < TU; ++tt)
                part[tt] = t0 + tt < n_rt
                               ? __ldcg(reinterpret_cast<const float4*>(cs + (int64_t)(t0 + tt) * a.m_pad + j0))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            // tile order: s_j has the same bits whatever the tiling above
#pragma unroll
            for (int tt = 0; tt < TU; ++tt)
                if (t0 + tt < n_rt) {
                    sv[0] += part[tt].x;
                    sv[1] += part[tt].y;
                    sv[2] += part[tt].z;
                    sv[3] += part[tt].w;
                }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = j0 + e;
            if (j < j_hi) {
                sv[e] *= a.inv_rows;
                scores[j] = sv[e];
                spos[j] = pv[e];
                if (m > B) {
                    const uint32_t k = a.window ? (uint32_t)pv[e] : __float_as_uint(sv[e]);
                    vals[j] = k;
                    k_and &= k;
                    k_or |= k;
                }
            }
        }
    }
    if (m <= B) {                               // state not full: keep all
        for (int j = max(c, j_lo) + tid; j < j_hi; j += NT) pos[j] = a.pos_base + (j - c);
        return;
    }
    // this CTA's keys to the other CTAs of the unit: each thread sends the
    // keys it stored itself above (the same indexing), so no barrier is needed
    if (CL && C > 1)
        for (int j0 = j_lo + 4 * tid; j0 < j_hi; j0 += 4 * NT)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0 + e;
                if (j >= j_hi) break;
                const uint32_t k = vals[j];
                for (int r = 0; r < C; ++r)
                    if (r != rank)
                        ptx::st_cluster_u32(ptx::cluster_map(vals_s + 4u * (uint32_t)j, (uint32_t)r), k);
            }

    // ---- 3. the cut of the E smallest keys
    {
        const uint32_t wa = __reduce_and_sync(0xffffffffu, k_and);
        const uint32_t wo = __reduce_or_sync(0xffffffffu, k_or);
        if (lane == 0) { s_and[warp] = wa; s_or[warp] = wo; }
    }
    __syncthreads();
    uint32_t all_and = __reduce_and_sync(0xffffffffu, lane < NW ? s_and[lane] : ~0u);
    uint32_t all_or = __reduce_or_sync(0xffffffffu, lane < NW ? s_or[lane] : 0u);
    if (CL && C > 1) {
        // every CTA's AND/OR to every CTA; then all keys and scores of the
        // unit are in place (the barrier orders the stores before it,
        // shared and global, for every thread of the cluster)
        if (tid < C) {
            ptx::st_cluster_u32(ptx::cluster_map(ptx::smem_u32(&c_and[rank]), (uint32_t)tid), all_and);
            ptx::st_cluster_u32(ptx::cluster_map(ptx::smem_u32(&c_or[rank]), (uint32_t)tid), all_or);
        }
        ptx::cluster_sync();
        all_and = __reduce_and_sync(0xffffffffu, lane < C ? c_and[lane] : ~0u);
        all_or = __reduce_or_sync(0xffffffffu, lane < C ? c_or[lane] : 0u);
    }
    const RadixScratch rs{hist, comb, gtot, rout};
    const uint32_t E = (uint32_t)(m - B);
    const Cut cut = radix_cut<NT>([&](int j, uint32_t& k) { k = vals[j]; return true; }, m, (uint32_t)m, E,
                                  all_and, all_or, rs);
    // equal scores on both sides of the cut (every bit compared, some of the
    // boundary keys kept): of those, the lower positions are kept
    Cut tie{0u, 0u, 0u, 0u};
    const bool split_tie = cut.r != cut.cnt;
    if (split_tie) {
        auto tie_pos = [&](int j, uint32_t& k) {
            k = (uint32_t)spos[j];
            return vals[j] == cut.pre;
        };
        uint32_t ta = ~0u, to = 0u;
        for (int j = tid; j < m; j += NT) {
            uint32_t k;
            if (tie_pos(j, k)) { ta &= k; to |= k; }
        }
        ta = __reduce_and_sync(0xffffffffu, ta);
        to = __reduce_or_sync(0xffffffffu, to);
        __syncthreads();                        // s_and / s_or reads above are done
        if (lane == 0) { s_and[warp] = ta; s_or[warp] = to; }
        __syncthreads();
        tie = radix_cut<NT>(tie_pos, m, cut.cnt, cut.cnt - cut.r,
                            __reduce_and_sync(0xffffffffu, lane < NW ? s_and[lane] : ~0u),
                            __reduce_or_sync(0xffffffffu, lane < NW ? s_or[lane] : 0u), rs);
    }
    auto evicted = [&](int j) -> bool {
        const uint32_t hv = hi_bits(vals[j], cut.shift);
        if (hv != cut.pre) return hv < cut.pre;
        if (!split_tie) return true;
        const uint32_t p = hi_bits((uint32_t)spos[j], tie.shift);     // kept: the lower positions
        return !(p < tie.pre || (p == tie.pre && tie.r == tie.cnt));
    };

    // ---- 4. holes (slots < B evicted) and movers (slots >= B kept) in slot
    // order: warp w takes the 32-slot chunks [w*cpw, (w+1)*cpw), a ballot per
    // chunk and kind, then a scan over the warps' totals
    const int nch = (m + 31) / 32;
    const int cpw = (nch + NW - 1) / NW;
    uint32_t nh = 0, nm = 0;
    for (int q = warp * cpw; q < min(nch, (warp + 1) * cpw); ++q) {
        const int j = q * 32 + lane;
        const bool ev = j < m && evicted(j);
        const uint32_t hb = __ballot_sync(0xffffffffu, ev && j < B);
        const uint32_t mb = __ballot_sync(0xffffffffu, !ev && j < m && j >= B);
        // surviving frame rows that stay in place get their position
        if (rank == 0 && !ev && j >= c && j < min(B, m)) pos[j] = a.pos_base + (j - c);
        if (lane == 0) { hmask[q] = hb; mmask[q] = mb; }
        nh += __popc(hb);
        nm += __popc(mb);
    }
    if (lane == 0) { wtot[0][warp] = nh; wtot[1][warp] = nm; }
    __syncthreads();                            // keys dead: holes / movers may overwrite them
    if (warp == 0) {
        const uint32_t th = lane < NW ? wtot[0][lane] : 0u, tm = lane < NW ? wtot[1][lane] : 0u;
        uint32_t ph = th, pm = tm;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t yh = __shfl_up_sync(0xffffffffu, ph, off);
            const uint32_t ym = __shfl_up_sync(0xffffffffu, pm, off);
            if (lane >= off) { ph += yh; pm += ym; }
        }
        wtot[0][lane] = ph - th;
        wtot[1][lane] = pm - tm;
        if (lane == 31) {
            // every hole gets a mover
            s_pairs = min(ph, pm);
            if (ph != pm && rank == 0)
                record_error(a.err, (uint32_t)STATEKV_E_DEVICE, kSiteSelect, ph * 65536u + pm);
        }
    }
    __syncthreads();
    {
        uint32_t oh = wtot[0][warp], om = wtot[1][warp];
        const uint32_t lt = (1u << lane) - 1u;
        for (int q = warp * cpw; q < min(nch, (warp + 1) * cpw); ++q) {
            const uint32_t hb = hmask[q], mb = mmask[q];
            const int j = q * 32 + lane;
            if ((hb >> lane) & 1u) holes[oh + __popc(hb & lt)] = j;
            if ((mb >> lane) & 1u) movers[om + __popc(mb & lt)] = j;
            oh += __popc(hb);
            om += __popc(mb);
        }
    }
    __syncthreads();
    const uint32_t np = s_pairs;
    // this CTA's pairs [p_lo, p_hi)
    const uint32_t p_lo = (uint32_t)((uint64_t)np * rank / C);
    const uint32_t p_hi = (uint32_t)((uint64_t)np * (rank + 1) / C);
    for (uint32_t r = p_lo + tid; r < p_hi; r += NT) pos[holes[r]] = a.pos_base + (movers[r] - c);

    // ---- row moves (K and V), 16-byte vectors.  Holes are slots < B and
    // movers slots >= B, so no row is both read and written: each thread
    // issues all its loads (up to 4 vectors of K and of V) before its stores,
    // one memory round trip instead of one per vector
    constexpr int MV = 4;
    const int vpr = a.row_bytes / 16;           // 16-byte vectors per row: a power of two
    const int vpr_shift = 31 - __clz(vpr);
    const int64_t unit_bytes = (int64_t)a.slots * a.row_bytes;
    uint4* pk = reinterpret_cast<uint4*>((char*)a.pool_k + u * unit_bytes);
    uint4* pv = reinterpret_cast<uint4*>((char*)a.pool_v + u * unit_bytes);
    const int64_t total = (int64_t)p_hi * vpr;
    for (int64_t e0 = (int64_t)p_lo * vpr + tid; e0 < total; e0 += MV * NT) {
        uint4 vk[MV], vv[MV];
        int64_t dst[MV];
#pragma unroll
        for (int q = 0; q < MV; ++q) {
            const int64_t e = e0 + (int64_t)q * NT;
            dst[q] = -1;
            if (e < total) {
                const int r = (int)(e >> vpr_shift), w = (int)(e & (vpr - 1));
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
    const size_t nchunk = (size_t)(slots + 31) / 32;
    return nchunk * 32 * sizeof(uint32_t) + (size_t)(kCopies + 1) * kBuckets * sizeof(uint32_t) +
           2 * nchunk * sizeof(uint32_t);
}

template <int NT>
cudaLaunchConfig_t select_config(const SelectArgs& a, cudaStream_t st, size_t smem, int C,
                                 cudaLaunchAttribute (&attr)[2]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.U * C));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

// CTAs per unit: the largest C in {8, 4} for which the device holds all U
// clusters at once (one 1024-thread CTA per SM), else 1.  Pairs (C = 2)
// measured no faster than one CTA per unit on the 56-unit stack, whose
// selection starts while the attention kernel's last wave still runs.
// Cached per (device, shared memory size).
int select_cluster_size(const SelectArgs& a, size_t smem) {
    if (const char* e = std::getenv("STATEKV_SELECT_CLUSTER")) {
        const int v = std::atoi(e);
        if (v == 1 || v == 2 || v == 4 || v == 8) return v;
    }
    if (a.U > a.num_sms / 4) return 1;
    static std::mutex mu;
    struct Entry { int dev; size_t smem; int per_wave[9]; };
    static std::vector<Entry> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    Entry* ent = nullptr;
    for (auto& x : cache)
        if (x.dev == dev && x.smem == smem) ent = &x;
    if (!ent) {
        cache.push_back(Entry{dev, smem, {}});
        ent = &cache.back();
        for (int C = 4; C <= 8; C *= 2) {
            cudaLaunchAttribute attr[2];
            SelectArgs probe = a;
            probe.U = 1;
            const cudaLaunchConfig_t cfg = select_config<1024>(probe, nullptr, smem, C, attr);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, select_kernel<1024, true>, &cfg) != cudaSuccess)
                n = 0;
            ent->per_wave[C] = n;
        }
        cudaGetLastError();
    }
    for (int C = 8; C >= 4; C /= 2)
        if (ent->per_wave[C] >= a.U) return C;
    return 1;
}

template <int NT, bool CL>
cudaError_t launch_select_nt(const SelectArgs& a, size_t smem, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel<NT, CL>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = select_config<NT>(a, st, smem, a.cluster, attr);
    return cudaLaunchKernelEx(&cfg, select_kernel<NT, CL>, a);
}

cudaError_t launch_select(const SelectArgs& a_in, cudaStream_t st) {
    // a handle that never evicts never reaches the key buffer
    const size_t smem = a_in.never_evicts ? 0 : select_smem_bytes(a_in.slots, a_in.T);
    SelectArgs a = a_in;
    a.cluster = 1;
    if (a.U > a.num_sms) return launch_select_nt<512, false>(a, smem, st);
    if (cudaFuncSetAttribute(select_kernel<1024, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return cudaGetLastError();
    a.cluster = select_cluster_size(a, smem);
    return a.cluster > 1 ? launch_select_nt<1024, true>(a, smem, st)
                         : launch_select_nt<1024, false>(a, smem, st);
}

}  // namespace statekv
