// Text-token decode over the detailed state D_N (tcgen05, TMA).
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"),
// 关键设计 1: the detailed state D_n keeps the K/V of every frame for text
// decoding; 关键设计 3: text tokens continue the virtual positions after the
// video (p = offset + N*T + j) with the same static RoPE scale.
//
// Per (stream, layer, KV head) unit the R = G*tok text query rows attend over
// every D row written so far (all visible) and over the tok new rows
// (causal).  D is read once per decode step: the kernel is HBM-bound, R is
// small.  So the products put the keys (and, for PV, the head dimension) on
// the 128 MMA rows and the query rows on the narrow N side ("swap AB"):
//   S^T[128 keys][N]  = K_tile[128][d] . Q^T          (A = K tile, B = Q)
//   O^T[d][N]        += V_tile^T[d][128] . P^T[128][N] (A = V tile MN-major,
//                                                      B = P^T K-major)
// with N = R rounded up to 16/32/64, so no MMA row is padding.
//
// Work items are (unit, chunk of CHUNK_KEYS keys); a persistent grid of one
// CTA per SM walks them, the TMA producer streaming K/V tiles across item
// boundaries.  Each item writes a partial (m, l, O) per query row; a second
// kernel merges the partials of a unit.
//
// Softmax: thread = key (TMEM lane).  Each row keeps one reference value for
// the whole item; p = exp2(s*scale*log2e - ref).  The reference is raised (and
// l and O rescaled) only when a score exceeds it by more than 2^8, which
// keeps exp2 in range without a max reduction per tile.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM allocator and MMA issuer,
// then the softmax / epilogue warps: warp w owns TMEM lane quarter w % 4
// (keys for S^T, head dimensions for O^T).  With 16 query rows there are 8
// of them (320 threads), with 32 or 64 there are 16 (576 threads): two or
// four per lane quarter, each taking an equal share of the rows, so a thread
// exponentiates 8 scores of its key per tile (16 at N = 64).
#include "pipeline.cuh"

namespace statekv {
namespace {

constexpr int kDecD = 128;                 // head dim served by this kernel
constexpr int kKeyTile = 128;              // keys per tile (MMA M of S^T)
constexpr int kChunkTiles = 16;            // tiles per work item
constexpr float kRefSlack = 8.f;           // raise the reference past 2^8

template <int N>
struct DecLayout {
    static constexpr int CHUNK = 128 * 128;          // [128 rows][64 bf16], 128B-swizzled
    static constexpr int KV_TILE = 2 * CHUNK;        // one K or V tile (d = 128)
    static constexpr int NS = N <= 32 ? 3 : 2;       // K/V stages (as many as fit)
    static constexpr int NCHUNK = N * 128;           // [N rows][64 bf16]
    static constexpr int Q_TILE = 2 * NCHUNK;        // Q [N][128]
    static constexpr int P_TILE = 2 * NCHUNK;        // P^T [N][128 keys]
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NS * KV_TILE;
    static constexpr int OFF_Q = OFF_V + NS * KV_TILE;       // [2]
    static constexpr int OFF_P = OFF_Q + 2 * Q_TILE;         // [2]
    // softmax warps per TMEM lane quarter, each taking an equal share of the
    // query rows (each thread exponentiates NH scores of its key per tile)
    static constexpr int WPQ = N >= 32 ? 4 : 2;
    static constexpr int SWARPS = 4 * WPQ;
    static constexpr int NH = N / WPQ;                       // query rows per softmax warp
    static constexpr int OFF_RED = OFF_P + 2 * P_TILE;       // float [4 lane quarters][N]
    static constexpr int OFF_REF = OFF_RED + 4 * N * 4;      // float [N] reference (log2 units)
    static constexpr int OFF_FAC = OFF_REF + N * 4;          // float [N] rescale factors
    static constexpr int OFF_FLAG = OFF_FAC + N * 4;         // uint32 [2 tile parities][SWARPS]
    static constexpr int OFF_BAR = OFF_FLAG + 8 * SWARPS;
    static constexpr int B_KV_FULL = 0;                      // [NS]
    static constexpr int B_KV_EMPTY = B_KV_FULL + NS;        // [NS]
    static constexpr int B_Q_FULL = B_KV_EMPTY + NS;         // [2]
    static constexpr int B_Q_EMPTY = B_Q_FULL + 2;           // [2]
    static constexpr int B_S_FULL = B_Q_EMPTY + 2;           // [2]
    static constexpr int B_S_READ = B_S_FULL + 2;            // [2]
    static constexpr int B_P_FULL = B_S_READ + 2;            // [2]
    static constexpr int B_P_FREE = B_P_FULL + 2;            // [2]
    static constexpr int B_O_FULL = B_P_FREE + 2;            // [2]
    static constexpr int B_O_FREE = B_O_FULL + 2;            // [2]
    static constexpr int B_DRAIN = B_O_FREE + 2;
    static constexpr int B_SYNC = B_DRAIN + 1;               // the softmax warps
    static constexpr int NBAR = B_SYNC + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static constexpr uint32_t TM_S = 0, TM_O = 2 * N;        // two S^T, two O^T buffers
    static constexpr uint32_t TMEM_COLS = 4 * N < 32 ? 32 : 4 * N;
    static constexpr int THREADS = 64 + 32 * SWARPS;
};

struct Item {
    int u, tile0, tiles;                       // unit, first key tile, tile count
};
__device__ __forceinline__ Item item_of(const DecodeArgs& a, int w) {
    Item it;
    it.u = w / a.chunks;
    const int c = w - it.u * a.chunks;
    it.tile0 = c * kChunkTiles;
    const int ntiles = (int)((a.keys + kKeyTile - 1) / kKeyTile);
    it.tiles = min(kChunkTiles, ntiles - it.tile0);
    return it;
}

// Byte offset of element (row, col) in a K-major, 128B-swizzled bf16 tile of
// `rows` rows: 64-column chunks of rows*128 bytes, 16-byte units XOR-ed with
// row % 8 inside each 128-byte row.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int rows) {
    const int chunk = col >> 6, c = col & 63;
    return (uint32_t)(chunk * rows * 128 + row * 128 + ((((c >> 3) ^ (row & 7)) << 4) | ((c & 7) << 1)));
}

template <int N>
__global__ void __launch_bounds__(DecLayout<N>::THREADS, 1)
decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, DecodeArgs a) {
    using L = DecLayout<N>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw_u32);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = a.U * a.chunks;

    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + L::OFF_MISC + 4);
    Sync sy{sbase + (uint32_t)L::OFF_BAR, abort_flag, a.err};
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::NS; ++s) {
            ptx::mbar_init(sy.bar(L::B_KV_FULL + s), 1);
            ptx::mbar_init(sy.bar(L::B_KV_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(sy.bar(L::B_Q_FULL + b), 1);
            ptx::mbar_init(sy.bar(L::B_Q_EMPTY + b), 1);
            ptx::mbar_init(sy.bar(L::B_S_FULL + b), 1);
            ptx::mbar_init(sy.bar(L::B_S_READ + b), L::SWARPS);
            ptx::mbar_init(sy.bar(L::B_P_FULL + b), L::SWARPS);
            ptx::mbar_init(sy.bar(L::B_P_FREE + b), 1);
            ptx::mbar_init(sy.bar(L::B_O_FULL + b), 1);
            ptx::mbar_init(sy.bar(L::B_O_FREE + b), L::SWARPS);
        }
        ptx::mbar_init(sy.bar(L::B_DRAIN), 1);
        ptx::mbar_init(sy.bar(L::B_SYNC), L::SWARPS);
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
    const uint32_t sK = sbase + L::OFF_K, sV = sbase + L::OFF_V;
    const uint32_t sQ = sbase + L::OFF_Q, sP = sbase + L::OFF_P;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            int g = 0, li = 0;                     // tiles and items loaded
            bool ok = true;
            for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x, ++li) {
                const Item it = item_of(a, w);
                const int qb = li & 1;
                if (!(ok = sy.wait(L::B_Q_EMPTY + qb, (uint32_t)(((li >> 1) & 1) ^ 1), kSiteKvEmpty)))
                    break;
                ptx::mbar_arrive_expect_tx(sy.bar(L::B_Q_FULL + qb), L::Q_TILE);
                for (int kc = 0; kc < 2; ++kc)
                    ptx::tma_load_3d(sQ + qb * L::Q_TILE + kc * L::NCHUNK, &tm_q,
                                     sy.bar(L::B_Q_FULL + qb), kc * 64, 0, it.u);
                for (int t = 0; t < it.tiles; ++t, ++g) {
                    const int s = g % L::NS, j = g / L::NS;
                    if (!(ok = sy.wait(L::B_KV_EMPTY + s, (uint32_t)(j & 1) ^ 1u, kSiteKvEmpty)))
                        break;
                    const uint32_t fb = sy.bar(L::B_KV_FULL + s);
                    ptx::mbar_arrive_expect_tx(fb, 2 * L::KV_TILE);
                    const int row = (it.tile0 + t) * kKeyTile;
                    for (int kc = 0; kc < 2; ++kc) {
                        ptx::tma_load_3d(sK + s * L::KV_TILE + kc * L::CHUNK, &tm_k, fb, kc * 64,
                                         row, it.u);
                        ptx::tma_load_3d(sV + s * L::KV_TILE + kc * L::CHUNK, &tm_v, fb, kc * 64,
                                         row, it.u);
                    }
                }
            }
            // never leave a copy in flight into this CTA's shared memory
            for (int s = 0; s < L::NS && s < g; ++s)
                sy.drain(L::B_KV_FULL + s, (uint32_t)(((g - 1 - s) / L::NS) & 1));
            for (int b = 0; b < 2 && b < li; ++b)
                sy.drain(L::B_Q_FULL + b, (uint32_t)(((li - 1 - b) / 2) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // per item: S^T(t) for every tile, each followed by PV(t-1); PV(last)
        // closes the item.  S^T runs one tile ahead of PV.
        constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, N, false, false);
        constexpr uint32_t idesc_o = ptx::idesc_bf16_f32(128, N, true, false);
        const uint32_t kmaj_hi = (uint32_t)(ptx::sdesc_sw128(0, 16, 1024) >> 32);
        const uint32_t mn_hi = (uint32_t)(ptx::sdesc_sw128(0, L::CHUNK, 1024) >> 32);
        const uint32_t kb0 = (uint32_t)ptx::sdesc_sw128(sK, 16, 1024);
        const uint32_t vb0 = (uint32_t)ptx::sdesc_sw128(sV, L::CHUNK, 1024);
        const uint32_t qb0 = (uint32_t)ptx::sdesc_sw128(sQ, 16, 1024);
        const uint32_t pb0 = (uint32_t)ptx::sdesc_sw128(sP, 16, 1024);
        int g = 0, li = 0;
        bool ok = true;
        // O^T(item buffer ob) += V(stage)^T P^T(buffer pb)
        auto issue_pv = [&](int gt, bool first, int ob) -> bool {
            const int s = gt % L::NS, pb = gt & 1;
            if (!sy.wait(L::B_P_FULL + pb, (uint32_t)((gt >> 1) & 1), kSitePFull)) return false;
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
                const uint32_t vb = vb0 + (uint32_t)s * (L::KV_TILE >> 4);
                const uint32_t pbd = pb0 + (uint32_t)pb * (L::P_TILE >> 4);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)            // 16 keys per step
                    ptx::umma_ss_lh(tmem + L::TM_O + (uint32_t)(ob * N), vb + 128u * ks, mn_hi,
                                    pbd + (uint32_t)((ks >> 2) * (L::NCHUNK >> 4) + 2 * (ks & 3)),
                                    kmaj_hi, idesc_o, (first && ks == 0) ? 0u : 1u);
                ptx::umma_commit(sy.bar(L::B_P_FREE + pb));
                ptx::umma_commit(sy.bar(L::B_KV_EMPTY + s));
            }
            __syncwarp();
            return true;
        };
        for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x, ++li) {
            const Item it = item_of(a, w);
            const int qb = li & 1, ob = li & 1;
            if (!(ok = sy.wait(L::B_Q_FULL + qb, (uint32_t)((li >> 1) & 1), kSiteQFull))) break;
            // O^T buffer ob free once the epilogue of item li-2 read it
            if (li >= 2 && !(ok = sy.wait(L::B_O_FREE + ob, (uint32_t)(((li - 2) >> 1) & 1), kSiteOFull)))
                break;
            ptx::tc_fence_after();
            const int g0 = g;
            for (int t = 0; t < it.tiles; ++t, ++g) {
                const int s = g % L::NS, sb = g & 1;
                if (!(ok = sy.wait(L::B_KV_FULL + s, (uint32_t)((g / L::NS) & 1), kSiteKvFull))) break;
                if (g >= 2 && !(ok = sy.wait(L::B_S_READ + sb, (uint32_t)(((g - 2) >> 1) & 1), kSiteSEmpty)))
                    break;
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                    const uint32_t kb = kb0 + (uint32_t)s * (L::KV_TILE >> 4);
                    const uint32_t qd = qb0 + (uint32_t)qb * (L::Q_TILE >> 4);
#pragma unroll
                    for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            ptx::umma_ss_lh(tmem + L::TM_S + (uint32_t)(sb * N),
                                            kb + kc * (L::CHUNK >> 4) + 2 * ks, kmaj_hi,
                                            qd + kc * (L::NCHUNK >> 4) + 2 * ks, kmaj_hi, idesc_s,
                                            (kc | ks) ? 1u : 0u);
                    ptx::umma_commit(sy.bar(L::B_S_FULL + sb));
                    if (t == it.tiles - 1) ptx::umma_commit(sy.bar(L::B_Q_EMPTY + qb));
                }
                __syncwarp();
                if (t > 0 && !(ok = issue_pv(g - 1, g - 1 == g0, ob))) break;
            }
            if (!ok) break;
            if (!(ok = issue_pv(g - 1, g - 1 == g0, ob))) break;
            if (ptx::elect_one()) ptx::umma_commit(sy.bar(L::B_O_FULL + ob));
            __syncwarp();
        }
        if (ptx::elect_one()) ptx::umma_commit(sy.bar(L::B_DRAIN));
        __syncwarp();
        sy.drain(L::B_DRAIN, 0);
    } else {
        // ------------------------------------------------ softmax / epilogue
        // warp w: TMEM lane quarter w % 4 (keys of S^T, head dimensions of
        // O^T) and query rows [r0, r0 + NH)
        constexpr int NH = L::NH;
        const int q4 = warp & 3;
        const int r0 = ((warp - 2) >> 2) * NH;
        const int kk = q4 * 32 + lane;                 // key of the tile / head dimension
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        float* red = reinterpret_cast<float*>(base + L::OFF_RED);
        float* ref = reinterpret_cast<float*>(base + L::OFF_REF);
        float* fac = reinterpret_cast<float*>(base + L::OFF_FAC);
        volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(base + L::OFF_FLAG);
        const float sc = a.scale_log2;
        const int visible = (int)a.visible, keys = (int)a.keys;
        int g = 0, li = 0;
        bool ok = true;
        // NH consecutive TMEM columns of this warp's lane quarter
        auto ld_cols = [&](uint32_t taddr, uint32_t (&v)[NH]) {
            if constexpr (NH == 8) ptx::tmem_ld_32x32b_x8(taddr, v);
            else if constexpr (NH == 16) ptx::tmem_ld_32x32b_x16(taddr, v);
            else ptx::tmem_ld_32x32b_x32(taddr, v);
        };
        auto st_cols = [&](uint32_t taddr, const uint32_t (&v)[NH]) {
            if constexpr (NH == 8) ptx::tmem_st_32x32b_x8(taddr, v);
            else if constexpr (NH == 16) ptx::tmem_st_32x32b_x16(taddr, v);
            else ptx::tmem_st_32x32b_x32(taddr, v);
        };
        // barrier of the softmax warps (a bounded mbarrier wait: a warp that
        // gave up cannot leave the others blocked)
        uint32_t sync_par = 0;
        auto sync_sm = [&]() -> bool {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_SYNC));
            const bool r = sy.wait(L::B_SYNC, sync_par, kSiteCol);
            sync_par ^= 1u;
            return r;
        };
        for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x, ++li) {
            const Item it = item_of(a, w);
            const int ob = li & 1;
            float l[NH];
#pragma unroll
            for (int j = 0; j < NH; ++j) l[j] = 0.f;
            if (threadIdx.x - 64 < N) ref[threadIdx.x - 64] = -INFINITY;
            if (!(ok = sync_sm())) break;
            for (int t = 0; t < it.tiles; ++t, ++g) {
                const int sb = g & 1, pb = g & 1;
                if (!(ok = sy.wait(L::B_S_FULL + sb, (uint32_t)((g >> 1) & 1), kSiteSFull))) break;
                ptx::tc_fence_after();
                uint32_t sr[NH];
                ld_cols(tmem + L::TM_S + sb * N + r0 + lane_base, sr);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_relaxed(sy.bar(L::B_S_READ + sb));
                // query row r is token r % tok of its head: key j is visible
                // to it iff j < keys and j <= visible + r % tok
                const int key = (it.tile0 + t) * kKeyTile + kk;
                const int kv = key - visible;          // >= 0 only among the new keys
                float x[NH];
                bool exceed = false;
                if ((it.tile0 + t + 1) * kKeyTile <= visible) {
                    // a tile of earlier keys only (every tile but the last one
                    // or two): each is visible to every row
#pragma unroll
                    for (int j = 0; j < NH; ++j) {
                        x[j] = __uint_as_float(sr[j]) * sc;
                        exceed |= x[j] > ref[r0 + j] + kRefSlack;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < NH; ++j) {
                        const int r = r0 + j;
                        const bool vis = key < keys && (kv < 0 || r % a.tok >= kv);
                        x[j] = vis ? __uint_as_float(sr[j]) * sc : -INFINITY;
                        exceed |= x[j] > ref[r] + kRefSlack;
                    }
                }
                // raise the reference of every row when any score got past it
                // (flags alternate between two sets by tile: a warp that runs
                // ahead writes the next tile's set while the others still
                // read this one; it cannot get two tiles ahead, as this
                // barrier waits for every warp)
                exceed = __any_sync(0xffffffffu, exceed);
                volatile uint32_t* fl = flag + L::SWARPS * (g & 1);
                if (lane == 0) fl[warp - 2] = exceed ? 1u : 0u;
                if (!(ok = sync_sm())) break;
                uint32_t any = 0u;
#pragma unroll
                for (int i = 0; i < L::SWARPS; ++i) any |= fl[i];
                if (any != 0u) {
#pragma unroll
                    for (int j = 0; j < NH; ++j) {
                        float m = x[j];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                        if (lane == 0) red[q4 * N + r0 + j] = m;
                    }
                    if (!(ok = sync_sm())) break;
                    if (threadIdx.x - 64 < N) {
                        const int r = threadIdx.x - 64;
                        const float m = fmaxf(fmaxf(red[r], red[N + r]), fmaxf(red[2 * N + r], red[3 * N + r]));
                        const float old = ref[r];
                        const float nw = fmaxf(old, m);
                        fac[r] = (old == -INFINITY) ? 0.f : ptx::ex2_approx(old - nw);
                        ref[r] = nw;
                    }
                    if (!(ok = sync_sm())) break;
                    // rescale l and the O^T accumulated so far in this item
#pragma unroll
                    for (int j = 0; j < NH; ++j) l[j] *= fac[r0 + j];
                    if (t > 0) {
                        // every PV of this item issued so far has completed
                        if (!(ok = sy.wait(L::B_P_FREE + ((g - 1) & 1), (uint32_t)(((g - 1) >> 1) & 1),
                                           kSitePEmpty))) break;
                        ptx::tc_fence_after();
                        uint32_t orr[NH];
                        const uint32_t ta = tmem + L::TM_O + ob * N + r0 + lane_base;
                        ld_cols(ta, orr);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < NH; ++j)
                            orr[j] = __float_as_uint(__uint_as_float(orr[j]) * fac[r0 + j]);
                        st_cols(ta, orr);
                        ptx::tmem_st_wait();
                    }
                }
                // P^T(t): row r, key kk (bf16) -- after PV(t-2) freed buffer pb
                if (g >= 2 && !(ok = sy.wait(L::B_P_FREE + pb, (uint32_t)(((g - 2) >> 1) & 1), kSitePEmpty)))
                    break;
                uint8_t* pt = base + L::OFF_P + pb * L::P_TILE;
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    // masked keys give 0 (a row's reference is finite once any
                    // key was visible to it)
                    const float p = x[j] == -INFINITY ? 0.f : ptx::ex2_approx(x[j] - ref[r0 + j]);
                    l[j] += p;
                    *reinterpret_cast<__nv_bfloat16*>(pt + sw128_offset(r0 + j, kk, N)) = __float2bfloat16_rn(p);
                }
                // generic-proxy stores -> visible to the tensor core
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_P_FULL + pb));
                // no barrier here: ref[] and fac[] are rewritten only in the
                // next tile's raise, after a barrier that every warp reaches
                // only once it has finished this tile
            }
            if (!ok) break;
            // ---- item epilogue: row sums, then O^T (thread = head dimension)
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                float sm = l[j];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
                if (lane == 0) red[q4 * N + r0 + j] = sm;
            }
            if (!(ok = sync_sm())) break;
            const int64_t pidx = (int64_t)w * N;      // partial rows of this item
            if (threadIdx.x - 64 < N) {
                const int r = threadIdx.x - 64;
                a.part_m[pidx + r] = ref[r];
                a.part_l[pidx + r] = red[r] + red[N + r] + red[2 * N + r] + red[3 * N + r];
            }
            if (!(ok = sy.wait(L::B_O_FULL + ob, (uint32_t)((li >> 1) & 1), kSiteOFull))) break;
            ptx::tc_fence_after();
            uint32_t orr[NH];
            ld_cols(tmem + L::TM_O + ob * N + r0 + lane_base, orr);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_O_FREE + ob));
            float* po = a.part_o + pidx * kDecD;
#pragma unroll
            for (int j = 0; j < NH; ++j) po[(int64_t)(r0 + j) * kDecD + kk] = __uint_as_float(orr[j]);
            if (!(ok = sync_sm())) break;              // ref[] / red[] reused by the next item
        }
    }
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// out[u][r][:] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the
// unit's chunks c (M = max m_c); rows r < R only.
// Merge a row's per-chunk partials (m, l, O) in chunk order.  Thread d owns
// output column d; the chunk weights exp2(m_c - max) and sums l_c are staged
// in shared memory per block of 128 chunks, and the partial-O loads of
// several chunks are in flight at once (the chunks' loads are independent).
__global__ void __launch_bounds__(kDecD) decode_combine_kernel(DecodeArgs a, int npad) {
    const int u = blockIdx.x, r = blockIdx.y, d = threadIdx.x;
    const int64_t i0 = (int64_t)u * a.chunks;
    __shared__ float s_w[kDecD], s_l[kDecD], s_red[kDecD / 32];
    float mx = -INFINITY;
    for (int c = d; c < a.chunks; c += kDecD) mx = fmaxf(mx, a.part_m[(i0 + c) * npad + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((d & 31) == 0) s_red[d >> 5] = mx;
    __syncthreads();
    mx = s_red[0];
#pragma unroll
    for (int w = 1; w < kDecD / 32; ++w) mx = fmaxf(mx, s_red[w]);
    float acc = 0.f, lsum = 0.f;
    for (int c0 = 0; c0 < a.chunks; c0 += kDecD) {
        const int n = min(kDecD, a.chunks - c0);
        __syncthreads();                            // the previous block's weights are used
        if (d < n) {
            const int64_t pr = (i0 + c0 + d) * npad + r;
            const float m = a.part_m[pr];
            // a chunk with no visible key contributes nothing
            s_w[d] = m == -INFINITY ? -1.f : ptx::ex2_approx(m - mx);
            s_l[d] = m == -INFINITY ? 0.f : a.part_l[pr];
        }
        __syncthreads();
        const float* po = a.part_o + ((i0 + c0) * npad + r) * kDecD + d;
#pragma unroll 8
        for (int c = 0; c < n; ++c) {
            const float o = po[(int64_t)c * npad * kDecD];
            const float w = s_w[c];
            if (w >= 0.f) {
                lsum = fmaf(w, s_l[c], lsum);
                acc = fmaf(w, o, acc);
            }
        }
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.o) + ((int64_t)u * a.R + r) * kDecD + d;
    *out = __float2bfloat16_rn(acc / lsum);
}

template <int N>
cudaError_t launch_n(const DecodeArgs& a, const DecodeMaps& m, cudaStream_t st) {
    using L = DecLayout<N>;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::SMEM);
    if (e != cudaSuccess) return e;
    const int items = a.U * a.chunks;
    const int grid = items < a.num_sms ? items : a.num_sms;
    decode_kernel<N><<<grid, L::THREADS, L::SMEM, st>>>(m.q, m.k, m.v, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    decode_combine_kernel<<<dim3((unsigned)a.U, (unsigned)a.R), kDecD, 0, st>>>(a, N);
    return cudaGetLastError();
}

}  // namespace

int decode_rows_pad(int R) { return R <= 16 ? 16 : R <= 32 ? 32 : R <= 64 ? 64 : -1; }
int decode_chunks(int64_t keys) {
    const int64_t tiles = (keys + kKeyTile - 1) / kKeyTile;
    return (int)((tiles + kChunkTiles - 1) / kChunkTiles);
}

bool make_decode_maps(DecodeMaps* m, const void* q_rot, int R, int npad, const void* det_k,
                      const void* det_v, int64_t det_pitch, int64_t units) {
    return encode_view(&m->q, q_rot, kDecD, R, units, npad) &&
           encode_view(&m->k, det_k, kDecD, det_pitch, units, kKeyTile) &&
           encode_view(&m->v, det_v, kDecD, det_pitch, units, kKeyTile);
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps& m, cudaStream_t st) {
    switch (decode_rows_pad(a.R)) {
        case 16: return launch_n<16>(a, m, st);
        case 32: return launch_n<32>(a, m, st);
        case 64: return launch_n<64>(a, m, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace statekv
