// bf16 frame attention on the 5th-generation tensor cores (tcgen05 + TMEM,
// operands staged by TMA), with the key column sums of P fused in.
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"):
//   关键设计 1 -- the frame's queries attend over [K̄_{n-1}; K_n]: every
//     compressed key is visible, frame keys are causal;
//   关键设计 2 -- key j's importance is the attention the frame's queries pay
//     to it, averaged over queries; this kernel emits, per 128-row query
//     tile, the column sums of the final normalised P (the select kernel
//     adds the tiles' partials in tile order);
//   整体框架 -- the per-frame cost O(T^2 + BT): the key loop covers only the
//     B compressed keys and the causally visible part of the frame.
//
// One CTA = one 128-row query tile of one (stream, layer, KV head); rows are
// (g, i) pairs of the G query heads that share the KV head, g-major.  Two
// sweeps over the 128-key tiles of the pool:
//   sweep 1: S = Q K^T (tcgen05, fp32 in TMEM) -> per thread and row, a sum
//            of exp2 against a reference (the row's max when last raised:
//            set by the first tile, raised only when a tile's sum passes
//            2^32, so no max per tile), combined across the row's threads at
//            the end -> log-sum-exp per row;
//   sweep 2: S again, P = exp2(S*scale - lse) (final, normalised): column
//            sums of fp32 P, and P -> bf16 into TMEM as the A operand of
//            O += P V (tcgen05 with A in TMEM, V read MN-major from shared
//            memory).  P is normalised before PV, so O needs no rescaling.
//
// Warp roles (608 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// issuer of the S = Q K^T MMAs, warp 2 issuer of the O += P V MMAs, warps
// 3..18 softmax.  Softmax warp w covers TMEM lane quarter w % 4 (the only
// lanes it may access) and 32-column chunk (w - 3) / 4 of every S tile;
// with the 16x256b load shape a thread holds 4 rows x 8 columns, so row
// statistics combine across 4 lanes (then across the 4 chunk warps once per
// sweep) and column sums need a 3-level shuffle reduction, then a sum over
// the 4 lane quarters in shared memory, which the PV-issuer warp does while
// the softmax warps move on (it waits for every warp's P anyway).
// Shared-memory bandwidth (128 B/clk/SM) is the scarce resource: an MMA with
// both operands in shared memory at M = N = 128 consumes all of it, leaving
// nothing for the TMA writes of the next K/V tiles.  So Q lives in TMEM: the
// softmax warps copy it there once, and both products read one operand from
// TMEM (S = Q K^T: Q; O += P V: P) and only K or V from shared memory, which
// halves the MMA's share of the bandwidth.
// TMEM (512 columns): Q (bf16 pairs) at 448..; sweep 1 -- three S buffers
// (0, 128, 256); sweep 2 -- two S buffers (0, 128), O (256..), P (384..447,
// bf16 pairs) in two 64-key halves, each with its own full/free barriers:
// the 8 warps of one half refill it as soon as that half's PV products are
// done, while the other half's still run.  An S buffer is handed back to the MMA issuer as soon as its
// tile has been loaded into registers, so S(t+1) is computed while the
// softmax works on S(t) and never waits for the signal that S(t) was read
// (that arrive sits in the same per-SMSP queue as the softmax's ex2 burst
// and completes late); P never aliases S.
// Every mbarrier wait is bounded; on timeout the CTA records
// STATEKV_E_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM, exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <type_traits>

#include "pipeline.cuh"

namespace statekv {
namespace {

constexpr int L_KSMAX = 8;                              // largest key split (cluster size)

template <int D>
struct TcLayout {
    static constexpr int BN = 128;
    static constexpr int KCH = D / 64;                  // 128-byte chunks along d
    static constexpr int CHUNK = 128 * 128;             // [128 rows][64 bf16], 128B-swizzled
    static constexpr int TILE = KCH * CHUNK;            // one K or V tile
    static constexpr int KS = 4, VS = 2;                // K and V pipeline stages
    static constexpr int SB1 = 3;                       // sweep-1 S buffers
    static constexpr int NCOL = 2;                      // column-sum exchange slots
    static constexpr int SW = 16;                       // softmax warps
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KS * TILE;
    static constexpr int OFF_COL = OFF_V + VS * TILE;   // float [NCOL][4 quarters][128]
    static constexpr int OFF_STAT = OFF_COL + NCOL * 4 * 128 * 4;   // float2 [16 threads][128 rows]
    static constexpr int OFF_LSE = OFF_STAT + 16 * 128 * 8;         // float [128 rows]
    static constexpr int KSMAX = L_KSMAX;
    static constexpr int OFF_XLSE = OFF_LSE + 128 * 4;  // float [KSMAX][128 rows]: the split's lse partials
    static constexpr int OFF_BAR = OFF_XLSE + KSMAX * 128 * 4;
    static constexpr int B_Q = 0;                       // Q in TMEM (all softmax warps)
    static constexpr int B_K_FULL = 1;
    static constexpr int B_K_EMPTY = B_K_FULL + KS;
    static constexpr int B_V_FULL = B_K_EMPTY + KS;
    static constexpr int B_V_EMPTY = B_V_FULL + VS;
    static constexpr int B_S_FULL = B_V_EMPTY + VS;     // [SB1] S buffer computed
    static constexpr int B_S_READ = B_S_FULL + SB1;     // [SB1] S buffer loaded by all softmax warps
    static constexpr int B_P_FULL = B_S_READ + SB1;     // [2] key half of P written by its 8 warps
    static constexpr int B_P_FREE = B_P_FULL + 2;       // [2] key half of P consumed by PV
    static constexpr int B_O_FULL = B_P_FREE + 2;
    static constexpr int B_DRAIN = B_O_FULL + 1;        // [2] each MMA issuer's teardown
    static constexpr int B_STAT = B_DRAIN + 2;          // row statistics of every softmax thread stored
    static constexpr int B_LSE = B_STAT + 1;            // lse of every row stored
    static constexpr int B_S1_DONE = B_LSE + 1;         // the PV warp issued its sweep-1 S tiles
    // split query tiles (the ks CTAs of a cluster, one key range each):
    static constexpr int B_XLSE = B_S1_DONE + 1;        // every other CTA's lse partials arrived
    static constexpr int B_XREADY = B_XLSE + 1;         // every other CTA's K stages may take our O
    static constexpr int B_XO = B_XREADY + 1;           // the O columns this CTA owns arrived
    static constexpr int NBAR = B_XO + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TM_O = 256, TM_P = 384, TM_Q = 448;
    static constexpr int THREADS = 96 + 32 * SW;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
    // a split tile's owner receives ks partial O blocks of bw columns x 128
    // rows (fp32) in its K stages
    static constexpr bool split_fits() {
        for (int ks = 2; ks <= KSMAX; ++ks) {
            const int bw = 8 * ((D + 8 * ks - 1) / (8 * ks));
            if (ks * bw * 128 * 4 > KS * TILE) return false;
        }
        return true;
    }
    static_assert(split_fits(), "split O exchange fits in the K stages");
};

// Key range of one 128-row query tile: tiles [0, nt) hold a key visible to
// some row; tiles [0, nfull) are visible to every row.
struct TileRange {
    int row0, nt, nfull;
};
__device__ __forceinline__ TileRange tile_range(int row0, int GT, int T, int c) {
    TileRange r{row0, 0, 0};
    if (row0 >= GT) return r;
    const int r1 = min(row0 + 128, GT) - 1;
    const bool one_head = (row0 / T) == (r1 / T);
    const int imax = one_head ? r1 % T : T - 1;
    const int imin = one_head ? row0 % T : 0;
    r.nt = (c + imax + 1 + 127) / 128;
    r.nfull = (c + imin + 1) / 128;
    return r;
}

// SPLIT: the grid is clusters of ks = a.split_ks CTAs.  The first
// split_item0 query tiles run whole, ks per cluster (the CTAs do not
// interact); each later tile is shared by the ks CTAs of a cluster ("coop"),
// CTA r taking key tiles [r*nt/ks, (r+1)*nt/ks): after sweep 1 every CTA
// sends its per-row lse partials to the others and all combine them in rank
// order (the same bits everywhere); at the end CTA r owns O columns
// [r*bw, (r+1)*bw) (bw a multiple of 8), receives the other CTAs' partial O
// of them through distributed shared memory and adds the ks partials in
// rank order.  Two uses: the last, partial wave of a launch of several
// waves runs as pairs (its tiles take about 60 % as long on twice as many
// SMs, and start as soon as SMs free up in the wave before), and a launch
// with fewer tiles than SMs (one layer at a time) spreads every tile's keys
// over ks CTAs.
// KSC: the split width, 1 = no split tiles, 2 = pairs (the tail of a launch
// of several waves), 0 = a.split_ks CTAs (a launch of fewer tiles than SMs).
template <int D, int KSC>
__global__ void __launch_bounds__(TcLayout<D>::THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, AttnArgs a) {
    using L = TcLayout<D>;
    constexpr bool SPLIT = KSC != 1;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rt = a.n_row_tiles;
    const int ks = KSC > 0 ? KSC : a.split_ks;
    const int cl = (int)blockIdx.x / ks;                 // cluster
    const bool coop = SPLIT && cl * ks >= a.split_item0;
    const int rank = coop ? (int)ptx::cluster_ctarank() : 0;
    const int item = coop ? a.split_item0 + (cl - a.split_item0 / ks) : (int)blockIdx.x;
    // O columns [rank*bw, (rank+1)*bw) are this CTA's to output in a split tile
    const int bw = 8 * ((D + 8 * ks - 1) / (8 * ks));
    const int u = item / n_rt;
    const int mt = item - u * n_rt;
    const TileRange me = tile_range(mt * 128, a.GT, a.T, a.c);
    // this CTA's key tiles: [t0, t0 + nt_mine) of the tile's [0, me.nt)
    const int t0 = coop ? rank * me.nt / ks : 0;
    const int nt_mine = coop ? (rank + 1) * me.nt / ks - t0 : me.nt;

    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::OFF_MISC);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(base + L::OFF_MISC + 4);
    Sync sy{sbase + (uint32_t)L::OFF_BAR, abort_flag, a.err};

    if (threadIdx.x == 0) {
        ptx::mbar_init(sy.bar(L::B_Q), L::SW);
        for (int s = 0; s < L::KS; ++s) {
            ptx::mbar_init(sy.bar(L::B_K_FULL + s), 1);
            ptx::mbar_init(sy.bar(L::B_K_EMPTY + s), 1);
        }
        for (int s = 0; s < L::VS; ++s) {
            ptx::mbar_init(sy.bar(L::B_V_FULL + s), 1);
            ptx::mbar_init(sy.bar(L::B_V_EMPTY + s), 1);
        }
        for (int b = 0; b < L::SB1; ++b) {
            ptx::mbar_init(sy.bar(L::B_S_FULL + b), 1);
            ptx::mbar_init(sy.bar(L::B_S_READ + b), L::SW);
        }
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(sy.bar(L::B_P_FULL + h), L::SW / 2);
            ptx::mbar_init(sy.bar(L::B_P_FREE + h), 1);
        }
        ptx::mbar_init(sy.bar(L::B_O_FULL), 1);
        ptx::mbar_init(sy.bar(L::B_DRAIN), 1);
        ptx::mbar_init(sy.bar(L::B_DRAIN + 1), 1);
        ptx::mbar_init(sy.bar(L::B_STAT), L::SW);
        ptx::mbar_init(sy.bar(L::B_LSE), 4);
        ptx::mbar_init(sy.bar(L::B_S1_DONE), 1);
        // split tiles: 128 rows of lse partials from each other CTA; its 16
        // softmax warps' "K stages consumed"; and one arrive per sending
        // lane (4 quarters x 32 lanes of every 32-column chunk that overlaps
        // this CTA's columns) from each other CTA
        const int lo = rank * bw, hi = min(D, lo + bw);
        const int nwin = lo < hi ? (hi - 1) / 32 - lo / 32 + 1 : 0;
        ptx::mbar_init(sy.bar(L::B_XLSE), (uint32_t)max(1, 128 * (ks - 1)));
        ptx::mbar_init(sy.bar(L::B_XREADY), (uint32_t)max(1, L::SW * (ks - 1)));
        ptx::mbar_init(sy.bar(L::B_XO), (uint32_t)max(1, 128 * nwin * (ks - 1)));
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), L::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // a split tile's other CTAs write into this CTA's shared memory and
    // arrive on its barriers: all of them must be initialised first
    if (coop) ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // set-up above may overlap the end of the RoPE kernel (programmatic
    // dependent launch); every read and write of global memory comes after
    ptx::dep_wait();
    // the split tail launch that may follow waits for this grid anyway
    ptx::dep_trigger();

    const uint32_t sK = sbase + L::OFF_K;
    const uint32_t sV = sbase + L::OFF_V;

    // S = Q K^T of K load kt into S buffer b, shared by the two issuer warps
    // (warp 1; warp 2 in sweep 1, where it has no PV products to issue).
    // Each issuer warp walks its schedule together and one elected lane
    // issues each batch of MMAs and their commits; an issuing thread stalls
    // while the tensor pipe's queue is full, and between batches its warp
    // waits for issue slots on a sub-partition with four softmax warps, so
    // two issuers halve that bookkeeping per tile in sweep 1.  prev_uses =
    // earlier S products into buffer b: the buffer may be overwritten once
    // every softmax warp loaded the last of them.  Phases follow from the
    // tile indices, so the two warps need no shared state.
    auto issue_s = [&](int kt, int b, int prev_uses) -> bool {
        constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 128, false, false);
        // a K step of 16 bf16 (32 bytes) adds 2 to the start-address field,
        // a stage (TILE bytes) adds TILE >> 4; in TMEM a K step of Q is 8 columns
        const uint32_t desc_hi = (uint32_t)(ptx::sdesc_sw128(0, 16, 1024) >> 32);
        const uint32_t kb0 = (uint32_t)ptx::sdesc_sw128(sK, 16, 1024);
        const int s = kt % L::KS, j = kt / L::KS;
        if (!sy.wait(L::B_K_FULL + s, (uint32_t)(j & 1), kSiteKvFull)) return false;
        ptx::tc_fence_after();
        if (prev_uses > 0) {
            if (!sy.wait(L::B_S_READ + b, (uint32_t)((prev_uses - 1) & 1), kSiteSEmpty)) return false;
            ptx::tc_fence_after();
        }
        if (ptx::elect_one()) {
            const uint32_t d = tmem + 128u * b;
            const uint32_t kb = kb0 + (uint32_t)s * (L::TILE >> 4);
#pragma unroll
            for (int kc = 0; kc < L::KCH; ++kc)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    ptx::umma_ts_lh(d, tmem + L::TM_Q + 32u * kc + 8u * ks,
                                    kb + kc * (L::CHUNK >> 4) + 2 * ks, desc_hi, idesc_qk,
                                    (kc | ks) ? 1u : 0u);
            ptx::umma_commit(sy.bar(L::B_S_FULL + b));
            // the stage is free once this product has read it
            ptx::umma_commit(sy.bar(L::B_K_EMPTY + s));
        }
        __syncwarp();
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_k);
            ptx::tma_prefetch_desc(&tm_v);
            int kt = 0, vt = 0;                        // K and V loads issued
            bool ok = true;
            // load number cnt of a ring of ns stages goes to stage cnt % ns
            // and completes phase cnt / ns of that stage's full barrier
            auto load = [&](int t, bool is_v) -> bool {
                const int ns = is_v ? L::VS : L::KS;
                const int cnt = is_v ? vt : kt;
                const int s = cnt % ns, j = cnt / ns;
                const int empty = (is_v ? L::B_V_EMPTY : L::B_K_EMPTY) + s;
                if (!sy.wait(empty, (uint32_t)(j & 1) ^ 1u, kSiteKvEmpty)) return false;
                const uint32_t fb = sy.bar((is_v ? L::B_V_FULL : L::B_K_FULL) + s);
                ptx::mbar_arrive_expect_tx(fb, L::TILE);
                const uint32_t dst = (is_v ? sV : sK) + s * L::TILE;
                const CUtensorMap* map = is_v ? &tm_v : &tm_k;
#pragma unroll
                for (int kc = 0; kc < L::KCH; ++kc)
                    ptx::tma_load_3d(dst + kc * L::CHUNK, map, fb, kc * 64, (t0 + t) * L::BN, u);
                if (is_v) ++vt; else ++kt;
                return true;
            };
            // the order of first use: sweep 1 K(0..), sweep 2 K(0) K(1) then
            // K(t+2) V(t) for every t -- S(t+2) is issued as soon as the
            // softmax has loaded S(t), PV(t) only once P(t) is written, so
            // K(t+2) goes first; behind V(t), which waits for PV(t-2) to free
            // its stage, it arrived just in time for S(t+2) to enter the
            // tensor pipe ahead of PV(t) and delay it by a whole product
            for (int t = 0; ok && t < nt_mine; ++t) ok = load(t, false);
            for (int t = 0; ok && t < min(2, nt_mine); ++t) ok = load(t, false);
            for (int t = 0; ok && t < nt_mine; ++t) {
                if (t + 2 < nt_mine) ok = load(t + 2, false);
                if (ok) ok = load(t, true);
            }
            // never leave a copy in flight into this CTA's shared memory: wait
            // for the last load of every stage (load n of stage s is number
            // s + n * stages, its phase parity n & 1)
            for (int s = 0; s < L::KS && s < kt; ++s)
                sy.drain(L::B_K_FULL + s, (uint32_t)(((kt - 1 - s) / L::KS) & 1));
            for (int s = 0; s < L::VS && s < vt; ++s)
                sy.drain(L::B_V_FULL + s, (uint32_t)(((vt - 1 - s) / L::VS) & 1));
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- S = Q K^T issuer
        // Q is in TMEM once every softmax warp has stored its part
        bool ok = sy.wait(L::B_Q, 0, kSiteQFull);
        ptx::tc_fence_after();
        // sweep 1: three S buffers in rotation; this warp issues the even
        // tiles, the PV warp (idle until sweep 2) the odd ones
        for (int t = 0; ok && t < nt_mine; t += 2) ok = issue_s(t, t % L::SB1, t / L::SB1);
        // sweep 2: S buffers 0 and 1; S(t+2) waits only for S(t) to have
        // been loaded, so it is computed while the softmax works on S(t+1).
        // This warp now also consumes the K stages and S buffers the PV warp
        // used in sweep 1: it starts once that warp passed its last sweep-1
        // waits, or a parity wait here could match a phase two back
        if (ok) ok = sy.wait(L::B_S1_DONE, 0, kSiteSEmpty);
        for (int t = 0; ok && t < nt_mine; ++t) {
            const int b = t & 1;
            const int s1_uses = nt_mine > b ? (nt_mine - 1 - b) / L::SB1 + 1 : 0;
            ok = issue_s(nt_mine + t, b, s1_uses + t / 2);
        }
        // all MMAs complete before TMEM is released
        if (ptx::elect_one()) ptx::umma_commit(sy.bar(L::B_DRAIN));
        __syncwarp();
        sy.drain(L::B_DRAIN, 0);
    } else if (warp == 2) {
        // ---------------------------------------------------------- O += P V issuer
        constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, D, false, true);
        // a 16-key step of V (2048 bytes) adds 128 to the start-address field
        const uint32_t v_hi = (uint32_t)(ptx::sdesc_sw128(0, L::CHUNK, 1024) >> 32);
        const uint32_t vb0 = (uint32_t)ptx::sdesc_sw128(sV, L::CHUNK, 1024);
        uint32_t pv_par = 0;                           // parity of the next P_FULL phase
        const float* colbuf = reinterpret_cast<const float*>(base + L::OFF_COL);
        float* colsum = a.colsum + ((int64_t)u * n_rt + mt) * a.m_pad;
        const uint64_t keep_l2 = ptx::l2_policy_evict_last();
        // sweep 1: the odd S tiles (warp 1 issues the even ones)
        bool ok = sy.wait(L::B_Q, 0, kSiteQFull);
        ptx::tc_fence_after();
        for (int t = 1; ok && t < nt_mine; t += 2) ok = issue_s(t, t % L::SB1, t / L::SB1);
        if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_S1_DONE));
        // O overlays sweep-1 S buffer 2: P(0) is written only after every
        // softmax warp finished sweep 1, so PV(0) waiting for P(0) is enough
        for (int t = 0; ok && t < nt_mine; ++t) {
            const int vs = t % L::VS, jv = t / L::VS;
            if (!(ok = sy.wait(L::B_V_FULL + vs, (uint32_t)(jv & 1), kSiteKvFull))) break;
            // each 64-key half of P(t) goes to the tensor pipe as soon as its
            // 8 warps wrote it, and is handed back as soon as its 4 MMAs are
            // done: the warps of one half refill it while the other half's
            // products still run
            for (int h = 0; h < 2; ++h) {
                if (!(ok = sy.wait(L::B_P_FULL + h, pv_par, kSitePFull))) break;
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                    const uint32_t p_tmem = tmem + L::TM_P;
                    const uint32_t vb = vb0 + (uint32_t)vs * (L::TILE >> 4);
                    // MN-major V: LBO = distance between 64-wide d chunks,
                    // SBO = distance between 8-key row groups
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int ks = 4 * h + k4;
                        ptx::umma_ts_lh(tmem + L::TM_O, p_tmem + 8u * ks, vb + 128u * ks, v_hi,
                                        idesc_pv, (t | ks) ? 1u : 0u);
                    }
                    ptx::umma_commit(sy.bar(L::B_P_FREE + h));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (ptx::elect_one()) ptx::umma_commit(sy.bar(L::B_V_EMPTY + vs));
            __syncwarp();
            {
                pv_par ^= 1u;
                // key column sums of P(t): the 4 lane quarters' partials (kept
                // in L2 for the select kernel that reads them after this grid)
                const float* cb = colbuf + (t % L::NCOL) * 512;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int e = 32 * j + lane;
                    ptx::st_global_hint(colsum + (t0 + t) * L::BN + e,
                                        cb[e] + cb[128 + e] + cb[256 + e] + cb[384 + e], keep_l2);
                }
            }
        }
        if (ptx::elect_one()) {
            if (ok) ptx::umma_commit(sy.bar(L::B_O_FULL));
            ptx::umma_commit(sy.bar(L::B_DRAIN + 1));
        }
        __syncwarp();
        sy.drain(L::B_DRAIN + 1, 0);
    } else {
        // ------------------------------------------------------------ softmax
        // thread rows: 32*q4 + 16*hh + lane/4 + 8*sub (ri = 2*hh + sub);
        // columns of chunk cq: 32*cq + 8*rp + 2*(lane%4) + {0,1}
        const int sw = warp - 3;
        const int q4 = warp & 3;                       // TMEM lane quarter
        const int cq = sw >> 2;                        // 32-column chunk of the tile
        const float sc = a.scale_log2;
        const uint32_t lane_h0 = (uint32_t)(q4 * 32) << 16;
        const uint32_t lane_h1 = (uint32_t)(q4 * 32 + 16) << 16;
        int lim[4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) {
            const int r_unit = me.row0 + q4 * 32 + 16 * (ri >> 1) + (lane >> 2) + 8 * (ri & 1);
            lim[ri] = r_unit < a.GT ? a.c + (r_unit % a.T) : -1;  // kk visible iff kk <= lim
        }
        const int colb = 32 * cq + 2 * (lane & 3);     // tile column of this thread's pair 0
        const int ph = cq >> 1;                        // key half of P this warp writes
        float* colbuf = reinterpret_cast<float*>(base + L::OFF_COL);
        float2* statbuf = reinterpret_cast<float2*>(base + L::OFF_STAT);
        float* colsum = a.colsum + ((int64_t)u * n_rt + mt) * a.m_pad;
        uint32_t s_par = 0;                            // per S buffer: parity of the next S_FULL phase
        bool ok = true;
        auto load_s = [&](uint32_t t_s, uint32_t (&r0)[16], uint32_t (&r1)[16]) {
            ptx::tmem_ld_16x256b_x4(t_s + lane_h0 + 32 * cq, r0);
            ptx::tmem_ld_16x256b_x4(t_s + lane_h1 + 32 * cq, r1);
            ptx::tmem_ld_wait();
        };

        // ---- Q -> TMEM: lane = query row, bf16 pairs (even element low) along
        // the columns; each warp copies its lane quarter's rows, its chunk's
        // quarter of the d columns.  Rows past the unit's end are zero.
        {
            constexpr int QW = D / 8;                  // TMEM columns per chunk warp
            const int r_unit = me.row0 + q4 * 32 + lane;
            uint32_t qv[QW];
            if (r_unit < a.GT) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const uint8_t*>(a.q_rot) + ((int64_t)u * a.GT + r_unit) * (D * 2) +
                    cq * (D / 2));
#pragma unroll
                for (int j = 0; j < QW / 4; ++j) {
                    const uint4 v = src[j];
                    qv[4 * j] = v.x; qv[4 * j + 1] = v.y; qv[4 * j + 2] = v.z; qv[4 * j + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < QW; ++j) qv[j] = 0u;
            }
            const uint32_t t_q = tmem + L::TM_Q + lane_h0 + QW * cq;
            if constexpr (QW == 16) ptx::tmem_st_32x32b_x16(t_q, qv);
            else ptx::tmem_st_32x32b_x8(t_q, qv);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_Q));
        }

        // ---- sweep 1: per-thread running max / sum of exp2 over its columns
        float mrow[4], lrow[4], nref[4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) { mrow[ri] = -INFINITY; lrow[ri] = 0.f; nref[ri] = 0.f; }
        for (int t = 0, b = 0; t < nt_mine; ++t, b = (b == L::SB1 - 1) ? 0 : b + 1) {
            if (!sy.wait(L::B_S_FULL + b, (s_par >> b) & 1u, kSiteSFull)) { ok = false; break; }
            ptx::tc_fence_after();
            uint32_t r0[16], r1[16];
            load_s(tmem + 128u * b, r0, r1);
            // the buffer is free for the next S as soon as it is in registers
            // (wait::ld above; the arrive orders no memory access, so it is
            // relaxed and does not wait for this warp's column-sum stores)
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_relaxed(sy.bar(L::B_S_READ + b));
            s_par ^= 1u << b;
            const int k0 = (t0 + t) * L::BN + colb;
            // fully visible tiles and the few diagonal ones are separate
            // instantiations: the per-element mask would otherwise be
            // if-converted into every tile (16 % of the kernel's instructions)
            auto rows1 = [&](auto diag_tag) {
            constexpr bool diag = decltype(diag_tag)::value;
            // the row's 8 scores of this tile (masked ones -inf)
            auto row_x = [&](int ri, float (&x)[8]) {
                const uint32_t* r = (ri >> 1) ? r1 : r0;
                const int sub = ri & 1;
#pragma unroll
                for (int rp = 0; rp < 4; ++rp) {
                    x[2 * rp] = __uint_as_float(r[4 * rp + 2 * sub]);
                    x[2 * rp + 1] = __uint_as_float(r[4 * rp + 2 * sub + 1]);
                }
                if constexpr (diag) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (k0 + 8 * (e >> 1) + (e & 1) > lim[ri]) x[e] = -INFINITY;
                }
            };
            auto row_sum = [&](const float (&x)[8], float nref) -> float {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float2 z = ptx::fma2(make_float2(x[e], x[e + 1]), make_float2(sc, sc),
                                         make_float2(nref, nref));
                    acc = ptx::add2(acc, make_float2(ptx::ex2_approx(z.x), ptx::ex2_approx(z.y)));
                }
                return acc.x + acc.y;
            };
            // each row sums exp2 against a reference (its running max as of the
            // last time it was raised); the reference is raised only when a
            // row is new or a tile's sum passes 2^32
            float part[4];
            bool raise = false;
#pragma unroll
            for (int ri = 0; ri < 4; ++ri) {
                float x[8];
                row_x(ri, x);
                part[ri] = row_sum(x, nref[ri]);
                raise |= !(part[ri] <= 0x1p32f) || mrow[ri] == -INFINITY;
            }
            if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
                for (int ri = 0; ri < 4; ++ri) {
                    if (!(part[ri] <= 0x1p32f) || mrow[ri] == -INFINITY) {
                        float x[8];
                        row_x(ri, x);
                        const float mx = ptx::max3(ptx::max3(x[0], x[1], x[2]),
                                                   ptx::max3(x[3], x[4], x[5]),
                                                   ptx::max3(x[6], x[7], mrow[ri]));
                        if (mx != -INFINITY) {
                            if (mrow[ri] != -INFINITY)
                                lrow[ri] *= ptx::ex2_approx((mrow[ri] - mx) * sc);
                            mrow[ri] = mx;
                            nref[ri] = -mx * sc;
                        }
                        part[ri] = row_sum(x, nref[ri]);
                    }
                }
            }
#pragma unroll
            for (int ri = 0; ri < 4; ++ri) lrow[ri] += part[ri];
            };
            if (t0 + t >= me.nfull) rows1(std::true_type{});
            else rows1(std::false_type{});
        }
        // combine once per row: every thread stores its (reference, sum) for
        // its 4 rows (16 threads hold parts of a row: 4 lanes x 4 chunk
        // warps), then the 4 warps of chunk 0 merge one row per thread and
        // publish its lse; merging in every thread instead repeats each
        // row's merge 16 times right where no other work overlaps it
        {
            const int e = cq * 4 + (lane & 3);
#pragma unroll
            for (int ri = 0; ri < 4; ++ri) {
                const int row = q4 * 32 + 16 * (ri >> 1) + (lane >> 2) + 8 * (ri & 1);
                statbuf[e * 128 + row] = make_float2(mrow[ri], lrow[ri]);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_STAT));
        float* lsebuf = reinterpret_cast<float*>(base + L::OFF_LSE);
        if (cq == 0) {
            if (!sy.wait(L::B_STAT, 0, kSiteCol)) ok = false;
            const int row = q4 * 32 + lane;
            float2 st[16];
            float m = -INFINITY;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                st[e] = statbuf[e * 128 + row];
                m = fmaxf(m, st[e].x);
            }
            float l = 0.f;
            if (m != -INFINITY) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (st[e].x != -INFINITY) l = fmaf(st[e].y, ptx::ex2_approx((st[e].x - m) * sc), l);
            }
            float lse = (me.row0 + row < a.GT && l > 0.f) ? fmaf(m, sc, log2f(l)) : INFINITY;
            if (SPLIT && coop) {
                // the row's lse over this CTA's key range (-inf: no key),
                // sent to every other CTA of the split; all combine the ks
                // partials in rank order, so every CTA gets the same bits
                const float part = l > 0.f ? fmaf(m, sc, log2f(l)) : -INFINITY;
                const uint32_t slot = sbase + L::OFF_XLSE + 4u * (uint32_t)(rank * 128 + row);
                for (int j = 0; j < ks; ++j)
                    if (j != rank) ptx::st_cluster_f32(ptx::cluster_map(slot, (uint32_t)j), part);
                // the warp's 32 rows, then one fence and one 32-count arrive
                // per destination
                __syncwarp();
                if (lane == 0) {
                    ptx::fence_acq_rel_cluster();
                    for (int j = 0; j < ks; ++j)
                        if (j != rank)
                            ptx::mbar_arrive_remote_relaxed(
                                ptx::cluster_map(sy.bar(L::B_XLSE), (uint32_t)j), 32u);
                }
                if (!sy.wait_cluster(L::B_XLSE, 0, kSiteCol)) ok = false;
                const float* xl = reinterpret_cast<const float*>(base + L::OFF_XLSE);
                float mx = -INFINITY;
                for (int j = 0; j < ks; ++j) mx = fmaxf(mx, j == rank ? part : xl[j * 128 + row]);
                float sum = 0.f;
                if (mx != -INFINITY)
                    for (int j = 0; j < ks; ++j)
                        sum += exp2f((j == rank ? part : xl[j * 128 + row]) - mx);
                lse = (me.row0 + row < a.GT && mx != -INFINITY) ? mx + log2f(sum) : INFINITY;
            }
            lsebuf[row] = lse;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_LSE));
        }
        float lse2[4];
        if (!sy.wait(L::B_LSE, 0, kSiteCol)) ok = false;
#pragma unroll
        for (int ri = 0; ri < 4; ++ri)
            lse2[ri] = lsebuf[q4 * 32 + 16 * (ri >> 1) + (lane >> 2) + 8 * (ri & 1)];

        // ---- sweep 2: P, its column sums, P -> TMEM (bf16) for PV
        uint32_t p_par = 0;                            // parity of the P_FREE phase of PV(t-1)
        for (int t = 0, slot = 0; ok && t < nt_mine; ++t, slot = (slot == L::NCOL - 1) ? 0 : slot + 1) {
            const int b = t & 1;
            if (!sy.wait(L::B_S_FULL + b, (s_par >> b) & 1u, kSiteSFull)) { ok = false; break; }
            ptx::tc_fence_after();
            uint32_t r0[16], r1[16];
            load_s(tmem + 128u * b, r0, r1);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_relaxed(sy.bar(L::B_S_READ + b));
            s_par ^= 1u << b;
            const int k0 = (t0 + t) * L::BN + colb;
            float c[8];                                // column partials: k = 2*rp + e
            uint32_t pk[2][8];
            auto rows2 = [&](auto diag_tag) {
            constexpr bool diag = decltype(diag_tag)::value;
#pragma unroll
            for (int ri = 0; ri < 4; ++ri) {
                const uint32_t* r = (ri >> 1) ? r1 : r0;
                const int sub = ri & 1;
                const float nl = -lse2[ri];
#pragma unroll
                for (int rp = 0; rp < 4; ++rp) {
                    float2 z = ptx::fma2(make_float2(__uint_as_float(r[4 * rp + 2 * sub]),
                                                     __uint_as_float(r[4 * rp + 2 * sub + 1])),
                                         make_float2(sc, sc), make_float2(nl, nl));
                    float2 p = make_float2(ptx::ex2_approx(z.x), ptx::ex2_approx(z.y));
                    if constexpr (diag) {
                        if (k0 + 8 * rp > lim[ri]) p.x = 0.f;
                        if (k0 + 8 * rp + 1 > lim[ri]) p.y = 0.f;
                    }
                    if (ri == 0) { c[2 * rp] = p.x; c[2 * rp + 1] = p.y; }
                    else {
                        const float2 cc = ptx::add2(make_float2(c[2 * rp], c[2 * rp + 1]), p);
                        c[2 * rp] = cc.x; c[2 * rp + 1] = cc.y;
                    }
                    pk[ri >> 1][2 * rp + sub] = ptx::pack_bf16x2(p.x, p.y);
                }
            }
            };
            if (t0 + t >= me.nfull) rows2(std::true_type{});
            else rows2(std::false_type{});
            // this warp's half of P is free once its half of PV(t-1) has
            // completed (issued when that half of P(t-1) was complete)
            if (t > 0 && !sy.wait(L::B_P_FREE + ph, p_par, kSitePEmpty)) {
                ok = false;
                break;
            }
            if (t > 0) p_par ^= 1u;
            ptx::tc_fence_after();
            const uint32_t t_p = tmem + L::TM_P + 16u * cq;
            ptx::tmem_st_16x128b_x4(t_p + lane_h0, pk[0]);
            ptx::tmem_st_16x128b_x4(t_p + lane_h1, pk[1]);
            // column sums over the warp's 32 rows: lanes sharing lane&3 hold the
            // same columns; reduce over lane bits 4, 3, 2 (keep half each)
#pragma unroll
            for (int half = 4, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
                const bool up = (lane & bit) != 0;
#pragma unroll
                for (int j = 0; j < half; ++j) {
                    const float send = up ? c[j] : c[j + half];
                    const float keep = up ? c[j + half] : c[j];
                    c[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
                }
            }
            // lane holds chunk column 8*((lane>>3)&3) + 2*(lane&3) + ((lane>>2)&1);
            // the PV issuer sums the 4 lane quarters once P_FULL(t) (a release
            // after this store) completes; slot t % NCOL is rewritten at tile
            // t + NCOL only after PV(t+NCOL-1), which that warp issues after
            // reading the slot
            colbuf[slot * 512 + q4 * 128 + 32 * cq + 8 * ((lane >> 3) & 3) + 2 * (lane & 3) +
                   ((lane >> 2) & 1)] = c[0];
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sy.bar(L::B_P_FULL + ph));
        }
        if (SPLIT && coop) {
            // this CTA's key tiles are consumed: the others may put their O
            // columns into our K stages (the signal orders no memory access:
            // the products that read the stages completed before S_FULL)
            __syncwarp();
            if (lane == 0)
                for (int j = 0; j < ks; ++j)
                    if (j != rank)
                        ptx::mbar_arrive_remote_relaxed(
                            ptx::cluster_map(sy.bar(L::B_XREADY), (uint32_t)j), 1u);
        }
        if (me.nt > 0 && (!coop || rank == ks - 1))    // the CTA holding the last tiles
            for (int kk = me.nt * L::BN + sw * 32 + lane; kk < a.m_pad; kk += 32 * L::SW)
                colsum[kk] = 0.f;

        // ---- output rows: quarter q4, 32 columns per warp
        if (SPLIT && coop) {
            // CTA r outputs columns [r*bw, (r+1)*bw): the others store their
            // partial O of them column-major into its K stages (slot of
            // sender j at [j*bw][128], so a warp's 32 lanes = 32 rows write
            // consecutive words) and it adds the ks partials in rank order
            if (cq < D / 32) {
                const int c0 = 32 * cq;
                const int row = q4 * 32 + lane;
                float v[32];
                bool have = false;
                if (ok && nt_mine > 0 && sy.wait(L::B_O_FULL, 0, kSiteOFull)) {
                    ptx::tc_fence_after();
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(tmem + L::TM_O + lane_h0 + 32 * cq, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    have = true;
                }
                if (!have) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;   // no key tiles: no mass
                }
                // owners of this warp's 32 columns (bw is a multiple of 8)
                const int o_lo = c0 / bw, o_hi = min((c0 + 31) / bw, ks - 1);
                if (o_lo != rank || o_hi != rank) {
                    if (sy.wait_cluster(L::B_XREADY, 0, kSiteCol)) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int o = (c0 + j) / bw;
                            if (o != rank) {
                                const uint32_t col = (uint32_t)(rank * bw + (c0 + j - o * bw));
                                ptx::st_cluster_f32(ptx::cluster_map(sK + 4u * (col * 128 + row),
                                                                     (uint32_t)o), v[j]);
                            }
                        }
                    }
                    // the warp's stores, then one fence and one 32-count
                    // arrive per owner
                    __syncwarp();
                    if (lane == 0) {
                        ptx::fence_acq_rel_cluster();
                        for (int o = o_lo; o <= o_hi; ++o)
                            if (o != rank)
                                ptx::mbar_arrive_remote_relaxed(
                                    ptx::cluster_map(sy.bar(L::B_XO), (uint32_t)o), 32u);
                    }
                }
                const int lo = max(c0, rank * bw), hi = min(c0 + 32, (rank + 1) * bw);
                if (lo < hi && sy.wait_cluster(L::B_XO, 0, kSiteCol) && me.row0 + row < a.GT) {
                    const float* xo = reinterpret_cast<const float*>(base + L::OFF_K);
                    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o) +
                                         ((int64_t)u * a.GT + me.row0 + row) * D + c0;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (c0 + 8 * g < lo || c0 + 8 * g >= hi) continue;
                        uint32_t wv[4];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const int j = 8 * g + e;
                            const int col = c0 + j - rank * bw;      // within this CTA's columns
                            float s0 = 0.f, s1 = 0.f;
                            for (int r = 0; r < ks; ++r) {
                                s0 += r == rank ? v[j] : xo[(r * bw + col) * 128 + row];
                                s1 += r == rank ? v[j + 1] : xo[(r * bw + col + 1) * 128 + row];
                            }
                            wv[e / 2] = ptx::pack_bf16x2(s0, s1);
                        }
                        reinterpret_cast<uint4*>(out)[g] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }
        } else if (me.nt > 0 && ok && cq < D / 32 && sy.wait(L::B_O_FULL, 0, kSiteOFull)) {
            ptx::tc_fence_after();
            const int r_unit = me.row0 + q4 * 32 + lane;
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tmem + L::TM_O + lane_h0 + 32 * cq, r);
            ptx::tmem_ld_wait();
            if (r_unit < a.GT) {
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.o) +
                                     ((int64_t)u * a.GT + r_unit) * D + 32 * cq;
                uint32_t wv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    wv[j] = ptx::pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(wv[4 * v4], wv[4 * v4 + 1], wv[4 * v4 + 2], wv[4 * v4 + 3]);
            }
        }
        ptx::tc_fence_before();
    }

    __syncthreads();
    // no CTA leaves while its split-tile peer may still write into it or
    // arrive on its barriers (every role above has drained its own traffic)
    if (coop) ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

template <int D>
cudaLaunchConfig_t grid_config(cudaStream_t st, int grid, int ks, cudaLaunchAttribute (&attr)[2]) {
    using L = TcLayout<D>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(L::THREADS);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

template <int D, int KSC>
cudaError_t launch_grid(const AttnArgs& a, const TcMaps& m, cudaStream_t st, int grid) {
    using L = TcLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, KSC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = grid_config<D>(st, grid, a.split_ks, attr);
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, KSC>, m.k, m.v, a);
}

// Clusters of ks split CTAs that one wave holds on this device (0 when the
// query fails), cached per (device, D, ks).
template <int D>
int clusters_per_wave(int ks) {
    static std::mutex mu;
    static int cache[64][L_KSMAX + 1];
    static bool init = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!init) {
        for (auto& row : cache)
            for (int& x : row) x = -1;
        init = true;
    }
    int& c = cache[dev][ks];
    if (c < 0) {
        c = 0;
        if (cudaFuncSetAttribute(attn_tc_kernel<D, 0>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcLayout<D>::SMEM) == cudaSuccess) {
            cudaLaunchAttribute attr[2];
            const cudaLaunchConfig_t cfg = grid_config<D>(nullptr, ks, ks, attr);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<D, 0>, &cfg) == cudaSuccess)
                c = n;
        }
        cudaGetLastError();
    }
    return c;
}

// Which query tiles run split over their keys, and over how many CTAs.
//  * At least one full wave (one CTA per SM, a.resident SMs): the tiles of
//    the last, partial wave, when it fills at most half the SMs, as pairs.
//  * Fewer tiles than SMs (e.g. one layer per launch): every tile, over the
//    ks in 1..8 with the least estimated time, waves(ks) * (P + nt / ks):
//    nt key tiles per query tile (at most), P ~ 4 key tiles' worth of
//    per-CTA set-up, exchange and output, waves from the clusters of ks CTAs
//    the device holds at once (a cluster needs ks free SMs of one GPC).
// STATEKV_ATTN_SPLIT overrides which tiles: 0 = none, all = every tile, n =
// the last n; STATEKV_ATTN_SPLIT_WAYS (2..8, default 2) the CTAs per tile.
struct SplitPlan {
    int split;      // tiles split (the last ones)
    int ks;         // CTAs per split tile
};

template <int D>
SplitPlan plan_split(const AttnArgs& a, int items) {
    const char* env = std::getenv("STATEKV_ATTN_SPLIT");
    if (env && *env) {
        int ks = 2;
        if (const char* w = std::getenv("STATEKV_ATTN_SPLIT_WAYS"))
            ks = std::max(2, std::min(L_KSMAX, std::atoi(w)));
        if (std::strcmp(env, "all") == 0) return {items, ks};
        const long n = std::strtol(env, nullptr, 10);
        return {(int)std::max(0L, std::min((long)items, n)), ks};
    }
    if (a.resident <= 0) return {0, 1};
    if (items >= a.resident) {
        const int full = items / a.resident * a.resident, tail = items - full;
        return {(tail > 0 && 2 * tail <= a.resident) ? tail : 0, 2};
    }
    const double nt = (double)((a.c + a.T + 127) / 128);
    constexpr double P = 4.0;
    int best = 1;
    double best_cost = P + nt;                   // unsplit: one wave
    for (int ks = 2; ks <= L_KSMAX; ++ks) {
        const int per_wave = clusters_per_wave<D>(ks);
        if (per_wave <= 0) continue;
        const double waves = (double)((items + per_wave - 1) / per_wave);
        const double cost = waves * (P + nt / ks);
        if (cost < best_cost) { best_cost = cost; best = ks; }
    }
    return best > 1 ? SplitPlan{items, best} : SplitPlan{0, 1};
}

template <int D>
cudaError_t launch_tc(const AttnArgs& a_in, const TcMaps& m, cudaStream_t st) {
    const int items = a_in.U * a_in.n_row_tiles;
    AttnArgs a = a_in;
    SplitPlan p = plan_split<D>(a, items);
    if (p.split == 0) {
        a.split_item0 = items;
        a.split_ks = 1;
        return launch_grid<D, 1>(a, m, st, items);
    }
    // whole tiles go ks per cluster: a multiple of ks of them
    const int ks = p.ks;
    int split = p.split + (items - p.split) % ks;
    a.split_item0 = items - split;
    a.split_ks = ks;
    const int grid = a.split_item0 + ks * split;
    return ks == 2 ? launch_grid<D, 2>(a, m, st, grid) : launch_grid<D, 0>(a, m, st, grid);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode_view(CUtensorMap* m, const void* base, int d, int64_t rows, int64_t units,
                 int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_tc_maps(TcMaps* m, const void* pool_k, const void* pool_v, int d, int64_t slots,
                  int64_t units) {
    return encode_view(&m->k, pool_k, d, slots, units, 128) &&
           encode_view(&m->v, pool_v, d, slots, units, 128);
}

cudaError_t launch_attention_tc(const AttnArgs& a, const TcMaps& m, cudaStream_t st) {
    if (a.d == 128) return launch_tc<128>(a, m, st);
    if (a.d == 64) return launch_tc<64>(a, m, st);
    return cudaErrorInvalidValue;
}

}  // namespace statekv
