// Internal declarations shared by the libstatekv translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "statekv.h"

namespace statekv {

// Device status word layout (uint32[4]): [0] status code (STATEKV_E_*),
// [1] site id of the first failure, [2] blockIdx.x, [3] extra.
constexpr int kErrWords = 4;

// Error sites recorded by bounded waits.
enum ErrSite : uint32_t {
    kSiteQFull = 1, kSiteKvFull, kSiteKvEmpty, kSiteSFull, kSiteSEmpty,
    kSitePFull, kSitePEmpty, kSiteOFull, kSiteDrain, kSiteTmemAddr, kSiteCol,
    kSiteSelect = 32,
};

// ------------------------------------------------------------- launchers
struct RopeArgs {
    const void* q; const void* k; const void* v;   // caller inputs
    void* q_rot;                                   // [U*G*T][d]
    void* pool_k; void* pool_v;                    // [U][slots][d]
    void* det_k; void* det_v;                      // [U][det_pitch][d]
    const float2* cs;                              // [T][d/2] (cos, sin), vector-interleaved
                                                   // rows (rope_cs_index)
    int64_t rows_q;      // S*L*Hq*T
    int64_t rows_kv;     // S*L*Hkv*T
    int32_t T, d, slots, c;
    int64_t det_pitch, det_row0;                   // det row of token 0 = n*T
};

struct RopeTableArgs {
    const double* omega;  // [d/2]
    float2* cs;           // [T][d/2], rows vector-interleaved (rope_cs_index)
    int64_t p0;           // virtual position of token 0 of this frame
    int32_t T, half;
    int32_t vec;          // pairs per RoPE thread: 8 (bf16) or 4 (fp32)
};

// Where pair k of a row sits in the (cos, sin) table.  A RoPE thread j
// rotates pairs [j*vec, (j+1)*vec) of a row; the table keeps its pairs 2e and
// 2e+1 side by side (one 16-byte load) and the same pair step of consecutive
// threads in consecutive 16 bytes, so a warp's loads of one step are
// contiguous instead of vec*8 bytes apart.
__host__ __device__ __forceinline__ int rope_cs_index(int k, int half, int vec) {
    const int tpr = half / vec, j = k / vec, e = k - j * vec;
    return ((e >> 1) * tpr + j) * 2 + (e & 1);
}

struct AttnArgs {
    const void* q_rot;    // [U][GT][d]
    const void* pool_k;   // [U][slots][d]
    const void* pool_v;
    void* o;              // [U][GT][d]
    float* colsum;        // [U][n_row_tiles][m_pad] per-tile key column sums of P
    uint32_t* err;
    int32_t U, GT, T, d, slots, c, m_pad, n_row_tiles;
    float scale_log2;     // mscale^2/sqrt(d) * log2(e)
    float scale;          // mscale^2/sqrt(d)
    // query tiles [split_item0, U * n_row_tiles) run split over the keys,
    // each by the split_ks CTAs of a cluster (set by the launcher); resident
    // = CTAs one wave holds (one per SM; 0: never split)
    int32_t split_item0;
    int32_t split_ks;
    int32_t resident;
};

struct SelectArgs {
    const float* colsum;  // [U][n_row_tiles][m_pad]
    float* scores;        // [U][m_pad]
    int32_t* score_pos;   // [U][m_pad]
    int32_t* pos;         // [U][slots] live positions of the compressed pool
    void* pool_k; void* pool_v;   // [U][slots][row_bytes]
    uint32_t* err;
    int32_t U, n_row_tiles, m_pad, slots, c, T, B, row_bytes;
    int32_t pos_base;     // virtual position of this frame's token 0
    float inv_rows;       // 1 / (G*T)
    int32_t window;       // 1: keep the B most recent tokens instead of Top-B
    int32_t never_evicts; // B >= every pool size this handle can reach
    int32_t num_sms;      // SMs of the device (sets the CTA size)
    int32_t cluster;      // CTAs per unit (a thread-block cluster; set by the launcher)
};

cudaError_t launch_rope_table(const RopeTableArgs& a, cudaStream_t st);
cudaError_t launch_rope(const RopeArgs& a, int dtype, cudaStream_t st, bool early);
// TMA views of the attention kernel's operands: K and V of the pool as
// [units][slots][d], read in 128-row boxes.
struct TcMaps {
    CUtensorMap k, v;
};
bool make_tc_maps(TcMaps* m, const void* pool_k, const void* pool_v, int d, int64_t slots,
                  int64_t units);
cudaError_t launch_attention_tc(const AttnArgs& a, const TcMaps& maps, cudaStream_t st);
cudaError_t launch_attention_simt(const AttnArgs& a, cudaStream_t st);

// Text decode over the detailed state (decode.cu): R = G*tok query rows per
// unit, keys = visible + tok D rows, partials per (unit, key chunk).
struct DecodeArgs {
    void* o;                     // [U][R][128] bf16
    float* part_m;               // [U*chunks][npad]  row reference (log2 units)
    float* part_l;               // [U*chunks][npad]  row sum
    float* part_o;               // [U*chunks][npad][128] unnormalised O
    uint32_t* err;
    int32_t U, R, tok, chunks, num_sms;
    int64_t visible, keys;
    float scale_log2;
};
struct DecodeMaps {
    CUtensorMap q, k, v;
};
int decode_rows_pad(int R);            // 16 / 32 / 64, or -1 when R > 64
int decode_chunks(int64_t keys);       // key chunks per unit
bool make_decode_maps(DecodeMaps* m, const void* q_rot, int R, int npad, const void* det_k,
                      const void* det_v, int64_t det_pitch, int64_t units);
cudaError_t launch_decode(const DecodeArgs& a, const DecodeMaps& m, cudaStream_t st);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);

// Query-row tile heights of the two attention paths (the column-sum buffer
// holds one row of partial sums per tile).
constexpr int kTcRowTile = 128;
constexpr int kSimtRowTile = 16;
// Dynamic shared memory of the select kernel for B + T candidates.
size_t select_smem_bytes(int slots, int T);
constexpr int kMaxSlots = 24576;
// dynamic shared memory the selection may take: the 227 KB a CTA can have
// less what the kernel declares statically (histogram, scan, flags)
constexpr size_t kSelectSmemMax = 227 * 1024 - 4096;

}  // namespace statekv

// ---------------------------------------------------------- device helpers
#ifdef __CUDACC__
namespace statekv {

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Record the first device-side failure; later ones are dropped.
__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code,
                                             uint32_t site, uint32_t extra) {
    if (atomicCAS(err, 0u, code) == 0u) {
        err[1] = site;
        err[2] = blockIdx.x;
        err[3] = extra;
        __threadfence();
    }
}

}  // namespace statekv
#endif
