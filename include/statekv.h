/*
 * statekv.h -- C ABI of libstatekv, the GB300 (sm_103a) implementation of
 * StateKV streaming video prefill.
 *
 * Method: "Linear Scaling Video VLMs for Long Video Understanding" (StateKV,
 * ECCV 2026), papernotes.org summary, section 方法详解:
 *   整体框架 (overall framework) -- frames arrive one at a time, T visual tokens
 *     each; in every layer the frame attends only to a fixed-capacity
 *     compressed state C_{n-1} and to itself, so the per-frame cost is
 *     O(T^2 + BT) and the prefill is linear in the number of frames N;
 *   关键设计 1 (dual state) -- per layer a detailed state D_n holding every
 *     frame's K/V (kept for text decoding) and a compressed state C_n with
 *     |K̄_n| = B; Q_n attends over [K̄_{n-1}; K_n];
 *   关键设计 2 (temporal-sink update) -- candidate pool U_n = S̄_{n-1} ∪ {1..T},
 *     score s_j = mean attention the frame's queries pay to key j,
 *     S̄_n = TopK({s_j}, B) rebuilds C_n;
 *   关键设计 3 (virtual length, static RoPE scale) -- RoPE angles use the
 *     logical stream position L_n = nT (+ i); one global scale alpha is fixed
 *     before prefill and never changes.
 *
 * Readings of points the page leaves open (fixed here, per KV head):
 *   - mask: compressed keys fully visible; frame key i' visible to query i iff
 *     i' <= i;
 *   - s_j averages P over all G*T query rows of the G query heads that share
 *     the KV head (a query that cannot see j contributes 0);
 *   - Top-B ties go to the lower virtual position;
 *   - positions p = position_offset + n*T + i, n 0-based;
 *   - alpha != 1 is YaRN NTK-by-parts (beta_fast 32, beta_slow 1) with logit
 *     factor mscale^2, mscale = 0.1 ln(alpha) + 1;
 *   - C and D hold post-RoPE keys in the storage dtype.
 *
 * Threading and streams: a handle is not thread-safe; calls on one handle
 * must be serialised by the caller.  All device work of a call is enqueued
 * asynchronously on the caller's CUDA stream (cudaStream_t passed as void*,
 * NULL = the legacy default stream); results are valid once that stream has
 * reached the point after the call.
 *
 * Errors: every entry point returns an int status (STATEKV_OK or a negative
 * STATEKV_E_*).  Nothing aborts and no C++ exception crosses the ABI.  Host
 * argument checks happen before any device work, so a call rejected with
 * E_INVALID_ARG / E_UNSUPPORTED / E_CAPACITY leaves the handle unchanged.
 * E_CUDA means a CUDA call failed (the handle's device state is then
 * unspecified; destroy it); the call clears the CUDA runtime's last-error
 * state before returning, so a refused launch does not resurface in later
 * calls.  Device-side bounded waits that give up record a
 * status that statekv_check_device_status() reports as E_TIMEOUT.
 */
#ifndef STATEKV_H_
#define STATEKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------ selection policy */
#define STATEKV_SELECT_TOPB    0    /* Top-B by attention score (StateKV)    */
#define STATEKV_SELECT_WINDOW  1    /* the B most recent tokens (ReKV-style)  */

/* ---------------------------------------------------------------- status */
#define STATEKV_OK              0
#define STATEKV_E_INVALID_ARG  -1   /* null pointer, bad size, bad index      */
#define STATEKV_E_UNSUPPORTED  -2   /* valid but not implemented (e.g. d=96)  */
#define STATEKV_E_CAPACITY     -3   /* detailed state full (n == max_frames)  */
#define STATEKV_E_OOM          -4   /* device allocation failed at create     */
#define STATEKV_E_CUDA         -5   /* a CUDA runtime/driver call failed      */
#define STATEKV_E_TIMEOUT      -6   /* a device-side bounded wait gave up     */
#define STATEKV_E_DEVICE       -7   /* a device-side consistency check failed */

/* storage dtypes */
#define STATEKV_BF16 0              /* bf16 storage, fp32 accumulation        */
#define STATEKV_F32  1              /* fp32 storage and arithmetic            */

/* kernels, for statekv_profile_read() */
#define STATEKV_KERNEL_ROPE_TABLE 0 /* cos/sin table (computed once, at create: */
                                    /* no launches inside a prefill)            */
#define STATEKV_KERNEL_ROPE       1 /* RoPE at virtual positions + appends    */
#define STATEKV_KERNEL_ATTENTION  2 /* two-sweep attention + key column sums  */
#define STATEKV_KERNEL_SELECT     3 /* score finish, Top-B, slot-reuse gather */
#define STATEKV_NUM_KERNELS       4

typedef struct statekv_handle statekv_handle;   /* opaque */

/*
 * Configuration of one handle.  Every (stream, layer, KV head) is an
 * independent unit with its own C and D; all units advance together, one
 * frame per statekv_prefill_frame call.
 *   num_streams   S >= 1   independent videos stepped together
 *   num_layers    L >= 1   transformer layers (inputs per layer are given)
 *   num_q_heads   Hq       query heads; Hq % Hkv == 0, G = Hq / Hkv
 *   num_kv_heads  Hkv >= 1 KV heads (query head j uses KV head j / G)
 *   head_dim      d        64 or 128
 *   frame_tokens  T >= 1   visual tokens per frame
 *   budget        B >= 0   compressed-state capacity (关键设计 1, |K̄| = B)
 *   max_frames    N_max    capacity of the detailed state D, in frames
 *   dtype         STATEKV_BF16 or STATEKV_F32
 *   device        CUDA device ordinal the handle lives on
 *   rope_theta    RoPE base theta (> 1)
 *   rope_alpha    static global RoPE scale alpha >= 1, fixed for the
 *                 handle's lifetime (关键设计 3)
 *   rope_orig_ctx YaRN original context L_orig (> 0 when alpha != 1)
 *   position_offset virtual position of the first video token (>= 0)
 *   select_policy STATEKV_SELECT_TOPB (the method, 关键设计 2) or
 *                 STATEKV_SELECT_WINDOW: keep the B most recent tokens
 *                 instead, the sliding-window baseline the page compares
 *                 against (ReKV, R frames = B/T).  Full self-attention is
 *                 budget >= max_frames*T with either policy (nothing is ever
 *                 evicted).
 * Limits: G*T <= 65536 query rows per unit; B + T <= 24576 unless
 * B >= max_frames*T (no eviction: then only memory bounds the pool);
 * positions must fit in int32.
 * The bf16 attention runs one CTA per 128-row query tile.  Some tiles are
 * split over their keys among the CTAs of a thread-block cluster, which
 * exchange their row log-sum-exps and partial outputs through distributed
 * shared memory (results agree with whole tiles up to rounding, and are
 * deterministic): with at least one full wave of tiles (one per SM), the
 * tiles of the last, partial wave when it fills at most half the SMs, as
 * pairs; with fewer tiles than SMs (for example one layer per call), every
 * tile, over 2..8 CTAs chosen from how many such clusters the device holds
 * at once.  The selection likewise spreads each unit over a cluster of up to
 * 8 CTAs when the units are few.  Test overrides, read at every prefill
 * launch: STATEKV_ATTN_SPLIT (0 = no split, all = every tile, n = the last n
 * tiles) with STATEKV_ATTN_SPLIT_WAYS (2..8, default 2), and
 * STATEKV_SELECT_CLUSTER (1, 2, 4 or 8 CTAs per unit).
 */
typedef struct statekv_config {
    int32_t num_streams;
    int32_t num_layers;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t frame_tokens;
    int32_t budget;
    int32_t max_frames;
    int32_t dtype;
    int32_t device;
    double  rope_theta;
    double  rope_alpha;
    int64_t rope_orig_ctx;
    int64_t position_offset;
    int32_t select_policy;
} statekv_config;

/* Human-readable name of a status code (static storage, never NULL). */
const char* statekv_status_string(int status);

/*
 * Create a handle: validates cfg, allocates on cfg->device (current device is
 * restored on return) the compressed pool [S][L][Hkv][B+T][d] for K and V,
 * its positions [S][L][Hkv][B+T] int32, the detailed state
 * [S][L][Hkv][N_max*T][d] for K and V, scratch (rotated queries, per-tile key
 * column sums, scores) and one frame of staging for the host-buffer entry
 * point.  All device memory is zero-filled.  The handle owns it all.
 * On failure *out is set to NULL and nothing is leaked.
 */
int statekv_create(const statekv_config* cfg, statekv_handle** out);

/* Free everything the handle owns (synchronises the device first). NULL ok. */
int statekv_destroy(statekv_handle* h);

/*
 * One frame step n (= statekv_frame_index(h)) for every unit (整体框架,
 * 关键设计 1-3):
 *   1. rotate Q and K at p = position_offset + n*T + i with the static
 *      frequencies, store K' and V into D rows [n*T, n*T+T) and into the
 *      compressed pool after the c = min(B, n*T) live slots;
 *   2. O = softmax(Q' [K̄_{n-1}; K'_n]^T * mscale^2/sqrt(d), masked) [V̄; V];
 *   3. s_j for every pool slot, Top-B with ties to the lower position;
 *   4. C_n keeps the B winners: evicted slots are refilled in place by the
 *      surviving frame rows (slot order is not position order).
 * Pointers are DEVICE pointers on the handle's device, caller-owned,
 * contiguous, in the storage dtype:
 *   q, o : [S][L][Hq][T][d]      (o is written, never read)
 *   k, v : [S][L][Hkv][T][d]     (pre-RoPE keys; values)
 * q/k/v must not alias o or handle memory.  Returns E_CAPACITY when
 * n == max_frames.  On success the frame index advances by one.
 */
int statekv_prefill_frame(statekv_handle* h, const void* q, const void* k,
                          const void* v, void* o, void* cuda_stream);

/*
 * Same step with HOST buffers (same layouts): copies q/k/v into the handle's
 * device staging, runs the step and copies o back, all enqueued on
 * cuda_stream.  Host buffers should be page-locked for the copies to be
 * asynchronous; they must stay valid and unmodified until the stream passes
 * the call.
 */
int statekv_prefill_frame_host(statekv_handle* h, const void* q_host,
                               const void* k_host, const void* v_host,
                               void* o_host, void* cuda_stream);

/*
 * `frames` consecutive steps from HOST buffers holding the frames back to
 * back (frame-major, each frame in the layouts above):
 *   q, o : [frames][S][L][Hq][T][d]      k, v : [frames][S][L][Hkv][T][d]
 * The same computation as `frames` calls of statekv_prefill_frame_host, but
 * the copies overlap the device work: the handle holds two staging slots,
 * and on side streams of its own (four per direction, each copying a quarter
 * of a frame's bytes) it copies frame i+1 in and frame i-1 out while frame i
 * runs on cuda_stream.  The whole batch is ordered on
 * cuda_stream like a single call: the side streams first wait for the work
 * already enqueued there, and cuda_stream waits for the last copy out, so
 * every o frame is valid (and q/k/v may be reused) once the stream passes
 * the call.  Host buffers should be page-locked.  Returns E_CAPACITY, with
 * nothing done, when n + frames > max_frames; frames == 0 is a no-op.  The
 * side streams and events are created on the first call (E_CUDA if that
 * fails); a handle's calls must not overlap with each other.
 * This entry point has no counterpart in the page; it streams a video from
 * host memory at device speed.
 */
int statekv_prefill_frames_host(statekv_handle* h, int32_t frames, const void* q_host,
                                const void* k_host, const void* v_host, void* o_host,
                                void* cuda_stream);

/*
 * Text decode over the detailed state (关键设计 1: D_n keeps every frame's
 * K/V for text decoding; 关键设计 3: text continues the virtual positions
 * with the same static scale).  `tokens` new text tokens (1..16, and at most
 * T) take positions p = position_offset + n*T + j, j counting every text
 * token decoded since the last frame; their K', V are appended to D after
 * the rows already there, and each query row attends over all earlier D rows
 * (the whole video and earlier text) and, causally, over the new tokens:
 *   O = softmax(Q' [D_K]^T * mscale^2/sqrt(d), causal on the new rows) D_V.
 * Device pointers, contiguous, storage dtype:
 *   q, o : [S][L][Hq][tokens][d]     k, v : [S][L][Hkv][tokens][d] (pre-RoPE)
 * Supported: bf16 storage, d = 128, G*tokens <= 64 (else E_UNSUPPORTED).
 * Returns E_CAPACITY (nothing done) when the new rows do not fit in D
 * (n*T + decoded + tokens > max_frames*T).  Once a handle has decoded text,
 * the prefill entry points return E_INVALID_ARG until statekv_reset.  The
 * first call allocates the handle's decode scratch (partial results per
 * 2048-key chunk of D; E_OOM if that fails).
 */
int statekv_decode(statekv_handle* h, int32_t tokens, const void* q, const void* k,
                   const void* v, void* o, void* cuda_stream);

/* Text tokens decoded since the last reset (-1 for a NULL handle). */
int64_t statekv_text_tokens(const statekv_handle* h);

/*
 * Borrowed DEVICE pointers to the compressed state C_{n-1} of (stream s,
 * layer) after the last step: k, v -> [Hkv][pitch][d], pos -> [Hkv][pitch]
 * int32 virtual positions; the first *count slots of each head are live
 * (count = min(B, n*T)), in slot order.  *pitch = B + T.  Valid until the
 * next call that changes the handle.  Any output pointer may be NULL.
 */
int statekv_get_compressed(statekv_handle* h, int32_t s, int32_t layer,
                           const void** k, const void** v, const int32_t** pos,
                           int32_t* count, int32_t* pitch);

/*
 * Borrowed DEVICE pointers to the detailed state D_{n-1} of (s, layer):
 * k, v -> [Hkv][pitch][d] with row r = virtual position r - position_offset
 * (post-RoPE K, V as given); *count = n*T (+ decoded text tokens) live rows per head,
 * *pitch = max_frames*T.  Any output pointer may be NULL.
 */
int statekv_get_detailed(statekv_handle* h, int32_t s, int32_t layer,
                         const void** k, const void** v, int64_t* count,
                         int64_t* pitch);

/* Frames processed so far (n). */
int64_t statekv_frame_index(const statekv_handle* h);

/* Forget all frames: n = 0, c = 0 (allocations kept, contents stale). */
int statekv_reset(statekv_handle* h);

/*
 * Synchronise cuda_stream, then report and clear the device status word:
 * STATEKV_OK, STATEKV_E_TIMEOUT (a bounded wait inside a kernel gave up; that
 * launch's outputs are invalid) or STATEKV_E_DEVICE.
 */
int statekv_check_device_status(statekv_handle* h, void* cuda_stream);

/* ------------------------------------------------------------- test hooks */

/*
 * Importance scores of the last step (关键设计 2) for (s, layer):
 * scores -> [Hkv][pitch] fp32, pool_pos -> [Hkv][pitch] int32, both in pool
 * slot order before the Top-B update (slots [0,c) held C_{n-1}, slots
 * [c, c+T) the frame's tokens); *m = c + T candidates.  Borrowed DEVICE
 * pointers, valid until the next step.
 */
int statekv_get_scores(statekv_handle* h, int32_t s, int32_t layer,
                       const float** scores, const int32_t** pool_pos,
                       int32_t* m, int32_t* pitch);

/* Borrowed DEVICE pointer to the rotated queries Q' of the last frame step
 * ([S][L][Hq][T][d], storage dtype) or, after a text decode, of the last
 * decode step ([S][L][Hq][tokens][d]).  Valid until the next step. */
int statekv_get_rotated_query(statekv_handle* h, const void** q_rot);

/* Set the frame index n (teacher forcing / resume); 0 <= n < max_frames. */
int statekv_set_frame_index(statekv_handle* h, int64_t n);

/*
 * Teacher forcing / resume: overwrite C of (s, layer) with count rows per KV
 * head from DEVICE buffers k, v [Hkv][count][d] (post-RoPE, storage dtype)
 * and pos [Hkv][count] int32.  count must equal min(B, n*T) for the current
 * frame index n.  Copies are enqueued on cuda_stream.
 */
int statekv_set_compressed(statekv_handle* h, int32_t s, int32_t layer,
                           const void* k, const void* v, const int32_t* pos,
                           int32_t count, void* cuda_stream);

/*
 * Per-kernel timing with CUDA events recorded on the launch stream around
 * every launch while enabled.  statekv_profile_read synchronises, then
 * returns for kernel id (STATEKV_KERNEL_*) the summed device milliseconds
 * and the number of launches since profiling was last enabled.
 * statekv_profile_kernels restricts the bracketing to the kernels whose bit
 * (1 << STATEKV_KERNEL_*) is set in mask (default: all).  An event recorded
 * between two launches also ends the overlap of the second launch's start
 * with the first one's end (below), so timing only the kernel of interest
 * keeps the others' overlap.
 *
 * Overlap of consecutive launches within a frame sequence: the RoPE kernel
 * of frame n+1 starts while the selection of frame n still runs (its query
 * rows do not depend on it; its writes of the frame's keys into the pool
 * wait for the selection to finish), the attention kernel's set-up
 * overlaps the RoPE kernel's end, and the selection is launched while the
 * attention kernel still runs and starts work as soon as it has finished
 * (programmatic dependent launch).  Any other
 * operation on the stream between two calls separates them as usual.
 */
int statekv_profile_enable(statekv_handle* h, int enable);
int statekv_profile_kernels(statekv_handle* h, uint32_t mask);
int statekv_profile_read(statekv_handle* h, int32_t kernel, double* total_ms,
                         int64_t* launches);

/* ------------------------------------------------- allocation-free entry */

/*
 * No counterpart in the paper: a deployment convenience.
 *
 * Frame attention and importance scores for callers that cannot allocate
 * device memory -- whose memory is owned by another allocator (an inference
 * server's pool, a framework hosting this library as a plugin) or that must
 * avoid the device-wide synchronisation cudaMalloc/cudaFree can cause.  It
 * creates no handle and calls no cudaMalloc, cudaFree or other allocating
 * routine; its only scratch (the per-query-tile column sums of P) is a
 * file-scope 16 MiB __device__ array that every GPU loading this library
 * holds until the process exits.
 *
 * Computes, per unit u (one KV head of one layer and stream), exactly the
 * attention and scores of one statekv_prefill_frame step:
 *   o      = softmax(q_rot pool_k^T * logit_scale, masked) pool_v
 *   scores = s_j, the mean over the group*frame_tokens query rows of P[:, j]
 * where pool rows [0, compressed) are compressed keys (visible to every
 * query) and rows [compressed, compressed + frame_tokens) are the frame's
 * keys in token order (frame key i' visible to query token i iff i' <= i).
 * DEVICE pointers on the current device, caller-owned, contiguous, storage
 * dtype (STATEKV_BF16 or STATEKV_F32), 16-byte aligned:
 *   q_rot  [units][group * frame_tokens][head_dim]  rotated queries, g-major
 *   pool_k, pool_v [units][pool_rows][head_dim]     pool_rows >= compressed + frame_tokens
 *   o      [units][group * frame_tokens][head_dim]  written
 *   scores [units][compressed + frame_tokens] fp32  written
 *   status uint32[4] device status word, required (4-byte aligned): the
 *          call first zeroes it on cuda_stream; a bounded device wait that
 *          gives up then writes STATEKV_E_TIMEOUT into status[0] (the wait
 *          site into status[1]) and leaves o and scores unspecified.  Read
 *          it once the stream has passed the call.
 * logit_scale = mscale^2 / sqrt(head_dim).  Returns STATEKV_E_CAPACITY when
 * units * ceil(group*frame_tokens / R) * round_up(pool_rows, 128) * 4 bytes
 * exceeds the 16 MiB scratch (R = 128 query rows per tile for bf16, 16 for
 * fp32), STATEKV_E_UNSUPPORTED for head_dim not in {64, 128}.
 * The first call on a device takes the scratch's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls on a device share the scratch:
 * calls that overlap on the GPU race and must be serialised by the caller.
 * Work is enqueued on cuda_stream; results are valid once it passes the call.
 */
int statekv_attend_scores_static(const void* q_rot, const void* pool_k,
                                 const void* pool_v, int32_t units,
                                 int32_t group, int32_t frame_tokens,
                                 int32_t head_dim, int32_t pool_rows,
                                 int32_t compressed, double logit_scale,
                                 int32_t dtype, void* o, float* scores,
                                 uint32_t* status, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* STATEKV_H_ */
