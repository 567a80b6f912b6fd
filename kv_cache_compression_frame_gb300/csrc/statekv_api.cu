// libstatekv C ABI: handle lifetime, argument checks, device memory layout,
// TMA descriptors and the per-frame launch sequence.
//
// StateKV ("Linear Scaling Video VLMs for Long Video Understanding"),
// 方法详解 / 整体框架 and 关键设计 1-3.  Per frame step n, on the caller's stream:
//   rope (+ D append, pool insert) -> attention (+ column sums)
//   -> select (scores, Top-B, slot-reuse gather);
// the cos/sin table of every position D can hold is built once, at create.
// Device memory per unit u = (stream, layer, KV head), all allocated at
// create:
//   pool K/V   [U][B+T][d]      compressed slots [0, c) then the frame's rows
//   pool pos   [U][B+T] int32   virtual positions of the compressed slots
//   D K/V      [U][N_max*T][d]  row r = virtual position r - offset
//   Q'         [U*G*T][d]       rotated queries (scratch)
//   colsum     [U][tiles][m_pad] per query-tile column sums of P
//   scores     [U][m_pad], score_pos [U][m_pad]
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "statekv_internal.cuh"

using namespace statekv;

namespace {

// copy streams per direction of the batched host entry point
constexpr int kCopyWays = 4;

struct PendingEvent {
    int kernel;
    cudaEvent_t start, stop;
};

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() { if (prev >= 0) cudaSetDevice(prev); }
};

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// A failed CUDA call: clear the runtime's last-error state (a refused launch,
// for instance, would otherwise be reported again by the next call that
// checks it, in this library or the caller's code) and report E_CUDA.
int cuda_fail() {
    cudaGetLastError();
    return STATEKV_E_CUDA;
}

}  // namespace

struct statekv_handle {
    statekv_config cfg{};
    int64_t n = 0;                      // frames processed
    int64_t text = 0;                   // text tokens decoded after frame n-1
    int num_sms = 0;
    float* dec_m = nullptr; float* dec_l = nullptr; float* dec_o = nullptr;  // decode partials
    int64_t dec_items = 0;              // capacity of the partials (items)
    int G = 0, U = 0, GT = 0, slots = 0, m_pad = 0, n_row_tiles = 0, esize = 0;
    int64_t det_pitch = 0;
    double mscale = 1.0;
    float scale = 0.f, scale_log2 = 0.f;

    double* omega = nullptr;            // [d/2]
    float2* cs = nullptr;               // [det_pitch][d/2] cos/sin of every D row's position
    void* pool_k = nullptr; void* pool_v = nullptr;
    int32_t* pos = nullptr;
    void* det_k = nullptr; void* det_v = nullptr;
    void* q_rot = nullptr;
    float* colsum = nullptr;
    float* scores = nullptr;
    int32_t* score_pos = nullptr;
    uint32_t* err = nullptr;            // device status word
    void* stage_q = nullptr; void* stage_k = nullptr; void* stage_v = nullptr; void* stage_o = nullptr;
    // second staging slot and the side streams / events of the batched host
    // entry point (streams and events are created on its first call)
    void* stage2_q = nullptr; void* stage2_k = nullptr; void* stage2_v = nullptr;
    void* stage2_o = nullptr;
    // kCopyWays copy streams per direction: one copy stream moved ~100 GB/s,
    // less than a frame's inputs per frame time need
    cudaStream_t s_in[kCopyWays] = {}, s_out[kCopyWays] = {};
    cudaEvent_t ev_entry = nullptr, ev_in[2][kCopyWays] = {}, ev_front[2] = {},
                ev_out[2][kCopyWays] = {};
    TcMaps tc{};                        // TMA views for the bf16 attention kernel

    bool profiling = false;
    uint32_t prof_mask = 0xffffffffu;   // kernels bracketed while profiling
    std::vector<PendingEvent> pending;
    std::vector<cudaEvent_t> spare;
    double prof_ms[STATEKV_NUM_KERNELS] = {0, 0, 0, 0};
    int64_t prof_n[STATEKV_NUM_KERNELS] = {0, 0, 0, 0};
    std::vector<void*> allocs;

    size_t q_bytes() const {
        return (size_t)cfg.num_streams * cfg.num_layers * cfg.num_q_heads * cfg.frame_tokens *
               cfg.head_dim * esize;
    }
    size_t kv_bytes() const {
        return (size_t)cfg.num_streams * cfg.num_layers * cfg.num_kv_heads * cfg.frame_tokens *
               cfg.head_dim * esize;
    }
    int c() const { return (int)std::min<int64_t>(cfg.budget, n * cfg.frame_tokens); }
};

namespace {

void destroy_pipeline(statekv_handle* h) {
    for (cudaEvent_t* e : {&h->ev_entry, &h->ev_front[0], &h->ev_front[1]})
        if (*e) { cudaEventDestroy(*e); *e = nullptr; }
    for (int sl = 0; sl < 2; ++sl)
        for (int j = 0; j < kCopyWays; ++j)
            for (cudaEvent_t* e : {&h->ev_in[sl][j], &h->ev_out[sl][j]})
                if (*e) { cudaEventDestroy(*e); *e = nullptr; }
    for (int j = 0; j < kCopyWays; ++j)
        for (cudaStream_t* st : {&h->s_in[j], &h->s_out[j]})
            if (*st) { cudaStreamDestroy(*st); *st = nullptr; }
}

void free_all(statekv_handle* h) {
    for (void* p : h->allocs) cudaFree(p);
    h->allocs.clear();
    for (auto& e : h->pending) { cudaEventDestroy(e.start); cudaEventDestroy(e.stop); }
    for (auto e : h->spare) cudaEventDestroy(e);
    h->pending.clear();
    h->spare.clear();
    destroy_pipeline(h);
}

template <typename T>
bool dalloc(statekv_handle* h, T** p, size_t bytes) {
    void* q = nullptr;
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(&q, bytes) != cudaSuccess) { cudaGetLastError(); return false; }
    if (cudaMemset(q, 0, bytes) != cudaSuccess) { cudaGetLastError(); cudaFree(q); return false; }
    h->allocs.push_back(q);
    *p = reinterpret_cast<T*>(q);
    return true;
}

int validate(const statekv_config* c) {
    if (!c) return STATEKV_E_INVALID_ARG;
    if (c->num_streams < 1 || c->num_layers < 1 || c->num_kv_heads < 1 || c->num_q_heads < 1 ||
        c->frame_tokens < 1 || c->budget < 0 || c->max_frames < 1 || c->device < 0)
        return STATEKV_E_INVALID_ARG;
    if (c->num_q_heads % c->num_kv_heads != 0) return STATEKV_E_INVALID_ARG;
    if (c->dtype != STATEKV_BF16 && c->dtype != STATEKV_F32) return STATEKV_E_INVALID_ARG;
    if (!(c->rope_theta > 1.0) || !(c->rope_alpha >= 1.0) || !std::isfinite(c->rope_theta) ||
        !std::isfinite(c->rope_alpha))
        return STATEKV_E_INVALID_ARG;
    if (c->rope_alpha != 1.0 && c->rope_orig_ctx <= 0) return STATEKV_E_INVALID_ARG;
    if (c->position_offset < 0) return STATEKV_E_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128) return STATEKV_E_UNSUPPORTED;
    int64_t G = c->num_q_heads / c->num_kv_heads;
    if (G * c->frame_tokens > 65536) return STATEKV_E_UNSUPPORTED;
    if (c->select_policy != STATEKV_SELECT_TOPB && c->select_policy != STATEKV_SELECT_WINDOW)
        return STATEKV_E_INVALID_ARG;
    // selection keeps the pool's keys in shared memory; a handle whose budget
    // covers every frame it can hold never selects (full self-attention)
    const bool never_evicts = (int64_t)c->budget >= (int64_t)c->max_frames * c->frame_tokens;
    if (!never_evicts && ((int64_t)c->budget + c->frame_tokens > kMaxSlots ||
                          select_smem_bytes(c->budget + c->frame_tokens, c->frame_tokens) >
                              kSelectSmemMax))
        return STATEKV_E_UNSUPPORTED;
    if ((int64_t)c->budget + c->frame_tokens > (1LL << 24)) return STATEKV_E_UNSUPPORTED;
    if (c->position_offset + (int64_t)c->max_frames * c->frame_tokens > 0x7fffffffLL)
        return STATEKV_E_UNSUPPORTED;
    int64_t units = (int64_t)c->num_streams * c->num_layers * c->num_kv_heads;
    if (units * G * c->frame_tokens > 0x7fffffffLL || units > 0x7fffffffLL / 1024)
        return STATEKV_E_UNSUPPORTED;
    return STATEKV_OK;
}

// Frequencies omega_k of the rotated pairs, and the logit temperature
// factor.  Plain RoPE omega_k = theta^(-2k/d); a static scale alpha != 1 uses
// YaRN's NTK-by-parts rule: r_k = L_orig * omega_k / (2 pi), ramp
// g_k = clamp((r_k - 1) / 31, 0, 1), omega'_k = (1 - g_k) omega_k / alpha +
// g_k omega_k, mscale = 0.1 ln(alpha) + 1.
void rope_frequencies(const statekv_config& c, std::vector<double>& om, double& mscale) {
    const int half = c.head_dim / 2;
    om.resize(half);
    for (int k = 0; k < half; ++k) {
        double w = std::pow(c.rope_theta, -2.0 * k / c.head_dim);
        if (c.rope_alpha != 1.0) {
            double r = (double)c.rope_orig_ctx * w / (2.0 * M_PI);
            double g = std::min(1.0, std::max(0.0, (r - 1.0) / 31.0));
            w = (1.0 - g) * w / c.rope_alpha + g * w;
        }
        om[k] = w;
    }
    mscale = c.rope_alpha == 1.0 ? 1.0 : 0.1 * std::log(c.rope_alpha) + 1.0;
}

// An event from the spare list or a new one; nullptr if none can be made.
cudaEvent_t take_event(statekv_handle* h) {
    if (!h->spare.empty()) { cudaEvent_t e = h->spare.back(); h->spare.pop_back(); return e; }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    return e;
}

// Runs one launch, bracketed by events when profiling (a launch whose events
// cannot be made or recorded runs unbracketed and is not counted).
template <typename F>
cudaError_t timed(statekv_handle* h, int kernel, cudaStream_t st, F&& launch) {
    if (!h->profiling || !((h->prof_mask >> kernel) & 1u)) return launch();
    PendingEvent pe{kernel, take_event(h), take_event(h)};
    if (!pe.start || !pe.stop || cudaEventRecord(pe.start, st) != cudaSuccess) {
        cudaGetLastError();
        for (cudaEvent_t ev : {pe.start, pe.stop})
            if (ev) h->spare.push_back(ev);
        return launch();
    }
    cudaError_t e = launch();
    if (cudaEventRecord(pe.stop, st) != cudaSuccess) {
        cudaGetLastError();
        h->spare.push_back(pe.start);
        h->spare.push_back(pe.stop);
        return e;
    }
    h->pending.push_back(pe);
    return e;
}

int check_ptr(const void* p) {
    if (!p) return STATEKV_E_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p) % 16) return STATEKV_E_INVALID_ARG;
    return STATEKV_OK;
}

// One frame step in two halves: RoPE + attention (reads q, k, v, writes o),
// then the selection.  A caller may put waits between the halves: there they
// cost only the selection's early launch (its CTAs then start when the wait
// is over instead of waiting on the GPU for the attention kernel), while
// between the selection and the next frame's RoPE they would end the overlap
// of the two (programmatic dependent launch).
int run_front(statekv_handle* h, const void* q, const void* k, const void* v, void* o,
              cudaStream_t st) {
    const statekv_config& c = h->cfg;
    const int T = c.frame_tokens, d = c.head_dim;
    const int cc = h->c();
    const int64_t p0 = c.position_offset + h->n * T;
    cudaError_t e;

    RopeArgs ra{};
    ra.q = q; ra.k = k; ra.v = v;
    ra.q_rot = h->q_rot; ra.pool_k = h->pool_k; ra.pool_v = h->pool_v;
    ra.det_k = h->det_k; ra.det_v = h->det_v;
    ra.cs = h->cs + (size_t)h->n * T * (d / 2);          // rows of this frame's positions
    ra.rows_q = (int64_t)h->U * h->GT;
    ra.rows_kv = (int64_t)h->U * T;
    ra.T = T; ra.d = d; ra.slots = h->slots; ra.c = cc;
    ra.det_pitch = h->det_pitch; ra.det_row0 = h->n * T;
    e = timed(h, STATEKV_KERNEL_ROPE, st, [&] { return launch_rope(ra, c.dtype, st, true); });
    if (e != cudaSuccess) return cuda_fail();

    AttnArgs aa{};
    aa.q_rot = h->q_rot; aa.pool_k = h->pool_k; aa.pool_v = h->pool_v; aa.o = o;
    aa.colsum = h->colsum; aa.err = h->err;
    aa.U = h->U; aa.GT = h->GT; aa.T = T; aa.d = d; aa.slots = h->slots; aa.c = cc;
    aa.m_pad = h->m_pad; aa.n_row_tiles = h->n_row_tiles;
    aa.scale = h->scale; aa.scale_log2 = h->scale_log2;
    aa.resident = h->num_sms;                            // one attention CTA per SM
    e = timed(h, STATEKV_KERNEL_ATTENTION, st, [&] {
        return c.dtype == STATEKV_BF16 ? launch_attention_tc(aa, h->tc, st)
                                       : launch_attention_simt(aa, st);
    });
    if (e != cudaSuccess) return cuda_fail();
    return STATEKV_OK;
}

int run_back(statekv_handle* h, cudaStream_t st) {
    const statekv_config& c = h->cfg;
    const int T = c.frame_tokens, d = c.head_dim;
    const int cc = h->c();
    const int64_t p0 = c.position_offset + h->n * T;
    SelectArgs sa{};
    sa.colsum = h->colsum; sa.scores = h->scores; sa.score_pos = h->score_pos;
    sa.pos = h->pos; sa.pool_k = h->pool_k; sa.pool_v = h->pool_v; sa.err = h->err;
    sa.U = h->U; sa.n_row_tiles = h->n_row_tiles; sa.m_pad = h->m_pad; sa.slots = h->slots;
    sa.c = cc; sa.T = T; sa.B = c.budget; sa.row_bytes = d * h->esize;
    sa.pos_base = (int32_t)p0;
    sa.inv_rows = (float)(1.0 / ((double)h->G * T));
    sa.window = c.select_policy == STATEKV_SELECT_WINDOW;
    sa.never_evicts = (int64_t)c.budget >= (int64_t)c.max_frames * T;
    sa.num_sms = h->num_sms;
    cudaError_t e = timed(h, STATEKV_KERNEL_SELECT, st, [&] { return launch_select(sa, st); });
    if (e != cudaSuccess) return cuda_fail();

    h->n += 1;
    return STATEKV_OK;
}

int run_frame(statekv_handle* h, const void* q, const void* k, const void* v, void* o,
              cudaStream_t st) {
    const int r = run_front(h, q, k, v, o, st);
    return r != STATEKV_OK ? r : run_back(h, st);
}

}  // namespace

extern "C" {

const char* statekv_status_string(int s) {
    switch (s) {
        case STATEKV_OK: return "ok";
        case STATEKV_E_INVALID_ARG: return "invalid argument";
        case STATEKV_E_UNSUPPORTED: return "unsupported configuration";
        case STATEKV_E_CAPACITY: return "detailed state is full (n == max_frames)";
        case STATEKV_E_OOM: return "device allocation failed";
        case STATEKV_E_CUDA: return "CUDA call failed";
        case STATEKV_E_TIMEOUT: return "device-side bounded wait timed out";
        case STATEKV_E_DEVICE: return "device-side consistency check failed";
        default: return "unknown status";
    }
}

int statekv_create(const statekv_config* cfg, statekv_handle** out) {
    if (!out) return STATEKV_E_INVALID_ARG;
    *out = nullptr;
    int v = validate(cfg);
    if (v != STATEKV_OK) return v;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return cuda_fail();
    if (cfg->device >= ndev) return STATEKV_E_INVALID_ARG;
    DeviceGuard g(cfg->device);
    if (!g.ok) return cuda_fail();

    statekv_handle* h = new (std::nothrow) statekv_handle();
    if (!h) return STATEKV_E_OOM;
    h->cfg = *cfg;
    const statekv_config& c = h->cfg;
    h->G = c.num_q_heads / c.num_kv_heads;
    h->U = c.num_streams * c.num_layers * c.num_kv_heads;
    h->GT = h->G * c.frame_tokens;
    h->slots = c.budget + c.frame_tokens;
    h->m_pad = (int)round_up(h->slots, 128);
    h->esize = c.dtype == STATEKV_BF16 ? 2 : 4;
    const int row_tile = c.dtype == STATEKV_BF16 ? kTcRowTile : kSimtRowTile;
    h->n_row_tiles = (h->GT + row_tile - 1) / row_tile;
    h->det_pitch = (int64_t)c.max_frames * c.frame_tokens;

    std::vector<double> om;
    rope_frequencies(c, om, h->mscale);
    const double scale = h->mscale * h->mscale / std::sqrt((double)c.head_dim);
    h->scale = (float)scale;
    h->scale_log2 = (float)(scale * 1.4426950408889634074);

    const int d = c.head_dim, T = c.frame_tokens;
    const size_t row = (size_t)d * h->esize;
    bool ok = true;
    ok = ok && dalloc(h, &h->omega, sizeof(double) * d / 2);
    ok = ok && dalloc(h, &h->cs, sizeof(float2) * (size_t)h->det_pitch * d / 2);
    ok = ok && dalloc(h, &h->pool_k, (size_t)h->U * h->slots * row);
    ok = ok && dalloc(h, &h->pool_v, (size_t)h->U * h->slots * row);
    ok = ok && dalloc(h, &h->pos, sizeof(int32_t) * (size_t)h->U * h->slots);
    ok = ok && dalloc(h, &h->det_k, (size_t)h->U * h->det_pitch * row);
    ok = ok && dalloc(h, &h->det_v, (size_t)h->U * h->det_pitch * row);
    ok = ok && dalloc(h, &h->q_rot, (size_t)h->U * h->GT * row);
    ok = ok && dalloc(h, &h->colsum, sizeof(float) * (size_t)h->U * h->n_row_tiles * h->m_pad);
    ok = ok && dalloc(h, &h->scores, sizeof(float) * (size_t)h->U * h->m_pad);
    ok = ok && dalloc(h, &h->score_pos, sizeof(int32_t) * (size_t)h->U * h->m_pad);
    ok = ok && dalloc(h, &h->err, sizeof(uint32_t) * kErrWords);
    ok = ok && dalloc(h, &h->stage_q, h->q_bytes());
    ok = ok && dalloc(h, &h->stage_k, h->kv_bytes());
    ok = ok && dalloc(h, &h->stage_v, h->kv_bytes());
    ok = ok && dalloc(h, &h->stage_o, h->q_bytes());
    ok = ok && dalloc(h, &h->stage2_q, h->q_bytes());
    ok = ok && dalloc(h, &h->stage2_k, h->kv_bytes());
    ok = ok && dalloc(h, &h->stage2_v, h->kv_bytes());
    ok = ok && dalloc(h, &h->stage2_o, h->q_bytes());
    if (!ok) { free_all(h); delete h; return STATEKV_E_OOM; }
    if (cudaMemcpy(h->omega, om.data(), sizeof(double) * om.size(), cudaMemcpyHostToDevice) !=
        cudaSuccess) {
        free_all(h); delete h; return cuda_fail();
    }
    // the rotation of every position D can hold (frames and decoded text),
    // computed once: D row r is at virtual position position_offset + r
    {
        RopeTableArgs ta{h->omega, h->cs, c.position_offset, (int32_t)h->det_pitch, d / 2,
                         c.dtype == STATEKV_BF16 ? 8 : 4};
        if (launch_rope_table(ta, nullptr) != cudaSuccess) { free_all(h); delete h; return cuda_fail(); }
    }
    if (c.dtype == STATEKV_BF16 &&
        !make_tc_maps(&h->tc, h->pool_k, h->pool_v, d, h->slots, h->U)) {
        free_all(h); delete h; return cuda_fail();
    }
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, c.device) !=
        cudaSuccess) {
        free_all(h); delete h; return cuda_fail();
    }
    if (cudaDeviceSynchronize() != cudaSuccess) { free_all(h); delete h; return cuda_fail(); }
    *out = h;
    return STATEKV_OK;
}

int statekv_destroy(statekv_handle* h) {
    if (!h) return STATEKV_OK;
    DeviceGuard g(h->cfg.device);
    cudaDeviceSynchronize();
    free_all(h);
    delete h;
    return STATEKV_OK;
}

int statekv_prefill_frame(statekv_handle* h, const void* q, const void* k, const void* v,
                          void* o, void* cuda_stream) {
    if (!h) return STATEKV_E_INVALID_ARG;
    int r;
    if ((r = check_ptr(q)) || (r = check_ptr(k)) || (r = check_ptr(v)) || (r = check_ptr(o)))
        return r;
    if (h->text > 0) return STATEKV_E_INVALID_ARG;   // decoding has started: reset first
    if (h->n >= h->cfg.max_frames) return STATEKV_E_CAPACITY;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return cuda_fail();
    return run_frame(h, q, k, v, o, reinterpret_cast<cudaStream_t>(cuda_stream));
}

int statekv_prefill_frame_host(statekv_handle* h, const void* q, const void* k, const void* v,
                               void* o, void* cuda_stream) {
    if (!h || !q || !k || !v || !o || h->text > 0) return STATEKV_E_INVALID_ARG;
    if (h->n >= h->cfg.max_frames) return STATEKV_E_CAPACITY;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return cuda_fail();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (cudaMemcpyAsync(h->stage_q, q, h->q_bytes(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(h->stage_k, k, h->kv_bytes(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaMemcpyAsync(h->stage_v, v, h->kv_bytes(), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return cuda_fail();
    int r = run_frame(h, h->stage_q, h->stage_k, h->stage_v, h->stage_o, st);
    if (r != STATEKV_OK) return r;
    if (cudaMemcpyAsync(o, h->stage_o, h->q_bytes(), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return cuda_fail();
    return STATEKV_OK;
}

namespace {

bool ensure_pipeline(statekv_handle* h) {
    if (h->s_in[0]) return true;
    bool ok = true;
    for (int j = 0; j < kCopyWays; ++j)
        for (cudaStream_t* st : {&h->s_in[j], &h->s_out[j]})
            ok = ok && cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* e : {&h->ev_entry, &h->ev_front[0], &h->ev_front[1]})
        ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    for (int sl = 0; sl < 2; ++sl)
        for (int j = 0; j < kCopyWays; ++j)
            for (cudaEvent_t* e : {&h->ev_in[sl][j], &h->ev_out[sl][j]})
                ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        destroy_pipeline(h);
        cudaGetLastError();
    }
    return ok;
}

}  // namespace

// Frames i = 0..F-1, staging slot i & 1.  Each direction's bytes of a frame
// are cut into kCopyWays equal ranges (256-byte aligned), one per stream j:
//   s_in[j] : [wait front(i-2)] H2D range j of q|k|v(i) -> slot  record ev_in[slot][j]
//   st      : front(i) (RoPE, attention)                         record ev_front[slot]
//   s_out[j]: wait ev_front[slot]  D2H range j of o(i) <- slot    record ev_out[slot][j]
//   st      : wait ev_in[next slot][*], [wait ev_out[next slot][*] of frame i-1],
//             back(i) (selection)
// so the copies of frames i+1 (in) and i (out) overlap the step of frame
// i, and the waits sit between the attention and the selection, never
// between the selection and the next frame's RoPE.  The side streams first
// wait for everything already on st; at the end st waits for the last
// copies, so the batch is ordered on st like one call.
int statekv_prefill_frames_host(statekv_handle* h, int32_t frames, const void* q, const void* k,
                                const void* v, void* o, void* cuda_stream) {
    if (!h || frames < 0 || !q || !k || !v || !o || h->text > 0) return STATEKV_E_INVALID_ARG;
    if (frames == 0) return STATEKV_OK;
    if (h->n + frames > h->cfg.max_frames) return STATEKV_E_CAPACITY;
    DeviceGuard g(h->cfg.device);
    if (!g.ok) return cuda_fail();
    if (!ensure_pipeline(h)) return cuda_fail();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    const size_t qb = h->q_bytes(), kvb = h->kv_bytes();
    void* sq[2] = {h->stage_q, h->stage2_q};
    void* sk[2] = {h->stage_k, h->stage2_k};
    void* sv[2] = {h->stage_v, h->stage2_v};
    void* so[2] = {h->stage_o, h->stage2_o};
    // range j of n bytes: [cut(n, j), cut(n, j + 1))
    auto cut = [](size_t n, int j) {
        return j >= kCopyWays ? n : std::min(n, (n * (size_t)j / kCopyWays + 255) / 256 * 256);
    };
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    if (!ok(cudaEventRecord(h->ev_entry, st))) return cuda_fail();
    for (int j = 0; j < kCopyWays; ++j)
        if (!ok(cudaStreamWaitEvent(h->s_in[j], h->ev_entry, 0)) ||
            !ok(cudaStreamWaitEvent(h->s_out[j], h->ev_entry, 0)))
            return cuda_fail();
    auto h2d = [&](int32_t i) -> bool {
        const int sl = i & 1;
        // the frame's inputs as one byte range [0, qb + 2 kvb): q, then k, then v
        const char* src[3] = {static_cast<const char*>(q) + (size_t)i * qb,
                              static_cast<const char*>(k) + (size_t)i * kvb,
                              static_cast<const char*>(v) + (size_t)i * kvb};
        char* dst[3] = {static_cast<char*>(sq[sl]), static_cast<char*>(sk[sl]),
                        static_cast<char*>(sv[sl])};
        const size_t off[4] = {0, qb, qb + kvb, qb + 2 * kvb};
        for (int j = 0; j < kCopyWays; ++j) {
            if (i >= 2 && !ok(cudaStreamWaitEvent(h->s_in[j], h->ev_front[sl], 0))) return false;
            const size_t lo = cut(off[3], j), hi = cut(off[3], j + 1);
            for (int t = 0; t < 3; ++t) {
                const size_t a = std::max(lo, off[t]), b = std::min(hi, off[t + 1]);
                if (b > a && !ok(cudaMemcpyAsync(dst[t] + (a - off[t]), src[t] + (a - off[t]), b - a,
                                                 cudaMemcpyHostToDevice, h->s_in[j])))
                    return false;
            }
            if (!ok(cudaEventRecord(h->ev_in[sl][j], h->s_in[j])) ||
                !ok(cudaStreamWaitEvent(st, h->ev_in[sl][j], 0)))
                return false;
        }
        return true;
    };
    if (!h2d(0)) return cuda_fail();
    for (int32_t i = 0; i < frames; ++i) {
        const int sl = i & 1;
        int r = run_front(h, sq[sl], sk[sl], sv[sl], so[sl], st);
        if (r != STATEKV_OK) return r;
        if (!ok(cudaEventRecord(h->ev_front[sl], st))) return cuda_fail();
        char* oi = static_cast<char*>(o) + (size_t)i * qb;
        const char* ds = static_cast<const char*>(so[sl]);
        for (int j = 0; j < kCopyWays; ++j) {
            const size_t b0 = cut(qb, j), b1 = cut(qb, j + 1);
            if (!ok(cudaStreamWaitEvent(h->s_out[j], h->ev_front[sl], 0)) ||
                (b1 > b0 && !ok(cudaMemcpyAsync(oi + b0, ds + b0, b1 - b0, cudaMemcpyDeviceToHost,
                                                h->s_out[j]))) ||
                !ok(cudaEventRecord(h->ev_out[sl][j], h->s_out[j])))
                return cuda_fail();
        }
        if (i + 1 < frames) {
            if (!h2d(i + 1)) return cuda_fail();
            // attention(i+1) rewrites the output slot of frame i-1
            for (int j = 0; j < kCopyWays; ++j)
                if (i >= 1 && !ok(cudaStreamWaitEvent(st, h->ev_out[(i + 1) & 1][j], 0)))
                    return cuda_fail();
        }
        r = run_back(h, st);
        if (r != STATEKV_OK) return r;
    }
    for (int s2 = 0; s2 < 2 && s2 < frames; ++s2)
        for (int j = 0; j < kCopyWays; ++j)
            if (!ok(cudaStreamWaitEvent(st, h->ev_out[(frames - 1 - s2) & 1][j], 0)))
                return cuda_fail();
    return STATEKV_OK;
}

int statekv_decode(statekv_handle* h, int32_t tokens, const void* q, const void* k, const void* v,
                   void* o, void* cuda_stream) {
    if (!h) return STATEKV_E_INVALID_ARG;
    int r;
    if ((r = check_ptr(q)) || (r = check_ptr(k)) || (r = check_ptr(v)) || (r = check_ptr(o)))
        return r;
    const statekv_config& c = h->cfg;
    if (tokens < 1 || tokens > 16 || tokens > c.frame_tokens) return STATEKV_E_INVALID_ARG;
    if (c.dtype != STATEKV_BF16 || c.head_dim != 128) return STATEKV_E_UNSUPPORTED;
    const int R = h->G * tokens;
    const int npad = decode_rows_pad(R);
    if (npad < 0) return STATEKV_E_UNSUPPORTED;
    const int64_t visible = h->n * c.frame_tokens + h->text;
    if (visible + tokens > h->det_pitch) return STATEKV_E_CAPACITY;
    DeviceGuard g(c.device);
    if (!g.ok) return cuda_fail();
    // partial-result buffers, sized once for the whole detailed state
    const int64_t items_max = (int64_t)h->U * decode_chunks(h->det_pitch);
    if (h->dec_items < items_max) {
        if (!dalloc(h, &h->dec_m, sizeof(float) * items_max * 64) ||
            !dalloc(h, &h->dec_l, sizeof(float) * items_max * 64) ||
            !dalloc(h, &h->dec_o, sizeof(float) * items_max * 64 * 128))
            return STATEKV_E_OOM;
        h->dec_items = items_max;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    RopeArgs ra{};
    ra.q = q; ra.k = k; ra.v = v;
    ra.q_rot = h->q_rot; ra.pool_k = nullptr; ra.pool_v = nullptr;
    ra.det_k = h->det_k; ra.det_v = h->det_v;
    ra.cs = h->cs + (size_t)visible * (c.head_dim / 2);
    ra.rows_q = (int64_t)h->U * R;
    ra.rows_kv = (int64_t)h->U * tokens;
    ra.T = tokens; ra.d = c.head_dim; ra.slots = h->slots; ra.c = 0;
    ra.det_pitch = h->det_pitch; ra.det_row0 = visible;
    if (launch_rope(ra, c.dtype, st, false) != cudaSuccess) return cuda_fail();
    DecodeMaps maps;
    if (!make_decode_maps(&maps, h->q_rot, R, npad, h->det_k, h->det_v, h->det_pitch, h->U))
        return cuda_fail();
    DecodeArgs da{};
    da.o = o; da.part_m = h->dec_m; da.part_l = h->dec_l; da.part_o = h->dec_o; da.err = h->err;
    da.U = h->U; da.R = R; da.tok = tokens; da.chunks = decode_chunks(visible + tokens);
    da.num_sms = h->num_sms; da.visible = visible; da.keys = visible + tokens;
    da.scale_log2 = h->scale_log2;
    if (launch_decode(da, maps, st) != cudaSuccess) return cuda_fail();
    h->text += tokens;
    return STATEKV_OK;
}

int64_t statekv_text_tokens(const statekv_handle* h) { return h ? h->text : -1; }

int statekv_get_compressed(statekv_handle* h, int32_t s, int32_t layer, const void** k,
                           const void** v, const int32_t** pos, int32_t* count, int32_t* pitch) {
    if (!h || s < 0 || s >= h->cfg.num_streams || layer < 0 || layer >= h->cfg.num_layers)
        return STATEKV_E_INVALID_ARG;
    const int64_t u0 = ((int64_t)s * h->cfg.num_layers + layer) * h->cfg.num_kv_heads;
    const size_t row = (size_t)h->cfg.head_dim * h->esize;
    if (k) *k = (const char*)h->pool_k + u0 * h->slots * row;
    if (v) *v = (const char*)h->pool_v + u0 * h->slots * row;
    if (pos) *pos = h->pos + u0 * h->slots;
    if (count) *count = h->c();
    if (pitch) *pitch = h->slots;
    return STATEKV_OK;
}

int statekv_get_detailed(statekv_handle* h, int32_t s, int32_t layer, const void** k,
                         const void** v, int64_t* count, int64_t* pitch) {
    if (!h || s < 0 || s >= h->cfg.num_streams || layer < 0 || layer >= h->cfg.num_layers)
        return STATEKV_E_INVALID_ARG;
    const int64_t u0 = ((int64_t)s * h->cfg.num_layers + layer) * h->cfg.num_kv_heads;
    const size_t row = (size_t)h->cfg.head_dim * h->esize;
    if (k) *k = (const char*)h->det_k + u0 * h->det_pitch * row;
    if (v) *v = (const char*)h->det_v + u0 * h->det_pitch * row;
    if (count) *count = h->n * h->cfg.frame_tokens + h->text;
    if (pitch) *pitch = h->det_pitch;
    return STATEKV_OK;
}

int64_t statekv_frame_index(const statekv_handle* h) { return h ? h->n : -1; }

int statekv_reset(statekv_handle* h) {
    if (!h) return STATEKV_E_INVALID_ARG;
    h->n = 0;
    h->text = 0;
    return STATEKV_OK;
}

int statekv_check_device_status(statekv_handle* h, void* cuda_stream) {
    if (!h) return STATEKV_E_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_fail();
    uint32_t w[kErrWords] = {0, 0, 0, 0};
    if (cudaMemcpy(w, h->err, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_fail();
    if (w[0] == 0) return STATEKV_OK;
    std::fprintf(stderr, "statekv: device status %d at site %u (block %u, extra %u)\n",
                 (int)w[0], w[1], w[2], w[3]);
    if (cudaMemset(h->err, 0, sizeof(w)) != cudaSuccess) return cuda_fail();
    return (int)(int32_t)w[0];
}

int statekv_get_scores(statekv_handle* h, int32_t s, int32_t layer, const float** scores,
                       const int32_t** pool_pos, int32_t* m, int32_t* pitch) {
    if (!h || s < 0 || s >= h->cfg.num_streams || layer < 0 || layer >= h->cfg.num_layers)
        return STATEKV_E_INVALID_ARG;
    if (h->n == 0) return STATEKV_E_INVALID_ARG;
    const int64_t u0 = ((int64_t)s * h->cfg.num_layers + layer) * h->cfg.num_kv_heads;
    if (scores) *scores = h->scores + u0 * h->m_pad;
    if (pool_pos) *pool_pos = h->score_pos + u0 * h->m_pad;
    if (m) *m = (int32_t)std::min<int64_t>(h->cfg.budget, (h->n - 1) * h->cfg.frame_tokens) +
                h->cfg.frame_tokens;
    if (pitch) *pitch = h->m_pad;
    return STATEKV_OK;
}

int statekv_get_rotated_query(statekv_handle* h, const void** q_rot) {
    if (!h || !q_rot) return STATEKV_E_INVALID_ARG;
    *q_rot = h->q_rot;
    return STATEKV_OK;
}

int statekv_set_frame_index(statekv_handle* h, int64_t n) {
    if (!h || n < 0 || n >= h->cfg.max_frames) return STATEKV_E_INVALID_ARG;
    h->n = n;
    return STATEKV_OK;
}

int statekv_set_compressed(statekv_handle* h, int32_t s, int32_t layer, const void* k,
                           const void* v, const int32_t* pos, int32_t count, void* cuda_stream) {
    if (!h || s < 0 || s >= h->cfg.num_streams || layer < 0 || layer >= h->cfg.num_layers)
        return STATEKV_E_INVALID_ARG;
    if (count != h->c()) return STATEKV_E_INVALID_ARG;
    if (count > 0 && (!k || !v || !pos)) return STATEKV_E_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(cuda_stream);
    const size_t row = (size_t)h->cfg.head_dim * h->esize;
    const int64_t u0 = ((int64_t)s * h->cfg.num_layers + layer) * h->cfg.num_kv_heads;
    for (int hk = 0; hk < h->cfg.num_kv_heads && count > 0; ++hk) {
        const int64_t u = u0 + hk;
        if (cudaMemcpyAsync((char*)h->pool_k + u * h->slots * row,
                            (const char*)k + (size_t)hk * count * row, count * row,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync((char*)h->pool_v + u * h->slots * row,
                            (const char*)v + (size_t)hk * count * row, count * row,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(h->pos + u * h->slots, pos + (size_t)hk * count,
                            count * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return cuda_fail();
    }
    return STATEKV_OK;
}

int statekv_profile_enable(statekv_handle* h, int enable) {
    if (!h) return STATEKV_E_INVALID_ARG;
    h->profiling = enable != 0;
    if (h->profiling) {
        for (auto& e : h->pending) { h->spare.push_back(e.start); h->spare.push_back(e.stop); }
        h->pending.clear();
        for (int i = 0; i < STATEKV_NUM_KERNELS; ++i) { h->prof_ms[i] = 0; h->prof_n[i] = 0; }
    }
    return STATEKV_OK;
}

int statekv_profile_kernels(statekv_handle* h, uint32_t mask) {
    if (!h) return STATEKV_E_INVALID_ARG;
    h->prof_mask = mask;
    return STATEKV_OK;
}

int statekv_profile_read(statekv_handle* h, int32_t kernel, double* total_ms, int64_t* launches) {
    if (!h || kernel < 0 || kernel >= STATEKV_NUM_KERNELS) return STATEKV_E_INVALID_ARG;
    DeviceGuard g(h->cfg.device);
    for (auto& e : h->pending) {
        if (cudaEventSynchronize(e.stop) != cudaSuccess) return cuda_fail();
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, e.start, e.stop) != cudaSuccess) return cuda_fail();
        h->prof_ms[e.kernel] += ms;
        h->prof_n[e.kernel] += 1;
        h->spare.push_back(e.start);
        h->spare.push_back(e.stop);
    }
    h->pending.clear();
    if (total_ms) *total_ms = h->prof_ms[kernel];
    if (launches) *launches = h->prof_n[kernel];
    return STATEKV_OK;
}

}  // extern "C"
