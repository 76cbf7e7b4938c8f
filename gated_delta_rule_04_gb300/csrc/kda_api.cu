// C ABI of the KDA mixer core: host-side validation, workspace layout and the
// launch sequence of each entry point.  Every check happens here, before
// anything is enqueued, so a rejected call writes nothing.
#include <math.h>
#include <string.h>

#include <vector>

#include <algorithm>
#include <numeric>

#include "kda_chunk_layout.cuh"

namespace kda {
namespace {

constexpr int CHUNK = 64;
constexpr size_t WS_ALIGN = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t count_chunks(const int64_t* cu, int32_t n) {
    int64_t c = 0;
    for (int32_t i = 0; i < n; ++i) c += (cu[i + 1] - cu[i] + CHUNK - 1) / CHUNK;
    return c;
}

// Which prefill algorithm a parameter set runs.
enum class Algo { Scan, Chunked };

bool chunked_available() { return chunked_kernel_built(); }

kda_status resolve_algo(const kda_params* p, Algo* out) {
    const bool bf16 = p->io_dtype == KDA_DTYPE_BF16;
    // bounded gate: 16 * 5.5 = 88 < ln(FLT_MAX) keeps every sub-tile factor in
    // range; the unbounded gate takes the diagonal blocks by position pairs
    const bool bound_ok = (p->gate_kind == KDA_GATE_BOUNDED && p->gate_lower_bound >= -5.5f) ||
                          p->gate_kind == KDA_GATE_SOFTPLUS;
    switch (p->algo) {
        case KDA_ALGO_SCAN: *out = Algo::Scan; return KDA_OK;
        case KDA_ALGO_CHUNKED:
        case KDA_ALGO_CHUNKED_SEGMENTS:
            if (!bf16 || !bound_ok || !chunked_available()) return KDA_ERR_UNSUPPORTED;
            *out = Algo::Chunked;
            return KDA_OK;
        case KDA_ALGO_AUTO:
            *out = (bf16 && bound_ok && chunked_available()) ? Algo::Chunked : Algo::Scan;
            return KDA_OK;
        default: return KDA_ERR_INVALID_ARG;
    }
}

kda_status check_params(const kda_params* p) {
    if (p == nullptr) return KDA_ERR_INVALID_ARG;
    if (p->num_heads < 1 || p->num_heads > (1 << 16)) return KDA_ERR_INVALID_ARG;
    if (p->head_dim != D || p->conv_kernel != CONV_K) return KDA_ERR_UNSUPPORTED;
    if (p->io_dtype != KDA_DTYPE_F32 && p->io_dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARG;
    if (p->gate_kind != KDA_GATE_BOUNDED && p->gate_kind != KDA_GATE_SOFTPLUS) return KDA_ERR_INVALID_ARG;
    if (p->gate_kind == KDA_GATE_BOUNDED && (!(p->gate_lower_bound < 0.f) || !isfinite(p->gate_lower_bound)))
        return KDA_ERR_INVALID_ARG;
    if (!(p->l2_eps >= 0.f) || !(p->norm_eps >= 0.f) || !isfinite(p->l2_eps) || !isfinite(p->norm_eps))
        return KDA_ERR_INVALID_ARG;
    if (!isfinite(p->q_scale)) return KDA_ERR_INVALID_ARG;
    if (!p->conv_w || !p->A_log || !p->dt_bias || !p->norm_w) return KDA_ERR_INVALID_ARG;
    if (!aligned16(p->conv_w) || !aligned16(p->dt_bias) || !aligned16(p->norm_w)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

float resolved_q_scale(const kda_params* p) {
    return p->q_scale != 0.f ? p->q_scale : 1.0f / sqrtf((float)D);
}

// Workspace regions.  meta = cu_seqlens (int64 [n+1]) | first chunk of each
// sequence (int64 [n+1]) | sequence order (int32 [n], padded) | chunk table.
struct WsLayout {
    size_t status = 0, meta = 0, qh = 0, kh = 0, vh = 0, g = 0, beta = 0, ocore = 0, rec = 0, total = 0;
    size_t meta_bytes = 0, off_chunk_off = 0, off_order = 0, off_chunks = 0;
};

WsLayout layout(const kda_params* p, Algo algo, int32_t n_seqs, int64_t T, int64_t n_chunks) {
    WsLayout L;
    const size_t W = (size_t)p->num_heads * D;
    const size_t op = 4;  // q^/k^/v^ of the scan path: fp32
    size_t off = 0;
    L.status = off; off += WS_ALIGN;
    L.meta = off;
    L.off_chunk_off = sizeof(int64_t) * (size_t)(n_seqs + 1);
    L.off_order = L.off_chunk_off + sizeof(int64_t) * (size_t)(n_seqs + 1);
    L.off_chunks = align_up(L.off_order + sizeof(int32_t) * (size_t)n_seqs, 16);
    L.meta_bytes = L.off_chunks + sizeof(ChunkDesc) * (size_t)n_chunks;
    off = align_up(off + L.meta_bytes, WS_ALIGN);
    // q^, k^, v^ (fp32), gate, beta and o_core: only the scan path has a
    // separate pre-stage and output stage; the chunked path keeps them on chip
    const bool scan = algo == Algo::Scan;
    const size_t tw = scan ? (size_t)T * W : 0;
    L.qh = off; off = align_up(off + op * tw, WS_ALIGN);
    L.kh = off; off = align_up(off + op * tw, WS_ALIGN);
    L.vh = off; off = align_up(off + op * tw, WS_ALIGN);
    L.g = off; off = align_up(off + 4 * tw, WS_ALIGN);
    L.beta = off; off = align_up(off + 4 * (scan ? (size_t)T * p->num_heads : 0), WS_ALIGN);
    L.ocore = off;
    off = align_up(off + 4 * tw, WS_ALIGN);
    L.rec = off;
    if (algo == Algo::Chunked) off = align_up(off + (size_t)REC_BYTES * (size_t)n_chunks * p->num_heads, WS_ALIGN);
    L.total = off;
    return L;
}

kda_status check_cu(const int64_t* cu, int32_t n, int64_t T) {
    if (n < 0 || T < 0) return KDA_ERR_INVALID_ARG;
    if (cu == nullptr) return KDA_ERR_INVALID_ARG;
    if (cu[0] != 0 || cu[n] != T) return KDA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (cu[i + 1] < cu[i]) return KDA_ERR_INVALID_ARG;
    if (T > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;  // chunk table uses int32 token indices
    return KDA_OK;
}

kda_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

struct OverlapPlan {
    int S = 0, sms = 0;
    int64_t seg = 0, seg_chunks = 0;
    size_t meta_stride = 0, off_meta = 0, off_cufull = 0, off_rec[2] = {0, 0}, total = 0;
};
constexpr size_t WS_COUNTER = 64;   // two work counters of the chunk preparation, inside the status block

// The windows and their workspace layout for a T-token sequence (false when it
// is too short for two windows).  No device query: the workspace size uses it.
// Shortest window.  With up to 64 heads the recurrence leaves most SMs to the
// chunk preparation, and windows of 16 chunks paid from 2048 tokens on (20-25 %
// at 8192-16384 tokens and 32 heads, measured on GB300).  With more heads the
// recurrence takes most SMs and windows shorter than 8192 tokens did not pay.
int64_t window_min(int H) { return H <= 64 ? 1024 : 8192; }

bool overlap_layout(const kda_params* p, int64_t T, OverlapPlan* pl) {
    const int64_t wmin = window_min(p->num_heads);
    if (T < 2 * wmin) return false;
    // Up to 4 windows of at least wmin tokens (3 above 48 heads), the last one 1/d
    // as long as the others, since its recurrence runs alone after every
    // preparation: d = 6 above 64 heads, 4 above 32, 2 up to 32.  Measured on
    // GB300 at T = 32768: 96 heads 3.85 ms with four equal windows, 3.78 with
    // four and d = 4, 3.72 with three and d = 6; 64 heads 2.66 / 2.56 (four,
    // d = 4) / 2.55 (three, d = 4); 48 heads 2.04 with four and d = 4 against
    // 2.06 with three; 32 heads 1.50 / 1.47 (four, d = 2) against 1.51 with three.
    const int64_t s0 = std::min<int64_t>(p->num_heads > 48 ? 3 : 4, T / wmin);
    const int64_t d = p->num_heads > 64 ? 6 : p->num_heads > 32 ? 4 : 2;
    const int64_t seg = ((d * T + d * s0 - d) / (d * s0 - (d - 1)) + CHUNK - 1) / CHUNK * CHUNK;
    pl->S = (int)((T + seg - 1) / seg);
    if (pl->S < 2) return false;
    pl->seg = seg;
    pl->seg_chunks = seg / CHUNK;
    pl->meta_stride = 4 * sizeof(int64_t) + sizeof(ChunkDesc) * (size_t)pl->seg_chunks;
    size_t off = WS_ALIGN;  // status block
    pl->off_meta = off;
    off = align_up(off + pl->meta_stride * pl->S, WS_ALIGN);
    pl->off_cufull = off;
    off += WS_ALIGN;
    const size_t rec_bytes = (size_t)REC_BYTES * (size_t)pl->seg_chunks * (size_t)p->num_heads;
    for (int r = 0; r < 2; ++r) {
        pl->off_rec[r] = off;
        off = align_up(off + rec_bytes, WS_ALIGN);
    }
    pl->total = off;
    return true;
}


// ---- segmented recurrence of one sequence -------------------------------------
// The sequence's chunks split into P segments; the recurrence of each segment
// runs in parallel from a zero state (and its linear part from the identity),
// an affine scan composes the segment maps, and a second pass runs every
// segment after the first from its true starting state (see kda_segments.cu).
struct SegPlan {
    int P = 0;
    int64_t c_first[MAX_SEGS + 1] = {};   // first chunk of each segment; c_first[P] = chunks
    size_t slot_bytes = 0, off_slots = 0, total = 0;
};
constexpr int64_t SEG_MIN_CHUNKS = 8;   // shortest segment
constexpr int SMS_GB300 = 152;

// The fewest segments a call runs as: KDA_ALGO_CHUNKED_SEGMENTS takes any
// P >= 3 and KDA_ALGO_CHUNKED none.  KDA_ALGO_AUTO takes P >= 5, and P >= 3
// for sequences of 64 to 128 chunks.  Measured on GB300 against the overlapped
// windows: with P >= 5 segments halve the step of long few-head sequences
// (T = 32768, H = 8: 1.07 -> 0.55 ms); with P = 3 or 4, two thirds or half of
// the chain stay serial, after the whole preparation, and the windows, which
// overlap the chain with the preparation, win on long sequences (T = 16384,
// H = 32: 0.81 against 0.87 ms) while segments win from 4096 to 8192 tokens
// (T = 4096, H = 32: 0.273 against 0.296 ms).
int segment_min(const kda_params* p, int64_t chunks) {
    if (p->algo == KDA_ALGO_CHUNKED_SEGMENTS) return 3;
    if (p->algo == KDA_ALGO_AUTO) return (chunks >= 64 && chunks <= 128) ? 3 : 5;
    return 1 << 30;
}

// The number of segments for H heads on `sms` SMs (0: not segmented): the
// first pass runs 2P - 3 CTAs per head, and every segment holds at least
// SEG_MIN_CHUNKS chunks.
int segment_count(int H, int sms, int64_t chunks) {
    int P = 0;
    for (int c = 3; c <= (MAX_SEGS + 3) / 2; ++c)
        if ((int64_t)H * (2 * c - 3) <= sms && chunks >= (int64_t)c * SEG_MIN_CHUNKS) P = c;
    return P;
}

// Workspace of the segmented schedule: the single pass's, then 3P - 5 state
// slots of H x 128 x 128 fp32 (the offsets B_0 .. B_{P-2}, the maps M_1 ..
// M_{P-2}, the composed states X_2 .. X_{P-1}).
// P is the most segments `sms` SMs take, reduced until the layout fits
// `ws_bytes` (0: no limit).
bool segment_layout(const kda_params* p, int64_t T, int sms, size_t single_bytes, size_t ws_bytes, SegPlan* sp) {
    const int64_t chunks = (T + CHUNK - 1) / CHUNK;
    const size_t slot = (size_t)p->num_heads * D * D * sizeof(float);
    const size_t base = align_up(single_bytes, WS_ALIGN);
    const int P_min = segment_min(p, chunks);
    int P = segment_count(p->num_heads, sms, chunks);
    while (P >= P_min && ws_bytes != 0 && base + (size_t)(3 * P - 5) * slot > ws_bytes) --P;
    if (P < P_min || P < 3) return false;
    sp->P = P;
    for (int i = 0; i <= P; ++i) sp->c_first[i] = chunks * i / P;
    sp->slot_bytes = (size_t)p->num_heads * D * D * sizeof(float);
    sp->off_slots = align_up(single_bytes, WS_ALIGN);
    sp->total = sp->off_slots + (size_t)(3 * P - 5) * sp->slot_bytes;
    return true;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char* kda_status_str(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
        case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    }
    return "unknown status";
}

int32_t kda_prefill_algo(const kda_params* p) {
    if (check_params(p) != KDA_OK) return -1;
    Algo algo;
    if (resolve_algo(p, &algo) != KDA_OK) return -1;
    return algo == Algo::Chunked ? KDA_ALGO_CHUNKED : KDA_ALGO_SCAN;
}

size_t kda_prefill_workspace_bytes(const kda_params* p, int32_t n_seqs, int64_t total_tokens) {
    if (check_params(p) != KDA_OK || n_seqs < 0 || total_tokens < 0) return 0;
    Algo algo;
    if (resolve_algo(p, &algo) != KDA_OK) return 0;
    if (n_seqs == 0 && total_tokens == 0) return 0;
    // upper bound on the chunk count: every sequence may add one partial chunk
    const int64_t n_chunks = total_tokens / CHUNK + n_seqs;
    size_t need = layout(p, algo, n_seqs, total_tokens, n_chunks).total;
    OverlapPlan pl;   // one long sequence may run as windows (see prefill_overlapped)
    if (algo == Algo::Chunked && n_seqs == 1 && overlap_layout(p, total_tokens, &pl)) need = std::max(need, pl.total);
    // one sequence may run as segments (prefill_segmented); the reserve assumes
    // GB300's 152 SMs, and a call with less workspace takes fewer segments
    SegPlan sp;
    if (algo == Algo::Chunked && n_seqs == 1 &&
        segment_layout(p, total_tokens, SMS_GB300, layout(p, algo, 1, total_tokens, n_chunks).total, 0, &sp))
        need = std::max(need, sp.total);
    return need;
}

}  // extern "C"

namespace {

// Records ev[i] (when given) on the stream; stage boundaries for profiling.
cudaError_t mark(void* const* ev, int i, cudaStream_t s) {
    if (ev == nullptr || ev[i] == nullptr) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
}

}  // namespace

namespace kda {
namespace {

// ---- overlapped chunked prefill ------------------------------------------------
// One sequence whose recurrence (one CTA per head) would leave SMs idle: the
// sequence runs as S windows of whole chunks, and the recurrence of window w
// overlaps the chunk preparation of window w + 1.  The preparation of a window
// is two launches sharing one work counter: part 1 on the caller's stream with
// as many CTAs as the recurrence leaves SMs free, part 2 on the recurrence
// stream behind the recurrence of the window before, with one CTA per SM it
// frees.  Windows start on the chunk grid of the sequence and read the conv halo
// from the inputs, so the result is the same, bit for bit, as the single pass;
// the state continues in S_out from window to window, and the ring is updated
// once at the end.
// Whether this call runs as windows: one long sequence, fewer heads than SMs.
bool plan_overlap(const kda_params* p, int64_t T, size_t ws_bytes, OverlapPlan* pl) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    if (p->num_heads >= sms || !overlap_layout(p, T, pl)) return false;
    pl->sms = sms;
    return pl->total <= ws_bytes;
}

// The recurrence stream (highest priority) and the events of the window
// schedule, per host thread and device: created on a thread's first windowed
// call on a device and kept for the thread's lifetime.  Two host threads never
// share them, so concurrent calls on different streams cannot wait on each
// other's events; calls from one thread are ordered by the events themselves.
struct WindowStreams {
    cudaStream_t sr = nullptr;
    cudaEvent_t ev[7] = {};
};
// A thread's window streams and events, released when the thread exits (while
// the runtime is still usable: at process exit it may already be unloading).
struct ThreadWindowStreams {
    std::vector<WindowStreams> per_device;
    ~ThreadWindowStreams() {
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        for (size_t d = 0; d < per_device.size(); ++d) {
            WindowStreams& w = per_device[d];
            if (w.sr == nullptr || cudaSetDevice((int)d) != cudaSuccess) continue;
            for (auto& e : w.ev)
                if (e) cudaEventDestroy(e);
            cudaStreamDestroy(w.sr);
        }
        cudaSetDevice(prev);
    }
};
WindowStreams* window_streams() {
    thread_local ThreadWindowStreams tws;
    std::vector<WindowStreams>& per_device = tws.per_device;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    if ((size_t)dev >= per_device.size()) per_device.resize(dev + 1);
    WindowStreams& w = per_device[dev];
    if (w.sr == nullptr) {
        int least = 0, greatest = 0;
        WindowStreams n;
        bool good = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
                    cudaStreamCreateWithPriority(&n.sr, cudaStreamNonBlocking, greatest) == cudaSuccess;
        for (auto& e : n.ev) good = good && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
        if (!good) {
            for (auto& e : n.ev)
                if (e) cudaEventDestroy(e);
            if (n.sr) cudaStreamDestroy(n.sr);
            return nullptr;
        }
        w = n;
    }
    return &w;
}

kda_status prefill_overlapped(const kda_params* p, const void* q, const void* k, const void* v, const void* z,
                              const void* b, const void* gout, int64_t T, const float* S_in, float* S_out,
                              const void* ring_in, void* ring_out, void* o, unsigned char* ws, cudaStream_t s,
                              const OverlapPlan& pl, bool reset_status) {
    const int H = p->num_heads, W = H * D;
    int32_t* status = reinterpret_cast<int32_t*>(ws);
    int32_t* counters = reinterpret_cast<int32_t*>(ws + WS_COUNTER);   // [2], by window parity

    WindowStreams* res = window_streams();
    if (res == nullptr) return KDA_ERR_CUDA;
    cudaStream_t sr = res->sr;
    cudaEvent_t* ev = res->ev;   // start, prep part 1 [2], recurrence [2], end, counter reset
    kda_status st = KDA_OK;
    auto ok = [&](cudaError_t e) { if (e != cudaSuccess) st = KDA_ERR_CUDA; return st == KDA_OK; };
    if (st == KDA_OK && ok(cudaEventRecord(ev[0], s)) && ok(cudaStreamWaitEvent(sr, ev[0], 0)) &&
        ok(reset_status ? cudaMemsetAsync(ws, 0, WS_ALIGN, s) : cudaSuccess) &&
        // every window's cu, chunk offsets and chunk table, built on the device
        ok(launch_build_window_meta(T, pl.seg, pl.S, (int64_t)pl.meta_stride, ws + pl.off_meta,
                                    reinterpret_cast<int64_t*>(ws + pl.off_cufull), s))) {
        const float qs = resolved_q_scale(p);
        // items per take: batches of PREP_BATCH amortise the counter, but a
        // window with few items per SM balances better one item at a time
        const int64_t win_items = pl.seg_chunks * H;
        const int32_t batch = win_items >= (int64_t)8 * PREP_BATCH * pl.sms ? PREP_BATCH : 1;
        for (int w = 0; w < pl.S && st == KDA_OK; ++w) {
            const int r = w & 1;
            unsigned char* rec = ws + pl.off_rec[r];
            const unsigned char* mw = ws + pl.off_meta + w * pl.meta_stride;
            const int64_t t0 = w * pl.seg, nck = (std::min(T, t0 + pl.seg) - t0 + CHUNK - 1) / CHUNK;
            int32_t* counter = counters + r;
            // records and counter of window w - 2 (same parity) are no longer in use
            if (w >= 2 && !ok(cudaStreamWaitEvent(s, ev[3 + r], 0))) break;
            if (!ok(cudaMemsetAsync(counter, 0, sizeof(int32_t), s))) break;
            // part 2 (on sr) takes items from this counter: it starts after the reset
            if (w > 0 && (!ok(cudaEventRecord(ev[6], s)) || !ok(cudaStreamWaitEvent(sr, ev[6], 0)))) break;
            PrepArgs pr{q, k, v, z, b, ring_in, p->conv_w, p->A_log, p->dt_bias, p->gate_lower_bound, p->l2_eps, qs,
                        reinterpret_cast<const ChunkDesc*>(mw + 4 * sizeof(int64_t)), (int32_t)nck, H, T, rec, status,
                        counter, batch, prep_wait_limit_ns(p), {}, {}, p->gate_kind};
            // part 1 alongside the recurrence of window w - 1 (all SMs for window 0)
            if (!ok(launch_chunk_prep(pr, s, w == 0 ? 0 : pl.sms - H)) || !ok(cudaEventRecord(ev[1 + r], s))) break;
            // part 2 on the SMs that recurrence frees
            if (w > 0 && !ok(launch_chunk_prep(pr, sr, H))) break;
            if (!ok(cudaStreamWaitEvent(sr, ev[1 + r], 0))) break;
            ChunkRecArgs ca{rec, w == 0 ? S_in : S_out, S_out, gout, p->norm_w, o, p->norm_eps,
                            reinterpret_cast<const int64_t*>(mw), reinterpret_cast<const int64_t*>(mw) + 2, nullptr,
                            status, 1, H};
            if (!ok(launch_chunk_recurrence(ca, sr)) || !ok(cudaEventRecord(ev[3 + r], sr))) break;
        }
        if (st == KDA_OK && ring_out) {
            RingArgs ra{q, k, v, ring_in, ring_out, reinterpret_cast<const int64_t*>(ws + pl.off_cufull), 1, W};
            ok(launch_ring_update(ra, 1, sr));
        }
    }
    // the caller's stream orders after everything on the recurrence stream
    if (cudaEventRecord(ev[5], sr) != cudaSuccess || cudaStreamWaitEvent(s, ev[5], 0) != cudaSuccess)
        st = KDA_ERR_CUDA;
    return st;
}

// Whether this call runs its recurrence as segments: one sequence whose heads
// leave most SMs idle (2P - 3 CTAs per head for P >= 3 segments of at least
// SEG_MIN_CHUNKS chunks) and a workspace that holds the state slots.
bool plan_segments(const kda_params* p, int64_t T, size_t single_bytes, size_t ws_bytes, SegPlan* sp) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return segment_layout(p, T, sms, single_bytes, ws_bytes, sp);
}

// The recurrence of one sequence (chunk preparation done, records in `rec`)
// as P segments: pass 1 runs segments 0 .. P-2 from their starting states
// (the caller's for segment 0, which writes its outputs there; zero for the
// others) and the linear parts of segments 1 .. P-2 from the identity; the
// scan composes X_{p+1} = M_p X_p + B_p; pass 2 runs segments 1 .. P-1 from
// their true starting states, writing their outputs and, for the last, S_out.
kda_status recurrence_segmented(const kda_params* p, const void* gout, int64_t T, const float* S_in, float* S_out,
                                void* o, const void* rec, int32_t* status, unsigned char* ws, const SegPlan& sp,
                                cudaStream_t s) {
    const int H = p->num_heads, P = sp.P;
    auto slot = [&](int i) { return reinterpret_cast<float*>(ws + sp.off_slots + (size_t)i * sp.slot_bytes); };
    // slots: B_0 .. B_{P-2} at 0 .. P-2, M_p (p = 1 .. P-2) at P-1 .. 2P-4, X_p (p = 2 .. P-1) at 2P-3 .. 3P-6
    auto B = [&](int q) { return slot(q); };
    auto M = [&](int q) { return slot(P - 2 + q); };
    auto X = [&](int q) { return slot(2 * P - 5 + q); };
    auto seg_t0 = [&](int q) { return (int64_t)CHUNK * sp.c_first[q]; };
    auto seg_t1 = [&](int q) { return std::min<int64_t>(T, (int64_t)CHUNK * sp.c_first[q + 1]); };
    ChunkRecArgs a{};
    a.records = rec; a.gout = gout; a.norm_w = p->norm_w; a.o = o; a.eps = p->norm_eps; a.status = status; a.H = H;
    int n = 0;
    auto add = [&](int q, const float* in, float* out, int32_t mode) {
        a.seg_t0[n] = seg_t0(q); a.seg_t1[n] = seg_t1(q); a.seg_c0[n] = sp.c_first[q];
        a.seg_S_in[n] = in; a.seg_S_out[n] = out; a.seg_mode[n] = mode;
        ++n;
    };
    add(0, S_in, B(0), 0);
    for (int q = 1; q + 1 < P; ++q) add(q, nullptr, B(q), SEG_NO_OUTPUT);
    for (int q = 1; q + 1 < P; ++q) add(q, nullptr, M(q), SEG_IDENTITY | SEG_LINEAR | SEG_NO_OUTPUT);
    a.n_segs = n;
    if (launch_chunk_recurrence(a, s) != cudaSuccess) return KDA_ERR_CUDA;
    {
        ScanArgs2 sa{};
        sa.P = P; sa.H = H;
        for (int q = 0; q + 1 < P; ++q) sa.B[q] = B(q);
        for (int q = 1; q + 1 < P; ++q) sa.M[q] = M(q);
        for (int q = 2; q < P; ++q) sa.X[q] = X(q);
        if (launch_affine_scan(sa, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    n = 0;
    for (int q = 1; q < P; ++q) add(q, q == 1 ? B(0) : X(q), q == P - 1 ? S_out : nullptr, 0);
    a.n_segs = n;
    if (launch_chunk_recurrence(a, s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

kda_status prefill_check(const kda_params* p) {
    kda_status st = check_params(p);
    if (st != KDA_OK) return st;
    Algo algo;
    return resolve_algo(p, &algo);
}

kda_status prefill_run(const kda_params* p, const void* q, const void* k, const void* v,
                       const void* z, const void* b, const void* gout,
                       const int64_t* cu_seqlens_host, int32_t n_seqs, int64_t total_tokens,
                       const float* S_in, float* S_out, const void* ring_in, void* ring_out,
                       void* o, void* workspace, size_t workspace_bytes, void* stream_,
                       void* const* ev, bool reset_status) {
    kda_status st = check_params(p);
    if (st != KDA_OK) return st;
    Algo algo;
    st = resolve_algo(p, &algo);
    if (st != KDA_OK) return st;
    st = check_cu(cu_seqlens_host, n_seqs, total_tokens);
    if (st != KDA_OK) return st;
    if (n_seqs == 0) return KDA_OK;
    if (total_tokens > 0) {
        const void* tok[7] = {q, k, v, z, gout, o, nullptr};
        for (int i = 0; i < 6; ++i)
            if (tok[i] == nullptr || !aligned16(tok[i])) return KDA_ERR_INVALID_ARG;
        if (b == nullptr) return KDA_ERR_INVALID_ARG;
    }
    if (S_out == nullptr || !aligned16(S_out) || (S_in && !aligned16(S_in))) return KDA_ERR_INVALID_ARG;
    if ((ring_in && !aligned16(ring_in)) || (ring_out && !aligned16(ring_out))) return KDA_ERR_INVALID_ARG;

    const int64_t n_chunks = count_chunks(cu_seqlens_host, n_seqs);
    const size_t need = kda_prefill_workspace_bytes(p, n_seqs, total_tokens);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % WS_ALIGN))
        return KDA_ERR_WORKSPACE;
    const WsLayout L = layout(p, algo, n_seqs, total_tokens, n_chunks);

    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    SegPlan sp;
    const bool segmented = algo == Algo::Chunked && n_seqs == 1 &&
                           plan_segments(p, total_tokens, L.total, workspace_bytes, &sp);
    if (algo == Algo::Chunked && ev == nullptr && n_seqs == 1 && !segmented) {
        OverlapPlan pl;
        if (plan_overlap(p, total_tokens, workspace_bytes, &pl))
            return prefill_overlapped(p, q, k, v, z, b, gout, total_tokens, S_in, S_out, ring_in, ring_out, o,
                                      static_cast<unsigned char*>(workspace), s, pl, reset_status);
    }
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const int H = p->num_heads, W = H * D;
    const int io_bf16 = p->io_dtype == KDA_DTYPE_BF16;

    // longest sequences first, so the sequential chunk walks start early
    std::vector<int32_t> order(n_seqs);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
        return cu_seqlens_host[x + 1] - cu_seqlens_host[x] > cu_seqlens_host[y + 1] - cu_seqlens_host[y];
    });
    const int64_t* d_cu = reinterpret_cast<const int64_t*>(ws + L.meta);
    const int64_t* d_coff = reinterpret_cast<const int64_t*>(ws + L.meta + L.off_chunk_off);
    const int32_t* d_order = reinterpret_cast<const int32_t*>(ws + L.meta + L.off_order);
    const ChunkDesc* d_chunks = reinterpret_cast<const ChunkDesc*>(ws + L.meta + L.off_chunks);
    // the status word reports bounded-wait timeouts of this call only (of
    // the whole segmented call when the caller clears it once)
    cudaError_t e = reset_status ? cudaMemsetAsync(ws + L.status, 0, WS_ALIGN, s) : cudaSuccess;
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    // cu_seqlens, chunk offsets, order and chunk table, built on the device from
    // kernel arguments (no copy from pageable host memory)
    e = build_meta(cu_seqlens_host, order.data(), n_seqs, 0, const_cast<int64_t*>(d_cu), const_cast<int64_t*>(d_coff),
                   const_cast<int32_t*>(d_order), const_cast<ChunkDesc*>(d_chunks), s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;

    if (mark(ev, 0, s) != cudaSuccess) return KDA_ERR_CUDA;
    const float qs = resolved_q_scale(p);
    float* gbuf = reinterpret_cast<float*>(ws + L.g);
    float* beta = reinterpret_cast<float*>(ws + L.beta);
    float* ocore = reinterpret_cast<float*>(ws + L.ocore);

    PrestageArgs pa{q, k, v, z, b, p->conv_w, p->A_log, p->dt_bias, ring_in, d_cu, d_chunks,
                    (int32_t)n_chunks, H, p->gate_lower_bound, p->l2_eps, qs, p->gate_kind,
                    ws + L.qh, ws + L.kh, ws + L.vh, gbuf, beta};
    if (algo == Algo::Scan) {
        e = launch_prestage(pa, io_bf16, /*out_fp16=*/0, /*cumsum=*/0, s);
        if (e != cudaSuccess || mark(ev, 1, s) != cudaSuccess || mark(ev, 2, s) != cudaSuccess) return KDA_ERR_CUDA;
        ScanArgs sa{reinterpret_cast<const float*>(ws + L.qh), reinterpret_cast<const float*>(ws + L.kh),
                    reinterpret_cast<const float*>(ws + L.vh), gbuf, beta, S_in, S_out, ocore, d_cu,
                    n_seqs, H};
        e = launch_scan(sa, s);
        if (e != cudaSuccess || mark(ev, 3, s) != cudaSuccess) return KDA_ERR_CUDA;
    } else {
        // the chunk preparation runs the pre-stage itself
        if (mark(ev, 1, s) != cudaSuccess) return KDA_ERR_CUDA;
        PrepArgs pr{q, k, v, z, b, ring_in, p->conv_w, p->A_log, p->dt_bias, p->gate_lower_bound, p->l2_eps, qs,
                    d_chunks, (int32_t)n_chunks, H, total_tokens, ws + L.rec, reinterpret_cast<int32_t*>(ws + L.status), nullptr,
                    PREP_BATCH, prep_wait_limit_ns(p), {}, {}, p->gate_kind};
        e = launch_chunk_prep(pr, s);
        if (e != cudaSuccess || mark(ev, 2, s) != cudaSuccess) return KDA_ERR_CUDA;
        // the recurrence kernel applies the output norm itself; one sequence with
        // few heads runs it as segments
        if (segmented) {
            const kda_status st2 = recurrence_segmented(p, gout, total_tokens, S_in, S_out, o, ws + L.rec,
                                                        reinterpret_cast<int32_t*>(ws + L.status), ws, sp, s);
            if (st2 != KDA_OK) return st2;
        } else {
            ChunkRecArgs ca{ws + L.rec, S_in, S_out, gout, p->norm_w, o, p->norm_eps, d_cu, d_coff, d_order,
                            reinterpret_cast<int32_t*>(ws + L.status), n_seqs, H};
            e = launch_chunk_recurrence(ca, s);
            if (e != cudaSuccess) return KDA_ERR_CUDA;
        }
        if (mark(ev, 3, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (algo == Algo::Scan) {
        EpilogueArgs ea{ocore, gout, p->norm_w, o, total_tokens, H, p->norm_eps};
        e = launch_epilogue(ea, io_bf16, s);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (mark(ev, 4, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (ring_out) {
        RingArgs ra{q, k, v, ring_in, ring_out, d_cu, n_seqs, W};
        e = launch_ring_update(ra, io_bf16, s);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (mark(ev, 5, s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace kda

extern "C" {

int32_t kda_prefill_windows(const kda_params* p, int32_t n_seqs, int64_t total_tokens, size_t workspace_bytes) {
    if (check_params(p) != KDA_OK || n_seqs < 0 || total_tokens < 0) return -1;
    Algo algo;
    if (resolve_algo(p, &algo) != KDA_OK) return -1;
    if (algo != Algo::Chunked || n_seqs != 1) return 1;
    SegPlan sp;
    int64_t n_chunks = (total_tokens + CHUNK - 1) / CHUNK;
    if (plan_segments(p, total_tokens, layout(p, algo, 1, total_tokens, n_chunks).total, workspace_bytes, &sp))
        return 1;
    OverlapPlan pl;
    if (plan_overlap(p, total_tokens, workspace_bytes, &pl)) return pl.S;
    return 1;
}

int32_t kda_prefill_segments(const kda_params* p, int32_t n_seqs, int64_t total_tokens, size_t workspace_bytes) {
    if (check_params(p) != KDA_OK || n_seqs < 0 || total_tokens < 0) return -1;
    Algo algo;
    if (resolve_algo(p, &algo) != KDA_OK) return -1;
    if (algo != Algo::Chunked || n_seqs != 1) return 0;
    SegPlan sp;
    const int64_t n_chunks = (total_tokens + CHUNK - 1) / CHUNK;
    if (plan_segments(p, total_tokens, layout(p, algo, 1, total_tokens, n_chunks).total, workspace_bytes, &sp))
        return sp.P;
    return 0;
}

kda_status kda_prefill(const kda_params* p, const void* q, const void* k, const void* v,
                       const void* z, const void* b, const void* gout,
                       const int64_t* cu_seqlens_host, int32_t n_seqs, int64_t total_tokens,
                       const float* S_in, float* S_out, const void* ring_in, void* ring_out,
                       void* o, void* workspace, size_t workspace_bytes, void* stream) {
    return prefill_run(p, q, k, v, z, b, gout, cu_seqlens_host, n_seqs, total_tokens, S_in, S_out, ring_in,
                       ring_out, o, workspace, workspace_bytes, stream, nullptr, true);
}

kda_status kda_prefill_with_events(const kda_params* p, const void* q, const void* k, const void* v,
                                   const void* z, const void* b, const void* gout,
                                   const int64_t* cu_seqlens_host, int32_t n_seqs,
                                   int64_t total_tokens, const float* S_in, float* S_out,
                                   const void* ring_in, void* ring_out, void* o, void* workspace,
                                   size_t workspace_bytes, void* stream, void* const* stage_events) {
    return prefill_run(p, q, k, v, z, b, gout, cu_seqlens_host, n_seqs, total_tokens, S_in, S_out, ring_in,
                       ring_out, o, workspace, workspace_bytes, stream, stage_events, true);
}

kda_status kda_decode_multi(const kda_params* p, int32_t n_sessions, int32_t n_tokens, const void* q,
                            const void* k, const void* v, const void* z, const void* b, const void* gout,
                            const int32_t* slots, int32_t n_slots, const float* S_in, float* S_out,
                            const void* ring_in, void* ring_out, void* o, void* stream_) {
    kda_status st = check_params(p);
    if (st != KDA_OK) return st;
    if (n_sessions < 0 || n_tokens < 1 || n_tokens > KDA_DECODE_MAX_TOKENS || n_slots < 0) return KDA_ERR_INVALID_ARG;
    if (n_sessions == 0) return KDA_OK;
    if (slots == nullptr && n_slots < n_sessions) return KDA_ERR_INVALID_ARG;
    const void* ptrs[10] = {q, k, v, z, gout, o, S_in, S_out, ring_in, ring_out};
    for (int i = 0; i < 10; ++i)
        if (ptrs[i] == nullptr || !aligned16(ptrs[i])) return KDA_ERR_INVALID_ARG;
    if (b == nullptr) return KDA_ERR_INVALID_ARG;
    if ((int64_t)n_sessions * p->num_heads > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    DecodeArgs da{q, k, v, z, b, gout, p->conv_w, p->A_log, p->dt_bias, p->norm_w, slots, S_in, S_out, ring_in,
                  ring_out, o, n_sessions, p->num_heads, n_tokens, n_slots, p->gate_lower_bound, p->l2_eps,
                  p->norm_eps, resolved_q_scale(p), p->gate_kind};
    return cuda_status(launch_decode(da, p->io_dtype == KDA_DTYPE_BF16, static_cast<cudaStream_t>(stream_)));
}

kda_status kda_decode(const kda_params* p, int32_t n_sessions, const void* q, const void* k,
                      const void* v, const void* z, const void* b, const void* gout, float* S,
                      void* ring, void* o, void* stream_) {
    return kda_decode_multi(p, n_sessions, 1, q, k, v, z, b, gout, nullptr, n_sessions, S, S, ring, ring, o,
                            stream_);
}

kda_status kda_workspace_status(void* workspace, void* stream_) {
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % WS_ALIGN)) return KDA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (word == ERR_NONE) return KDA_OK;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    return word == ERR_TIMEOUT ? KDA_ERR_TIMEOUT : KDA_ERR_CUDA;
}

}  // extern "C"
