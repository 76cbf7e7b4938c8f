// kda_prefill_host: the prefill of a packed batch that lives in host memory,
// with the host<->device copies hidden behind the kernels.
//
// The batch is cut into consecutive token segments.  Each segment is a
// kda_prefill call over the pieces of the sequences that fall inside it; a
// piece continues from the state and conv ring the previous piece of its
// sequence left in S_out / ring_out (updated in place), so the segments
// together compute the prefill of the whole batch.  Three staging sets
// rotate over three streams: while the compute stream runs segment s, the
// copy-in stream loads segment s + 1 and the copy-out stream reads back the
// output of segment s - 1.  A set is reloaded only after its output has been
// read back.
#include <algorithm>
#include <vector>

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr size_t HS_ALIGN = 256;
constexpr int N_SETS = 3;
size_t hs_up(size_t x) { return (x + HS_ALIGN - 1) / HS_ALIGN * HS_ALIGN; }

// One staging set for `seg` tokens: planes q, k, v, z, gout, o [seg][H*128]
// and the beta logits b [seg][H], each 256-byte aligned.
struct StageLayout {
    size_t plane = 0, set = 0;
};
StageLayout stage_layout(int H, size_t esize, int64_t seg) {
    StageLayout L;
    L.plane = hs_up((size_t)seg * H * D * esize);
    L.set = 6 * L.plane + hs_up((size_t)seg * H * esize);
    return L;
}

// The sequence pieces inside tokens [t0, t1): sequences first..last, with the
// cumulative piece lengths in sub (sub[0] = 0).  `first` only moves forward
// between consecutive segments.  Sequences that end at or before t0 are
// skipped (empty ones keep the state copied through at the start).
void segment_pieces(const int64_t* cu, int32_t n, int64_t t0, int64_t t1, int32_t& first, int32_t& last,
                    std::vector<int64_t>& sub) {
    while (first < n && cu[first + 1] <= t0) ++first;
    last = first;
    while (last + 1 < n && cu[last + 1] < t1) ++last;
    sub.assign(1, 0);
    for (int32_t i = first; i <= last; ++i) {
        const int64_t a = std::max(cu[i], t0), c = std::min(cu[i + 1], t1);
        sub.push_back(sub.back() + std::max<int64_t>(c - a, 0));
    }
}

bool cu_ok(const int64_t* cu, int32_t n, int64_t T) {
    if (cu == nullptr || n < 0 || T < 0 || cu[0] != 0 || cu[n] != T) return false;
    for (int32_t i = 0; i < n; ++i)
        if (cu[i + 1] < cu[i]) return false;
    return true;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest kda_prefill workspace any segment needs.
size_t max_segment_workspace(const kda_params* p, const int64_t* cu, int32_t n, int64_t T, int64_t seg) {
    size_t need = 0;
    std::vector<int64_t> sub;
    int32_t first = 0, last = 0;
    for (int64_t t0 = 0; t0 < T; t0 += seg) {
        const int64_t t1 = std::min(T, t0 + seg);
        segment_pieces(cu, n, t0, t1, first, last, sub);
        need = std::max(need, kda_prefill_workspace_bytes(p, last - first + 1, t1 - t0));
    }
    return hs_up(need);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

size_t kda_prefill_host_scratch_bytes(const kda_params* p, const int64_t* cu_seqlens_host, int32_t n_seqs,
                                      int64_t total_tokens, int64_t segment_tokens) {
    if (prefill_check(p) != KDA_OK || segment_tokens <= 0 || segment_tokens > (int64_t)INT32_MAX) return 0;
    if (!cu_ok(cu_seqlens_host, n_seqs, total_tokens) || total_tokens == 0) return 0;
    const size_t esize = p->io_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const int64_t seg = std::min(segment_tokens, total_tokens);
    return max_segment_workspace(p, cu_seqlens_host, n_seqs, total_tokens, seg) +
           N_SETS * stage_layout(p->num_heads, esize, seg).set;
}

kda_status kda_prefill_host(const kda_params* p, const void* q, const void* k, const void* v, const void* z,
                            const void* b, const void* gout, const int64_t* cu, int32_t n_seqs,
                            int64_t total_tokens, const float* S_in, float* S_out, const void* ring_in,
                            void* ring_out, void* o, int64_t segment_tokens, void* scratch, size_t scratch_bytes,
                            void* stream_, void* h2d_stream_, void* d2h_stream_) {
    // ---- every check before anything is enqueued
    kda_status st = prefill_check(p);
    if (st != KDA_OK) return st;
    if (!cu_ok(cu, n_seqs, total_tokens) || segment_tokens <= 0) return KDA_ERR_INVALID_ARG;
    if (segment_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (n_seqs == 0) return KDA_OK;
    if (S_out == nullptr || ring_out == nullptr || !al16(S_out) || !al16(ring_out)) return KDA_ERR_INVALID_ARG;
    if ((S_in && !al16(S_in)) || (ring_in && !al16(ring_in))) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !z || !b || !gout || !o)) return KDA_ERR_INVALID_ARG;
    const int H = p->num_heads, W = H * D;
    const size_t esize = p->io_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const int64_t seg = std::min(segment_tokens, std::max<int64_t>(total_tokens, 1));
    size_t ws_bytes = 0, set_bytes = 0;
    if (total_tokens > 0) {
        ws_bytes = max_segment_workspace(p, cu, n_seqs, total_tokens, seg);
        set_bytes = stage_layout(H, esize, seg).set;
        if (scratch == nullptr || scratch_bytes < ws_bytes + N_SETS * set_bytes ||
            (reinterpret_cast<uintptr_t>(scratch) % HS_ALIGN))
            return KDA_ERR_WORKSPACE;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    cudaStream_t s_in = h2d_stream_ ? static_cast<cudaStream_t>(h2d_stream_) : s;
    cudaStream_t s_out = d2h_stream_ ? static_cast<cudaStream_t>(d2h_stream_) : s;

    // ---- the state and ring every piece continues from
    const size_t state_bytes = (size_t)n_seqs * H * D * D * sizeof(float);
    const size_t ring_bytes = (size_t)n_seqs * 3 * RING * W * esize;
    cudaError_t e = cudaSuccess;
    if (S_in == nullptr) e = cudaMemsetAsync(S_out, 0, state_bytes, s);
    else if (S_in != S_out) e = cudaMemcpyAsync(S_out, S_in, state_bytes, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (ring_in == nullptr) e = cudaMemsetAsync(ring_out, 0, ring_bytes, s);
    else if (ring_in != ring_out) e = cudaMemcpyAsync(ring_out, ring_in, ring_bytes, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (total_tokens == 0) return KDA_OK;
    char* ws = static_cast<char*>(scratch);
    // the error word covers every segment: cleared once here
    if (cudaMemsetAsync(ws, 0, HS_ALIGN, s) != cudaSuccess) return KDA_ERR_CUDA;

    cudaEvent_t ev[3 * N_SETS + 1] = {};
    for (auto& x : ev)
        if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) st = KDA_ERR_CUDA;
    cudaEvent_t *loaded = ev, *computed = ev + N_SETS, *freed = ev + 2 * N_SETS, start = ev[3 * N_SETS];
    // both copy streams start after the work already on the caller's stream
    if (st == KDA_OK && (cudaEventRecord(start, s) != cudaSuccess || cudaStreamWaitEvent(s_in, start, 0) ||
                         cudaStreamWaitEvent(s_out, start, 0)))
        st = KDA_ERR_CUDA;

    const char* src[6] = {static_cast<const char*>(q), static_cast<const char*>(k), static_cast<const char*>(v),
                          static_cast<const char*>(z), static_cast<const char*>(gout), static_cast<const char*>(b)};
    const size_t row[6] = {W * esize, W * esize, W * esize, W * esize, W * esize, H * esize};
    std::vector<int64_t> sub;
    int32_t first = 0, last = 0;
    for (int64_t t0 = 0, si = 0; st == KDA_OK && t0 < total_tokens; t0 += seg, ++si) {
        const int64_t t1 = std::min(total_tokens, t0 + seg), len = t1 - t0;
        const int j = (int)(si % N_SETS);
        char* set = ws + ws_bytes + (size_t)j * set_bytes;
        const size_t plane = stage_layout(H, esize, seg).plane;
        char* dst[6] = {set, set + plane, set + 2 * plane, set + 3 * plane, set + 4 * plane, set + 6 * plane};
        char* d_o = set + 5 * plane;
        // copy in, once the set's previous output has been read back
        if (si >= N_SETS && cudaStreamWaitEvent(s_in, freed[j], 0) != cudaSuccess) { st = KDA_ERR_CUDA; break; }
        for (int x = 0; x < 6; ++x)
            if (cudaMemcpyAsync(dst[x], src[x] + (size_t)t0 * row[x], (size_t)len * row[x], cudaMemcpyHostToDevice,
                                s_in) != cudaSuccess)
                st = KDA_ERR_CUDA;
        if (st != KDA_OK || cudaEventRecord(loaded[j], s_in) != cudaSuccess) { st = KDA_ERR_CUDA; break; }
        // compute: the pieces of this segment, continuing in place
        segment_pieces(cu, n_seqs, t0, t1, first, last, sub);
        if (cudaStreamWaitEvent(s, loaded[j], 0) != cudaSuccess) { st = KDA_ERR_CUDA; break; }
        float* Sp = S_out + (size_t)first * H * D * D;
        char* rp = static_cast<char*>(ring_out) + (size_t)first * 3 * RING * W * esize;
        st = prefill_run(p, dst[0], dst[1], dst[2], dst[3], dst[5], dst[4], sub.data(), last - first + 1, len, Sp,
                         Sp, rp, rp, d_o, ws, ws_bytes, s, nullptr, false);
        if (st != KDA_OK) break;
        if (cudaEventRecord(computed[j], s) != cudaSuccess) { st = KDA_ERR_CUDA; break; }
        // copy out
        if (cudaStreamWaitEvent(s_out, computed[j], 0) != cudaSuccess ||
            cudaMemcpyAsync(static_cast<char*>(o) + (size_t)t0 * W * esize, d_o, (size_t)len * W * esize,
                            cudaMemcpyDeviceToHost, s_out) != cudaSuccess ||
            cudaEventRecord(freed[j], s_out) != cudaSuccess)
            st = KDA_ERR_CUDA;
    }
    // the caller's stream orders after both copy streams
    if (cudaEventRecord(loaded[0], s_in) != cudaSuccess || cudaStreamWaitEvent(s, loaded[0], 0) != cudaSuccess ||
        cudaEventRecord(freed[0], s_out) != cudaSuccess || cudaStreamWaitEvent(s, freed[0], 0) != cudaSuccess)
        st = KDA_ERR_CUDA;
    for (auto& x : ev)
        if (x) cudaEventDestroy(x);
    return st;
}

}  // extern "C"
