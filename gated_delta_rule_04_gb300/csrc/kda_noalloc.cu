// kda_prefill_noalloc: the prefill for callers that may not allocate memory.
//
// kda_prefill asks its caller for a workspace.  Some callers cannot provide
// one on demand: code whose device memory is fully planned up front (a plugin
// inside an inference engine that owns every byte, a serving loop whose
// memory plan is fixed at start-up) and code that must not call cudaMalloc or
// cudaFree, which can synchronise the whole device and stall every other
// stream.  This entry point takes the same inputs and outputs as kda_prefill
// but no workspace: its scratch is a fixed array in device memory that every
// GPU which loads this library holds until the process exits.  It calls no
// memory-allocating routine, on the device or on the host.
//
// Set-up: the first call in each CUDA context (one per device for runtime-API
// callers) looks up the array's device address with cudaGetSymbolAddress,
// with that device current, and caches it with the context it belongs to;
// make that first call before any stream capture.
// Sharing: every call uses the same array and leaves its contents behind.
// The only part that must start at zero (the error word) is cleared by each
// call; every other byte is written before it is read.  Calls whose work can
// overlap on the GPU (concurrent streams, or host threads on one device)
// race on the array: order them on one stream.
#include <string.h>

#include <mutex>

#include "kda_chunk_layout.cuh"

namespace kda {
namespace {

constexpr size_t NA_ALIGN = 256;
constexpr int NA_CHUNK = CHUNK_T;
constexpr int NA_MAX_DEVICES = 64;
constexpr int NA_MAX_SEQS = 512;           // sequences per call (their order is sorted on the stack)

// The scratch array.  In host code this name is only a handle for
// cudaGetSymbolAddress, never an address to pass to a kernel.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// The cached address per device, with the context it was looked up in: a
// cudaDeviceReset (or another context on the device) invalidates it.
struct ScratchSlot {
    void* ctx;
    void* addr;
};
ScratchSlot g_scratch[NA_MAX_DEVICES];
std::mutex g_scratch_mu;

typedef int (*CtxGetCurrentFn)(void**);   // CUresult cuCtxGetCurrent(CUcontext*)
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<CtxGetCurrentFn>(nullptr);
        return reinterpret_cast<CtxGetCurrentFn>(f);
    }();
    return fn;
}

size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct NaLayout {
    size_t status, meta, meta_bytes, off_coff, off_order, off_chunks;
    size_t qh, kh, vh, g, beta, ocore, rec, total;
};

// Same region order as the caller-provided workspace of kda_prefill.
NaLayout na_layout(int H, bool chunked, int32_t n, int64_t T, int64_t nc) {
    NaLayout L{};
    const size_t W = (size_t)H * D, op = 4;
    const size_t tw = chunked ? 0 : (size_t)T * W;  // pre-stage outputs: scan path only
    size_t off = 0;
    L.status = off; off += NA_ALIGN;
    L.meta = off;
    L.off_coff = sizeof(int64_t) * (size_t)(n + 1);
    L.off_order = L.off_coff + sizeof(int64_t) * (size_t)(n + 1);
    L.off_chunks = up(L.off_order + sizeof(int32_t) * (size_t)n, 16);
    L.meta_bytes = L.off_chunks + sizeof(ChunkDesc) * (size_t)nc;
    off = up(off + L.meta_bytes, NA_ALIGN);
    L.qh = off; off = up(off + op * tw, NA_ALIGN);
    L.kh = off; off = up(off + op * tw, NA_ALIGN);
    L.vh = off; off = up(off + op * tw, NA_ALIGN);
    L.g = off; off = up(off + 4 * tw, NA_ALIGN);
    L.beta = off; off = up(off + 4 * (chunked ? 0 : (size_t)T * H), NA_ALIGN);
    L.ocore = off;
    off = up(off + 4 * tw, NA_ALIGN);
    L.rec = off;
    if (chunked) off = up(off + (size_t)REC_BYTES * (size_t)nc * H, NA_ALIGN);
    L.total = off;
    return L;
}

// Device address of the scratch array in the current context (looked up once
// per context).
cudaError_t scratch_address(unsigned char** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= NA_MAX_DEVICES) return cudaErrorInvalidDevice;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (get_ctx == nullptr) return cudaErrorDeviceUninitialized;
    void* ctx = nullptr;
    if (get_ctx(&ctx) != 0) return cudaErrorDeviceUninitialized;
    if (ctx == nullptr) {
        // no context current yet: the runtime's symbol lookup makes the device's
        // primary context current
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (get_ctx(&ctx) != 0 || ctx == nullptr) return cudaErrorDeviceUninitialized;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchSlot& sl = g_scratch[dev];
    if (sl.ctx != ctx || sl.addr == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        sl.ctx = ctx;
        sl.addr = p;
    }
    *out = static_cast<unsigned char*>(sl.addr);
    return cudaSuccess;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_prefill_noalloc(const kda_params* p, const void* q, const void* k, const void* v,
                                          const void* z, const void* b, const void* gout,
                                          const int64_t* cu, int32_t n_seqs, int64_t total_tokens,
                                          const float* S_in, float* S_out, const void* ring_in, void* ring_out,
                                          void* o, void* stream_) {
    // the parameter checks and the algorithm choice of kda_prefill, with its statuses
    const kda_status pst = prefill_check(p);
    if (pst != KDA_OK) return pst;
    const bool chunked = kda_prefill_algo(p) == KDA_ALGO_CHUNKED;
    if (n_seqs < 0 || total_tokens < 0 || cu == nullptr) return KDA_ERR_INVALID_ARG;
    if (cu[0] != 0 || cu[n_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_seqs; ++i)
        if (cu[i + 1] < cu[i]) return KDA_ERR_INVALID_ARG;
    if (n_seqs == 0) return KDA_OK;
    if (total_tokens > 0) {
        const void* tok[6] = {q, k, v, z, gout, o};
        for (int i = 0; i < 6; ++i)
            if (tok[i] == nullptr || !al16(tok[i])) return KDA_ERR_INVALID_ARG;
        if (b == nullptr) return KDA_ERR_INVALID_ARG;
    }
    if (S_out == nullptr || !al16(S_out) || (S_in && !al16(S_in))) return KDA_ERR_INVALID_ARG;
    if ((ring_in && !al16(ring_in)) || (ring_out && !al16(ring_out))) return KDA_ERR_INVALID_ARG;

    // size limits of the fixed scratch and of the on-stack sequence order
    int64_t nc = 0;
    for (int32_t i = 0; i < n_seqs; ++i) nc += (cu[i + 1] - cu[i] + NA_CHUNK - 1) / NA_CHUNK;
    const int H = p->num_heads, W = H * D;
    if (n_seqs > NA_MAX_SEQS) return KDA_ERR_UNSUPPORTED;
    if (total_tokens > (int64_t)INT32_MAX) return KDA_ERR_UNSUPPORTED;   // (as kda_prefill)
    const NaLayout L = na_layout(H, chunked, n_seqs, total_tokens, nc);
    if (L.total > KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;

    unsigned char* ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return KDA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream_);

    // longest sequences first (insertion sort on the stack: stable, no allocation)
    int32_t order[NA_MAX_SEQS];
    for (int32_t i = 0; i < n_seqs; ++i) order[i] = i;
    for (int32_t i = 1; i < n_seqs; ++i) {
        const int32_t x = order[i];
        const int64_t lx = cu[x + 1] - cu[x];
        int32_t j = i - 1;
        while (j >= 0 && cu[order[j] + 1] - cu[order[j]] < lx) { order[j + 1] = order[j]; --j; }
        order[j + 1] = x;
    }
    const int64_t* d_cu = reinterpret_cast<const int64_t*>(ws + L.meta);
    const int64_t* d_coff = reinterpret_cast<const int64_t*>(ws + L.meta + L.off_coff);
    const int32_t* d_order = reinterpret_cast<const int32_t*>(ws + L.meta + L.off_order);
    const ChunkDesc* d_chunks = reinterpret_cast<const ChunkDesc*>(ws + L.meta + L.off_chunks);
    cudaError_t e = cudaMemsetAsync(ws + L.status, 0, NA_ALIGN, s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    // cu_seqlens, chunk offsets, order and chunk table, built on the device from
    // kernel arguments
    e = build_meta(cu, order, n_seqs, 0, const_cast<int64_t*>(d_cu), const_cast<int64_t*>(d_coff),
                   const_cast<int32_t*>(d_order), const_cast<ChunkDesc*>(d_chunks), s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;

    const int io_bf16 = p->io_dtype == KDA_DTYPE_BF16;
    const float qs = p->q_scale != 0.f ? p->q_scale : 1.0f / sqrtf((float)D);
    float* gbuf = reinterpret_cast<float*>(ws + L.g);
    float* beta = reinterpret_cast<float*>(ws + L.beta);
    float* ocore = reinterpret_cast<float*>(ws + L.ocore);
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    PrestageArgs pa{q, k, v, z, b, p->conv_w, p->A_log, p->dt_bias, ring_in, d_cu, d_chunks,
                    (int32_t)nc, H, p->gate_lower_bound, p->l2_eps, qs, p->gate_kind,
                    ws + L.qh, ws + L.kh, ws + L.vh, gbuf, beta};
    if (!chunked) {
        if (launch_prestage(pa, io_bf16, 0, 0, s) != cudaSuccess) return KDA_ERR_CUDA;
        ScanArgs sa{reinterpret_cast<const float*>(ws + L.qh), reinterpret_cast<const float*>(ws + L.kh),
                    reinterpret_cast<const float*>(ws + L.vh), gbuf, beta, S_in, S_out, ocore, d_cu,
                    n_seqs, H};
        if (launch_scan(sa, s) != cudaSuccess) return KDA_ERR_CUDA;
    } else {
        PrepArgs pr{q, k, v, z, b, ring_in, p->conv_w, p->A_log, p->dt_bias, p->gate_lower_bound, p->l2_eps, qs,
                    d_chunks, (int32_t)nc, H, total_tokens, ws + L.rec, status, nullptr, PREP_BATCH, prep_wait_limit_ns(p), {}, {}, p->gate_kind};
        if (launch_chunk_prep(pr, s) != cudaSuccess) return KDA_ERR_CUDA;
        ChunkRecArgs ca{ws + L.rec, S_in, S_out, gout, p->norm_w, o, p->norm_eps, d_cu, d_coff, d_order, status,
                        n_seqs, H};
        if (launch_chunk_recurrence(ca, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (!chunked) {
        EpilogueArgs ea{ocore, gout, p->norm_w, o, total_tokens, H, p->norm_eps};
        if (launch_epilogue(ea, io_bf16, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (ring_out) {
        RingArgs ra{q, k, v, ring_in, ring_out, d_cu, n_seqs, W};
        if (launch_ring_update(ra, io_bf16, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

// Reads (and clears) the error word of the scratch array, as kda_workspace_status
// does for a caller's workspace.
extern "C" kda_status kda_noalloc_status(void* stream_) {
    unsigned char* ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return KDA_ERR_CUDA;
    return kda_workspace_status(ws, stream_);
}
