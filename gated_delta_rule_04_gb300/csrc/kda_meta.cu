// Prefill metadata built on the device: token offsets, first chunk of each
// sequence, the sequence order of the recurrence's CTAs and the chunk table,
// from cu_seqlens (and the order) passed by value as kernel arguments.  The
// host never copies pageable memory to the device for them, so a call stays
// asynchronous.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int MT = 256;        // threads per block
constexpr int MCHUNK = 64;     // tokens per chunk

// Every block recomputes the chunk prefix of the slice's sequences in shared
// memory (at most META_SEQS of them); thread g of the grid then writes chunk g
// of the slice, and block 0 also writes the per-sequence entries.
__global__ void __launch_bounds__(MT) build_meta_kernel(const __grid_constant__ MetaSlice m) {
    __shared__ int64_t pref[META_SEQS + 1];
    __shared__ int64_t part[MT];
    const int tid = threadIdx.x;
    // per-thread sums of chunk counts over a contiguous range of sequences, then a scan
    constexpr int PER = (META_SEQS + MT - 1) / MT;
    int64_t loc[PER];
    int64_t sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = tid * PER + j;
        const int64_t c = i < m.n ? (m.cu[i + 1] - m.cu[i] + MCHUNK - 1) / MCHUNK : 0;
        loc[j] = c;
        sum += c;
    }
    part[tid] = sum;
    __syncthreads();
    for (int off = 1; off < MT; off <<= 1) {   // inclusive Hillis-Steele scan of the partial sums
        const int64_t v = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    int64_t run = part[tid] - sum;              // exclusive prefix of this thread's range
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int i = tid * PER + j;
        if (i <= m.n) pref[i] = run;
        run += loc[j];
    }
    if (tid == MT - 1 && MT * PER <= m.n) pref[m.n] = run;   // (m.n <= META_SEQS = MT * PER)
    __syncthreads();
    const int64_t total = pref[m.n];
    if (blockIdx.x == 0) {
        for (int i = tid; i < m.n + (m.tail ? 1 : 0); i += MT) {
            if (m.d_cu) m.d_cu[m.seq0 + i] = m.cu[i];
            if (m.d_coff) m.d_coff[m.seq0 + i] = m.chunk0 + pref[i];
            if (m.d_order && i < m.n) m.d_order[m.seq0 + i] = m.order[i];
        }
    }
    if (m.d_chunks == nullptr) return;
    for (int64_t g = (int64_t)blockIdx.x * MT + tid; g < total; g += (int64_t)gridDim.x * MT) {
        int lo = 0, hi = m.n - 1;               // the sequence i with pref[i] <= g < pref[i + 1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pref[mid] <= g) lo = mid; else hi = mid - 1;
        }
        const int64_t t0 = m.cu[lo] + MCHUNK * (g - pref[lo]);
        const int64_t len = m.cu[lo + 1] - t0 < MCHUNK ? m.cu[lo + 1] - t0 : MCHUNK;
        m.d_chunks[m.chunk0 + g] =
            ChunkDesc{m.seq0 + lo, (int32_t)t0, (int32_t)len, (int32_t)(t0 - m.cu[lo] + m.pos_base)};
    }
}

}  // namespace

cudaError_t launch_build_meta(const MetaSlice& m, cudaStream_t s) {
    if (m.n < 0 || m.n > META_SEQS) return cudaErrorInvalidValue;
    int64_t chunks = 0;
    for (int i = 0; i < m.n; ++i) chunks += (m.cu[i + 1] - m.cu[i] + MCHUNK - 1) / MCHUNK;
    int64_t blocks = (chunks + MT - 1) / MT;
    if (blocks < 1) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    build_meta_kernel<<<(unsigned)blocks, MT, 0, s>>>(m);
    return cudaGetLastError();
}

cudaError_t build_meta(const int64_t* cu, const int32_t* order, int32_t n, int64_t pos_base, int64_t* d_cu,
                       int64_t* d_coff, int32_t* d_order, ChunkDesc* d_chunks, cudaStream_t s) {
    MetaSlice m;
    m.pos_base = pos_base;
    m.d_cu = d_cu;
    m.d_coff = d_coff;
    m.d_order = d_order;
    m.d_chunks = d_chunks;
    int64_t chunk0 = 0;
    int32_t seq0 = 0;
    do {
        const int32_t k = n - seq0 < META_SEQS ? n - seq0 : META_SEQS;
        m.n = k;
        m.seq0 = seq0;
        m.tail = seq0 + k == n;
        m.chunk0 = chunk0;
        for (int32_t i = 0; i <= k; ++i) m.cu[i] = cu[seq0 + i];
        for (int32_t i = 0; i < k; ++i) m.order[i] = order ? order[seq0 + i] : seq0 + i;
        cudaError_t e = launch_build_meta(m, s);
        if (e != cudaSuccess) return e;
        for (int32_t i = 0; i < k; ++i) chunk0 += (cu[seq0 + i + 1] - cu[seq0 + i] + MCHUNK - 1) / MCHUNK;
        seq0 += k;
    } while (seq0 < n);
    return cudaSuccess;
}

}  // namespace kda

namespace kda {
namespace {

// Metadata of the overlapped windows of one T-token sequence: window w covers
// tokens [w seg, min(T, (w + 1) seg)); its block of `stride` bytes holds
// {t0, t1, 0, nck} (int64) and its chunk table, with chunk positions taken in
// the whole sequence.  Thread 0 also writes the whole sequence's cu {0, T}.
__global__ void __launch_bounds__(MT) build_window_meta_kernel(int64_t T, int64_t seg, int32_t S, int64_t stride,
                                                               unsigned char* meta, int64_t* cufull) {
    const int64_t seg_chunks = seg / MCHUNK;
    const int64_t g = (int64_t)blockIdx.x * MT + threadIdx.x;
    if (g == 0) {
        cufull[0] = 0;
        cufull[1] = T;
    }
    if (g >= (int64_t)S * seg_chunks) return;
    const int64_t w = g / seg_chunks, i = g % seg_chunks;
    const int64_t t0 = w * seg, t1 = t0 + seg < T ? t0 + seg : T;
    const int64_t nck = (t1 - t0 + MCHUNK - 1) / MCHUNK;
    int64_t* m = reinterpret_cast<int64_t*>(meta + w * stride);
    if (i == 0) {
        m[0] = t0; m[1] = t1; m[2] = 0; m[3] = nck;
    }
    if (i < nck) {
        const int64_t t = t0 + MCHUNK * i;
        reinterpret_cast<ChunkDesc*>(m + 4)[i] =
            ChunkDesc{0, (int32_t)t, (int32_t)(t1 - t < MCHUNK ? t1 - t : MCHUNK), (int32_t)t};
    }
}

}  // namespace

cudaError_t launch_build_window_meta(int64_t T, int64_t seg, int32_t S, int64_t stride, unsigned char* meta,
                                     int64_t* cufull, cudaStream_t s) {
    const int64_t n = (int64_t)S * (seg / MCHUNK);
    const int64_t blocks = n > 0 ? (n + MT - 1) / MT : 1;
    build_window_meta_kernel<<<(unsigned)blocks, MT, 0, s>>>(T, seg, S, stride, meta, cufull);
    return cudaGetLastError();
}

}  // namespace kda
