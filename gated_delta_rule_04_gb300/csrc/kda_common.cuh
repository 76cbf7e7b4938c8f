// Device helpers shared by the KDA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int D = 128;      // head_dim (the only width instantiated)
constexpr int CONV_K = 4;   // short conv kernel size
constexpr int RING = 3;     // conv ring slots = CONV_K - 1

// Error words written to the workspace status slot by bounded waits.
constexpr int32_t ERR_NONE = 0;
constexpr int32_t ERR_TIMEOUT = 1;

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }

// ---- 8-channel vector I/O for fp32 and bf16 token tensors ------------------
template <typename T> struct Vec8;

template <> struct Vec8<float> {
    static __device__ __forceinline__ void load(const float* p, float (&x)[8]) {
        float4 a = __ldg(reinterpret_cast<const float4*>(p));
        float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    // shared-memory (or any generic, 16-byte aligned) load without the read-only path
    static __device__ __forceinline__ void lds(const float* p, float (&x)[8]) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&x)[8]) {
        reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
};

template <> struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[8]) {
        uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(h[i]);
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[8]) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};

template <> struct Vec8<__half> {
    static __device__ __forceinline__ void load(const __half* p, float (&x)[8]) {
        uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __half22float2(h[i]);
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__half* p, const float (&x)[8]) {
        uint4 u;
        __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};

// 8 values from shared memory (16-byte aligned) as fp32
__device__ __forceinline__ void lds8(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void lds8(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x; x[2 * i + 1] = f.y;
    }
}

// x * sigmoid(x) and sigmoid(x) with the fast exponential and divide
// (relative error a few ulp; every consumer rounds to fp16/bf16 or compares
// at 1e-4).
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// The decay gate g of channel value z + dt_bias (e_a = exp(A_log)): the
// lower-bounded sigmoid gate (kind 0) or -e_a softplus(z + dt_bias) (kind 1).
__device__ __forceinline__ float decay_gate(int kind, float lb, float e_a, float zb) {
    if (kind == 1) return -e_a * (zb > 20.f ? zb : log1pf(expf(zb)));
    return lb / (1.0f + expf(-e_a * zb));
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Sum over the 16 lanes of a half warp (lanes 0-15 and 16-31 reduce apart).
__device__ __forceinline__ float halfwarp_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One unit of prefill work: `len` tokens of sequence `seq` starting at the
// global token index `t0`; `pos` is t0's index inside its sequence.
struct ChunkDesc {
    int32_t seq;
    int32_t t0;
    int32_t len;
    int32_t pos;
};

}  // namespace kda

// ---- launch wrappers (defined in the per-kernel .cu files) -----------------
namespace kda {

struct PrestageArgs {
    const void *q, *k, *v, *z, *b;
    const float *conv_w, *A_log, *dt_bias;
    const void* ring_in;
    const int64_t* cu;        // device [n+1]
    const ChunkDesc* chunks;  // device [n_chunks]
    int32_t n_chunks, H;
    float lb, l2_eps, q_scale;
    int32_t gate_kind;        // kda_gate
    void *qh, *kh, *vh;       // outputs, fp16 (chunked path) or fp32 (scan path)
    float *gbuf, *beta;       // gate (raw g, or chunk-local cumulative sum) and beta
};

cudaError_t launch_prestage(const PrestageArgs& a, int io_bf16, int out_fp16, int cumsum,
                            cudaStream_t s);

struct RingArgs {
    const void *q, *k, *v;
    const void* ring_in;
    void* ring_out;
    const int64_t* cu;
    int32_t n_seqs, W;
};
cudaError_t launch_ring_update(const RingArgs& a, int io_bf16, cudaStream_t s);

struct ScanArgs {
    const float *qh, *kh, *vh, *g, *beta;
    const float* S_in;
    float* S_out;
    float* o_core;
    const int64_t* cu;
    int32_t n_seqs, H;
};
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);

struct EpilogueArgs {
    const float* o_core;
    const void* gout;
    const float* norm_w;
    void* o;
    int64_t T;
    int32_t H;
    float eps;
};
cudaError_t launch_epilogue(const EpilogueArgs& a, int io_bf16, cudaStream_t s);

bool chunked_kernel_built();

struct DecodeArgs {
    const void *q, *k, *v, *z, *b, *gout;   // [n][n_tok][H*128]; b [n][n_tok][H]
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    const int32_t* slots;                   // [n] state-pool slot per session, or NULL (slot = session)
    const float* S_in;                      // pools [n_slots][H][128][128]; S_out may alias S_in
    float* S_out;
    const void* ring_in;                    // pools [n_slots][3][3][H*128]; ring_out may alias ring_in
    void* ring_out;
    void* o;                                // [n][n_tok][H*128]
    int32_t n, H, n_tok, n_slots;
    float lb, l2_eps, norm_eps, q_scale;
    int32_t gate_kind;                      // kda_gate
};
cudaError_t launch_decode(const DecodeArgs& a, int io_bf16, cudaStream_t s);

// Prefill metadata built on the device from values passed as kernel
// arguments (no host-to-device copy): for a slice of up to META_SEQS sequences
// seq0 .. seq0 + n - 1, their token offsets, first chunk index, order entry and
// the ChunkDesc of each 64-token chunk.  pos_base is added to every chunk's
// position in its sequence (the start of a window inside one sequence).  Any
// output pointer may be null to skip it; `tail` also writes the entries of
// index seq0 + n of cu and chunk_off.
constexpr int META_SEQS = 1024;
struct MetaSlice {
    int64_t cu[META_SEQS + 1];
    int32_t order[META_SEQS];
    int32_t n, seq0, tail;
    int64_t chunk0, pos_base;
    int64_t* d_cu;
    int64_t* d_coff;
    int32_t* d_order;
    ChunkDesc* d_chunks;
};
cudaError_t launch_build_meta(const MetaSlice& m, cudaStream_t s);
// The whole table for n sequences with host offsets cu[0..n] (cu[0] may be
// nonzero) and an optional host order[n], in slices of META_SEQS.
cudaError_t build_meta(const int64_t* cu, const int32_t* order, int32_t n, int64_t pos_base, int64_t* d_cu,
                       int64_t* d_coff, int32_t* d_order, ChunkDesc* d_chunks, cudaStream_t s);

// The metadata of the overlapped windows of one T-token sequence (S windows of
// `seg` tokens, blocks of `stride` bytes at `meta`) and the sequence's cu {0, T}.
cudaError_t launch_build_window_meta(int64_t T, int64_t seg, int32_t S, int64_t stride, unsigned char* meta,
                                     int64_t* cufull, cudaStream_t s);

// The parameter checks of kda_prefill: KDA_OK or the status it would return.
kda_status prefill_check(const kda_params* p);

// The checks and launch sequence of kda_prefill (ev: optional stage events).
// reset_status = false leaves the workspace's error word as earlier calls
// left it, so a caller that runs one problem as several calls on one
// workspace reads the timeouts of all of them.
kda_status prefill_run(const kda_params* p, const void* q, const void* k, const void* v, const void* z,
                       const void* b, const void* gout, const int64_t* cu_seqlens_host, int32_t n_seqs,
                       int64_t total_tokens, const float* S_in, float* S_out, const void* ring_in, void* ring_out,
                       void* o, void* workspace, size_t workspace_bytes, void* stream, void* const* ev,
                       bool reset_status);

}  // namespace kda
