// Fused pre-stage of the KDA prefill (one CTA per (chunk, head)):
//   short causal conv (kernel 4) + SiLU on q, k, v; L2 norm of q and k with
//   q scaled by q_scale; lower-bounded decay gate; beta = sigmoid(b).
// Sources: "Kimi Delta Attention (KDA) -- analysis & C kernel plan", section
// "The KDA layer, precisely"; "ferrox-models 0.8.0, module kda", module
// overview (L2 eps 1e-6, q * head_dim^-0.5, depthwise causal Conv1d);
// "Kimi K3 - Retention gate - OpenModelAtlas" (g = lb*sigmoid(e^A (z + b))).
//
// Layout: the CTA stages the raw q/k/v rows t0-3 .. t0+len-1 of its head
// (128 channels) in shared memory with cp.async, taking rows before the
// sequence start from the conv ring.  Each half warp then owns four
// consecutive tokens and 8 channels (16-byte vectors).  With `cumsum` the gate
// is written as the inclusive cumulative sum inside the chunk (the chunked
// prefill's per-channel log decay); otherwise the raw gate is written.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int PS_THREADS = 256;
constexpr int PS_MAXLEN = 64;      // tokens per chunk (16 half warps x 4)
constexpr int PS_ROWS = PS_MAXLEN + RING;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(PS_THREADS, 2) prestage_kernel(PrestageArgs a, int cumsum) {
    constexpr int VEC = 16 / sizeof(TI);          // elements per 16-byte vector
    constexpr int VPR = D / VEC;                  // vectors per 128-channel row
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TI* xs = reinterpret_cast<TI*>(smem_raw);     // [3][PS_ROWS][D]
    float* tot = reinterpret_cast<float*>(smem_raw + sizeof(TI) * 3 * PS_ROWS * D);  // [16][D]
    float* cw = tot + 16 * D;                     // [3][D][4] conv weights of this head
    TI* zs = reinterpret_cast<TI*>(cw + 3 * D * CONV_K);  // [PS_MAXLEN][D] gate inputs

    const int item = blockIdx.x;
    const int H = a.H, W = H * D;
    const int chunk = item / H, h = item % H;
    const ChunkDesc cd = a.chunks[chunk];
    const int len = cd.len;
    const int rows = len + RING;
    const int tid = threadIdx.x;
    const TI* planes[3] = {static_cast<const TI*>(a.q), static_cast<const TI*>(a.k),
                           static_cast<const TI*>(a.v)};
    const TI* ring = static_cast<const TI*>(a.ring_in);

    // ---- phase 1: stage raw rows (row r holds local token pos + r - 3)
    for (int idx = tid; idx < 3 * rows * VPR; idx += PS_THREADS) {
        const int p = idx / (rows * VPR);
        const int rem = idx - p * rows * VPR;
        const int r = rem / VPR, vv = rem - r * VPR;
        TI* dst = xs + ((size_t)p * PS_ROWS + r) * D + vv * VEC;
        const int local = cd.pos + r - RING;  // index inside the sequence
        const int ch = h * D + vv * VEC;
        if (local >= 0) {
            cp_async16(dst, planes[p] + (size_t)(cd.t0 + r - RING) * W + ch);
        } else if (ring != nullptr) {
            cp_async16(dst, ring + (((size_t)cd.seq * 3 + p) * RING + (RING + local)) * W + ch);
        } else {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
    }

    for (int idx = tid; idx < 3 * D; idx += PS_THREADS) {  // conv weights: one 16-byte row per channel
        const int p = idx / D, c = idx % D;
        cp_async16(cw + 4 * idx, a.conv_w + ((size_t)p * W + h * D + c) * CONV_K);
    }

    // gate inputs of the chunk's tokens, staged with the same copies
    for (int idx = tid; idx < len * VPR; idx += PS_THREADS) {
        const int r = idx / VPR, vv = idx - r * VPR;
        cp_async16(zs + (size_t)r * D + vv * VEC, static_cast<const TI*>(a.z) + (size_t)(cd.t0 + r) * W + h * D + vv * VEC);
    }
    const int hw = tid >> 4, l16 = tid & 15;
    const int cb = l16 * 8;                       // first channel (inside the head)
    float dtb[8];
    Vec8<float>::load(a.dt_bias + h * D + cb, dtb);
    const float eA = expf(a.A_log[h]);
    if (tid < len) {
        const float bl = to_f32(static_cast<const TI*>(a.b)[(size_t)(cd.t0 + tid) * H + h]);
        a.beta[(size_t)(cd.t0 + tid) * H + h] = 1.0f / (1.0f + expf(-bl));
    }

    cp_async_wait_all();
    __syncthreads();

    // ---- phase 2: conv + SiLU + norms, four consecutive tokens per half warp
    TO* outs[3] = {static_cast<TO*>(a.qh), static_cast<TO*>(a.kh), static_cast<TO*>(a.vh)};
#pragma unroll 1
    for (int p = 0; p < 3; ++p) {
        float wt[8][4];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 w4 = *reinterpret_cast<const float4*>(cw + 4 * (p * D + cb + e));
            wt[e][0] = w4.x; wt[e][1] = w4.y; wt[e][2] = w4.z; wt[e][3] = w4.w;
        }
        float win[7][8];  // smem rows hw*4 .. hw*4+6 = tokens hw*4-3 .. hw*4+3
#pragma unroll
        for (int r = 0; r < 7; ++r) {
            const int row = hw * 4 + r;
            if (row < rows) {
                lds8(xs + ((size_t)p * PS_ROWS + row) * D + cb, win[r]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) win[r][e] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int tau = hw * 4 + j;
            float y[8];
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float acc = wt[e][0] * win[j][e];
                acc = fmaf(wt[e][1], win[j + 1][e], acc);
                acc = fmaf(wt[e][2], win[j + 2][e], acc);
                acc = fmaf(wt[e][3], win[j + 3][e], acc);
                y[e] = silu_fast(acc);
                ss = fmaf(y[e], y[e], ss);
            }
            if (p < 2) {
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                float r = rsqrtf(ss + a.l2_eps);
                if (p == 0) r *= a.q_scale;
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] *= r;
            }
            if (tau < len) Vec8<TO>::store(outs[p] + (size_t)(cd.t0 + tau) * W + h * D + cb, y);
        }
    }

    // ---- gate (and its cumulative sum inside the chunk)
    float gv[4][8];
    float run[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) run[e] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int tau = hw * 4 + j;
        float z8[8];
        if (tau < len) lds8(zs + (size_t)tau * D + cb, z8);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float g = tau < len ? decay_gate(a.gate_kind, a.lb, eA, z8[e] + dtb[e]) : 0.f;
            run[e] += g;
            gv[j][e] = cumsum ? run[e] : g;
        }
    }
    if (cumsum) {
        Vec8<float>::store(tot + hw * D + cb, run);
        __syncthreads();
        float pre[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pre[e] = 0.f;
        for (int k = 0; k < hw; ++k) {
            float t8[8];
            const float4 a0 = *reinterpret_cast<const float4*>(tot + k * D + cb);
            const float4 a1 = *reinterpret_cast<const float4*>(tot + k * D + cb + 4);
            t8[0] = a0.x; t8[1] = a0.y; t8[2] = a0.z; t8[3] = a0.w;
            t8[4] = a1.x; t8[5] = a1.y; t8[6] = a1.z; t8[7] = a1.w;
#pragma unroll
            for (int e = 0; e < 8; ++e) pre[e] += t8[e];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) gv[j][e] += pre[e];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int tau = hw * 4 + j;
        if (tau < len) Vec8<float>::store(a.gbuf + (size_t)(cd.t0 + tau) * W + h * D + cb, gv[j]);
    }
}

// Final conv ring of each sequence: slot s holds the raw input at local index
// L-3+s, taken from ring_in (or zero) when that index is negative.  Each
// thread reads all three of its old slots before writing, so ring_out may
// alias ring_in.
template <typename TI>
__global__ void ring_update_kernel(RingArgs a) {
    constexpr int VEC = 16 / sizeof(TI);
    const int vpr = a.W / VEC;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)a.n_seqs * 3 * vpr;
    if (idx >= total) return;
    const int n = (int)(idx / (3 * vpr));
    const int rem = (int)(idx - (int64_t)n * 3 * vpr);
    const int p = rem / vpr, vv = rem - p * vpr;
    const int64_t bos = a.cu[n], L = a.cu[n + 1] - bos;
    const TI* plane = static_cast<const TI*>(p == 0 ? a.q : (p == 1 ? a.k : a.v));
    const TI* rin = static_cast<const TI*>(a.ring_in);
    TI* rout = static_cast<TI*>(a.ring_out);
    uint4 vals[RING];
#pragma unroll
    for (int s = 0; s < RING; ++s) {
        const int64_t src = L - RING + s;
        if (src >= 0)
            vals[s] = *reinterpret_cast<const uint4*>(plane + (size_t)(bos + src) * a.W + vv * VEC);
        else if (rin != nullptr)
            vals[s] = *reinterpret_cast<const uint4*>(rin + (((size_t)n * 3 + p) * RING + (RING + src)) * a.W + vv * VEC);
        else
            vals[s] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int s = 0; s < RING; ++s)
        *reinterpret_cast<uint4*>(rout + (((size_t)n * 3 + p) * RING + s) * a.W + vv * VEC) = vals[s];
}

template <typename TI, typename TO>
cudaError_t launch_prestage_t(const PrestageArgs& a, int cumsum, cudaStream_t s) {
    const size_t smem = sizeof(TI) * 3 * PS_ROWS * D + sizeof(float) * 16 * D + sizeof(float) * 3 * D * CONV_K +
                        sizeof(TI) * PS_MAXLEN * D;
    cudaError_t e = cudaFuncSetAttribute(prestage_kernel<TI, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.n_chunks * a.H;
    if (blocks == 0) return cudaSuccess;
    prestage_kernel<TI, TO><<<(unsigned)blocks, PS_THREADS, smem, s>>>(a, cumsum);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prestage(const PrestageArgs& a, int io_bf16, int out_fp16, int cumsum,
                            cudaStream_t s) {
    if (io_bf16) {
        return out_fp16 ? launch_prestage_t<__nv_bfloat16, __half>(a, cumsum, s)
                        : launch_prestage_t<__nv_bfloat16, float>(a, cumsum, s);
    }
    return out_fp16 ? launch_prestage_t<float, __half>(a, cumsum, s)
                    : launch_prestage_t<float, float>(a, cumsum, s);
}

cudaError_t launch_ring_update(const RingArgs& a, int io_bf16, cudaStream_t s) {
    const int vec = io_bf16 ? 8 : 4;
    const int64_t total = (int64_t)a.n_seqs * 3 * (a.W / vec);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((total + threads - 1) / threads);
    if (io_bf16) ring_update_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(a);
    else ring_update_kernel<float><<<blocks, threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
