// Chunk recurrence of the chunked prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory).  One CTA per (sequence, head)
// walks the sequence's 64-token chunks in order; the 128 x 128 fp32 state
// never leaves the SM.
//
// Per chunk, with the operands prepared by the chunk-preparation kernel
// (W, Q+, Kt, U0, P, decay; see kda_chunk_prep.cu) and S the state at the
// chunk start (the inter-chunk step of the chunked UT form, "memra-engine
// 0.124.0, module kda", PREFILL DISPATCH):
//   U   = U0 - W S
//   O   = Q+ S + P U
//   S'  = Diag(decay) S + Kt^T U
// Everything is computed transposed so that every MMA has M = 128 (the value
// dimension) and the state lives in TMEM as S^T (lane = value index, column
// = key index):
//   MMA1  D[:, 0:64]   = S^T W^T           (A = S^T fp16 copy, B = W)
//         D[:, 64:128] = S^T Q+^T          (B = Q+)
//   SIMT  U^T = U0^T - D[:, 0:64]  -> fp16 tile
//   MMA2  S^T += U^T Kt                     (onto the decayed state, B = Kt^T tile)
//   MMA3  D[:, 64:128] += U^T P^T           (B = P)
//   SIMT  O^T = D[:, 64:128] -> o_core ; S^T -> fp16 copy, scaled by next decay
// Each chunk's record arrives with one bulk copy into a two-stage ring, two
// chunks ahead of use.  Every wait is bounded; on timeout the kernel records
// KDA timeout in the workspace status word, drains its own copies and
// returns after freeing its tensor memory.
#include "kda_chunk_layout.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int NT = 128;                 // 4 warps: thread t <-> TMEM lane t <-> value index t
constexpr uint32_t TMEM_COLS = 256;     // [0,128) state S^T, [128,256) D
constexpr uint32_t STAGE_STRIDE = 75776;  // REC_BYTES rounded up to 1 KiB
constexpr uint32_t OFF_ST = 2 * STAGE_STRIDE;      // S^T fp16, 2 panels x 128 rows x 128 B
constexpr uint32_t OFF_UT = OFF_ST + 32768;        // U^T fp16, 1 panel x 128 rows x 128 B
constexpr uint32_t OFF_BAR = OFF_UT + 16384;       // 3 mbarriers + TMEM slot + flags
constexpr uint32_t SMEM_BYTES = OFF_BAR + 128 + 1024;  // + slack for 1 KiB alignment
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s

constexpr uint32_t IDESC_N64 = ptx::idesc_f16_f32(128, 64);
constexpr uint32_t IDESC_N128 = ptx::idesc_f16_f32(128, 128);

__device__ __forceinline__ uint4 pack8_f16(const float* v) {
    uint4 u;
    __half2* p = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
    return u;
}

__global__ void __launch_bounds__(NT, 1) chunk_recurrence_kernel(ChunkRecArgs a) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sb = smem_raw + (base - raw);
    const uint32_t bar_load[2] = {base + OFF_BAR, base + OFF_BAR + 8};
    const uint32_t bar_mma = base + OFF_BAR + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sb + OFF_BAR + 32);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sb + OFF_BAR + 36);
    int* pend = reinterpret_cast<int*>(sb + OFF_BAR + 40);  // [0],[1] load pending per stage, [2] mma pending

    const int tid = threadIdx.x, warp = tid >> 5;
    const int H = a.H, W = H * D;
    const int n = a.seq_order ? a.seq_order[blockIdx.x / H] : (int)(blockIdx.x / H);
    const int h = blockIdx.x % H;
    const int64_t c0 = a.chunk_off[n];
    const int64_t nc = a.chunk_off[n + 1] - c0;
    const int64_t bos = a.cu[n], L = a.cu[n + 1] - bos;

    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(bar_load[0], 1);
        ptx::mbar_init(bar_load[1], 1);
        ptx::mbar_init(bar_mma, 1);
        *abort_flag = 0;
        pend[0] = pend[1] = pend[2] = 0;
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane;         // this warp's lanes, state columns
    const uint32_t tD = tmem + lane + 128;   // this warp's lanes, D columns

    const unsigned char* recs = static_cast<const unsigned char*>(a.records);
    auto issue_load = [&](int64_t c) {
        const int s = (int)(c & 1);
        ptx::mbar_expect_tx(bar_load[s], REC_BYTES);
        ptx::bulk_g2s(base + s * STAGE_STRIDE, recs + ((size_t)(c0 + c) * H + h) * REC_BYTES, REC_BYTES,
                      bar_load[s]);
        pend[s] = 1;
    };
    if (tid == 0) {
        for (int64_t c = 0; c < nc && c < 2; ++c) issue_load(c);
    }

    // initial state: S^T into TMEM (thread t holds value column t, all keys)
    const size_t soff = ((size_t)n * H + h) * D * D;
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
        float v[32];
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] = a.S_in ? a.S_in[soff + (size_t)(32 * j + x) * D + tid] : 0.f;
        ptx::tmem_st32(tS + 32 * j, v);
    }

    uint32_t mma_phase = 0;
    uint32_t load_phase[2] = {0, 0};
    float* o_core = a.o_core;
#pragma unroll 1
    for (int64_t c = 0; c < nc; ++c) {
        const int s = (int)(c & 1);
        const uint32_t stg = base + s * STAGE_STRIDE;
        const unsigned char* sp = sb + s * STAGE_STRIDE;
        const int64_t rem = L - (int64_t)CHUNK_T * c;
        const int Lc = rem < CHUNK_T ? (int)rem : CHUNK_T;

        if (!ptx::mbar_wait(bar_load[s], load_phase[s], WAIT_LIMIT_NS)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) break;
        load_phase[s] ^= 1;
        if (tid == 0) pend[s] = 0;

        // ---- state transition: fp16 copy of S^T for MMA1, then S^T *= decay (per key column)
        const float* decay = reinterpret_cast<const float*>(sp + REC_DECAY);
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float v[32];
            ptx::tmem_ld32(tS + 32 * j, v);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(sb + OFF_ST + sw128_off(tid, 32 * j + 8 * q, 128)) = pack8_f16(v + 8 * q);
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] *= decay[32 * j + x];
            ptx::tmem_st32(tS + 32 * j, v);
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t koff = (kk & 3) * 32;  // 16 fp16 of K inside the 128-byte row
                const uint64_t ad = ptx::sdesc_sw128(base + OFF_ST + (kk >> 2) * 16384 + koff);
                const uint64_t bw = ptx::sdesc_sw128(stg + REC_W + (kk >> 2) * 8192 + koff);
                const uint64_t bq = ptx::sdesc_sw128(stg + REC_Q + (kk >> 2) * 8192 + koff);
                ptx::mma_f16(tmem + 128, ad, bw, IDESC_N64, kk > 0);
                ptx::mma_f16(tmem + 192, ad, bq, IDESC_N64, kk > 0);
            }
            ptx::mma_commit(bar_mma);
            pend[2] = 1;
        }
        if (!ptx::mbar_wait(bar_mma, mma_phase, WAIT_LIMIT_NS)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) break;
        mma_phase ^= 1;
        if (tid == 0) pend[2] = 0;
        ptx::tc_fence_after();

        // ---- U^T = U0^T - (W S)^T, as the fp16 A operand of MMA2 / MMA3
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            float v[32];
            ptx::tmem_ld32(tD + 32 * j, v);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t off = sw128_off(tid, 32 * j + 8 * q, 128);
                const uint4 u0 = *reinterpret_cast<const uint4*>(sp + REC_UT + off);
                const __half2* p = reinterpret_cast<const __half2*>(&u0);
                float u[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(p[e]);
                    u[2 * e] = f.x - v[8 * q + 2 * e];
                    u[2 * e + 1] = f.y - v[8 * q + 2 * e + 1];
                }
                *reinterpret_cast<uint4*>(sb + OFF_UT + off) = pack8_f16(u);
            }
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t au = ptx::sdesc_sw128(base + OFF_UT + kk * 32);
                const uint64_t bk = ptx::sdesc_sw128(stg + REC_KT + kk * 32);
                const uint64_t bp = ptx::sdesc_sw128(stg + REC_P + kk * 32);
                ptx::mma_f16(tmem, au, bk, IDESC_N128, 1);
                ptx::mma_f16(tmem + 192, au, bp, IDESC_N64, 1);
            }
            ptx::mma_commit(bar_mma);
            pend[2] = 1;
        }
        if (!ptx::mbar_wait(bar_mma, mma_phase, WAIT_LIMIT_NS)) *abort_flag = 1;
        __syncthreads();
        if (*abort_flag) break;
        mma_phase ^= 1;
        if (tid == 0) pend[2] = 0;
        ptx::tc_fence_after();

        // ---- O^T -> o_core (lanes are consecutive value columns: coalesced)
        float* orow = o_core + (size_t)(bos + CHUNK_T * c) * W + (size_t)h * D + tid;
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            float v[32];
            ptx::tmem_ld32(tD + 64 + 32 * j, v);
#pragma unroll
            for (int x = 0; x < 32; ++x)
                if (32 * j + x < Lc) orow[(size_t)(32 * j + x) * W] = v[x];
        }
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0 && c + 2 < nc) {
            ptx::fence_async_smem();
            issue_load(c + 2);
        }
    }

    if (!*abort_flag) {
        // final state: S_out[key][value] = S^T[value][key]
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float v[32];
            ptx::tmem_ld32(tS + 32 * j, v);
#pragma unroll
            for (int x = 0; x < 32; ++x) a.S_out[soff + (size_t)(32 * j + x) * D + tid] = v[x];
        }
    } else if (tid == 0) {
        // record the timeout, then let this CTA's own copies and MMAs land
        atomicExch(a.status, ERR_TIMEOUT);
        for (int s = 0; s < 2; ++s)
            if (pend[s]) ptx::mbar_wait(bar_load[s], load_phase[s], WAIT_LIMIT_NS);
        if (pend[2]) ptx::mbar_wait(bar_mma, mma_phase, WAIT_LIMIT_NS);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

bool chunked_kernel_built() { return true; }

cudaError_t launch_chunk_recurrence(const ChunkRecArgs& a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(chunk_recurrence_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.n_seqs * a.H;
    if (blocks == 0) return cudaSuccess;
    chunk_recurrence_kernel<<<(unsigned)blocks, NT, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
