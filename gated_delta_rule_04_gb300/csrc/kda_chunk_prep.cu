// Chunk preparation for the chunked prefill: everything inside a 64-token
// chunk that does not depend on the recurrent state, for all chunks and heads
// in parallel.  The chunked form follows the "chunked UT transform" with a
// per-channel cumulative log gate described on "memra-engine 0.124.0, module
// kda" (PREFILL DISPATCH) and the 16-token tile bound of "Kimi K3 - Retention
// gate - OpenModelAtlas" (section "Why": with g >= -5 every rescaling over a
// 16-token tile stays below e^80).
//
// With G_r the inclusive cumulative gate inside the chunk (per key channel):
//   A[r][s] = beta_r sum_i k_ri k_si e^{G_ri - G_si}   (s < r)
//   P[r][s] =        sum_i q_ri k_si e^{G_ri - G_si}   (s <= r)
//   T  = (I + A)^{-1} Diag(beta)
//   W  = T (k * e^{G}),  U0 = T v,  Q+ = q * e^{G},  Kt = k * e^{G_last - G},
//   decay = e^{G_last}
// The sequential kernel then needs only U = U0 - W S, O = Q+ S + P U and
// S' = Diag(decay) S + Kt^T U per chunk.
//
// Range.  e^{G_r - G_s} is split at the 16-token sub-tile boundaries.  With
// st(a)/en(a) the first/last token of sub-tile a, Y_s = e^{G_en(b) - G_s} <= 1
// for s in sub-tile b, and for r in sub-tile a:
//   a > b:  e^{G_r - G_s} = [e^{G_r - G_st(a)} e^{G_st(a) - G_en(b)}] * Y_s
//           both brackets <= 1: these six off-diagonal 16 x 16 blocks run on
//           the tensor cores with fp16 operands (two M=128 MMAs, rows =
//           (block pair, r) for k and for q, columns = all 64 s);
//   a = b:  e^{G_r - G_s} = (1 / Y_r) * Y_s with 1/Y_r <= e^{75}: the four
//           diagonal blocks stay in fp32 on the CUDA cores (fp16 cannot hold
//           e^{75}, and bf16 operands there triple the end-to-end error).
// The unit lower-triangular solve is blockwise: the four 16 x 16 diagonal
// inverses by forward substitution, then the off-diagonal blocks of the
// inverse by 16 x 16 products, diagonal by diagonal.  W^T = (k e^G)^T T^T and
// U0^T = v^T T^T run as two M=128 tensor-core MMAs.
//
// Output: one record per (chunk, head) holding the operand tiles in the exact
// shared-memory image the tcgen05 recurrence kernel consumes (fp16, K-major,
// 128-byte swizzle: 16-byte chunk j of row r stored at chunk position j ^ (r & 7)).
#include "kda_chunk_layout.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int PT = 256;        // threads (8 warps)
constexpr int C = CHUNK_T;     // 64 tokens
constexpr int LDS = 65;        // padded fp32 row stride of the 64 x 64 matrices
constexpr uint32_t TMEM_COLS = 256;  // [0,64) A-rows D, [64,128) P-rows D, [128,192) W^T, [192,256) U0^T
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// shared-memory map (bytes, from a 1 KiB aligned base)
constexpr uint32_t S_G = 0;                    // fp32 [64][128] G (rows past the chunk repeat the last)
constexpr uint32_t S_Y = S_G + 32768;          // fp32 [64][128] Y, later X = (I+A)^{-1} fp32 [64][65]
constexpr uint32_t S_KH = S_Y + 32768;         // fp16 [64][128] k^ (plain row-major)
constexpr uint32_t S_QH = S_KH + 16384;        // fp16 [64][128] q^
constexpr uint32_t S_LOFF = S_QH + 16384;      // fp16 2 tiles x [128 rows][128 keys] (swizzled), later KPT/VT/TT
constexpr uint32_t S_KPT = S_LOFF;             //   fp16 [128 key][64 tok]  (k e^G)^T
constexpr uint32_t S_VT = S_LOFF + 16384;      //   fp16 [128 val][64 tok]  v^T
constexpr uint32_t S_TT = S_LOFF + 32768;      //   fp16 [64 r][64 s]       T
constexpr uint32_t S_RT = S_LOFF + 65536;      // fp16 [64 s][128 keys] (swizzled) k Y
constexpr uint32_t S_AM = S_RT + 16384;        // fp32 [64][65] A (with beta)
constexpr uint32_t S_PM = S_AM + 64 * LDS * 4; // fp32 [64][65] P
constexpr uint32_t S_MT = S_PM + 64 * LDS * 4; // fp32 [6 pairs][128] e^{G_st(a) - G_en(b)}; [4][128] e^{G_en(a)-G_st(a)}; [4][128] e^{G_st(a)}
constexpr uint32_t S_BT = S_MT + 14 * 128 * 4; // fp32 [64] beta
constexpr uint32_t S_BAR = S_BT + 256;         // mbarrier + TMEM slot
constexpr uint32_t SMEM_BYTES = S_BAR + 64 + 1024;

__constant__ int8_t kPairA[6] = {1, 2, 3, 2, 3, 3};
__constant__ int8_t kPairB[6] = {0, 0, 0, 1, 1, 2};

__device__ __forceinline__ uint4 pack8_f16(const float* v) {
    uint4 u;
    __half2* p = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
    return u;
}

// eight fp16 values from shared memory (16-byte aligned) as fp32
__device__ __forceinline__ void lds_h8(const __half* p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(PT, 1) chunk_prep_kernel(PrepArgs a) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sb = smem_raw + (base - raw);
    float* G = reinterpret_cast<float*>(sb + S_G);
    float* Y = reinterpret_cast<float*>(sb + S_Y);
    float* Xm = reinterpret_cast<float*>(sb + S_Y);
    const __half* KH = reinterpret_cast<const __half*>(sb + S_KH);
    const __half* QH = reinterpret_cast<const __half*>(sb + S_QH);
    const __half* VH = reinterpret_cast<const __half*>(sb + S_RT);  // v^ rows, after the off-diagonal MMAs
    float* Am = reinterpret_cast<float*>(sb + S_AM);
    float* Pm = reinterpret_cast<float*>(sb + S_PM);
    float* Mt = reinterpret_cast<float*>(sb + S_MT);
    float* bt = reinterpret_cast<float*>(sb + S_BT);
    const uint32_t bar = base + S_BAR;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sb + S_BAR + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sb + S_BAR + 20);

    const int H = a.H, W = H * D;
    const int chunk = blockIdx.x / H, h = blockIdx.x % H;
    const ChunkDesc cd = a.chunks[chunk];
    const int L = cd.len, t0 = cd.t0;
    const int tid = threadIdx.x, warp = tid >> 5;
    const __half* qh = static_cast<const __half*>(a.qh);
    const __half* kh = static_cast<const __half*>(a.kh);
    const __half* vh = static_cast<const __half*>(a.vh);
    const size_t hb = (size_t)h * D;
    auto gidx = [&](int r, int i) { return (size_t)(t0 + r) * W + hb + i; };

    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }

    // ---- 1. G, beta, k^, q^ into shared memory (16-byte cp.async copies, all in flight at once)
    for (int idx = tid; idx < C * 32; idx += PT) {          // G: 64 rows x 32 x 16 B
        const int r = idx >> 5, v4 = idx & 31;
        const int rr = r < L ? r : L - 1;
        cp_async16(sb + S_G + 16 * idx, a.gcum + gidx(rr, 4 * v4));
    }
    for (int idx = tid; idx < C * 16; idx += PT) {          // k^, q^: 64 rows x 16 x 16 B
        const int r = idx >> 4, v8 = idx & 15;
        if (r < L) {
            cp_async16(sb + S_KH + 16 * idx, kh + gidx(r, 8 * v8));
            cp_async16(sb + S_QH + 16 * idx, qh + gidx(r, 8 * v8));
        } else {
            reinterpret_cast<uint4*>(sb + S_KH)[idx] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(sb + S_QH)[idx] = make_uint4(0, 0, 0, 0);
        }
    }
    cp_async_wait_all();
    if (tid < C) bt[tid] = tid < L ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- 2. Y, per-tile factors, right operand R = k Y (fp16 swizzled)
    for (int idx = tid; idx < C * D; idx += PT) {
        const int r = idx >> 7, i = idx & 127;
        const int en = min((r & ~15) + 15, L - 1);
        Y[idx] = __expf(G[en * D + i] - G[idx]);
    }
    for (int idx = tid; idx < 14 * D; idx += PT) {
        const int m = idx >> 7, i = idx & 127;
        float val;
        if (m < 6) {          // e^{G_st(a) - G_en(b)}, a > b
            const int st = min(16 * kPairA[m], L - 1), en = min(16 * kPairB[m] + 15, L - 1);
            val = expf(G[st * D + i] - G[en * D + i]);
        } else if (m < 10) {  // e^{G_en(a) - G_st(a)}
            const int ta = m - 6;
            const int st = min(16 * ta, L - 1), en = min(16 * ta + 15, L - 1);
            val = expf(G[en * D + i] - G[st * D + i]);
        } else {              // e^{G_st(a)}
            const int st = min(16 * (m - 10), L - 1);
            val = expf(G[st * D + i]);
        }
        Mt[idx] = val;
    }
    __syncthreads();
    for (int idx = tid; idx < C * 16; idx += PT) {           // R: 64 rows x 16 chunks of 8 keys
        const int s = idx >> 4, ch = idx & 15;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = ch * 8 + e;
            v[e] = __half2float(KH[s * D + i]) * Y[s * D + i];
        }
        *reinterpret_cast<uint4*>(sb + S_RT + sw128_off(s, ch * 8, C)) = pack8_f16(v);
    }
    // left operand of the off-diagonal blocks: row (pair p, r_local) =
    //   k_r e^{G_r - G_st(a)} e^{G_st(a) - G_en(b)}, with
    //   e^{G_r - G_st(a)} = e^{G_en(a) - G_st(a)} / Y_r   (both <= 1 after the division)
    // tile 0 holds the k rows, tile 1 the q rows; rows 96..127 are zero.
    for (int idx = tid; idx < 2 * 128 * 16; idx += PT) {
        const int tile = idx >> 11, rem = idx & 2047;
        const int row = rem >> 4, ch = rem & 15;
        float v[8];
        if (row < 96) {
            const int p = row >> 4, rl = row & 15;
            const int ta = kPairA[p];
            const int r = 16 * ta + rl;
            const __half* src = tile == 0 ? KH : QH;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = ch * 8 + e;
                const float x = Mt[(6 + ta) * D + i] * __frcp_rn(Y[r * D + i]);
                v[e] = __half2float(src[r * D + i]) * x * Mt[p * D + i];
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
        *reinterpret_cast<uint4*>(sb + S_LOFF + tile * 32768 + sw128_off(row, ch * 8, 128)) = pack8_f16(v);
    }
    ptx::fence_async_smem();
    ptx::tc_fence_before();
    __syncthreads();

    // ---- 3. off-diagonal blocks on the tensor cores: D[row][s] for all 64 s
    constexpr uint32_t IDESC_N64 = ptx::idesc_f16_f32(128, 64);
    if (tid == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk & 3) * 32;
            const uint64_t bR = ptx::sdesc_sw128(base + S_RT + (kk >> 2) * 8192 + koff);
            const uint64_t aK = ptx::sdesc_sw128(base + S_LOFF + (kk >> 2) * 16384 + koff);
            const uint64_t aQ = ptx::sdesc_sw128(base + S_LOFF + 32768 + (kk >> 2) * 16384 + koff);
            ptx::mma_f16(tmem, aK, bR, IDESC_N64, kk > 0);
            ptx::mma_f16(tmem + 64, aQ, bR, IDESC_N64, kk > 0);
        }
        ptx::mma_commit(bar);
    }

    // ---- 4. diagonal blocks in fp32 while the MMAs run: e^{G_r - G_s} = Y_s / Y_r.
    // Thread (tile a, 4 rows x 4 cols block, K quarter); partial sums reduced in
    // shared memory.  Blocks above the diagonal of a tile are skipped.
    {
        // zero A and P (the off-diagonal blocks are filled from TMEM later)
        for (int idx = tid; idx < C * LDS; idx += PT) { Am[idx] = 0.f; Pm[idx] = 0.f; }
        __syncthreads();
        const int ta = tid >> 6;            // tile
        const int rem = tid & 63;
        const int blk = rem >> 2, kq = rem & 3;
        const int br = blk >> 2, bc = blk & 3;  // 4x4 sub-blocks of the 16x16 tile
        float accA[4][4], accP[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) { accA[x][y] = 0.f; accP[x][y] = 0.f; }
        if (bc <= br) {
            const int r0 = 16 * ta + 4 * br, s0 = 16 * ta + 4 * bc;
#pragma unroll 1
            for (int i0 = 32 * kq; i0 < 32 * kq + 32; i0 += 8) {
                float lk[4][8], lq[4][8], rr[4][8];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    float y8[8], k8[8], q8[8], ys8[8], ks8[8];
                    Vec8<float>::lds(Y + (r0 + x) * D + i0, y8);
                    Vec8<float>::lds(Y + (s0 + x) * D + i0, ys8);
                    lds_h8(KH + (r0 + x) * D + i0, k8);
                    lds_h8(QH + (r0 + x) * D + i0, q8);
                    lds_h8(KH + (s0 + x) * D + i0, ks8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float inv = __frcp_rn(y8[e]);
                        lk[x][e] = k8[e] * inv;
                        lq[x][e] = q8[e] * inv;
                        rr[x][e] = ks8[e] * ys8[e];
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int y = 0; y < 4; ++y) {
                            accA[x][y] = fmaf(lk[x][e], rr[y][e], accA[x][y]);
                            accP[x][y] = fmaf(lq[x][e], rr[y][e], accP[x][y]);
                        }
            }
        }
        // reduce the four K quarters with shuffles (lanes kq = 0..3 are adjacent)
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                float va = accA[x][y], vp = accP[x][y];
                va += __shfl_xor_sync(0xffffffffu, va, 1);
                va += __shfl_xor_sync(0xffffffffu, va, 2);
                vp += __shfl_xor_sync(0xffffffffu, vp, 1);
                vp += __shfl_xor_sync(0xffffffffu, vp, 2);
                accA[x][y] = va;
                accP[x][y] = vp;
            }
        if (kq == 0 && bc <= br) {
            const int r0 = 16 * ta + 4 * br, s0 = 16 * ta + 4 * bc;
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const int r = r0 + x, s = s0 + y;
                    if (s < r) Am[r * LDS + s] = bt[r] * accA[x][y];
                    if (s <= r) Pm[r * LDS + s] = accP[x][y];
                }
        }
    }

    // ---- 5. off-diagonal blocks out of TMEM (warps 0-3: k rows -> A, 4-7: q rows -> P)
    if (!ptx::mbar_wait(bar, 0, WAIT_LIMIT_NS)) *abort_flag = 1;
    ptx::tc_fence_after();
    {
        const int lane_row = 32 * (warp & 3) + (tid & 31);  // TMEM lane = tile row
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp < 4 ? 0 : 64);
        float v[64];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            float part[16];
            tmem_ld16(taddr + 16 * q4, part);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[16 * q4 + j] = part[j];
        }
        if (lane_row < 96 && !*abort_flag) {
            const int p = lane_row >> 4, rl = lane_row & 15;
            const int r = 16 * kPairA[p] + rl, sb0 = 16 * kPairB[p];
            if (warp < 4) {
                const float be = bt[r];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    // the pair's columns sit at [16 b, 16 b + 16) of the 64
                    float val = 0.f;
#pragma unroll
                    for (int bb = 0; bb < 3; ++bb)
                        if (kPairB[p] == bb) val = v[16 * bb + j];
                    Am[r * LDS + sb0 + j] = be * val;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float val = 0.f;
#pragma unroll
                    for (int bb = 0; bb < 3; ++bb)
                        if (kPairB[p] == bb) val = v[16 * bb + j];
                    Pm[r * LDS + sb0 + j] = val;
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();

    // v^ rows into the (now free) right-operand space, landing during the solve
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, v8 = idx & 15;
        if (r < L) cp_async16(sb + S_RT + 16 * idx, vh + gidx(r, 8 * v8));
        else reinterpret_cast<uint4*>(sb + S_RT)[idx] = make_uint4(0, 0, 0, 0);
    }

    // ---- 6. X = (I + A)^{-1}: diagonal 16 x 16 inverses by forward substitution
    for (int idx = tid; idx < C * LDS; idx += PT) Xm[idx] = 0.f;
    __syncthreads();
    if (tid < 64) {
        const int ta = tid >> 4, j = tid & 15;
        const int o = 16 * ta;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float t = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < r; ++s) t = fmaf(-Am[(o + r) * LDS + o + s], x[s], t);
            x[r] = (r < j) ? 0.f : t;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Xm[(o + r) * LDS + o + j] = x[r];
    }
    __syncthreads();
    // off-diagonal blocks, one diagonal at a time:
    //   X_ab = -X_aa * sum_{k=b}^{a-1} A_ak X_kb
    // Am's upper-right 16x16 blocks are zero and unused by the solve; they
    // hold the temporaries M_ab = sum_k A_ak X_kb at block (b, a).
    for (int d = 1; d < 4; ++d) {
        const int nblk = 4 - d;
        for (int idx = tid; idx < nblk * 256; idx += PT) {
            const int bidx = idx >> 8, e = idx & 255;
            const int b = bidx, ab = bidx + d;
            const int r = e >> 4, cc = e & 15;
            float acc = 0.f;
            for (int kb = b; kb < ab; ++kb)
#pragma unroll
                for (int s = 0; s < 16; ++s)
                    acc = fmaf(Am[(16 * ab + r) * LDS + 16 * kb + s], Xm[(16 * kb + s) * LDS + 16 * b + cc], acc);
            Am[(16 * b + r) * LDS + 16 * ab + cc] = acc;  // temporary in the unused upper block
        }
        __syncthreads();
        for (int idx = tid; idx < nblk * 256; idx += PT) {
            const int bidx = idx >> 8, e = idx & 255;
            const int b = bidx, ab = bidx + d;
            const int r = e >> 4, cc = e & 15;
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < 16; ++s)
                acc = fmaf(Xm[(16 * ab + r) * LDS + 16 * ab + s], Am[(16 * b + s) * LDS + 16 * ab + cc], acc);
            Xm[(16 * ab + r) * LDS + 16 * b + cc] = -acc;
        }
        __syncthreads();
    }

    cp_async_wait_all();
    __syncthreads();

    // ---- 7. operands of W^T and U0^T (the left tiles are dead: reuse their space)
    //   TT[r][s] = X[r][s] beta_s ; KPT[key][s] = k_s e^{G_s} ; VT[val][s] = v_s
    for (int idx = tid; idx < C * 8; idx += PT) {           // TT: 64 rows x 8 chunks
        const int r = idx >> 3, ch = idx & 7;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = ch * 8 + e;
            v[e] = Xm[r * LDS + s] * bt[s];
        }
        *reinterpret_cast<uint4*>(sb + S_TT + sw128_off(r, ch * 8, C)) = pack8_f16(v);
    }
    for (int idx = tid; idx < D * 8; idx += PT) {           // KPT, VT: 128 rows x 8 chunks of 8 tokens
        const int row = idx & 127, ch = idx >> 7;
        float vk[8], vv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = ch * 8 + e;
            vk[e] = __half2float(KH[s * D + row]) * __expf(G[s * D + row]);
            vv[e] = __half2float(VH[s * D + row]);
        }
        *reinterpret_cast<uint4*>(sb + S_KPT + sw128_off(row, ch * 8, 128)) = pack8_f16(vk);
        *reinterpret_cast<uint4*>(sb + S_VT + sw128_off(row, ch * 8, 128)) = pack8_f16(vv);
    }
    ptx::fence_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0 && !*abort_flag) {
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bT = ptx::sdesc_sw128(base + S_TT + kk * 32);
            const uint64_t aK = ptx::sdesc_sw128(base + S_KPT + kk * 32);
            const uint64_t aV = ptx::sdesc_sw128(base + S_VT + kk * 32);
            ptx::mma_f16(tmem + 128, aK, bT, IDESC_N64, kk > 0);
            ptx::mma_f16(tmem + 192, aV, bT, IDESC_N64, kk > 0);
        }
        ptx::mma_commit(bar);
    }

    unsigned char* rec = static_cast<unsigned char*>(a.records) + ((size_t)chunk * H + h) * REC_BYTES;

    // ---- 8. tiles that need no MMA: Q+ [tok][key], Kt^T [key][tok], P [r][s], decay
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, ch = idx & 15;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = ch * 8 + e;
            v[e] = __half2float(QH[r * D + i]) * __expf(G[r * D + i]);
        }
        *reinterpret_cast<uint4*>(rec + REC_Q + sw128_off(r, ch * 8, C)) = pack8_f16(v);
    }
    for (int idx = tid; idx < D * 8; idx += PT) {
        const int key = idx & 127, ch = idx >> 7;
        const float glast = G[(C - 1) * D + key];
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = ch * 8 + e;
            v[e] = __half2float(KH[s * D + key]) * __expf(glast - G[s * D + key]);
        }
        *reinterpret_cast<uint4*>(rec + REC_KT + sw128_off(key, ch * 8, 128)) = pack8_f16(v);
    }
    for (int idx = tid; idx < C * 8; idx += PT) {
        const int r = idx >> 3, ch = idx & 7;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = Pm[r * LDS + ch * 8 + e];
        *reinterpret_cast<uint4*>(rec + REC_P + sw128_off(r, ch * 8, C)) = pack8_f16(v);
    }
    if (tid < D) reinterpret_cast<float*>(rec + REC_DECAY)[tid] = expf(G[(C - 1) * D + tid]);

    // ---- 9. W and U0^T out of TMEM: warps 0-3 hold W^T (lane = key), 4-7 U0^T (lane = value)
    if (!ptx::mbar_wait(bar, 1, WAIT_LIMIT_NS)) *abort_flag = 1;
    ptx::tc_fence_after();
    {
        const int row = 32 * (warp & 3) + (tid & 31);
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp < 4 ? 128 : 192);
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            float v[16];
            tmem_ld16(taddr + 16 * q4, v);
            if (*abort_flag) continue;
            if (warp < 4) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<__half*>(rec + REC_W + sw128_off(16 * q4 + j, row, C)) = __float2half_rn(v[j]);
            } else {
                *reinterpret_cast<uint4*>(rec + REC_UT + sw128_off(row, 16 * q4, 128)) = pack8_f16(v);
                *reinterpret_cast<uint4*>(rec + REC_UT + sw128_off(row, 16 * q4 + 8, 128)) = pack8_f16(v + 8);
            }
        }
    }
    if (tid == 0 && *abort_flag) atomicExch(a.status, ERR_TIMEOUT);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

size_t chunk_prep_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_chunk_prep(const PrepArgs& a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.n_chunks * a.H;
    if (blocks == 0) return cudaSuccess;
    chunk_prep_kernel<<<(unsigned)blocks, PT, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
