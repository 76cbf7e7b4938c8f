// Chunk preparation for the chunked prefill: everything inside a 64-token
// chunk that does not depend on the recurrent state, for all chunks and heads
// in parallel.  The chunked form follows the "chunked UT transform" with a
// per-channel cumulative log gate described on "memra-engine 0.124.0, module
// kda" (PREFILL DISPATCH) and the 16-token tile bound of "Kimi K3 - Retention
// gate - OpenModelAtlas" (section "Why": with g >= -5 every rescaling over a
// 16-token tile stays below e^80, inside bf16's range).
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
// Range.  For s in 16-token sub-tile b the reference point is the last token
// of that sub-tile, en(b):  e^{G_r - G_s} = e^{G_r - G_en(b)} * Y_s with
// Y_s = e^{G_en(b) - G_s} <= 1.  The left factor is <= 1 when r lies in a
// later sub-tile and at most e^{75} inside the diagonal sub-tile, which bf16
// holds.  All of A and the off-diagonal blocks of P therefore run on the
// tensor cores as two bf16 MMAs (M = 128, N = 64 = every s, K = 128 keys):
// 256 left rows = (A rows grouped by column sub-tile b: 64+48+32+16) +
// (off-diagonal P rows: 48+32+16).  The diagonal blocks of P stay in fp32 on
// the CUDA cores: P reaches the output directly, and bf16 there would triple
// the end-to-end error, while bf16 in A changes it by under 5%.
// Left factors for a later sub-tile a > b are formed as a product of two
// factors <= 1, e^{G_r - G_st(a)} e^{G_st(a) - G_en(b)}, so nothing
// overflows or loses precision to fp32 subnormals.
//
// The unit lower-triangular solve is blockwise: the four 16 x 16 diagonal
// inverses by forward substitution, then the off-diagonal blocks of the
// inverse by 16 x 16 products, diagonal by diagonal.  W^T = (k e^G)^T T^T and
// U0^T = v^T T^T run as two fp16 M=128 MMAs.
//
// Output: one record per (chunk, head) holding the operand tiles in the exact
// shared-memory image the tcgen05 recurrence kernel consumes (fp16, K-major,
// 128-byte swizzle: 16-byte chunk j of row r stored at chunk position j ^ (r & 7)).
#include "kda_chunk_layout.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int PT = 512;        // threads (16 warps: four per scheduler to hide latency)
constexpr int C = CHUNK_T;     // 64 tokens
constexpr int LDS = 65;        // padded fp32 row stride of the 64 x 64 matrices
constexpr int LDY = 132;       // padded fp32 row stride of Y
constexpr uint32_t TMEM_COLS = 256;  // [0,64) left tile 0, [64,128) left tile 1, [128,192) W^T, [192,256) U0^T
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// shared-memory map (bytes, from a 1 KiB aligned base)
constexpr uint32_t S_G = 0;                      // fp32 [64][128] G (rows past the chunk repeat the last)
constexpr uint32_t S_Y = S_G + 32768;            // fp32 [64][132] Y; later X = (I+A)^{-1} fp32 [64][65]
constexpr uint32_t S_KH = S_Y + 33792;           // fp16 [64][128] k^ (plain row-major)
constexpr uint32_t S_QH = S_KH + 16384;          // fp16 [64][128] q^
constexpr uint32_t S_VH = S_QH + 16384;          // fp16 [64][128] v^
constexpr uint32_t S_LAP = S_VH + 16384;         // bf16 2 tiles x [128 rows][128 keys] (swizzled); later KPT/VT/TT
constexpr uint32_t S_KPT = S_LAP;                //   fp16 [128 key][64 tok]  (k e^G)^T
constexpr uint32_t S_VT = S_LAP + 16384;         //   fp16 [128 val][64 tok]  v^T
constexpr uint32_t S_TT = S_LAP + 32768;         //   fp16 [64 r][64 s]       T
constexpr uint32_t S_RT = S_LAP + 65536;         // bf16 [64 s][128 keys] k Y (swizzled); later the W tile
constexpr uint32_t S_AM = S_RT + 16384;          // fp32 [64][65] A (with beta)
constexpr uint32_t S_PT = S_AM + 64 * LDS * 4;   // fp16 [64 r][64 s] P, in the record's swizzled layout
constexpr uint32_t S_MT = S_PT + 8192;           // fp32 [6][128] e^{G_st(a) - G_en(b)} per pair a > b; [4][128] e^{G_en(a) - G_st(a)}
constexpr uint32_t S_BT = S_MT + 10 * 128 * 4;   // fp32 [64] beta
constexpr uint32_t S_BAR = S_BT + 256;           // mbarrier, TMEM slot, flag
constexpr uint32_t SMEM_BYTES = S_BAR + 64 + 1024;

// sub-tile pairs a > b in the order of the factor table
__constant__ int8_t kPairA[6] = {1, 2, 3, 2, 3, 3};
__constant__ int8_t kPairB[6] = {0, 0, 0, 1, 1, 2};
__device__ __forceinline__ int pair_of(int a, int b) { return b == 0 ? a - 1 : (b == 1 ? a + 1 : 5); }

// Row groups of the 256 left rows: (is_P, column sub-tile b, first r, first row)
__constant__ int16_t kGroup[7][4] = {
    {0, 0, 0, 0}, {0, 1, 16, 64}, {0, 2, 32, 112}, {0, 3, 48, 144},
    {1, 0, 16, 160}, {1, 1, 32, 208}, {1, 2, 48, 240}};
__device__ __forceinline__ int group_of(int row) {
    int g = 0;
#pragma unroll
    for (int j = 1; j < 7; ++j)
        if (row >= kGroup[j][3]) g = j;
    return g;
}

__device__ __forceinline__ uint4 pack8_f16(const float* v) {
    uint4 u;
    __half2* p = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
    return u;
}
__device__ __forceinline__ uint4 pack8_bf16(const float* v) {
    uint4 u;
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    return u;
}

// eight fp16 / fp32 values from shared memory (16-byte aligned) as fp32
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
__device__ __forceinline__ void lds_f8(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void sts_f8(float* p, const float (&x)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// One-instruction reciprocal (max error 1 ulp); every argument here is a
// normal number in [e^-75, 1].
__device__ __forceinline__ float rcp_approx(float y) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

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

// One diagonal of the blockwise inverse (block pairs (b + d, b)), with the
// inner products unrolled so every load is issued ahead of its FMA.
template <int Dg>
__device__ __forceinline__ void solve_level(float* Am, float* Xm, int tid) {
    constexpr int nblk = 4 - Dg;
    for (int idx = tid; idx < nblk * 256; idx += PT) {
        const int b = idx >> 8, e = idx & 255, ab = b + Dg;
        const int r = e >> 4, cc = e & 15;
        float acc = 0.f;
#pragma unroll
        for (int kk = 0; kk < Dg; ++kk)
#pragma unroll
            for (int s = 0; s < 16; ++s)
                acc = fmaf(Am[(16 * ab + r) * LDS + 16 * (b + kk) + s], Xm[(16 * (b + kk) + s) * LDS + 16 * b + cc], acc);
        Am[(16 * b + r) * LDS + 16 * ab + cc] = acc;
    }
    __syncthreads();
    for (int idx = tid; idx < nblk * 256; idx += PT) {
        const int b = idx >> 8, e = idx & 255, ab = b + Dg;
        const int r = e >> 4, cc = e & 15;
        float acc = 0.f;
#pragma unroll
        for (int s = 0; s < 16; ++s)
            acc = fmaf(Xm[(16 * ab + r) * LDS + 16 * ab + s], Am[(16 * b + s) * LDS + 16 * ab + cc], acc);
        Xm[(16 * ab + r) * LDS + 16 * b + cc] = -acc;
    }
    __syncthreads();
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
    const __half* VH = reinterpret_cast<const __half*>(sb + S_VH);
    float* Am = reinterpret_cast<float*>(sb + S_AM);
    unsigned char* ptile = sb + S_PT;
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

    // ---- 1. G, k^, q^, v^ into shared memory: three cp.async groups, all in
    // flight at once, each awaited where it is first needed
    for (int idx = tid; idx < C * 32; idx += PT) {
        const int r = idx >> 5, v4 = idx & 31;
        const int rr = r < L ? r : L - 1;
        cp_async16(sb + S_G + 16 * idx, a.gcum + gidx(rr, 4 * v4));
    }
    cp_async_commit();
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, v8 = idx & 15;
        if (r < L) {
            cp_async16(sb + S_KH + 16 * idx, kh + gidx(r, 8 * v8));
            cp_async16(sb + S_QH + 16 * idx, qh + gidx(r, 8 * v8));
        } else {
            reinterpret_cast<uint4*>(sb + S_KH)[idx] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(sb + S_QH)[idx] = make_uint4(0, 0, 0, 0);
        }
    }
    cp_async_commit();
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, v8 = idx & 15;
        if (r < L) cp_async16(sb + S_VH + 16 * idx, vh + gidx(r, 8 * v8));
        else reinterpret_cast<uint4*>(sb + S_VH)[idx] = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
    if (tid < C) bt[tid] = tid < L ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    for (int idx = tid; idx < 512; idx += PT) reinterpret_cast<uint4*>(ptile)[idx] = make_uint4(0, 0, 0, 0);
    cp_async_wait_group<2>();  // G
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // ---- 2. Y_s = e^{G_en(b) - G_s} and the per-sub-tile factors (8 channels per step)
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, ch = idx & 15;
        const int en = min((r & ~15) + 15, L - 1);
        float g[8], ge[8], y[8];
        lds_f8(G + r * D + 8 * ch, g);
        lds_f8(G + en * D + 8 * ch, ge);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __expf(ge[e] - g[e]);
        sts_f8(Y + r * LDY + 8 * ch, y);
    }
    for (int idx = tid; idx < 10 * D; idx += PT) {
        const int m = idx >> 7, i = idx & 127;
        int st, en;
        if (m < 6) { st = min(16 * kPairA[m], L - 1); en = min(16 * kPairB[m] + 15, L - 1); }
        else { st = min(16 * (m - 6) + 15, L - 1); en = min(16 * (m - 6), L - 1); }  // e^{G_en(a) - G_st(a)}
        Mt[idx] = __expf(G[st * D + i] - G[en * D + i]);
    }
    __syncthreads();

    // ---- 3. right operand R_s = k_s Y_s and the 256 left rows (bf16, swizzled).
    // One item = (token r, 8 channels): the reciprocal 1/Y_r is formed once and
    // every left row that token appears in (A rows for b <= a, P rows for
    // b < a) is written from it.
    cp_async_wait_group<1>();  // k^, q^
    __syncthreads();
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, ch = idx & 15;
        const int ta = r >> 4;
        float k8[8], q8[8], y8[8], iy[8], v[8];
        lds_h8(KH + r * D + 8 * ch, k8);
        lds_h8(QH + r * D + 8 * ch, q8);
        lds_f8(Y + r * LDY + 8 * ch, y8);
#pragma unroll
        for (int e = 0; e < 8; ++e) { v[e] = k8[e] * y8[e]; iy[e] = rcp_approx(y8[e]); }
        *reinterpret_cast<uint4*>(sb + S_RT + sw128_off(r, 8 * ch, C)) = pack8_bf16(v);
        float va[8];
        lds_f8(Mt + (6 + ta) * D + 8 * ch, va);
#pragma unroll
        for (int e = 0; e < 8; ++e) va[e] *= iy[e];  // e^{G_r - G_st(a)} = e^{G_en(a) - G_st(a)} / Y_r
        for (int b = 0; b <= ta; ++b) {
            // A row of (column sub-tile b, r)
            const int arow = kGroup[b][3] + (r - kGroup[b][2]);
            float f[8];
            if (b == ta) {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = iy[e];
            } else {
                float cab[8];
                lds_f8(Mt + pair_of(ta, b) * D + 8 * ch, cab);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = va[e] * cab[e];
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = k8[e] * f[e];
            *reinterpret_cast<uint4*>(sb + S_LAP + (arow >> 7) * 32768 + sw128_off(arow & 127, 8 * ch, 128)) =
                pack8_bf16(v);
            if (b < ta) {  // off-diagonal P row of (b, r)
                const int prow = kGroup[4 + b][3] + (r - kGroup[4 + b][2]);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = q8[e] * f[e];
                *reinterpret_cast<uint4*>(sb + S_LAP + (prow >> 7) * 32768 + sw128_off(prow & 127, 8 * ch, 128)) =
                    pack8_bf16(v);
            }
        }
    }
    ptx::fence_async_smem();
    ptx::tc_fence_before();
    __syncthreads();

    // ---- 4. A and the off-diagonal P blocks on the tensor cores
    constexpr uint32_t IDESC_BF16_N64 = ptx::idesc_bf16_f32(128, 64);
    constexpr uint32_t IDESC_F16_N64 = ptx::idesc_f16_f32(128, 64);
    if (tid == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk & 3) * 32;
            const uint64_t bR = ptx::sdesc_sw128(base + S_RT + (kk >> 2) * 8192 + koff);
            const uint64_t a0 = ptx::sdesc_sw128(base + S_LAP + (kk >> 2) * 16384 + koff);
            const uint64_t a1 = ptx::sdesc_sw128(base + S_LAP + 32768 + (kk >> 2) * 16384 + koff);
            ptx::mma_f16(tmem, a0, bR, IDESC_BF16_N64, kk > 0);
            ptx::mma_f16(tmem + 64, a1, bR, IDESC_BF16_N64, kk > 0);
        }
        ptx::mma_commit(bar);
    }

    // ---- 5. diagonal blocks of P in fp32 while the MMAs run: e^{G_r - G_s} = Y_s / Y_r.
    // Thread = (sub-tile, 4x4 block, K quarter); the quarters interleave 8-channel
    // chunks so that neighbouring lanes read different banks.
    for (int idx = tid; idx < C * LDS; idx += PT) Am[idx] = 0.f;
    __syncthreads();
    {
        const int ta = tid >> 7, rem = tid & 127;
        const int blk = rem >> 3, kq = rem & 7;   // 16 blocks of 4x4 x 8 interleaved K slices
        const int br = blk >> 2, bc = blk & 3;
        float acc[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
        const int r0 = 16 * ta + 4 * br, s0 = 16 * ta + 4 * bc;
        if (bc <= br) {
#pragma unroll 1
            for (int c8 = kq; c8 < 16; c8 += 8) {
                float lq[4][8], rr[4][8];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    float q8[8], yr[8], k8[8], ys[8];
                    lds_h8(QH + (r0 + x) * D + 8 * c8, q8);
                    lds_f8(Y + (r0 + x) * LDY + 8 * c8, yr);
                    lds_h8(KH + (s0 + x) * D + 8 * c8, k8);
                    lds_f8(Y + (s0 + x) * LDY + 8 * c8, ys);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        lq[x][e] = q8[e] * rcp_approx(yr[e]);
                        rr[x][e] = k8[e] * ys[e];
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
#pragma unroll
                    for (int x = 0; x < 4; ++x)
#pragma unroll
                        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(lq[x][e], rr[y][e], acc[x][y]);
            }
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                float v = acc[x][y];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                acc[x][y] = v;
            }
        if (kq == 0 && bc <= br) {
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y)
                    if (s0 + y <= r0 + x)
                        *reinterpret_cast<__half*>(ptile + sw128_off(r0 + x, s0 + y, C)) = __float2half_rn(acc[x][y]);
        }
    }

    // ---- 6. A and off-diagonal P out of TMEM (warps 0-3: left tile 0, 4-7: tile 1)
    if (!ptx::mbar_wait(bar, 0, WAIT_LIMIT_NS)) *abort_flag = 1;
    ptx::tc_fence_after();
    if (warp < 8) {
        const int lane_row = 32 * (warp & 3) + (tid & 31);
        const int row = (warp < 4 ? 0 : 128) + lane_row;
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp < 4 ? 0 : 64);
        const int g = group_of(row);
        const int isP = kGroup[g][0], b = kGroup[g][1];
        const int r = kGroup[g][2] + (row - kGroup[g][3]);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            float v[16];
            tmem_ld16(taddr + 16 * q4, v);  // columns s = 16 q4 .. 16 q4 + 15
            if (q4 == b && !*abort_flag) {
                if (isP) {
                    *reinterpret_cast<uint4*>(ptile + sw128_off(r, 16 * b, C)) = pack8_f16(v);
                    *reinterpret_cast<uint4*>(ptile + sw128_off(r, 16 * b + 8, C)) = pack8_f16(v + 8);
                } else {
                    const float be = bt[r];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (16 * b + j < r) Am[r * LDS + 16 * b + j] = be * v[j];
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();

    // ---- 7. X = (I + A)^{-1}: diagonal 16 x 16 inverses by forward substitution
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
    // off-diagonal blocks, one diagonal at a time: X_ab = -X_aa sum_{k=b}^{a-1} A_ak X_kb.
    // The temporaries M_ab live in A's unused upper-right block (b, a).
    solve_level<1>(Am, Xm, tid);
    solve_level<2>(Am, Xm, tid);
    solve_level<3>(Am, Xm, tid);
    cp_async_wait_group<0>();  // v^
    __syncthreads();

    // ---- 8. operands of W^T and U0^T (fp16; the left tiles are dead, reuse their space)
    //   TT[r][s] = X[r][s] beta_s ; KPT[key][s] = k_s e^{G_s} ; VT[val][s] = v_s
    for (int idx = tid; idx < C * 8; idx += PT) {
        const int r = idx >> 3, ch = idx & 7;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = Xm[r * LDS + 8 * ch + e] * bt[8 * ch + e];
        *reinterpret_cast<uint4*>(sb + S_TT + sw128_off(r, 8 * ch, C)) = pack8_f16(v);
    }
    for (int idx = tid; idx < D * 8; idx += PT) {
        const int row = idx & 127, ch = idx >> 7;
        float vk[8], vv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = 8 * ch + e;
            vk[e] = __half2float(KH[s * D + row]) * __expf(G[s * D + row]);
            vv[e] = __half2float(VH[s * D + row]);
        }
        *reinterpret_cast<uint4*>(sb + S_KPT + sw128_off(row, 8 * ch, 128)) = pack8_f16(vk);
        *reinterpret_cast<uint4*>(sb + S_VT + sw128_off(row, 8 * ch, 128)) = pack8_f16(vv);
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
            ptx::mma_f16(tmem + 128, aK, bT, IDESC_F16_N64, kk > 0);
            ptx::mma_f16(tmem + 192, aV, bT, IDESC_F16_N64, kk > 0);
        }
        ptx::mma_commit(bar);
    }

    unsigned char* rec = static_cast<unsigned char*>(a.records) + ((size_t)chunk * H + h) * REC_BYTES;

    // ---- 9. tiles that need no MMA, straight to the record: Q+ [tok][key], Kt^T [key][tok], P, decay
    for (int idx = tid; idx < C * 16; idx += PT) {
        const int r = idx >> 4, ch = idx & 15;
        float q8[8], g8[8], v[8];
        lds_h8(QH + r * D + 8 * ch, q8);
        lds_f8(G + r * D + 8 * ch, g8);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = q8[e] * __expf(g8[e]);
        *reinterpret_cast<uint4*>(rec + REC_Q + sw128_off(r, 8 * ch, C)) = pack8_f16(v);
    }
    for (int idx = tid; idx < D * 8; idx += PT) {
        const int key = idx & 127, ch = idx >> 7;
        const float glast = G[(C - 1) * D + key];
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = 8 * ch + e;
            v[e] = __half2float(KH[s * D + key]) * __expf(glast - G[s * D + key]);
        }
        *reinterpret_cast<uint4*>(rec + REC_KT + sw128_off(key, 8 * ch, 128)) = pack8_f16(v);
    }
    for (int idx = tid; idx < 512; idx += PT)  // the 8 KiB P image
        reinterpret_cast<uint4*>(rec + REC_P)[idx] = reinterpret_cast<const uint4*>(ptile)[idx];
    if (tid < D) reinterpret_cast<float*>(rec + REC_DECAY)[tid] = expf(G[(C - 1) * D + tid]);

    // ---- 10. W^T (warps 0-3, lane = key) through a shared-memory W tile; U0^T (warps 4-7, lane = value) direct
    if (!ptx::mbar_wait(bar, 1, WAIT_LIMIT_NS)) *abort_flag = 1;
    ptx::tc_fence_after();
    if (warp < 8) {
        const int row = 32 * (warp & 3) + (tid & 31);
        const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp < 4 ? 128 : 192);
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            float v[16];
            tmem_ld16(taddr + 16 * q4, v);
            if (warp < 4) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<__half*>(sb + S_RT + sw128_off(16 * q4 + j, row, C)) = __float2half_rn(v[j]);
            } else if (!*abort_flag) {
                *reinterpret_cast<uint4*>(rec + REC_UT + sw128_off(row, 16 * q4, 128)) = pack8_f16(v);
                *reinterpret_cast<uint4*>(rec + REC_UT + sw128_off(row, 16 * q4 + 8, 128)) = pack8_f16(v + 8);
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (!*abort_flag) {
        for (int idx = tid; idx < 1024; idx += PT)  // the 16 KiB W image, 16 bytes per thread step
            reinterpret_cast<uint4*>(rec + REC_W)[idx] = reinterpret_cast<const uint4*>(sb + S_RT)[idx];
    } else if (tid == 0) {
        atomicExch(a.status, ERR_TIMEOUT);
    }
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
