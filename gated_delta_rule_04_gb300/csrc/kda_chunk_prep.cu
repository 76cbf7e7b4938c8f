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
// Range: e^{G_r - G_s} is split at the sub-tile boundaries so that no factor
// exceeds e^{75}: for r in sub-tile a and s in sub-tile b (16 tokens each),
//   a > b:  e^{G_r - G_st(a)} * e^{G_st(a) - G_end(b)} * e^{G_end(b) - G_s}   (all <= 1)
//   a = b:  e^{G_r - G_st(a)} * e^{G_st(a) - G_end(a)} * e^{G_end(a) - G_s}   (middle <= e^{75})
// where st(a) is the first and end(b) the last token of a sub-tile.
//
// Output: one record per (chunk, head) holding the operand tiles in the exact
// shared-memory image the tcgen05 kernel consumes (fp16, K-major, 128-byte
// swizzle: 16-byte chunk j of row r stored at chunk position j ^ (r & 7)).
#include "kda_common.cuh"
#include "kda_chunk_layout.cuh"

namespace kda {
namespace {

constexpr int PT = 256;        // threads
constexpr int C = CHUNK_T;     // 64 tokens
constexpr int LDL = 129;       // padded fp32 row stride (bank-conflict free columns)
constexpr int LDS = 65;

__device__ __forceinline__ float bf(const __half* p) { return __half2float(*p); }

__global__ void __launch_bounds__(PT, 1) chunk_prep_kernel(PrepArgs a) {
    extern __shared__ __align__(16) float sm[];
    float* LK = sm;                  // [64][129] k * X   (X = e^{G_r - G_st(tile r)})
    float* LQ = LK + C * LDL;        // [64][129] q * X
    float* R = LQ + C * LDL;         // [64][129] k * Y   (Y = e^{G_end(tile s) - G_s})
    float* G = R + C * LDL;          // [64][128] G (rows past the chunk repeat the last row)
    float* Am = G + C * D;           // [64][65]  A (with beta)
    float* Pm = Am + C * LDS;        // [64][65]  P
    float* Tm = Pm + C * LDS;        // [64][65]  T
    float* Mt = Tm + C * LDS;        // [10][128] Z_a (4 diagonal tiles), C_ab (6 pairs a > b)
    float* bt = Mt + 10 * D;         // [64] beta

    const int H = a.H, W = H * D;
    const int chunk = blockIdx.x / H, h = blockIdx.x % H;
    const ChunkDesc cd = a.chunks[chunk];
    const int L = cd.len, t0 = cd.t0;
    const int tid = threadIdx.x;
    const __half* qh = static_cast<const __half*>(a.qh);
    const __half* kh = static_cast<const __half*>(a.kh);
    const __half* vh = static_cast<const __half*>(a.vh);
    const size_t hb = (size_t)h * D;
    auto gidx = [&](int r, int i) { return (size_t)(t0 + r) * W + hb + i; };

    // ---- 1a. cumulative gate and beta
    for (int idx = tid; idx < C * D; idx += PT) {
        const int r = idx / D, i = idx % D;
        const int rr = r < L ? r : L - 1;
        G[r * D + i] = a.gcum[gidx(rr, i)];
    }
    if (tid < C) bt[tid] = tid < L ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    __syncthreads();

    // ---- 1b. scaled operands of A and P, tile factors
    for (int idx = tid; idx < C * D; idx += PT) {
        const int r = idx / D, i = idx % D;
        const int st = r & ~15;
        const int en = min(st + 15, L - 1);
        const float g = G[r * D + i];
        const float X = expf(g - G[st * D + i]);
        const float Y = expf(G[en * D + i] - g);
        const float kv = r < L ? bf(kh + gidx(r, i)) : 0.f;
        const float qv = r < L ? bf(qh + gidx(r, i)) : 0.f;
        LK[r * LDL + i] = kv * X;
        LQ[r * LDL + i] = qv * X;
        R[r * LDL + i] = kv * Y;
    }
    for (int idx = tid; idx < 10 * D; idx += PT) {
        const int m = idx / D, i = idx % D;
        int ta, tb;
        if (m < 4) { ta = m; tb = m; }
        else { const int pairs[6][2] = {{1, 0}, {2, 0}, {3, 0}, {2, 1}, {3, 1}, {3, 2}}; ta = pairs[m - 4][0]; tb = pairs[m - 4][1]; }
        const int st = min(16 * ta, L - 1);
        const int en = min(16 * tb + 15, L - 1);
        Mt[m * D + i] = expf(G[st * D + i] - G[en * D + i]);
    }
    __syncthreads();

    // ---- 2. A and P, 4x4 pair blocks per thread
    {
        const int ti = tid / 16, tj = tid % 16;
        const int r0 = 4 * ti, s0 = 4 * tj;
        const int ta = r0 >> 4, tb = s0 >> 4;
        float accA[4][4], accP[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) { accA[x][y] = 0.f; accP[x][y] = 0.f; }
        if (tb <= ta) {
            int m;
            if (ta == tb) m = ta;
            else m = 4 + (tb == 0 ? ta - 1 : (tb == 1 ? 3 + ta - 2 : 5));
            const float* Mrow = Mt + m * D;
            for (int i = 0; i < D; ++i) {
                const float mm = Mrow[i];
                float lk[4], lq[4], rr[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    lk[x] = LK[(r0 + x) * LDL + i] * mm;
                    lq[x] = LQ[(r0 + x) * LDL + i] * mm;
                    rr[x] = R[(s0 + x) * LDL + i];
                }
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        accA[x][y] = fmaf(lk[x], rr[y], accA[x][y]);
                        accP[x][y] = fmaf(lq[x], rr[y], accP[x][y]);
                    }
            }
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const int r = r0 + x, s = s0 + y;
                Am[r * LDS + s] = (s < r) ? bt[r] * accA[x][y] : 0.f;
                Pm[r * LDS + s] = (s <= r) ? accP[x][y] : 0.f;
            }
    }
    __syncthreads();

    // ---- 3. T = (I + A)^{-1} Diag(beta), one column per thread
    if (tid < C) {
        const int j = tid;
        for (int r = 0; r < j; ++r) Tm[r * LDS + j] = 0.f;
        for (int r = j; r < C; ++r) {
            float t = (r == j) ? bt[r] : 0.f;
            for (int s = j; s < r; ++s) t = fmaf(-Am[r * LDS + s], Tm[s * LDS + j], t);
            Tm[r * LDS + j] = t;
        }
    }
    __syncthreads();

    unsigned char* rec = static_cast<unsigned char*>(a.records) + ((size_t)chunk * H + h) * REC_BYTES;

    // ---- 4. W = T (k e^G) (row-major tile [tok][key]) and U0^T = (T v)^T ([val][tok])
    {
        const int c = tid & 127;
        const bool isW = tid < 128;
        float xc[C];
#pragma unroll
        for (int s = 0; s < C; ++s) {
            float x = 0.f;
            if (s < L) x = isW ? bf(kh + gidx(s, c)) * expf(G[s * D + c]) : bf(vh + gidx(s, c));
            xc[s] = x;
        }
        uint32_t pack[4];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s <= r; ++s) acc = fmaf(Tm[r * LDS + s], xc[s], acc);
            if (isW) {
                *reinterpret_cast<__half*>(rec + REC_W + sw128_off(r, c, C)) = __float2half_rn(acc);
            } else {
                // pack 8 consecutive tokens of row `c` into one 16-byte chunk
                const uint32_t bits = (uint32_t)__half_as_ushort(__float2half_rn(acc));
                if ((r & 1) == 0) pack[(r & 7) >> 1] = bits;
                else pack[(r & 7) >> 1] |= bits << 16;
                if ((r & 7) == 7)
                    *reinterpret_cast<uint4*>(rec + REC_UT + sw128_off(c, r & ~7, 128)) =
                        make_uint4(pack[0], pack[1], pack[2], pack[3]);
            }
        }
    }

    // ---- 5. Q+ ([tok][key]), Kt^T ([key][tok]), P ([r][s]), decay
    for (int idx = tid; idx < C * 16; idx += PT) {      // Q+: 64 rows x 16 chunks of 8 keys
        const int r = idx / 16, ch = idx % 16;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int i = ch * 8 + e;
            v[e] = r < L ? bf(qh + gidx(r, i)) * expf(G[r * D + i]) : 0.f;
        }
        uint4 u;
        __half2* p2 = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) p2[e] = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
        *reinterpret_cast<uint4*>(rec + REC_Q + sw128_off(r, ch * 8, C)) = u;
    }
    for (int idx = tid; idx < D * 8; idx += PT) {       // Kt^T: 128 key rows x 8 chunks of 8 tokens
        const int key = idx % D, ch = idx / D;
        const float glast = G[(L - 1) * D + key];
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = ch * 8 + e;
            v[e] = s < L ? bf(kh + gidx(s, key)) * expf(glast - G[s * D + key]) : 0.f;
        }
        uint4 u;
        __half2* p2 = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) p2[e] = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
        *reinterpret_cast<uint4*>(rec + REC_KT + sw128_off(key, ch * 8, 128)) = u;
    }
    for (int idx = tid; idx < C * 8; idx += PT) {       // P: 64 rows x 8 chunks of 8 columns
        const int r = idx / 8, ch = idx % 8;
        uint4 u;
        __half2* p2 = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            p2[e] = __floats2half2_rn(Pm[r * LDS + ch * 8 + 2 * e], Pm[r * LDS + ch * 8 + 2 * e + 1]);
        *reinterpret_cast<uint4*>(rec + REC_P + sw128_off(r, ch * 8, C)) = u;
    }
    if (tid < D) {
        reinterpret_cast<float*>(rec + REC_DECAY)[tid] = expf(G[(L - 1) * D + tid]);
    }
}

}  // namespace

size_t chunk_prep_smem_bytes() {
    return sizeof(float) * (3 * C * LDL + C * D + 3 * C * LDS + 10 * D + C);
}

cudaError_t launch_chunk_prep(const PrepArgs& a, cudaStream_t s) {
    const size_t smem = chunk_prep_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.n_chunks * a.H;
    if (blocks == 0) return cudaSuccess;
    chunk_prep_kernel<<<(unsigned)blocks, PT, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
