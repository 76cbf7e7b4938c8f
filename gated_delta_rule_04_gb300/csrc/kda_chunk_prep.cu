// Chunk preparation of the chunked prefill, with the pre-stage fused in:
// from the raw projections of a 64-token chunk of one head to the record of
// operand tiles the tcgen05 recurrence consumes.  Everything here is
// independent of the recurrent state, so all (chunk, head) items run in
// parallel.
//
// Per item (sources: "Kimi Delta Attention (KDA) -- analysis & C kernel
// plan", sections "The KDA layer, precisely" and "Recurrence"; "ferrox-models
// 0.8.0, module kda", module overview; "Kimi K3 - Retention gate -
// OpenModelAtlas", gate formula):
//   1. short causal conv (kernel 4) + SiLU of q, k, v; q^ = q / |q| * q_scale,
//      k^ = k / |k| (eps inside the root); g = lb * sigmoid(e^A (z + dt_bias));
//      beta = sigmoid(b); G = chunk-local inclusive cumulative sum of g.
//   2. the chunked form ("chunked UT transform" with a per-channel cumulative
//      log gate, "memra-engine 0.124.0, module kda", PREFILL DISPATCH; 16-token
//      tiles kept in range by the lower bound, "Kimi K3 - Retention gate",
//      section "Why"):
//        A[r][s] = beta_r sum_i k_ri k_si e^{G_ri - G_si}   (s < r)
//        P[r][s] =        sum_i q_ri k_si e^{G_ri - G_si}   (s <= r)
//        T = (I + A)^{-1} Diag(beta),  W = T (k e^G),  U0 = T v,
//        Q+ = q e^G,  Kt = k e^{G_last - G},  decay = e^{G_last}
//      The recurrence then needs only U = U0 - W S, O = Q+ S + P U and
//      S' = Diag(decay) S + Kt^T U per chunk.
//
// Range.  For s in 16-token sub-tile b the reference point is the last token
// of b, en(b): e^{G_r - G_s} = e^{G_r - G_en(b)} Y_s with Y_s = e^{G_en(b) - G_s}
// <= 1.  For r in sub-tile a the left factor is iY_r C_ab with
// iY_r = e^{G_r - G_en(a)} in [1, e^{75}] and C_ab = e^{G_en(a) - G_en(b)} <= 1,
// which bf16 holds; a factor that underflows stands for a product far below
// every other term.
//
// Tensor cores.  A and the off-diagonal blocks of P are two bf16 M = 128 MMAs
// against the right operand R = k Y (N = 64, K = 128 keys).  The 256 left
// rows are the A rows grouped by column sub-tile b (64 + 48 + 32 + 16) and the
// off-diagonal P rows (48 + 32 + 16).  The diagonal blocks of P reach the
// output directly and need more than bf16: their operands are split into
// bf16 high and low parts: one N = 128 MMA multiplies [q hi; q lo] by
// [R hi | R lo] and the readout adds hi*hi + hi*lo + lo*hi, good to about 16 bits.  W = T (k e^G) and U0^T = v^T T^T are
// fp16 MMAs; the unit lower-triangular solve is fp32 on the CUDA cores
// (16 x 16 diagonal inverses, then the off-diagonal blocks diagonal by
// diagonal).
//
// Thread mapping of the element-wise part: warp w, lane l -> token octet
// o = w / 2 (tokens 8o .. 8o+7, inside sub-tile o / 2) and channel pair
// p = 32 (w % 2) + l (channels 2p, 2p+1).  Each thread keeps its 16 elements
// in registers from the conv to the operand tiles; token sums (L2 norms) are
// warp reduce-scatters plus one shared-memory exchange, and the cumulative
// gate is a per-thread running sum plus a prefix over octets.
//
// Schedule.  The grid is persistent (one CTA per SM, or fewer when the
// launch shares the GPU).  A CTA walks its items in head-major order, either a
// fixed contiguous range or batches taken from a work counter.  The next
// item's raw rows (TMA tensor copies) and its head's conv taps and dt_bias
// (bulk copies) arrive while the current item is being solved.
//
// Output: one record per (chunk, head) in the exact shared-memory image the
// recurrence kernel consumes (fp16, K-major, 128-byte swizzle).  Q+ and the
// decay are stored from registers; Kt, P, W and U0^T are assembled in shared
// memory and leave as contiguous bulk stores.
#include <type_traits>

#include "kda_chunk_layout.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int PT = 512;
constexpr int C = CHUNK_T;                 // 64 tokens
constexpr int RAW_ROWS = C + RING;         // raw q/k/v rows incl. the three before the chunk
constexpr uint32_t ROW_B = D * 2;          // one bf16 row of a head
constexpr int LDS = 68;                    // fp32 row stride of the 64 x 64 matrices (16-byte rows)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_D0 = 0, TM_D1 = 64, TM_D2 = 128, TM_W = 256, TM_U = 384;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;

// shared-memory map (bytes from a 1 KiB aligned base)
constexpr uint32_t S_RQ = 0;                               // bf16 [67][128] raw q (row 0 = token t0 - 3)
constexpr uint32_t S_RK = S_RQ + RAW_ROWS * ROW_B;
constexpr uint32_t S_RV = S_RK + RAW_ROWS * ROW_B;
constexpr uint32_t S_WUSTAGE = S_RQ;                       // between the conv stage and the next raw rows:
                                                           //   the previous item's W and U0^T (2 x 16 KiB)
constexpr uint32_t S_KTSTAGE = S_RQ + 32768;               //   and Kt (16 KiB), staged for bulk stores
constexpr uint32_t S_OPS = 52224;                          // operand region (1 KiB aligned)
constexpr uint32_t S_LAP = S_OPS;                          //   bf16 2 x [128 rows][128 keys]
constexpr uint32_t S_QD = S_OPS + 65536;                   //   bf16 [128][128]: rows 0-63 hi, 64-127 lo
constexpr uint32_t S_RHL = S_OPS + 98304;                  //   bf16 [128][128 keys] R: rows 0-63 hi, 64-127 lo
constexpr uint32_t S_AM = S_OPS;                           // after the first MMAs: fp32 [64][68] A
constexpr uint32_t S_XM = S_OPS + 17408;                   //   fp32 [64][68] X = (I + A)^{-1}
constexpr uint32_t S_TAPS = S_OPS + 36864;                 //   the next item's conv taps [3][128][4] and
                                                           //   dt_bias [128] (fp32), arriving with its raw rows
constexpr uint32_t TAPS_BYTES = 3 * 2048 + 512;
constexpr uint32_t S_PSTAGE = S_RHL;                       //   P (8 KiB), staged for a bulk store
constexpr uint32_t S_TT = S_OPS + 131072;                  // fp16 [64 r][64 s] T; the W product reads it as
                                                           //   128 A rows, rows 64-127 being the first 8 KiB of
                                                           //   the next tile (their output lanes are unused)
constexpr uint32_t S_KPT = S_TT + 8192;                    // fp16 [128 key][64 s] (k e^G)^T
constexpr uint32_t S_VT = S_KPT + 16384;                   // fp16 [128 val][64 s] v^T
constexpr uint32_t S_NRM = S_VT + 16384;                   // fp32 [16 warps][16] partial sums of squares
constexpr uint32_t S_TOT = S_NRM + 1024;                   // fp32 [8 octets][128] gate sums
constexpr uint32_t S_BT = S_TOT + 4096;                    // fp32 [64] beta
constexpr uint32_t S_BAR = S_BT + 256;                     // 3 mbarriers, TMEM slot, abort flag
constexpr uint32_t SMEM_BYTES = S_BAR + 64 + 1024;
static_assert(S_RV + RAW_ROWS * ROW_B <= S_OPS, "raw rows overlap the operand region");
static_assert(S_KTSTAGE + 16384 <= S_RV + RAW_ROWS * ROW_B, "Kt staging stays inside the raw rows");
static_assert(S_XM + 64 * LDS * 4 <= S_TAPS && S_TAPS + TAPS_BYTES <= S_QD, "solve tiles, taps");
static_assert(S_PSTAGE + 8192 <= S_OPS + 131072, "P staging");
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(S_TT + 16384 <= S_VT, "the W product's A rows stay inside the T and (k e^G)^T tiles");

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

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcpf(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 bf2f(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack8_f16(const float* v) {
    return make_uint4(pack_f16(v[0], v[1]), pack_f16(v[2], v[3]), pack_f16(v[4], v[5]), pack_f16(v[6], v[7]));
}
// named barrier over `count` threads (id 0 is __syncthreads)
__device__ __forceinline__ void bar_sync_n(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void sts32(unsigned char* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }

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

// Blockwise inverse X = (I + A)^{-1} over 16 x 16 blocks, once the diagonal
// blocks X_aa are known:  X_ab = -X_aa sum_{k=b}^{a-1} A_ak X_kb.  First
// At_ak = X_aa A_ak for every a > k (one pass, kept in A's unused upper block
// (k, a)); then one pass per block diagonal, X_ab = -sum_k At_ak X_kb.
// Thread = (block pair, row, 4 consecutive columns): one broadcast load of the
// left factor and one 16-byte load of the right row per 4 FMAs.
__device__ __forceinline__ void solve_premultiply(float* Am, const float* Xm, int tid) {
    if (tid < 6 * 64) {
        const int p = tid >> 6, r = (tid >> 2) & 15, c = 4 * (tid & 3);
        const int a = p < 3 ? p + 1 : (p < 5 ? p - 1 : 3);   // (a, k): (1,0) (2,0) (3,0) (2,1) (3,1) (3,2)
        const int k = p < 3 ? 0 : (p < 5 ? 1 : 2);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const float l = Xm[(16 * a + r) * LDS + 16 * a + s];
            const float4 m = *reinterpret_cast<const float4*>(Am + (16 * a + s) * LDS + 16 * k + c);
            acc.x = fmaf(l, m.x, acc.x); acc.y = fmaf(l, m.y, acc.y);
            acc.z = fmaf(l, m.z, acc.z); acc.w = fmaf(l, m.w, acc.w);
        }
        *reinterpret_cast<float4*>(Am + (16 * k + r) * LDS + 16 * a + c) = acc;
    }
    __syncthreads();
}

template <int Dg>
__device__ __forceinline__ void solve_level(const float* Am, float* Xm, int tid) {
    constexpr int nthr = (4 - Dg) * 64;
    const int b = tid >> 6, r = (tid >> 2) & 15, c = 4 * (tid & 3), a = b + Dg;
    if (tid < nthr) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int kk = 0; kk < Dg; ++kk)
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const float l = Am[(16 * (b + kk) + r) * LDS + 16 * a + s];   // At_{a, b+kk}[r][s]
                const float4 x = *reinterpret_cast<const float4*>(Xm + (16 * (b + kk) + s) * LDS + 16 * b + c);
                acc.x = fmaf(l, x.x, acc.x); acc.y = fmaf(l, x.y, acc.y);
                acc.z = fmaf(l, x.z, acc.z); acc.w = fmaf(l, x.w, acc.w);
            }
        *reinterpret_cast<float4*>(Xm + (16 * a + r) * LDS + 16 * b + c) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Raw q/k/v rows of one item into shared memory, issued by one warp: one TMA
// box per plane (the chunk and the three rows before it).  At a sequence
// start the three rows before the chunk belong to the conv ring (16-byte
// copies by the warp, awaited with cp.async.wait) or are zero (left unloaded
// and read as zero).  Rows past the end of the tensor read as zero;
// rows past the chunk are never used.
__device__ __forceinline__ void issue_raw(const PrepArgs& a, const ChunkDesc& cd, int h, uint32_t base, uint32_t bar,
                                          int lane) {
    const int W = a.H * D;
    if (lane == 0) {
        // one arrival on the barrier, expecting every byte below
        ptx::mbar_expect_tx(bar, TAPS_BYTES + (cd.pos > 0 ? 3u * RAW_ROWS * ROW_B : 3u * C * ROW_B));
        // the head's conv taps and dt_bias
#pragma unroll
        for (int pl = 0; pl < 3; ++pl)
            ptx::bulk_g2s(base + S_TAPS + pl * 2048, a.conv_w + ((size_t)pl * W + h * D) * CONV_K, 2048, bar);
        ptx::bulk_g2s(base + S_TAPS + 3 * 2048, a.dt_bias + h * D, 512, bar);
        if (cd.pos > 0) {
#pragma unroll
            for (int pl = 0; pl < 3; ++pl)
                ptx::tma_load_2d(base + S_RQ + (uint32_t)pl * RAW_ROWS * ROW_B, &a.map67[pl], h * D, cd.t0 - RING, bar);
        } else {
#pragma unroll
            for (int pl = 0; pl < 3; ++pl)
                ptx::tma_load_2d(base + S_RQ + (uint32_t)pl * RAW_ROWS * ROW_B + RING * ROW_B, &a.map64[pl], h * D,
                                 cd.t0, bar);
        }
    }
    if (cd.pos == 0 && a.ring_in != nullptr) {
        for (int i = lane; i < 3 * RING * 16; i += 32) {
            const int pl = i / (RING * 16), r = (i / 16) % RING, piece = i & 15;  // ring slot r = raw row r
            const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.ring_in) +
                                       (((size_t)cd.seq * 3 + pl) * RING + r) * W + (size_t)h * D;
            cp_async16(base + S_RQ + (uint32_t)pl * RAW_ROWS * ROW_B + (uint32_t)r * ROW_B + 16 * piece,
                       src + 8 * piece);
        }
        cp_async_commit();
    }
}

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 h2f(uint32_t u) { return __half22float2(*reinterpret_cast<const __half2*>(&u)); }

__global__ void __launch_bounds__(PT, 1) chunk_prep_kernel(const __grid_constant__ PrepArgs a) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sb = smem_raw + (base - raw);
    float* Am = reinterpret_cast<float*>(sb + S_AM);
    float* Xm = reinterpret_cast<float*>(sb + S_XM);
    float* nrm = reinterpret_cast<float*>(sb + S_NRM);
    float* tot = reinterpret_cast<float*>(sb + S_TOT);
    float* bt = reinterpret_cast<float*>(sb + S_BT);
    const uint32_t bar_raw = base + S_BAR, bar_mma1 = base + S_BAR + 8, bar_mma2 = base + S_BAR + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sb + S_BAR + 24);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sb + S_BAR + 28);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, W = H * D;
    const int n_items = a.n_chunks * H;
    const int o = warp >> 1;                       // token octet
    const int a_sub = o >> 1;                      // 16-token sub-tile of the octet
    const int c0 = 2 * (32 * (warp & 1) + lane);   // first of this thread's two channels
    const int tok0 = 8 * o;

    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(bar_raw, 1);
        ptx::mbar_init(bar_mma1, 1);
        ptx::mbar_init(bar_mma2, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // gate inputs (this thread's tokens and channels) and the beta logit of an
    // item, loaded into registers one item ahead of use
    uint32_t zr[8];
    unsigned short b_raw = 0;   // bf16 bits

    auto load_zb = [&](const ChunkDesc& cn, int hn) {
        const uint32_t* zp = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.z) +
                                                               (size_t)(cn.t0 + tok0) * W + hn * D + c0);
#pragma unroll
        for (int j = 0; j < 8; ++j) zr[j] = tok0 + j < cn.len ? __ldcg(zp + (size_t)j * (W / 2)) : 0u;
        b_raw = tid < cn.len ? static_cast<const unsigned short*>(a.b)[(size_t)(cn.t0 + tid) * H + hn] : 0;
    };

    // This CTA's items, in head-major order (item j is chunk j % n_chunks of head
    // j / n_chunks, so consecutive items share their head's constants): either one
    // contiguous range, or batches of a.batch taken from the work counter one
    // batch ahead (the next item must be known an item ahead for its loads).
    // [jt, j_stop) is the current batch and nb_start the first item of the next.
    const int NC = a.n_chunks;
    volatile int* s_take = reinterpret_cast<volatile int*>(sb + S_BAR + 32);
    int jt, j_stop, nb_start;
    if (a.work_counter != nullptr) {
        if (tid == 0) {
            s_take[0] = atomicAdd(a.work_counter, 1);
            s_take[1] = atomicAdd(a.work_counter, 1);
        }
        __syncthreads();
        jt = min(s_take[0] * a.batch, n_items);
        j_stop = min(jt + a.batch, n_items);
        nb_start = min(s_take[1] * a.batch, n_items);
        __syncthreads();   // read before the loop rewrites s_take
    } else {
        jt = (int)(((int64_t)blockIdx.x * n_items) / gridDim.x);
        j_stop = (int)(((int64_t)(blockIdx.x + 1) * n_items) / gridDim.x);
        nb_start = n_items;
    }
    // chunk descriptor of the current item, carried from the previous iteration
    ChunkDesc cd = jt < j_stop ? a.chunks[jt % NC] : ChunkDesc{0, 0, 0, 0};
    if (jt < j_stop) {
        if (warp == PT / 32 - 1) issue_raw(a, cd, jt / NC, base, bar_raw, lane);
        load_zb(cd, jt / NC);
    }
    // in-flight bookkeeping for the drain after a timeout: a raw load issued by
    // the last warp and not yet consumed (flag in that warp's lane 0), and the
    // MMAs of thread 0 (1 = bar_mma1, 2 = bar_mma2 in flight)
    int pend_raw = jt < j_stop && tid == PT - 32;
    uint32_t raw_par = 0;                           // phase parity of that load
    int mma_pending = 0;
    uint32_t mma_par = 0;                           // phase parity of those MMAs
    uint32_t k_iter = 0;

    // W (lanes = tokens 0-63) and U0^T (lanes = values) of an item, from TMEM to its
    // record, by warps 4-15 (warps 0-3 issue the first MMAs meanwhile): warp w reads TMEM
    // lane quarter w % 4 and, with gq = w / 4 - 1, the 16-column groups
    // W: 3gq .. 3gq+2 (gq 2: 6-7; quarters 0-1 only), U0^T: {0,1}, {2}, {3}.
    // The two tiles are assembled in shared memory in their record image and
    // leave as two contiguous 16 KiB bulk stores (16-byte pieces scattered over
    // 128-byte lines would cost one memory transaction each).  Every caller is
    // CTA-uniform; warps 4-15 meet at named barrier 2.
    unsigned char* rec_prev = nullptr;
    auto wu_out = [&](unsigned char* rp) {
        if (warp < 4) return;
        const int qd = warp & 3, gq = (warp >> 2) - 1;
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        auto group_out = [&](uint32_t tcol, unsigned char* dst, int row, int col, int rows) {
            float v[16];
            tmem_ld16(tl + tcol, v);
            *reinterpret_cast<uint4*>(dst + sw128_off(row, col, rows)) = pack8_f16(v);
            *reinterpret_cast<uint4*>(dst + sw128_off(row, col + 8, rows)) = pack8_f16(v + 8);
        };
        if (qd < 2) {
            const int wend = gq == 2 ? 8 : 3 * gq + 3;
#pragma unroll 1
            for (int c = 3 * gq; c < wend; ++c) group_out(TM_W + 16 * c, sb + S_WUSTAGE, 32 * qd + lane, 16 * c, C);
        }
#pragma unroll 1
        for (int c = gq == 0 ? 0 : gq + 1; c < gq + 2; ++c)
            group_out(TM_U + 16 * c, sb + S_WUSTAGE + 16384, 32 * qd + lane, 16 * c, 128);
        ptx::fence_async_smem();
        bar_sync_n(2, PT - 128);
        if (tid == PT - 32) {
            ptx::bulk_s2g(rp + REC_W, base + S_WUSTAGE, 8192);                  // W keys 0-63
            ptx::bulk_s2g(rp + REC_W + REC_PANEL, base + S_WUSTAGE + 8192, 8192);  // W keys 64-127
            ptx::bulk_s2g(rp + REC_UT, base + S_WUSTAGE + 16384, 16384);
            ptx::bulk_commit();
        }
    };

#pragma unroll 1
    while (jt < j_stop) {
        const uint32_t par = k_iter & 1u;
        const int h = jt / NC, len = cd.len;
        // the next item's descriptor, read now so that nothing waits on it later
        const bool last_of_batch = jt + 1 == j_stop;
        const int next = last_of_batch ? nb_start : jt + 1;
        const bool has_next = next < n_items;
        const ChunkDesc cn = a.chunks[(has_next ? next : jt) % NC];
        const int hn = next / NC;
        unsigned char* rec = static_cast<unsigned char*>(a.records) + ((size_t)(jt % NC) * H + h) * REC_BYTES;

        const float eA = __expf(__ldg(a.A_log + h));   // used late in the conv stage
        const bool zero_halo = cd.pos == 0 && a.ring_in == nullptr;

        // raw rows, conv taps and dt_bias of this item
        if (!ptx::mbar_wait(bar_raw, par, WAIT_LIMIT_NS)) *abort_flag = 1;
        else pend_raw = 0;
        cp_async_wait_all();   // ring rows at a sequence start
        __syncthreads();
        if (*abort_flag) break;
        float2 wt[3][4];   // conv taps of the two channels
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
            const float4 w0 = *reinterpret_cast<const float4*>(sb + S_TAPS + pl * 2048 + 16 * c0);
            const float4 w1 = *reinterpret_cast<const float4*>(sb + S_TAPS + pl * 2048 + 16 * c0 + 16);
            // taps times 1/2: the conv yields x/2, the argument of tanh in the SiLU
            wt[pl][0] = make_float2(0.5f * w0.x, 0.5f * w1.x); wt[pl][1] = make_float2(0.5f * w0.y, 0.5f * w1.y);
            wt[pl][2] = make_float2(0.5f * w0.z, 0.5f * w1.z); wt[pl][3] = make_float2(0.5f * w0.w, 0.5f * w1.w);
        }
        const float2 dtb = *reinterpret_cast<const float2*>(sb + S_TAPS + 3 * 2048 + 4 * c0);

        // ---- 1. conv + SiLU of q, k, v (kept as fp16 pairs); gate; sums of squares.
        // Octets inside the chunk (all but a ragged tail) skip the token masks.
        uint32_t aq[8], ak[8], av[8];
        float sq[16];
        float2 gc[8];
        float2 run = make_float2(0.f, 0.f);
        const bool halo0 = zero_halo && tok0 == 0;        // rows 0-2 read as zero
        const float2 gsc = f2(-eA * LOG2E);                 // gate argument: (z + dt_bias) e^A, as -log2 e units
        const float2 gof = __fmul2_rn(dtb, gsc);
        const float2 lb2 = f2(a.lb);
        auto stage = [&](auto full_c) {
            constexpr bool FULL = decltype(full_c)::value;
#pragma unroll
            for (int pl = 0; pl < 3; ++pl) {
                float2 xr[11];
#pragma unroll
                for (int j = 0; j < 11; ++j) {
                    const uint32_t u =
                        *reinterpret_cast<const uint32_t*>(sb + S_RQ + pl * RAW_ROWS * ROW_B + (tok0 + j) * ROW_B + 2 * c0);
                    xr[j] = bf2f(u);
                    if (j < RING && halo0) xr[j] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // h = x / 2;  x sigmoid(x) = h + h tanh(h), tanh in half precision: the
                    // result is rounded to fp16 next, and the error (about 2^-11 of x) is at that level
                    float2 hx = __fmul2_rn(wt[pl][0], xr[j]);
                    hx = __ffma2_rn(wt[pl][1], xr[j + 1], hx);
                    hx = __ffma2_rn(wt[pl][2], xr[j + 2], hx);
                    hx = __ffma2_rn(wt[pl][3], xr[j + 3], hx);
                    const __half2 hin = __float22half2_rn(hx);
                    uint32_t t;
                    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hin)));
                    const float2 y = __ffma2_rn(hx, h2f(t), hx);
                    const bool valid = FULL || tok0 + j < len;
                    const uint32_t hv = valid ? pack_f16(y.x, y.y) : 0u;
                    const float yy = valid ? fmaf(y.x, y.x, y.y * y.y) : 0.f;
                    if (pl == 0) { aq[j] = hv; sq[j] = yy; }
                    if (pl == 1) { ak[j] = hv; sq[8 + j] = yy; }
                    if (pl == 2) av[j] = hv;
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 sarg = __ffma2_rn(bf2f(zr[j]), gsc, gof);
                const float2 g = __fmul2_rn(lb2, make_float2(rcpf(1.f + ex2f(sarg.x)), rcpf(1.f + ex2f(sarg.y))));
                if (FULL || tok0 + j < len) run = __fadd2_rn(run, g);
                gc[j] = run;
            }
        };
        if (tok0 + 8 <= len) stage(std::true_type{});
        else stage(std::false_type{});
        // sums of squares of q (values 0-7) and k (8-15) per token, reduce-scattered
        // over the warp: afterwards lanes 2v and 2v+1 hold value v's sum over 64 channels
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool up = lane & 16;
            const float send = up ? sq[i] : sq[i + 8], keep = up ? sq[i + 8] : sq[i];
            sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool up = lane & 8;
            const float send = up ? sq[i] : sq[i + 4], keep = up ? sq[i + 4] : sq[i];
            sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const bool up = lane & 4;
            const float send = up ? sq[i] : sq[i + 2], keep = up ? sq[i + 2] : sq[i];
            sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
            const bool up = lane & 2;
            const float send = up ? sq[0] : sq[1], keep = up ? sq[1] : sq[0];
            sq[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], 1);
        if ((lane & 1) == 0) nrm[warp * 16 + (lane >> 1)] = sq[0];
        *reinterpret_cast<float2*>(tot + o * D + c0) = run;
        if (tid < C) bt[tid] = tid < len ? rcpf(1.f + ex2f(-__uint_as_float((uint32_t)b_raw << 16) * LOG2E)) : 0.f;
        // the previous item's staged P has left the operand region
        if (tid == PT - 32) ptx::bulk_wait_read_all();
        __syncthreads();

        // ---- norms (lane 2v, 2v+1 computes value v; then broadcast)
        float nv;
        {
            const int v = lane >> 1;
            const float ss = nrm[(2 * o) * 16 + v] + nrm[(2 * o + 1) * 16 + v];
            nv = rsqrtf(ss + a.l2_eps) * (v < 8 ? a.q_scale : 1.f);
        }
        // ---- cumulative gate: prefix over octets, sub-tile ends, last token
        float2 pre = make_float2(0.f, 0.f), gen[4];
        {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int oo = 0; oo < 8; ++oo) {
                const float2 t2 = *reinterpret_cast<const float2*>(tot + oo * D + c0);
                if (oo == o) pre = acc;
                acc = __fadd2_rn(acc, t2);
                if (oo & 1) gen[oo >> 1] = acc;
            }
        }
        const float2 ge = a_sub == 0 ? gen[0] : a_sub == 1 ? gen[1] : a_sub == 2 ? gen[2] : gen[3];
        const float2 L2 = f2(LOG2E);
        // per-channel factors: E = e^{G_en(a)}, F = e^{G_last - G_en(a)}, Cb = e^{G_en(a) - G_en(b)}
        const float2 E = make_float2(ex2f(ge.x * LOG2E), ex2f(ge.y * LOG2E));
        const float2 F = make_float2(ex2f((gen[3].x - ge.x) * LOG2E), ex2f((gen[3].y - ge.y) * LOG2E));
        float2 Cb[3];
#pragma unroll
        for (int b = 0; b < 3; ++b) Cb[b] = make_float2(ex2f((ge.x - gen[b].x) * LOG2E), ex2f((ge.y - gen[b].y) * LOG2E));
        if (o == 0)
            *reinterpret_cast<float2*>(rec + REC_DECAY + 4 * c0) =
                make_float2(ex2f(gen[3].x * LOG2E), ex2f(gen[3].y * LOG2E));
        const float2 dofs = __fmul2_rn(__fadd2_rn(pre, make_float2(-ge.x, -ge.y)), L2);  // (G_oct_start - G_en(a)) log2 e

        // ---- 2. operand tiles.  Per token: R (hi, lo), the A / P left rows, the
        // diagonal P rows (hi, lo), Q+ and Kt to the record; (k e^G) and v stay
        // packed for the later fp16 MMAs.
        uint32_t kt[2][4], kp[2][4], vp[2][4];
        uint32_t kt_prev = 0, kp_prev = 0;
        // Store addresses.  Every row-major tile here is K-major with the 128-byte
        // swizzle and every row index is (multiple of 8) + j, so element (row0 + j,
        // c0) sits at  tile + row-block offset + colpart + 128 j + ((lane/4 ^ j) << 4).
        const uint32_t colpart = (uint32_t)(warp & 1) * 16384u + 4u * (lane & 3);   // 128-row tiles
        const uint32_t colrec = (uint32_t)(warp & 1) * REC_PANEL + 4u * (lane & 3); // Q+ record panels
        const uint32_t chunk = (uint32_t)lane >> 2;
        auto lap_off = [&](int row0) {   // row0: LAP row of token tok0 (a multiple of 8)
            return (uint32_t)(row0 >> 7) * 32768u + (uint32_t)(row0 & 127) * 128u + colpart;
        };
        constexpr int kRowA[4] = {0, 48, 80, 96};     // LAP row - r of the A rows of column sub-tile b
        constexpr int kRowP[3] = {144, 176, 192};     // LAP row - r of the off-diagonal P rows of b
        const int rowA_diag = (a_sub == 0 ? 0 : a_sub == 1 ? 48 : a_sub == 2 ? 80 : 96) + tok0;
        const uint32_t offA_diag = lap_off(rowA_diag);
        unsigned char* const sRHL = sb + S_RHL + (uint32_t)tok0 * 128u + colpart;
        unsigned char* const sQD = sb + S_QD + (uint32_t)tok0 * 128u + colpart;
        unsigned char* const sLAP = sb + S_LAP;
        unsigned char* const gQ = rec + REC_Q + (uint32_t)tok0 * 128u + colrec;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t jo = 128u * j + ((chunk ^ j) << 4);   // row j of the 8-row block, swizzled
            const float nq = __shfl_sync(0xffffffffu, nv, 2 * j);
            const float nk = __shfl_sync(0xffffffffu, nv, 16 + 2 * j);
            const float2 q = __fmul2_rn(h2f(aq[j]), f2(nq));
            const float2 k = __fmul2_rn(h2f(ak[j]), f2(nk));
            const float2 d = __ffma2_rn(gc[j], L2, dofs);                  // (G_r - G_en(a)) log2 e >= 0
            const float2 y = make_float2(ex2f(-d.x), ex2f(-d.y));          // Y  = e^{G_en(a) - G_r} <= 1
            const float2 iy = make_float2(ex2f(d.x), ex2f(d.y));           // iY = e^{G_r - G_en(a)} >= 1
            const float2 ky = __fmul2_rn(k, y);
            const uint32_t rh = pack_bf16(ky.x, ky.y);
            const float2 rhf = bf2f(rh);
            const float2 rlo = __fadd2_rn(ky, make_float2(-rhf.x, -rhf.y));
            sts32(sRHL + jo, rh);
            sts32(sRHL + 64 * 128 + jo, pack_bf16(rlo.x, rlo.y));
            const float2 ki = __fmul2_rn(k, iy), qi = __fmul2_rn(q, iy);
            sts32(sLAP + offA_diag + jo, pack_bf16(ki.x, ki.y));      // A row of the diagonal sub-tile
#pragma unroll
            for (int b = 0; b < 3; ++b) {
                if (b < a_sub) {
                    const float2 kf = __fmul2_rn(ki, Cb[b]), qf = __fmul2_rn(qi, Cb[b]);
                    sts32(sLAP + lap_off(kRowA[b] + tok0) + jo, pack_bf16(kf.x, kf.y));
                    sts32(sLAP + lap_off(kRowP[b] + tok0) + jo, pack_bf16(qf.x, qf.y));
                }
            }
            const uint32_t qh = pack_bf16(qi.x, qi.y);
            const float2 qhf = bf2f(qh);
            const float2 qlo = __fadd2_rn(qi, make_float2(-qhf.x, -qhf.y));
            sts32(sQD + jo, qh);
            sts32(sQD + 64 * 128 + jo, pack_bf16(qlo.x, qlo.y));
            // record: Q+ = q e^{G} = q iY E
            const float2 qp = __fmul2_rn(qi, E);
            *reinterpret_cast<uint32_t*>(gQ + jo) = pack_f16(qp.x, qp.y);
            // Kt = k e^{G_last - G} = k Y F;  (k e^G) = k iY E;  v.  Pairs of tokens are
            // transposed into per-channel rows: word w of channel e holds tokens 2w, 2w+1.
            const float2 ktf = __fmul2_rn(ky, F), kpf = __fmul2_rn(ki, E);
            const uint32_t t_kt = pack_f16(ktf.x, ktf.y), t_kp = pack_f16(kpf.x, kpf.y);
            if (j & 1) {
                const int w = j >> 1;
                kt[0][w] = __byte_perm(kt_prev, t_kt, 0x5410);
                kt[1][w] = __byte_perm(kt_prev, t_kt, 0x7632);
                kp[0][w] = __byte_perm(kp_prev, t_kp, 0x5410);
                kp[1][w] = __byte_perm(kp_prev, t_kp, 0x7632);
                vp[0][w] = __byte_perm(av[j - 1], av[j], 0x5410);
                vp[1][w] = __byte_perm(av[j - 1], av[j], 0x7632);
            } else {
                kt_prev = t_kt;
                kp_prev = t_kp;
            }
        }
        // the previous item's W / U0 MMAs read (k e^G)^T, v^T and T: they have long finished
        if (k_iter > 0 && !ptx::mbar_wait(bar_mma2, par ^ 1u, WAIT_LIMIT_NS)) *abort_flag = 1;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            *reinterpret_cast<uint4*>(sb + S_KTSTAGE + sw128_off(c0 + e, tok0, 128)) =
                make_uint4(kt[e][0], kt[e][1], kt[e][2], kt[e][3]);
            *reinterpret_cast<uint4*>(sb + S_KPT + sw128_off(c0 + e, tok0, 128)) =
                make_uint4(kp[e][0], kp[e][1], kp[e][2], kp[e][3]);
            *reinterpret_cast<uint4*>(sb + S_VT + sw128_off(c0 + e, tok0, 128)) =
                make_uint4(vp[e][0], vp[e][1], vp[e][2], vp[e][3]);
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == PT - 32) {
            ptx::bulk_s2g(rec + REC_KT, base + S_KTSTAGE, 16384);
            ptx::bulk_commit();
        }
        // no one sets the abort flag between here and the first-MMA wait, so this
        // read is the same in every thread
        const bool live = !*abort_flag;

        // ---- 3. A, off-diagonal P, diagonal P on the tensor cores
        constexpr uint32_t IDESC_BF16_N64 = ptx::idesc_bf16_f32(128, 64);
        constexpr uint32_t IDESC_BF16_N128 = ptx::idesc_bf16_f32(128, 128);
        if (tid == 0) {
            ptx::tc_fence_after();
            // three independent accumulator chains, interleaved by K step: A and the
            // off-diagonal P (two M = 128 halves of the left rows) and the diagonal P
            // ([q hi; q lo] x [R hi; R lo], N = 128; the readout adds hi*hi + hi*lo + lo*hi)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t koff = (kk & 3) * 32, pn = kk >> 2;
                const uint64_t bR = ptx::sdesc_sw128(base + S_RHL + pn * 16384 + koff);   // R hi rows
                ptx::mma_f16(tmem + TM_D0, ptx::sdesc_sw128(base + S_LAP + pn * 16384 + koff), bR, IDESC_BF16_N64, kk > 0);
                ptx::mma_f16(tmem + TM_D1, ptx::sdesc_sw128(base + S_LAP + 32768 + pn * 16384 + koff), bR, IDESC_BF16_N64,
                             kk > 0);
                ptx::mma_f16(tmem + TM_D2, ptx::sdesc_sw128(base + S_QD + pn * 16384 + koff), bR, IDESC_BF16_N128, kk > 0);
            }
            ptx::mma_commit(bar_mma1);
            mma_pending = 1;
            mma_par = par;
        }
        // the previous item's W and U0^T (warps 4-15) while the MMAs run; then the
        // next item's gate inputs
        if (k_iter > 0 && live) {
            ptx::tc_fence_after();
            wu_out(rec_prev);
        }
        if (has_next) load_zb(cn, hn);
        if (!ptx::mbar_wait(bar_mma1, par, WAIT_LIMIT_NS)) *abort_flag = 1;
        ptx::tc_fence_after();
        if (tid == 0 && !*abort_flag) mma_pending = 0;

        // ---- 4. read out A (to fp32 Am, times beta_r) and P (to the record)
        if (!*abort_flag) {
            if (warp < 8) {
                const int row = 128 * (warp >> 2) + 32 * (warp & 3) + lane;
                const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (warp < 4 ? TM_D0 : TM_D1);
                const int g = group_of(row);
                const int isP = kGroup[g][0], b = kGroup[g][1];
                const int r = kGroup[g][2] + (row - kGroup[g][3]);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float v[16];
                    tmem_ld16(taddr + 16 * q4, v);
                    if (q4 == b) {
                        if (isP) {
                            *reinterpret_cast<uint4*>(sb + S_PSTAGE + sw128_off(r, 16 * b, C)) = pack8_f16(v);
                            *reinterpret_cast<uint4*>(sb + S_PSTAGE + sw128_off(r, 16 * b + 8, C)) = pack8_f16(v + 8);
                        } else {  // beta_r A, strictly lower part (zeros above in the diagonal block)
                            const float be = bt[r];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                float4 w4;
                                w4.x = 16 * b + 4 * q + 0 < r ? be * v[4 * q + 0] : 0.f;
                                w4.y = 16 * b + 4 * q + 1 < r ? be * v[4 * q + 1] : 0.f;
                                w4.z = 16 * b + 4 * q + 2 < r ? be * v[4 * q + 2] : 0.f;
                                w4.w = 16 * b + 4 * q + 3 < r ? be * v[4 * q + 3] : 0.f;
                                *reinterpret_cast<float4*>(Am + r * LDS + 16 * b + 4 * q) = w4;
                            }
                        }
                    }
                }
            } else if (warp < 12) {
                // diagonal P blocks: D2 rows are [q hi; q lo], columns [R hi | R lo].
                // Warps 10-11 hand the lo*hi terms (lanes 64-127) to warps 8-9 through
                // shared memory; warps 8-9 add hi*hi + hi*lo + lo*hi.
                float* pdl = tot;   // fp32 [64 r][16]; the gate totals are no longer needed
                const int qd = warp & 3;
                const int r = 32 * (qd & 1) + lane;                    // 0..63
                const int ta = r >> 4;
                const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + TM_D2;
                if (qd >= 2) {
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const int blk = 2 * (qd & 1) + q2;             // sub-tiles of this warp's rows
                        float v[16];
                        tmem_ld16(taddr + 16 * blk, v);                // q lo x R hi
                        if (blk == ta) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                *reinterpret_cast<float4*>(pdl + r * 16 + 4 * q) =
                                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        }
                    }
                }
                bar_sync_n(1, 128);
                if (qd < 2) {
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        const int blk = 2 * qd + q2;
                        float v[16], w[16];
                        tmem_ld16(taddr + 16 * blk, v);                // q hi x R hi
                        tmem_ld16(taddr + 64 + 16 * blk, w);           // q hi x R lo
                        if (blk == ta) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float4 l4 = *reinterpret_cast<const float4*>(pdl + r * 16 + 4 * q);
                                v[4 * q] += w[4 * q] + l4.x;
                                v[4 * q + 1] += w[4 * q + 1] + l4.y;
                                v[4 * q + 2] += w[4 * q + 2] + l4.z;
                                v[4 * q + 3] += w[4 * q + 3] + l4.w;
                            }
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                if (16 * ta + jj > r) v[jj] = 0.f;
                            *reinterpret_cast<uint4*>(sb + S_PSTAGE + sw128_off(r, 16 * ta, C)) = pack8_f16(v);
                            *reinterpret_cast<uint4*>(sb + S_PSTAGE + sw128_off(r, 16 * ta + 8, C)) = pack8_f16(v + 8);
                        }
                    }
                    for (int tb = ta + 1; tb < 4; ++tb) {
                        *reinterpret_cast<uint4*>(sb + S_PSTAGE + sw128_off(r, 16 * tb, C)) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(sb + S_PSTAGE + sw128_off(r, 16 * tb + 8, C)) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;
        // the last warp (idle in the solve) stores P and fetches the next item's raw
        // rows and taps, once the staged W, U0^T and Kt have been read from that memory
        if (warp == PT / 32 - 1) {
            if (lane == 0) {
                ptx::bulk_s2g(rec + REC_P, base + S_PSTAGE, 8192);
                ptx::bulk_commit();
                ptx::bulk_wait_read_all();
            }
            __syncwarp();
            if (has_next) {
                issue_raw(a, cn, hn, base, bar_raw, lane);
                if (lane == 0) { pend_raw = 1; raw_par = (k_iter + 1) & 1u; }
            }
        }

        // ---- 5. X = (I + A)^{-1}: diagonal 16 x 16 inverses by forward substitution
        if (tid < 64) {
            const int ta = tid >> 4, j = tid & 15;
            const int ob = 16 * ta;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                // x_r = e_j - sum_{s<r} A[r][s] x_s, as four interleaved partial sums
                const float* Lr = Am + (ob + r) * LDS + ob;
                float p[4] = {(r == j) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; 4 * q < r; ++q) {
                    const float4 l4 = *reinterpret_cast<const float4*>(Lr + 4 * q);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * q + e < r) p[e] = fmaf(-lv[e], x[4 * q + e], p[e]);
                }
                x[r] = (r < j) ? 0.f : (p[0] + p[1]) + (p[2] + p[3]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Xm[(ob + r) * LDS + ob + j] = x[r];
        }
        // the batch after the next one (read at the end of this item)
        if (tid == PT - 32 && last_of_batch && a.work_counter != nullptr) s_take[0] = atomicAdd(a.work_counter, 1);
        __syncthreads();
        solve_premultiply(Am, Xm, tid);
        solve_level<1>(Am, Xm, tid);
        solve_level<2>(Am, Xm, tid);
        solve_level<3>(Am, Xm, tid);

        // ---- 6. T = X Diag(beta) (fp16, blocks above the diagonal zero)
        {
            const int r = tid >> 3, ch = tid & 7;   // 512 threads = 64 rows x 8 column groups
            float v[8], xr[8], b8[8];
            lds8(Xm + r * LDS + 8 * ch, xr);
            lds8(bt + 8 * ch, b8);
            const bool keep = (ch >> 1) <= (r >> 4);   // blocks above the diagonal are zero
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = keep ? xr[e] * b8[e] : 0.f;
            *reinterpret_cast<uint4*>(sb + S_TT + sw128_off(r, 8 * ch, 128)) = pack8_f16(v);
        }
        ptx::fence_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            ptx::tc_fence_after();
            constexpr uint32_t IDESC_W = ptx::idesc_f16_f32(128, 128);
            constexpr uint32_t IDESC_U = ptx::idesc_f16_f32(128, 64);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t dT = ptx::sdesc_sw128(base + S_TT + kk * 32);
                ptx::mma_f16(tmem + TM_W, dT, ptx::sdesc_sw128(base + S_KPT + kk * 32), IDESC_W, kk > 0);
                ptx::mma_f16(tmem + TM_U, ptx::sdesc_sw128(base + S_VT + kk * 32), dT, IDESC_U, kk > 0);
            }
            ptx::mma_commit(bar_mma2);
            mma_pending = 2;
            mma_par = par;
        }
        // W and U0^T of this item are read out while the next item's first MMAs run
        rec_prev = rec;
        cd = cn;
        ptx::tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;
        ++k_iter;
        if (!last_of_batch) {
            ++jt;
        } else {
            jt = nb_start;
            j_stop = min(nb_start + a.batch, n_items);
            nb_start = a.work_counter != nullptr ? min(s_take[0] * a.batch, n_items) : n_items;
        }
    }

    // (the loop leaves right after a barrier, so the flag reads the same everywhere)
    if (!*abort_flag && rec_prev != nullptr) {
        if (!ptx::mbar_wait(bar_mma2, (k_iter - 1) & 1u, WAIT_LIMIT_NS)) *abort_flag = 1;
        ptx::tc_fence_after();
        if (tid == PT - 32) ptx::bulk_wait_read_all();   // the staging tiles are free
        __syncthreads();
        if (!*abort_flag) wu_out(rec_prev);
        if (tid == 0 && !*abort_flag) mma_pending = 0;
    }
    if (tid == PT - 32) ptx::bulk_wait_all();   // the staged record stores have landed
    cp_async_wait_all();  // this thread's copies of a prefetch that was not consumed
    if (*abort_flag && pend_raw) ptx::mbar_wait(bar_raw, raw_par, WAIT_LIMIT_NS);
    if (*abort_flag && tid == 0) {
        // record the timeout, then let this CTA's own MMAs land
        atomicExch(a.status, ERR_TIMEOUT);
        if (mma_pending == 1) ptx::mbar_wait(bar_mma1, mma_par, WAIT_LIMIT_NS);
        if (mma_pending == 2) ptx::mbar_wait(bar_mma2, mma_par, WAIT_LIMIT_NS);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

size_t chunk_prep_smem_bytes() { return SMEM_BYTES; }

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// [T][W] bf16 tensor, boxes of `rows` rows x 128 channels, zero fill out of bounds
bool encode_rows(CUtensorMap* m, const void* base, int64_t T, int64_t W, uint32_t rows) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)W, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)W * 2};
    const cuuint32_t box[2] = {(cuuint32_t)D, rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_prep(const PrepArgs& args, cudaStream_t s, int max_ctas) {
    const int64_t items = (int64_t)args.n_chunks * args.H;
    if (items == 0) return cudaSuccess;
    if (items > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    PrepArgs a = args;
    const void* planes[3] = {a.q, a.k, a.v};
    for (int pl = 0; pl < 3; ++pl)
        if (!encode_rows(&a.map67[pl], planes[pl], a.T, (int64_t)a.H * D, RAW_ROWS) ||
            !encode_rows(&a.map64[pl], planes[pl], a.T, (int64_t)a.H * D, C))
            return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int64_t grid = items < sms ? items : sms;
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    chunk_prep_kernel<<<(unsigned)grid, PT, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
