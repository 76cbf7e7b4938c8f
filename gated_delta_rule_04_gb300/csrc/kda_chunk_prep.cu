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
// every other term.  Under the unbounded gate (template flag SP) iY_r has no
// bound: the off-diagonal factors are then taken as one exponential each,
// e^{G_r - G_en(b)} <= 1, and the diagonal blocks of A and P by position pairs
// on the CUDA cores (see dg_index).
//
// Tensor cores.  A and the off-diagonal blocks of P are two bf16 M = 128 MMAs
// against the right operand R = k Y (N = 64, K = 128 keys).  The 256 left
// rows are the A rows grouped by column sub-tile b (64 + 48 + 32 + 16) and the
// off-diagonal P rows (48 + 32 + 16).  The diagonal blocks of P reach the
// output directly and need more than bf16: their operands are split into
// bf16 high and low parts: one N = 128 MMA multiplies [q hi; q lo] by
// [R hi | R lo] and the readout adds hi*hi + hi*lo + lo*hi, good to about 16
// bits.  W = T (k e^G) and U0^T = v^T T^T are fp16 MMAs; the unit
// lower-triangular solve is fp32 on the CUDA cores (16 x 16 diagonal
// inverses, then the off-diagonal blocks diagonal by diagonal).
//
// Two warp groups, two items in flight per SM.  The persistent CTA (one per
// SM) splits its 16 warps:
//   front (warps 0-7): conv, SiLU, gate and norms of item j, its operand tiles
//     (shared memory) and its Q+ / Kt / decay records, then the first tcgen05
//     batch (A, off-diagonal P, split diagonal P) of item j;
//   back (warps 8-15): for item j - 1, the readout of A and P from tensor
//     memory, the solve, T, the W / U0^T products, their readout and the
//     record stores of P, W and U0^T.  One thread of warp 11 issues the
//     tcgen05 batches, TMA boxes and bulk stores.
// So the element-wise work of one item overlaps the short, dependent solve of
// the one before.  The raw q/k/v rows of an item (with the three rows before
// the chunk) arrive by TMA into the operand region, issued by the back once
// the previous item's first batch has read that region; the gate inputs and
// beta logits are plain loads, and an L2 prefetch runs one item ahead.
//
// Front thread mapping: warp w, lane l -> sub-tile a = w / 2 (tokens 16a ..
// 16a+15) and channel pair p = 32 (w % 2) + l (channels 2p, 2p+1).  Each
// thread keeps its 32 elements per plane in registers from the conv to the
// operand tiles; token sums (L2 norms) are warp reduce-scatters plus one
// shared-memory exchange between the two warps of a sub-tile, and the
// cumulative gate is a per-thread running sum plus a prefix over sub-tiles.
//
// Hand-offs (all mbarriers, one phase per item, in item order):
//   mma1   the first batch of item j finished: the back may read A and P, and
//          the next item's raw rows may land in the operand region;
//   raw    one per plane: the raw q (k, v) rows of item j have landed: the
//          front may start on it (on the conv of k, of v);
//   info   item j's record address and beta are published to the back (a
//          null address ends the back's loop);
//   mma2   the W / U0^T products of item j finished: the front may overwrite
//          (k e^G)^T and v^T.
// Every wait is bounded; loop exits are agreed on with bar.red.or so that no
// named barrier waits for a warp that left.  After a timeout the kernel
// records it in the workspace status word, lets its own MMAs and bulk stores
// finish and frees its tensor memory.
//
// Output: one record per (chunk, head) in the exact shared-memory image the
// recurrence kernel consumes (fp16, K-major, 128-byte swizzle).  Q+ and the
// decay are stored from registers; Kt, P, W and U0^T are assembled in shared
// memory and leave as contiguous bulk stores.
#include "kda_chunk_layout.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int PT = 512;                    // 16 warps
constexpr int NF = 256;                    // front threads (warps 0-7)
constexpr int NB = 256;                    // back threads (warps 8-15)
constexpr int BAR_FRONT = 1, BAR_BACK = 2; // named barrier ids
// the back thread that issues the tcgen05 batches, TMA boxes and bulk stores (and
// waits for them): lane 0 of warp 11, on the SM sub-partition (warp index mod 4)
// that the rest of the back group loads least
constexpr int ISSUER = 96;
constexpr int REG_LAUNCH = 65536 / PT;     // registers per thread at launch (__launch_bounds__(PT, 1))
// register split (front, back): the latency-bound front gets the larger share;
// at 160 / 96 both variants' backs are spill-free (the unbounded gate's kernel
// spills 12 bytes in all, the fewest of the splits tried)
constexpr int REG_FRONT = 160;
constexpr int REG_BACK = 96;
static_assert(REG_LAUNCH == 128 && NF * REG_FRONT + NB * REG_BACK <= PT * REG_LAUNCH && REG_FRONT % 8 == 0 &&
                  REG_BACK % 8 == 0 && REG_BACK >= 24 && REG_FRONT <= 256,
              "the register split must fit the launch's registers, or setmaxnreg.inc waits forever");
constexpr int C = CHUNK_T;                 // 64 tokens
constexpr int XR = 16 + RING;              // raw rows a front thread reads per plane
constexpr int LDS = 68;                    // fp32 row stride of the 64 x 64 matrices (16-byte rows)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_D0 = 0, TM_D1 = 64, TM_D2 = 128, TM_W = 256, TM_U = 384;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int NSLOT = 3;                   // slots of the per-item hand-off (beta, record address)

// shared-memory map (bytes from a 1 KiB aligned base)
constexpr uint32_t RAW_ROW = D * 2;                // one bf16 row of a head
constexpr uint32_t RAW_PLANE = (C + RING) * RAW_ROW;
constexpr uint32_t S_RAW = 0;                      // bf16 [3 planes][67 rows][128]: raw q, k, v of the next item
                                                   //   (row 0 = token t0 - 3), in the operand tiles: it lands
                                                   //   after the previous item's first batch has read them, and
                                                   //   is read before this item's tiles are written
constexpr uint32_t S_LAP = 0;                      // bf16 2 x [128 rows][128 keys]: A / off-diagonal P left rows
constexpr uint32_t S_QD = S_LAP + 65536;           // bf16 [128][128]: rows 0-63 q hi, 64-127 q lo
constexpr uint32_t S_DG = S_QD;                    //   softplus gate (no split P): fp32 [2 slots][4 sub-tiles]
                                                   //   [2 halves][128] position-pair sums of the diagonal
                                                   //   blocks below level 3, then the level-3 operand tiles:
constexpr uint32_t S_L3A = S_QD + 8192;            //   fp16 2 panels x [64 rows][64 ch]: k^, q^ of rows 8-15
constexpr uint32_t S_L3B = S_QD + 24576;           //   fp16 2 panels x [32 rows][64 ch]: k^ of columns 0-7
constexpr uint32_t S_L3T = 0;                      //   (offset in the X tile) fp32 [A, P][4][8][8] level-3 sums
constexpr uint32_t S_RHL = S_QD + 32768;           // bf16 [128][128 keys] R: rows 0-63 hi, 64-127 lo
constexpr uint32_t S_TT = S_RHL + 32768;           // fp16 [64 r][64 s] T; the W product reads it as 128 A
                                                   //   rows, rows 64-127 being the first 8 KiB of (k e^G)^T
                                                   //   (their output lanes are unused).  Before T: P staged
                                                   //   for its bulk store.
constexpr uint32_t S_KPT = S_TT + 8192;            // fp16 [128 key][64 s] (k e^G)^T
constexpr uint32_t S_VT = S_KPT + 16384;           // fp16 [128 val][64 s] v^T
constexpr uint32_t S_TAPS = S_VT + 16384;          // float2 [3 planes][64 pairs][4 taps]: the head's conv taps
                                                   //   times 1/2, channel pairs interleaved
constexpr uint32_t S_AM = S_TAPS + 6144;           // fp32 [64][68] beta A (back)
constexpr uint32_t S_XM = S_AM + 64 * LDS * 4;     // fp32 [64][68] X = (I + A)^{-1} (back)
constexpr uint32_t S_WUST = S_AM;                  //   after T: W (2 x 8 KiB) and U0^T (16 KiB) staged
constexpr uint32_t S_PDL = S_XM;                   //   during the readout: lo*hi terms of diagonal P
constexpr uint32_t S_NRM = S_XM + 64 * LDS * 4;    // float2 [8 warps][16]: partial sums of squares (q, k)
constexpr uint32_t S_TOT = S_NRM + 1024;           // float2 [4 sub-tiles][64 pairs]: gate sums
constexpr uint32_t S_BT = S_TOT + 2048;            // fp32 [NSLOT][64] beta
constexpr uint32_t S_INFO = S_BT + NSLOT * 256;    // [NSLOT] Handoff: record address, the next item
constexpr uint32_t S_BAR = S_INFO + NSLOT * 32;    // mbarriers, TMEM slot, flags
constexpr uint32_t S_DGX = S_BAR + 128;             // u8 [A, P][16 r][16 s]: unbounded gate's pair codes
constexpr uint32_t SMEM_BYTES = S_DGX + 512 + 1024;
static_assert(S_RAW + 3 * RAW_PLANE <= S_QD, "raw rows inside the left-row tiles");
static_assert(S_KPT == S_TT + 8192, "the W product's junk A rows are the first 8 KiB of (k e^G)^T");
static_assert(S_WUST + 32768 <= S_NRM, "W / U0^T staging inside the solve tiles");
static_assert(S_XM + 64 * 16 * 4 <= S_NRM, "lo*hi exchange inside X");
static_assert(2 * 4 * 2 * 128 * 4 <= S_L3A - S_DG && S_L3B + 2 * 4096 == S_QD + 32768,
              "pair sums and level-3 tiles inside the diagonal-P operand tile");
static_assert(S_L3A % 1024 == 0 && S_L3B % 1024 == 0, "level-3 tiles on 1 KiB boundaries");
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(S_LAP % 1024 == 0 && S_QD % 1024 == 0 && S_RHL % 1024 == 0 && S_TT % 1024 == 0 &&
                  S_KPT % 1024 == 0 && S_VT % 1024 == 0,
              "MMA operand tiles start on 1 KiB boundaries");

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
__device__ __forceinline__ float lg2f(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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
__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 h2f(uint32_t u) { return __half22float2(*reinterpret_cast<const __half2*>(&u)); }
__device__ __forceinline__ void bar_sync_n(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void sts32(unsigned char* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 32 lanes x 16 consecutive 32-bit TMEM columns into registers, without
// waiting: several loads in flight, then tmem_wait_ld.
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 8 consecutive 32-bit TMEM columns, without waiting.
__device__ __forceinline__ void tmem_ld8_nw(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// Waits for phase `parity` of an mbarrier for at most `limit_ns`, giving up
// early once the CTA's abort flag is set.  Returns false when it gave up; a
// timeout also sets the flag.  The waiting thread sleeps in the barrier test
// (a few microseconds at a time) rather than spinning: the other group's
// warps share its SM sub-partition.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
    constexpr uint32_t SLEEP_NS = 4000;
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    const uint32_t hint = limit_ns < SLEEP_NS ? (uint32_t)limit_ns : SLEEP_NS;
    while (!ptx::mbar_try_wait_sleep(bar, parity, hint)) {
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// Blockwise inverse X = (I + A)^{-1} over 16 x 16 blocks, once the diagonal
// blocks X_aa are known:  X_ab = -X_aa sum_{k=b}^{a-1} A_ak X_kb.  First
// At_ak = X_aa A_ak for every a > k (one pass, kept in A's unused upper block
// (k, a)); then one pass per block diagonal, X_ab = -sum_k At_ak X_kb.
// Task = (block pair, row, 4 consecutive columns): one broadcast load of the
// left factor and one 16-byte load of the right row per 4 FMAs.  The back
// group's 256 threads (index bt) run them; each pass ends with its barrier.
__device__ __forceinline__ void solve_premultiply(float* Am, const float* Xm, int bt) {
#pragma unroll 1
    for (int task = bt; task < 6 * 64; task += NB) {
        const int p = task >> 6, r = (task >> 2) & 15, c = 4 * (task & 3);
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
    bar_sync_n(BAR_BACK, NB);
}

template <int Dg>
__device__ __forceinline__ void solve_level(const float* Am, float* Xm, int bt) {
    constexpr int ntask = (4 - Dg) * 64;
    static_assert(ntask <= NB, "one task per thread");
    const int b = bt >> 6, r = (bt >> 2) & 15, c = 4 * (bt & 3), a = b + Dg;
    if (bt < ntask) {
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
    bar_sync_n(BAR_BACK, NB);
}

// ---- diagonal blocks under the unbounded (softplus) gate ----------------------
// Without a lower bound on g, the factors e^{G_r - G_en(a)} of a diagonal
// sub-tile overflow, so its pairs (r, s) are summed position by position on
// the CUDA cores ("Kimi K3 - Retention gate", section "Why": the old gate
// needed an explicit position-pair computation on the diagonal tiles).  Each
// pair takes its factor from a recursive halving of the 16-token sub-tile:
// at level t (halves of h = 2^t tokens) the pairs with r in the upper and s in
// the lower half of a 2h-block use the last token m of the lower half,
// e^{G_r - G_s} = e^{G_r - G_m} e^{G_m - G_s}, both factors <= 1.  Level 3
// (rows 8-15 against columns 0-7 through token 7, 64 of the 120 A pairs and 64
// of the 136 P pairs) is one rank-128 product per sub-tile, so it runs on the
// tensor cores in fp16 (every factor <= 1); the other pair values are
// numbered level by level (t = 2, 1, 0), block by block, row by row, A before
// P within a row, and the 16 values P[r][r] come last (indices 112 + r).
__device__ __forceinline__ bool dg_level3(int jr, int js) { return jr >= 8 && js < 8; }
__device__ __forceinline__ int dg_index(int jr, int js, int isP) {
    if (jr == js) return 112 + jr;
    const int t = 31 - __clz(jr ^ js), h = 1 << t, b0 = (jr >> (t + 1)) << (t + 1);
    const int lvl = t == 2 ? 0 : t == 1 ? 64 : 96;
    return lvl + (b0 >> (t + 1)) * 2 * h * h + (jr - b0 - h) * 2 * h + isP * h + (js - b0);
}
// The back group reads the pair values through a table of one code per (A or P,
// r, s), built once per CTA: the index above, DG_L3 for a level-3 pair, DG_ZERO
// above the diagonal (and on it for A).
constexpr uint32_t DG_L3 = 0xFE, DG_ZERO = 0xFF;
__device__ __forceinline__ uint32_t dg_code(int isP, int jr, int js) {
    if (isP ? js > jr : js >= jr) return DG_ZERO;
    return dg_level3(jr, js) ? DG_L3 : (uint32_t)dg_index(jr, js, isP);
}

// Sum of v[i] over the warp's 32 lanes, lanes 2i and 2i + 1 keeping the sum
// of v[i] (recursive halving: 16 shuffles for 16 values).
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
    for (int o = 16; o >= 2; o >>= 1) {
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < o / 2; ++i) {
            const float send = up ? v[i] : v[i + o / 2], keep = up ? v[i + o / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Read-only 4-byte load that does not allocate in L1: the rows are read once,
// and the L1 left beside the shared-memory tiles is too small to stage them.
__device__ __forceinline__ uint32_t ldg_na(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Address of raw row i (0 .. XR-1, chunk-relative token 16a + i - 3) of one
// plane for this thread's channel pair, or null where the row reads as zero:
// past the chunk's last token, or before a sequence start without a ring.
__device__ __forceinline__ const uint32_t* raw_row(const PrepArgs& A, const void* plane, int pl,
                                                   const ChunkDesc& cd, int h, int a, int i, int c0) {
    const int W = A.H * D;
    const int r = 16 * a + i - RING;
    if (r >= cd.len) return nullptr;
    if (r >= 0 || cd.pos > 0)
        return reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(plane) +
                                                 (size_t)(cd.t0 + r) * W + (size_t)h * D + c0);
    if (A.ring_in == nullptr) return nullptr;
    // ring slot RING + r (slot 0 oldest) of sequence cd.seq, plane pl
    return reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(A.ring_in) +
                                             (((size_t)cd.seq * 3 + pl) * RING + (RING + r)) * W + (size_t)h * D + c0);
}

// Hand-off of one item from the front to the back group: its record, and the
// item after it (whose raw rows the back loads once this item's first batch
// has finished).
struct Handoff {
    unsigned char* rec;   // null: no more items
    int32_t has_next, t0, len, pos, h;
    int32_t pad;
};
static_assert(sizeof(Handoff) == 32, "hand-off slot");

// The raw q, k, v rows of one item into the raw-row tile, by one thread, counted
// on `bar`: the chunk and the three rows before it, or at a sequence start the
// chunk alone (rows 3-66; the rows before it come from the conv ring or are zero).
// Rows past the end of the tensor read as zero; rows past the chunk are not used.
__device__ __forceinline__ void issue_raw(const PrepArgs& a, int32_t t0, int32_t pos, int h, uint32_t base,
                                          const uint32_t (&bar)[3]) {
#pragma unroll
    for (int pl = 0; pl < 3; ++pl) {   // one mbarrier per plane: the conv of q starts while k and v land
        ptx::mbar_expect_tx(bar[pl], pos > 0 ? RAW_PLANE : C * RAW_ROW);
        if (pos > 0) ptx::tma_load_2d(base + S_RAW + pl * RAW_PLANE, &a.map67[pl], h * D, t0 - RING, bar[pl]);
        else ptx::tma_load_2d(base + S_RAW + pl * RAW_PLANE + RING * RAW_ROW, &a.map64[pl], h * D, t0, bar[pl]);
    }
}

// L2 prefetch of one item's raw q/k/v rows (with the three rows before the
// chunk), gate inputs and beta logits, one item ahead of their loads: 530
// 128-byte lines (3 planes x 67 rows x 2 halves of the head's row, z 64 x 2),
// two or three per front thread, and the beta logits of threads ft < len.
// Plain prefetches: they neither block the thread nor hold a register.
__device__ __forceinline__ void prefetch_item(const PrepArgs& a, const ChunkDesc& cn, int hn, int ft) {
    const int W = a.H * D;
    constexpr int PLANE_LINES = (C + RING) * 2, LINES = 3 * PLANE_LINES + 2 * C;
    const int first = cn.pos > 0 ? -RING : 0;                 // rows before the chunk inside the sequence
#pragma unroll
    for (int li = ft; li < LINES; li += NF) {
        const int pl = li < 3 * PLANE_LINES ? li / PLANE_LINES : 3;
        const int rest = pl < 3 ? li - pl * PLANE_LINES : li - 3 * PLANE_LINES;
        const int row = (pl < 3 ? -RING : 0) + (rest >> 1), half = rest & 1;
        if (row < first || row >= cn.len) continue;
        const void* base = pl == 0 ? a.q : pl == 1 ? a.k : pl == 2 ? a.v : a.z;
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + (size_t)(cn.t0 + row) * W +
                                 (size_t)hn * D + 64 * half;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
    if (ft < cn.len) {
        const unsigned short* bp = static_cast<const unsigned short*>(a.b) + (size_t)(cn.t0 + ft) * a.H + hn;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(bp));
    }
}

// SP: the unbounded gate g = -e^A softplus(z + dt_bias) (diagonal blocks by
// position pairs); otherwise the lower-bounded gate.
template <bool SP>
__global__ void __launch_bounds__(PT, 1) chunk_prep_kernel(const __grid_constant__ PrepArgs a) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sb = smem_raw + (base - raw);
    float* Am = reinterpret_cast<float*>(sb + S_AM);
    float* Xm = reinterpret_cast<float*>(sb + S_XM);
    float* btab = reinterpret_cast<float*>(sb + S_BT);
    volatile Handoff* info = reinterpret_cast<volatile Handoff*>(sb + S_INFO);
    const uint32_t bar_mma1 = base + S_BAR, bar_mma2 = base + S_BAR + 8, bar_info = base + S_BAR + 16,
                   bar_drain = base + S_BAR + 24;
    // the raw q, k, v rows of an item, one mbarrier per plane
    const uint32_t bar_raw[3] = {base + S_BAR + 32, base + S_BAR + 72, base + S_BAR + 80};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sb + S_BAR + 48);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sb + S_BAR + 52);
    volatile int* s_take = reinterpret_cast<volatile int*>(sb + S_BAR + 56);
    // raw-row loads issued (for the drain after a timeout)
    volatile int* raw_issued = reinterpret_cast<volatile int*>(sb + S_BAR + 64);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t lim = a.wait_limit_ns ? a.wait_limit_ns : WAIT_LIMIT_NS;

    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid == 0) {
        ptx::mbar_init(bar_mma1, 1);
        ptx::mbar_init(bar_mma2, 1);
        ptx::mbar_init(bar_info, 1);
        ptx::mbar_init(bar_drain, 1);
        for (int pl = 0; pl < 3; ++pl) ptx::mbar_init(bar_raw[pl], 1);
        *raw_issued = 0;
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (SP) sb[S_DGX + tid] = (unsigned char)dg_code(tid >> 8, (tid >> 4) & 15, tid & 15);   // (PT = 512)
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < NF / 32) {
        // ================================ front ================================
        // registers move from the back group to this one: 256 x REG_FRONT +
        // 256 x REG_BACK is exactly the 512 x 128 the CTA was launched with
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_FRONT));
        const int ft = tid;
        const int H = a.H, W = H * D, NC = a.n_chunks;
        const int n_items = NC * H;
        const int a_sub = warp >> 1, hf = warp & 1;
        const int c0 = 2 * (32 * hf + lane);           // first of this thread's two channels
        const int tok0 = 16 * a_sub;
        float2* nrm = reinterpret_cast<float2*>(sb + S_NRM);
        float2* tot = reinterpret_cast<float2*>(sb + S_TOT);

        // This CTA's items, in head-major order (item j is chunk j % NC of head
        // j / NC, so consecutive items share their head's constants): either one
        // contiguous range, or batches of a.batch taken from the work counter one
        // batch ahead (the next item must be known an item ahead for its prefetch).
        // [jt, j_stop) is the current batch and nb_start the first item of the next.
        int jt, j_stop, nb_start;
        if (a.work_counter != nullptr) {
            if (ft == 0) {
                s_take[0] = atomicAdd(a.work_counter, 1);
                s_take[1] = atomicAdd(a.work_counter, 1);
            }
            bar_sync_n(BAR_FRONT, NF);
            jt = min(s_take[0] * a.batch, n_items);
            j_stop = min(jt + a.batch, n_items);
            nb_start = min(s_take[1] * a.batch, n_items);
        } else {
            jt = (int)(((int64_t)blockIdx.x * n_items) / gridDim.x);
            j_stop = (int)(((int64_t)(blockIdx.x + 1) * n_items) / gridDim.x);
            nb_start = n_items;
        }
        ChunkDesc cd = jt < j_stop ? a.chunks[jt % NC] : ChunkDesc{0, 0, 0, 0};
        if (jt < j_stop) prefetch_item(a, cd, jt / NC, ft);
        // gate inputs and the beta logit of an item (the raw q, k, v rows arrive in
        // shared memory)
        uint32_t zr[16];
        unsigned short b_raw = 0;   // bf16 bits
        auto issue_loads = [&](const ChunkDesc& cl, int hl) {
            const uint32_t* zp = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.z) +
                                                                   (size_t)(cl.t0 + tok0) * W + (size_t)hl * D + c0);
#pragma unroll
            for (int j = 0; j < 16; ++j) zr[j] = tok0 + j < cl.len ? ldg_na(zp + (size_t)j * (W / 2)) : 0u;
            b_raw = ft < cl.len ? static_cast<const unsigned short*>(a.b)[(size_t)(cl.t0 + ft) * H + hl]
                                : (unsigned short)0;
        };
        // the first item's raw rows; the back group loads each later item's once
        // the first batch of the item before has read the operand tiles
        if (ft == 0 && jt < j_stop) {
            issue_raw(a, cd.t0, cd.pos, jt / NC, base, bar_raw);
            *raw_issued = 1;
        }
        // The head's constants, reloaded only when the head changes (items are
        // head-major): conv taps times 1/2 (the conv then yields x/2, the argument of
        // tanh in the SiLU) in shared memory, and the gate's scale and offset in
        // registers.  With the operand tiles in shared memory the L1 cache is small,
        // so loading them from global memory per item would wait on L2 every time.
        int cur_h = -1;
        float2 gsc = make_float2(0.f, 0.f), gof = make_float2(0.f, 0.f);
        float4* taps = reinterpret_cast<float4*>(sb + S_TAPS);   // [3][64 pairs][2] float4
        uint32_t k_iter = 0;
        // (the top-of-item barrier also orders the reads of s_take above before
        // the next atomicAdd rewrites it)
#pragma unroll 1
        while (jt < j_stop) {
            if (ptx::bar_sync_or(BAR_FRONT, NF, *abort_flag != 0)) break;
            const int h = jt / NC, len = cd.len;
            const bool last_of_batch = jt + 1 == j_stop;
            const int next = last_of_batch ? nb_start : jt + 1;
            const bool has_next = next < n_items;
            const ChunkDesc cn = a.chunks[(has_next ? next : jt) % NC];
            const int hn = next / NC;
            unsigned char* rec = static_cast<unsigned char*>(a.records) + ((size_t)(jt % NC) * H + h) * REC_BYTES;
            const int slot = (int)(k_iter % NSLOT);
            if (has_next) prefetch_item(a, cn, hn, ft);
            // the batch after the next one (read after this item's last barrier)
            if (ft == 0 && last_of_batch && a.work_counter != nullptr) s_take[0] = atomicAdd(a.work_counter, 1);

            // this item's gate inputs and beta logit (in flight while its raw rows land)
            issue_loads(cd, h);
            if (h != cur_h) {   // (CTA-uniform)
                cur_h = h;
                // thread ft < 192 writes plane ft / 64, pair ft % 64: taps 0-3 of both channels
                if (ft < 3 * 64) {
                    const int pl = ft >> 6, pr = ft & 63;
                    const float4 w0 = __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)pl * W + h * D + 2 * pr) * CONV_K));
                    const float4 w1 =
                        __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)pl * W + h * D + 2 * pr + 1) * CONV_K));
                    taps[2 * ft] = make_float4(0.5f * w0.x, 0.5f * w1.x, 0.5f * w0.y, 0.5f * w1.y);
                    taps[2 * ft + 1] = make_float4(0.5f * w0.z, 0.5f * w1.z, 0.5f * w0.w, 0.5f * w1.w);
                }
                bar_sync_n(BAR_FRONT, NF);
                const float eA = __expf(__ldg(a.A_log + h));
                const float2 dtb = __ldg(reinterpret_cast<const float2*>(a.dt_bias + h * D + c0));
                if (SP) {
                    gsc = f2(-eA);             // g = -e^A softplus(z + dt_bias)
                    gof = dtb;
                } else {
                    gsc = f2(-eA * LOG2E);     // argument of 2^x: -(z + dt_bias) e^A log2 e
                    gof = __fmul2_rn(dtb, gsc);
                }
            }
            const bool full = tok0 + 16 <= len;

            // this item's raw q rows (one thread polls, the others wait in the barrier;
            // the k and v rows are waited for before their conv)
            {
                bool late = false;
                if (ft == 0) late = !wait_or_abort(bar_raw[0], k_iter & 1u, lim, abort_flag);
                if (ptx::bar_sync_or(BAR_FRONT, NF, late)) break;
            }

            // ---- gate g = lb sigmoid(e^A (z + dt_bias)) (or -e^A softplus(z + dt_bias))
            // and its running sum over the thread's 16 tokens (tokens past the chunk's
            // end add nothing)
            float2 gc[16];
            {
                const float2 lb2 = f2(a.lb);
                float2 run = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float2 g;
                    if (SP) {
                        // softplus(x) = max(x, 0) + ln 2 log2(1 + 2^{-|x| log2 e})
                        const float2 x = __fadd2_rn(bf2f(zr[j]), gof);
                        const float2 l = make_float2(lg2f(1.f + ex2f(-fabsf(x.x) * LOG2E)),
                                                     lg2f(1.f + ex2f(-fabsf(x.y) * LOG2E)));
                        const float2 sp = __ffma2_rn(l, f2(0.6931471805599453f),
                                                     make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
                        g = __fmul2_rn(gsc, sp);
                    } else {
                        const float2 sarg = __ffma2_rn(bf2f(zr[j]), gsc, gof);
                        g = __fmul2_rn(lb2, make_float2(rcpf(1.f + ex2f(sarg.x)), rcpf(1.f + ex2f(sarg.y))));
                    }
                    if (full || tok0 + j < len) run = __fadd2_rn(run, g);
                    gc[j] = run;
                }
            }


            // ---- conv (kernel 4) + SiLU of one plane, kept as fp16 pairs; the sums of
            // squares of its 16 tokens are reduce-scattered over the warp, so that
            // lanes 2t and 2t + 1 return token t's sum over this warp's 64 channels
            auto conv_plane = [&](const uint32_t (&x)[XR], int pl, uint32_t (&outp)[16], bool want_sq) -> float {
                const float4 t01 = taps[2 * (64 * pl + 32 * hf + lane)], t23 = taps[2 * (64 * pl + 32 * hf + lane) + 1];
                const float2 wt0 = make_float2(t01.x, t01.y), wt1 = make_float2(t01.z, t01.w);
                const float2 wt2 = make_float2(t23.x, t23.y), wt3 = make_float2(t23.z, t23.w);
                float sq[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    // h = x / 2;  x sigmoid(x) = h + h tanh(h), tanh in half precision: the
                    // result is rounded to fp16 next, and the error (about 2^-11 of x) is at that level
                    float2 hx = __fmul2_rn(wt0, bf2f(x[j]));
                    hx = __ffma2_rn(wt1, bf2f(x[j + 1]), hx);
                    hx = __ffma2_rn(wt2, bf2f(x[j + 2]), hx);
                    hx = __ffma2_rn(wt3, bf2f(x[j + 3]), hx);
                    const __half2 hin = __float22half2_rn(hx);
                    uint32_t t;
                    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(*reinterpret_cast<const uint32_t*>(&hin)));
                    const float2 y = __ffma2_rn(hx, h2f(t), hx);
                    const bool valid = full || tok0 + j < len;
                    outp[j] = valid ? pack_f16(y.x, y.y) : 0u;
                    sq[j] = valid ? fmaf(y.x, y.x, y.y * y.y) : 0.f;
                }
                if (!want_sq) return 0.f;
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
                return sq[0] + __shfl_xor_sync(0xffffffffu, sq[0], 1);
            };
            // raw rows 16a - 3 .. 16a + 15 of a plane (the 67-row tile's rows 16a .. 16a + 18);
            // at a sequence start the three rows before the chunk come from the ring or are zero
            const bool ring_rows = cd.pos == 0 && a_sub == 0;
            auto raw_rows = [&](int pl, uint32_t (&x)[XR]) {
                const unsigned char* src = sb + S_RAW + pl * RAW_PLANE + tok0 * RAW_ROW + 4 * (32 * hf + lane);
#pragma unroll
                for (int i = 0; i < XR; ++i) x[i] = *reinterpret_cast<const uint32_t*>(src + i * RAW_ROW);
                if (ring_rows) {
#pragma unroll
                    for (int i = 0; i < RING; ++i) {
                        const uint32_t* p = raw_row(a, pl == 0 ? a.q : pl == 1 ? a.k : a.v, pl, cd, h, 0, i, c0);
                        x[i] = p ? ldg_na(p) : 0u;
                    }
                }
            };
            uint32_t aq[16], ak[16], av[16];
            float sqq, sqk;
            {
                uint32_t x[XR];
                raw_rows(0, x);
                sqq = conv_plane(x, 0, aq, true);
                // (every thread observes the plane's barrier itself; after a timeout it
                // reads stale rows, and the next agreement on the abort flag ends the loop)
                wait_or_abort(bar_raw[1], k_iter & 1u, lim, abort_flag);
                raw_rows(1, x);
                sqk = conv_plane(x, 1, ak, true);
                wait_or_abort(bar_raw[2], k_iter & 1u, lim, abort_flag);
                raw_rows(2, x);
                conv_plane(x, 2, av, false);
            }
            const float beta = ft < len ? rcpf(1.f + ex2f(-__uint_as_float((uint32_t)b_raw << 16) * LOG2E)) : 0.f;

            // ---- hand the token sums, sub-tile gate totals and beta to the other warps
            if ((lane & 1) == 0) nrm[warp * 16 + (lane >> 1)] = make_float2(sqq, sqk);
            tot[a_sub * 64 + 32 * hf + lane] = gc[15];
            if (ft < C) btab[slot * C + ft] = beta;
            // (this barrier also ends every read of the raw-row tile, which the operand
            // tiles below overwrite; the first batch of the previous item had finished
            // before those rows were loaded)
            bar_sync_n(BAR_FRONT, NF);

            // ---- norms of this lane's token (lane >> 1), both channel halves
            float nvq, nvk;
            {
                const float2 mine = nrm[warp * 16 + (lane >> 1)], other = nrm[(warp ^ 1) * 16 + (lane >> 1)];
                nvq = rsqrtf(mine.x + other.x + a.l2_eps) * a.q_scale;
                nvk = rsqrtf(mine.y + other.y + a.l2_eps);
            }
            if (SP) {
                // ---- the diagonal blocks of A and P by position pairs (see dg_index).
                // Level 3: this thread's two channels of k^ and q^ (norm factor and
                // e^{G_r - G_7}) for rows 8-15 and of k^ (norm factor and e^{G_7 - G_s})
                // for columns 0-7 into the level-3 operand tiles, for the back's first
                // tcgen05 batch.  Levels 2-0: this thread's share of every pair sum of its
                // sub-tile, on the conv outputs (the norm factors of both tokens are
                // applied after the sum over the warp's 64 channels); the back adds the
                // two warps.
                float* dg = reinterpret_cast<float*>(sb + S_DG) + (((k_iter & 1u) * 4 + a_sub) * 2 + hf) * 128;
                auto ex2d = [&](float2 hi, float2 lo) {   // e^{hi - lo} per channel (hi <= lo)
                    return make_float2(ex2f((hi.x - lo.x) * LOG2E), ex2f((hi.y - lo.y) * LOG2E));
                };
                auto dot2 = [](float2 x, float2 y) { return fmaf(x.x, y.x, x.y * y.y); };
                // one batch of 16 pair values: lanes 2q and 2q + 1 hold value 16 kb + q,
                // whose row jr, column js and matrix (A or P) they name
                const int q = lane >> 1;
                auto finish = [&](float (&v)[16], int kb, int jr, int js, int isP) {
                    const float sum = reduce_scatter16(v, lane);
                    const float nq_r = __shfl_sync(0xffffffffu, nvq, 2 * jr);
                    const float nk_r = __shfl_sync(0xffffffffu, nvk, 2 * jr);
                    const float nk_s = __shfl_sync(0xffffffffu, nvk, 2 * js);
                    if ((lane & 1) == 0) dg[16 * kb + q] = sum * (isP ? nq_r : nk_r) * nk_s;
                };
                // level 3 operand tiles: fp16, K-major with the 128-byte swizzle; channel
                // pair c0 sits at chunk lane / 4, bytes 4 (lane & 3) of a 128-byte row of
                // panel hf; rows 8 a_sub + i are one 8-row swizzle group
                {
                    const uint32_t cpart = ((uint32_t)(lane >> 2)) << 4, cbyte = 4u * (lane & 3);
                    unsigned char* const tA = sb + S_L3A + (uint32_t)hf * 8192u + (uint32_t)(8 * a_sub) * 128u + cbyte;
                    unsigned char* const tB = sb + S_L3B + (uint32_t)hf * 4096u + (uint32_t)(8 * a_sub) * 128u + cbyte;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t ro = 128u * i + (cpart ^ ((uint32_t)i << 4));
                        // column s = i: k^_s e^{G_7 - G_s}
                        const float nks = __shfl_sync(0xffffffffu, nvk, 2 * i);
                        float2 ks = __fmul2_rn(h2f(ak[i]), f2(nks));
                        if (i < 7) ks = __fmul2_rn(ks, ex2d(gc[7], gc[i]));
                        sts32(tB + ro, pack_f16(ks.x, ks.y));
                        // row r = 8 + i: k^_r and q^_r times e^{G_r - G_7}
                        const float nkr = __shfl_sync(0xffffffffu, nvk, 2 * (8 + i));
                        const float nqr = __shfl_sync(0xffffffffu, nvq, 2 * (8 + i));
                        const float2 rho = ex2d(gc[8 + i], gc[7]);
                        const float2 kr = __fmul2_rn(__fmul2_rn(h2f(ak[8 + i]), f2(nkr)), rho);
                        const float2 qr = __fmul2_rn(__fmul2_rn(h2f(aq[8 + i]), f2(nqr)), rho);
                        sts32(tA + ro, pack_f16(kr.x, kr.y));
                        sts32(tA + 32u * 128u + ro, pack_f16(qr.x, qr.y));
                    }
                }
                // level 2: in each half, rows 4-7 against columns 0-3, through token 3
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int m = 8 * bb + 3;
                    float2 ks[4];
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        ks[s] = s == 3 ? h2f(ak[m]) : __fmul2_rn(h2f(ak[8 * bb + s]), ex2d(gc[m], gc[8 * bb + s]));
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float v[16];
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int r = 8 * bb + 4 + 2 * half + rr;
                            const float2 rho = ex2d(gc[r], gc[m]);
                            const float2 kr = __fmul2_rn(h2f(ak[r]), rho), qr = __fmul2_rn(h2f(aq[r]), rho);
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                v[8 * rr + s] = dot2(kr, ks[s]);
                                v[8 * rr + 4 + s] = dot2(qr, ks[s]);
                            }
                        }
                        finish(v, 2 * bb + half, 8 * bb + 4 + 2 * half + (q >> 3), 8 * bb + (q & 3), (q >> 2) & 1);
                    }
                }
                // level 1: in each quarter, rows 2-3 against columns 0-1, through token 1
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    float v[16];
#pragma unroll
                    for (int bq = 0; bq < 2; ++bq) {
                        const int bb = 2 * hb + bq, m = 4 * bb + 1;
                        const float2 ks0 = __fmul2_rn(h2f(ak[4 * bb]), ex2d(gc[m], gc[4 * bb])), ks1 = h2f(ak[m]);
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int r = 4 * bb + 2 + rr;
                            const float2 rho = ex2d(gc[r], gc[m]);
                            const float2 kr = __fmul2_rn(h2f(ak[r]), rho), qr = __fmul2_rn(h2f(aq[r]), rho);
                            v[8 * bq + 4 * rr + 0] = dot2(kr, ks0);
                            v[8 * bq + 4 * rr + 1] = dot2(kr, ks1);
                            v[8 * bq + 4 * rr + 2] = dot2(qr, ks0);
                            v[8 * bq + 4 * rr + 3] = dot2(qr, ks1);
                        }
                    }
                    const int bb = 2 * hb + (q >> 3), w = q & 7;
                    finish(v, 4 + hb, 4 * bb + 2 + (w >> 2), 4 * bb + (w & 1), (w >> 1) & 1);
                }
                // level 0: each odd row against the token before it
                {
                    float v[16];
#pragma unroll
                    for (int bb = 0; bb < 8; ++bb) {
                        const int r = 2 * bb + 1, s = 2 * bb;
                        const float2 ks = __fmul2_rn(h2f(ak[s]), ex2d(gc[r], gc[s]));
                        v[2 * bb] = dot2(h2f(ak[r]), ks);
                        v[2 * bb + 1] = dot2(h2f(aq[r]), ks);
                    }
                    finish(v, 6, 2 * (q >> 1) + 1, 2 * (q >> 1), q & 1);
                }
                // P[r][r]
                {
                    float v[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) v[r] = dot2(h2f(aq[r]), h2f(ak[r]));
                    finish(v, 7, q, q, 1);
                }
            }
            // ---- per-channel factors from the sub-tile ends G_en(b):
            // E = e^{G_en(a)}, F = e^{G_last - G_en(a)}, Cb = e^{G_en(a) - G_en(b)}
            float2 gen[4];
            {
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    acc = __fadd2_rn(acc, tot[b * 64 + 32 * hf + lane]);
                    gen[b] = acc;
                }
            }
            const float2 ge = a_sub == 0 ? gen[0] : a_sub == 1 ? gen[1] : a_sub == 2 ? gen[2] : gen[3];
            const float2 F = make_float2(ex2f((gen[3].x - ge.x) * LOG2E), ex2f((gen[3].y - ge.y) * LOG2E));
            // bounded gate: E and Cb as factors (iY E and iY Cb stay in range);
            // unbounded: their exponents, added to the token's before one 2^x each
            float2 E, Cb[3];
            if (SP) {
                E = make_float2(ge.x * LOG2E, ge.y * LOG2E);
#pragma unroll
                for (int b = 0; b < 3; ++b) Cb[b] = make_float2((ge.x - gen[b].x) * LOG2E, (ge.y - gen[b].y) * LOG2E);
            } else {
                E = make_float2(ex2f(ge.x * LOG2E), ex2f(ge.y * LOG2E));
#pragma unroll
                for (int b = 0; b < 3; ++b)
                    Cb[b] = make_float2(ex2f((ge.x - gen[b].x) * LOG2E), ex2f((ge.y - gen[b].y) * LOG2E));
            }
            if (a_sub == 0)
                *reinterpret_cast<float2*>(rec + REC_DECAY + 4 * c0) =
                    make_float2(ex2f(gen[3].x * LOG2E), ex2f(gen[3].y * LOG2E));
            const float2 gl = gc[15];


            // ---- operand tiles.  Per token: R (hi, lo), the A / P left rows, the
            // diagonal P rows (hi, lo), Q+ to the record; Kt and (k e^G) are kept as
            // fp16 pairs transposed into per-channel rows (word w of channel e holds
            // tokens 2w, 2w+1) for the tiles written after the loop.
            // Store addresses: every row-major tile here is K-major with the 128-byte
            // swizzle and every row index is (multiple of 16) + j, so element (row, c0)
            // sits at  tile + row-block offset + 128 j + ((lane/4 ^ (j & 7)) << 4) + 4 (lane & 3).
            uint32_t kt[2][8], kp[2][8];
            uint32_t kt_prev = 0, kp_prev = 0;
            const uint32_t colpart = (uint32_t)hf * 16384u + 4u * (lane & 3);     // 128-row tiles
            const uint32_t colrec = (uint32_t)hf * REC_PANEL + 4u * (lane & 3);   // Q+ record panels
            const uint32_t chunk = (uint32_t)lane >> 2;
            auto lap_off = [&](int row0) {   // row0: LAP row of token tok0 (a multiple of 16)
                return (uint32_t)(row0 >> 7) * 32768u + (uint32_t)(row0 & 127) * 128u + colpart;
            };
            constexpr int kRowA[4] = {0, 48, 80, 96};     // LAP row - r of the A rows of column sub-tile b
            constexpr int kRowP[3] = {144, 176, 192};     // LAP row - r of the off-diagonal P rows of b
            const uint32_t offA_diag = lap_off((a_sub == 0 ? 0 : a_sub == 1 ? 48 : a_sub == 2 ? 80 : 96) + tok0);
            unsigned char* const sRHL = sb + S_RHL + (uint32_t)tok0 * 128u + colpart;
            unsigned char* const sQD = sb + S_QD + (uint32_t)tok0 * 128u + colpart;
            unsigned char* const sLAP = sb + S_LAP;
            unsigned char* const gQ = rec + REC_Q + (uint32_t)tok0 * 128u + colrec;
            const float2 L2 = f2(LOG2E);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t jo = 128u * j + ((chunk ^ (uint32_t)(j & 7)) << 4);   // row j, swizzled
                const float nq = __shfl_sync(0xffffffffu, nvq, 2 * j);
                const float nk = __shfl_sync(0xffffffffu, nvk, 2 * j);
                const float2 q = __fmul2_rn(h2f(aq[j]), f2(nq));
                const float2 k = __fmul2_rn(h2f(ak[j]), f2(nk));
                // (G_r - G_en(a)) log2 e >= 0 (the running sum decreases)
                const float2 d = __fmul2_rn(__fadd2_rn(gc[j], make_float2(-gl.x, -gl.y)), L2);
                const float2 y = make_float2(ex2f(-d.x), ex2f(-d.y));          // Y  = e^{G_en(a) - G_r} <= 1
                const float2 ky = __fmul2_rn(k, y);
                const uint32_t rh = pack_bf16(ky.x, ky.y);
                const float2 rhf = bf2f(rh);
                const float2 rlo = __fadd2_rn(ky, make_float2(-rhf.x, -rhf.y));
                sts32(sRHL + jo, rh);
                sts32(sRHL + 64 * 128 + jo, pack_bf16(rlo.x, rlo.y));
                float2 qp, kpf;   // q e^G (the Q+ record) and k e^G
                if (SP) {
                    // every factor is one 2^x of a non-positive exponent
#pragma unroll
                    for (int b = 0; b < 3; ++b) {
                        if (b < a_sub) {   // e^{G_r - G_en(b)}
                            const float2 f = make_float2(ex2f(d.x + Cb[b].x), ex2f(d.y + Cb[b].y));
                            const float2 kf = __fmul2_rn(k, f), qf = __fmul2_rn(q, f);
                            sts32(sLAP + lap_off(kRowA[b] + tok0) + jo, pack_bf16(kf.x, kf.y));
                            sts32(sLAP + lap_off(kRowP[b] + tok0) + jo, pack_bf16(qf.x, qf.y));
                        }
                    }
                    const float2 eg = make_float2(ex2f(d.x + E.x), ex2f(d.y + E.y));   // e^{G_r}
                    qp = __fmul2_rn(q, eg);
                    kpf = __fmul2_rn(k, eg);
                } else {
                    const float2 iy = make_float2(ex2f(d.x), ex2f(d.y));       // iY = e^{G_r - G_en(a)} >= 1
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
                    qp = __fmul2_rn(qi, E);    // q iY E
                    kpf = __fmul2_rn(ki, E);   // k iY E
                }
                // record: Q+ = q e^{G}
                *reinterpret_cast<uint32_t*>(gQ + jo) = pack_f16(qp.x, qp.y);
                // Kt = k e^{G_last - G} = k Y F
                const float2 ktf = __fmul2_rn(ky, F);
                const uint32_t t_kt = pack_f16(ktf.x, ktf.y), t_kp = pack_f16(kpf.x, kpf.y);
                if (j & 1) {
                    const int w = j >> 1;
                    kt[0][w] = __byte_perm(kt_prev, t_kt, 0x5410);
                    kt[1][w] = __byte_perm(kt_prev, t_kt, 0x7632);
                    kp[0][w] = __byte_perm(kp_prev, t_kp, 0x5410);
                    kp[1][w] = __byte_perm(kp_prev, t_kp, 0x7632);
                } else {
                    kt_prev = t_kt;
                    kp_prev = t_kp;
                }
            }
            uint32_t vp[2][8];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                vp[0][w] = __byte_perm(av[2 * w], av[2 * w + 1], 0x5410);
                vp[1][w] = __byte_perm(av[2 * w], av[2 * w + 1], 0x7632);
            }
            // Kt, (k e^G)^T and v^T rows c0 + e, tokens tok0 .. tok0 + 15: two 16-byte
            // pieces per row.  The two pieces of a row are one aligned 32-byte sector of
            // Kt's record tile, stored straight to global memory.  In shared memory the
            // lanes of each 8-lane phase spread over all eight swizzle positions (lanes
            // 4-7 of each group of 8 write their second piece first).
            // (selects rather than a lane-dependent index, which would put the arrays in
            // local memory)
            const int x0 = (lane >> 2) & 1;
            auto pick = [](const uint32_t (&w)[8], int x) {
                return x ? make_uint4(w[4], w[5], w[6], w[7]) : make_uint4(w[0], w[1], w[2], w[3]);
            };
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int x = 0; x < 2; ++x)
                    *reinterpret_cast<uint4*>(rec + REC_KT + sw128_off(c0 + e, tok0 + 8 * x, 128)) = pick(kt[e], x);
            }
            // the previous item's W / U0 products have read (k e^G)^T and v^T (and T)
            bool bad = ft == 0 && k_iter > 0 && !wait_or_abort(bar_mma2, (k_iter - 1) & 1u, lim, abort_flag);
            if (ptx::bar_sync_or(BAR_FRONT, NF, bad)) break;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int xx = 0; xx < 2; ++xx) {
                    const int x = xx ^ x0;
                    const uint32_t off = sw128_off(c0 + e, tok0 + 8 * x, 128);
                    *reinterpret_cast<uint4*>(sb + S_KPT + off) = pick(kp[e], x);
                    *reinterpret_cast<uint4*>(sb + S_VT + off) = pick(vp[e], x);
                }
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before();
            if (ptx::bar_sync_or(BAR_FRONT, NF, *abort_flag != 0)) break;

            // ---- hand the item to the back group (which issues its first tcgen05 batch)
            if (ft == 0) {
                info[slot].rec = rec;
                info[slot].has_next = has_next;
                info[slot].t0 = cn.t0;
                info[slot].len = cn.len;
                info[slot].pos = cn.pos;
                info[slot].h = hn;
                mbar_arrive(bar_info);
            }
            ++k_iter;
            cd = cn;
            if (!last_of_batch) {
                ++jt;
            } else {
                jt = nb_start;
                j_stop = min(nb_start + a.batch, n_items);
                nb_start = a.work_counter != nullptr ? min(s_take[0] * a.batch, n_items) : n_items;
            }
        }
        // Tell the back group there are no more items: once the last item's first
        // batch has finished (so that the back has seen that item's hand-off), a null
        // record.
        if (ft == 0) {
            if (k_iter == 0 || wait_or_abort(bar_mma1, (k_iter - 1) & 1u, lim, abort_flag)) {
                info[k_iter % NSLOT].rec = nullptr;
                mbar_arrive(bar_info);
            }
        }
    } else {
        // ================================ back =================================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_BACK));
        const int bt = tid - NF, bw = warp - NF / 32;   // 0..255, 0..7
        const int qd = warp & 3;                          // TMEM lane quarter of this warp
        const float* dgb = reinterpret_cast<const float*>(sb + S_DG);
        float* l3t = reinterpret_cast<float*>(sb + S_XM + S_L3T);   // free until the diagonal inverses
        uint32_t k = 0;
#pragma unroll 1
        while (true) {
            // one thread polls the hand-off, the others wait in the barrier
            bool bad = bt == ISSUER && !wait_or_abort(bar_info, k & 1u, lim, abort_flag);
            if (ptx::bar_sync_or(BAR_BACK, NB, bad)) break;
            unsigned char* rec = info[k % NSLOT].rec;   // the same value in every thread
            if (rec == nullptr) break;
            // ---- the first tcgen05 batch: A, off-diagonal P, diagonal P
            if (bt == ISSUER) {
                ptx::tc_fence_after();
                constexpr uint32_t IDESC_BF16_N64 = ptx::idesc_bf16_f32(128, 64);
                constexpr uint32_t IDESC_BF16_N128 = ptx::idesc_bf16_f32(128, 128);
                // three independent accumulator chains, interleaved by K step: A and the
                // off-diagonal P (two M = 128 halves of the left rows) and the diagonal P
                // ([q hi; q lo] x [R hi; R lo], N = 128; the readout adds hi*hi + hi*lo + lo*hi)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk & 3) * 32, pn = kk >> 2;
                    const uint64_t bR = ptx::sdesc_sw128(base + S_RHL + pn * 16384 + koff);   // R hi rows
                    ptx::mma_f16(tmem + TM_D0, ptx::sdesc_sw128(base + S_LAP + pn * 16384 + koff), bR,
                                 IDESC_BF16_N64, kk > 0);
                    ptx::mma_f16(tmem + TM_D1, ptx::sdesc_sw128(base + S_LAP + 32768 + pn * 16384 + koff), bR,
                                 IDESC_BF16_N64, kk > 0);
                    if (!SP)
                        ptx::mma_f16(tmem + TM_D2, ptx::sdesc_sw128(base + S_QD + pn * 16384 + koff), bR,
                                     IDESC_BF16_N128, kk > 0);
                }
                if (SP) {   // the diagonal blocks' level-3 pairs: [k^ rows; q^ rows] x columns
                    constexpr uint32_t IDESC_L3 = ptx::idesc_f16_f32(128, 32);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk & 3) * 32, pn = kk >> 2;
                        // (A rows 64-127 are the next tile's bytes; their lanes are not read)
                        ptx::mma_f16(tmem + TM_D2, ptx::sdesc_sw128(base + S_L3A + pn * 8192 + koff),
                                     ptx::sdesc_sw128(base + S_L3B + pn * 4096 + koff), IDESC_L3, kk > 0);
                    }
                }
                ptx::mma_commit(bar_mma1);
            }
            const float* bta = btab + (k % NSLOT) * C;
            if (bt == ISSUER) {
                bad = !wait_or_abort(bar_mma1, k & 1u, lim, abort_flag);
                // the operand tiles are free: the next item's raw rows go there
                const volatile Handoff& hd = info[k % NSLOT];
                if (!bad && hd.has_next) {
                    issue_raw(a, hd.t0, hd.pos, hd.h, base, bar_raw);
                    *raw_issued = *raw_issued + 1;
                }
                ptx::bulk_wait_read_all();   // the previous W / U0^T staging (solve tiles) has been read
            }
            ptx::tc_fence_before();
            if (ptx::bar_sync_or(BAR_BACK, NB, bad)) break;
            ptx::tc_fence_after();

            // ---- unbounded gate: the level-3 pair sums of the diagonal blocks, from the
            // diagonal 8 x 8 blocks of the tcgen05 product (warp 8: k^ rows, lanes 0-31;
            // warp 9: q^ rows, lanes 32-63; row 8 a + i of sub-tile a), to l3t
            if (SP) {
                if (bw < 2) {
                    const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + TM_D2;
                    const int a3 = lane >> 3, i3 = lane & 7;
                    float* dst = l3t + (bw * 4 + a3) * 64 + i3 * 8;
#pragma unroll 1
                    for (int g = 0; g < 4; ++g) {   // column block g; lanes of sub-tile g keep it
                        uint32_t rg[8];
                        tmem_ld8_nw(taddr + 8 * g, rg);
                        tmem_wait_ld();
                        if (a3 == g) {
                            *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(rg[0]), __uint_as_float(rg[1]),
                                                                          __uint_as_float(rg[2]), __uint_as_float(rg[3]));
                            *reinterpret_cast<float4*>(dst + 4) = make_float4(__uint_as_float(rg[4]), __uint_as_float(rg[5]),
                                                                              __uint_as_float(rg[6]), __uint_as_float(rg[7]));
                        }
                    }
                }
                bar_sync_n(BAR_BACK, NB);
            }

            // ---- read out A (to fp32 Am, times beta_r) and the off-diagonal P (to its
            // staging tile).  A warp's 32 rows need the 16-column block of their column
            // sub-tile b: one or two blocks per warp, loaded together.
            {
                const int row0 = 128 * (bw >> 2) + 32 * qd, row = row0 + lane;
                const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + ((bw >> 2) == 0 ? TM_D0 : TM_D1);
                const int g = group_of(row);
                const int isP = kGroup[g][0], b = kGroup[g][1];
                const int r = kGroup[g][2] + (row - kGroup[g][3]);
                const int b_first = kGroup[group_of(row0)][1], b_last = kGroup[group_of(row0 + 31)][1];
                uint32_t r0[16], r1[16];
                tmem_ld16_nw(taddr + 16 * b_first, r0);
                if (b_last != b_first) tmem_ld16_nw(taddr + 16 * b_last, r1);   // (warp-uniform)
                tmem_wait_ld();
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(b == b_first ? r0[i] : r1[i]);
                if (SP && !isP && (r >> 4) == b) {   // diagonal block: the position-pair sums
                    const float* d = dgb + ((k & 1u) * 4 + b) * 256;
                    const float* t3 = l3t + b * 64;
                    const int jr = r & 15;
                    const uint4 cw = *reinterpret_cast<const uint4*>(sb + S_DGX + 16 * jr);
                    const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t code = (cws[i >> 2] >> (8 * (i & 3))) & 0xFFu, x = code & 127u;
                        v[i] = code == DG_ZERO ? 0.f : code == DG_L3 ? t3[(jr & 7) * 8 + i] : d[x] + d[128 + x];
                    }
                }
                if (isP) {
                    // (an off-diagonal block: both chunks lie in the lower triangle)
                    *reinterpret_cast<uint4*>(sb + S_TT + 16 * p_chunk(r, 2 * b)) = pack8_f16(v);
                    *reinterpret_cast<uint4*>(sb + S_TT + 16 * p_chunk(r, 2 * b + 1)) = pack8_f16(v + 8);
                } else {  // beta_r A, strictly lower part (zeros above in the diagonal block)
                    const float be = bta[r];
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
            // ---- diagonal P blocks, unbounded gate (warps 8-11): the front's position-pair
            // sums, row r = bt % 64, columns 8 (bt / 64) .. + 7 of each block
            if (SP && bw < 4) {
                const int r = bt & 63, hh = bt >> 6, ta = r >> 4, jr = r & 15;
                const float* d = dgb + ((k & 1u) * 4 + ta) * 256;
                const float* t3 = l3t + (4 + ta) * 64;
                const uint2 cw = *reinterpret_cast<const uint2*>(sb + S_DGX + 256 + 16 * jr + 8 * hh);
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t code = ((e < 4 ? cw.x : cw.y) >> (8 * (e & 3))) & 0xFFu, x = code & 127u;
                    v[e] = code == DG_ZERO ? 0.f : code == DG_L3 ? t3[(jr & 7) * 8 + 8 * hh + e] : d[x] + d[128 + x];
                }
                if (2 * ta + hh <= (r >> 3))   // (the chunk above the diagonal is zero, and not stored)
                    *reinterpret_cast<uint4*>(sb + S_TT + 16 * p_chunk(r, 2 * ta + hh)) = pack8_f16(v);
            }
            // ---- diagonal P blocks (warps 8-11): D2 rows are [q hi; q lo], columns
            // [R hi | R lo].  Warps 10-11 hand the lo*hi terms (lanes 64-127) to warps
            // 8-9 through shared memory; warps 8-9 add hi*hi + hi*lo + lo*hi.
            if (!SP && bw < 4) {
                float* pdl = reinterpret_cast<float*>(sb + S_PDL);   // fp32 [64 r][16]
                const int r = 32 * (qd & 1) + lane;                  // 0..63
                const int ta = r >> 4;
                const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + TM_D2;
                if (qd >= 2) {
                    // q lo x R hi: sub-tile ta's block (lanes 0-15: 2 (qd & 1), 16-31: the next)
                    uint32_t r0[16], r1[16];
                    tmem_ld16_nw(taddr + 16 * (2 * (qd & 1)), r0);
                    tmem_ld16_nw(taddr + 16 * (2 * (qd & 1) + 1), r1);
                    tmem_wait_ld();
                    const bool second = lane >= 16;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<float4*>(pdl + r * 16 + 4 * q) =
                            make_float4(__uint_as_float(second ? r1[4 * q] : r0[4 * q]),
                                        __uint_as_float(second ? r1[4 * q + 1] : r0[4 * q + 1]),
                                        __uint_as_float(second ? r1[4 * q + 2] : r0[4 * q + 2]),
                                        __uint_as_float(second ? r1[4 * q + 3] : r0[4 * q + 3]));
                }
                bar_sync_n(3, 128);
                if (qd < 2) {
                    // q hi x R hi, then q hi x R lo, of sub-tile ta's block (lanes 0-15:
                    // 2 qd, 16-31: the next), one load pair in flight at a time
                    const bool second = lane >= 16;
                    float v[16];
                    {
                        uint32_t r0[16], r1[16];
                        tmem_ld16_nw(taddr + 16 * (2 * qd), r0);
                        tmem_ld16_nw(taddr + 16 * (2 * qd + 1), r1);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(second ? r1[i] : r0[i]);
                    }
                    {
                        uint32_t r0[16], r1[16];
                        tmem_ld16_nw(taddr + 64 + 16 * (2 * qd), r0);
                        tmem_ld16_nw(taddr + 64 + 16 * (2 * qd + 1), r1);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 l4 = *reinterpret_cast<const float4*>(pdl + r * 16 + 4 * q);
                            const float l[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                v[4 * q + e] += __uint_as_float(second ? r1[4 * q + e] : r0[4 * q + e]) + l[e];
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        if (16 * ta + jj > r) v[jj] = 0.f;
                    *reinterpret_cast<uint4*>(sb + S_TT + 16 * p_chunk(r, 2 * ta)) = pack8_f16(v);
                    if (2 * ta + 1 <= (r >> 3))   // (otherwise above the diagonal: zero, not stored)
                        *reinterpret_cast<uint4*>(sb + S_TT + 16 * p_chunk(r, 2 * ta + 1)) = pack8_f16(v + 8);
                }
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before();
            bar_sync_n(BAR_BACK, NB);
            // P leaves
            if (bt == ISSUER) {
                ptx::bulk_s2g(rec + REC_P, base + S_TT, REC_P_BYTES);
                ptx::bulk_commit();
            }

            // ---- X = (I + A)^{-1}: diagonal 16 x 16 inverses by forward substitution
            // (warps 10-11: warps 8-9 read out diagonal P and warp 8 issues the batches,
            // so this spreads the back's work over the four SM sub-partitions)
            if (bt >= 64 && bt < 128) {
                const int ta = (bt - 64) >> 4, j = bt & 15;
                const int ob = 16 * ta;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    // x_r = e_j - sum_{s<r} A[r][s] x_s, as four interleaved partial sums
                    const float* Lr = Am + (ob + r) * LDS + ob;
                    float p4[4] = {(r == j) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int q = 0; 4 * q < r; ++q) {
                        const float4 l4 = *reinterpret_cast<const float4*>(Lr + 4 * q);
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * q + e < r) p4[e] = fmaf(-lv[e], x[4 * q + e], p4[e]);
                    }
                    x[r] = (r < j) ? 0.f : (p4[0] + p4[1]) + (p4[2] + p4[3]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Xm[(ob + r) * LDS + ob + j] = x[r];
            }
            bar_sync_n(BAR_BACK, NB);
            solve_premultiply(Am, Xm, bt);
            solve_level<1>(Am, Xm, bt);
            solve_level<2>(Am, Xm, bt);
            solve_level<3>(Am, Xm, bt);
            if (bt == ISSUER) ptx::bulk_wait_read_all();   // P has left its staging tile, where T goes
            bar_sync_n(BAR_BACK, NB);

            // ---- T = X Diag(beta) (fp16, blocks above the diagonal zero)
#pragma unroll
            for (int task = bt; task < 2 * NB; task += NB) {
                const int r = task >> 3, ch = task & 7;   // 64 rows x 8 column groups
                float v[8], xr[8], b8[8];
                lds8(Xm + r * LDS + 8 * ch, xr);
                lds8(bta + 8 * ch, b8);
                const bool keep = (ch >> 1) <= (r >> 4);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = keep ? xr[e] * b8[e] : 0.f;
                *reinterpret_cast<uint4*>(sb + S_TT + sw128_off(r, 8 * ch, 128)) = pack8_f16(v);
            }
            ptx::fence_async_smem();
            ptx::tc_fence_before();
            bar_sync_n(BAR_BACK, NB);
            if (bt == ISSUER) {
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
            }
            if (bt == ISSUER) bad = !wait_or_abort(bar_mma2, k & 1u, lim, abort_flag);
            ptx::tc_fence_before();
            if (ptx::bar_sync_or(BAR_BACK, NB, bad)) break;
            ptx::tc_fence_after();

            // ---- W (lanes = tokens 0-63) and U0^T (lanes = values) from TMEM to their
            // record image in the solve tiles: warp (quarter qd, half x = bw / 4) takes
            // W column groups 4x .. 4x+3 (quarters 0-1 only) and U0^T groups 2x, 2x+1
            {
                const int x = bw >> 2;
                const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
                // two 16-column groups per load batch, packed to fp16 into the record image
                auto group_out2 = [&](uint32_t tcol, unsigned char* dst, int col, int rows) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16_nw(tl + tcol, r0);
                    tmem_ld16_nw(tl + tcol + 16, r1);
                    tmem_wait_ld();
                    const int row = 32 * qd + lane;
                    auto pk = [](const uint32_t* w) {
                        return make_uint4(pack_f16(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                          pack_f16(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                          pack_f16(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                          pack_f16(__uint_as_float(w[6]), __uint_as_float(w[7])));
                    };
                    *reinterpret_cast<uint4*>(dst + sw128_off(row, col, rows)) = pk(r0);
                    *reinterpret_cast<uint4*>(dst + sw128_off(row, col + 8, rows)) = pk(r0 + 8);
                    *reinterpret_cast<uint4*>(dst + sw128_off(row, col + 16, rows)) = pk(r1);
                    *reinterpret_cast<uint4*>(dst + sw128_off(row, col + 24, rows)) = pk(r1 + 8);
                };
                if (qd < 2) {
#pragma unroll 1
                    for (int c = 4 * x; c < 4 * x + 4; c += 2) group_out2(TM_W + 16 * c, sb + S_WUST, 16 * c, C);
                }
                group_out2(TM_U + 32 * x, sb + S_WUST + 16384, 32 * x, 128);
            }
            ptx::fence_async_smem();
            bar_sync_n(BAR_BACK, NB);
            if (bt == ISSUER) {
                ptx::bulk_s2g(rec + REC_W, base + S_WUST, 8192);                   // W keys 0-63
                ptx::bulk_s2g(rec + REC_W + REC_PANEL, base + S_WUST + 8192, 8192);  // W keys 64-127
                ptx::bulk_s2g(rec + REC_UT, base + S_WUST + 16384, 16384);
                ptx::bulk_commit();
            }
            ++k;
        }
    }

    // ---- drain: the MMA issuer lets its MMAs finish (a commit covers every earlier
    // one of that thread), and its bulk stores land, before TMEM is freed
    if (tid == NF + ISSUER) {
        ptx::mma_commit(bar_drain);
        ptx::mbar_wait(bar_drain, 0, WAIT_LIMIT_NS);
        ptx::bulk_wait_all();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) {
        atomicExch(a.status, ERR_TIMEOUT);
        // raw-row loads still in flight land before the CTA leaves (the phases of a
        // barrier complete in order: the last issued one covers the earlier ones)
        if (*raw_issued > 0)
            for (int pl = 0; pl < 3; ++pl) ptx::mbar_wait(bar_raw[pl], (uint32_t)(*raw_issued - 1) & 1u, WAIT_LIMIT_NS);
    }
    if (warp == 0) {
        __syncwarp();   // (thread 0 may have waited above; the dealloc is warp-collective)
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
        if (!encode_rows(&a.map67[pl], planes[pl], a.T, (int64_t)a.H * D, C + RING) ||
            !encode_rows(&a.map64[pl], planes[pl], a.T, (int64_t)a.H * D, C))
            return cudaErrorInvalidValue;
    void (*kern)(PrepArgs) = a.gate_kind == KDA_GATE_SOFTPLUS ? chunk_prep_kernel<true> : chunk_prep_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int64_t grid = items < sms ? items : sms;
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    kern<<<(unsigned)grid, PT, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
