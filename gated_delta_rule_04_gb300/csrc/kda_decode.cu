// Batched decode, fully fused: for each session, n_tok consecutive tokens
// (1 for plain decode, K+1 for a speculative verify round) through conv ring
// + SiLU, L2 norms, gate, beta, the gated delta rule on the fp32 state and
// RMSNormGated.  One CTA per (session, head), 256 threads; the 64 KiB state of
// the (session, head) stays in registers across the tokens and moves through
// HBM once in each direction.
//
// The step follows the decode plan on "Kimi Delta Attention (KDA) --
// analysis & C kernel plan" (section "C kernel plan", Decode): u = S'^T k,
// d = beta (v - u), S = Diag(g) S + k d^T, o = S^T q, with S streamed once.
// Here o is formed as S'^T q + (q.k) d, so one pass over S gives both GEMVs.
// The conv arm with its ring roll mirrors the fused assemble+conv+roll
// dispatch on "memra-engine 0.124.0, module kda" (kda_attn_decode); the
// multi-token form is the batched verify-rows call of the same page
// (kda_verify_rows_cached: the recurrence stays sequential inside one launch
// over register-resident state), and keeping the input state untouched gives
// its snapshot-and-replay rollback (kda_verify_rollback_rows).
//
// Work split.  Everything that does not touch S (conv, SiLU, gate, beta, the
// L2 norms) runs for a group of up to DG tokens at once, and the output norm
// for the group runs after it.  In both kernels warp w owns key rows
// 16w..16w+15 of S and lane l value columns 4l..4l+3, so every load and store
// instruction of S moves 512 contiguous bytes and every per-row value is one
// shared-memory broadcast; the sums over key rows meet in shared memory.
// A token costs two block barriers in the round kernel (partial sums in,
// d out).  A layout that keeps the key-row sums inside a warp (an 8 x 8
// lane tile and a shuffle butterfly) needs no barrier per token, but its
// 32-byte row pieces made the state traffic alone 0.044 ms slower on 8192
// session-heads, more than the barriers cost.
//
// The state and ring are read from the input pools before anything is
// written, so input and output may alias (in-place update).
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "kda_common.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

constexpr int DC_THREADS = 256;
constexpr int DG = 8;    // tokens per group
constexpr int RP = 144;  // padded row vector: key row r at rix(r)

// Key row r of a padded row vector (a 4-float step after every 32 rows
// spreads the rows that the L2-norm step writes at once over all banks).
__device__ __forceinline__ int rix(int r) { return r + ((r >> 5) << 2); }

template <typename TI>
struct DecodeSmem {
    TI x[4][DG][D];   // raw q, k, v, z of the group
    TI go[2][DG][D];  // raw output-gate logits, double-buffered across groups
    float qc[DG][D], kc[DG][D];  // conv + SiLU of q and k, before the L2 norm
    float va[DG][D];             // conv + SiLU of v
    float so[DG][D];             // o before RMSNormGated
    float e[DG][RP];             // exp(g)
    float kh[DG][RP];            // k^
    float av[DG][RP];            // exp(g) k^  (u = S^T av = S'^T k^)
    float bv[DG][RP];            // exp(g) q^  (S^T bv = S'^T q^)
    float beta[DG], qk[DG];      // beta, q^.k^
    float red[8][2][D];          // per-warp partial sums of S^T av and S^T bv
    float sd[D];                 // d of the current token
};

// Persistent CTAs walk the (session, head) items with a stride of the grid.
// While one item computes, its successor's state (64 KiB), token rows and
// conv ring are fetched into L2, so the HBM traffic of the next item overlaps
// this item's arithmetic.  Threads 0..(5 + 3 * RING) each issue one prefetch.
template <typename TI>
__device__ __forceinline__ void prefetch_item(const DecodeArgs& a, int item, int n_tok, int tid) {
    const int H = a.H, W = H * D;
    const int n = item / H, h = item % H;
    if (tid > 5 + 3 * RING) return;
    const int slot = a.slots ? a.slots[n] : n;
    if (slot < 0 || slot >= a.n_slots) return;
    const size_t rowb = (size_t)D * sizeof(TI);
    if (tid == 0) {
        ptx::bulk_prefetch_l2(a.S_in + ((size_t)slot * H + h) * D * D, D * D * sizeof(float));
    } else if (tid <= 5) {
        const void* pl = tid == 1 ? a.q : tid == 2 ? a.k : tid == 3 ? a.v : tid == 4 ? a.z : a.gout;
        const char* base = static_cast<const char*>(pl) + ((size_t)n * n_tok * W + (size_t)h * D) * sizeof(TI);
        for (int t = 0; t < n_tok; ++t) ptx::bulk_prefetch_l2(base + (size_t)t * W * sizeof(TI), (uint32_t)rowb);
    } else {
        const int r = tid - 6;  // ring row (plane r / RING, slot r % RING)
        ptx::bulk_prefetch_l2(static_cast<const char*>(a.ring_in) +
                                  (((size_t)slot * 3 * RING + r) * W + (size_t)h * D) * sizeof(TI),
                              (uint32_t)rowb);
    }
}

// ---- one token per session (plain decode) ----------------------------------
// The token's inputs are read straight into registers (no group staging), and
// its conv, norms and gate run on the threads that own the channels; four
// block barriers in all.
template <typename TI>
__global__ void __launch_bounds__(DC_THREADS, 2) decode_kernel(DecodeArgs a) {
    const int H = a.H, W = H * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = a.n * H;
    __shared__ float s_e[D], s_k[D], s_a[D], s_b[D], s_v[D], s_d[D];
    __shared__ float s_red[8][2][D];
    __shared__ float s_sum[8][4];
    __shared__ float s_scal[2];
#pragma unroll 1
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        if (item + (int)gridDim.x < n_items) prefetch_item<TI>(a, item + gridDim.x, 1, tid);
        const int n = item / H, h = item % H;
        const int slot = a.slots ? a.slots[n] : n;
        if (slot < 0 || slot >= a.n_slots) continue;  // invalid pool index: the session is skipped

        const float* Sg_in = a.S_in + ((size_t)slot * H + h) * D * D;
        float* Sg_out = a.S_out + ((size_t)slot * H + h) * D * D;
        float4 Sr[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            Sr[r] = __ldcs(reinterpret_cast<const float4*>(Sg_in + (size_t)(16 * warp + r) * D) + lane);

        // conv windows: threads 0-127 own channel i of planes q and k, threads
        // 128-255 channel i of plane v (and the gate); slot 0 is the oldest
        const int i = tid & (D - 1);
        const int c = h * D + i;
        const int p0 = tid < D ? 0 : 2;            // first plane of this thread
        const size_t tok = (size_t)n * W + c;
        const TI* ring_in = static_cast<const TI*>(a.ring_in) + (size_t)slot * 3 * RING * W;
        TI win[2][RING];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            if (pp == 1 && p0 == 2) break;
#pragma unroll
            for (int s = 0; s < RING; ++s) win[pp][s] = ring_in[((size_t)(p0 + pp) * RING + s) * W + c];
        }
        const TI* plane0 = static_cast<const TI*>(p0 == 0 ? a.q : a.v);   // this thread's first plane
        const TI* plane1 = static_cast<const TI*>(a.k);
        auto conv_plane = [&](int pp) -> float {
            const TI xr = (pp == 0 ? plane0 : plane1)[tok];
            const float4 w = __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)(p0 + pp) * W + c) * CONV_K));
            float y = w.x * to_f32(win[pp][0]);
            y = fmaf(w.y, to_f32(win[pp][1]), y);
            y = fmaf(w.z, to_f32(win[pp][2]), y);
            y = fmaf(w.w, to_f32(xr), y);
            win[pp][0] = win[pp][1];
            win[pp][1] = win[pp][2];
            win[pp][2] = xr;
            return silu_fast(y);
        };

        // ---- conv + SiLU (threads 0-127: planes q, k; 128-255: v + gate)
        float aq = 0.f, ak = 0.f;
        if (tid < D) {
            aq = conv_plane(0);
            ak = conv_plane(1);
            const float s0 = warp_sum(aq * aq), s1 = warp_sum(ak * ak), s2 = warp_sum(aq * ak);
            if (lane == 0) { s_sum[warp][0] = s0; s_sum[warp][1] = s1; s_sum[warp][2] = s2; }
        } else {
            s_v[i] = conv_plane(0);
            const float z = to_f32(static_cast<const TI*>(a.z)[tok]);
            s_e[i] = __expf(decay_gate(a.gate_kind, a.lb, expf(a.A_log[h]), z + a.dt_bias[c]));
        }
        __syncthreads();
        if (tid < D) {
            const float sq = s_sum[0][0] + s_sum[1][0] + s_sum[2][0] + s_sum[3][0];
            const float sk = s_sum[0][1] + s_sum[1][1] + s_sum[2][1] + s_sum[3][1];
            const float sqk = s_sum[0][2] + s_sum[1][2] + s_sum[2][2] + s_sum[3][2];
            const float rq = rsqrtf(sq + a.l2_eps) * a.q_scale, rk = rsqrtf(sk + a.l2_eps);
            const float qh = aq * rq, kh = ak * rk;
            const float e = s_e[i];
            s_k[i] = kh;
            s_a[i] = e * kh;
            s_b[i] = e * qh;
            if (tid == 0) {
                s_scal[0] = sqk * rq * rk;  // q^.k^
                const float bl = to_f32(static_cast<const TI*>(a.b)[(size_t)n * H + h]);
                s_scal[1] = sigmoid_fast(bl);
            }
        }
        __syncthreads();

        // ---- u = S'^T k^ and w = S'^T q^ over this warp's 16 rows
        float u[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float ar = s_a[16 * warp + r], br = s_b[16 * warp + r];
            u[0] = fmaf(ar, Sr[r].x, u[0]); u[1] = fmaf(ar, Sr[r].y, u[1]);
            u[2] = fmaf(ar, Sr[r].z, u[2]); u[3] = fmaf(ar, Sr[r].w, u[3]);
            w[0] = fmaf(br, Sr[r].x, w[0]); w[1] = fmaf(br, Sr[r].y, w[1]);
            w[2] = fmaf(br, Sr[r].z, w[2]); w[3] = fmaf(br, Sr[r].w, w[3]);
        }
        *reinterpret_cast<float4*>(&s_red[warp][0][4 * lane]) = make_float4(u[0], u[1], u[2], u[3]);
        *reinterpret_cast<float4*>(&s_red[warp][1][4 * lane]) = make_float4(w[0], w[1], w[2], w[3]);
        __syncthreads();

        float oj = 0.f;
        if (tid < D) {
            float uj = 0.f, wj = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) { uj += s_red[k][0][tid]; wj += s_red[k][1][tid]; }
            const float dj = s_scal[1] * (s_v[tid] - uj);
            s_d[tid] = dj;
            oj = fmaf(s_scal[0], dj, wj);
            const float so = warp_sum(oj * oj);
            if (lane == 0) s_sum[warp][3] = so;
        }
        __syncthreads();

        // ---- S = Diag(e) S + k^ d^T, each row streamed out as soon as it is final
        const float4 d4 = *reinterpret_cast<const float4*>(&s_d[4 * lane]);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int rr = 16 * warp + r;
            const float er = s_e[rr], kr = s_k[rr];
            Sr[r].x = fmaf(er, Sr[r].x, kr * d4.x);
            Sr[r].y = fmaf(er, Sr[r].y, kr * d4.y);
            Sr[r].z = fmaf(er, Sr[r].z, kr * d4.z);
            Sr[r].w = fmaf(er, Sr[r].w, kr * d4.w);
            __stcs(reinterpret_cast<float4*>(Sg_out + (size_t)rr * D) + lane, Sr[r]);
        }

        // ---- RMSNormGated
        if (tid < D) {
            const float ss = s_sum[0][3] + s_sum[1][3] + s_sum[2][3] + s_sum[3][3];
            const float r = rsqrtf(ss * (1.0f / D) + a.norm_eps);
            const float gt = to_f32(static_cast<const TI*>(a.gout)[tok]);
            static_cast<TI*>(a.o)[tok] = from_f32<TI>(oj * r * a.norm_w[tid] * sigmoid_fast(gt));
        }

        // ---- ring out (after every read of the inputs)
        TI* ring_out = static_cast<TI*>(a.ring_out) + (size_t)slot * 3 * RING * W;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            if (pp == 1 && p0 == 2) break;
#pragma unroll
            for (int s = 0; s < RING; ++s) ring_out[((size_t)(p0 + pp) * RING + s) * W + c] = win[pp][s];
        }
        __syncthreads();  // the shared vectors are rewritten by the next item
    }
}

// ---- a round of n_tok >= 2 tokens per session -------------------------------
template <typename TI>
__global__ void __launch_bounds__(DC_THREADS, 2) decode_round_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) unsigned char dc_smem[];
    DecodeSmem<TI>& sm = *reinterpret_cast<DecodeSmem<TI>*>(dc_smem);
    const int H = a.H, W = H * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = a.n * H;
    const int n_tok = a.n_tok;
#pragma unroll 1
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        if (item + (int)gridDim.x < n_items) prefetch_item<TI>(a, item + gridDim.x, n_tok, tid);
        const int n = item / H, h = item % H;
        const int slot = a.slots ? a.slots[n] : n;
        if (slot < 0 || slot >= a.n_slots) continue;  // invalid pool index: the session is skipped
        const size_t row0 = (size_t)n * n_tok;      // token row of (session, token 0)

        // ---- raw inputs of the group starting at token g0, into buffer `buf`.
        // Warps 0-3 copy channels 32(w%4).. of q and k, warps 4-7 of v and z:
        // exactly what each warp's threads read in the conv step.  Warp t copies
        // the gate logits of token t, which it reads in the output step; warp 7
        // lane t prefetches the beta logit of token t into a register.
        TI b_next = TI(0.f);
        auto stage = [&](int g0, int buf) {
            const TI* pl0 = static_cast<const TI*>(warp < 4 ? a.q : a.v);
            const TI* pl1 = static_cast<const TI*>(warp < 4 ? a.k : a.z);
            const int pbase = warp < 4 ? 0 : 2, cbase = 32 * (warp & 3);
            const int ng = min(DG, n_tok - g0);
            constexpr int EPC = 16 / sizeof(TI);    // elements per 16-byte chunk
            constexpr int CPR = 32 / EPC;           // chunks per 32 channels
            for (int c = lane; c < 2 * ng * CPR; c += 32) {
                const int part = c % CPR, t = (c / CPR) % ng, pp = c / (CPR * ng);
                const size_t off = (row0 + g0 + t) * W + (size_t)h * D + cbase + part * EPC;
                ptx::cp_async16(&sm.x[pbase + pp][t][cbase + part * EPC], (pp == 0 ? pl0 : pl1) + off);
            }
            if (warp < ng) {
                const TI* gsrc = static_cast<const TI*>(a.gout) + (row0 + g0 + warp) * W + (size_t)h * D;
                for (int c = lane; c < D / EPC; c += 32) ptx::cp_async16(&sm.go[buf][warp][c * EPC], gsrc + c * EPC);
            }
            ptx::cp_async_commit();
            if (warp == 7 && lane < ng) b_next = static_cast<const TI*>(a.b)[(row0 + g0 + lane) * H + h];
        };
        stage(0, 0);

        // ---- the state: rows 16w + r, columns 4l..4l+3
        const float* Sg_in = a.S_in + ((size_t)slot * H + h) * D * D;
        float* Sg_out = a.S_out + ((size_t)slot * H + h) * D * D;
        float4 Sr[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            Sr[r] = __ldcs(reinterpret_cast<const float4*>(Sg_in + (size_t)(16 * warp + r) * D) + lane);

        // ---- conv windows in registers: threads 0-127 own channel i of planes q
        // and k, threads 128-255 channel i of plane v (and the gate); slot 0 is
        // the oldest
        const int i = tid & (D - 1);
        const int c = h * D + i;
        const int p0 = tid < D ? 0 : 2;  // first ring plane of this thread
        const TI* ring_in = static_cast<const TI*>(a.ring_in) + (size_t)slot * 3 * RING * W;
        // raw values; they become the new ring (bit-exact copy).  Plane 1 of
        // threads 128-255 is the gate logit z, which has no ring: it stays zero.
        TI win[2][RING];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
            for (int s = 0; s < RING; ++s)
                win[pp][s] = (pp == 1 && p0 == 2) ? TI(0.f) : ring_in[((size_t)(p0 + pp) * RING + s) * W + c];
        }
        float4 wconv[2];
        wconv[0] = __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)p0 * W + c) * CONV_K));
        wconv[1] = p0 == 0 ? __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)1 * W + c) * CONV_K))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        const float eA = expf(a.A_log[h]);
        const float dtb = a.dt_bias[c];

#pragma unroll 1
        for (int g0 = 0, gi = 0; g0 < n_tok; g0 += DG, ++gi) {
            const int ng = min(DG, n_tok - g0);
            const TI bl = b_next;
            ptx::cp_async_wait_all();
            __syncwarp();

            // ---- conv + SiLU, gate, beta of the group's tokens.  The conv reads a
            // sequence of the 3 window values and the group's raw inputs, so the
            // tokens do not depend on one another and their exponentials and
            // divides overlap.  NT (2, 4 or 8) rows are computed, those past the
            // group's end dropped.
            auto conv_group = [&](auto nt_c) {
                constexpr int NT = decltype(nt_c)::value;
                TI xs[2][RING + NT];
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
                    for (int s = 0; s < RING; ++s) xs[pp][s] = win[pp][s];
#pragma unroll
                    for (int t = 0; t < NT; ++t) xs[pp][RING + t] = sm.x[p0 + pp][t][i];
                }
                auto conv_at = [&](int pp, int t) -> float {
                    const float4 w = wconv[pp];
                    float y = w.x * to_f32(xs[pp][t]);
                    y = fmaf(w.y, to_f32(xs[pp][t + 1]), y);
                    y = fmaf(w.z, to_f32(xs[pp][t + 2]), y);
                    y = fmaf(w.w, to_f32(xs[pp][t + 3]), y);
                    return silu_fast(y);
                };
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (tid < D) {
                        const float yq = conv_at(0, t), yk = conv_at(1, t);
                        if (t < ng) {
                            sm.qc[t][i] = yq;
                            sm.kc[t][i] = yk;
                        }
                    } else {
                        const float yv = conv_at(0, t);
                        const float ee = __expf(decay_gate(a.gate_kind, a.lb, eA, to_f32(xs[1][RING + t]) + dtb));
                        if (t < ng) {
                            sm.va[t][i] = yv;
                            sm.e[t][rix(i)] = ee;
                        }
                    }
                }
                // the window after the group: raw inputs ng .. ng + 2 of the sequence
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
                    for (int s = 0; s < RING; ++s) {
                        TI v = xs[pp][s];
#pragma unroll
                        for (int m = 1; m <= NT; ++m) v = ng == m ? xs[pp][m + s] : v;
                        win[pp][s] = v;
                    }
                }
            };
            if (ng <= 2) conv_group(std::integral_constant<int, 2>{});
            else if (ng <= 4) conv_group(std::integral_constant<int, 4>{});
            else conv_group(std::integral_constant<int, DG>{});
            if (warp == 7 && lane < ng) sm.beta[lane] = sigmoid_fast(to_f32(bl));
            __syncthreads();
            if (g0 + DG < n_tok) stage(g0 + DG, (gi + 1) & 1);  // the staged inputs are consumed

            // ---- L2 norms: warp t normalises token t, lane l channels 4l..4l+3
            if (warp < ng) {
                const int t = warp, ro = rix(4 * lane);
                const float4 q4 = *reinterpret_cast<const float4*>(&sm.qc[t][4 * lane]);
                const float4 k4 = *reinterpret_cast<const float4*>(&sm.kc[t][4 * lane]);
                const float4 e4 = *reinterpret_cast<const float4*>(&sm.e[t][ro]);
                float sq = q4.x * q4.x, sk = k4.x * k4.x, sqk = q4.x * k4.x;
                sq = fmaf(q4.y, q4.y, sq); sk = fmaf(k4.y, k4.y, sk); sqk = fmaf(q4.y, k4.y, sqk);
                sq = fmaf(q4.z, q4.z, sq); sk = fmaf(k4.z, k4.z, sk); sqk = fmaf(q4.z, k4.z, sqk);
                sq = fmaf(q4.w, q4.w, sq); sk = fmaf(k4.w, k4.w, sk); sqk = fmaf(q4.w, k4.w, sqk);
                sq = warp_sum(sq);
                sk = warp_sum(sk);
                sqk = warp_sum(sqk);
                const float rq = rsqrtf(sq + a.l2_eps) * a.q_scale, rk = rsqrtf(sk + a.l2_eps);
                const float4 kh = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
                const float4 qh = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
                *reinterpret_cast<float4*>(&sm.kh[t][ro]) = kh;
                *reinterpret_cast<float4*>(&sm.av[t][ro]) =
                    make_float4(e4.x * kh.x, e4.y * kh.y, e4.z * kh.z, e4.w * kh.w);
                *reinterpret_cast<float4*>(&sm.bv[t][ro]) =
                    make_float4(e4.x * qh.x, e4.y * qh.y, e4.z * qh.z, e4.w * qh.w);
                if (lane == 0) sm.qk[t] = sqk * rq * rk;
            }
            __syncthreads();

            // ---- the recurrence over the group: per token, partial S^T av and
            // S^T bv over this warp's 16 rows, their sums and d per column, and
            // the rank-1 update; column pairs run as packed fp32 pairs
#pragma unroll 1
            for (int t = 0; t < ng; ++t) {
                const float* A = &sm.av[t][rix(16 * warp)];
                const float* B = &sm.bv[t][rix(16 * warp)];
                const float2 z2 = make_float2(0.f, 0.f);
                float2 u01[2] = {z2, z2}, u23[2] = {z2, z2}, w01[2] = {z2, z2}, w23[2] = {z2, z2};
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(A + 4 * r4);
                    const float4 b4 = *reinterpret_cast<const float4*>(B + 4 * r4);
                    const float ar[4] = {a4.x, a4.y, a4.z, a4.w}, br[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int r = 4 * r4 + m, p = m & 1;
                        const float2 aa = make_float2(ar[m], ar[m]), bb = make_float2(br[m], br[m]);
                        const float2 s01 = make_float2(Sr[r].x, Sr[r].y), s23 = make_float2(Sr[r].z, Sr[r].w);
                        u01[p] = __ffma2_rn(aa, s01, u01[p]); u23[p] = __ffma2_rn(aa, s23, u23[p]);
                        w01[p] = __ffma2_rn(bb, s01, w01[p]); w23[p] = __ffma2_rn(bb, s23, w23[p]);
                    }
                }
                const float2 uu01 = __fadd2_rn(u01[0], u01[1]), uu23 = __fadd2_rn(u23[0], u23[1]);
                const float2 ww01 = __fadd2_rn(w01[0], w01[1]), ww23 = __fadd2_rn(w23[0], w23[1]);
                *reinterpret_cast<float4*>(&sm.red[warp][0][4 * lane]) = make_float4(uu01.x, uu01.y, uu23.x, uu23.y);
                *reinterpret_cast<float4*>(&sm.red[warp][1][4 * lane]) = make_float4(ww01.x, ww01.y, ww23.x, ww23.y);
                __syncthreads();
                if (tid < D) {
                    float uj = 0.f, wj = 0.f;
#pragma unroll
                    for (int k = 0; k < 8; ++k) { uj += sm.red[k][0][tid]; wj += sm.red[k][1][tid]; }
                    const float dj = sm.beta[t] * (sm.va[t][tid] - uj);
                    sm.sd[tid] = dj;
                    sm.so[t][tid] = fmaf(sm.qk[t], dj, wj);
                }
                __syncthreads();
                const float4 d4 = *reinterpret_cast<const float4*>(&sm.sd[4 * lane]);
                const float2 d01 = make_float2(d4.x, d4.y), d23 = make_float2(d4.z, d4.w);
                const float* E = &sm.e[t][rix(16 * warp)];
                const float* K = &sm.kh[t][rix(16 * warp)];
                // S = Diag(e) S + k^ d^T; after the last token each row streams out
                // as soon as it is final (every read of S_in is behind us)
                const bool last = g0 + t + 1 == n_tok;
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const float4 e4 = *reinterpret_cast<const float4*>(E + 4 * r4);
                    const float4 k4 = *reinterpret_cast<const float4*>(K + 4 * r4);
                    const float er[4] = {e4.x, e4.y, e4.z, e4.w}, kr[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int r = 4 * r4 + m;
                        const float2 ee = make_float2(er[m], er[m]), kk = make_float2(kr[m], kr[m]);
                        const float2 s01 = __ffma2_rn(ee, make_float2(Sr[r].x, Sr[r].y), __fmul2_rn(kk, d01));
                        const float2 s23 = __ffma2_rn(ee, make_float2(Sr[r].z, Sr[r].w), __fmul2_rn(kk, d23));
                        Sr[r] = make_float4(s01.x, s01.y, s23.x, s23.y);
                        if (last) __stcs(reinterpret_cast<float4*>(Sg_out + (size_t)(16 * warp + r) * D) + lane, Sr[r]);
                    }
                }
            }
            __syncthreads();

            // ---- RMSNormGated: warp t finishes token t, lane l channels 4l..4l+3
            if (warp < ng) {
                const int t = warp;
                const float4 o4 = *reinterpret_cast<const float4*>(&sm.so[t][4 * lane]);
                float ss = o4.x * o4.x;
                ss = fmaf(o4.y, o4.y, ss);
                ss = fmaf(o4.z, o4.z, ss);
                ss = fmaf(o4.w, o4.w, ss);
                ss = warp_sum(ss);
                const float r = rsqrtf(ss * (1.0f / D) + a.norm_eps);
                const float4 nw = __ldg(reinterpret_cast<const float4*>(a.norm_w) + lane);
                const TI* gg = &sm.go[gi & 1][t][4 * lane];
                const float ov[4] = {o4.x, o4.y, o4.z, o4.w}, nv[4] = {nw.x, nw.y, nw.z, nw.w};
                TI y[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) y[m] = from_f32<TI>(ov[m] * r * nv[m] * sigmoid_fast(to_f32(gg[m])));
                TI* dst = static_cast<TI*>(a.o) + (row0 + g0 + t) * W + (size_t)h * D + 4 * lane;
                if constexpr (sizeof(TI) == 4) {
                    *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(y);
                } else {
                    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(y);
                }
            }
        }

        // ---- ring out (written once, after every read of the inputs)
        TI* ring_out = static_cast<TI*>(a.ring_out) + (size_t)slot * 3 * RING * W;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            if (pp == 1 && p0 == 2) break;
#pragma unroll
            for (int s = 0; s < RING; ++s) ring_out[((size_t)(p0 + pp) * RING + s) * W + c] = win[pp][s];
        }
        __syncthreads();  // the staging buffers are rewritten by the next item
    }
}

// Resident CTAs of a decode kernel: two per SM (the register budget of
// __launch_bounds__), looked up once per device.
int decode_grid(int64_t items) {
    static std::atomic<int> sms_cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return (int)std::min<int64_t>(items, 2 * 152);
    int sms = dev < 64 ? sms_cache[dev].load() : 0;
    if (sms == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
        if (dev < 64) sms_cache[dev].store(sms);
    }
    return (int)std::min<int64_t>(items, 2 * (int64_t)sms);
}

template <typename TI>
cudaError_t launch_round(const DecodeArgs& a, int64_t blocks, cudaStream_t s) {
    constexpr size_t smem = sizeof(DecodeSmem<TI>);
    // above the 48 KiB default the kernel needs the opt-in, once per device
    static std::atomic<uint64_t> opted{0};
    if (smem > 48 * 1024) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = dev < 64 ? uint64_t(1) << dev : 0;
        if (!bit || !(opted.load() & bit)) {
            e = cudaFuncSetAttribute(decode_round_kernel<TI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            opted.fetch_or(bit);
        }
    }
    // Short rounds walk the items persistently, prefetching the next one; from
    // 8 tokens on, the arithmetic of an item covers the latency of the next
    // load anyway and one CTA per item measured faster.
    const int grid = a.n_tok <= 4 ? decode_grid(blocks) : (int)blocks;
    decode_round_kernel<TI><<<grid, DC_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int io_bf16, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.n * a.H;
    if (blocks == 0 || a.n_tok == 0) return cudaSuccess;
    if (a.n_tok == 1) {
        const int grid = decode_grid(blocks);
        if (io_bf16) decode_kernel<__nv_bfloat16><<<grid, DC_THREADS, 0, s>>>(a);
        else decode_kernel<float><<<grid, DC_THREADS, 0, s>>>(a);
        return cudaGetLastError();
    }
    return io_bf16 ? launch_round<__nv_bfloat16>(a, blocks, s) : launch_round<float>(a, blocks, s);
}

}  // namespace kda
