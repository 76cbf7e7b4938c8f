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
// Memory: warp w owns key rows 16w..16w+15 of S, lane l value columns
// 4l..4l+3, so every load and store instruction moves 512 contiguous bytes.
// The state and ring are read from the input pools before anything is
// written, so input and output may alias (in-place update).
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int DC_THREADS = 256;

// ONE: a.n_tok == 1 (plain decode), compiled without the token loop
template <typename TI, bool ONE>
__global__ void __launch_bounds__(DC_THREADS, 2) decode_kernel(DecodeArgs a) {
    const int H = a.H, W = H * D;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = a.slots ? a.slots[n] : n;
    if (slot < 0 || slot >= a.n_slots) return;  // invalid pool index: the session is skipped

    const float* Sg_in = a.S_in + ((size_t)slot * H + h) * D * D;
    float* Sg_out = a.S_out + ((size_t)slot * H + h) * D * D;
    float4 Sr[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        Sr[r] = __ldcs(reinterpret_cast<const float4*>(Sg_in + (size_t)(16 * warp + r) * D) + lane);

    __shared__ float s_e[D], s_k[D], s_a[D], s_b[D], s_v[D], s_d[D];
    __shared__ float s_red[8][2][D];
    __shared__ float s_sum[8][4];
    __shared__ float s_scal[2];

    // conv windows in registers: threads 0-127 own channel i of planes q and k,
    // threads 128-255 channel i of plane v (and the gate); slot 0 is the oldest
    const int i = tid & (D - 1);
    const int c = h * D + i;
    const int p0 = tid < D ? 0 : 2;            // first plane of this thread
    const TI* ring_in = static_cast<const TI*>(a.ring_in) + (size_t)slot * 3 * RING * W;
    float win[2][RING];
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        if (pp == 1 && p0 == 2) break;
#pragma unroll
        for (int s = 0; s < RING; ++s) win[pp][s] = to_f32(ring_in[((size_t)(p0 + pp) * RING + s) * W + c]);
    }
    TI raw_last[2][RING];                      // raw values of the new ring (bit-exact copy)
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        if (pp == 1 && p0 == 2) break;
#pragma unroll
        for (int s = 0; s < RING; ++s) raw_last[pp][s] = ring_in[((size_t)(p0 + pp) * RING + s) * W + c];
    }
    float4 wconv[2];
    wconv[0] = __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)p0 * W + c) * CONV_K));
    wconv[1] = p0 == 0 ? __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)1 * W + c) * CONV_K))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    const TI* plane0 = static_cast<const TI*>(p0 == 0 ? a.q : a.v);   // this thread's first plane
    const TI* plane1 = static_cast<const TI*>(a.k);
    const float eA = expf(a.A_log[h]);
    const float dtb = a.dt_bias[c];

    const int n_tok = ONE ? 1 : a.n_tok;
#pragma unroll 1
    for (int t = 0; t < n_tok; ++t) {
        const size_t row = (size_t)n * n_tok + t;     // token row of (session, t)
        const size_t tok = row * W + c;
        auto conv_plane = [&](int pp) -> float {
            const TI xr = (pp == 0 ? plane0 : plane1)[tok];
            const float xv = to_f32(xr);
            const float4 w = wconv[pp];
            float y = w.x * win[pp][0];
            y = fmaf(w.y, win[pp][1], y);
            y = fmaf(w.z, win[pp][2], y);
            y = fmaf(w.w, xv, y);
            win[pp][0] = win[pp][1];
            win[pp][1] = win[pp][2];
            win[pp][2] = xv;
            raw_last[pp][0] = raw_last[pp][1];
            raw_last[pp][1] = raw_last[pp][2];
            raw_last[pp][2] = xr;
            return y / (1.0f + expf(-y));
        };

        // ---- prologue: conv + SiLU (threads 0-127: planes q, k; 128-255: v + gate)
        float aq = 0.f, ak = 0.f;
        if (tid < D) {
            aq = conv_plane(0);
            ak = conv_plane(1);
            const float s0 = warp_sum(aq * aq), s1 = warp_sum(ak * ak), s2 = warp_sum(aq * ak);
            if (lane == 0) { s_sum[warp][0] = s0; s_sum[warp][1] = s1; s_sum[warp][2] = s2; }
        } else {
            s_v[i] = conv_plane(0);
            const float z = to_f32(static_cast<const TI*>(a.z)[tok]);
            const float g = decay_gate(a.gate_kind, a.lb, eA, z + dtb);
            s_e[i] = expf(g);
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
                const float bl = to_f32(static_cast<const TI*>(a.b)[row * H + h]);
                s_scal[1] = 1.0f / (1.0f + expf(-bl));
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

        // ---- S = Diag(e) S + k^ d^T (registers); after the last token each row
        // streams out as soon as it is final (every read of S_in is behind us)
        const float4 d4 = *reinterpret_cast<const float4*>(&s_d[4 * lane]);
        const bool last = t + 1 == n_tok;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int rr = 16 * warp + r;
            const float er = s_e[rr], kr = s_k[rr];
            Sr[r].x = fmaf(er, Sr[r].x, kr * d4.x);
            Sr[r].y = fmaf(er, Sr[r].y, kr * d4.y);
            Sr[r].z = fmaf(er, Sr[r].z, kr * d4.z);
            Sr[r].w = fmaf(er, Sr[r].w, kr * d4.w);
            if (last) __stcs(reinterpret_cast<float4*>(Sg_out + (size_t)rr * D) + lane, Sr[r]);
        }

        // ---- RMSNormGated epilogue
        if (tid < D) {
            const float ss = s_sum[0][3] + s_sum[1][3] + s_sum[2][3] + s_sum[3][3];
            const float r = rsqrtf(ss * (1.0f / D) + a.norm_eps);
            const float gt = to_f32(static_cast<const TI*>(a.gout)[tok]);
            const float y = oj * r * a.norm_w[tid] / (1.0f + expf(-gt));
            static_cast<TI*>(a.o)[tok] = from_f32<TI>(y);
        }
        if (!last) __syncthreads();  // the shared vectors are rewritten by the next token
    }

    // ---- ring out (written once, after every read of the inputs)
    TI* ring_out = static_cast<TI*>(a.ring_out) + (size_t)slot * 3 * RING * W;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        if (pp == 1 && p0 == 2) break;
#pragma unroll
        for (int s = 0; s < RING; ++s) ring_out[((size_t)(p0 + pp) * RING + s) * W + c] = raw_last[pp][s];
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int io_bf16, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.n * a.H;
    if (blocks == 0 || a.n_tok == 0) return cudaSuccess;
    const bool one = a.n_tok == 1;
    if (io_bf16) {
        if (one) decode_kernel<__nv_bfloat16, true><<<(unsigned)blocks, DC_THREADS, 0, s>>>(a);
        else decode_kernel<__nv_bfloat16, false><<<(unsigned)blocks, DC_THREADS, 0, s>>>(a);
    } else {
        if (one) decode_kernel<float, true><<<(unsigned)blocks, DC_THREADS, 0, s>>>(a);
        else decode_kernel<float, false><<<(unsigned)blocks, DC_THREADS, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
