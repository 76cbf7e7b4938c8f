// Batched one-token decode, fully fused: conv ring + SiLU, L2 norms, gate,
// beta, one pass of the gated delta rule over the fp32 state, RMSNormGated,
// ring roll.  One CTA per (session, head), 256 threads.
//
// The step follows the decode plan on "Kimi Delta Attention (KDA) --
// analysis & C kernel plan" (section "C kernel plan", Decode): u = S'^T k,
// d = beta (v - u), S = Diag(g) S + k d^T, o = S^T q, with S streamed once.
// Here o is formed as S'^T q + (q.k) d, so S is read once (both GEMVs in one
// pass) and written once.  The conv arm with its ring roll mirrors the fused
// assemble+conv+roll dispatch on "memra-engine 0.124.0, module kda"
// (kda_attn_decode).
//
// Memory: the 64 KiB state of a (session, head) is loaded into registers at
// kernel entry (16 float4 per thread, issued before any other work so the
// whole tile is in flight while the prologue runs) and written back once with
// streaming stores.  Warp w owns key rows 16w..16w+15, lane l value columns
// 4l..4l+3, so every load and store instruction moves 512 contiguous bytes.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int DC_THREADS = 256;

template <typename TI>
__global__ void __launch_bounds__(DC_THREADS, 2) decode_kernel(DecodeArgs a) {
    const int H = a.H, W = H * D;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    float* Sg = a.S + ((size_t)n * H + h) * D * D;
    float4 Sr[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
        Sr[r] = __ldcs(reinterpret_cast<const float4*>(Sg + (size_t)(16 * warp + r) * D) + lane);

    __shared__ float s_e[D], s_k[D], s_a[D], s_b[D], s_v[D], s_d[D];
    __shared__ float s_red[8][2][D];
    __shared__ float s_sum[8][4];
    __shared__ float s_scal[2];

    // ---- prologue: conv + SiLU (threads 0-127: planes q, k; 128-255: v + gate)
    const int i = tid & (D - 1);
    const int c = h * D + i;
    TI* ring = static_cast<TI*>(a.ring) + (size_t)n * 3 * RING * W;
    const size_t tok = (size_t)n * W + c;
    auto conv_plane = [&](int p, const TI* x) -> float {
        TI* rp = ring + (size_t)p * RING * W + c;
        const float r0 = to_f32(rp[0]), r1 = to_f32(rp[W]), r2 = to_f32(rp[2 * W]);
        const TI xr = x[tok];
        const float xv = to_f32(xr);
        const float4 w = __ldg(reinterpret_cast<const float4*>(a.conv_w + ((size_t)p * W + c) * CONV_K));
        float y = w.x * r0;
        y = fmaf(w.y, r1, y);
        y = fmaf(w.z, r2, y);
        y = fmaf(w.w, xv, y);
        // roll the ring: slots (0,1,2) <- (1,2,new); this thread owns the channel
        rp[0] = rp[W];
        rp[W] = rp[2 * W];
        rp[2 * W] = xr;
        return y / (1.0f + expf(-y));
    };
    float aq = 0.f, ak = 0.f;
    if (tid < D) {
        aq = conv_plane(0, static_cast<const TI*>(a.q));
        ak = conv_plane(1, static_cast<const TI*>(a.k));
        float s0 = warp_sum(aq * aq), s1 = warp_sum(ak * ak), s2 = warp_sum(aq * ak);
        if (lane == 0) { s_sum[warp][0] = s0; s_sum[warp][1] = s1; s_sum[warp][2] = s2; }
    } else {
        s_v[i] = conv_plane(2, static_cast<const TI*>(a.v));
        const float z = to_f32(static_cast<const TI*>(a.z)[tok]);
        const float g = a.lb / (1.0f + expf(-expf(a.A_log[h]) * (z + a.dt_bias[c])));
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
            const float bl = to_f32(static_cast<const TI*>(a.b)[(size_t)n * H + h]);
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

    // ---- S = Diag(e) S + k^ d^T, written once
    const float4 d4 = *reinterpret_cast<const float4*>(&s_d[4 * lane]);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int row = 16 * warp + r;
        const float er = s_e[row], kr = s_k[row];
        float4 s = Sr[r];
        s.x = fmaf(er, s.x, kr * d4.x);
        s.y = fmaf(er, s.y, kr * d4.y);
        s.z = fmaf(er, s.z, kr * d4.z);
        s.w = fmaf(er, s.w, kr * d4.w);
        __stcs(reinterpret_cast<float4*>(Sg + (size_t)row * D) + lane, s);
    }

    // ---- RMSNormGated epilogue
    if (tid < D) {
        const float ss = s_sum[0][3] + s_sum[1][3] + s_sum[2][3] + s_sum[3][3];
        const float r = rsqrtf(ss * (1.0f / D) + a.norm_eps);
        const float gt = to_f32(static_cast<const TI*>(a.gout)[tok]);
        const float y = oj * r * a.norm_w[tid] / (1.0f + expf(-gt));
        static_cast<TI*>(a.o)[tok] = from_f32<TI>(y);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int io_bf16, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.n * a.H;
    if (blocks == 0) return cudaSuccess;
    if (io_bf16) decode_kernel<__nv_bfloat16><<<(unsigned)blocks, DC_THREADS, 0, s>>>(a);
    else decode_kernel<float><<<(unsigned)blocks, DC_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
