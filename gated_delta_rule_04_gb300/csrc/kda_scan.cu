// Sequential-scan prefill of the gated delta recurrence in fp32 (the path
// for fp32 I/O, and an independent GPU cross-check of the chunked kernel).
//
//   S' = Diag(exp(g_t)) S;  u = S'^T k;  S = S' + beta k (v - u)^T;  o = S^T q
// ("Kimi Delta Attention (KDA) -- analysis & C kernel plan", section
// "Recurrence").  The output is formed without a second pass over S:
//   o = S'^T q + (q.k) beta (v - u),
// so each token needs one reduction over the key axis for u, w = S'^T q and
// q.k together.  The T-loop runs inside the kernel with the state resident in
// registers, as the sequential scan on the memra-engine page
// ("memra-engine 0.124.0, module kda", PREFILL DISPATCH) does.
//
// Mapping: one warp per (sequence, head, 4 value columns); lane l owns key
// rows l, l+32, l+64, l+96, so a thread holds a 4x4 block of S and the
// reduction over keys is a warp butterfly.  Four warps (16 columns) per CTA
// share the q/k/g rows through L1.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int SC_WARPS = 4;
constexpr int SC_COLS = SC_WARPS * 4;      // value columns per CTA
constexpr int SC_VBLOCKS = D / SC_COLS;    // CTAs per (sequence, head)

__global__ void __launch_bounds__(SC_WARPS * 32) scan_kernel(ScanArgs a) {
    const int H = a.H, W = H * D;
    const int vb = blockIdx.x % SC_VBLOCKS;
    const int h = (blockIdx.x / SC_VBLOCKS) % H;
    const int n = blockIdx.x / (SC_VBLOCKS * H);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = vb * SC_COLS + warp * 4;

    const size_t soff = ((size_t)n * H + h) * D * D;
    float S[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.S_in) s4 = *reinterpret_cast<const float4*>(a.S_in + soff + (size_t)(lane + 32 * m) * D + col0);
        S[m][0] = s4.x; S[m][1] = s4.y; S[m][2] = s4.z; S[m][3] = s4.w;
    }

    const int64_t bos = a.cu[n], eos = a.cu[n + 1];
    // software pipeline: the next token's inputs are loaded before this one's math
    float qn[4], kn[4], gn[4], bn = 0.f;
    float4 vn = make_float4(0.f, 0.f, 0.f, 0.f);
    auto load = [&](int64_t t) {
        const size_t base = (size_t)t * W + h * D;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            qn[m] = __ldg(a.qh + base + lane + 32 * m);
            kn[m] = __ldg(a.kh + base + lane + 32 * m);
            gn[m] = __ldg(a.g + base + lane + 32 * m);
        }
        vn = __ldg(reinterpret_cast<const float4*>(a.vh + base + col0));
        bn = __ldg(a.beta + (size_t)t * H + h);
    };
    if (bos < eos) load(bos);
    for (int64_t t = bos; t < eos; ++t) {
        float q[4], k[4], g[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) { q[m] = qn[m]; k[m] = kn[m]; g[m] = gn[m]; }
        const float4 v4 = vn;
        const float beta = bn;
        if (t + 1 < eos) load(t + 1);

        float e[4], red[9];
#pragma unroll
        for (int j = 0; j < 9; ++j) red[j] = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            e[m] = expf(g[m]);
            const float ak = e[m] * k[m], aq = e[m] * q[m];
            red[8] = fmaf(q[m], k[m], red[8]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                red[j] = fmaf(ak, S[m][j], red[j]);       // u = S'^T k
                red[4 + j] = fmaf(aq, S[m][j], red[4 + j]);  // w = S'^T q
            }
        }
#pragma unroll
        for (int j = 0; j < 9; ++j) red[j] = warp_sum(red[j]);
        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
        float d[4], o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            d[j] = beta * (vv[j] - red[j]);
            o[j] = fmaf(red[8], d[j], red[4 + j]);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) S[m][j] = fmaf(e[m], S[m][j], k[m] * d[j]);
        if (lane == 0)
            *reinterpret_cast<float4*>(a.o_core + (size_t)t * W + h * D + col0) = make_float4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
        *reinterpret_cast<float4*>(a.S_out + soff + (size_t)(lane + 32 * m) * D + col0) =
            make_float4(S[m][0], S[m][1], S[m][2], S[m][3]);
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s) {
    const int64_t blocks = (int64_t)a.n_seqs * a.H * SC_VBLOCKS;
    if (blocks == 0) return cudaSuccess;
    scan_kernel<<<(unsigned)blocks, SC_WARPS * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
