// Output RMSNormGated with a sigmoid gate, per (token, head):
//   o = o_core / sqrt(mean_i o_core^2 + eps) * norm_w[i] * sigmoid(gout)
// ("Kimi Delta Attention (KDA) -- analysis & C kernel plan", section "The KDA
// layer, precisely": o = RMSNormGated(o, gate); "ferrox-models 0.8.0, module
// kda", fact 2: the gate activation is sigmoid).
// One half warp per (token, head), 8 channels per lane in 16/32-byte vectors.
#include "kda_common.cuh"

namespace kda {
namespace {

template <typename TI>
__global__ void __launch_bounds__(256) epilogue_kernel(EpilogueArgs a) {
    const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
    const int l16 = threadIdx.x & 15;
    const int H = a.H, W = H * D;
    const bool live = item < a.T * H;
    const int64_t t = live ? item / H : 0;
    const int h = live ? (int)(item % H) : 0;
    const size_t off = (size_t)t * W + h * D + l16 * 8;
    float x[8], gt[8], w[8];
    float ss = 0.f;
    if (live) {
        Vec8<float>::load(a.o_core + off, x);
        Vec8<TI>::load(static_cast<const TI*>(a.gout) + off, gt);
        Vec8<float>::load(a.norm_w + l16 * 8, w);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
    }
    ss = halfwarp_sum(ss);
    if (!live) return;
    const float r = rsqrtf(ss * (1.0f / D) + a.eps);
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = x[e] * r * w[e] / (1.0f + expf(-gt[e]));
    Vec8<TI>::store(static_cast<TI*>(a.o) + off, y);
}

}  // namespace

cudaError_t launch_epilogue(const EpilogueArgs& a, int io_bf16, cudaStream_t s) {
    const int64_t halves = a.T * a.H;
    if (halves == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((halves * 16 + 255) / 256);
    if (io_bf16) epilogue_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(a);
    else epilogue_kernel<float><<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
