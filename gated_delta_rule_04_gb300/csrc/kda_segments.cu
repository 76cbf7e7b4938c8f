// Composition of segment maps for the segmented recurrence of one sequence
// (the context-parallel state exchange run inside one GPU).
//
// The chunk step of the recurrence is affine in the state and acts on every
// value column alike: S' = A S + B with A = Diag(decay) - Kt^T W and
// B = Kt^T U0 ("memra-engine 0.124.0, module kda", PREFILL DISPATCH: the
// chunked form; the segment maps are the exchange a context-parallel split of
// one sequence needs).  Over a segment the steps compose to S_end = M S_start
// + B_seg: M comes from running the segment's linear part from the identity,
// B_seg from running it from zero.  With X_1 = B_0 (the state after segment 0,
// which starts from the caller's state), the state entering segment p + 1 is
// X_{p+1} = M_p X_p + B_p.  Value columns never mix, so each CTA takes one
// head and a block of 16 value columns through every segment in order.
#include "kda_chunk_layout.cuh"

namespace kda {
namespace {

constexpr int ST = 256;   // threads
constexpr int VB = 16;    // value columns per CTA

__global__ void __launch_bounds__(ST) affine_scan_kernel(const __grid_constant__ ScanArgs2 a) {
    __shared__ float xs[D][VB];   // X_p, this block of columns
    const int h = blockIdx.x, vb = blockIdx.y * VB;
    const int tid = threadIdx.x;
    const int key = tid >> 1, vh = (tid & 1) * (VB / 2);   // thread: one key row, 8 value columns
    const size_t hoff = (size_t)h * D * D;
    // X_1 = B_0
    for (int i = tid; i < D * VB; i += ST) xs[i / VB][i % VB] = a.B[0][hoff + (size_t)(i / VB) * D + vb + i % VB];
    __syncthreads();
    for (int p = 1; p + 1 < a.P; ++p) {
        const float* Mp = a.M[p] + hoff + (size_t)key * D;
        const float* Bp = a.B[p] + hoff + (size_t)key * D + vb + vh;
        float acc[VB / 2];
#pragma unroll
        for (int e = 0; e < VB / 2; ++e) acc[e] = Bp[e];
#pragma unroll 4
        for (int j = 0; j < D; ++j) {
            const float m = __ldg(Mp + j);
#pragma unroll
            for (int e = 0; e < VB / 2; ++e) acc[e] = fmaf(m, xs[j][vh + e], acc[e]);
        }
        __syncthreads();   // every thread has read X_p
        float* Xn = a.X[p + 1] + hoff + (size_t)key * D + vb + vh;
#pragma unroll
        for (int e = 0; e < VB / 2; ++e) {
            xs[key][vh + e] = acc[e];
            Xn[e] = acc[e];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_affine_scan(const ScanArgs2& a, cudaStream_t s) {
    if (a.P < 3 || a.P > MAX_SEGS || a.H < 1) return cudaSuccess;
    affine_scan_kernel<<<dim3((unsigned)a.H, D / VB), ST, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
