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
// head and a block of 8 value columns through every segment in order, M_p
// passing through shared memory 32 keys at a time.
#include "kda_chunk_layout.cuh"

namespace kda {
namespace {

constexpr int ST = 128;   // threads: one key row each
constexpr int VB = 8;     // value columns per CTA
constexpr int JC = 32;    // keys of M_p staged in shared memory at a time

__global__ void __launch_bounds__(ST) affine_scan_kernel(const __grid_constant__ ScanArgs2 a) {
    __shared__ float xs[D][VB];        // X_p, this block of columns
    __shared__ float ms[D][JC + 1];    // 32 columns of M_p (padded: row reads are conflict-free)
    const int h = blockIdx.x, vb = blockIdx.y * VB;
    const int key = threadIdx.x;
    const size_t hoff = (size_t)h * D * D;
    constexpr int NLD = D * JC / 4 / ST;   // float4 loads per thread per block of M_p
    // the next block of M_p is loaded into registers while the current one is used:
    // the loads do not depend on X, so the chain waits for one block's latency at most
    float4 nx[NLD];
    auto load_block = [&](int p, int jc) {
        const float* Mp = a.M[p] + hoff;
#pragma unroll
        for (int i = 0; i < NLD; ++i) {
            const int idx = key + ST * i, r = idx >> 3, c = (idx & 7) * 4;
            nx[i] = __ldg(reinterpret_cast<const float4*>(Mp + (size_t)r * D + jc + c));
        }
    };
    // X_1 = B_0
    for (int i = key; i < D * VB; i += ST) xs[i / VB][i % VB] = a.B[0][hoff + (size_t)(i / VB) * D + vb + i % VB];
    load_block(1, 0);
    for (int p = 1; p + 1 < a.P; ++p) {
        const float* Bp = a.B[p] + hoff + (size_t)key * D + vb;
        float acc[VB];
#pragma unroll
        for (int e = 0; e < VB; ++e) acc[e] = Bp[e];
        for (int jc = 0; jc < D; jc += JC) {
            __syncthreads();   // the previous block of M_p (and X_p's update) is done with
            // rows of 32 keys as float4: each warp holds four whole 128-byte row pieces
#pragma unroll
            for (int i = 0; i < NLD; ++i) {
                const int idx = key + ST * i, r = idx >> 3, c = (idx & 7) * 4;
                ms[r][c] = nx[i].x;
                ms[r][c + 1] = nx[i].y;
                ms[r][c + 2] = nx[i].z;
                ms[r][c + 3] = nx[i].w;
            }
            __syncthreads();
            if (jc + JC < D) load_block(p, jc + JC);
            else if (p + 2 < a.P) load_block(p + 1, 0);
#pragma unroll 8
            for (int jj = 0; jj < JC; ++jj) {
                const float m = ms[key][jj];
#pragma unroll
                for (int e = 0; e < VB; ++e) acc[e] = fmaf(m, xs[jc + jj][e], acc[e]);
            }
        }
        __syncthreads();   // every thread has read X_p
        float* Xn = a.X[p + 1] + hoff + (size_t)key * D + vb;
#pragma unroll
        for (int e = 0; e < VB; ++e) {
            xs[key][e] = acc[e];
            Xn[e] = acc[e];
        }
    }
}

}  // namespace

cudaError_t launch_affine_scan(const ScanArgs2& a, cudaStream_t s) {
    if (a.P < 3 || a.P > MAX_SEGS || a.H < 1) return cudaSuccess;
    affine_scan_kernel<<<dim3((unsigned)a.H, D / VB), ST, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
