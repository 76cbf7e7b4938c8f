// Layout shared by the chunk-preparation kernel (producer) and the tcgen05
// chunk-recurrence kernel (consumer): one record per (chunk, head) holding
// that chunk's operand tiles as the byte image of the consumer's shared
// memory, so one bulk copy moves a whole record.
#pragma once

#include <cuda.h>

#include "kda_common.cuh"

namespace kda {

constexpr int CHUNK_T = 64;  // tokens per chunk
constexpr int MAX_SEGS = 16;  // pseudo-sequences of one segmented recurrence launch
constexpr int32_t SEG_IDENTITY = 1, SEG_LINEAR = 2, SEG_NO_OUTPUT = 4;

// Record layout (bytes).  Every tile is fp16, K-major with the 128-byte
// swizzle, and starts on a 1024-byte boundary.  fp16 rather than bf16: every
// operand here is bounded (unit-norm keys and queries scaled by decays <= 1,
// values of order 1-10, the UT-solve products), so the 3 extra mantissa bits
// cut the operand rounding error 8x at the same tensor-core rate.
// W and Q+ are interleaved panel by panel (W keys 0-63, Q+ keys 0-63, W keys
// 64-127, Q+ keys 64-127), so that [W; Q+] is one 128-row operand with the
// 64-row W and Q+ panels REC_PANEL bytes apart.
constexpr int REC_W = 0;          // W     [64 tok rows][128 key]  2 panels x 64 rows x 128 B, stride REC_PANEL
constexpr int REC_Q = 8192;       // Q+    [64 tok rows][128 key]  2 panels, stride REC_PANEL
constexpr int REC_PANEL = 16384;  // panel stride of W and Q+
constexpr int REC_KT = 32768;     // Kt^T  [128 key rows][64 tok]  1 panel x 128 rows
constexpr int REC_UT = 49152;     // U0^T  [128 val rows][64 tok]  1 panel x 128 rows
constexpr int REC_P = 65536;      // P     lower triangle [64 r rows][64 s]: see p_chunk
constexpr int REC_P_BYTES = 288 * 16;
constexpr int REC_DECAY = REC_P + REC_P_BYTES;  // decay [128] fp32 = e^{G_last}
constexpr int REC_BYTES = REC_DECAY + 512;

// P (s <= r) is stored as its lower triangle of 16-byte chunks: row r holds the
// 8-column chunks c <= r / 8 (every element past them is zero), rows in order,
// 288 chunks in all; p_chunk is the index of chunk c of row r.  The recurrence
// expands it into a swizzled tile in shared memory.
__host__ __device__ constexpr int p_chunk(int r, int c) {
    return 4 * (r >> 3) * ((r >> 3) + 1) + (r & 7) * ((r >> 3) + 1) + c;
}
static_assert(p_chunk(63, 7) == 287 && p_chunk(8, 0) == 8 && p_chunk(16, 0) == 24, "P chunk numbering");

// Byte offset of 16-bit element (row, k) in a K-major tile with the 128-byte
// swizzle: 64 elements of K per 128-byte row, panels of `rows` rows for each
// further 64 elements of K, 8-row groups 1024 bytes apart.
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int k, int rows) {
    const int panel = k >> 6, kk = k & 63;
    const int chunk = kk >> 3, within = kk & 7;
    return (uint32_t)(panel * rows * 128 + row * 128 + (((chunk ^ (row & 7)) & 7) << 4) + within * 2);
}

// Inputs of the chunk preparation (pre-stage fused in): the raw bf16
// projections and the layer parameters.
struct PrepArgs {
    const void *q, *k, *v, *z, *b;  // bf16 [T][H*128]; b [T][H]
    const void* ring_in;            // bf16 [n][3][3][H*128] or NULL (zero)
    const float *conv_w, *A_log, *dt_bias;
    float lb, l2_eps, q_scale;
    const ChunkDesc* chunks;
    int32_t n_chunks, H;
    int64_t T;                      // total tokens
    void* records;                  // [n_chunks][H][REC_BYTES]
    int32_t* status;                // workspace error word
    // NULL: each CTA takes a fixed contiguous range of items.  Otherwise a
    // zeroed counter from which CTAs take batches of `batch` items in turn
    // (1 <= batch <= PREP_BATCH), so that CTAs starting late (other kernels
    // hold their SMs) take fewer.
    int32_t* work_counter;
    int32_t batch;
    // Limit of the waits between the kernel's two warp groups, in ns (0: the
    // default 2 s).  The drain after a timeout always uses the default.
    uint64_t wait_limit_ns;
    // set by launch_chunk_prep: TMA descriptors of q, k, v as [T][H*128] bf16
    // with a 67-row box (a chunk and the three rows before it) and a 64-row box
    CUtensorMap map67[3], map64[3];
    int32_t gate_kind;              // KDA_GATE_BOUNDED or KDA_GATE_SOFTPLUS
};
constexpr int PREP_BATCH = 4;        // most items per take from PrepArgs::work_counter
// PrepArgs::wait_limit_ns from the parameters' test hook (0: the default)
inline uint64_t prep_wait_limit_ns(const kda_params* p) { return (uint64_t)p->wait_limit_us * 1000ull; }
// max_ctas > 0 caps the persistent grid (for a launch that shares the GPU).
cudaError_t launch_chunk_prep(const PrepArgs& a, cudaStream_t s, int max_ctas = 0);
size_t chunk_prep_smem_bytes();

struct ChunkRecArgs {
    const void* records;
    const float* S_in;
    float* S_out;
    const void* gout;          // bf16 [T][H*128] output-gate logits
    const float* norm_w;       // [128]
    void* o;                   // bf16 [T][H*128]
    float eps;                 // RMSNorm eps
    const int64_t* cu;         // [n+1] token offsets
    const int64_t* chunk_off;  // [n+1] first chunk of each sequence
    const int32_t* seq_order;  // [n] sequences by decreasing length (CTA order), or NULL
    int32_t* status;
    int32_t n_seqs, H;
    // Segments of one sequence (n_segs > 0; then cu, chunk_off, seq_order and
    // S_in / S_out are not used): CTA (n, h) runs tokens [seg_t0[n], seg_t1[n])
    // whose first chunk is seg_c0[n], from the state seg_S_in[n] (NULL: zero),
    // writing its final state to seg_S_out[n] (NULL: not written); states are
    // [H][128][128].  seg_mode[n] bits: SEG_IDENTITY starts from the identity
    // instead, SEG_LINEAR runs the linear part of the chunk step only (U0 read
    // as zero), SEG_NO_OUTPUT writes no output rows.
    int32_t n_segs;
    int64_t seg_t0[MAX_SEGS], seg_t1[MAX_SEGS], seg_c0[MAX_SEGS];
    const float* seg_S_in[MAX_SEGS];
    float* seg_S_out[MAX_SEGS];
    int32_t seg_mode[MAX_SEGS];
};
cudaError_t launch_chunk_recurrence(const ChunkRecArgs& a, cudaStream_t s);

// Affine composition of segment maps, column block by column block:
// X_{p+1} = M_p X_p + B_p for p = 1 .. P - 2, with X_1 = B_0 (all [H][128][128]
// fp32, key-major rows; M_p maps keys to keys).  X[p] receives X_p.
struct ScanArgs2 {
    const float* B[MAX_SEGS];
    const float* M[MAX_SEGS];
    float* X[MAX_SEGS];
    int32_t P, H;
};
cudaError_t launch_affine_scan(const ScanArgs2& a, cudaStream_t s);

}  // namespace kda
