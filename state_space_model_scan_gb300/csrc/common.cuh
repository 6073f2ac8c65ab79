// common.cuh -- types and device helpers shared by the libssd kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/ssd.h"

namespace ssd {

// ---------------------------------------------------------------------------
// Workspace header: 64 int32 words at offset 0 of every workspace.
enum HeaderWord {
    HDR_NCHUNKS = 0,   // number of chunks in the chunk list
    HDR_NUNITS = 1,    // number of work units (fused path)
    HDR_NSEQS = 2,
    HDR_STATUS = 3,    // device-side ssd_status (first error wins)
    HDR_TICKET = 4,    // fused path: next unit ticket
    HDR_MAXSEG = 5,    // fused path: largest number of units in one sequence
    HDR_TICKET2 = 6,   // tensor-core backward: next work item of the gradient kernel
    HDR_PROBE = 7,     // ssd_selftest_bounded_wait: the flag nothing sets
    HDR_WORDS = 64
};

// The chunk grid runs over each batch row's token axis: physical chunk c of a row holds
// tokens [cQ, (c+1)Q).  With packed sequences (cu_seqlens) a chunk may hold parts of
// several sequences; each part (a segment) is processed as one chunk tile: the Q rows
// from the chunk's first token, of which rows [lo, len) belong to the segment.  Rows
// outside get dt := 0 (decay 1, no input) and are never written, which is the
// sequence mask seq_idx[l] == seq_idx[s] of the intra-chunk matrix.

// One sequence: tokens [t0, t0 + len) of batch row b; its nch chunk tiles start at chunk0.
struct SeqInfo {
    int32_t b, t0, len, chunk0;
    int32_t nch, pad0, pad1, pad2;
};
// Number of chunk tiles of a sequence: the physical chunks its tokens touch.
__host__ __device__ __forceinline__ int seq_nchunks(int t0, int len, int Q) {
    return len > 0 ? (t0 + len + Q - 1) / Q - t0 / Q : 0;
}
// One chunk tile: the segment of one sequence in the physical chunk starting at token t0
// of batch row b; rows [lo, len) of the tile belong to it (0 <= lo < len <= Q).  16 bytes
// (the gradient kernel keeps two of these live at its register limit).
struct ChunkInfo {
    int32_t seq, b, t0;
    int16_t len, lo;
};
// One work unit of the fused forward: segment j (`nchunk` consecutive chunk tiles) of one
// sequence; t0 = first token of its first tile's physical chunk, rows [lo, len) from t0
// belong to the sequence (lo > 0 only for a sequence starting inside its first chunk).
struct UnitInfo {
    int32_t seq, b, t0, len;          // rows [lo, len) from token t0 of row b
    int32_t nchunk, prev, j;          // prev: index of unit (seq, j-1) or -1
    int16_t last, lo;                 // last: j is the sequence's final unit
};

// Shape of one call, as the kernels see it.
struct Shape {
    int B, L, H, P, G, N, S;
    int Nio;          // dstate of the caller's B, C, dB, dC (the tensor-core path computes N = 128
                      // and reads a dstate-64 problem as its zero-extended half: TMA fills past Nio)
    int Q;            // internal chunk length
    int hpg;          // H / G
    int kmax;         // capacity of the chunk list
    int umax;         // capacity of the unit list
    int R;            // most chunks per unit (fused path)
    int useg_num, useg_den;   // units per chunk of a sequence (>= 1/R): see the metadata kernel
};

// Arguments of the tensor-core backward kernels (bwd_tc.cu).
struct BwdTcArgs {
    const void *x, *Bp, *Cp;
    const int64_t *sx, *sb, *sc;
    const float *dt_raw;
    int64_t sdb, sdl;
    const float *A, *D, *bias;
    const void *dy, *z;
    const int64_t *sdy, *sz;
    void *dx, *dz;
    const int64_t *sdx, *sdz;
    float *ddt;
    int64_t sddb, sddl;
    const __nv_bfloat16 *states;   // carried state entering each chunk: 16 KB swizzled tile per (chunk, head)
    __nv_bfloat16 *dS;    // [chunk][H][P][N] bf16: local dS from the dstates kernel, then (in place) the
                          // gradient of the state leaving every chunk (carried in fp32 by the reverse scan)
    float *chunk_lam, *dBh, *dCh, *partials;
    int hs;                         // heads per CTA of the gradient kernel (divides H/G)
    int hs_ds;                      // heads per CTA of the dstates kernel (divides H/G)
    // gradient kernel work items: pairs (chunk, group) below k_pairs in H/G/hs subsets of hs
    // heads, the rest in nsub_tail subsets whose dB/dC shares (tpart) are summed afterwards
    int k_pairs, nsub_tail, n_items, grid;   // grid: persistent CTAs (one per SM at most)
    float *tpart;                   // [tail item][2][Q][N] fp32
    void *dB, *dC;                  // final dB/dC (written directly when hs == H/G)
    float *dA, *dD, *dbias;         // per-head gradients (sums of the per-(chunk, head) partials)
    const int64_t *sdB, *sdC;
};

// Strided views (element strides of the three outer dims; innermost stride 1).
struct View3 {
    const void *p;
    int64_t s0, s1, s2;
};
struct MView3 {
    void *p;
    int64_t s0, s1, s2;
};

// Raises a kernel's dynamic shared memory limit when a launch needs more than
// was set before on this device (state: the largest limit set per device < 64).
template <typename K>
inline cudaError_t ensure_smem_attr(K kernel, int bytes, int *set_bytes /* [64] */) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (set_bytes[dev & 63] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) set_bytes[dev & 63] = bytes;
    return e;
}

__device__ __forceinline__ void set_status(int32_t *hdr, int32_t code) {
    atomicCAS(&hdr[HDR_STATUS], 0, code);
}

// ---------------------------------------------------------------------------
// dtype helpers
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// softplus in fp32: log(1 + exp(v)); for v > 20 the exact value differs from v
// by less than 2.1e-9 relative, so v is returned there.
__device__ __forceinline__ float softplus_f(float v) { return v > 20.f ? v : log1pf(expf(v)); }
__device__ __forceinline__ float sigmoid_f(float v) { return 1.f / (1.f + expf(-v)); }

// Inclusive warp prefix sum.
__device__ __forceinline__ float warp_incl_sum(float v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float t = __shfl_up_sync(0xffffffffu, v, o);
        if ((threadIdx.x & 31) >= o) v += t;
    }
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace ssd
