// simt_fwd.cu -- the staged SIMT forward, one kernel per step of the chunked scan.
//
// Steps (Mamba-3-Lite "SSD Reference", section "ssd_complex_chunkwise -- the
// production scan", restated for the real Mamba-2 recurrence with dt on the input):
//   a1 chunk_cumsum  : dt = softplus(dt_raw + dt_bias), cs = inclusive in-chunk cumsum of dt*A
//                      ("Chunking and the discretized log-decay")
//   a3 chunk_state   : S_c[p][n] = sum_l x[l][p] * dt[l] * exp(cs[Q-1] - cs[l]) * B[l][n]
//                      ("Intra-chunk outputs and per-chunk states", the states einsum)
//   a4 state_passing : carry-in of chunk c+1 = exp(cs_c[Q-1]) * carry-in of c + S_c, from the
//                      initial state ("Inter-chunk propagation -- the fixed contract": the
//                      telescoped exp(CD[z-1] - CD[c]) weights as a left-to-right scan)
//   a5 chunk_scan    : y = (sum_{s<=l} C_l.B_s exp(cs[l]-cs[s]) dt[s] x[s]
//                          + exp(cs[l]) C_l . S_in + D x) * silu(z)
//                      ("Readout, real cast, slice-back": Y_diag + Y_off)
// Arithmetic is fp32 throughout (fp32 inputs are never rounded to tf32/bf16).
// Rows of a chunk tile outside its segment [lo, len) get dt := 0 (decay 1, no input) and
// are not written.
#include "common.cuh"

namespace ssd {

namespace {

// ---------------------------------------------------------------------------- a1
// grid (kmax, H), block Q (a multiple of 32, <= 256)
__global__ void k_chunk_cumsum(Shape sh, const int32_t *__restrict__ hdr, const ChunkInfo *__restrict__ chunks,
                               const float *__restrict__ dt_raw, int64_t sdb, int64_t sdl,
                               const float *__restrict__ A, const float *__restrict__ bias,
                               float *__restrict__ dt_out, float *__restrict__ cs_out) {
    __shared__ float wsum[8];
    const int k = blockIdx.x, h = blockIdx.y, l = threadIdx.x;
    if (k >= hdr[HDR_NCHUNKS]) return;
    const ChunkInfo ci = chunks[k];
    float dt = 0.f;
    if (l >= ci.lo && l < ci.len) {
        float v = dt_raw[(int64_t)ci.b * sdb + (int64_t)(ci.t0 + l) * sdl + h] + (bias ? bias[h] : 0.f);
        dt = softplus_f(v);
    }
    float v = warp_incl_sum(dt * A[h]);
    const int w = l >> 5;
    if ((l & 31) == 31) wsum[w] = v;
    __syncthreads();
    for (int i = 0; i < w; ++i) v += wsum[i];
    const int64_t o = ((int64_t)k * sh.H + h) * sh.Q + l;
    dt_out[o] = dt;
    cs_out[o] = v;
}

// ---------------------------------------------------------------------------- a3
// grid (kmax, H), block 256.  Thread t owns n = t % N and rows p = t / N + (256/N) j.
template <typename T>
__global__ void __launch_bounds__(256)
k_chunk_state(Shape sh, const int32_t *__restrict__ hdr, const ChunkInfo *__restrict__ chunks,
              View3 x, View3 Bm, const float *__restrict__ dtw, const float *__restrict__ csw,
              float *__restrict__ states) {
    constexpr int LT = 16;
    __shared__ float xs[LT][129];
    __shared__ float bs[LT][129];
    __shared__ float w[256];
    const int k = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (k >= hdr[HDR_NCHUNKS]) return;
    const ChunkInfo ci = chunks[k];
    const int P = sh.P, N = sh.N, Q = sh.Q, g = h / sh.hpg;
    const float *dtk = dtw + ((int64_t)k * sh.H + h) * Q;
    const float *csk = csw + ((int64_t)k * sh.H + h) * Q;
    const float clast = csk[Q - 1];
    for (int l = tid; l < Q; l += 256) w[l] = dtk[l] * expf(clast - csk[l]);
    const int np = 256 / N, n = tid % N, p0 = tid / N, J = P / np;
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
    const T *xb = (const T *)x.p + (int64_t)ci.b * x.s0 + (int64_t)h * x.s2;
    const T *bb = (const T *)Bm.p + (int64_t)ci.b * Bm.s0 + (int64_t)g * Bm.s2;
    __syncthreads();
    for (int l0 = 0; l0 < ci.len; l0 += LT) {
        for (int i = tid; i < LT * P; i += 256) {
            int r = i / P, c = i % P;
            int l = l0 + r;
            xs[r][c] = (l < ci.len) ? to_f(xb[(int64_t)(ci.t0 + l) * x.s1 + c]) * w[l] : 0.f;
        }
        for (int i = tid; i < LT * N; i += 256) {
            int r = i / N, c = i % N;
            int l = l0 + r;
            bs[r][c] = (l < ci.len) ? to_f(bb[(int64_t)(ci.t0 + l) * Bm.s1 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < LT; ++r) {
            const float bv = bs[r][n];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < J) acc[j] += xs[r][p0 + np * j] * bv;
        }
        __syncthreads();
    }
    float *out = states + ((int64_t)k * sh.H + h) * P * N;
#pragma unroll
    for (int j = 0; j < 64; ++j)
        if (j < J) out[(int64_t)(p0 + np * j) * N + n] = acc[j];
}

// ---------------------------------------------------------------------------- a4
// Inter-chunk scan: sequential over the chunks of a sequence, parallel over the
// state elements.  grid (S*H, ceil(P*N/1024)), block 256; thread = four consecutive
// elements (p, n) of (sequence, head) (one float4), their running carries in
// registers.  In place: the chunk's local state S_c is replaced by the carry entering
// the chunk, and
//   carry <- exp(lam_c) carry + S_c
// passes the chunk; the carry after the last chunk is the final state.  Per batch of
// 8 chunks, lane j < 8 holds chunk j's decay exp(lam_c) and the warp broadcasts it
// with a shuffle at each step; the batch's 8 loads of S_c are issued ahead of the
// recurrence (they do not depend on the carry), so a warp keeps 8 contiguous
// 512-byte pieces in flight, and all blocks are resident at once.  The chunk's total
// log-decay is lamw[(chunk * H + h) * lam_stride].  With reverse = 1 the chunks are
// visited last to first: that is the backward recursion dS_out[c] = exp(cs_{c+1}[Q-1])
// dS_out[c+1] + dS_loc[c+1] (same affine form, the chunk's own decay), with `init` =
// dfinal and `final_` = dinit (caller tensors: read and written per element, since
// their 16-byte alignment is not guaranteed).  P*N is a multiple of 256.  The chunk tiles are
// fp32, or bf16 (the tensor-core backward's dS: stored rounded, carried in fp32).
__device__ __forceinline__ float4 ld_st4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld_st4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st_st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void st_st4(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

template <typename T>
__global__ void __launch_bounds__(256)
k_state_passing(Shape sh, const int32_t *__restrict__ hdr, const SeqInfo *__restrict__ seqs,
                const float *__restrict__ lamw, int lam_stride, T *__restrict__ states,
                const float *__restrict__ init, float *__restrict__ final_, int reverse) {
    constexpr int CB = 8;   // chunks per batch
    if (hdr[HDR_STATUS] != 0) return;
    const int s = blockIdx.x / sh.H, h = blockIdx.x % sh.H;
    const int PN = sh.P * sh.N;
    const int e = (blockIdx.y * 256 + threadIdx.x) * 4, lane = threadIdx.x & 31;
    if ((blockIdx.y * 256 + (threadIdx.x & ~31)) * 4 >= PN) return;   // whole warp past the end
    const SeqInfo si = seqs[s];
    const int nch = si.nch;   // (a division by the runtime chunk length here measurably slowed the scan)
    const int64_t sbase = ((int64_t)s * sh.H + h) * PN;
    const bool act = e < PN;
    float4 carry = make_float4(0.f, 0.f, 0.f, 0.f);
    if (init != nullptr && act) carry = make_float4(init[sbase + e], init[sbase + e + 1], init[sbase + e + 2], init[sbase + e + 3]);
    auto chunk_of = [&](int pos) { return reverse ? si.chunk0 + nch - 1 - pos : si.chunk0 + pos; };
    auto slot = [&](int pos) { return states + ((int64_t)chunk_of(pos) * sh.H + h) * PN + e; };
    for (int c0 = 0; c0 < nch; c0 += CB) {
        const int nc = min(CB, nch - c0);
        const float mydec = lane < nc ? expf(lamw[((int64_t)chunk_of(c0 + lane) * sh.H + h) * lam_stride]) : 0.f;
        float4 v[CB];
#pragma unroll
        for (int j = 0; j < CB; ++j) v[j] = (act && j < nc) ? ld_st4(slot(c0 + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const float d = __shfl_sync(0xffffffffu, mydec, j);
            if (j < nc) {
                if (act) st_st4(slot(c0 + j), carry);   // carry entering the chunk
                carry.x = fmaf(d, carry.x, v[j].x);
                carry.y = fmaf(d, carry.y, v[j].y);
                carry.z = fmaf(d, carry.z, v[j].z);
                carry.w = fmaf(d, carry.w, v[j].w);
            }
        }
    }
    if (final_ != nullptr && act) {
        final_[sbase + e] = carry.x;
        final_[sbase + e + 1] = carry.y;
        final_[sbase + e + 2] = carry.z;
        final_[sbase + e + 3] = carry.w;
    }
}

// ---------------------------------------------------------------------------- a5
// grid (kmax, H, Q/32), block 256: 32 output rows of one chunk and head.
template <typename T>
__global__ void __launch_bounds__(256)
k_chunk_scan(Shape sh, const int32_t *__restrict__ hdr, const ChunkInfo *__restrict__ chunks,
             View3 x, View3 Bm, View3 Cm, View3 z, const float *__restrict__ D,
             const float *__restrict__ dtw, const float *__restrict__ csw, const float *__restrict__ states,
             MView3 y) {
    constexpr int RT = 32;
    extern __shared__ float smem[];
    const int k = blockIdx.x, h = blockIdx.y, r0 = blockIdx.z * RT, tid = threadIdx.x;
    if (k >= hdr[HDR_NCHUNKS] || hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = chunks[k];
    if (r0 >= ci.len) return;
    const int P = sh.P, N = sh.N, Q = sh.Q, g = h / sh.hpg;
    float *cs = smem;                 // Q
    float *dt = cs + Q;               // Q
    float *Cs = dt + Q;               // RT x (N+1)
    float *Bs = Cs + RT * (N + 1);    // RT x (N+1)
    float *Ms = Bs + RT * (N + 1);    // RT x Q
    float *xs = Ms + RT * Q;          // RT x (P+1)
    float *Ss = xs + RT * (P + 1);    // P x (N+1): the carried state entering the chunk
    const float *dtk = dtw + ((int64_t)k * sh.H + h) * Q;
    const float *csk = csw + ((int64_t)k * sh.H + h) * Q;
    for (int l = tid; l < Q; l += 256) { cs[l] = csk[l]; dt[l] = dtk[l]; }
    const T *xb = (const T *)x.p + (int64_t)ci.b * x.s0 + (int64_t)h * x.s2;
    const T *bb = (const T *)Bm.p + (int64_t)ci.b * Bm.s0 + (int64_t)g * Bm.s2;
    const T *cb = (const T *)Cm.p + (int64_t)ci.b * Cm.s0 + (int64_t)g * Cm.s2;
    for (int i = tid; i < RT * N; i += 256) {
        int r = i / N, c = i % N, l = r0 + r;
        Cs[r * (N + 1) + c] = (l < ci.len) ? to_f(cb[(int64_t)(ci.t0 + l) * Cm.s1 + c]) : 0.f;
    }
    {   // S_in staged once (coalesced), so the Y_off dot products read shared memory
        const float *sk = states + ((int64_t)k * sh.H + h) * P * N;
        for (int i = tid; i < P * N; i += 256) Ss[(i / N) * (N + 1) + i % N] = sk[i];
    }
    __syncthreads();
    // M[l][s] = (C_l . B_s) exp(cs[l] - cs[s]) dt[s] for s <= l, over s-tiles up to this row tile
    for (int s0 = 0; s0 <= r0; s0 += RT) {
        for (int i = tid; i < RT * N; i += 256) {
            int r = i / N, c = i % N, s = s0 + r;
            Bs[r * (N + 1) + c] = (s < ci.len) ? to_f(bb[(int64_t)(ci.t0 + s) * Bm.s1 + c]) : 0.f;
        }
        __syncthreads();
        for (int i = tid; i < RT * RT; i += 256) {
            int r = i / RT, c = i % RT;
            int l = r0 + r, s = s0 + c;
            float v = 0.f;
            if (s <= l && s < ci.len) {
                float acc = 0.f;
                for (int n = 0; n < N; ++n) acc += Cs[r * (N + 1) + n] * Bs[c * (N + 1) + n];
                v = acc * expf(cs[l] - cs[s]) * dt[s];
            }
            Ms[r * Q + s] = v;
        }
        __syncthreads();
    }
    // Y_diag[l][p] = sum_s M[l][s] x[s][p]
    const int pr = 256 / P, p = tid % P, lr = tid / P, J = RT / pr;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int s0 = 0; s0 <= r0; s0 += RT) {
        for (int i = tid; i < RT * P; i += 256) {
            int r = i / P, c = i % P, s = s0 + r;
            xs[r * (P + 1) + c] = (s < ci.len) ? to_f(xb[(int64_t)(ci.t0 + s) * x.s1 + c]) : 0.f;
        }
        __syncthreads();
        for (int c = 0; c < RT; ++c) {
            const float xv = xs[c * (P + 1) + p];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < J) acc[j] += Ms[(lr + pr * j) * Q + s0 + c] * xv;
        }
        __syncthreads();
    }
    // Y_off[l][p] = exp(cs[l]) sum_n C[l][n] S_in[p][n]; then D skip, gate, store
    const float *sin = Ss + p * (N + 1);
    const float Dh = D ? D[h] : 0.f;
    T *yb = (T *)y.p + (int64_t)ci.b * y.s0 + (int64_t)h * y.s2;
    const T *zb = z.p ? (const T *)z.p + (int64_t)ci.b * z.s0 + (int64_t)h * z.s2 : nullptr;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (j >= J) continue;
        const int r = lr + pr * j, l = r0 + r;
        if (l < ci.lo || l >= ci.len) continue;
        float yo = 0.f;
        for (int n = 0; n < N; ++n) yo += Cs[r * (N + 1) + n] * sin[n];
        const int64_t tok = (int64_t)(ci.t0 + l);
        float v = acc[j] + expf(cs[l]) * yo + Dh * to_f(xb[tok * x.s1 + p]);
        if (zb) {
            float zz = to_f(zb[tok * z.s1 + p]);
            v *= zz * sigmoid_f(zz);
        }
        yb[tok * y.s1 + p] = from_f<T>(v);
    }
}

}  // namespace

// ---------------------------------------------------------------------------- launchers
cudaError_t launch_chunk_cumsum(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks,
                                const float *dt_raw, int64_t sdb, int64_t sdl, const float *A,
                                const float *bias, float *dt_out, float *cs_out, cudaStream_t st) {
    k_chunk_cumsum<<<dim3(sh.kmax, sh.H), sh.Q, 0, st>>>(sh, hdr, chunks, dt_raw, sdb, sdl, A, bias, dt_out, cs_out);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_chunk_state(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 x,
                               View3 Bm, const float *dtw, const float *csw, float *states, cudaStream_t st) {
    k_chunk_state<T><<<dim3(sh.kmax, sh.H), 256, 0, st>>>(sh, hdr, chunks, x, Bm, dtw, csw, states);
    return cudaGetLastError();
}

cudaError_t launch_state_passing(const Shape &sh, const int32_t *hdr, const SeqInfo *seqs, const float *lamw,
                                 int lam_stride, float *states, const float *init, float *final_, int reverse,
                                 cudaStream_t st) {
    const int PN = sh.P * sh.N;
    if (sh.S * sh.H == 0) return cudaSuccess;
    if (PN % 256 != 0) return cudaErrorInvalidValue;   // float4 per thread, whole warps
    k_state_passing<float><<<dim3(sh.S * sh.H, (PN + 1023) / 1024), 256, 0, st>>>(sh, hdr, seqs, lamw, lam_stride,
                                                                                  states, init, final_, reverse);
    return cudaGetLastError();
}
cudaError_t launch_state_passing(const Shape &sh, const int32_t *hdr, const SeqInfo *seqs, const float *lamw,
                                 int lam_stride, __nv_bfloat16 *states, const float *init, float *final_, int reverse,
                                 cudaStream_t st) {
    const int PN = sh.P * sh.N;
    if (sh.S * sh.H == 0) return cudaSuccess;
    if (PN % 256 != 0) return cudaErrorInvalidValue;
    k_state_passing<__nv_bfloat16><<<dim3(sh.S * sh.H, (PN + 1023) / 1024), 256, 0, st>>>(
        sh, hdr, seqs, lamw, lam_stride, states, init, final_, reverse);
    return cudaGetLastError();
}

size_t chunk_scan_smem(const Shape &sh) {
    return sizeof(float) * (size_t)(2 * sh.Q + 2 * 32 * (sh.N + 1) + 32 * sh.Q + 32 * (sh.P + 1) +
                                    sh.P * (sh.N + 1));
}

template <typename T>
cudaError_t launch_chunk_scan(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 x, View3 Bm,
                              View3 Cm, View3 z, const float *D, const float *dtw, const float *csw,
                              const float *states, MView3 y, cudaStream_t st) {
    const size_t smem = chunk_scan_smem(sh);
    static int attr_done[64] = {0};
    cudaError_t e = ensure_smem_attr(k_chunk_scan<T>, (int)smem, attr_done);
    if (e != cudaSuccess) return e;
    k_chunk_scan<T><<<dim3(sh.kmax, sh.H, sh.Q / 32), 256, smem, st>>>(sh, hdr, chunks, x, Bm, Cm, z, D, dtw, csw,
                                                                        states, y);
    return cudaGetLastError();
}

template cudaError_t launch_chunk_state<float>(const Shape &, const int32_t *, const ChunkInfo *, View3, View3,
                                               const float *, const float *, float *, cudaStream_t);
template cudaError_t launch_chunk_state<__nv_bfloat16>(const Shape &, const int32_t *, const ChunkInfo *, View3,
                                                       View3, const float *, const float *, float *, cudaStream_t);
template cudaError_t launch_chunk_scan<float>(const Shape &, const int32_t *, const ChunkInfo *, View3, View3, View3,
                                              View3, const float *, const float *, const float *, const float *,
                                              MView3, cudaStream_t);
template cudaError_t launch_chunk_scan<__nv_bfloat16>(const Shape &, const int32_t *, const ChunkInfo *, View3, View3,
                                                      View3, View3, const float *, const float *, const float *,
                                                      const float *, MView3, cudaStream_t);

}  // namespace ssd
