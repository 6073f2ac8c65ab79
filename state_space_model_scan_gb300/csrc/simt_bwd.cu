// simt_bwd.cu -- the staged SIMT backward of the chunked SSD scan.
//
// Recompute-based, as the Mamba-3-Lite "SSD Reference" page's section "6. The
// autograd backward contract" prescribes for its kernel (re-run the forward math,
// inject the true upstream gradients): the forward's dt, cs and carry-in states
// are recomputed by the forward's own a1/a3/a4 kernels, then
//   bwd_dstates      : dS_loc[c][p][n] = sum_l exp(cs[l]) dyp[l][p] C[l][n]
//   state_passing    : reverse scan  dS_out[c] = exp(cs_{c+1}[Q-1]) dS_out[c+1] + dS_loc[c+1],
//                      dS_out[last] = dfinal, dinit = exp(cs_0[Q-1]) dS_out[0] + dS_loc[0]
//   bwd_chunk        : per chunk and head, every gradient of the chunk's closed form:
//     with E[l][s] = exp(cs[l]-cs[s]) (s <= l), CB = C B^T, dM = dyp x^T, M = E dt_s CB,
//     w_s = dt[s] exp(cs[Q-1]-cs[s]), u[s][p] = sum_n B[s][n] dS_out[p][n]:
//       dx[s]   = sum_l M[l][s] dyp[l] + w_s u[s] + D dyp[s]
//       dB[s]   = sum_l E dt_s dM[l][s] C[l]      + w_s x[s]^T dS_out
//       dC[l]   = sum_s E dt_s dM[l][s] B[s]      + exp(cs[l]) dyp[l]^T S_in
//       ddt[s] (direct) = sum_l E CB dM[l][s]     + exp(cs[Q-1]-cs[s]) x[s].u[s]
//       dcs[i]  = sum_{s<i} T1[i][s] - sum_{l>i} T1[l][i] + T2[i] - T4[i] + [i = Q-1](T3 + sum_s T4[s])
//         T1 = M o dM, T2[l] = dyp[l].Y_off[l], T4[s] = w_s x[s].u[s], T3 = exp(cs[Q-1]) <S_in, dS_out>
//         (the diagonal s = l of T1 does not depend on cs: its row and column terms cancel exactly
//         and are left out of both sums)
//       da[u] = sum_{i>=u} dcs[i] = sum_{i>=u} (dcs[i] without T4) + T3 + sum_{s<u} T4[s], formed
//         that way (a reverse scan and a forward exclusive scan), so no large term cancels against
//         itself;  ddt = ddt_direct + A da;  dA += sum dt da
//       ddt_raw = ddt * sigmoid(dt_raw + dt_bias);  dz = dy ypre silu'(z)
//   reductions       : dB/dC over the heads of a group, dA/dD/ddt_bias over chunks, in a
//                      fixed order (bitwise reproducible; no atomics).
// Chunk lengths QS = 32 or 64 (a template argument): one chunk row per 256 / QS threads.
#include "common.cuh"

namespace ssd {

namespace {

// sum over the NP consecutive lanes that share a chunk row (fixed order)
template <int NP>
__device__ __forceinline__ float sum_parts(float v) {
#pragma unroll
    for (int o = 1; o < NP; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ bwd_dstates
// grid (kmax, H), block 256; mapping as the forward chunk_state kernel.
template <typename T, int QS>
__global__ void __launch_bounds__(256)
k_bwd_dstates(Shape sh, const int32_t *__restrict__ hdr, const ChunkInfo *__restrict__ chunks,
              View3 dy, View3 z, View3 Cm, const float *__restrict__ csw, float *__restrict__ dstates) {
    constexpr int LT = 16;
    __shared__ float ds[LT][129];
    __shared__ float cs_[LT][129];
    __shared__ float w[QS];
    const int k = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (k >= hdr[HDR_NCHUNKS] || hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = chunks[k];
    const int P = sh.P, N = sh.N, g = h / sh.hpg;
    const float *csk = csw + ((int64_t)k * sh.H + h) * QS;
    if (tid < QS) w[tid] = expf(csk[tid]);
    const int np = 256 / N, n = tid % N, p0 = tid / N, J = P / np;
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
    const T *dyb = (const T *)dy.p + (int64_t)ci.b * dy.s0 + (int64_t)h * dy.s2;
    const T *zb = z.p ? (const T *)z.p + (int64_t)ci.b * z.s0 + (int64_t)h * z.s2 : nullptr;
    const T *cb = (const T *)Cm.p + (int64_t)ci.b * Cm.s0 + (int64_t)g * Cm.s2;
    __syncthreads();
    for (int l0 = 0; l0 < ci.len; l0 += LT) {
        for (int i = tid; i < LT * P; i += 256) {
            int r = i / P, c = i % P, l = l0 + r;
            float v = 0.f;
            if (l >= ci.lo && l < ci.len) {
                int64_t tok = ci.t0 + l;
                v = to_f(dyb[tok * dy.s1 + c]);
                if (zb) { float zz = to_f(zb[tok * z.s1 + c]); v *= zz * sigmoid_f(zz); }
                v *= w[l];
            }
            ds[r][c] = v;
        }
        for (int i = tid; i < LT * N; i += 256) {
            int r = i / N, c = i % N, l = l0 + r;
            cs_[r][c] = (l >= ci.lo && l < ci.len) ? to_f(cb[(int64_t)(ci.t0 + l) * Cm.s1 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < LT; ++r) {
            const float cv = cs_[r][n];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < J) acc[j] += ds[r][p0 + np * j] * cv;
        }
        __syncthreads();
    }
    float *out = dstates + ((int64_t)k * sh.H + h) * P * N;
#pragma unroll
    for (int j = 0; j < 64; ++j)
        if (j < J) out[(int64_t)(p0 + np * j) * N + n] = acc[j];
}

// ------------------------------------------------------------------ bwd_chunk
// grid (kmax, H), block 256 = QS rows x NP threads.  Dynamic shared memory.
template <typename T, int QS>
__global__ void __launch_bounds__(256)
k_bwd_chunk(Shape sh, const int32_t *__restrict__ hdr, const ChunkInfo *__restrict__ chunks,
            View3 x, View3 Bm, View3 Cm, View3 z, View3 dy, const float *__restrict__ dt_raw, int64_t sdb,
            int64_t sdl, const float *__restrict__ A, const float *__restrict__ D, const float *__restrict__ bias,
            const float *__restrict__ dtw, const float *__restrict__ csw, const float *__restrict__ states,
            const float *__restrict__ dstates, MView3 dx, MView3 dz, float *__restrict__ ddt, int64_t sddb,
            int64_t sddl, float *__restrict__ dBh, float *__restrict__ dCh, float *__restrict__ partials,
            int stage_states) {
    constexpr int NP = 256 / QS;   // threads per chunk row
    constexpr int NQ = QS / 32;    // 32-position blocks of the per-position scalars
    extern __shared__ float sm[];
    const int k = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (k >= hdr[HDR_NCHUNKS] || hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = chunks[k];
    const int P = sh.P, N = sh.N, g = h / sh.hpg;
    const int P1 = P + 1, N1 = N + 1, Q1 = QS + 1;
    float *cs = sm;                  // QS
    float *dt = cs + QS;             // QS
    float *wst = dt + QS;            // QS
    float *vec = wst + QS;           // 8 x QS per-row scalars
    float *xs = vec + 8 * QS;        // QS x P1
    float *dys = xs + QS * P1;       // QS x P1  (dyp = dy * silu(z))
    float *Bs = dys + QS * P1;       // QS x N1
    float *Cs = Bs + QS * N1;        // QS x N1
    float *Mm = Cs + QS * N1;        // QS x Q1  CB, then M
    float *Em = Mm + QS * Q1;        // QS x Q1  dM, then E dt dM
    float *Tm = Em + QS * Q1;        // QS x Q1  E CB dM
    float *Dso = Tm + QS * Q1;       // P x N1   dS_out, S_in (when stage_states: the per-row dot
    float *Sis = Dso + P * N1;       //          products then read shared memory, not global)
    float *rowXU = vec, *rowT2 = vec + QS, *rowD = vec + 2 * QS;

    const float *dtk = dtw + ((int64_t)k * sh.H + h) * QS;
    const float *csk = csw + ((int64_t)k * sh.H + h) * QS;
    if (tid < QS) { cs[tid] = csk[tid]; dt[tid] = dtk[tid]; }
    __syncthreads();
    const float clast = cs[QS - 1];
    if (tid < QS) wst[tid] = dt[tid] * expf(clast - cs[tid]);
    const T *xb = (const T *)x.p + (int64_t)ci.b * x.s0 + (int64_t)h * x.s2;
    const T *bb = (const T *)Bm.p + (int64_t)ci.b * Bm.s0 + (int64_t)g * Bm.s2;
    const T *cb = (const T *)Cm.p + (int64_t)ci.b * Cm.s0 + (int64_t)g * Cm.s2;
    const T *zb = z.p ? (const T *)z.p + (int64_t)ci.b * z.s0 + (int64_t)h * z.s2 : nullptr;
    const T *dyb = (const T *)dy.p + (int64_t)ci.b * dy.s0 + (int64_t)h * dy.s2;
    for (int i = tid; i < QS * P; i += 256) {
        int r = i / P, c = i % P;
        float xv = 0.f, dv = 0.f;
        if (r >= ci.lo && r < ci.len) {
            int64_t tok = ci.t0 + r;
            xv = to_f(xb[tok * x.s1 + c]);
            dv = to_f(dyb[tok * dy.s1 + c]);
            if (zb) { float zz = to_f(zb[tok * z.s1 + c]); dv *= zz * sigmoid_f(zz); }
        }
        xs[r * P1 + c] = xv;
        dys[r * P1 + c] = dv;
    }
    for (int i = tid; i < QS * N; i += 256) {
        int r = i / N, c = i % N;
        bool in = r >= ci.lo && r < ci.len;
        Bs[r * N1 + c] = in ? to_f(bb[(int64_t)(ci.t0 + r) * Bm.s1 + c]) : 0.f;
        Cs[r * N1 + c] = in ? to_f(cb[(int64_t)(ci.t0 + r) * Cm.s1 + c]) : 0.f;
    }
    const float *dsg = dstates + ((int64_t)k * sh.H + h) * P * N;
    const float *sig = states + ((int64_t)k * sh.H + h) * P * N;
    if (stage_states) {
        for (int i = tid; i < P * N; i += 256) {
            Dso[(i / N) * N1 + i % N] = dsg[i];
            Sis[(i / N) * N1 + i % N] = sig[i];
        }
    }
    __syncthreads();
    // CB[l][s], dM[l][s]
    for (int i = tid; i < QS * QS; i += 256) {
        int l = i / QS, s = i % QS;
        float a = 0.f, b = 0.f;
        if (s <= l) {
            for (int n = 0; n < N; ++n) a += Cs[l * N1 + n] * Bs[s * N1 + n];
            for (int p = 0; p < P; ++p) b += dys[l * P1 + p] * xs[s * P1 + p];
        }
        const float E = (s <= l) ? expf(cs[l] - cs[s]) : 0.f;
        Mm[l * Q1 + s] = E * dt[s] * a;
        Em[l * Q1 + s] = E * dt[s] * b;
        Tm[l * Q1 + s] = E * a * b;
    }
    __syncthreads();

    const int r = tid / NP, part = tid % NP;     // row r, part `part` of its columns
    const float *dso = stage_states ? Dso : dsg;
    const float *sin = stage_states ? Sis : sig;
    const int ld = stage_states ? N1 : N;   // row stride of dso / sin
    const float Dh = D ? D[h] : 0.f;
    const bool live = r >= ci.lo && r < ci.len;
    const int64_t tok = (int64_t)ci.t0 + r;
    // dx[r][p] and x.u row sums
    {
        float xu = 0.f;
        for (int p = part; p < P; p += NP) {
            float a = 0.f;
            for (int l = r; l < QS; ++l) a += Mm[l * Q1 + r] * dys[l * P1 + p];
            float u = 0.f;
            const float *drow = dso + p * ld;
            for (int n = 0; n < N; ++n) u += Bs[r * N1 + n] * drow[n];
            xu += xs[r * P1 + p] * u;
            if (live) {
                T *o = (T *)dx.p + (int64_t)ci.b * dx.s0 + tok * dx.s1 + (int64_t)h * dx.s2;
                o[p] = from_f<T>(a + wst[r] * u + Dh * dys[r * P1 + p]);
            }
        }
        xu = sum_parts<NP>(xu);
        if (part == 0) rowXU[r] = xu;
    }
    // dB (this head) [r][n]
    {
        float *o = dBh + (((int64_t)k * sh.H + h) * QS + r) * N;
        for (int n = part; n < N; n += NP) {
            float a = 0.f;
            for (int l = r; l < QS; ++l) a += Em[l * Q1 + r] * Cs[l * N1 + n];
            float b = 0.f;
            for (int p = 0; p < P; ++p) b += xs[r * P1 + p] * dso[p * ld + n];
            o[n] = a + wst[r] * b;
        }
    }
    // dC (this head) [r][n]
    {
        float *o = dCh + (((int64_t)k * sh.H + h) * QS + r) * N;
        const float er = expf(cs[r]);
        for (int n = part; n < N; n += NP) {
            float a = 0.f;
            for (int s = 0; s <= r; ++s) a += Em[r * Q1 + s] * Bs[s * N1 + n];
            float b = 0.f;
            for (int p = 0; p < P; ++p) b += dys[r * P1 + p] * sin[p * ld + n];
            o[n] = a + er * b;
        }
    }
    // ypre, dz, T2, dD row sums
    {
        const float er = expf(cs[r]);
        float t2 = 0.f, dd = 0.f;
        for (int p = part; p < P; p += NP) {
            float yd = 0.f;
            for (int s = 0; s <= r; ++s) yd += Mm[r * Q1 + s] * xs[s * P1 + p];
            float yb = 0.f;
            const float *srow = sin + p * ld;
            for (int n = 0; n < N; ++n) yb += Cs[r * N1 + n] * srow[n];
            const float yo = er * yb;
            t2 += dys[r * P1 + p] * yo;
            dd += dys[r * P1 + p] * xs[r * P1 + p];
            if (zb && live) {
                const float ypre = yd + yo + Dh * xs[r * P1 + p];
                const float zz = to_f(zb[tok * z.s1 + p]);
                const float sg = sigmoid_f(zz);
                const float dyv = to_f(dyb[tok * dy.s1 + p]);
                T *o = (T *)dz.p + (int64_t)ci.b * dz.s0 + tok * dz.s1 + (int64_t)h * dz.s2;
                o[p] = from_f<T>(dyv * ypre * sg * (1.f + zz * (1.f - sg)));
            }
        }
        t2 = sum_parts<NP>(t2);
        dd = sum_parts<NP>(dd);
        if (part == 0) { rowT2[r] = t2; rowD[r] = dd; }
    }
    __syncthreads();
    // T3 = exp(cs[Q-1]) <S_in, dS_out>: fixed-order block reduction
    float t3p = 0.f;
    for (int i = tid; i < P * N; i += 256) t3p += sin[(i / N) * ld + i % N] * dso[(i / N) * ld + i % N];
    t3p = warp_sum(t3p);
    float *red = vec + 3 * QS;    // 8 warp partials
    if ((tid & 31) == 0) red[tid >> 5] = t3p;
    __syncthreads();
    if (tid < 32) {
        // per-position scalars: thread i handles positions i + 32 q (q < NQ)
        float T3 = 0.f;
        for (int w = 0; w < 8; ++w) T3 += red[w];
        T3 *= expf(clast);
        float dcs[NQ], t4[NQ], ddir[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int i = tid + 32 * q;
            float rowT1 = 0.f, colTm = 0.f;
            for (int s = 0; s < i; ++s) rowT1 += dt[s] * Tm[i * Q1 + s];
            for (int l = i + 1; l < QS; ++l) colTm += Tm[l * Q1 + i];
            t4[q] = wst[i] * rowXU[i];
            ddir[q] = colTm + Tm[i * Q1 + i] + expf(clast - cs[i]) * rowXU[i];
            dcs[q] = rowT1 - dt[i] * colTm + rowT2[i];
        }
        // sum_{i >= u} dcs[i]: reverse inclusive scans within each block of 32 positions;
        // sum_{s < u} T4[s]: exclusive forward scans within each block; then the other
        // blocks' totals
        float rs[NQ], ps[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) { rs[q] = dcs[q]; ps[q] = t4[q]; }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float t = __shfl_down_sync(0xffffffffu, rs[q], o);
                if (tid + o < 32) rs[q] += t;
            }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float t = __shfl_up_sync(0xffffffffu, ps[q], o);
                if (tid >= o) ps[q] += t;
            }
        }
        float da[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            float later = 0.f, earlier = 0.f;   // later blocks' dcs totals, earlier blocks' T4 totals
#pragma unroll
            for (int q2 = q + 1; q2 < NQ; ++q2) later += __shfl_sync(0xffffffffu, rs[q2], 0);
#pragma unroll
            for (int q2 = 0; q2 < q; ++q2) earlier += __shfl_sync(0xffffffffu, ps[q2], 31);
            float ex = __shfl_up_sync(0xffffffffu, ps[q], 1);
            if (tid == 0) ex = 0.f;
            da[q] = rs[q] + later + T3 + earlier + ex;
        }
        const float Ah = A[h];
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int i = tid + 32 * q;
            if (i >= ci.lo && i < ci.len) {
                const float v = dt_raw[(int64_t)ci.b * sdb + (int64_t)(ci.t0 + i) * sdl + h] + (bias ? bias[h] : 0.f);
                const float g_ = (ddir[q] + Ah * da[q]) * sigmoid_f(v);
                ddt[(int64_t)ci.b * sddb + (int64_t)(ci.t0 + i) * sddl + h] = g_;
                pa += dt[i] * da[q];
                pb += g_;
            }
        }
        pa = warp_sum(pa);
        pb = warp_sum(pb);
        float pd = 0.f;
#pragma unroll
        for (int q = 0; q < NQ; ++q) pd += rowD[tid + 32 * q];
        pd = warp_sum(pd);
        if (tid == 0) {
            float *pp = partials + ((int64_t)k * sh.H + h) * 4;
            pp[0] = pa; pp[1] = pd; pp[2] = pb; pp[3] = 0.f;
        }
    }
}

// ------------------------------------------------------------------ reductions
// dB and dC: sum the per-head rows of each group in head order.  grid (kmax, G,
// 2 * ceil(Q/16)): z picks dB or dC and a slab of 16 rows of the chunk; block 256.
template <typename T>
__global__ void k_reduce_group(Shape sh, const int32_t *__restrict__ hdr, const ChunkInfo *__restrict__ chunks,
                               const float *__restrict__ srcB, MView3 dstB, const float *__restrict__ srcC,
                               MView3 dstC) {
    const int k = blockIdx.x, g = blockIdx.y;
    const int nslab = (sh.Q + 15) / 16;
    const int which = blockIdx.z / nslab, l0 = (blockIdx.z % nslab) * 16;
    if (k >= hdr[HDR_NCHUNKS] || hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = chunks[k];
    const float *src = which == 0 ? srcB : srcC;
    const MView3 dst = which == 0 ? dstB : dstC;
    const int N = sh.N, No = sh.Nio;   // share row stride; columns the caller's tensors hold
    const int rows = min(16, ci.len - l0);
    for (int i = threadIdx.x; i < rows * No; i += blockDim.x) {
        const int l = l0 + i / No, n = i % No;
        if (l < ci.lo) continue;   // rows of another sequence sharing the chunk
        float a = 0.f;
        const float *s = src + (((int64_t)k * sh.H + (int64_t)g * sh.hpg) * sh.Q + l) * N + n;
        for (int j = 0; j < sh.hpg; ++j) a += s[(int64_t)j * sh.Q * N];
        T *o = (T *)dst.p + (int64_t)ci.b * dst.s0 + (int64_t)(ci.t0 + l) * dst.s1 + (int64_t)g * dst.s2;
        o[n] = from_f<T>(a);
    }
}

// dA, dD, ddt_bias: sum chunk partials in a fixed order.  grid H, block 256.
__global__ void k_reduce_heads(Shape sh, const int32_t *__restrict__ hdr, const float *__restrict__ partials,
                               float *dA, float *dD, float *dbias) {
    __shared__ float red[3][8];
    const int h = blockIdx.x, tid = threadIdx.x;
    const int nk = hdr[HDR_STATUS] != 0 ? 0 : hdr[HDR_NCHUNKS];
    float a = 0.f, d = 0.f, b = 0.f;
    for (int k = tid; k < nk; k += 256) {
        const float *pp = partials + ((int64_t)k * sh.H + h) * 4;
        a += pp[0]; d += pp[1]; b += pp[2];
    }
    a = warp_sum(a); d = warp_sum(d); b = warp_sum(b);
    if ((tid & 31) == 0) { red[0][tid >> 5] = a; red[1][tid >> 5] = d; red[2][tid >> 5] = b; }
    __syncthreads();
    if (tid == 0) {
        float ta = 0.f, td = 0.f, tb = 0.f;
        for (int w = 0; w < 8; ++w) { ta += red[0][w]; td += red[1][w]; tb += red[2][w]; }
        dA[h] = ta;
        if (dD) dD[h] = td;
        if (dbias) dbias[h] = tb;
    }
}

}  // namespace

size_t bwd_chunk_smem(const Shape &sh) {
    const int QS = sh.Q, P1 = sh.P + 1, N1 = sh.N + 1, Q1 = QS + 1;
    return sizeof(float) * (size_t)(11 * QS + 2 * QS * P1 + 2 * QS * N1 + 3 * QS * Q1);
}
// dS_out and S_in of the chunk staged in shared memory too, where they fit (227 KB per block)
static size_t bwd_chunk_stage_bytes(const Shape &sh) { return sizeof(float) * 2 * (size_t)sh.P * (sh.N + 1); }
static bool bwd_chunk_stages(const Shape &sh) { return bwd_chunk_smem(sh) + bwd_chunk_stage_bytes(sh) <= 227 * 1024; }

template <typename T>
cudaError_t launch_bwd_dstates(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 dy, View3 z,
                               View3 Cm, const float *csw, float *dstates, cudaStream_t st) {
    if (sh.Q == 32)
        k_bwd_dstates<T, 32><<<dim3(sh.kmax, sh.H), 256, 0, st>>>(sh, hdr, chunks, dy, z, Cm, csw, dstates);
    else if (sh.Q == 64)
        k_bwd_dstates<T, 64><<<dim3(sh.kmax, sh.H), 256, 0, st>>>(sh, hdr, chunks, dy, z, Cm, csw, dstates);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_chunk(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 x, View3 Bm,
                             View3 Cm, View3 z, View3 dy, const float *dt_raw, int64_t sdb, int64_t sdl,
                             const float *A, const float *D, const float *bias, const float *dtw, const float *csw,
                             const float *states, const float *dstates, MView3 dx, MView3 dz, float *ddt,
                             int64_t sddb, int64_t sddl, float *dBh, float *dCh, float *partials, cudaStream_t st) {
    const int stage = bwd_chunk_stages(sh) ? 1 : 0;
    const size_t smem = bwd_chunk_smem(sh) + (stage ? bwd_chunk_stage_bytes(sh) : 0);
    if (sh.Q == 32) {
        static int attr_done[64] = {0};
        cudaError_t e = ensure_smem_attr(k_bwd_chunk<T, 32>, (int)smem, attr_done);
        if (e != cudaSuccess) return e;
        k_bwd_chunk<T, 32><<<dim3(sh.kmax, sh.H), 256, smem, st>>>(sh, hdr, chunks, x, Bm, Cm, z, dy, dt_raw, sdb, sdl,
                                                                   A, D, bias, dtw, csw, states, dstates, dx, dz, ddt,
                                                                   sddb, sddl, dBh, dCh, partials, stage);
    } else if (sh.Q == 64) {
        static int attr_done[64] = {0};
        cudaError_t e = ensure_smem_attr(k_bwd_chunk<T, 64>, (int)smem, attr_done);
        if (e != cudaSuccess) return e;
        k_bwd_chunk<T, 64><<<dim3(sh.kmax, sh.H), 256, smem, st>>>(sh, hdr, chunks, x, Bm, Cm, z, dy, dt_raw, sdb, sdl,
                                                                   A, D, bias, dtw, csw, states, dstates, dx, dz, ddt,
                                                                   sddb, sddl, dBh, dCh, partials, stage);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_reduce_group(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const float *srcB,
                                MView3 dstB, const float *srcC, MView3 dstC, cudaStream_t st) {
    const int nslab = (sh.Q + 15) / 16;
    k_reduce_group<T><<<dim3(sh.kmax, sh.G, 2 * nslab), 256, 0, st>>>(sh, hdr, chunks, srcB, dstB, srcC, dstC);
    return cudaGetLastError();
}

cudaError_t launch_reduce_heads(const Shape &sh, const int32_t *hdr, const float *partials, float *dA, float *dD,
                                float *dbias, cudaStream_t st) {
    k_reduce_heads<<<sh.H, 256, 0, st>>>(sh, hdr, partials, dA, dD, dbias);
    return cudaGetLastError();
}

#define SSD_INST(T)                                                                                              \
    template cudaError_t launch_bwd_dstates<T>(const Shape &, const int32_t *, const ChunkInfo *, View3, View3,  \
                                               View3, const float *, float *, cudaStream_t);                     \
    template cudaError_t launch_bwd_chunk<T>(const Shape &, const int32_t *, const ChunkInfo *, View3, View3,    \
                                             View3, View3, View3, const float *, int64_t, int64_t, const float *, \
                                             const float *, const float *, const float *, const float *,          \
                                             const float *, const float *, MView3, MView3, float *, int64_t,      \
                                             int64_t, float *, float *, float *, cudaStream_t);                   \
    template cudaError_t launch_reduce_group<T>(const Shape &, const int32_t *, const ChunkInfo *, const float *, \
                                                MView3, const float *, MView3, cudaStream_t);
SSD_INST(float)
SSD_INST(__nv_bfloat16)
#undef SSD_INST

}  // namespace ssd
