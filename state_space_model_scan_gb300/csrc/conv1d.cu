// conv1d.cu -- causal depthwise convolution over the sequence axis with an optional SiLU,
// forward and backward: the step before the scan in a Mamba-2 block, run on the packed
// xBC = [x | B | C] channels (the Helion pull request for the Mamba-2 SSD path, "Summary":
// mamba_split_conv1d_scan_combined; "Testing": x, B and C are views of one packed buffer):
//
//   pre[t,c] = bias[c] + sum_{k<K} w[c,k] u[t-(K-1)+k, c]   (u := 0 before t's sequence start)
//   out[t,c] = silu(pre[t,c])  (or pre)
//
// The scan then reads x, B and C as strided views of `out` (no copy: the split is the view).
// A thread owns 8 consecutive channels and sweeps a tile of TT tokens with its inputs' last
// K rows in registers (forward), and, for the backward, also the K input-gradient rows still
// receiving contributions; the weight and bias gradients are per-tile partial sums added in a
// fixed order afterwards (bitwise reproducible).  Every access of a warp is one contiguous
// 512-byte (bf16) or 1 KB (fp32) row piece.
#include <algorithm>

#include "common.cuh"

namespace ssd {

namespace {

constexpr int TT = 64;        // tokens per thread
constexpr int CT = 256;       // threads per block (8 channels each)
constexpr int KMAX = 8;

__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float *v) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(e[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void ld8(const float *p, float *v) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8(__nv_bfloat16 *p, const float *v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void st8(float *p, const float *v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

struct ConvArgs {
    int64_t B, L, Cn, S;          // batch rows, tokens per row, channels, sequences (packed) or 0
    int K;
    bool silu;
    const void *u, *dout;
    int64_t su_b, su_l, sd_b, sd_l;
    const float *w, *bias;        // w: [Cn][K]
    const int32_t *cu;            // packed sequences (B = 1) or NULL
    void *out, *du;
    int64_t so_b, so_l, sdu_b, sdu_l;
    float *partials;              // [tiles][Cn][K + 1]: dw shares, then the dbias share
    int64_t tiles_per_row;
};

// Sequence bookkeeping along a sweep: the start of the current token's sequence and the
// first token of the next one.
struct SeqCursor {
    int64_t start, next;
    int s;
    __device__ void init(const ConvArgs &a, int64_t t) {
        if (a.cu == nullptr) {
            start = 0;
            next = a.L;
            s = 0;
            return;
        }
        int lo = 0, hi = (int)a.S - 1;   // last s with cu[s] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        s = lo;
        start = max(a.cu[s], 0);   // clamped: a malformed cu_seqlens never moves a load off the row
        next = a.cu[s + 1];
    }
    // advances to token t (non-decreasing); true when t starts a new sequence
    __device__ bool advance(const ConvArgs &a, int64_t t) {
        if (a.cu == nullptr || t < next) return false;
        while (s + 1 < a.S && a.cu[s + 1] <= t) ++s;
        start = max(a.cu[s], 0);
        next = a.cu[s + 1];
        return true;
    }
};

template <typename T, int K>
__global__ void __launch_bounds__(CT)
k_conv_fwd(const ConvArgs a) {
    const int64_t c0 = ((int64_t)blockIdx.y * CT + threadIdx.x) * 8;
    if (c0 >= a.Cn) return;
    const int64_t b = blockIdx.x / a.tiles_per_row, t0 = (blockIdx.x % a.tiles_per_row) * TT;
    const int64_t t1 = std::min(a.L, t0 + TT);
    const T *u = static_cast<const T *>(a.u) + b * a.su_b + c0;
    T *o = static_cast<T *>(a.out) + b * a.so_b + c0;
    float w[K][8], bias[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        bias[e] = a.bias ? a.bias[c0 + e] : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) w[k][e] = a.w[(c0 + e) * K + k];
    }
    SeqCursor cur;
    cur.init(a, t0);
    float ring[K][8];   // ring[k] = u[t - (K-1) + k] for the current t (k < K-1 filled before t)
#pragma unroll
    for (int k = 0; k < K - 1; ++k) {
        const int64_t tp = t0 - (K - 1) + k;
        if (tp >= cur.start) ld8(u + tp * a.su_l, ring[k]);
        else {
#pragma unroll
            for (int e = 0; e < 8; ++e) ring[k][e] = 0.f;
        }
    }
    for (int64_t t = t0; t < t1; ++t) {
        if (cur.advance(a, t)) {   // a new sequence: nothing before it counts
#pragma unroll
            for (int k = 0; k < K - 1; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) ring[k][e] = 0.f;
        }
        ld8(u + t * a.su_l, ring[K - 1]);
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = bias[e];
#pragma unroll
            for (int k = 0; k < K; ++k) acc = fmaf(w[k][e], ring[k][e], acc);
            v[e] = a.silu ? acc * sigmoid_f(acc) : acc;
        }
        st8(o + t * a.so_l, v);
#pragma unroll
        for (int k = 0; k < K - 1; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) ring[k][e] = ring[k + 1][e];
    }
}

// Backward over the tile [t0, t1): the sweep runs t from t0 to t1 + K - 2 computing
// g[t] = dout[t] act'(pre[t]); g[t] reaches du[t - (K-1) + k] (same sequence) for every k;
// du[t'] is complete once t passes t' + K - 1 and leaves then.  dw and dbias take the tile's
// tokens t in [t0, t1).
template <typename T, int K>
__global__ void __launch_bounds__(CT)
k_conv_bwd(const ConvArgs a) {
    const int64_t c0 = ((int64_t)blockIdx.y * CT + threadIdx.x) * 8;
    if (c0 >= a.Cn) return;
    const int64_t b = blockIdx.x / a.tiles_per_row, t0 = (blockIdx.x % a.tiles_per_row) * TT;
    const int64_t t1 = std::min(a.L, t0 + TT);
    const T *u = static_cast<const T *>(a.u) + b * a.su_b + c0;
    const T *d = static_cast<const T *>(a.dout) + b * a.sd_b + c0;
    T *du = static_cast<T *>(a.du) + b * a.sdu_b + c0;
    float w[K][8], bias[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        bias[e] = a.bias ? a.bias[c0 + e] : 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) w[k][e] = a.w[(c0 + e) * K + k];
    }
    float dw[K][8], db[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        db[e] = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) dw[k][e] = 0.f;
    }
    SeqCursor cur;
    cur.init(a, t0);
    float ring[K][8];   // inputs u[t - (K-1) + k]
    float acc[K][8];    // du[t - (K-1) + k] being summed
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;
#pragma unroll
    for (int k = 0; k < K - 1; ++k) {
        const int64_t tp = t0 - (K - 1) + k;
        if (tp >= cur.start) ld8(u + tp * a.su_l, ring[k]);
        else {
#pragma unroll
            for (int e = 0; e < 8; ++e) ring[k][e] = 0.f;
        }
    }
    const int64_t tend = std::min(a.L, t1 + K - 1);
    for (int64_t t = t0; t < tend; ++t) {
        if (cur.advance(a, t)) {
#pragma unroll
            for (int k = 0; k < K - 1; ++k)
#pragma unroll
                for (int e = 0; e < 8; ++e) ring[k][e] = 0.f;
        }
        ld8(u + t * a.su_l, ring[K - 1]);
        float dv[8];
        ld8(d + t * a.sd_l, dv);
        float g[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float pre = bias[e];
#pragma unroll
            for (int k = 0; k < K; ++k) pre = fmaf(w[k][e], ring[k][e], pre);
            if (a.silu) {
                const float sg = sigmoid_f(pre);
                g[e] = dv[e] * sg * (1.f + pre * (1.f - sg));
            } else {
                g[e] = dv[e];
            }
        }
        const bool own = t < t1;   // this tile's token: its dw / dbias shares
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t tp = t - (K - 1) + k;
            if (tp >= cur.start) {   // u[tp] fed pre[t] (same sequence)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    acc[k][e] = fmaf(w[k][e], g[e], acc[k][e]);
                    if (own) dw[k][e] = fmaf(g[e], ring[k][e], dw[k][e]);
                }
            }
        }
        if (own) {
#pragma unroll
            for (int e = 0; e < 8; ++e) db[e] += g[e];
        }
        // du[t - (K-1)] has all its contributions now
        const int64_t tdone = t - (K - 1);
        if (tdone >= t0 && tdone < t1) st8(du + tdone * a.sdu_l, acc[0]);
#pragma unroll
        for (int k = 0; k < K - 1; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                ring[k][e] = ring[k + 1][e];
                acc[k][e] = acc[k + 1][e];
            }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[K - 1][e] = 0.f;
    }
    // the tile's last rows, whose windows would run past the end of the row: acc[0] now holds
    // du[tend - (K-1)]; rows before t0 are skipped over
    for (int64_t tdone = tend - (K - 1); tdone < t1; ++tdone) {
        if (tdone >= t0) st8(du + tdone * a.sdu_l, acc[0]);
#pragma unroll
        for (int k = 0; k < K - 1; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[k][e] = acc[k + 1][e];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[K - 1][e] = 0.f;
    }
    float *pp = a.partials + (int64_t)blockIdx.x * a.Cn * (K + 1);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
        for (int k = 0; k < K; ++k) pp[(c0 + e) * (K + 1) + k] = dw[k][e];
        pp[(c0 + e) * (K + 1) + K] = db[e];
    }
}

__global__ void k_conv_dw(const float *partials, int64_t tiles, int64_t Cn, int K, float *dw, float *db) {
    const int64_t n = Cn * (K + 1);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int64_t t = 0; t < tiles; ++t) s += partials[t * n + i];
        const int64_t c = i / (K + 1);
        const int k = (int)(i - c * (K + 1));
        if (k < K) dw[c * K + k] = s;
        else if (db) db[c] = s;
    }
}

template <typename T>
cudaError_t launch_fwd(const ConvArgs &a, dim3 grid, cudaStream_t st) {
    switch (a.K) {
        case 1: k_conv_fwd<T, 1><<<grid, CT, 0, st>>>(a); break;
        case 2: k_conv_fwd<T, 2><<<grid, CT, 0, st>>>(a); break;
        case 3: k_conv_fwd<T, 3><<<grid, CT, 0, st>>>(a); break;
        case 4: k_conv_fwd<T, 4><<<grid, CT, 0, st>>>(a); break;
        case 5: k_conv_fwd<T, 5><<<grid, CT, 0, st>>>(a); break;
        case 6: k_conv_fwd<T, 6><<<grid, CT, 0, st>>>(a); break;
        case 7: k_conv_fwd<T, 7><<<grid, CT, 0, st>>>(a); break;
        default: k_conv_fwd<T, 8><<<grid, CT, 0, st>>>(a); break;
    }
    return cudaGetLastError();
}
template <typename T>
cudaError_t launch_bwd(const ConvArgs &a, dim3 grid, cudaStream_t st) {
    switch (a.K) {
        case 1: k_conv_bwd<T, 1><<<grid, CT, 0, st>>>(a); break;
        case 2: k_conv_bwd<T, 2><<<grid, CT, 0, st>>>(a); break;
        case 3: k_conv_bwd<T, 3><<<grid, CT, 0, st>>>(a); break;
        case 4: k_conv_bwd<T, 4><<<grid, CT, 0, st>>>(a); break;
        case 5: k_conv_bwd<T, 5><<<grid, CT, 0, st>>>(a); break;
        case 6: k_conv_bwd<T, 6><<<grid, CT, 0, st>>>(a); break;
        case 7: k_conv_bwd<T, 7><<<grid, CT, 0, st>>>(a); break;
        default: k_conv_bwd<T, 8><<<grid, CT, 0, st>>>(a); break;
    }
    return cudaGetLastError();
}

bool al16(const void *p) { return ((uintptr_t)p) % 16 == 0; }

// Host checks shared by both directions.  Token tensors: [batch, seqlen, channels] at element
// strides (row, token); channels contiguous.
ssd_status check_conv(const ssd_conv_problem *p, bool varlen) {
    if (p == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    if (p->batch < 1 || p->seqlen < 0 || p->channels < 1 || p->width < 1 || p->reserved != 0)
        return SSD_ERR_INVALID_ARGUMENT;
    if (p->dtype < SSD_F32 || p->dtype > SSD_BF16 || p->activation < 0 || p->activation > 1)
        return SSD_ERR_INVALID_ARGUMENT;
    if (varlen && (p->batch != 1 || p->nseqs < 1)) return SSD_ERR_INVALID_ARGUMENT;
    if (!varlen && p->nseqs != 0) return SSD_ERR_INVALID_ARGUMENT;
    if (p->width > KMAX || p->channels % 8 != 0 || p->seqlen > ((int64_t)1 << 31) || p->nseqs > ((int64_t)1 << 24))
        return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}
ssd_status check_tok(const ssd_conv_problem *p, const void *t, int64_t sb, int64_t sl) {
    if (p->seqlen == 0) return SSD_OK;
    if (t == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    if (sl < p->channels || (p->batch > 1 && sb < sl * p->seqlen)) return SSD_ERR_INVALID_ARGUMENT;
    if (!al16(t) || sl % 8 != 0 || sb % 8 != 0) return SSD_ERR_MISALIGNED;
    return SSD_OK;
}

#define CONV_TRY(expr)                 \
    do {                               \
        ssd_status _s = (expr);        \
        if (_s != SSD_OK) return _s;   \
    } while (0)

ConvArgs make_args(const ssd_conv_problem *p, const float *w, const float *bias, const int32_t *cu) {
    ConvArgs a{};
    a.B = p->batch; a.L = p->seqlen; a.Cn = p->channels; a.S = cu ? p->nseqs : 0; a.K = (int)p->width;
    a.silu = p->activation == 1;
    a.w = w; a.bias = bias; a.cu = cu;
    a.tiles_per_row = (p->seqlen + TT - 1) / TT;
    return a;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status ssd_conv1d_fwd(const ssd_conv_problem *p, const void *x, int64_t x_sb, int64_t x_sl, const float *weight,
                          const float *bias, const int32_t *cu_seqlens, void *out, int64_t out_sb, int64_t out_sl,
                          void *stream) {
    CONV_TRY(check_conv(p, cu_seqlens != nullptr));
    CONV_TRY(check_tok(p, x, x_sb, x_sl));
    CONV_TRY(check_tok(p, out, out_sb, out_sl));
    if (weight == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    if (p->seqlen == 0) return SSD_OK;
    ConvArgs a = make_args(p, weight, bias, cu_seqlens);
    a.u = x; a.su_b = x_sb; a.su_l = x_sl; a.out = out; a.so_b = out_sb; a.so_l = out_sl;
    const dim3 grid((unsigned)(a.B * a.tiles_per_row), (unsigned)((a.Cn / 8 + CT - 1) / CT));
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = p->dtype == SSD_BF16 ? launch_fwd<__nv_bfloat16>(a, grid, st) : launch_fwd<float>(a, grid, st);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_conv1d_bwd_workspace_size(const ssd_conv_problem *p, size_t *bytes) {
    if (bytes == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    CONV_TRY(check_conv(p, p != nullptr && p->nseqs != 0));
    const int64_t tiles = p->batch * ((p->seqlen + TT - 1) / TT);
    *bytes = (size_t)std::max<int64_t>(tiles, 1) * (size_t)p->channels * (size_t)(p->width + 1) * sizeof(float);
    return SSD_OK;
}

ssd_status ssd_conv1d_bwd(const ssd_conv_problem *p, const void *x, int64_t x_sb, int64_t x_sl, const float *weight,
                          const float *bias, const int32_t *cu_seqlens, const void *dout, int64_t dout_sb,
                          int64_t dout_sl, void *dx, int64_t dx_sb, int64_t dx_sl, float *dweight, float *dbias,
                          void *workspace, size_t workspace_bytes, void *stream) {
    CONV_TRY(check_conv(p, cu_seqlens != nullptr));
    CONV_TRY(check_tok(p, x, x_sb, x_sl));
    CONV_TRY(check_tok(p, dout, dout_sb, dout_sl));
    CONV_TRY(check_tok(p, dx, dx_sb, dx_sl));
    if (weight == nullptr || dweight == nullptr || (bias != nullptr && dbias == nullptr)) return SSD_ERR_INVALID_ARGUMENT;
    const int64_t tiles = p->batch * ((p->seqlen + TT - 1) / TT);
    const size_t need = (size_t)std::max<int64_t>(tiles, 1) * (size_t)p->channels * (size_t)(p->width + 1) * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need) return SSD_ERR_WORKSPACE_TOO_SMALL;
    if (!al16(workspace)) return SSD_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    ConvArgs a = make_args(p, weight, bias, cu_seqlens);
    a.u = x; a.su_b = x_sb; a.su_l = x_sl; a.dout = dout; a.sd_b = dout_sb; a.sd_l = dout_sl;
    a.du = dx; a.sdu_b = dx_sb; a.sdu_l = dx_sl; a.partials = static_cast<float *>(workspace);
    if (tiles > 0) {
        const dim3 grid((unsigned)tiles, (unsigned)((a.Cn / 8 + CT - 1) / CT));
        const cudaError_t e =
            p->dtype == SSD_BF16 ? launch_bwd<__nv_bfloat16>(a, grid, st) : launch_bwd<float>(a, grid, st);
        if (e != cudaSuccess) return SSD_ERR_CUDA;
    } else {
        if (cudaMemsetAsync(workspace, 0, need, st) != cudaSuccess) return SSD_ERR_CUDA;
    }
    const int64_t n = p->channels * (p->width + 1);
    k_conv_dw<<<(unsigned)std::min<int64_t>((n + 255) / 256, 1024), 256, 0, st>>>(
        a.partials, std::max<int64_t>(tiles, 1), p->channels, (int)p->width, dweight, dbias);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
