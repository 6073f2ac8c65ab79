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

// ---- staged sweeps.  A block covers TT tokens x CB channels; its threads first copy the tile
// (plus the K-1 rows before it, and for the backward after it) into shared memory with
// cp.async -- a whole tile of loads in flight at once -- and then thread (piece j, token group
// g) sweeps its W channels over TG = 8 tokens (forward: W = 8, 256 threads) or TGB = 16 tokens
// (backward: W = 4, 256 threads, about 110 registers, two blocks per SM) from shared memory.
// (Measured: a forward with W = 4 is a third slower; a backward with W = 8 or 2 a tenth.)
constexpr int CB = 256;              // channels per block (32 pieces of 8)
constexpr int TG = TT / (CT / 32);   // tokens per thread: 8
constexpr int CTB = 128;             // backward: threads per block (two blocks per SM) ...
constexpr int TGB = TT / (CTB / 32); // ... and tokens per thread: 16
#define TAPS_BYTES(K) ((size_t)((K) + 1) * CB * sizeof(float))   // staged taps and bias
#ifndef CONV_BWD_W
#define CONV_BWD_W 4
#endif
#ifndef CONV_FWD_W
#define CONV_FWD_W 8
#endif

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Copies rows [tb, tb + nrows) of a [L][channels] token matrix (row stride sl elements),
// channels [cbase, cbase + CB), into `dst` (row r at r * 32 pieces); rows outside [0, L) and
// channels past Cn are not copied (never read unmasked).
template <typename T>
__device__ __forceinline__ void stage_rows(const T *src, int64_t sl, int64_t tb, int nrows, int64_t L, int64_t cbase,
                                           int64_t Cn, T *dst) {
    for (int i = threadIdx.x; i < nrows * 32; i += blockDim.x) {
        const int r = i >> 5, j = i & 31;
        const int64_t t = tb + r, c = cbase + 8 * j;
        if (t >= 0 && t < L && c < Cn) {
            const T *g = src + t * sl + c;
            T *d = dst + (int64_t)r * (32 * 8) + 8 * j;
            if (sizeof(T) == 2) {
                cp_async16(d, g);
            } else {
                cp_async16(d, g);
                cp_async16(d + 4, g + 4);
            }
        }
    }
    cp_async_commit_wait();
}

template <typename T>
__device__ __forceinline__ void lds8(const T *p, float *v) { ld8(p, v); }
// 4 channels: 8 bytes (bf16) or 16 bytes (fp32)
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float *v) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void ld4(const float *p, float *v) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float *v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}
__device__ __forceinline__ void st4(float *p, const float *v) {
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
// 2 channels: 4 bytes (bf16) or 8 bytes (fp32)
__device__ __forceinline__ void ld2(const __nv_bfloat16 *p, float *v) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    v[0] = a.x; v[1] = a.y;
}
__device__ __forceinline__ void ld2(const float *p, float *v) {
    const float2 a = *reinterpret_cast<const float2 *>(p);
    v[0] = a.x; v[1] = a.y;
}
__device__ __forceinline__ void st2(__nv_bfloat16 *p, const float *v) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(v[0], v[1]);
}
__device__ __forceinline__ void st2(float *p, const float *v) { *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]); }
template <int W, typename T>
__device__ __forceinline__ void ldw(const T *p, float *v) {
    if (W == 8) ld8(p, v); else if (W == 4) ld4(p, v); else ld2(p, v);
}
template <int W, typename T>
__device__ __forceinline__ void stw(T *p, const float *v) {
    if (W == 8) st8(p, v); else if (W == 4) st4(p, v); else st2(p, v);
}

// logistic function with the fast exponential and divide (relative error ~1e-6; 1/inf = 0
// gives the right limit for very negative arguments)
__device__ __forceinline__ float sig_fast(float v) { return __fdividef(1.f, 1.f + __expf(-v)); }
// the same through one tanh.approx (relative error ~2^-11): (1 + tanh(v/2)) / 2, for bf16 data,
// whose own rounding is 2^-9
__device__ __forceinline__ float sig_tanh(float v) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * v));
    return fmaf(0.5f, t, 0.5f);
}
template <typename T>
__device__ __forceinline__ float sig_t(float v) { return sizeof(T) == 2 ? sig_tanh(v) : sig_fast(v); }

// The block's taps and biases, staged once in shared memory as [k][channel] (then [K][c] =
// the bias): weight [Cn][K] holds channels cbase .. cbase+255 as 256K contiguous floats, read
// with consecutive threads on consecutive floats; a thread then reads its 8 channels of tap k
// as two 16-byte pieces.
template <int K>
__device__ __forceinline__ void stage_taps(const float *w, const float *bias, int64_t cbase, int64_t Cn, float *ws) {
    const int64_t nch = std::min<int64_t>(CB, Cn - cbase);
    for (int i = threadIdx.x; i < CB * K; i += blockDim.x) {
        const int c = i / K, k = i % K;
        ws[k * CB + c] = c < nch ? w[cbase * K + i] : 0.f;
    }
    for (int c = threadIdx.x; c < CB; c += blockDim.x)
        ws[K * CB + c] = (bias != nullptr && c < nch) ? bias[cbase + c] : 0.f;
}

template <typename T, int K, int W>   // W channels per thread (8: 256 threads, 4: 512 threads)
__global__ void __launch_bounds__(CT * 8 / W, 4)   // four blocks per SM (64 registers) measured 2-3% faster than three
k_conv_fwd(const ConvArgs a) {
    constexpr int NPC = CB / W;        // channel pieces per row
    extern __shared__ __align__(16) uint8_t conv_sm[];
    float *ws = reinterpret_cast<float *>(conv_sm);                  // taps [K][CB], bias [CB]
    T *tile = reinterpret_cast<T *>(conv_sm + TAPS_BYTES(K));        // rows t0-(K-1) .. t0+TT-1
    const int j = threadIdx.x % NPC, grp = threadIdx.x / NPC;
    const int64_t cbase = (int64_t)blockIdx.y * CB, c0 = cbase + W * j;
    const int64_t b = blockIdx.x / a.tiles_per_row, t0 = (blockIdx.x % a.tiles_per_row) * TT;
    const int64_t tb = t0 - (K - 1);
    stage_taps<K>(a.w, a.bias, cbase, a.Cn, ws);
    stage_rows(static_cast<const T *>(a.u) + b * a.su_b, a.su_l, tb, TT + K - 1, a.L, cbase, a.Cn, tile);
    __syncthreads();
    if (c0 >= a.Cn) return;
    const int64_t s0 = t0 + (int64_t)grp * TG, s1 = std::min(a.L, s0 + TG);   // this thread's tokens
    if (s0 >= s1) return;
    T *o = static_cast<T *>(a.out) + b * a.so_b + c0;
    float w[K][W], bias[W];
#pragma unroll
    for (int k = 0; k <= K; ++k) {   // the thread's W channels of tap k (k = K: the bias)
        float *dst = k < K ? w[k < K ? k : 0] : bias;
#pragma unroll
        for (int e = 0; e < W; ++e) dst[e] = ws[k * CB + W * j + e];
    }
    SeqCursor cur;
    cur.init(a, s0);
    const T *col = tile + W * j;   // row t at (t - tb) * 256 (offsets below fit 32 bits)
    if (s0 - (K - 1) >= cur.start && s1 <= cur.next) {
        // The thread's tokens and the K-1 before them lie in one sequence: no sequence starts
        // to test, a 32-bit counter, pointers that step a row.
        const T *rp = col + (int)(s0 - t0) * 256;   // row t - (K-1) of the current t
        T *op = o + s0 * a.so_l;
        const int n = (int)(s1 - s0);
        for (int i = 0; i < n; ++i) {
            float acc[W];
#pragma unroll
            for (int e = 0; e < W; ++e) acc[e] = bias[e];
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float v[W];
                ldw<W>(rp + k * 256, v);
#pragma unroll
                for (int e = 0; e < W; ++e) acc[e] = fmaf(w[k][e], v[e], acc[e]);
            }
            if (a.silu) {
#pragma unroll
                for (int e = 0; e < W; ++e) acc[e] *= sig_t<T>(acc[e]);
            }
            stw<W>(op, acc);
            rp += 256;
            op += a.so_l;
        }
        return;
    }
    for (int64_t t = s0; t < s1; ++t) {
        cur.advance(a, t);
        float acc[W];
#pragma unroll
        for (int e = 0; e < W; ++e) acc[e] = bias[e];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int64_t tp = t - (K - 1) + k;   // u[tp] feeds pre[t] when in t's sequence
            if (tp >= cur.start) {
                float v[W];
                ldw<W>(col + (int)(tp - tb) * 256, v);
#pragma unroll
                for (int e = 0; e < W; ++e) acc[e] = fmaf(w[k][e], v[e], acc[e]);
            }
        }
        if (a.silu) {
#pragma unroll
            for (int e = 0; e < W; ++e) acc[e] *= sig_t<T>(acc[e]);
        }
        stw<W>(o + t * a.so_l, acc);
    }
}

// Backward over the thread's tokens [s0, s1): the sweep runs t from s0 to s1 + K - 2 computing
// g[t] = dout[t] act'(pre[t]); g[t] reaches du[t - (K-1) + k] (same sequence) for every k;
// du[t'] is complete once t passes t' + K - 1 and leaves then.  dw and dbias take the thread's
// tokens t in [s0, s1); the eight token groups' shares are summed in order in shared memory.
template <typename T, int K, int W>   // W channels per thread (8: 128 threads, 4: 256 threads)
__global__ void __launch_bounds__(CTB * 8 / W)
k_conv_bwd(const ConvArgs a) {
    constexpr int NPC = CB / W;        // channel pieces per row
    constexpr int NT = NPC * (TT / TGB);
    extern __shared__ __align__(16) uint8_t conv_sm[];
    constexpr int RU = TT + 2 * (K - 1), RD = TT + K - 1;
    float *ws = reinterpret_cast<float *>(conv_sm);                    // taps [K][CB], bias [CB]
    T *tu = reinterpret_cast<T *>(conv_sm + TAPS_BYTES(K));            // u rows t0-(K-1) .. t0+TT+K-2
    T *td = tu + RU * 256;                                             // dout rows t0 .. t0+TT+K-2
    float *red = reinterpret_cast<float *>(conv_sm + TAPS_BYTES(K));   // after the sweep: [group][K+1][256]
    const int j = threadIdx.x % NPC, grp = threadIdx.x / NPC;
    const int64_t cbase = (int64_t)blockIdx.y * CB, c0 = cbase + W * j;
    const int64_t b = blockIdx.x / a.tiles_per_row, t0 = (blockIdx.x % a.tiles_per_row) * TT;
    const int64_t tb = t0 - (K - 1);
    stage_taps<K>(a.w, a.bias, cbase, a.Cn, ws);
    stage_rows(static_cast<const T *>(a.u) + b * a.su_b, a.su_l, tb, RU, a.L, cbase, a.Cn, tu);
    stage_rows(static_cast<const T *>(a.dout) + b * a.sd_b, a.sd_l, t0, RD, a.L, cbase, a.Cn, td);
    __syncthreads();
    const bool live = c0 < a.Cn;
    const int64_t s0 = t0 + (int64_t)grp * TGB, s1 = std::min(a.L, s0 + TGB);
    float w[K][W], bias[W], dw[K][W], db[W];
#pragma unroll
    for (int k = 0; k <= K; ++k) {   // the thread's W channels of tap k (k = K: the bias)
        float *dst = k < K ? w[k < K ? k : 0] : bias;
#pragma unroll
        for (int e = 0; e < W; ++e) dst[e] = ws[k * CB + W * j + e];
    }
#pragma unroll
    for (int e = 0; e < W; ++e) {
        db[e] = 0.f;
#pragma unroll
        for (int k = 0; k < K; ++k) dw[k][e] = 0.f;
    }
    if (live && s0 < s1) {
        T *du = static_cast<T *>(a.du) + b * a.sdu_b + c0;
        const T *ucol = tu + W * j, *dcol = td + W * j;
        SeqCursor cur;
        cur.init(a, s0);
        float ring[K][W];   // inputs u[t - (K-1) + k]
        float acc[K][W];    // du[t - (K-1) + k] being summed
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int e = 0; e < W; ++e) acc[k][e] = 0.f;
        const int64_t tend_all = std::min(a.L, s1 + K - 1);
        if (s0 - (K - 1) >= cur.start && tend_all <= cur.next) {
            // The thread's whole window (its tokens, the K-1 before and after) lies in one
            // sequence: no sequence starts to test, 32-bit counters, pointers that step a row.
            const T *up = ucol + (int)(s0 - t0) * 256, *dp = dcol + (int)(s0 - t0) * 256;
#pragma unroll
            for (int k = 0; k < K - 1; ++k) ldw<W>(up + k * 256, ring[k]);
            up += (K - 1) * 256;
            T *dup = du + (s0 - (K - 1)) * a.sdu_l;   // du[t - (K-1)] of the current t
            const int nown = (int)(s1 - s0), ntot = (int)(tend_all - s0);
#pragma unroll 4   // the ring and accumulator rotation becomes register renaming
            for (int i = 0; i < ntot; ++i) {
                ldw<W>(up, ring[K - 1]);
                up += 256;
                float dv[W];
                ldw<W>(dp, dv);
                dp += 256;
                float g[W];
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    float pre = bias[e];
#pragma unroll
                    for (int k = 0; k < K; ++k) pre = fmaf(w[k][e], ring[k][e], pre);
                    if (a.silu) {
                        const float sg = sig_t<T>(pre);
                        g[e] = dv[e] * sg * (1.f + pre * (1.f - sg));
                    } else {
                        g[e] = dv[e];
                    }
                }
#pragma unroll
                for (int k = 0; k < K; ++k)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[k][e] = fmaf(w[k][e], g[e], acc[k][e]);
                if (i < nown) {   // this thread's token: its dw / dbias shares
#pragma unroll
                    for (int e = 0; e < W; ++e) {
#pragma unroll
                        for (int k = 0; k < K; ++k) dw[k][e] = fmaf(g[e], ring[k][e], dw[k][e]);
                        db[e] += g[e];
                    }
                }
                if (i >= K - 1) stw<W>(dup, acc[0]);   // du[s0 + i - (K-1)] is complete
                dup += a.sdu_l;
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        ring[k][e] = ring[k + 1][e];
                        acc[k][e] = acc[k + 1][e];
                    }
#pragma unroll
                for (int e = 0; e < W; ++e) acc[K - 1][e] = 0.f;
            }
            // rows whose windows would run past the end of the row (tend_all clamped to L)
            for (int64_t tdone = tend_all - (K - 1); tdone < s1; ++tdone) {
                if (tdone >= s0) stw<W>(du + tdone * a.sdu_l, acc[0]);
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int e = 0; e < W; ++e) acc[k][e] = acc[k + 1][e];
#pragma unroll
                for (int e = 0; e < W; ++e) acc[K - 1][e] = 0.f;
            }
        } else {
#pragma unroll
        for (int k = 0; k < K - 1; ++k) {
            const int64_t tp = s0 - (K - 1) + k;
            if (tp >= cur.start) ldw<W>(ucol + (int)(tp - tb) * 256, ring[k]);
            else {
#pragma unroll
                for (int e = 0; e < W; ++e) ring[k][e] = 0.f;
            }
        }
        const int64_t tend = std::min(a.L, s1 + K - 1);
        for (int64_t t = s0; t < tend; ++t) {
            if (cur.advance(a, t)) {
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
#pragma unroll
                    for (int e = 0; e < W; ++e) ring[k][e] = 0.f;
            }
            ldw<W>(ucol + (int)(t - tb) * 256, ring[K - 1]);
            float dv[W];
            ldw<W>(dcol + (int)(t - t0) * 256, dv);
            float g[W];
#pragma unroll
            for (int e = 0; e < W; ++e) {
                float pre = bias[e];
#pragma unroll
                for (int k = 0; k < K; ++k) pre = fmaf(w[k][e], ring[k][e], pre);
                if (a.silu) {
                    const float sg = sig_t<T>(pre);
                    g[e] = dv[e] * sg * (1.f + pre * (1.f - sg));
                } else {
                    g[e] = dv[e];
                }
            }
            const bool own = t < s1;   // this thread's token: its dw / dbias shares
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int64_t tp = t - (K - 1) + k;
                if (tp >= cur.start) {   // u[tp] fed pre[t] (same sequence)
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        acc[k][e] = fmaf(w[k][e], g[e], acc[k][e]);
                        if (own) dw[k][e] = fmaf(g[e], ring[k][e], dw[k][e]);
                    }
                }
            }
            if (own) {
#pragma unroll
                for (int e = 0; e < W; ++e) db[e] += g[e];
            }
            const int64_t tdone = t - (K - 1);   // du[tdone] has all its contributions now
            if (tdone >= s0 && tdone < s1) stw<W>(du + tdone * a.sdu_l, acc[0]);
#pragma unroll
            for (int k = 0; k < K - 1; ++k)
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    ring[k][e] = ring[k + 1][e];
                    acc[k][e] = acc[k + 1][e];
                }
#pragma unroll
            for (int e = 0; e < W; ++e) acc[K - 1][e] = 0.f;
        }
        // the last rows, whose windows would run past the end of the row: acc[0] now holds
        // du[tend - (K-1)]; rows before s0 are skipped over
        for (int64_t tdone = tend - (K - 1); tdone < s1; ++tdone) {
            if (tdone >= s0) stw<W>(du + tdone * a.sdu_l, acc[0]);
#pragma unroll
            for (int k = 0; k < K - 1; ++k)
#pragma unroll
                for (int e = 0; e < W; ++e) acc[k][e] = acc[k + 1][e];
#pragma unroll
            for (int e = 0; e < W; ++e) acc[K - 1][e] = 0.f;
        }
        }   // general path
    }
    __syncthreads();   // the staged tiles are no longer read: reuse them for the group sums
#pragma unroll
    for (int e = 0; e < W; ++e) {
#pragma unroll
        for (int k = 0; k < K; ++k) red[((grp * (K + 1)) + k) * 256 + W * j + e] = dw[k][e];
        red[((grp * (K + 1)) + K) * 256 + W * j + e] = db[e];
    }
    __syncthreads();
    float *pp = a.partials + (int64_t)blockIdx.x * a.Cn * (K + 1);
    for (int i = threadIdx.x; i < 256 * (K + 1); i += NT) {
        const int c = i / (K + 1), k = i % (K + 1);   // channel within the block, tap (K: bias)
        if (cbase + c >= a.Cn) continue;
        float sum = 0.f;
        for (int q = 0; q < TT / TGB; ++q) sum += red[(q * (K + 1) + k) * 256 + c];
        pp[(cbase + c) * (K + 1) + k] = sum;
    }
}

// dw / dbias: the column sums of the per-tile shares [tiles][Cn (K+1)] in a fixed order.  A
// block takes 32 columns; warp w sums tiles w, w + 8, ... in ascending order (four loads in
// flight), and the eight warp sums are added in warp order.
__global__ void __launch_bounds__(256) k_conv_dw(const float *partials, int64_t tiles, int64_t Cn, int K, float *dw,
                                                 float *db) {
    __shared__ float red[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t n = Cn * (K + 1), i = (int64_t)blockIdx.x * 32 + lane;
    float s = 0.f;
    if (i < n) {
        const float *col = partials + i;
        int64_t t = w;
        for (; t + 24 < tiles; t += 32) {
            const float a0 = col[t * n], a1 = col[(t + 8) * n], a2 = col[(t + 16) * n], a3 = col[(t + 24) * n];
            s += a0;
            s += a1;
            s += a2;
            s += a3;
        }
        for (; t < tiles; t += 8) s += col[t * n];
    }
    red[w][lane] = s;
    __syncthreads();
    if (w == 0 && i < n) {
        float tot = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) tot += red[q][lane];
        const int64_t c = i / (K + 1);
        const int k = (int)(i - c * (K + 1));
        if (k < K) dw[c * K + k] = tot;
        else if (db) db[c] = tot;
    }
}

template <typename T, int K>
size_t fwd_smem() { return TAPS_BYTES(K) + (size_t)(TT + K - 1) * 256 * sizeof(T); }
template <typename T, int K>
size_t bwd_smem() {
    const size_t stage = (size_t)(2 * TT + 3 * (K - 1)) * 256 * sizeof(T);
    const size_t red = (size_t)(TT / TGB) * (K + 1) * 256 * sizeof(float);
    return TAPS_BYTES(K) + (stage > red ? stage : red);
}
constexpr int kFwdW = CONV_FWD_W;   // channels per thread of the forward sweep
template <typename T, int K>
cudaError_t launch_fwd_k(const ConvArgs &a, dim3 grid, cudaStream_t st) {
    static int attr[64] = {0};
    const size_t sm = fwd_smem<T, K>();
    cudaError_t e = ensure_smem_attr(k_conv_fwd<T, K, kFwdW>, (int)sm, attr);
    if (e != cudaSuccess) return e;
    k_conv_fwd<T, K, kFwdW><<<grid, CT * 8 / kFwdW, sm, st>>>(a);
    return cudaGetLastError();
}
constexpr int kBwdW = CONV_BWD_W;   // channels per thread of the backward sweep
template <typename T, int K>
cudaError_t launch_bwd_k(const ConvArgs &a, dim3 grid, cudaStream_t st) {
    static int attr[64] = {0};
    const size_t sm = bwd_smem<T, K>();
    cudaError_t e = ensure_smem_attr(k_conv_bwd<T, K, kBwdW>, (int)sm, attr);
    if (e != cudaSuccess) return e;
    k_conv_bwd<T, K, kBwdW><<<grid, CTB * 8 / kBwdW, sm, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fwd(const ConvArgs &a, dim3 grid, cudaStream_t st) {
    switch (a.K) {
        case 1: return launch_fwd_k<T, 1>(a, grid, st);
        case 2: return launch_fwd_k<T, 2>(a, grid, st);
        case 3: return launch_fwd_k<T, 3>(a, grid, st);
        case 4: return launch_fwd_k<T, 4>(a, grid, st);
        case 5: return launch_fwd_k<T, 5>(a, grid, st);
        case 6: return launch_fwd_k<T, 6>(a, grid, st);
        case 7: return launch_fwd_k<T, 7>(a, grid, st);
        default: return launch_fwd_k<T, 8>(a, grid, st);
    }
}
template <typename T>
cudaError_t launch_bwd(const ConvArgs &a, dim3 grid, cudaStream_t st) {
    switch (a.K) {
        case 1: return launch_bwd_k<T, 1>(a, grid, st);
        case 2: return launch_bwd_k<T, 2>(a, grid, st);
        case 3: return launch_bwd_k<T, 3>(a, grid, st);
        case 4: return launch_bwd_k<T, 4>(a, grid, st);
        case 5: return launch_bwd_k<T, 5>(a, grid, st);
        case 6: return launch_bwd_k<T, 6>(a, grid, st);
        case 7: return launch_bwd_k<T, 7>(a, grid, st);
        default: return launch_bwd_k<T, 8>(a, grid, st);
    }
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
    const dim3 grid((unsigned)(a.B * a.tiles_per_row), (unsigned)((a.Cn + CB - 1) / CB));
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
        const dim3 grid((unsigned)tiles, (unsigned)((a.Cn + CB - 1) / CB));
        const cudaError_t e =
            p->dtype == SSD_BF16 ? launch_bwd<__nv_bfloat16>(a, grid, st) : launch_bwd<float>(a, grid, st);
        if (e != cudaSuccess) return SSD_ERR_CUDA;
    } else {
        if (cudaMemsetAsync(workspace, 0, need, st) != cudaSuccess) return SSD_ERR_CUDA;
    }
    const int64_t n = p->channels * (p->width + 1);
    k_conv_dw<<<(unsigned)((n + 31) / 32), 256, 0, st>>>(
        a.partials, std::max<int64_t>(tiles, 1), p->channels, (int)p->width, dweight, dbias);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
