// gated_norm.cu -- gated normalisation over feature groups, forward and backward: the
// normalisation that follows the SSD scan in a Mamba-2 block (the gated LayerNorm / RMSNorm
// whose backward the Helion pull request for the Mamba-2 SSD path times as layer_norm_bwd,
// "Measurements").  Per row t and group g of features i, with s = silu(z) (s = 1 without z):
//
//   u = y s (gate first, the default) or u = y (normalise, then gate),
//   mu = mean_{i in g} u (LayerNorm) or 0 (RMS),  rstd[t,g] = 1/sqrt(mean_{i in g} (u-mu)^2 + eps),
//   out[t,i] = (u - mu) rstd w[i]  (times s when the gate comes after)
//
// and its exact derivative.  Memory-bound: one warp per (row, group) item, each lane eight
// consecutive features per 16-byte (bf16) or 32-byte (fp32) access; the backward's weight
// gradient is summed in a fixed order (per-warp shared-memory rows, then row chunks), so
// every result is bitwise reproducible.
#include <algorithm>

#include "common.cuh"

namespace ssd {

namespace {

constexpr int NW = 8;                 // warps per block
constexpr int64_t kMaxGroup = 6144;   // features per group at most (backward: NW rows of it in shared memory)

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *v) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(e[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float *p, float *v) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// 8 elements as loaded (raw bits), converted later: lets a warp keep the next item's loads in flight
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> { uint4 u; };
template <> struct Raw8<float> { float4 a, b; };
__device__ __forceinline__ void ldraw(const __nv_bfloat16 *p, Raw8<__nv_bfloat16> &r) {
    r.u = *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ void ldraw(const float *p, Raw8<float> &r) {
    r.a = reinterpret_cast<const float4 *>(p)[0];
    r.b = reinterpret_cast<const float4 *>(p)[1];
}
__device__ __forceinline__ void cvt8(const Raw8<__nv_bfloat16> &r, float *v) {
    const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&r.u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(e[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void cvt8(const Raw8<float> &r, float *v) {
    v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w; v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float *v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float *p, const float *v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// logistic function with the fast exponential and divide (relative error ~1e-6, far inside the
// fp32 tolerance; 1/inf = 0 gives the right limit for very negative arguments)
__device__ __forceinline__ float sig(float v) { return __fdividef(1.f, 1.f + __expf(-v)); }
// for bf16 data, whose own rounding is 2^-9: (1 + tanh(v/2)) / 2 through one tanh.approx
// (relative error ~2^-11) instead of an exponential and a reciprocal
template <typename T>
__device__ __forceinline__ float sig_t(float v) {
    if (sizeof(T) == 2) {
        float t;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * v));
        return fmaf(0.5f, t, 0.5f);
    }
    return sig(v);
}

struct NormArgs {
    int64_t rows, width, G;   // G = features per group
    int ng;                   // groups per row
    float eps;
    const void *y, *z, *dout;
    int64_t sy, sz, sdout;
    const float *w, *rstd_in;
    void *out, *dy, *dz;
    int64_t sout, sdy, sdz;
    float *rstd;
    float *partials;          // [row chunk][width] (backward)
    int64_t rows_per_chunk;
    int ln, bg;               // LayerNorm (subtract the group mean); gate applied after the norm
};

template <typename T>
__global__ void __launch_bounds__(NW * 32)
k_norm_fwd(const NormArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t items = a.rows * a.ng, nw = (int64_t)gridDim.x * NW;
    const int pieces = (int)(a.G / 8);
    for (int64_t it = (int64_t)blockIdx.x * NW + (threadIdx.x >> 5); it < items; it += nw) {
        const int64_t r = it / a.ng;
        const int g = (int)(it - r * a.ng);
        const T *yr = static_cast<const T *>(a.y) + r * a.sy + (int64_t)g * a.G;
        const T *zr = a.z ? static_cast<const T *>(a.z) + r * a.sz + (int64_t)g * a.G : nullptr;
        // u of piece j (each pass re-reads the lines the warp just read: cache hits)
        auto load_u = [&](int j, float (&u)[8]) {
            load8(yr + 8 * j, u);
            if (zr && !a.bg) {
                float zz[8];
                load8(zr + 8 * j, zz);
#pragma unroll
                for (int e = 0; e < 8; ++e) u[e] *= zz[e] * sig_t<T>(zz[e]);
            }
        };
        float mu = 0.f;
        if (a.ln) {
            float ls = 0.f;
            for (int j = lane; j < pieces; j += 32) {
                float u[8];
                load_u(j, u);
#pragma unroll
                for (int e = 0; e < 8; ++e) ls += u[e];
            }
            mu = warp_sum(ls) / (float)a.G;
        }
        float ss = 0.f;
        for (int j = lane; j < pieces; j += 32) {
            float u[8];
            load_u(j, u);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float c = u[e] - mu;
                ss = fmaf(c, c, ss);
            }
        }
        ss = warp_sum(ss);
        const float rs = 1.f / sqrtf(ss / (float)a.G + a.eps);
        if (lane == 0) a.rstd[r * a.ng + g] = rs;
        T *orow = static_cast<T *>(a.out) + r * a.sout + (int64_t)g * a.G;
        const float *wr = a.w + (int64_t)g * a.G;
        for (int j = lane; j < pieces; j += 32) {
            float u[8], wv[8];
            load_u(j, u);
            load8(wr + 8 * j, wv);
            if (zr && a.bg) {
                float zz[8];
                load8(zr + 8 * j, zz);
#pragma unroll
                for (int e = 0; e < 8; ++e) wv[e] *= zz[e] * sig_t<T>(zz[e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] = (u[e] - mu) * rs * wv[e];
            store8(orow + 8 * j, u);
        }
    }
}

// grid (row chunks, groups), NW warps: warp w takes rows chunk_start + w, + NW, ...; its share
// of dw for the group's columns accumulates in its own shared-memory row, the rows are summed
// in warp order at the end, and k_norm_dw sums the row chunks in a fixed order.
template <typename T>
__global__ void __launch_bounds__(NW * 32)
k_norm_bwd(const NormArgs a) {
    extern __shared__ float acc[];   // [NW][G]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.y;
    const int pieces = (int)(a.G / 8);
    float *mine = acc + (int64_t)warp * a.G;
    for (int64_t i = lane; i < a.G; i += 32) mine[i] = 0.f;
    const int64_t r0 = (int64_t)blockIdx.x * a.rows_per_chunk, r1 = std::min(a.rows, r0 + a.rows_per_chunk);
    const float *wr = a.w + (int64_t)g * a.G;
    for (int64_t r = r0 + warp; r < r1; r += NW) {
        const T *yr = static_cast<const T *>(a.y) + r * a.sy + (int64_t)g * a.G;
        const T *zr = a.z ? static_cast<const T *>(a.z) + r * a.sz + (int64_t)g * a.G : nullptr;
        const T *dr = static_cast<const T *>(a.dout) + r * a.sdout + (int64_t)g * a.G;
        const float rs = a.rstd_in[r * a.ng + g];
        // piece j: y, the gate s = silu(z) and sigma(z), dout, w (re-read by each pass: cache hits)
        auto load_piece = [&](int j, float (&y8)[8], float (&sg)[8], float (&sgate)[8], float (&z8)[8]) {
            load8(yr + 8 * j, y8);
            if (zr) {
                load8(zr + 8 * j, z8);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sg[e] = sig_t<T>(z8[e]);
                    sgate[e] = z8[e] * sg[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) { sg[e] = 0.f; sgate[e] = 1.f; z8[e] = 0.f; }
            }
        };
        float mu = 0.f;
        if (a.ln) {
            float ls = 0.f;
            for (int j = lane; j < pieces; j += 32) {
                float y8[8], sg[8], sgate[8], z8[8];
                load_piece(j, y8, sg, sgate, z8);
#pragma unroll
                for (int e = 0; e < 8; ++e) ls += a.bg ? y8[e] : y8[e] * sgate[e];
            }
            mu = warp_sum(ls) / (float)a.G;
        }
        float dot = 0.f, gs = 0.f;   // sums over the group of g x_hat and of g, g = d out / d x_hat
        for (int j = lane; j < pieces; j += 32) {
            float y8[8], sg[8], sgate[8], z8[8], d[8], wv[8];
            load_piece(j, y8, sg, sgate, z8);
            load8(dr + 8 * j, d);
            load8(wr + 8 * j, wv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xh = ((a.bg ? y8[e] : y8[e] * sgate[e]) - mu) * rs;
                const float gw = a.bg ? d[e] * wv[e] * sgate[e] : d[e] * wv[e];
                dot = fmaf(gw, xh, dot);
                gs += gw;
            }
        }
        dot = warp_sum(dot) / (float)a.G;
        gs = a.ln ? warp_sum(gs) / (float)a.G : 0.f;
        T *dyr = static_cast<T *>(a.dy) + r * a.sdy + (int64_t)g * a.G;
        T *dzr = a.z ? static_cast<T *>(a.dz) + r * a.sdz + (int64_t)g * a.G : nullptr;
        for (int j = lane; j < pieces; j += 32) {
            float y8[8], sg[8], sgate[8], z8[8], d[8], wv[8];
            load_piece(j, y8, sg, sgate, z8);
            load8(dr + 8 * j, d);
            load8(wr + 8 * j, wv);
            float o1[8], o2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float xh = ((a.bg ? y8[e] : y8[e] * sgate[e]) - mu) * rs;
                const float gw = a.bg ? d[e] * wv[e] * sgate[e] : d[e] * wv[e];
                const float du = rs * (gw - gs - xh * dot);                  // d out / d u
                const float dsilu = sg[e] * (1.f + z8[e] * (1.f - sg[e]));    // silu'(z)
                o1[e] = a.bg ? du : du * sgate[e];                                          // dy
                o2[e] = a.bg ? d[e] * wv[e] * xh * dsilu : du * y8[e] * dsilu;              // dz
                mine[8 * j + e] += d[e] * (a.bg ? xh * sgate[e] : xh);                      // dw share
            }
            store8(dyr + 8 * j, o1);
            if (zr) store8(dzr + 8 * j, o2);
        }
    }
    __syncthreads();
    float *dst = a.partials + (int64_t)blockIdx.x * a.width + (int64_t)g * a.G;
    for (int64_t i = threadIdx.x; i < a.G; i += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < NW; ++w) s += acc[(int64_t)w * a.G + i];
        dst[i] = s;
    }
}

// Register-resident variants for groups of at most 32 * PPL * 8 features: a lane keeps its PPL
// pieces of y (and z, dout) in registers, so every load of a row is issued at once and nothing is
// read twice; in the backward the lane's slice of w and of the dw sums stay in registers too.
// GEN = false compiles the default mode only (RMS, the gate first); true reads a.ln and a.bg.
template <typename T, int PPL, bool GEN>
__global__ void __launch_bounds__(NW * 32)
k_norm_fwd_reg(const NormArgs a) {
    const bool ln = GEN && a.ln, bg = GEN && a.bg;
    const int lane = threadIdx.x & 31;
    const int64_t items = a.rows * a.ng, nw = (int64_t)gridDim.x * NW;
    const int pieces = (int)(a.G / 8);
    const bool hasz = a.z != nullptr;
    // y and z of an item are loaded one item ahead (raw bits), so a warp's loads stay in flight
    // while it normalises the current item
    Raw8<T> ry[PPL], rz[PPL];
    auto fetch = [&](int64_t it2) {
        const int64_t r2 = it2 / a.ng;
        const int g2 = (int)(it2 - r2 * a.ng);
        const T *y2 = static_cast<const T *>(a.y) + r2 * a.sy + (int64_t)g2 * a.G;
        const T *z2 = hasz ? static_cast<const T *>(a.z) + r2 * a.sz + (int64_t)g2 * a.G : nullptr;
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            const int j = lane + 32 * k;
            if (j < pieces) {
                ldraw(y2 + 8 * j, ry[k]);
                if (hasz) ldraw(z2 + 8 * j, rz[k]);
            }
        }
    };
    const int64_t first = (int64_t)blockIdx.x * NW + (threadIdx.x >> 5);
    if (first < items) fetch(first);
    for (int64_t it = first; it < items; it += nw) {
        const int64_t r = it / a.ng;
        const int g = (int)(it - r * a.ng);
        float v[PPL][8], zz[PPL][8];
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            if (lane + 32 * k < pieces) {
                cvt8(ry[k], v[k]);
                if (hasz) cvt8(rz[k], zz[k]);
            }
        }
        if (it + nw < items) fetch(it + nw);
        // u in place: the gate multiplies now unless it comes after the norm
        if (hasz && !bg) {
#pragma unroll
            for (int k = 0; k < PPL; ++k)
                if (lane + 32 * k < pieces)
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[k][e] *= zz[k][e] * sig_t<T>(zz[k][e]);
        }
        float mu = 0.f;
        if (ln) {
            float ls = 0.f;
#pragma unroll
            for (int k = 0; k < PPL; ++k)
                if (lane + 32 * k < pieces)
#pragma unroll
                    for (int e = 0; e < 8; ++e) ls += v[k][e];
            mu = warp_sum(ls) / (float)a.G;
        }
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            if (lane + 32 * k < pieces) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float c = v[k][e] - mu;
                    ss = fmaf(c, c, ss);
                }
            }
        }
        ss = warp_sum(ss);
        const float rs = 1.f / sqrtf(ss / (float)a.G + a.eps);
        if (lane == 0) a.rstd[r * a.ng + g] = rs;
        T *orow = static_cast<T *>(a.out) + r * a.sout + (int64_t)g * a.G;
        const float *wr = a.w + (int64_t)g * a.G;
#pragma unroll
        for (int k = 0; k < PPL; ++k) {
            const int j = lane + 32 * k;
            if (j < pieces) {
                float wv[8];
                load8(wr + 8 * j, wv);
                if (hasz && bg)
#pragma unroll
                    for (int e = 0; e < 8; ++e) wv[e] *= zz[k][e] * sig_t<T>(zz[k][e]);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[k][e] = (v[k][e] - mu) * rs * wv[e];
                store8(orow + 8 * j, v[k]);
            }
        }
    }
}

// The backward of one (row, group) from a lane's PPL pieces of y, z, dout and w held in
// registers (the warp holds the row): dy, dz stored, the dw shares accumulated.
template <typename T, int PPL, bool GEN>
__device__ __forceinline__ void bwd_row(const NormArgs &a, int lane, int pieces, bool hasz, float rs,
                                        const float (&y8)[PPL][8], const float (&z8)[PPL][8],
                                        const float (&d)[PPL][8], const float (&wv)[PPL][8], float (&dw)[PPL][8],
                                        T *dyr, T *dzr) {
    const bool ln = GEN && a.ln, bg = GEN && a.bg;
    float mu = 0.f;
    if (ln) {
        float ls = 0.f;
#pragma unroll
        for (int k = 0; k < PPL; ++k)
            if (lane + 32 * k < pieces)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    ls += (hasz && !bg) ? y8[k][e] * (z8[k][e] * sig_t<T>(z8[k][e])) : y8[k][e];
        mu = warp_sum(ls) / (float)a.G;
    }
    float dot = 0.f, gs = 0.f;   // sums over the group of g x_hat and of g, g = d out / d x_hat
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        if (lane + 32 * k < pieces) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float sgate = hasz ? z8[k][e] * sig_t<T>(z8[k][e]) : 1.f;
                const float xh = ((bg ? y8[k][e] : y8[k][e] * sgate) - mu) * rs;
                const float gw = bg ? d[k][e] * wv[k][e] * sgate : d[k][e] * wv[k][e];
                dot = fmaf(gw, xh, dot);
                if (ln) gs += gw;
            }
        }
    }
    dot = warp_sum(dot) / (float)a.G;
    gs = ln ? warp_sum(gs) / (float)a.G : 0.f;
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const int j = lane + 32 * k;
        if (j < pieces) {
            float o1[8], o2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float sg = hasz ? sig_t<T>(z8[k][e]) : 0.f;
                const float sgate = hasz ? z8[k][e] * sg : 1.f;
                const float xh = ((bg ? y8[k][e] : y8[k][e] * sgate) - mu) * rs;
                const float gw = bg ? d[k][e] * wv[k][e] * sgate : d[k][e] * wv[k][e];
                const float du = rs * (gw - gs - xh * dot);                     // d out / d u
                const float dsilu = sg * (1.f + z8[k][e] * (1.f - sg));         // silu'(z)
                o1[e] = bg ? du : du * sgate;                                                    // dy
                o2[e] = hasz ? (bg ? d[k][e] * wv[k][e] * xh * dsilu : du * y8[k][e] * dsilu) : 0.f;  // dz
                dw[k][e] = fmaf(d[k][e], bg ? xh * sgate : xh, dw[k][e]);                       // dw share
            }
            store8(dyr + 8 * j, o1);
            if (hasz) store8(dzr + 8 * j, o2);
        }
    }
}

// Backward with the rows staged in shared memory: a block takes its row chunk of one group in
// batches of NW rows (one per warp); each warp copies y, z and dout of its row of the next batch
// by cp.async (double-buffered) while it computes the current one, so the loads in flight do
// not depend on how many warps the registers allow.  A lane keeps its slice of w and of the dw sums in
// registers; the block's dw rows are summed in warp order at the end, as in the kernels above.
__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
template <typename T, int PPL, bool GEN>
__global__ void __launch_bounds__(NW * 32)
k_norm_bwd_staged(const NormArgs a) {
    extern __shared__ __align__(16) uint8_t nsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.y;
    const int G = (int)a.G, pieces = G / 8;
    const int cpr = G * (int)sizeof(T) / 16;                  // 16-byte pieces per row
    const int ntens = a.z ? 3 : 2;                            // y, dout, z
    T *stage = reinterpret_cast<T *>(nsm);                    // [2][ntens][NW][G]
    const int64_t r0 = (int64_t)blockIdx.x * a.rows_per_chunk, r1 = std::min(a.rows, r0 + a.rows_per_chunk);
    const float *wr = a.w + (int64_t)g * G;
    float wv[PPL][8], dw[PPL][8];
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const int j = lane + 32 * k;
#pragma unroll
        for (int e = 0; e < 8; ++e) { dw[k][e] = 0.f; wv[k][e] = 0.f; }
        if (j < pieces) load8(wr + 8 * j, wv[k]);
    }
    auto tile = [&](int buf, int t, int rw) { return stage + (((int64_t)buf * 3 + t) * NW + rw) * G; };
    // Each warp stages the row it computes (y, dout, z of row rb + warp): the copies and the
    // reads of a row stay within one warp, so a warp barrier orders them.
    auto issue = [&](int64_t rb, int buf) {
        const int64_t r = rb + warp;
        if (r < r1) {
            const T *src[3] = {static_cast<const T *>(a.y) + r * a.sy + (int64_t)g * G,
                               static_cast<const T *>(a.dout) + r * a.sdout + (int64_t)g * G,
                               a.z ? static_cast<const T *>(a.z) + r * a.sz + (int64_t)g * G : nullptr};
            for (int t = 0; t < ntens; ++t) {
                uint8_t *dst = reinterpret_cast<uint8_t *>(tile(buf, t, warp));
                const uint8_t *sp = reinterpret_cast<const uint8_t *>(src[t]);
                for (int q = lane; q < cpr; q += 32) cp16(dst + 16 * q, sp + 16 * q);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    int buf = 0;
    if (r0 < r1) issue(r0, 0);
    for (int64_t rb = r0; rb < r1; rb += NW, buf ^= 1) {
        if (rb + NW < r1) {
            issue(rb + NW, buf ^ 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncwarp();
        const int64_t r = rb + warp;
        if (r < r1) {
            const T *ys = tile(buf, 0, warp), *ds = tile(buf, 1, warp), *zs = a.z ? tile(buf, 2, warp) : nullptr;
            float y8[PPL][8], z8[PPL][8] = {}, d[PPL][8];
#pragma unroll
            for (int k = 0; k < PPL; ++k) {
                const int j = lane + 32 * k;
                if (j < pieces) {
                    load8(ys + 8 * j, y8[k]);
                    load8(ds + 8 * j, d[k]);
                    if (zs) load8(zs + 8 * j, z8[k]);
                }
            }
            const float rs = a.rstd_in[r * a.ng + g];
            T *dyr = static_cast<T *>(a.dy) + r * a.sdy + (int64_t)g * G;
            T *dzr = a.z ? static_cast<T *>(a.dz) + r * a.sdz + (int64_t)g * G : nullptr;
            bwd_row<T, PPL, GEN>(a, lane, pieces, zs != nullptr, rs, y8, z8, d, wv, dw, dyr, dzr);
        }
        __syncwarp();   // this warp's reads of the buffer precede its refill at the next step
    }
    __syncthreads();   // every warp is done with the stage before it becomes the dw rows
    float *acc = reinterpret_cast<float *>(nsm);   // [NW][G], over the (now idle) stage
    float *mine = acc + (int64_t)warp * G;
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
        const int j = lane + 32 * k;
        if (j < pieces)
#pragma unroll
            for (int e = 0; e < 8; ++e) mine[8 * j + e] = dw[k][e];
    }
    __syncthreads();
    float *dst = a.partials + (int64_t)blockIdx.x * a.width + (int64_t)g * G;
    for (int i = threadIdx.x; i < G; i += NW * 32) {
        float sum = 0.f;
        for (int q = 0; q < NW; ++q) sum += acc[(int64_t)q * G + i];
        dst[i] = sum;
    }
}
template <typename T>
size_t staged_smem(int64_t G) {
    const size_t stage = (size_t)2 * 3 * NW * (size_t)G * sizeof(T);
    const size_t red = (size_t)NW * (size_t)G * sizeof(float);
    return stage > red ? stage : red;
}

// dw: the column sums of the per-chunk shares [chunks][width] in a fixed order.  A block takes
// 32 columns; warp w sums chunks w, w + 8, ... in ascending order (four loads in flight), and the
// eight warp sums are added in warp order, so the result is bitwise reproducible.
__global__ void __launch_bounds__(256) k_norm_dw(const float *partials, int64_t chunks, int64_t width, float *dw) {
    __shared__ float red[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t i = (int64_t)blockIdx.x * 32 + lane;
    float s = 0.f;
    if (i < width) {
        const float *col = partials + i;
        int64_t c = w;
        for (; c + 24 < chunks; c += 32) {
            const float a0 = col[c * width], a1 = col[(c + 8) * width], a2 = col[(c + 16) * width],
                        a3 = col[(c + 24) * width];
            s += a0;
            s += a1;
            s += a2;
            s += a3;
        }
        for (; c < chunks; c += 8) s += col[c * width];
    }
    red[w][lane] = s;
    __syncthreads();
    if (w == 0 && i < width) {
        float tot = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) tot += red[q][lane];
        dw[i] = tot;
    }
}

template <typename K>
cudaError_t launch_one(K kernel, const NormArgs &a, dim3 grid, size_t smem, cudaStream_t st, int *attr) {
    cudaError_t e = ensure_smem_attr(kernel, (int)smem, attr);
    if (e == cudaSuccess) kernel<<<grid, NW * 32, smem, st>>>(a);
    return e;
}
template <typename T, bool GEN>
cudaError_t launch_norm_bwd_g(const NormArgs &a, int64_t ppl, dim3 grid, size_t smem, cudaStream_t st) {
    static int attr[4][64] = {};
    const size_t ssm = staged_smem<T>(a.G);
    if (ppl <= 1) return launch_one(k_norm_bwd_staged<T, 1, GEN>, a, grid, ssm, st, attr[0]);
    if (ppl <= 2) return launch_one(k_norm_bwd_staged<T, 2, GEN>, a, grid, ssm, st, attr[1]);
    if (ppl <= 4) return launch_one(k_norm_bwd_staged<T, 4, GEN>, a, grid, ssm, st, attr[2]);
    return launch_one(k_norm_bwd<T>, a, grid, smem, st, attr[3]);
}
template <typename T>
cudaError_t launch_norm_bwd(const NormArgs &a, int64_t ppl, dim3 grid, size_t smem, cudaStream_t st) {
    return (a.ln || a.bg) ? launch_norm_bwd_g<T, true>(a, ppl, grid, smem, st)
                          : launch_norm_bwd_g<T, false>(a, ppl, grid, smem, st);
}
// The grid-stride kernels run one wave: at most the blocks that are resident at once (the
// occupancy of the instantiation at hand times the SMs), so no block waits for a free SM.
template <typename K>
void launch_wave(K kernel, const NormArgs &a, int blocks, int sms, cudaStream_t st) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, NW * 32, 0) == cudaSuccess && per_sm > 0)
        blocks = std::min(blocks, per_sm * sms);
    kernel<<<blocks, NW * 32, 0, st>>>(a);
}
template <typename T, bool GEN>
void launch_norm_fwd_g(const NormArgs &a, int64_t ppl, int blocks, int sms, cudaStream_t st) {
    if (ppl <= 1) launch_wave(k_norm_fwd_reg<T, 1, GEN>, a, blocks, sms, st);
    else if (ppl <= 2) launch_wave(k_norm_fwd_reg<T, 2, GEN>, a, blocks, sms, st);
    else if (ppl <= 4) launch_wave(k_norm_fwd_reg<T, 4, GEN>, a, blocks, sms, st);
    else launch_wave(k_norm_fwd<T>, a, blocks, sms, st);
}
template <typename T>
void launch_norm_fwd(const NormArgs &a, int64_t ppl, int blocks, int sms, cudaStream_t st) {
    if (a.ln || a.bg) launch_norm_fwd_g<T, true>(a, ppl, blocks, sms, st);
    else launch_norm_fwd_g<T, false>(a, ppl, blocks, sms, st);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

bool aligned16(const void *p) { return ((uintptr_t)p) % 16 == 0; }

// Shared checks of both directions; *chunks = the backward's row chunks: two blocks per SM
// over all groups (one resident wave of the staged backward, about 120 registers a thread).
ssd_status check_norm(const ssd_norm_problem *p, int64_t *chunks) {
    if (p == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    if (p->rows < 0 || p->width < 1 || p->group_size < 1 || p->width % p->group_size != 0)
        return SSD_ERR_INVALID_ARGUMENT;
    if (!(p->eps >= 0.f) || p->dtype < SSD_F32 || p->dtype > SSD_BF16 ||
        (p->flags & ~(SSD_NORM_LAYER | SSD_NORM_GATE_AFTER)) != 0)
        return SSD_ERR_INVALID_ARGUMENT;
    if (p->group_size % 8 != 0 || p->group_size > kMaxGroup || p->rows > ((int64_t)1 << 31) ||
        p->width > ((int64_t)1 << 24))
        return SSD_ERR_UNSUPPORTED;
    const int64_t ng = p->width / p->group_size;
    const int64_t want = std::max<int64_t>(1, (2 * (int64_t)sm_count() + ng - 1) / ng);
    *chunks = std::max<int64_t>(1, std::min<int64_t>(p->rows, want));
    return SSD_OK;
}

// A row-major [rows, width] tensor with element row stride `stride`.
ssd_status check_rows(const ssd_norm_problem *p, const void *t, int64_t stride, bool required) {
    if (t == nullptr) return required && p->rows > 0 ? SSD_ERR_INVALID_ARGUMENT : SSD_OK;
    if (p->rows > 1 && stride < p->width) return SSD_ERR_INVALID_ARGUMENT;
    if (!aligned16(t) || stride % 8 != 0) return SSD_ERR_MISALIGNED;
    return SSD_OK;
}

#define NORM_TRY(expr)                 \
    do {                               \
        ssd_status _s = (expr);        \
        if (_s != SSD_OK) return _s;   \
    } while (0)

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status ssd_gated_norm_fwd(const ssd_norm_problem *p, const void *y, int64_t y_stride, const void *z,
                              int64_t z_stride, const float *weight, void *out, int64_t out_stride, float *rstd,
                              void *stream) {
    int64_t chunks = 0;
    NORM_TRY(check_norm(p, &chunks));
    NORM_TRY(check_rows(p, y, y_stride, true));
    NORM_TRY(check_rows(p, z, z_stride, false));
    NORM_TRY(check_rows(p, out, out_stride, true));
    if (p->rows > 0 && (weight == nullptr || rstd == nullptr)) return SSD_ERR_INVALID_ARGUMENT;
    if (weight != nullptr && !aligned16(weight)) return SSD_ERR_MISALIGNED;
    if (p->rows == 0) return SSD_OK;
    NormArgs a{};
    a.rows = p->rows; a.width = p->width; a.G = p->group_size; a.ng = (int)(p->width / p->group_size);
    a.eps = p->eps; a.y = y; a.z = z; a.sy = y_stride; a.sz = z_stride; a.w = weight; a.out = out;
    a.sout = out_stride; a.rstd = rstd;
    a.ln = (p->flags & SSD_NORM_LAYER) != 0; a.bg = (p->flags & SSD_NORM_GATE_AFTER) != 0;
    const int64_t items = p->rows * a.ng;
    const int sms = sm_count();
    const int blocks = (int)std::min<int64_t>((items + NW - 1) / NW, 8LL * sms);
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t ppl = (p->group_size / 8 + 31) / 32;   // pieces per lane
    if (p->dtype == SSD_BF16) launch_norm_fwd<__nv_bfloat16>(a, ppl, blocks, sms, st);
    else launch_norm_fwd<float>(a, ppl, blocks, sms, st);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_gated_norm_bwd_workspace_size(const ssd_norm_problem *p, size_t *bytes) {
    if (bytes == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    int64_t chunks = 0;
    NORM_TRY(check_norm(p, &chunks));
    *bytes = (size_t)chunks * (size_t)p->width * sizeof(float);
    return SSD_OK;
}

ssd_status ssd_gated_norm_bwd(const ssd_norm_problem *p, const void *y, int64_t y_stride, const void *z,
                              int64_t z_stride, const float *weight, const float *rstd, const void *dout,
                              int64_t dout_stride, void *dy, int64_t dy_stride, void *dz, int64_t dz_stride,
                              float *dweight, void *workspace, size_t workspace_bytes, void *stream) {
    int64_t chunks = 0;
    NORM_TRY(check_norm(p, &chunks));
    NORM_TRY(check_rows(p, y, y_stride, true));
    NORM_TRY(check_rows(p, z, z_stride, false));
    NORM_TRY(check_rows(p, dout, dout_stride, true));
    NORM_TRY(check_rows(p, dy, dy_stride, true));
    NORM_TRY(check_rows(p, dz, dz_stride, z != nullptr));
    if (weight == nullptr || dweight == nullptr || (p->rows > 0 && rstd == nullptr)) return SSD_ERR_INVALID_ARGUMENT;
    if (!aligned16(weight)) return SSD_ERR_MISALIGNED;
    const size_t need = (size_t)chunks * (size_t)p->width * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need) return SSD_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = (cudaStream_t)stream;
    NormArgs a{};
    a.rows = p->rows; a.width = p->width; a.G = p->group_size; a.ng = (int)(p->width / p->group_size);
    a.eps = p->eps; a.y = y; a.z = z; a.dout = dout; a.sy = y_stride; a.sz = z_stride; a.sdout = dout_stride;
    a.w = weight; a.rstd_in = rstd; a.dy = dy; a.dz = dz; a.sdy = dy_stride; a.sdz = dz_stride;
    a.partials = static_cast<float *>(workspace);
    a.ln = (p->flags & SSD_NORM_LAYER) != 0; a.bg = (p->flags & SSD_NORM_GATE_AFTER) != 0;
    a.rows_per_chunk = p->rows > 0 ? (p->rows + chunks - 1) / chunks : 1;
    const size_t smem = (size_t)NW * (size_t)p->group_size * sizeof(float);
    const dim3 grid((unsigned)chunks, (unsigned)a.ng);
    const int64_t ppl = (p->group_size / 8 + 31) / 32;   // pieces per lane
    cudaError_t e;
    if (p->dtype == SSD_BF16)
        e = launch_norm_bwd<__nv_bfloat16>(a, ppl, grid, smem, st);
    else
        e = launch_norm_bwd<float>(a, ppl, grid, smem, st);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    k_norm_dw<<<(unsigned)((p->width + 31) / 32), 256, 0, st>>>(a.partials, chunks, p->width, dweight);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
