// bwd_tc.cu -- tensor-core backward of the SSD chunked scan (bf16 inputs, fp32
// accumulation), headdim 64, dstate 128, chunk 128.
//
// Recompute-based, as the Mamba-3-Lite "SSD Reference" page's section "6. The
// autograd backward contract" prescribes (re-run the forward math, inject the true
// upstream gradients).  Per chunk c of a sequence and head h, with
//   E[l][s] = exp(cs[l] - cs[s]) 1[s<=l], CB = C B^T, dyp = dy silu(z), dM = dyp x^T,
//   M = E dt_s CB, E' = E dt_s dM, w_s = dt_s exp(cs[Q-1] - cs[s]), e_l = exp(cs[l]),
//   S_in = carried state entering the chunk, dS = gradient of the state leaving it:
//     dx = M^T dyp + w o (B dS^T) + D dyp
//     dB = E'^T C + (w o x) dS            (this head's share; summed over the group later)
//     dC = E' B + (e o dyp) S_in
//     ddt[s] = sum_l E CB dM [l][s] + exp(cs[Q-1]-cs[s]) x[s].(B dS^T)[s] + A da[s]
//     da[u] = sum_{i>=u} dcs[i],
//     dcs[i] = sum_s (M o dM)[i][s] - sum_l (M o dM)[l][i] + dyp[i].(e_i C S_in^T)[i] - T4[i]
//              + [i = Q-1](exp(cs[Q-1]) <S_in, dS> + sum_s T4[s]),  T4[s] = w_s x[s].(B dS^T)[s]
//     dz = dy ypre silu'(z),  ypre = M x + e o (C S_in^T) + D x
// k_bwd_dstates computes the per-chunk state gradient source
//     dS_loc[p][n] = sum_l e_l dyp[l][p] C[l][n]
// which the reverse warp-shuffle scan turns into dS for every chunk.
// All contractions run as tcgen05.mma chains on 128-byte-swizzled shared-memory
// tiles (TMA for x, B, C and the bf16 carried states); reductions are fixed-order.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace ssd {

namespace {

using namespace tc;

constexpr int QT = 128, PT = 64, NT = 128;
constexpr uint32_t X_BYTES = QT * PT * 2;    // 16 KB
constexpr uint32_t BC_BYTES = QT * NT * 2;   // 32 KB
constexpr uint32_t S_BYTES = PT * NT * 2;    // 16 KB
constexpr float LOG2E = 1.4426950408889634f;

struct BwdParams {
    Shape sh;
    const int32_t *hdr;
    const ChunkInfo *chunks;
    const float *dt_raw;
    int64_t sdb, sdl;
    const float *A, *D, *bias;
    const __nv_bfloat16 *dy, *z;
    int64_t sdyb, sdyl, sdyh, szb, szl, szh;
    __nv_bfloat16 *dx, *dz;
    int64_t sdxb, sdxl, sdxh, sdzb, sdzl, sdzh;
    float *ddt;
    int64_t sddb, sddl;
    const float *dS;         // [chunk][H][P][N] fp32: gradient of the state leaving the chunk
    float *dS_loc;           // [chunk][H][P][N] fp32 (dstates kernel output)
    float *chunk_lam;        // [chunk][H] total log-decay of the chunk (dstates kernel output)
    float *dBh, *dCh;        // [chunk][H][Q][N] fp32 per-head shares
    float *partials;         // [chunk][H][4]: dA, dD, ddt_bias shares
};

__device__ __forceinline__ uint64_t kmaj(uint32_t base, int k, uint32_t col_bytes) {
    return sdesc(base + (uint32_t)(k >> 2) * col_bytes + (uint32_t)(k & 3) * 32u, 16u, 1024u);
}
// MN-major operand with K rows of 128 B; `mn_atom` = byte distance between 64-wide MN atoms.
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int k, uint32_t mn_atom) {
    return sdesc(base + (uint32_t)k * 2048u, mn_atom, 1024u);
}
__device__ __forceinline__ float silu_f(float z) { return z * rcp(1.f + ex2(-z * LOG2E)); }
__device__ __forceinline__ float sig_f(float z) { return rcp(1.f + ex2(-z * LOG2E)); }

// Loads 32 bf16 (64 bytes) of a row into floats.
__device__ __forceinline__ void load_row32(const __nv_bfloat16 *src, float *v) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u = __ldg(s + q);
        const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(e[i]);
            v[q * 8 + 2 * i] = f.x;
            v[q * 8 + 2 * i + 1] = f.y;
        }
    }
}
// Writes 32 floats as bf16 into the 4 chunks (4*hf .. 4*hf+3) of a 128-byte swizzled row.
__device__ __forceinline__ void store_row32_swz(uint8_t *row_base, int row, int hf, const float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = (4 * hf + q) ^ (row & 7);
        *reinterpret_cast<uint4 *>(row_base + c * 16) =
            make_uint4(pack_bf16(v[q * 8], v[q * 8 + 1]), pack_bf16(v[q * 8 + 2], v[q * 8 + 3]),
                       pack_bf16(v[q * 8 + 4], v[q * 8 + 5]), pack_bf16(v[q * 8 + 6], v[q * 8 + 7]));
    }
}
__device__ __forceinline__ void load_row32_swz(const uint8_t *row_base, int row, int hf, float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = (4 * hf + q) ^ (row & 7);
        uint4 u = *reinterpret_cast<const uint4 *>(row_base + c * 16);
        const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(e[i]);
            v[q * 8 + 2 * i] = f.x;
            v[q * 8 + 2 * i + 1] = f.y;
        }
    }
}
// Column sums of a 32x32 block held one row per lane (v[i] = column i): after the
// call lane j holds the sum over the warp's 32 rows of column j (fixed order).
__device__ __forceinline__ float colsum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? v[i] : v[i + o];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = (upper ? v[i + o] : v[i]) + recv;
        }
    }
    return v[0];
}

__device__ __forceinline__ float block_scan256(float v, float *wsum, float *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float x = warp_incl_sum(v);
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    float off = 0.f, tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < w) off += wsum[i];
        tot += wsum[i];
    }
    *total = tot;
    __syncthreads();
    return x + off;
}

// dt and the in-chunk cumulative log-decay of (chunk, head) into smem (cs2 = cs*log2 e).
__device__ __forceinline__ float chunk_scan_dt(const BwdParams &p, const ChunkInfo &ci, int h, float *dtc,
                                               float *cs2, float *wsum) {
    const int tid = threadIdx.x;
    float dt = 0.f;
    if (tid < ci.len) {
        const float v = p.dt_raw[(int64_t)ci.b * p.sdb + (int64_t)(ci.t0 + tid) * p.sdl + h] + (p.bias ? p.bias[h] : 0.f);
        dt = softplus_f(v);
    }
    float tot;
    const float cs = block_scan256(tid < QT ? dt * p.A[h] : 0.f, wsum, &tot);
    if (tid < QT) {
        dtc[tid] = dt;
        cs2[tid] = cs * LOG2E;
    }
    __syncthreads();
    return tot;
}

// ------------------------------------------------------------------ dstates
// grid (kmax, H), 256 threads.  dS_loc^T[n][p] = sum_l C[l][n] (e o dyp)[l][p] on the
// tensor cores (A = C^T, M-major; B = e o dyp, N-major), written as fp32 [p][n].
constexpr uint32_t DS_OFF_C = 0, DS_OFF_Y = BC_BYTES, DS_OFF_MISC = BC_BYTES + X_BYTES;
constexpr uint32_t DS_SMEM = DS_OFF_MISC + 2048 + 1024;

__global__ void __launch_bounds__(256)
k_bwd_dstates_tc(const __grid_constant__ CUtensorMap tmC, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, hf = tid >> 7;
    const int k = blockIdx.x, h = blockIdx.y;
    if (k >= p.hdr[HDR_NCHUNKS] || p.hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = p.chunks[k];
    const int g = h / p.sh.hpg;
    float *dtc = reinterpret_cast<float *>(sm + DS_OFF_MISC);
    float *cs2 = dtc + QT;
    float *wsum = cs2 + QT;
    uint64_t *bar = reinterpret_cast<uint64_t *>(wsum + 8);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        mbar_expect_tx(&bar[0], BC_BYTES);
        tma_load_4d(sm + DS_OFF_C, &tmC, &bar[0], 0, g, ci.t0, ci.b);
        tma_load_4d(sm + DS_OFF_C + BC_BYTES / 2, &tmC, &bar[0], 64, g, ci.t0, ci.b);
    }
    if (warp == 0) tmem_alloc(tslot, 64);
    tc_fence_before();
    const float lam = chunk_scan_dt(p, ci, h, dtc, cs2, wsum);   // contains __syncthreads
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) p.chunk_lam[(int64_t)k * p.sh.H + h] = lam;
    // (e o dyp) row `row`, half hf -> swizzled [l][p] tile
    {
        float v[32];
        if (row < ci.len) {
            const int64_t tok = (int64_t)ci.t0 + row;
            float zz[32];
            load_row32(p.dy + (int64_t)ci.b * p.sdyb + tok * p.sdyl + (int64_t)h * p.sdyh + 32 * hf, v);
            const float el = ex2(cs2[row]);
            if (p.z) {
                load_row32(p.z + (int64_t)ci.b * p.szb + tok * p.szl + (int64_t)h * p.szh + 32 * hf, zz);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= silu_f(zz[i]) * el;
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= el;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        store_row32_swz(sm + DS_OFF_Y + row * 128, row, hf, v);
    }
    fence_proxy_async_smem();
    const bool ok = mbar_wait(&bar[0], 0);
    __syncthreads();
    if (ok && tid == 0) {
        tc_fence_after();
        const uint32_t sC = smem_u32(sm + DS_OFF_C), sY = smem_u32(sm + DS_OFF_Y);
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk)
            umma_bf16(tmem, mnmaj(sC, kk, BC_BYTES / 2), mnmaj(sY, kk, 16384u), idesc_bf16(128, 64, 1, 1), kk > 0);
        umma_commit(&bar[1]);
    }
    bool ok2 = ok && mbar_wait(&bar[1], 0);
    if (!ok || !ok2) set_status(const_cast<int32_t *>(p.hdr), SSD_ERR_DEVICE_TIMEOUT);
    tc_fence_after();
    if (ok2) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + 32 * hf, v);
        tmem_wait_ld();
        float *dst = p.dS_loc + ((int64_t)k * p.sh.H + h) * (PT * NT) + (int64_t)(32 * hf) * NT + row;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[(int64_t)i * NT] = v[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// ------------------------------------------------------------------ main backward chunk kernel
// smem map (1024-aligned offsets)
constexpr uint32_t O_X = 0;                        // x      [s][p]   16 KB (TMA)
constexpr uint32_t O_B = O_X + X_BYTES;            // B      [s][n]   32 KB (TMA)
constexpr uint32_t O_C = O_B + BC_BYTES;           // C      [l][n]   32 KB (TMA)
constexpr uint32_t O_SI = O_C + BC_BYTES;          // S_in   [p][n]   16 KB (TMA, bf16)
constexpr uint32_t O_DY = O_SI + S_BYTES;          // dyp, then e o dyp [l][p] 16 KB
constexpr uint32_t O_WX = O_DY + X_BYTES;          // w o x  [s][p]   16 KB
constexpr uint32_t O_M = O_WX + X_BYTES;           // M      [l][s]   32 KB
constexpr uint32_t O_E = O_M + BC_BYTES;           // E'     [l][s]   32 KB
constexpr uint32_t O_SD = O_E + BC_BYTES;          // dS     [p][n]   16 KB (bf16)
constexpr uint32_t O_MISC = O_SD + S_BYTES;
// misc floats
constexpr int F_CS2 = 0, F_DT = 128, F_W = 256, F_ROWT1 = 384, F_ROWXU = 640, F_ROWT2 = 896, F_ROWD = 1152,
              F_COLP = 1408, F_RED = 1920, F_WSUM = 1936, F_END = 1952;
constexpr uint32_t BWD_SMEM = O_MISC + F_END * 4 + 64 + 1024;

// TMEM columns
constexpr uint32_t T_CB = 0, T_DM = 128;                       // group 1
constexpr uint32_t T_DXD = 0, T_DXS = 64, T_DB = 128, T_DC = 256;  // group 2 (+ dC part 2 in group 3)
constexpr uint32_t T_YD = 384, T_YO = 448;                     // group 3

__global__ void __launch_bounds__(256, 1)
k_bwd_chunk_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmS, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, hf = tid >> 7, quad = warp & 3;
    const int lane = tid & 31;
    const int k = blockIdx.x, h = blockIdx.y;
    if (k >= p.hdr[HDR_NCHUNKS] || p.hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = p.chunks[k];
    const int g = h / p.sh.hpg;
    const int H = p.sh.H;
    float *fm = reinterpret_cast<float *>(sm + O_MISC);
    float *cs2 = fm + F_CS2, *dtc = fm + F_DT, *wst = fm + F_W;
    uint64_t *bar = reinterpret_cast<uint64_t *>(fm + F_END);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    __shared__ int s_abort;
    if (tid == 0) {
        s_abort = 0;
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        mbar_expect_tx(&bar[0], X_BYTES + 2 * BC_BYTES + S_BYTES);
        tma_load_4d(sm + O_X, &tmX, &bar[0], 0, h, ci.t0, ci.b);
        tma_load_4d(sm + O_B, &tmB, &bar[0], 0, g, ci.t0, ci.b);
        tma_load_4d(sm + O_B + BC_BYTES / 2, &tmB, &bar[0], 64, g, ci.t0, ci.b);
        tma_load_4d(sm + O_C, &tmC, &bar[0], 0, g, ci.t0, ci.b);
        tma_load_4d(sm + O_C + BC_BYTES / 2, &tmC, &bar[0], 64, g, ci.t0, ci.b);
        // S_in (bf16 [p][n]) of (chunk, head): rows p of the [chunk*H + h] slab
        const int slab = k * H + h;
        tma_load_4d(sm + O_SI, &tmS, &bar[0], 0, 0, slab * PT, 0);
        tma_load_4d(sm + O_SI + S_BYTES / 2, &tmS, &bar[0], 64, 0, slab * PT, 0);
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    const float lam = chunk_scan_dt(p, ci, h, dtc, cs2, fm + F_WSUM);   // syncs
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lb = (uint32_t)(quad * 32) << 16;
    const float cl2 = cs2[QT - 1];
    if (tid < QT) wst[tid] = dtc[tid] * ex2(cl2 - cs2[tid]);
    __syncthreads();
    const float Dh = p.D ? p.D[h] : 0.f;
    const float Ah = p.A[h];
    const int64_t tok = (int64_t)ci.t0 + row;
    const bool live = row < ci.len;
    uint32_t mma_phase = 0;
    auto wait_mma = [&]() {
        if (!mbar_wait(&bar[1], mma_phase & 1)) {
            s_abort = 1;
            set_status(const_cast<int32_t *>(p.hdr), SSD_ERR_DEVICE_TIMEOUT);
        }
        ++mma_phase;
        tc_fence_after();
    };
    // dyp rows -> smem; dS (fp32 -> bf16 [p][n]) -> smem; T3 partial
    float dyp[32];
    {
        if (live) {
            float zz[32];
            load_row32(p.dy + (int64_t)ci.b * p.sdyb + tok * p.sdyl + (int64_t)h * p.sdyh + 32 * hf, dyp);
            if (p.z) {
                load_row32(p.z + (int64_t)ci.b * p.szb + tok * p.szl + (int64_t)h * p.szh + 32 * hf, zz);
#pragma unroll
                for (int i = 0; i < 32; ++i) dyp[i] *= silu_f(zz[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) dyp[i] = 0.f;
        }
        store_row32_swz(sm + O_DY + row * 128, row, hf, dyp);
    }
    float t3p = 0.f;
    {
        const float *src = p.dS + ((int64_t)k * H + h) * (PT * NT) + (int64_t)(32 * hf) * NT + row;
        const int n = row, ac = n >> 6, cn = (n & 63) >> 3;
        uint8_t *base = sm + O_SD + ac * (S_BYTES / 2) + (n & 7) * 2;
        const uint8_t *sib = sm + O_SI + ac * (S_BYTES / 2) + (n & 7) * 2;
        float dsv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) dsv[i] = __ldg(src + (int64_t)i * NT);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int pp = 32 * hf + i;
            *reinterpret_cast<__nv_bfloat16 *>(base + pp * 128 + ((cn ^ (pp & 7)) << 4)) = __float2bfloat16_rn(dsv[i]);
        }
        const bool okS = mbar_wait(&bar[0], 0);   // S_in (and x, B, C) landed
        if (!okS) {
            s_abort = 1;
            set_status(const_cast<int32_t *>(p.hdr), SSD_ERR_DEVICE_TIMEOUT);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int pp = 32 * hf + i;
            t3p += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sib + pp * 128 + ((cn ^ (pp & 7)) << 4))) *
                   dsv[i];
        }
    }
    // w o x
    {
        float xv[32];
        load_row32_swz(sm + O_X + row * 128, row, hf, xv);
        const float wl = wst[row];
#pragma unroll
        for (int i = 0; i < 32; ++i) xv[i] *= wl;
        store_row32_swz(sm + O_WX + row * 128, row, hf, xv);
    }
    fence_proxy_async_smem();
    __syncthreads();
    const uint32_t sX = smem_u32(sm + O_X), sB = smem_u32(sm + O_B), sC = smem_u32(sm + O_C);
    const uint32_t sSI = smem_u32(sm + O_SI), sDY = smem_u32(sm + O_DY), sWX = smem_u32(sm + O_WX);
    const uint32_t sM = smem_u32(sm + O_M), sE = smem_u32(sm + O_E), sSD = smem_u32(sm + O_SD);
    if (!s_abort && tid == 0) {   // group 1: CB = C B^T, dM = dyp x^T
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < NT / 16; ++kk)
            umma_bf16(tmem + T_CB, kmaj(sC, kk, BC_BYTES / 2), kmaj(sB, kk, BC_BYTES / 2), idesc_bf16(128, 128, 0, 0),
                      kk > 0);
#pragma unroll
        for (int kk = 0; kk < PT / 16; ++kk)
            umma_bf16(tmem + T_DM, kmaj(sDY, kk, X_BYTES), kmaj(sX, kk, X_BYTES), idesc_bf16(128, 128, 0, 0), kk > 0);
        umma_commit(&bar[1]);
    }
    if (!s_abort) wait_mma();
    // ---- M, E' (bf16) rows; row sums of M o dM; column sums of E CB dM (fixed order)
    float rowt1 = 0.f;
    {
        const int l = row;
        const float c2l = cs2[l];
        float *colp = fm + F_COLP;   // [8 warps][64]
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
            const int sb = hf == 0 ? (bi == 0 ? 0 : 3) : (bi == 0 ? 1 : 2);
            uint32_t pm[16], pe[16];
            float tmv[32];
            if (sb <= quad && !s_abort) {
                float cb[32], dm[32];
                tmem_ld32(tmem + lb + T_CB + sb * 32, cb);
                tmem_ld32(tmem + lb + T_DM + sb * 32, dm);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float mv[2], ev[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int s = sb * 32 + i + j;
                        float m = 0.f, e = 0.f, t = 0.f;
                        if (s <= l) {
                            const float E = ex2(c2l - cs2[s]);
                            const float ec = E * cb[i + j];
                            m = ec * dtc[s];
                            e = E * dtc[s] * dm[i + j];
                            t = ec * dm[i + j];
                            rowt1 += m * dm[i + j];
                        }
                        mv[j] = m;
                        ev[j] = e;
                        tmv[i + j] = t;
                    }
                    pm[i >> 1] = pack_bf16(mv[0], mv[1]);
                    pe[i >> 1] = pack_bf16(ev[0], ev[1]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) { pm[i] = 0u; pe[i] = 0u; }
#pragma unroll
                for (int i = 0; i < 32; ++i) tmv[i] = 0.f;
            }
            const float cs_ = colsum32(tmv);
            colp[warp * 64 + bi * 32 + lane] = cs_;
            uint8_t *rm = sm + O_M + (sb >> 1) * (BC_BYTES / 2) + l * 128;
            uint8_t *re = sm + O_E + (sb >> 1) * (BC_BYTES / 2) + l * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int cidx = (((sb & 1) << 2) + q) ^ (l & 7);
                *reinterpret_cast<uint4 *>(rm + (cidx << 4)) = make_uint4(pm[4 * q], pm[4 * q + 1], pm[4 * q + 2], pm[4 * q + 3]);
                *reinterpret_cast<uint4 *>(re + (cidx << 4)) = make_uint4(pe[4 * q], pe[4 * q + 1], pe[4 * q + 2], pe[4 * q + 3]);
            }
        }
        fm[F_ROWT1 + hf * 128 + l] = rowt1;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (!s_abort && tid == 0) {   // group 2
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk)   // dx_diag[s][p] = sum_l M[l][s] dyp[l][p]
            umma_bf16(tmem + T_DXD, mnmaj(sM, kk, BC_BYTES / 2), mnmaj(sDY, kk, 16384u), idesc_bf16(128, 64, 1, 1),
                      kk > 0);
#pragma unroll
        for (int kk = 0; kk < NT / 16; ++kk)   // u[s][p] = sum_n B[s][n] dS[p][n]
            umma_bf16(tmem + T_DXS, kmaj(sB, kk, BC_BYTES / 2), kmaj(sSD, kk, S_BYTES / 2), idesc_bf16(128, 64, 0, 0),
                      kk > 0);
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk)   // dB[s][n] = sum_l E'[l][s] C[l][n]
            umma_bf16(tmem + T_DB, mnmaj(sE, kk, BC_BYTES / 2), mnmaj(sC, kk, BC_BYTES / 2),
                      idesc_bf16(128, 128, 1, 1), kk > 0);
#pragma unroll
        for (int kk = 0; kk < PT / 16; ++kk)   // dB[s][n] += sum_p (w o x)[s][p] dS[p][n]
            umma_bf16(tmem + T_DB, kmaj(sWX, kk, X_BYTES), mnmaj(sSD, kk, S_BYTES / 2),
                      idesc_bf16(128, 128, 0, 1), 1);
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk)   // dC[l][n] = sum_s E'[l][s] B[s][n]
            umma_bf16(tmem + T_DC, kmaj(sE, kk, BC_BYTES / 2), mnmaj(sB, kk, BC_BYTES / 2),
                      idesc_bf16(128, 128, 0, 1), kk > 0);
        umma_commit(&bar[1]);
    }
    if (!s_abort) wait_mma();
    // ---- dx = dx_diag + w o u + D dyp; x.u row sums
    {
        float dxd[32], u[32], xv[32];
        tmem_ld32(tmem + lb + T_DXD + 32 * hf, dxd);
        tmem_ld32(tmem + lb + T_DXS + 32 * hf, u);
        tmem_wait_ld();
        load_row32_swz(sm + O_X + row * 128, row, hf, xv);
        const float ws = wst[row];
        float xu = 0.f;
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            xu += xv[i] * u[i];
            o[i] = dxd[i] + ws * u[i] + Dh * dyp[i];
        }
        fm[F_ROWXU + hf * 128 + row] = xu;
        if (live) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.dx + (int64_t)ci.b * p.sdxb + tok * p.sdxl + (int64_t)h * p.sdxh + 32 * hf);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                                    pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
        }
        // e o dyp over the dyp tile (row-uniform scale)
        const float el = ex2(cs2[row]);
        float ev[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) ev[i] = dyp[i] * el;
        store_row32_swz(sm + O_DY + row * 128, row, hf, ev);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (!s_abort && tid == 0) {   // group 3
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < PT / 16; ++kk)   // dC[l][n] += sum_p (e o dyp)[l][p] S_in[p][n]
            umma_bf16(tmem + T_DC, kmaj(sDY, kk, X_BYTES), mnmaj(sSI, kk, S_BYTES / 2), idesc_bf16(128, 128, 0, 1), 1);
#pragma unroll
        for (int kk = 0; kk < QT / 16; ++kk)   // Y_diag[l][p] = sum_s M[l][s] x[s][p]
            umma_bf16(tmem + T_YD, kmaj(sM, kk, BC_BYTES / 2), mnmaj(sX, kk, 16384u), idesc_bf16(128, 64, 0, 1), kk > 0);
#pragma unroll
        for (int kk = 0; kk < NT / 16; ++kk)   // Ybar[l][p] = sum_n C[l][n] S_in[p][n]
            umma_bf16(tmem + T_YO, kmaj(sC, kk, BC_BYTES / 2), kmaj(sSI, kk, S_BYTES / 2), idesc_bf16(128, 64, 0, 0),
                      kk > 0);
        umma_commit(&bar[1]);
    }
    if (!s_abort) wait_mma();
    // ---- dB, dC shares; ypre -> dz; T2, dD row sums
    {
        const int64_t base = ((int64_t)k * H + h) * QT * NT + (int64_t)row * NT + 64 * hf;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float v[32];
            tmem_ld32(tmem + lb + T_DB + 64 * hf + 32 * half, v);
            tmem_wait_ld();
            float4 *d = reinterpret_cast<float4 *>(p.dBh + base + 32 * half);
#pragma unroll
            for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            tmem_ld32(tmem + lb + T_DC + 64 * hf + 32 * half, v);
            tmem_wait_ld();
            d = reinterpret_cast<float4 *>(p.dCh + base + 32 * half);
#pragma unroll
            for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        float yd[32], yb[32], xv[32];
        tmem_ld32(tmem + lb + T_YD + 32 * hf, yd);
        tmem_ld32(tmem + lb + T_YO + 32 * hf, yb);
        tmem_wait_ld();
        load_row32_swz(sm + O_X + row * 128, row, hf, xv);
        const float el = ex2(cs2[row]);
        float t2 = 0.f, dd = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            t2 += dyp[i] * el * yb[i];
            dd += dyp[i] * xv[i];
        }
        fm[F_ROWT2 + hf * 128 + row] = t2;
        fm[F_ROWD + hf * 128 + row] = dd;
        if (live && p.z) {
            float dyv[32], zz[32], o[32];
            load_row32(p.dy + (int64_t)ci.b * p.sdyb + tok * p.sdyl + (int64_t)h * p.sdyh + 32 * hf, dyv);
            load_row32(p.z + (int64_t)ci.b * p.szb + tok * p.szl + (int64_t)h * p.szh + 32 * hf, zz);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float ypre = yd[i] + el * yb[i] + Dh * xv[i];
                const float sg = sig_f(zz[i]);
                o[i] = dyv[i] * ypre * sg * (1.f + zz[i] * (1.f - sg));
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.dz + (int64_t)ci.b * p.sdzb + tok * p.sdzl + (int64_t)h * p.sdzh + 32 * hf);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_uint4(pack_bf16(o[8 * q], o[8 * q + 1]), pack_bf16(o[8 * q + 2], o[8 * q + 3]),
                                    pack_bf16(o[8 * q + 4], o[8 * q + 5]), pack_bf16(o[8 * q + 6], o[8 * q + 7]));
        }
    }
    // T3 = exp(cs[Q-1]) <S_in, dS>: fixed-order block reduction
    {
        const float w = warp_sum(t3p);
        if (lane == 0) fm[F_RED + warp] = w;
    }
    __syncthreads();
    // ---- per-position scalars (threads 0..127 = position i)
    {
        const int i = tid;
        float dcs = 0.f, ddir = 0.f, t4 = 0.f;
        if (i < QT) {
            // column sums of E CB dM for column i: warps with the half that built block i/32, quads >= i/32
            const int sb = i >> 5, j = i & 31;
            const int hsel = (sb == 0 || sb == 3) ? 0 : 1;
            const int bi = (sb == 0 || sb == 1) ? 0 : 1;
            float colTm = 0.f;
            for (int q = sb; q < 4; ++q) colTm += fm[F_COLP + (hsel * 4 + q) * 64 + bi * 32 + j];
            const float xu = fm[F_ROWXU + i] + fm[F_ROWXU + 128 + i];
            const float r1 = fm[F_ROWT1 + i] + fm[F_ROWT1 + 128 + i];
            const float r2 = fm[F_ROWT2 + i] + fm[F_ROWT2 + 128 + i];
            t4 = wst[i] * xu;
            ddir = colTm + ex2(cl2 - cs2[i]) * xu;
            dcs = r1 - dtc[i] * colTm + r2 - t4;
        }
        float t4tot;
        (void)block_scan256(t4, fm + F_WSUM, &t4tot);   // total of T4 (positions >= len contribute 0)
        float T3 = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) T3 += fm[F_RED + w];
        T3 *= ex2(cl2);
        if (i == QT - 1) dcs += T3 + t4tot;
        // da[u] = sum_{i >= u} dcs[i] = total - (inclusive prefix up to u) + dcs[u]
        float dtot;
        const float inc = block_scan256(i < QT ? dcs : 0.f, fm + F_WSUM, &dtot);
        float pa = 0.f, pb = 0.f, pd = 0.f;
        if (i < QT) {
            const float da = dtot - inc + dcs;
            if (i < ci.len) {
                const float v = p.dt_raw[(int64_t)ci.b * p.sdb + (int64_t)(ci.t0 + i) * p.sdl + h] + (p.bias ? p.bias[h] : 0.f);
                const float gv = (ddir + Ah * da) * sigmoid_f(v);
                p.ddt[(int64_t)ci.b * p.sddb + (int64_t)(ci.t0 + i) * p.sddl + h] = gv;
                pa = dtc[i] * da;
                pb = gv;
            }
            pd = fm[F_ROWD + i] + fm[F_ROWD + 128 + i];
        }
        float ta, tb, td;
        (void)block_scan256(pa, fm + F_WSUM, &ta);
        (void)block_scan256(pb, fm + F_WSUM, &tb);
        (void)block_scan256(pd, fm + F_WSUM, &td);
        if (tid == 0) {
            float *pp = p.partials + ((int64_t)k * H + h) * 4;
            pp[0] = ta; pp[1] = td; pp[2] = tb; pp[3] = 0.f;
        }
    }
    (void)lam;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_b() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool map4(CUtensorMap *m, const void *ptr, int64_t inner, int64_t d1, int64_t d2, int64_t d3, int64_t s1, int64_t s2,
          int64_t s3, uint32_t box2) {
    auto fn = encode_fn_b();
    if (fn == nullptr) return false;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)d1, (cuuint64_t)d2, (cuuint64_t)d3};
    cuuint64_t strides[3] = {(cuuint64_t)(s1 * 2), (cuuint64_t)(s2 * 2), (cuuint64_t)(s3 * 2)};
    cuuint32_t box[4] = {64, 1, box2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

static BwdParams make_params(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a) {
    BwdParams p;
    p.sh = sh; p.hdr = hdr; p.chunks = chunks; p.dt_raw = a.dt_raw; p.sdb = a.sdb; p.sdl = a.sdl;
    p.A = a.A; p.D = a.D; p.bias = a.bias;
    p.dy = (const __nv_bfloat16 *)a.dy; p.sdyb = a.sdy[0]; p.sdyl = a.sdy[1]; p.sdyh = a.sdy[2];
    p.z = (const __nv_bfloat16 *)a.z;
    p.szb = a.sz ? a.sz[0] : 0; p.szl = a.sz ? a.sz[1] : 0; p.szh = a.sz ? a.sz[2] : 0;
    p.dx = (__nv_bfloat16 *)a.dx; p.sdxb = a.sdx[0]; p.sdxl = a.sdx[1]; p.sdxh = a.sdx[2];
    p.dz = (__nv_bfloat16 *)a.dz;
    p.sdzb = a.sdz ? a.sdz[0] : 0; p.sdzl = a.sdz ? a.sdz[1] : 0; p.sdzh = a.sdz ? a.sdz[2] : 0;
    p.ddt = a.ddt; p.sddb = a.sddb; p.sddl = a.sddl;
    p.dS = a.dS; p.dS_loc = a.dS; p.chunk_lam = a.chunk_lam; p.dBh = a.dBh; p.dCh = a.dCh; p.partials = a.partials;
    return p;
}

cudaError_t launch_bwd_dstates_tc(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a,
                                  cudaStream_t st) {
    CUtensorMap mc;
    if (!map4(&mc, a.Cp, NT, sh.G, sh.L, sh.B, a.sc[2], a.sc[1], a.sc[0], QT)) return cudaErrorInvalidValue;
    BwdParams p = make_params(sh, hdr, chunks, a);
    static int attr_done[64] = {0};
    cudaError_t e = ensure_smem_attr(k_bwd_dstates_tc, (int)DS_SMEM, attr_done);
    if (e != cudaSuccess) return e;
    k_bwd_dstates_tc<<<dim3(sh.kmax, sh.H), 256, DS_SMEM, st>>>(mc, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_chunk_tc(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a,
                                cudaStream_t st) {
    CUtensorMap mx, mb, mc, ms;
    if (!map4(&mx, a.x, PT, sh.H, sh.L, sh.B, a.sx[2], a.sx[1], a.sx[0], QT)) return cudaErrorInvalidValue;
    if (!map4(&mb, a.Bp, NT, sh.G, sh.L, sh.B, a.sb[2], a.sb[1], a.sb[0], QT)) return cudaErrorInvalidValue;
    if (!map4(&mc, a.Cp, NT, sh.G, sh.L, sh.B, a.sc[2], a.sc[1], a.sc[0], QT)) return cudaErrorInvalidValue;
    // carried states as a [rows = chunk*H*P][N] matrix, box {64, 64 rows}
    const int64_t rows = (int64_t)sh.kmax * sh.H * PT;
    if (!map4(&ms, a.states, NT, 1, rows, 1, NT, NT, rows * NT, PT)) return cudaErrorInvalidValue;
    BwdParams p = make_params(sh, hdr, chunks, a);
    static int attr_done[64] = {0};
    cudaError_t e = ensure_smem_attr(k_bwd_chunk_tc, (int)BWD_SMEM, attr_done);
    if (e != cudaSuccess) return e;
    k_bwd_chunk_tc<<<dim3(sh.kmax, sh.H), 256, BWD_SMEM, st>>>(mx, mb, mc, ms, p);
    return cudaGetLastError();
}

}  // namespace ssd
