// bwd_tc.cu -- tensor-core backward of the SSD chunked scan (bf16 inputs, fp32
// accumulation), headdim 64, dstate 128, chunk 128.
//
// The forward math is re-run per chunk with the true upstream gradients injected, as the
// Mamba-3-Lite "SSD Reference" page's section "6. The autograd backward contract"
// describes; the carried states S_in are the ones the forward kept (ssd_fwd_args.chunk_states)
// or, when it did not, recomputed by the fused forward in states-only mode.  Per chunk c
// of a sequence and head h, with
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
// k_bwd_dstates_tc computes the per-chunk state gradient source
//     dS_loc[p][n] = sum_l e_l dyp[l][p] C[l][n]
// which the reverse warp-shuffle scan turns into dS for every chunk.
// The row sums of M o dM and the dt-weighted column sums of E CB dM cancel along the
// suffix sums of dcs, so both come from the same fp32 products (never from bf16 tiles).
// All contractions run as tcgen05.mma chains on 128-byte-swizzled shared-memory
// tiles (TMA for x, B, C, dy, z; one bulk copy for the carried state of a (chunk, head),
// stored by the forward as the image of its swizzled [n][p] tile); reductions are
// fixed-order.
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
    const __nv_bfloat16 *dS; // [chunk][H][P][N] bf16: gradient of the state leaving the chunk
    const __nv_bfloat16 *states;   // 16 KB tile per (chunk, head): row n = S_in[0..63][n], 128-byte swizzle
    __nv_bfloat16 *dS_loc;   // [chunk][H][P][N] bf16 (dstates kernel output)
    float *chunk_lam;        // [chunk][H] total log-decay of the chunk (dstates kernel output)
    float *dBh, *dCh;        // [chunk][H/hs][Q][N] fp32 shares of head subsets (when hs < H/G)
    float *partials;         // [chunk][H][4]: dA, dD, ddt_bias shares
    int hs;                  // heads per CTA of the gradient kernel
    int hs_ds;               // heads per CTA of the dstates kernel
    __nv_bfloat16 *dB, *dC;  // final outputs when hs == H/G
    int64_t sdBb, sdBl, sdBg, sdCb, sdCl, sdCg;
    int k_pairs, nsub_tail, n_items;   // gradient kernel work items
    int st32;                // dx and dz rows are 32-byte aligned: stored with 256-bit stores
    float *tpart;
    float *dA, *dD, *dbias;
};

__device__ __forceinline__ uint64_t kmaj(uint32_t base, int k, uint32_t col_bytes) {
    return sdesc(base + (uint32_t)(k >> 2) * col_bytes + (uint32_t)(k & 3) * 32u, 16u, 1024u);
}
// MN-major operand with K rows of 128 B; `mn_atom` = byte distance between 64-wide MN atoms.
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int k, uint32_t mn_atom) {
    return sdesc(base + (uint32_t)k * 2048u, mn_atom, 1024u);
}
// logistic (1 + tanh(z/2)) / 2 through one tanh.approx (relative error ~2^-11, below the bf16
// rounding of the data it gates)
__device__ __forceinline__ float sig_f(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
}
__device__ __forceinline__ float silu_f(float z) { return z * sig_f(z); }

// 32 floats as bf16 to 64 contiguous bytes of global memory: two 256-bit stores when the
// address is 32-byte aligned (`st32`, checked on the host for base and strides), else four
// 128-bit stores.
__device__ __forceinline__ void store_row32_global(__nv_bfloat16 *dst, const float *o, bool st32) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(o[2 * i], o[2 * i + 1]);
    if (st32) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 16 * j),
                         "r"(w[8 * j]), "r"(w[8 * j + 1]), "r"(w[8 * j + 2]), "r"(w[8 * j + 3]), "r"(w[8 * j + 4]),
                         "r"(w[8 * j + 5]), "r"(w[8 * j + 6]), "r"(w[8 * j + 7])
                         : "memory");
    } else {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
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
// 16 floats as bf16 into the 16-byte chunks 2 qt, 2 qt + 1 of a 128-byte swizzled row, and back.
__device__ __forceinline__ void store_row16_swz(uint8_t *row_base, int row, int qt, const float *v) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int c = (2 * qt + q) ^ (row & 7);
        *reinterpret_cast<uint4 *>(row_base + c * 16) =
            make_uint4(pack_bf16(v[q * 8], v[q * 8 + 1]), pack_bf16(v[q * 8 + 2], v[q * 8 + 3]),
                       pack_bf16(v[q * 8 + 4], v[q * 8 + 5]), pack_bf16(v[q * 8 + 6], v[q * 8 + 7]));
    }
}
__device__ __forceinline__ void load_row16_swz(const uint8_t *row_base, int row, int qt, float *v) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int c = (2 * qt + q) ^ (row & 7);
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

// Over threads 0..127 (four warps, named barrier 2), in one pass and a fixed order: *vrev =
// the sum of v over this position and all later ones (reverse inclusive scan), *uexcl = the
// sum of u over all earlier positions (exclusive scan).  Both are formed directly, never as a
// total minus a prefix, so a large term never has to cancel against itself.  wsum holds 8
// floats and must not be rewritten before every participant has read it.
__device__ __forceinline__ void rev_excl_scan128(float v, float u, float *wsum, float *vrev, float *uexcl) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_down_sync(0xffffffffu, x, o);
        if (lane + o < 32) x += t;
    }
    const float y = warp_incl_sum(u);
    float ye = __shfl_up_sync(0xffffffffu, y, 1);
    if (lane == 0) ye = 0.f;
    if (lane == 0) wsum[w] = x;          // warp total of v
    if (lane == 31) wsum[4 + w] = y;     // warp total of u
    asm volatile("bar.sync 2, 128;" ::: "memory");
    float offv = 0.f, offu = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i > w) offv += wsum[i];
        if (i < w) offu += wsum[4 + i];
    }
    *vrev = x + offv;
    *uexcl = ye + offu;
}

// ------------------------------------------------------------------ dstates
// grid (kmax, H / hs_ds), 256 threads, three CTAs per SM: one chunk and hs_ds heads of one
// group per CTA.  Per head, dS_loc^T[n][p] = sum_l C[l][n] (e o dyp)[l][p] on the tensor
// cores (A = C^T, M-major; B = e o dyp, N-major), written as bf16 [p][n].  C is loaded
// once; e o dyp is formed in place over the dy tile (each thread rewrites the bytes it read),
// so the next head's z travels as soon as this head's e o dyp is formed and its dy once the
// MMA has read the tile.
constexpr uint32_t DS_OFF_C = 0, DS_OFF_ST = BC_BYTES, DS_OFF_Y = BC_BYTES,
                   DS_OFF_MISC = DS_OFF_ST + 2 * X_BYTES;
constexpr uint32_t DS_SMEM = DS_OFF_MISC + 2048 + 1024;

__global__ void __launch_bounds__(256, 3)
k_bwd_dstates_tc(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmDY,
                 const __grid_constant__ CUtensorMap tmZ, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, hf = tid >> 7;
    const int k = blockIdx.x, HS = p.hs_ds, h0 = blockIdx.y * HS;
    if (k >= p.hdr[HDR_NCHUNKS] || p.hdr[HDR_STATUS] != 0) return;
    const ChunkInfo ci = p.chunks[k];
    const int g = h0 / p.sh.hpg;
    const bool has_z = p.z != nullptr;
    float *dtc = reinterpret_cast<float *>(sm + DS_OFF_MISC);
    float *cs2 = dtc + QT;
    float *wsum = cs2 + QT;                                        // 16
    uint64_t *bar = reinterpret_cast<uint64_t *>(wsum + 16);       // 0: C, 1: dy, 2: MMA, 3: z
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);
    auto stage_dy = [&](int h) {   // one thread
        mbar_expect_tx(&bar[1], X_BYTES);
        tma_load_4d(sm + DS_OFF_ST, &tmDY, &bar[1], 0, h, ci.t0, ci.b);
    };
    auto stage_z = [&](int h) {   // one thread
        mbar_expect_tx(&bar[3], X_BYTES);
        tma_load_4d(sm + DS_OFF_ST + X_BYTES, &tmZ, &bar[3], 0, h, ci.t0, ci.b);
    };
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
        mbar_expect_tx(&bar[0], BC_BYTES);
        tma_load_4d(sm + DS_OFF_C, &tmC, &bar[0], 0, g, ci.t0, ci.b);
        tma_load_4d(sm + DS_OFF_C + BC_BYTES / 2, &tmC, &bar[0], 64, g, ci.t0, ci.b);
        stage_dy(h0);
        if (has_z) stage_z(h0);
    }
    auto load_dtv = [&](int h) -> float {
        return (tid >= ci.lo && tid < ci.len) ? p.dt_raw[(int64_t)ci.b * p.sdb + (int64_t)(ci.t0 + tid) * p.sdl + h] +
                                  (p.bias ? p.bias[h] : 0.f)
                            : 0.f;
    };
    float dt_next = load_dtv(h0), A_next = p.A[h0];
    if (warp == 0) tmem_alloc(tslot, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    uint32_t st_done = 0, st_issued = 1, mma_phase = 0, c_done = 0;
    int bad = 0;
    const uint32_t sC = smem_u32(sm + DS_OFF_C), sY = smem_u32(sm + DS_OFF_Y);
    for (int hi = 0; hi < HS; ++hi) {
        const int h = h0 + hi;
        const float vcur = dt_next, Ah = A_next;
        {   // dt and the in-chunk cumulative log-decay (cs2 = cs log2 e); chunk total -> chunk_lam
            const float dt = (tid >= ci.lo && tid < ci.len) ? softplus_f(vcur) : 0.f;
            float tot;
            const float cs = block_scan256(tid < QT ? dt * Ah : 0.f, wsum, &tot);
            if (tid < QT) {
                dtc[tid] = dt;
                cs2[tid] = cs * LOG2E;
            }
            if (tid == 0) p.chunk_lam[(int64_t)k * p.sh.H + h] = tot;
            __syncthreads();
        }
        if (!mbar_wait(&bar[1], st_done & 1)) bad = 1;   // dy (and z) of this head
        if (has_z && !mbar_wait(&bar[3], st_done & 1)) bad = 1;
        ++st_done;
        {   // (e o dyp) row `row`, half hf, in place over the dy tile (two 16-column pieces)
            const float el = (row >= ci.lo && row < ci.len) ? ex2(cs2[row]) : 0.f;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                uint8_t *yrow = sm + DS_OFF_ST + row * 128;
                const int qt = 2 * hf + q2;   // 16-column piece of the row
                float v[16];
                load_row16_swz(yrow, row, qt, v);
                if (has_z) {
                    float zz[16];
                    load_row16_swz(sm + DS_OFF_ST + X_BYTES + row * 128, row, qt, zz);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= silu_f(zz[i]) * el;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] *= el;
                }
                store_row16_swz(yrow, row, qt, v);
            }
        }
        fence_proxy_async_smem();
        if (__syncthreads_or(bad)) break;
        if (tid == 0) {
            if (hi + 1 < HS && has_z) stage_z(h + 1);   // the z tile is read
            if (hi == 0) {
                if (!mbar_wait(&bar[0], 0)) bad = 1;
                ++c_done;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < QT / 16; ++kk)
                umma_bf16(tmem, mnmaj(sC, kk, BC_BYTES / 2), mnmaj(sY, kk, 16384u), idesc_bf16(128, 64, 1, 1), kk > 0);
            umma_commit(&bar[2]);
        }
        if (hi + 1 < HS) {
            ++st_issued;
            dt_next = load_dtv(h + 1);
            A_next = p.A[h + 1];
        }
        if (!mbar_wait(&bar[2], mma_phase & 1)) bad = 1;
        ++mma_phase;
        tc_fence_after();
        if (tid == 0 && hi + 1 < HS) stage_dy(h + 1);   // the MMA has read the e o dyp tile
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)((warp & 3) * 32) << 16) + 32 * hf + 16 * q2, v);
            tmem_wait_ld();
            __nv_bfloat16 *dst =
                p.dS_loc + ((int64_t)k * p.sh.H + h) * (PT * NT) + (int64_t)(32 * hf + 16 * q2) * NT + row;
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[(int64_t)i * NT] = __float2bfloat16_rn(v[i]);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (bad) set_status(const_cast<int32_t *>(p.hdr), SSD_ERR_DEVICE_TIMEOUT);
    for (uint32_t q = st_done; q < st_issued; ++q) {
        mbar_wait(&bar[1], q & 1);
        if (has_z) mbar_wait(&bar[3], q & 1);
    }
    if (tid == 0 && c_done == 0) mbar_wait(&bar[0], 0);
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
constexpr uint32_t O_SI = O_C + BC_BYTES;          // S_in   [n][p]   16 KB (bulk copy, bf16)
constexpr uint32_t O_DY = O_SI + S_BYTES;          // dyp, then e o dyp [l][p] 16 KB
constexpr uint32_t O_M = O_DY + X_BYTES;           // M      [l][s]   32 KB
constexpr uint32_t O_E = O_M + BC_BYTES;           // E'     [l][s]   32 KB; before: dy, z of the head (TMA)
constexpr uint32_t O_WX = O_E + BC_BYTES;          // w o x  [s][p]   16 KB; before: dS of the head, bf16 [p][n] (bulk copy)
constexpr uint32_t O_SD = O_WX + X_BYTES;          // dS     [p][n]   16 KB (swizzled MMA tile)
constexpr uint32_t O_MISC = O_SD + S_BYTES;
// misc floats
constexpr int F_ROWT1 = 0, F_ROWXU = 256, F_ROWT2 = 512, F_ROWD = 768, F_COLP = 1024, F_RED = 1536,
              F_WSUM = 1552, F_PB = 1568, F_TSUM = 1576, F_TAB = 1584, F_DIAG = 3120, F_END = 3248;
// Per-head position tables, two sets (the next head's is built while this head runs):
// T_CS2 cs log2 e, T_DT dt, T_W w = dt exp(cs[Q-1] - cs), T_GD {exp(cs[a] - cs[s]), dt[s]}
// with a the last position of s's 32-block, T_VR dt_raw + dt_bias.
constexpr int T_CS2 = 0, T_DT = 128, T_W = 256, T_GD = 384, T_VR = 640, TAB_STRIDE = 768;
constexpr uint32_t BWD_SMEM = O_MISC + F_END * 4 + 64 + 1024;

// TMEM columns: dB and dC accumulate over the CTA's heads and C B^T (shared by the
// group's heads) is computed once; columns 384.. serve each head's three MMA groups.
constexpr uint32_t T_DB = 0, T_DC = 128, T_CB = 256;      // whole CTA
constexpr uint32_t T_DM = 384;                            // group 1
constexpr uint32_t T_DXD = 384, T_DXS = 448;              // group 2
constexpr uint32_t T_YD = 384, T_YO = 448;                // group 3 (+ dB, dC)

// Persistent: at most one CTA per SM, taking work items (chunk, group, subset of HS
// heads; HS divides H/G) from a ticket.  An item loads B and C once and computes C B^T
// once for its heads.  Every per-head input arrives one head ahead: dy, z and dS land in
// the E', w o x and dS tiles once the previous head's MMAs have consumed them, x and S_in
// likewise, and dt is read into a register, so no head waits on global memory; the next
// item's B/C and first-head inputs are loaded during the current item's last head.  dB and
// dC accumulate over the item's heads in TMEM and are written once: as bf16 outputs when
// the item covers the whole group, else as fp32 shares summed afterwards in subset order.
__global__ void __launch_bounds__(256, 1)
k_bwd_chunk_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmDY,
               const __grid_constant__ CUtensorMap tmZ, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, hf = tid >> 7, quad = warp & 3;
    const int lane = tid & 31;
    const int H = p.sh.H, G = p.sh.G, hpg = p.sh.hpg, nsub_main = hpg / p.hs;
    const bool has_z = p.z != nullptr;
    float *fm = reinterpret_cast<float *>(sm + O_MISC);
    int tb = 0;   // table set of the current head
    float *cs2 = fm + F_TAB + T_CS2, *dtc = fm + F_TAB + T_DT, *wst = fm + F_TAB + T_W, *vrt = fm + F_TAB + T_VR;
    const float2 *gdt = reinterpret_cast<const float2 *>(fm + F_TAB + T_GD);
    // 0: B/C, 1: x/S_in, 2: MMA (dx and y tiles), 3: dy/z/dS, 4: MMA (dB/dC chains)
    uint64_t *bar = reinterpret_cast<uint64_t *>(fm + F_END);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 5);
    int *s_item = reinterpret_cast<int *>(tslot + 1);   // [0] item, [1] finished-subset count
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lb = (uint32_t)(quad * 32) << 16;
    uint32_t mma_phase = 0, mma2_phase = 0, ld_done = 0, ld_issued = 0, st_done = 0, st_issued = 0, bc_done = 0,
             bc_issued = 0;
    int bad = 0;          // this thread saw a wait run out
    bool aborted = false; // uniform: some thread did (checked once per head)
    auto fail = [&]() {
        bad = 1;
        set_status(const_cast<int32_t *>(p.hdr), SSD_ERR_DEVICE_TIMEOUT);
    };
    auto wait_mma = [&]() {
        if (!mbar_wait(&bar[2], mma_phase & 1)) fail();
        ++mma_phase;
        tc_fence_after();
    };
    auto wait_mma2 = [&]() {
        if (!mbar_wait(&bar[4], mma2_phase & 1)) fail();
        ++mma2_phase;
        tc_fence_after();
    };
    const uint32_t sX = smem_u32(sm + O_X), sB = smem_u32(sm + O_B), sC = smem_u32(sm + O_C);
    const uint32_t sSI = smem_u32(sm + O_SI), sDY = smem_u32(sm + O_DY), sWX = smem_u32(sm + O_WX);
    const uint32_t sM = smem_u32(sm + O_M), sE = smem_u32(sm + O_E), sSD = smem_u32(sm + O_SD);

    // ---- work items: (chunk k, group g, subset of HS heads), in ticket order.  The next
    // item is taken during the current item's last head, and its B/C tiles and first-head
    // inputs are loaded while the current item finishes.
    struct Item {
        int item, pair, nsub, k, g, HS, h0;
        bool tail;
        ChunkInfo ci;
    };
    const int n_main = p.k_pairs * nsub_main;
    auto pair_of = [&](int it) { return it >= n_main ? p.k_pairs + (it - n_main) / p.nsub_tail : it / nsub_main; };
    auto decode = [&](int it, Item &w) {
        w.item = it;
        w.tail = it >= n_main;
        w.pair = pair_of(it);
        const int sub = w.tail ? (it - n_main) % p.nsub_tail : it % nsub_main;
        w.nsub = w.tail ? p.nsub_tail : nsub_main;
        w.k = w.pair / G;
        w.g = w.pair % G;
        w.HS = hpg / w.nsub;
        w.h0 = w.g * hpg + sub * w.HS;
        w.ci = p.chunks[w.k];
    };
    auto take = [&]() -> int {   // one thread: the next item whose chunk exists, else n_items
        const int nch = p.hdr[HDR_NCHUNKS];
        for (;;) {
            if (p.hdr[HDR_STATUS] != 0) return p.n_items;   // an error anywhere ends the work
            const int it = atomicAdd(const_cast<int32_t *>(p.hdr) + HDR_TICKET2, 1);
            if (it >= p.n_items) return p.n_items;
            if (pair_of(it) / G < nch) return it;
        }
    };
    auto load_head = [&](const Item &w, int h) {   // one thread: x and S_in
        const int slab = w.k * H + h;
        mbar_expect_tx(&bar[1], X_BYTES + S_BYTES);
        tma_load_4d(sm + O_X, &tmX, &bar[1], 0, h, w.ci.t0, w.ci.b);
        bulk_load(sm + O_SI, p.states + (int64_t)slab * (PT * NT), S_BYTES, &bar[1]);
    };
    auto stage_head = [&](const Item &w, int h) {   // one thread: dy, z and bf16 dS
        const __nv_bfloat16 *src = p.dS + ((int64_t)w.k * H + h) * (PT * NT);
        mbar_expect_tx(&bar[3], X_BYTES * (has_z ? 2u : 1u) + S_BYTES);
        tma_load_4d(sm + O_E, &tmDY, &bar[3], 0, h, w.ci.t0, w.ci.b);
        if (has_z) tma_load_4d(sm + O_E + X_BYTES, &tmZ, &bar[3], 0, h, w.ci.t0, w.ci.b);
        bulk_load(sm + O_WX, src, S_BYTES, &bar[3]);
    };
    auto load_first = [&](const Item &w) {   // one thread: B/C and the first head's inputs of an item
        mbar_expect_tx(&bar[0], 2 * BC_BYTES);
        tma_load_4d(sm + O_B, &tmB, &bar[0], 0, w.g, w.ci.t0, w.ci.b);
        tma_load_4d(sm + O_B + BC_BYTES / 2, &tmB, &bar[0], 64, w.g, w.ci.t0, w.ci.b);
        tma_load_4d(sm + O_C, &tmC, &bar[0], 0, w.g, w.ci.t0, w.ci.b);
        tma_load_4d(sm + O_C + BC_BYTES / 2, &tmC, &bar[0], 64, w.g, w.ci.t0, w.ci.b);
        stage_head(w, w.h0);
        load_head(w, w.h0);
    };
    auto issue_first = [&](const Item &w) {   // the same, issued by thread 0, counted by all
        if (tid == 0) load_first(w);
        ++bc_issued;
        ++st_issued;
        ++ld_issued;
    };
    // dt_raw + bias of position tid for a head (0 past the chunk's end)
    // dt_raw + bias at position tid - 128 (warps 4..7; 0 past the chunk's end)
    auto load_dtv = [&](const ChunkInfo &c, int h) -> float {
        const int pos = tid - 128;
        return (pos >= c.lo && pos < c.len) ? p.dt_raw[(int64_t)c.b * p.sdb + (int64_t)(c.t0 + pos) * p.sdl + h] +
                                 (p.bias ? p.bias[h] : 0.f)
                           : 0.f;
    };
    // Warps 4..7 (position tid - 128): a head's tables into set `set` (dt, the in-chunk cumulative
    // log-decay by a fixed-order scan over the four warps' partial sums, w, the block factors)
    auto build_tables = [&](int set, float vraw, float Aval, int clo, int clen) {
        const int pos = tid - 128, wl = warp - 4;
        float *T = fm + F_TAB + set * TAB_STRIDE;
        const float dt = (pos >= clo && pos < clen) ? softplus_f(vraw) : 0.f;
        const float x = warp_incl_sum(dt * Aval);
        if (lane == 31) fm[F_TSUM + wl] = x;
        asm volatile("bar.sync 1, 128;" ::: "memory");
        float off = 0.f, tot = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < wl) off += fm[F_TSUM + i];
            tot += fm[F_TSUM + i];
        }
        const float c2 = (x + off) * LOG2E, cl = tot * LOG2E;
        const float c31 = __shfl_sync(0xffffffffu, c2, 31);   // position pos | 31
        T[T_CS2 + pos] = c2;
        T[T_DT + pos] = dt;
        T[T_W + pos] = dt * ex2(cl - c2);
        reinterpret_cast<float2 *>(T + T_GD)[pos] = make_float2(ex2(c31 - c2), dt);
        T[T_VR + pos] = vraw;
        asm volatile("bar.sync 1, 128;" ::: "memory");   // F_TSUM read before a later build rewrites it
    };
    if (tid == 0) s_item[0] = take();
    __syncthreads();
    Item cur;
    bool have = s_item[0] < p.n_items;
    float A_next = 0.f, D_next = 0.f;
    if (have) {
        decode(s_item[0], cur);
        issue_first(cur);
        A_next = p.A[cur.h0];
        D_next = p.D ? p.D[cur.h0] : 0.f;
        if (tid >= 128) build_tables(0, load_dtv(cur.ci, cur.h0), A_next, cur.ci.lo, cur.ci.len);
    }
    __syncthreads();

    while (have) {   // work items
    const int item = cur.item, nsub = cur.nsub, k = cur.k, g = cur.g, HS = cur.HS, h0 = cur.h0;
    const bool tail = cur.tail;
    const ChunkInfo ci = cur.ci;
    Item nxt;
    bool have_next = false;
    const int64_t tok = (int64_t)ci.t0 + row;
    const bool live = row >= ci.lo && row < ci.len;

    for (int hi = 0; hi < HS; ++hi) {
        const int h = h0 + hi;
        if (hi + 1 == HS && tid == 0) s_item[0] = take();   // the item after this one (read after the head's syncs)
        const float Dh = D_next, Ah = A_next;
        {   // this head's tables (built during the previous head, or before the first)
            float *T = fm + F_TAB + tb * TAB_STRIDE;
            cs2 = T + T_CS2; dtc = T + T_DT; wst = T + T_W; vrt = T + T_VR;
            gdt = reinterpret_cast<const float2 *>(T + T_GD);
        }
        const float cl2 = cs2[QT - 1];
        if (!mbar_wait(&bar[3], st_done & 1)) fail();   // dy, z, dS of this head landed
        ++st_done;
        if (!mbar_wait(&bar[1], ld_done & 1)) fail();   // x and S_in of this head landed
        ++ld_done;
        if (hi == 0) {
            if (!mbar_wait(&bar[0], bc_done & 1)) fail();
            ++bc_done;
        }
        __syncthreads();
        // the next head (this item's, or the first of the item taken at this head's start): its
        // dt (warps 4..7), A and D are read now; warps 4..7 build its tables during group 2
        bool nh_has = false;
        int nh = 0, nh_lo = 0, nh_len = 0;
        if (hi + 1 < HS) {
            nh_has = true; nh = h + 1; nh_lo = ci.lo; nh_len = ci.len;
        } else if (s_item[0] < p.n_items) {
            decode(s_item[0], nxt);
            nh_has = true; nh = nxt.h0; nh_lo = nxt.ci.lo; nh_len = nxt.ci.len;
        }
        float v_next = 0.f;
        if (nh_has) {
            if (tid >= 128) v_next = load_dtv(hi + 1 < HS ? ci : nxt.ci, nh);
            A_next = p.A[nh];
            D_next = p.D ? p.D[nh] : 0.f;
        }
        float fz[32];   // dy silu'(z): dz = fz o ypre
        float t3p = 0.f;
        {
            float xv[32];
            {   // dyp = dy silu(z) -> dyp tile; dD row sums dyp . x
                float dyp[32];
                load_row32_swz(sm + O_E + row * 128, row, hf, dyp);
                if (has_z) {
                    float zz[32];
                    load_row32_swz(sm + O_E + X_BYTES + row * 128, row, hf, zz);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float sg = sig_f(zz[i]);
                        fz[i] = dyp[i] * sg * (1.f + zz[i] * (1.f - sg));
                        dyp[i] *= zz[i] * sg;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) fz[i] = 0.f;
                }
                if (!live) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) dyp[i] = 0.f;
                }
                store_row32_swz(sm + O_DY + row * 128, row, hf, dyp);
                load_row32_swz(sm + O_X + row * 128, row, hf, xv);
                float dd = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) dd += dyp[i] * xv[i];
                fm[F_ROWD + hf * 128 + row] = dd;
            }
            fence_proxy_async_smem();
            if (__syncthreads_or(bad)) {
                aborted = true;
                break;
            }
            if (tid == 0) {   // group 1 (runs during the dS work below): CB = C B^T (first head), dM = dyp x^T
                tc_fence_after();
                if (hi == 0) {
#pragma unroll
                    for (int kk = 0; kk < NT / 16; ++kk)
                        umma_bf16(tmem + T_CB, kmaj(sC, kk, BC_BYTES / 2), kmaj(sB, kk, BC_BYTES / 2),
                                  idesc_bf16(128, 128, 0, 0), kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < PT / 16; ++kk)
                    umma_bf16(tmem + T_DM, kmaj(sDY, kk, X_BYTES), kmaj(sX, kk, X_BYTES), idesc_bf16(128, 128, 0, 0),
                              kk > 0);
                umma_commit(&bar[2]);
            }
            const float wl = wst[row];
#pragma unroll
            for (int i = 0; i < 32; ++i) xv[i] *= wl;
            // dS (bf16 [p][n], staged in the w o x tile): T3 partial and the swizzled MMA copy.
            // Thread: 4 runs of 8 consecutive n (run c = tid + 256 j: p = c / 16, n0 = 8 (c % 16)).
            float dsv[4][8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = tid + 256 * j, pp = c >> 4, nc = c & 15;
                const uint4 raw = *reinterpret_cast<const uint4 *>(sm + O_WX + (pp * NT + 8 * nc) * 2);
                const __nv_bfloat162 *e2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(e2[i]);
                    dsv[j][2 * i] = f.x;
                    dsv[j][2 * i + 1] = f.y;
                }
            }
            // <S_in, dS> partial: thread takes 8 consecutive p at one n (run r = tid + 256 j:
            // n = r % 128, p = 8 (r / 128) ..), one 16-byte piece of the S_in tile's row n
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = tid + 256 * j, n = r & 127, q = r >> 7;
                const uint4 si = *reinterpret_cast<const uint4 *>(sm + O_SI + n * 128 + ((q ^ (n & 7)) << 4));
                const __nv_bfloat162 *e2 = reinterpret_cast<const __nv_bfloat162 *>(&si);
                const __nv_bfloat16 *dsn = reinterpret_cast<const __nv_bfloat16 *>(sm + O_WX) + 8 * q * NT + n;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 sv = __bfloat1622float2(e2[i]);
                    t3p = fmaf(sv.x, __bfloat162float(dsn[(2 * i) * NT]), t3p);
                    t3p = fmaf(sv.y, __bfloat162float(dsn[(2 * i + 1) * NT]), t3p);
                }
            }
            __syncthreads();   // the staged dS is read: its space becomes the w o x and dS tiles
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = tid + 256 * j, pp = c >> 4, nc = c & 15;
                *reinterpret_cast<uint4 *>(sm + O_SD + (nc >> 3) * (S_BYTES / 2) + pp * 128 + (((nc & 7) ^ (pp & 7)) << 4)) =
                    make_uint4(pack_bf16(dsv[j][0], dsv[j][1]), pack_bf16(dsv[j][2], dsv[j][3]),
                               pack_bf16(dsv[j][4], dsv[j][5]), pack_bf16(dsv[j][6], dsv[j][7]));
            }
            store_row32_swz(sm + O_WX + row * 128, row, hf, xv);
        }
        fence_proxy_async_smem();
        wait_mma();   // group 1
        // ---- M = E dt_s CB and E' = E dt_s dM (bf16) rows; row sums of M o dM; column sums of
        // E CB dM (fixed order).  Blocks of 32 columns below the diagonal take
        // E = exp(cs[l] - cs[a]) exp(cs[a] - cs[s]) (a = the block's last column; both factors
        // <= 1), the diagonal block exp per element.  The diagonal (s = l, E = 1) does not
        // depend on cs: it stays out of both sums (in exact arithmetic its row and column terms
        // cancel in dcs; in fp32, with dt large, they would leave rounding of their own size)
        // and is kept apart for the direct dt term.
        {
            float rowt1 = 0.f;
            const int l = row;
            const float c2l = cs2[l];
            const float2 *gd = gdt;
            float *colp = fm + F_COLP;   // [8 warps][64]
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
                const int sb = hf == 0 ? (bi == 0 ? 0 : 3) : (bi == 0 ? 1 : 2);   // warp-uniform
                uint8_t *rm = sm + O_M + (sb >> 1) * (BC_BYTES / 2) + l * 128;
                uint8_t *re = sm + O_E + (sb >> 1) * (BC_BYTES / 2) + l * 128;
                if (sb > quad) {   // above the diagonal: zeros (no column sums are read for it)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int cidx = (((sb & 1) << 2) + q) ^ (l & 7);
                        *reinterpret_cast<uint4 *>(rm + (cidx << 4)) = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(re + (cidx << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    continue;
                }
                uint32_t pm[16], pe[16];
                float cb[32], dm[32];
                tmem_ld32(tmem + lb + T_CB + sb * 32, cb);
                tmem_ld32(tmem + lb + T_DM + sb * 32, dm);
                tmem_wait_ld();
                if (sb < quad) {
                    const float r = ex2(c2l - cs2[sb * 32 + 31]);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float mv[2], ev[2];
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const float2 g = gd[sb * 32 + i + jj];
                            const float E = r * g.x;
                            const float ec = E * cb[i + jj], ed = E * g.y;
                            mv[jj] = ed * cb[i + jj];
                            ev[jj] = ed * dm[i + jj];
                            rowt1 = fmaf(mv[jj], dm[i + jj], rowt1);
                            cb[i + jj] = ec * dm[i + jj];   // E CB dM, for the column sums
                        }
                        pm[i >> 1] = pack_bf16(mv[0], mv[1]);
                        pe[i >> 1] = pack_bf16(ev[0], ev[1]);
                    }
                } else {
                    float dg = 0.f;   // the diagonal's E CB dM (E = 1)
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float mv[2], ev[2];
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int s = sb * 32 + i + jj;
                            float m = 0.f, e = 0.f, t = 0.f;
                            if (s <= l) {
                                const float E = ex2(c2l - cs2[s]);
                                const float ec = E * cb[i + jj], ed = E * dtc[s];
                                m = ed * cb[i + jj];
                                e = ed * dm[i + jj];
                                t = ec * dm[i + jj];
                                const bool dia = s == l;
                                rowt1 = fmaf(dia ? 0.f : m, dm[i + jj], rowt1);
                                dg = dia ? t : dg;
                                t = dia ? 0.f : t;
                            }
                            mv[jj] = m;
                            ev[jj] = e;
                            cb[i + jj] = t;
                        }
                        pm[i >> 1] = pack_bf16(mv[0], mv[1]);
                        pe[i >> 1] = pack_bf16(ev[0], ev[1]);
                    }
                    fm[F_DIAG + l] = dg;
                }
                colp[warp * 64 + bi * 32 + lane] = colsum32(cb);
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
        if (tid == 0) {   // group 2
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < QT / 16; ++kk)   // dx_diag[s][p] = sum_l M[l][s] dyp[l][p]
                umma_bf16(tmem + T_DXD, mnmaj(sM, kk, BC_BYTES / 2), mnmaj(sDY, kk, 16384u), idesc_bf16(128, 64, 1, 1),
                          kk > 0);
#pragma unroll
            for (int kk = 0; kk < NT / 16; ++kk)   // u[s][p] = sum_n B[s][n] dS[p][n]
                umma_bf16(tmem + T_DXS, kmaj(sB, kk, BC_BYTES / 2), kmaj(sSD, kk, S_BYTES / 2), idesc_bf16(128, 64, 0, 0),
                          kk > 0);
            umma_commit(&bar[2]);
        }
        if (nh_has && tid >= 128) build_tables(tb ^ 1, v_next, A_next, nh_lo, nh_len);   // while group 2 runs
        wait_mma();
        {   // dx = dx_diag + w o u + D dyp; x.u row sums; then e o dyp over the dyp tile
            float dxd[32], u[32], xv[32], dyp[32];
            tmem_ld32(tmem + lb + T_DXD + 32 * hf, dxd);
            tmem_ld32(tmem + lb + T_DXS + 32 * hf, u);
            load_row32_swz(sm + O_X + row * 128, row, hf, xv);
            load_row32_swz(sm + O_DY + row * 128, row, hf, dyp);
            tmem_wait_ld();
            const float ws = wst[row];
            float xu = 0.f;
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                xu = fmaf(xv[i], u[i], xu);
                o[i] = dxd[i] + ws * u[i] + Dh * dyp[i];
            }
            fm[F_ROWXU + hf * 128 + row] = xu;
            if (live)
                store_row32_global(p.dx + (int64_t)ci.b * p.sdxb + tok * p.sdxl + (int64_t)h * p.sdxh + 32 * hf, o,
                                   p.st32 != 0);
            const float el = ex2(cs2[row]);
#pragma unroll
            for (int i = 0; i < 32; ++i) dyp[i] *= el;
            store_row32_swz(sm + O_DY + row * 128, row, hf, dyp);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {   // group 3
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < QT / 16; ++kk)   // Y_diag[l][p] = sum_s M[l][s] x[s][p]
                umma_bf16(tmem + T_YD, kmaj(sM, kk, BC_BYTES / 2), mnmaj(sX, kk, 16384u), idesc_bf16(128, 64, 0, 1), kk > 0);
#pragma unroll
            for (int kk = 0; kk < NT / 16; ++kk)   // Ybar[l][p] = sum_n C[l][n] S_in[p][n]
                umma_bf16(tmem + T_YO, kmaj(sC, kk, BC_BYTES / 2), mnmaj(sSI, kk, 16384u), idesc_bf16(128, 64, 0, 1),
                          kk > 0);
            umma_commit(&bar[2]);   // the y tiles; the dB/dC chains below run on during the dz epilogue
            const uint32_t first = hi == 0 ? 0u : 1u;   // dB, dC start at the CTA's first head
#pragma unroll
            for (int kk = 0; kk < QT / 16; ++kk)   // dB[s][n] (+)= sum_l E'[l][s] C[l][n]
                umma_bf16(tmem + T_DB, mnmaj(sE, kk, BC_BYTES / 2), mnmaj(sC, kk, BC_BYTES / 2),
                          idesc_bf16(128, 128, 1, 1), (kk > 0) ? 1u : first);
#pragma unroll
            for (int kk = 0; kk < PT / 16; ++kk)   // dB[s][n] += sum_p (w o x)[s][p] dS[p][n]
                umma_bf16(tmem + T_DB, kmaj(sWX, kk, X_BYTES), mnmaj(sSD, kk, S_BYTES / 2), idesc_bf16(128, 128, 0, 1), 1);
#pragma unroll
            for (int kk = 0; kk < QT / 16; ++kk)   // dC[l][n] (+)= sum_s E'[l][s] B[s][n]
                umma_bf16(tmem + T_DC, kmaj(sE, kk, BC_BYTES / 2), mnmaj(sB, kk, BC_BYTES / 2),
                          idesc_bf16(128, 128, 0, 1), (kk > 0) ? 1u : first);
#pragma unroll
            for (int kk = 0; kk < PT / 16; ++kk)   // dC[l][n] += sum_p (e o dyp)[l][p] S_in[p][n]
                umma_bf16(tmem + T_DC, kmaj(sDY, kk, X_BYTES), kmaj(sSI, kk, S_BYTES), idesc_bf16(128, 128, 0, 0), 1);
            umma_commit(&bar[4]);
        }
        wait_mma();
        float xv[32];
        load_row32_swz(sm + O_X + row * 128, row, hf, xv);
        {   // ypre -> dz; T2 row sums
            float yd[32], yb[32], ev[32];
            tmem_ld32(tmem + lb + T_YD + 32 * hf, yd);
            tmem_ld32(tmem + lb + T_YO + 32 * hf, yb);
            load_row32_swz(sm + O_DY + row * 128, row, hf, ev);
            tmem_wait_ld();
            const float el = ex2(cs2[row]);
            float t2 = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) t2 += ev[i] * yb[i];
            fm[F_ROWT2 + hf * 128 + row] = t2;
            if (live && has_z) {
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = fz[i] * (yd[i] + el * yb[i] + Dh * xv[i]);
                store_row32_global(p.dz + (int64_t)ci.b * p.sdzb + tok * p.sdzl + (int64_t)h * p.sdzh + 32 * hf, o,
                                   p.st32 != 0);
            }
        }
        {   // T3 = exp(cs[Q-1]) <S_in, dS>: fixed-order block reduction
            const float w = warp_sum(t3p);
            if (lane == 0) fm[F_RED + warp] = w;
        }
        __syncthreads();   // the row sums and T3 shares are visible; every thread has read x and e o dyp
        // Thread 128 waits for the dB/dC chains (the last MMAs reading shared memory) and at once
        // fetches the next head's inputs (or the next item's B/C and first-head inputs, nxt having
        // been decoded during this head) into the freed tiles, while threads 0..127 compute the
        // per-position scalars.
        if (hi + 1 < HS) {
            if (tid == 128) {
                if (!mbar_wait(&bar[4], mma2_phase & 1)) fail();
                stage_head(cur, h + 1);
                load_head(cur, h + 1);
            }
            ++st_issued;
            ++ld_issued;
        } else if (s_item[0] < p.n_items) {
            have_next = true;
            if (tid == 128) {
                if (!mbar_wait(&bar[4], mma2_phase & 1)) fail();
                load_first(nxt);
            }
            ++bc_issued;
            ++st_issued;
            ++ld_issued;
        }
        if (tid < QT) {   // ---- per-position scalars (threads 0..127 = position i; named barrier 2)
            const int i = tid;
            float dcs, ddir, t4;
            {
                const int sb = i >> 5, jj = i & 31;
                const int hsel = (sb == 0 || sb == 3) ? 0 : 1;
                const int bi = (sb == 0 || sb == 1) ? 0 : 1;
                float colTm = 0.f;   // sum_{l > i} (E CB dM)[l][i], rows in quads >= sb, in quad order
                for (int q = sb; q < 4; ++q) colTm += fm[F_COLP + (hsel * 4 + q) * 64 + bi * 32 + jj];
                const float xu = fm[F_ROWXU + i] + fm[F_ROWXU + 128 + i];
                const float r1 = fm[F_ROWT1 + i] + fm[F_ROWT1 + 128 + i];
                const float r2 = fm[F_ROWT2 + i] + fm[F_ROWT2 + 128 + i];
                t4 = wst[i] * xu;
                ddir = colTm + fm[F_DIAG + i] + ex2(cl2 - cs2[i]) * xu;
                dcs = r1 - dtc[i] * colTm + r2;
            }
            float T3 = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) T3 += fm[F_RED + w];
            T3 *= ex2(cl2);
            // da[u] = sum_{i>=u} dcs[i] + T3 + sum_{s<u} T4[s]  (T4[s] enters dcs at the chunk's
            // last position with + and at s with -: their net share of da[u] is the prefix below u)
            float drev, t4ex;
            rev_excl_scan128(dcs, t4, fm + F_WSUM, &drev, &t4ex);
            float pa = 0.f, pb = 0.f;
            const float da = drev + T3 + t4ex;
            if (i >= ci.lo && i < ci.len) {
                const float gv = (ddir + Ah * da) * sigmoid_f(vrt[i]);
                p.ddt[(int64_t)ci.b * p.sddb + (int64_t)(ci.t0 + i) * p.sddl + h] = gv;
                pa = dtc[i] * da;
                pb = gv;
            }
            float pd = fm[F_ROWD + i] + fm[F_ROWD + 128 + i];
            // dA, ddt_bias, dD shares: fixed-order sums of pa, pb, pd over the four warps (the
            // T3 slots were read by every participant before the scan's barrier)
            pa = warp_sum(pa);
            pb = warp_sum(pb);
            pd = warp_sum(pd);
            if (lane == 0) {
                fm[F_RED + warp] = pa;
                fm[F_PB + warp] = pb;
                fm[F_RED + 8 + warp] = pd;
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (tid == 0) {
                float ta = 0.f, tb = 0.f, td = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    ta += fm[F_RED + w];
                    tb += fm[F_PB + w];
                    td += fm[F_RED + 8 + w];
                }
                float *pp = p.partials + ((int64_t)k * H + h) * 4;
                pp[0] = ta; pp[1] = td; pp[2] = tb; pp[3] = 0.f;
            }
        }
        wait_mma2();   // every thread: the dB/dC chains are done (thread 128 has seen it already)
        tb ^= 1;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // ---- dB, dC of the item's heads: final bf16 rows when the item covers the group; else
    // fp32 shares, summed in subset order afterwards by k_reduce_group (main items) or
    // k_bwd_finish (the split pairs of the tail)
    if (aborted || __syncthreads_or(bad)) {
        aborted = true;
        break;
    }
    {
        auto store_bf16 = [&](int which, const float *v) {
            const int ncols = p.sh.Nio - 64 * hf;   // of this half's 64 columns, those the caller's dB/dC hold
            if (!live || ncols <= 0) return;
            __nv_bfloat16 *dst = (which == 0 ? p.dB : p.dC) + (int64_t)ci.b * (which == 0 ? p.sdBb : p.sdCb) +
                                 tok * (which == 0 ? p.sdBl : p.sdCl) + (int64_t)g * (which == 0 ? p.sdBg : p.sdCg) +
                                 64 * hf;
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (8 * q < ncols)
                    d4[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                       pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
        };
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t col0 = (which == 0 ? T_DB : T_DC) + 64 * hf;
            float v[64];
            {
                float t[32];
                tmem_ld32(tmem + lb + col0, t);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = t[i];
                tmem_ld32(tmem + lb + col0 + 32, t);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[32 + i] = t[i];
            }
            if (nsub == 1) {
                store_bf16(which, v);
            } else {
                float *dst = tail ? p.tpart + (((int64_t)(item - n_main) * 2 + which) * QT + row) * NT + 64 * hf
                                  : (which == 0 ? p.dBh : p.dCh) +
                                        (((int64_t)k * (H / p.hs) + h0 / p.hs) * QT + row) * NT + 64 * hf;
                float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
                for (int q = 0; q < 16; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();   // dB/dC read from TMEM: the next item may start its chains
    tc_fence_after();
    have = have_next;
    if (have) cur = nxt;
    }   // work items
    // drain (only after an early stop) and free TMEM
    for (uint32_t q = ld_done; q < ld_issued; ++q) mbar_wait(&bar[1], q & 1);
    for (uint32_t q = st_done; q < st_issued; ++q) mbar_wait(&bar[3], q & 1);
    for (uint32_t q = bc_done; q < bc_issued; ++q) mbar_wait(&bar[0], q & 1);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// The two sums after the gradient kernel, one launch (their outputs are disjoint):
//  - blocks [0, tail_blocks): dB/dC of the pairs (chunk, group) split into subsets at the tail
//    of the gradient kernel, the subsets' fp32 shares summed in subset order; block =
//    (tail pair, dB or dC, 16 rows), 256 threads: 16 rows x 128 columns, 8 values a thread;
//  - the next H blocks: dA, dD, ddt_bias of a head, its per-chunk partials summed in a fixed
//    order.
__global__ void __launch_bounds__(256)
k_bwd_finish(const BwdParams p, int tail_blocks) {
    if ((int)blockIdx.x >= tail_blocks) {
        __shared__ float red[3][8];
        const int h = blockIdx.x - tail_blocks, tid = threadIdx.x;
        const int nk = p.hdr[HDR_STATUS] != 0 ? 0 : p.hdr[HDR_NCHUNKS];
        float a = 0.f, d = 0.f, b = 0.f;
        for (int k = tid; k < nk; k += 256) {
            const float *pp = p.partials + ((int64_t)k * p.sh.H + h) * 4;
            a += pp[0]; d += pp[1]; b += pp[2];
        }
        a = warp_sum(a); d = warp_sum(d); b = warp_sum(b);
        if ((tid & 31) == 0) { red[0][tid >> 5] = a; red[1][tid >> 5] = d; red[2][tid >> 5] = b; }
        __syncthreads();
        if (tid == 0) {
            float ta = 0.f, td = 0.f, tb = 0.f;
            for (int w = 0; w < 8; ++w) { ta += red[0][w]; td += red[1][w]; tb += red[2][w]; }
            p.dA[h] = ta;
            if (p.dD) p.dD[h] = td;
            if (p.dbias) p.dbias[h] = tb;
        }
        return;
    }
    const int per = 2 * (QT / 16);
    const int tp = blockIdx.x / per, which = (blockIdx.x % per) / (QT / 16), l0 = (blockIdx.x % (QT / 16)) * 16;
    const int pair = p.k_pairs + tp, k = pair / p.sh.G, g = pair % p.sh.G;
    if (p.hdr[HDR_STATUS] != 0 || k >= p.hdr[HDR_NCHUNKS]) return;
    const ChunkInfo ci = p.chunks[k];
    const int l = l0 + (threadIdx.x >> 4), n0 = (threadIdx.x & 15) * 8;
    if (l < ci.lo || l >= ci.len || n0 >= p.sh.Nio) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < p.nsub_tail; ++j) {
        const float4 *src = reinterpret_cast<const float4 *>(
            p.tpart + ((((int64_t)tp * p.nsub_tail + j) * 2 + which) * QT + l) * NT + n0);
        const float4 a = src[0], b = src[1];
        acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
        acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    __nv_bfloat16 *dst = (which == 0 ? p.dB : p.dC) + (int64_t)ci.b * (which == 0 ? p.sdBb : p.sdCb) +
                         (int64_t)(ci.t0 + l) * (which == 0 ? p.sdBl : p.sdCl) + (int64_t)g * (which == 0 ? p.sdBg : p.sdCg) + n0;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]),
                                                 pack_bf16(acc[4], acc[5]), pack_bf16(acc[6], acc[7]));
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
    p.states = a.states;
    p.dS = a.dS; p.dS_loc = a.dS; p.chunk_lam = a.chunk_lam; p.dBh = a.dBh; p.dCh = a.dCh; p.partials = a.partials;
    p.hs = a.hs;
    p.hs_ds = a.hs_ds;
    p.dB = (__nv_bfloat16 *)a.dB; p.dC = (__nv_bfloat16 *)a.dC;
    p.sdBb = a.sdB ? a.sdB[0] : 0; p.sdBl = a.sdB ? a.sdB[1] : 0; p.sdBg = a.sdB ? a.sdB[2] : 0;
    p.sdCb = a.sdC ? a.sdC[0] : 0; p.sdCl = a.sdC ? a.sdC[1] : 0; p.sdCg = a.sdC ? a.sdC[2] : 0;
    p.k_pairs = a.k_pairs; p.nsub_tail = a.nsub_tail; p.n_items = a.n_items; p.tpart = a.tpart;
    p.dA = a.dA; p.dD = a.dD; p.dbias = a.dbias;
    // 256-bit row stores need every dx / dz row piece 32-byte aligned: base and all strides
    auto a32 = [](const void *ptr, const int64_t *st) {
        return ptr == nullptr || ((uintptr_t)ptr % 32 == 0 && st[0] % 16 == 0 && st[1] % 16 == 0 && st[2] % 16 == 0);
    };
    p.st32 = (a32(a.dx, a.sdx) && a32(a.dz, a.sdz)) ? 1 : 0;
    return p;
}

cudaError_t launch_bwd_dstates_tc(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a,
                                  cudaStream_t st) {
    CUtensorMap mc, mdy, mz;
    if (!map4(&mc, a.Cp, sh.Nio, sh.G, sh.L, sh.B, a.sc[2], a.sc[1], a.sc[0], QT)) return cudaErrorInvalidValue;
    if (!map4(&mdy, a.dy, PT, sh.H, sh.L, sh.B, a.sdy[2], a.sdy[1], a.sdy[0], QT)) return cudaErrorInvalidValue;
    if (a.z != nullptr) {
        if (!map4(&mz, a.z, PT, sh.H, sh.L, sh.B, a.sz[2], a.sz[1], a.sz[0], QT)) return cudaErrorInvalidValue;
    } else {
        mz = mdy;   // not read
    }
    BwdParams p = make_params(sh, hdr, chunks, a);
    static int attr_done[64] = {0};
    cudaError_t e = ensure_smem_attr(k_bwd_dstates_tc, (int)DS_SMEM, attr_done);
    if (e != cudaSuccess) return e;
    k_bwd_dstates_tc<<<dim3(sh.kmax, sh.H / a.hs_ds), 256, DS_SMEM, st>>>(mc, mdy, mz, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_chunk_tc(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a,
                                cudaStream_t st) {
    CUtensorMap mx, mb, mc, mdy, mz;
    if (!map4(&mx, a.x, PT, sh.H, sh.L, sh.B, a.sx[2], a.sx[1], a.sx[0], QT)) return cudaErrorInvalidValue;
    if (!map4(&mdy, a.dy, PT, sh.H, sh.L, sh.B, a.sdy[2], a.sdy[1], a.sdy[0], QT)) return cudaErrorInvalidValue;
    if (a.z != nullptr) {
        if (!map4(&mz, a.z, PT, sh.H, sh.L, sh.B, a.sz[2], a.sz[1], a.sz[0], QT)) return cudaErrorInvalidValue;
    } else {
        mz = mdy;   // not read
    }
    if (!map4(&mb, a.Bp, sh.Nio, sh.G, sh.L, sh.B, a.sb[2], a.sb[1], a.sb[0], QT)) return cudaErrorInvalidValue;
    if (!map4(&mc, a.Cp, sh.Nio, sh.G, sh.L, sh.B, a.sc[2], a.sc[1], a.sc[0], QT)) return cudaErrorInvalidValue;
    BwdParams p = make_params(sh, hdr, chunks, a);
    static int attr_done[64] = {0};
    cudaError_t e = ensure_smem_attr(k_bwd_chunk_tc, (int)BWD_SMEM, attr_done);
    if (e != cudaSuccess) return e;
    if (a.grid > 0) k_bwd_chunk_tc<<<a.grid, 256, BWD_SMEM, st>>>(mx, mb, mc, mdy, mz, p);   // persistent
    const int tail_pairs = sh.kmax * sh.G - a.k_pairs;
    const int tail_blocks = (a.grid > 0 && tail_pairs > 0 && a.nsub_tail > 1 && a.hs == sh.hpg) ? tail_pairs * 2 * (QT / 16) : 0;
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
    k_bwd_finish<<<tail_blocks + sh.H, 256, 0, st>>>(p, tail_blocks);
    return cudaGetLastError();
}

}  // namespace ssd
