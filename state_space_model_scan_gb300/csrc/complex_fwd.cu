// complex_fwd.cu -- forward of the complex-A SSD scan (the Mamba-3-Lite variant), on the
// tensor cores in tf32 with fp32 accumulation.
//
// What it computes (Mamba-3-Lite "SSD Reference -- complex scan API & kernel contract",
// section "Math: the recurrence both functions implement"; section "ssd_complex_chunkwise"
// for the chunked evaluation and its inter-chunk contract): per (batch row, head), with
// abar_t = exp(softplus(dt_t) A_h) (A complex, dt real) and a complex state h_t [D, N],
//     h_t = abar_t h_{t-1} + x_t (outer) B_t ,   y_t[d] = sum_n C_t[n] h_t[d, n]
// from h_{-1} = initial_states (or 0); y_real = Re y, y_imag = Im y, final = h_{T-1}.
//
// Design.  One CTA per (batch row, head) walks its chunks of 64 positions in order and
// carries the state in shared memory (fp32), so no state ever goes to HBM between chunks.
// Complex products run as real tf32 MMAs over interleaved (re, im) K: with u, v complex
// K-vectors stored as [re, im] pairs, sum u v = [u_re, u_im] . [v_re, -v_im]  (real part)
// and [u_re, u_im] . [v_im, v_re]  (imaginary part), so the as-loaded interleaved operand
// pairs with a "conjugated" and a "swapped" copy of the other one; equally
// [u_re, -u_im] . [v_re, v_im] and [u_im, u_re] . [v_re, v_im] are the real and imaginary parts.
// An M = 128 MMA costs the issuing thread no more than an M = 64 one, and an N = 128 one about
// 1.4 times an N = 64 one, so operands are stacked on both sides:
//   batch 1  A = [conj(C) ; swap(C)]    B = [B tile ; S]  -> [Re Cb | Re Yraw ; Im Cb | Im Yraw]
//   batch 2  A = [M ; (w o B)^T],  M = L o Cb
//                                       B = conj(X^T)    -> [Re Ydiag ; Re Sloc]
//                                       B = swap(X^T)    -> [Im Ydiag ; Im Sloc]
//   y = Ydiag + exp(cs_l) Yraw ;  S <- exp(cs_63) S + Sloc
// (Cb = C B^T, Yraw = C S^T with S the carry-in state, Ydiag = M X, Sloc = (w o B)^T X) with
// cs the in-chunk inclusive cumulative sum of softplus(dt) A, L[l, s] = exp(cs_l - cs_s) for
// l >= s and w_l = exp(cs_63 - cs_l).  TMEM lanes 0..63 (the upper half of the CTA's warps)
// hold the real parts of rows l of Cb, Yraw and Ydiag; lanes 64..127 (the lower half) the
// imaginary parts of Cb and Yraw, and Sloc, whose rows n they fold into the carried state.
// Both halves build M, in alternating 8-column groups, passing each other the component of
// the other's groups through shared memory; the lower half passes Im Yraw to the upper half,
// which writes y.  Batch 2's two chains are committed separately, so the real outputs are
// written while the imaginary chain runs.  MMAs (K = 128: 16 of K = 8 each): 16 of M = 128,
// N = 128 and 32 of M = 128, N = 64 per chunk.  Operands are written as fp32; the tensor cores
// read their tf32 part (10 mantissa bits, truncated).  Positions past the end of the sequence
// read as zero (TMA bounds fill) and carry no decay.
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "tc_common.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int CQ = 64;                      // chunk length
constexpr int CD = 64;                      // head dimension (P)
constexpr int CN = 64;                      // state dimension
constexpr int CX_THREADS = 512;             // 16 warps: four per TMEM lane quadrant
constexpr uint32_t SLOT = 32768;            // a 64-row operand: 64 rows x 128 fp32, 4 K-atoms of 8 KB
constexpr uint32_t ATOM = 8192;
constexpr uint32_t ATOM128 = 16384;         // K-atom of a 128-row operand (rows 64.. at +8 KB)
constexpr uint32_t OFF_CC = 0;              // 128-row: [conj(C) ; swap(C)] (batch 1), then [M ; (w o B)^T]
constexpr uint32_t OFF_BS = 2 * SLOT;       // 128-row: [B tile (then swap(X^T)) ; carried state S]
constexpr uint32_t OFF_X = 4 * SLOT;        // X tile as loaded
constexpr uint32_t OFF_XC = 5 * SLOT;       // conj(X^T)
constexpr uint32_t OFF_E = 6 * SLOT;        // exchange, [64][65] fp32: Cb parts for the M build, then Im Yraw
constexpr uint32_t E_STRIDE = 65;
constexpr uint32_t OFF_MISC = OFF_E + 64 * E_STRIDE * 4 + 256;
// per-chunk tables, two sets (chunk c uses set c & 1; the next chunk's is built meanwhile)
constexpr uint32_t MISC_CS = 0, MISC_E = 1024, MISC_W = 2048, MISC_ROT = 3072, MISC_BAR = 4096, MISC_TMEM = 4160,
                   MISC_ABORT = 4164;
constexpr uint32_t CX_SMEM = OFF_MISC + 4608 + 1024;       // + alignment slack
constexpr uint32_t TX_BYTES = 3 * SLOT;                    // C, B and X tiles of one chunk

// TMEM columns: batch 1 [Cb | Yraw] 128 (real parts in lanes 0..63, imaginary in 64..127);
// batch 2 [Ydiag ; Sloc] real parts 64, imaginary parts 64.
constexpr uint32_t TC_CB = 0, TC_YR = 64, TC_Y2 = 128, TM_COLS = 256;

enum { BAR_IN = 0, BAR_M1 = 1, BAR_M2 = 2, BAR_M3 = 3 };

struct CxParams {
    int64_t Bt, T, H;
    const float *dt;        // [Bt][T][H]
    const float *A;         // [H] complex (re, im)
    const float *init;      // [Bt][H][D][N] complex or null
    float *y_re, *y_im;     // [Bt][T][H][D]; y_im may be null
    float *final_;          // [Bt][H][D][N] complex or null
    int32_t *hdr;           // status header
};

__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// K step k (8 fp32 = 32 bytes) of a 64-row operand slot.
__device__ __forceinline__ uint64_t opdesc(uint32_t slot, int k) {
    return sdesc(slot + (uint32_t)(k >> 2) * ATOM + (uint32_t)(k & 3) * 32u, 16u, 1024u);
}
// K step k of a 128-row operand.
__device__ __forceinline__ uint64_t opdesc128(uint32_t slot, int k) {
    return sdesc(slot + (uint32_t)(k >> 2) * ATOM128 + (uint32_t)(k & 3) * 32u, 16u, 1024u);
}
// Byte offset of fp32 element (row r, k) inside a 64-row slot (128-byte swizzle, K-major) ...
__device__ __forceinline__ uint32_t elem_off(int r, int k) {
    return (uint32_t)(k >> 5) * ATOM + (uint32_t)r * 128u + ((uint32_t)(((k & 31) >> 2) ^ (r & 7)) << 4) +
           (uint32_t)(k & 3) * 4u;
}
// ... and inside a 128-row operand
__device__ __forceinline__ uint32_t elem_off128(int r, int k) {
    return (uint32_t)(k >> 5) * ATOM128 + (uint32_t)r * 128u + ((uint32_t)(((k & 31) >> 2) ^ (r & 7)) << 4) +
           (uint32_t)(k & 3) * 4u;
}
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
__device__ __forceinline__ float2 cexp(float2 a) {
    float s, c;
    sincosf(a.y, &s, &c);
    const float m = __expf(a.x);
    return make_float2(m * c, m * s);
}
__device__ __forceinline__ float softplus_f(float v) {
    return v > 20.f ? v : log1pf(__expf(v));
}
// Named barrier 1 over the whole CTA: one half arrives (no wait), the other waits for it.
__device__ __forceinline__ void halves_arrive() { asm volatile("barrier.arrive 1, %0;" ::"n"(CX_THREADS) : "memory"); }
__device__ __forceinline__ void halves_sync() { asm volatile("barrier.sync 1, %0;" ::"n"(CX_THREADS) : "memory"); }
__device__ __forceinline__ void st_pair(uint8_t *slot, int r, int k, float a, float b) {
    *reinterpret_cast<float2 *>(slot + elem_off(r, k)) = make_float2(a, b);
}

__global__ void __launch_bounds__(CX_THREADS, 1)
k_complex_fwd(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const CxParams p) {
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
    uint8_t *CC = sm + OFF_CC, *BS = sm + OFF_BS, *XT = sm + OFF_X, *XC = sm + OFF_XC;
    float *E = reinterpret_cast<float *>(sm + OFF_E);
    float2 *cs_t = reinterpret_cast<float2 *>(sm + OFF_MISC + MISC_CS);    // [2][CQ] in-chunk cumsum
    float2 *ecs_t = reinterpret_cast<float2 *>(sm + OFF_MISC + MISC_E);    // [2][CQ] exp(cs_l)
    float2 *wv_t = reinterpret_cast<float2 *>(sm + OFF_MISC + MISC_W);     // [2][CQ] exp(cs_63 - cs_l)
    float2 *rot_t = reinterpret_cast<float2 *>(sm + OFF_MISC + MISC_ROT);  // [2][CQ] exp(i Im cs_l)
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_MISC + MISC_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + MISC_TMEM);
    volatile int *abort_ = reinterpret_cast<volatile int *>(sm + OFF_MISC + MISC_ABORT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t item = blockIdx.x;
    const int64_t b = item / p.H, h = item % p.H;
    const int nc = (int)((p.T + CQ - 1) / CQ);
    const float2 Ah = make_float2(p.A[2 * h], p.A[2 * h + 1]);
    // TMEM-phase mapping (M = 128 accumulators): warp w reads lanes 32 (w & 3) .. + 31, i.e.
    // accumulator row r = 32 (w & 3) + lane; the four warps of a lane quadrant take 16 columns
    // each.  Upper half (rows 0..63): row l = r; lower half: l or n = r - 64.
    const int quad = warp & 3, sub = warp >> 2;
    const bool upper = quad < 2;
    const int r64 = 32 * (quad & 1) + lane;   // l (upper) or the lower half's row - 64
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        *abort_ = 0;
        fence_mbar_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    if (warp == 0) tmem_alloc(tmem_slot, TM_COLS);
    // carried state from initial_states (or zero): rows 64 + d of BS, K = 2n + part, (Sr, Si)
    for (int i = tid; i < CD * CN; i += CX_THREADS) {
        const int d = i / CN, n = i % CN;
        float2 v = make_float2(0.f, 0.f);
        if (p.init != nullptr) v = reinterpret_cast<const float2 *>(p.init)[((b * p.H + h) * CD + d) * CN + n];
        *reinterpret_cast<float2 *>(BS + elem_off128(64 + d, 2 * n)) = v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sCC = smem_u32(CC), sBS = smem_u32(BS), sXC = smem_u32(XC);
    const uint32_t id128 = idesc_tf32(128, 64), id128n = idesc_tf32(128, 128);

    // One BAR_IN phase per chunk, armed for all three tiles when the X tile is issued; the C
    // and B tiles follow later into the same phase.
    auto load_x = [&](int c) {
        mbar_expect_tx(&bar[BAR_IN], TX_BYTES);
        for (int a = 0; a < 4; ++a) tma_load_4d(XT + a * ATOM, &tmX, &bar[BAR_IN], 32 * a, (int)h, c * CQ, (int)b);
    };
    auto load_cb = [&](int c) {
        for (int a = 0; a < 4; ++a) {
            tma_load_4d(CC + a * ATOM128, &tmC, &bar[BAR_IN], 32 * a, (int)h, c * CQ, (int)b);   // rows 0..63
            tma_load_4d(BS + a * ATOM128, &tmB, &bar[BAR_IN], 32 * a, (int)h, c * CQ, (int)b);   // rows 0..63
        }
    };
    // thread 0's record of what may still be in flight when a bounded wait gives up
    bool in_pending = false, m1_pending = false, m2_pending = false;
    uint32_t in_par = 0, m_par = 0;
    if (tid == 0 && nc > 0) {
        load_x(0);
        load_cb(0);
        in_pending = true;
    }
    // Warp 2 builds the per-chunk tables (one lane: two positions), the next chunk's while the
    // current chunk's second MMA batch runs; it reads dt one chunk ahead of that.
    float dtn[2] = {0.f, 0.f};
    auto fetch_dt = [&](int c) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t t = (int64_t)c * CQ + 2 * lane + j;
            dtn[j] = t < p.T ? p.dt[(b * p.T + t) * p.H + h] : 0.f;
        }
    };
    auto build_tables = [&](int c) {   // warp 2; dtn holds chunk c's dt
        const int set = c & 1;
        const int64_t t0 = (int64_t)c * CQ;
        float2 a2[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float sp = (t0 + 2 * lane + j < p.T) ? softplus_f(dtn[j]) : 0.f;
            a2[j] = make_float2(sp * Ah.x, sp * Ah.y);
        }
        if (c + 1 < nc) fetch_dt(c + 1);
        float2 s = make_float2(a2[0].x + a2[1].x, a2[0].y + a2[1].y);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float ux = __shfl_up_sync(0xffffffffu, s.x, o), uy = __shfl_up_sync(0xffffffffu, s.y, o);
            if (lane >= o) { s.x += ux; s.y += uy; }
        }
        float2 ex = make_float2(__shfl_up_sync(0xffffffffu, s.x, 1), __shfl_up_sync(0xffffffffu, s.y, 1));
        if (lane == 0) ex = make_float2(0.f, 0.f);
        const float2 last = make_float2(__shfl_sync(0xffffffffu, s.x, 31), __shfl_sync(0xffffffffu, s.y, 31));
        const float2 cl[2] = {make_float2(ex.x + a2[0].x, ex.y + a2[0].y), s};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int l = 2 * lane + j;
            cs_t[set * CQ + l] = cl[j];
            ecs_t[set * CQ + l] = cexp(cl[j]);
            wv_t[set * CQ + l] = cexp(make_float2(last.x - cl[j].x, last.y - cl[j].y));
            float sn, cn;
            sincosf(cl[j].y, &sn, &cn);
            rot_t[set * CQ + l] = make_float2(cn, sn);
        }
    };
    if (warp == 2 && nc > 0) {
        fetch_dt(0);
        build_tables(0);
    }
    __syncthreads();

    for (int c = 0; c < nc; ++c) {
        const uint32_t par = (uint32_t)(c & 1);
        const int64_t t0 = (int64_t)c * CQ;
        const float2 *cs = cs_t + (c & 1) * CQ, *ecs = ecs_t + (c & 1) * CQ;
        const float2 *wv = wv_t + (c & 1) * CQ, *rot = rot_t + (c & 1) * CQ;
        // ---- chunk inputs
        if (tid == 0) {
            in_par = par;
            if (!mbar_wait_abort(&bar[BAR_IN], par, abort_)) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
            else in_pending = false;
        }
        __syncthreads();
        if (*abort_) break;
        // conj(C) in place (rows 0..63 of CC) and swap(C) below it (rows 64..127, the same
        // swizzled position 8 KB on); B and S are used as they are
        for (int i = tid; i < (int)(SLOT / 16); i += CX_THREADS) {
            float4 *cp = reinterpret_cast<float4 *>(CC + (i >> 9) * ATOM128) + (i & 511);
            const float4 cv = *cp;
            *cp = make_float4(cv.x, -cv.y, cv.z, -cv.w);
            cp[ATOM / 16] = make_float4(cv.y, cv.x, cv.w, cv.z);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- batch 1: [Re Cb | Re Yraw ; Im Cb | Im Yraw] (B tile and state stacked, N = 128)
        if (tid == 0) {
            for (int k = 0; k < 16; ++k) umma_tf32(tmem + TC_CB, opdesc128(sCC, k), opdesc128(sBS, k), id128n, k > 0);
            umma_commit(&bar[BAR_M1]);
            m_par = par;
            m1_pending = true;
        }
        // ---- meanwhile conj(X^T) into XC (rows d, K = 2s + part: Xr, -Xi).  A warp reads one
        // 16-byte piece (two complex columns d) of 32 consecutive rows s and writes a contiguous
        // 256-byte run of rows d and d+1.
        {
            const int s = lane + 32 * (warp & 1);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d0 = 2 * ((warp >> 1) + 8 * i);
                const float4 v = *reinterpret_cast<const float4 *>(XT + elem_off(s, 2 * d0));
                st_pair(XC, d0, 2 * s, v.x, -v.y);
                st_pair(XC, d0 + 1, 2 * s, v.z, -v.w);
            }
        }
        if (tid == 0) {
            if (!mbar_wait_abort(&bar[BAR_M1], par, abort_)) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
            else m1_pending = false;
        }
        __syncthreads();
        tc_fence_after();
        if (*abort_) break;
        // ---- M = L o Cb is built by both halves, in 8-column groups g of row l: the upper half (Re Cb
        // in its lanes) takes the even groups, the lower half (Im Cb) the odd ones, so the causal
        // work splits evenly.  Each half passes the other the component of the other's groups
        // through E, keeping its own; both halves share the (w o B)^T and swap(X^T) builds.
        float own[8];
        {
            float v[16];
            tmem_ld16(tmem + lane_base + TC_CB + 16 * sub, v);
            tmem_wait_ld();
            // the upper half keeps group 2 sub and passes group 2 sub + 1; the lower half the reverse
            float *ex = E + r64 * E_STRIDE + 16 * sub + (upper ? 8 : 0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                own[j] = upper ? v[j] : v[8 + j];
                ex[j] = upper ? v[8 + j] : v[j];
            }
        }
        {   // (w o B)^T into rows 64..127 of CC (rows n, K = 2l + part) from the B tile
            const int l = r64;
            const float2 wl = wv[l];
#pragma unroll
            for (int i0 = 0; i0 < 4; ++i0) {
                const int i = upper ? i0 : i0 + 4;
                const int n0 = 2 * (sub + 4 * i);
                const float4 bv = *reinterpret_cast<const float4 *>(BS + elem_off128(l, 2 * n0));
                const float2 v0 = cmul(wl, make_float2(bv.x, bv.y)), v1 = cmul(wl, make_float2(bv.z, bv.w));
                *reinterpret_cast<float2 *>(CC + elem_off128(64 + n0, 2 * l)) = make_float2(v0.x, v0.y);
                *reinterpret_cast<float2 *>(CC + elem_off128(65 + n0, 2 * l)) = make_float2(v1.x, v1.y);
            }
        }
        __syncthreads();
        {   // ---- M rows l, group g, into rows 0..63 of CC (K = 2s + part)
            const int l = r64;
            const int g = 2 * sub + (upper ? 0 : 1);
            // L[l, s] = exp(Re(cs_l - cs_s)) rot_l conj(rot_s): the phase factors have modulus one,
            // so splitting them costs no range; the magnitude stays a difference
            const float lre = cs[l].x * 1.4426950408889634f;
            const float2 rl = rot[l];
            float out[16];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int s = 8 * g + j;
                const float other = E[l * E_STRIDE + s];
                const float2 cb = upper ? make_float2(own[j], other) : make_float2(other, own[j]);
                float2 m = make_float2(0.f, 0.f);
                if (s <= l) {
                    const float2 rs = rot[s];
                    const float mag = ex2(lre - cs[s].x * 1.4426950408889634f);
                    const float2 ph = make_float2(rl.x * rs.x + rl.y * rs.y, rl.y * rs.x - rl.x * rs.y);
                    m = cmul(make_float2(mag * ph.x, mag * ph.y), cb);
                }
                out[2 * j] = m.x;
                out[2 * j + 1] = m.y;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4 *>(CC + elem_off128(l, 16 * g + 4 * j)) =
                    make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
        }
        {   // swap(X^T) into the B-tile rows of BS (Xi, Xr)
            const int s = r64;
#pragma unroll
            for (int i0 = 0; i0 < 4; ++i0) {
                const int i = upper ? i0 : i0 + 4;
                const int d0 = 2 * (sub + 4 * i);
                const float4 v = *reinterpret_cast<const float4 *>(XT + elem_off(s, 2 * d0));
                *reinterpret_cast<float2 *>(BS + elem_off128(d0, 2 * s)) = make_float2(v.y, v.x);
                *reinterpret_cast<float2 *>(BS + elem_off128(d0 + 1, 2 * s)) = make_float2(v.w, v.z);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- batch 2: chain 1 [Re Ydiag ; Re Sloc] (B = conj(X^T)) and chain 2 [Im Ydiag ; Im Sloc]
        // (B = swap(X^T)), committed separately, so the upper half writes the real outputs while
        // chain 2 runs; the lower half (the state update) waits for both.
        if (tid == 0) {
            if (c + 1 < nc) {   // the X tile of the next chunk into its freed slot
                load_x(c + 1);
                in_pending = true;
            }
            for (int k = 0; k < 16; ++k) umma_tf32(tmem + TC_Y2, opdesc128(sCC, k), opdesc(sXC, k), id128, k > 0);
            umma_commit(&bar[BAR_M2]);
            for (int k = 0; k < 16; ++k) umma_tf32(tmem + TC_Y2 + 64, opdesc128(sCC, k), opdesc128(sBS, k), id128, k > 0);
            umma_commit(&bar[BAR_M3]);
            m_par = par;
            m2_pending = true;
        }
        // Every thread of a half waits on the chain barrier itself; the outcome is made uniform per
        // warp before any warp-collective TMEM access.
        if (!upper) {
            {   // Im Yraw to the upper half
                float yi[16];
                tmem_ld16(tmem + lane_base + TC_YR + 16 * sub, yi);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) E[r64 * E_STRIDE + 16 * sub + j] = yi[j];
            }
            __syncwarp();
            halves_arrive();
            if (warp == 2 && c + 1 < nc) build_tables(c + 1);   // the next chunk's tables meanwhile
            bool ok = mbar_wait_abort(&bar[BAR_M3], par, abort_);
            if (!ok) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (ok) {
                // C and B slots are free again: the next chunk's tiles overlap the state update
                if (tid == 64 && c + 1 < nc) load_cb(c + 1);
                __syncwarp();
                // ---- state of rows n: S <- exp(cs_63) S + Sloc (columns d); each (d, n) has one owner
                const int n = r64;
                float sr[16], si[16];
                tmem_ld16(tmem + lane_base + TC_Y2 + 16 * sub, sr);
                tmem_ld16(tmem + lane_base + TC_Y2 + 64 + 16 * sub, si);
                tmem_wait_ld();
                const float2 e = ecs[CQ - 1];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int d = 16 * sub + j;
                    float2 *sp = reinterpret_cast<float2 *>(BS + elem_off128(64 + d, 2 * n));
                    const float2 o = *sp;   // (Sr, Si)
                    *sp = make_float2(e.x * o.x - e.y * o.y + sr[j], e.x * o.y + e.y * o.x + si[j]);
                }
            }
        } else {
            __syncwarp();
            halves_sync();   // E holds Im Yraw
            bool ok = mbar_wait_abort(&bar[BAR_M2], par, abort_);
            if (!ok) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            const int l = r64;
            const int64_t t = t0 + l;
            const float2 e = ecs[l];
            const float *yi = E + l * E_STRIDE + 16 * sub;
            const int64_t off = ((b * p.T + t) * p.H + h) * CD + 16 * sub;
            float yr[16];
            if (ok) {   // ---- outputs of rows l: y = Ydiag + exp(cs_l) Yraw
                float dr[16];
                tmem_ld16(tmem + lane_base + TC_YR + 16 * sub, yr);
                tmem_ld16(tmem + lane_base + TC_Y2 + 16 * sub, dr);
                tmem_wait_ld();
                if (t < p.T) {
                    float o[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] = dr[j] + e.x * yr[j] - e.y * yi[j];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        reinterpret_cast<float4 *>(p.y_re + off)[j] =
                            make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                }
            }
            if (ok && p.y_im != nullptr) {
                ok = mbar_wait_abort(&bar[BAR_M3], par, abort_);
                if (!ok) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (ok) {
                    float di[16];
                    tmem_ld16(tmem + lane_base + TC_Y2 + 64 + 16 * sub, di);
                    tmem_wait_ld();
                    if (t < p.T) {
                        float o[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = di[j] + e.x * yi[j] + e.y * yr[j];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            reinterpret_cast<float4 *>(p.y_im + off)[j] =
                                make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (*abort_) break;
        if (tid == 0) m2_pending = false;   // both chains were waited for
    }
    if (*abort_) {
        // let copies and MMAs still in flight finish (bounded) before shared memory and
        // tensor memory are released
        if (tid == 0) {
            if (in_pending) mbar_wait(&bar[BAR_IN], in_par);
            if (m1_pending) mbar_wait(&bar[BAR_M1], m_par);
            if (m2_pending) {
                mbar_wait(&bar[BAR_M2], m_par);
                mbar_wait(&bar[BAR_M3], m_par);
            }
        }
    } else if (p.final_ != nullptr) {
        for (int i = tid; i < CD * CN; i += CX_THREADS) {
            const int d = i / CN, n = i % CN;
            reinterpret_cast<float2 *>(p.final_)[((b * p.H + h) * CD + d) * CN + n] =
                *reinterpret_cast<const float2 *>(BS + elem_off128(64 + d, 2 * n));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_cx() {
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

// fp32 map over a contiguous [Bt][T][H][128 floats] tensor, box {32, 1, 64, 1}, 128-byte swizzle.
bool map_cx(CUtensorMap *m, const void *ptr, int64_t Bt, int64_t T, int64_t H) {
    auto fn = encode_fn_cx();
    if (fn == nullptr) return false;
    cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)Bt};
    cuuint64_t strides[3] = {512, (cuuint64_t)(H * 512), (cuuint64_t)(T * H * 512)};
    cuuint32_t box[4] = {32, 1, (cuuint32_t)CQ, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status ssd_complex_fwd_workspace_size(const ssd_complex_problem *p, size_t *bytes) {
    if (p == nullptr || bytes == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    *bytes = HDR_WORDS * sizeof(int32_t);
    return SSD_OK;
}

ssd_status ssd_complex_fwd(const ssd_complex_problem *p, const void *x, const float *dt, const void *A,
                          const void *B, const void *C, const void *initial_states, float *y_real, float *y_imag,
                          void *final_states, void *workspace, size_t workspace_bytes, void *stream) {
    if (p == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    if (p->batch < 1 || p->seqlen < 0 || p->nheads < 1 || p->headdim < 1 || p->dstate < 1 || p->chunk_size < 1)
        return SSD_ERR_INVALID_ARGUMENT;
    if (p->headdim != CD || p->dstate != CN || p->chunk_size != CQ) return SSD_ERR_UNSUPPORTED;
    if (p->seqlen > ((int64_t)1 << 30) || p->nheads > ((int64_t)1 << 20) || p->batch * p->nheads > ((int64_t)1 << 30))
        return SSD_ERR_UNSUPPORTED;
    if (A == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    if (p->seqlen > 0 && (x == nullptr || dt == nullptr || B == nullptr || C == nullptr || y_real == nullptr))
        return SSD_ERR_INVALID_ARGUMENT;
    if (workspace == nullptr || workspace_bytes < HDR_WORDS * sizeof(int32_t)) return SSD_ERR_WORKSPACE_TOO_SMALL;
    auto al16 = [](const void *q) { return ((uintptr_t)q & 15u) == 0; };
    for (const void *q : {x, (const void *)B, (const void *)C, (const void *)y_real, (const void *)y_imag,
                          initial_states, (const void *)final_states, (const void *)workspace})
        if (q != nullptr && !al16(q)) return SSD_ERR_MISALIGNED;
    if (((uintptr_t)A & 7u) != 0 || ((uintptr_t)dt & 3u) != 0) return SSD_ERR_MISALIGNED;
    if (p->seqlen == 0 && final_states == nullptr) return SSD_OK;   // nothing to compute
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(workspace, 0, HDR_WORDS * sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
    CUtensorMap mx{}, mb{}, mc{};
    if (p->seqlen > 0) {
        if (!map_cx(&mx, x, p->batch, p->seqlen, p->nheads) || !map_cx(&mb, B, p->batch, p->seqlen, p->nheads) ||
            !map_cx(&mc, C, p->batch, p->seqlen, p->nheads))
            return SSD_ERR_CUDA;
    } else {
        // no tokens: maps are never read; the kernel only copies the initial state out
        if (!map_cx(&mx, final_states, 1, 1, 1)) return SSD_ERR_CUDA;
        mb = mx;
        mc = mx;
    }
    CxParams q{};
    q.Bt = p->batch; q.T = p->seqlen; q.H = p->nheads;
    q.dt = dt; q.A = static_cast<const float *>(A); q.init = static_cast<const float *>(initial_states);
    q.y_re = y_real; q.y_im = y_imag; q.final_ = static_cast<float *>(final_states);
    q.hdr = static_cast<int32_t *>(workspace);
    static int attr[64] = {0};
    if (ensure_smem_attr(k_complex_fwd, (int)CX_SMEM, attr) != cudaSuccess) return SSD_ERR_CUDA;
    k_complex_fwd<<<(unsigned)(p->batch * p->nheads), CX_THREADS, CX_SMEM, st>>>(mx, mb, mc, q);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
