// fused_fwd.cu -- single-pass tensor-core forward of the SSD chunked scan (bf16
// inputs, fp32 state and accumulation), headdim 64, dstate 128, chunk 128.
//
// Work decomposition.  A work unit is (sequence, head, R consecutive 128-token
// chunks).  Units are handed out in list order through an atomic ticket (the
// metadata kernel lists them by segment index, then sequence; tickets put the
// heads of one unit next to each other so the heads of a group share B/C tiles
// in L2).  For one unit a CTA:
//   phase 1  loads x, B per chunk (TMA, two stages) and accumulates, on the tensor cores, the
//            unit's end-state contribution from a zero start,
//              agg[n][p] = sum_l B[l][n] * dt[l] exp(cs_u[end] - cs_u[l]) * x[l][p],
//            then publishes agg and the unit's total log-decay;
//   carry-in folds, in a fixed order, the aggregates of the unit's predecessors
//            inside its block of KB segments and the end state published by the
//            previous block's last unit (or the initial state) -- the inter-chunk
//            propagation of the Mamba-3-Lite "SSD Reference" page ("Inter-chunk
//            propagation -- the fixed contract"), telescoped per unit, plus the
//            initial-state term.  The last unit of a block publishes its end state.
//            The association never depends on timing, so results are bitwise
//            reproducible;
//   phase 2  walks its chunks again (x, B now L2-resident) with the state in
//            registers and, per chunk on the tensor cores,
//              CB   = C B^T                           (segment-sum mask applied on chip)
//              S_c^T = B^T (w o x)                     (chunk state, w = dt exp(cs[Q-1]-cs))
//              Y_off = C S_in^T                        (carried state readout)
//              Y_diag = M x,  M = CB o exp(cs[l]-cs[s]) dt[s] 1[s<=l]
//            y = (Y_diag + exp(cs) Y_off + D x) silu(z) is written once (bf16).
// dt, cs, CB, M and chunk states never reach global memory, nor do the carried
// states unless the caller keeps them for the backward (FusedParams::states_out);
// only the per-unit aggregates / end states (fp32, small) are exchanged.
//
// Every wait (TMA, MMA completion, predecessor flags) is bounded; on expiry the
// kernel records SSD_ERR_DEVICE_TIMEOUT, stops taking work, frees its TMEM and
// exits.
#include <cudaTypedefs.h>

#include "tc_common.cuh"

namespace ssd {

namespace {

using namespace tc;

constexpr int QT = 128;   // chunk length
constexpr int PT = 64;    // head dim
constexpr int NT = 128;   // state dim
constexpr int RMAX = 5;   // max chunks per unit (states-only mode: 4, one 64-column TMEM slice each)
constexpr int RMAX_STATES = 4;
constexpr int KB = 4;     // segments per block of the carry-in fold
constexpr int NTHR = 256; // two threads per tile row / TMEM lane: half hf holds head-dim columns [32 hf, 32 hf + 32)

constexpr uint32_t X_BYTES = QT * PT * 2;    // 16 KB
constexpr uint32_t BC_BYTES = QT * NT * 2;   // 32 KB

// Shared memory (offsets from a 1024-aligned base), about 102 KB so that two CTAs
// share an SM and fill each other's load / tensor-core waits.
//   X  : x tile                     phase 1: stage-0 x (scaled in place to w o x)
//   B  : B tile                     phase 1: stage-0 B
//   C  : C tile                     phase 1: stage-1 B
//   W  : w o x, then S_in (bf16), then z (TMA), then y (TMA store)   phase 1: stage-1 x (scaled in place)
constexpr uint32_t OFF_X = 0;
constexpr uint32_t OFF_B = OFF_X + X_BYTES;        // 16384
constexpr uint32_t OFF_C = OFF_B + BC_BYTES;       // 49152
constexpr uint32_t OFF_W = OFF_C + BC_BYTES;       // 81920
constexpr uint32_t OFF_DTU = OFF_W + X_BYTES;      // 98304
constexpr uint32_t OFF_WU = OFF_DTU + RMAX * QT * 4;
constexpr uint32_t OFF_CS2 = OFF_WU + RMAX * QT * 4;    // chunk-local cumsum * log2 e, every chunk of the unit
constexpr uint32_t OFF_CF = OFF_CS2 + RMAX * QT * 4;     // per-column decay factors of the M build, every chunk
constexpr uint32_t OFF_DTN = OFF_CF + RMAX * QT * 4;     // raw dt of the next unit (cp.async during the fold)
constexpr uint32_t OFF_MISC = OFF_DTN + RMAX * QT * 4;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 256 + 1024;   // + alignment slack

// TMEM columns (256 per CTA)
constexpr uint32_t TM_CB = 0;     // [0,128) CB; then [0,64) M (bf16 pairs, the Y_diag A operand), [64,128) Y_diag
constexpr uint32_t TM_M = 0, TM_YD = 64;
constexpr uint32_t TM_SC = 128;   // [128,192) chunk state^T (phase 1: unit aggregate^T)
constexpr uint32_t TM_YO = 192;   // [192,256) C S_in^T
constexpr uint32_t TM_COLS = 256;

constexpr float LOG2E = 1.4426950408889634f;

struct FusedParams {
    Shape sh;
    int32_t *hdr;
    const UnitInfo *units;
    const float *dt_raw;
    int64_t sdb, sdl;
    const float *A, *D, *bias;
    const __nv_bfloat16 *z;
    int64_t szb, szl, szh;
    __nv_bfloat16 *y;
    int64_t syb, syl, syh;
    const float *init;
    float *final_;
    float *agg, *incl, *lam;
    uint32_t *flags;
    // Optional: the carried state entering every chunk, one 16 KB tile per (chunk, head)
    // at tile index chunk * H + head (chunk = seqs[seq].chunk0 + (t0 - seqs[seq].t0)/Q + c):
    // bf16, 128-byte row n = S[0..63][n], its 16-byte pieces q (p = 8q..8q+7) stored at
    // position q ^ (n & 7) -- the image of a 128-byte-swizzled shared-memory tile, so a
    // plain bulk copy into 1024-aligned shared memory gives the backward's MMA operand.
    // The states-only mode (template argument; used by the backward when the forward did
    // not keep them) computes nothing else: no CB, M, Y_off, Y_diag or y; phase 1 then
    // keeps each chunk's own state in TMEM, so phase 2 needs neither loads nor MMAs.
    __nv_bfloat16 *states_out;
    const SeqInfo *seqs;
};

// Barriers: x (phase-1 stage 0 / phase-2 x), b (phase-2 B), c (phase-1 stage 1 / phase-2 C),
// mma (tensor-core completion), z (phase-2 gate tile).  Each counts its own completed phases.
enum { BAR_X = 0, BAR_B = 1, BAR_C = 2, BAR_MMA = 3, BAR_Z = 4, NBAR = 5 };

struct Misc {
    uint64_t bar[NBAR];
    uint32_t tmem_base;
    int tnext;        // ticket of the next unit (taken at the start of the current one)
    int abort_;
    float wsum[8];      // chunk totals of the unit prologue
    float A_next, bias_next;   // A and dt_bias of the next unit's head (cp.async)
    UnitInfo ui_next;
};

// silu(z) = z sigmoid(z), sigmoid(z) = (1 + tanh(z/2)) / 2 (one tanh.approx).
__device__ __forceinline__ float silu_tanh(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return 0.5f * z * (1.f + t);
}

// 4-byte asynchronous global -> shared copy (completion: cp_async_wait_all by the issuing thread).
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// TMEM column (from TM_M) of M's 32-column block sb (see the M build in phase 2).
__device__ __forceinline__ uint32_t mcol(int sb) { return sb == 0 ? 0u : sb == 1 ? 32u : sb == 2 ? 48u : 16u; }

// Row n of the carried-state tile of (chunk k, head h) in FusedParams::states_out.
__device__ __forceinline__ uint8_t *state_tile_row(__nv_bfloat16 *base, int64_t k, int H, int h, int n) {
    return reinterpret_cast<uint8_t *>(base) + ((k * H + h) * (int64_t)(PT * NT) + (int64_t)n * PT) * 2;
}

// K-major SW128 operand: rows of 64 bf16 (128 B), atom columns of `col_bytes`.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int k, uint32_t col_bytes) {
    return sdesc(base + (uint32_t)(k >> 2) * col_bytes + (uint32_t)(k & 3) * 32u, 16u, 1024u);
}
// MN-major SW128 operand: K rows of 128 B; 16-row K step = 2048 B; MN atoms 16 KB apart.
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int k) {
    return sdesc(base + (uint32_t)k * 2048u, 16384u, 1024u);
}

// dst row = src row * w, half hf of the row's eight 16-byte pieces (the two halves of a
// row are disjoint; visited in swizzled order so eight consecutive rows hit eight
// different bank groups).
__device__ __forceinline__ void scale_half(const uint8_t *src_row, uint8_t *dst_row, int row, int hf, float wl) {
    const uint4 *src = reinterpret_cast<const uint4 *>(src_row);
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const int q = (4 * hf + qq) ^ (row & 7);
        uint4 v = src[q];
        __nv_bfloat162 *e = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f = __bfloat1622float2(e[i]);
            e[i] = __floats2bfloat162_rn(f.x * wl, f.y * wl);
        }
        dst[q] = v;
    }
}

// acc[i] += sc * src[i * NT] for 32 state columns p (a [P][N] state: for each column p
// the warp reads one contiguous 128-byte line).
__device__ __forceinline__ void fma_col32(float *acc, const float *src, float sc) {
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __ldcg(src + (int64_t)(j + i) * NT);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j + i] += sc * v[i];
    }
}

// Row n of a carried-state tile (bf16, 128-byte swizzled [n][p]), half hf: the four
// 16-byte pieces of columns p = 32 hf .. 32 hf + 31, from the thread's 32 values.
__device__ __forceinline__ void store_state_half(uint8_t *rowp, int row, int hf, const float *v) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(rowp + (((4 * hf + q) ^ (row & 7)) << 4)) =
            make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}

// kStatesOnly: the states-only mode (only FusedParams::states_out is written), compiled
// separately so that neither mode's code shapes the other's register allocation.
template <bool kStatesOnly>
__global__ void __launch_bounds__(NTHR, 2)
k_fused_fwd(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmZ,
            const __grid_constant__ CUtensorMap tmY, const FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & 127, hf = tid >> 7, quad = warp & 3;
    Misc *ms = reinterpret_cast<Misc *>(sm + OFF_MISC);
    float *dtu = reinterpret_cast<float *>(sm + OFF_DTU);
    float *wu = reinterpret_cast<float *>(sm + OFF_WU);
    float *cs2u = reinterpret_cast<float *>(sm + OFF_CS2);
    float *cfu = reinterpret_cast<float *>(sm + OFF_CF);
    float *dtn = reinterpret_cast<float *>(sm + OFF_DTN);
    uint8_t *Xs = sm + OFF_X, *Bs = sm + OFF_B, *Cs = sm + OFF_C, *Ws = sm + OFF_W;
    const Shape sh = p.sh;

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&ms->bar[i], 1);
        fence_mbar_init();
        ms->abort_ = 0;
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
        if (p.z) prefetch_tmap(&tmZ);
        if (p.y) prefetch_tmap(&tmY);
    }
    if (warp == 0) tmem_alloc(&ms->tmem_base, TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;

    // Per barrier, kept identically by every thread (all issue decisions are uniform):
    // the parity of its completed phases (bit b of par) and the count of issued-but-
    // unwaited operations (4-bit field b of pend, at most 2) for the drain after an
    // early stop.
    uint32_t par = 0u, pend = 0u;
    const int total = (p.hdr[HDR_STATUS] != 0) ? 0 : p.hdr[HDR_NUNITS] * sh.H;

    auto fail = [&]() {
        ms->abort_ = 1;
        set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
    };
    auto wait_bar = [&](int b) {
        if (!mbar_wait(&ms->bar[b], (par >> b) & 1u)) fail();
        par ^= 1u << b;
        pend -= 1u << (4 * b);
        if (b == BAR_MMA) tc_fence_after();
    };
    // TMA issue helpers (one thread issues; every thread counts)
    auto load_xb = [&](int b_, uint8_t *xd, uint8_t *bd, int h, int g, int t, int bb) {
        if (tid == 0) {
            uint64_t *bar = &ms->bar[b_];
            mbar_expect_tx(bar, X_BYTES + BC_BYTES);
            tma_load_4d(xd, &tmX, bar, 0, h, t, bb);
            tma_load_4d(bd, &tmB, bar, 0, g, t, bb);
            tma_load_4d(bd + BC_BYTES / 2, &tmB, bar, 64, g, t, bb);
        }
        pend += 1u << (4 * b_);
    };
    auto load_x = [&](int h, int t, int bb) {
        if (tid == 0) {
            mbar_expect_tx(&ms->bar[BAR_X], X_BYTES);
            tma_load_4d(Xs, &tmX, &ms->bar[BAR_X], 0, h, t, bb);
        }
        pend += 1u << (4 * BAR_X);
    };
    auto load_bc = [&](int b_, const CUtensorMap *map, uint8_t *dst, int g, int t, int bb) {
        if (tid == 0) {
            mbar_expect_tx(&ms->bar[b_], BC_BYTES);
            tma_load_4d(dst, map, &ms->bar[b_], 0, g, t, bb);
            tma_load_4d(dst + BC_BYTES / 2, map, &ms->bar[b_], 64, g, t, bb);
        }
        pend += 1u << (4 * b_);
    };
    auto load_z = [&](int h, int t, int bb) {
        if (tid == 0) {
            mbar_expect_tx(&ms->bar[BAR_Z], X_BYTES);
            tma_load_4d(Ws, &tmZ, &ms->bar[BAR_Z], 0, h, t, bb);
        }
        pend += 1u << (4 * BAR_Z);
    };
    auto commit = [&]() {
        if (tid == 0) umma_commit(&ms->bar[BAR_MMA]);
        pend += 1u << (4 * BAR_MMA);
    };

    const uint32_t idesc_cb = idesc_bf16(128, 128, 0, 0);
    const uint32_t idesc_sc = idesc_bf16(128, 64, 1, 1);
    const uint32_t idesc_yo = idesc_bf16(128, 64, 0, 1);
    const uint32_t idesc_yd = idesc_bf16(128, 64, 0, 1);
    const uint32_t sX = smem_u32(Xs), sB = smem_u32(Bs), sC = smem_u32(Cs), sW = smem_u32(Ws);
    const int64_t unit_stride = (int64_t)NT * PT;   // floats per (unit, head) aggregate

    // Inputs of a unit's dt prologue, fetched ahead by cp.async: thread (warp w, lane j)
    // copies raw dt of chunks w and w+4, positions 4j..4j+3 (the values it scans), thread 0
    // A and dt_bias.
    const int lane = tid & 31;
    auto fetch_unit_inputs = [&](const UnitInfo &un, int hn) {
        for (int c = warp; c < un.nchunk; c += NTHR / 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pos = c * QT + 4 * lane + i;
                if (pos >= un.lo && pos < un.len)
                    cp_async4(dtn + pos, p.dt_raw + (int64_t)un.b * p.sdb + (int64_t)(un.t0 + pos) * p.sdl + hn);
            }
        }
        if (tid == 0) {
            cp_async4(&ms->A_next, p.A + hn);
            if (p.bias) cp_async4(&ms->bias_next, p.bias + hn);
        }
    };
    if (tid == 0) {
        ms->tnext = atomicAdd(&p.hdr[HDR_TICKET], 1);
        if (ms->tnext < total) ms->ui_next = p.units[ms->tnext / sh.H];
    }
    __syncthreads();
    int ticket = ms->tnext;
    if (ticket < total) fetch_unit_inputs(ms->ui_next, ticket % sh.H);

    bool y_inflight = false;   // a y tile is being stored out of W (uniform)
    for (;;) {
        __syncthreads();
        if (tid == 0) bulk_wait_read0();   // W is refilled below (phase-1 loads)
        y_inflight = false;
        if (ticket >= total || ms->abort_) break;
        const int u = ticket / sh.H, h = ticket % sh.H, g = h / sh.hpg;
        const UnitInfo ui = ms->ui_next;
        __syncthreads();   // ui_next and tnext read: the next unit's may be written
        if (tid == 0) ms->tnext = atomicAdd(&p.hdr[HDR_TICKET], 1);   // fetched during the fold

        // phase-1 loads of the first two chunks go out first: stage 0 = (X, B), stage 1 = (W, C)
        load_xb(BAR_X, Xs, Bs, h, g, ui.t0, ui.b);
        if (ui.nchunk > 1) load_xb(BAR_C, Ws, Cs, h, g, ui.t0 + QT, ui.b);

        // ---- dt over the unit, chunk-local and unit-level cumulative log-decay, phase-1 weights.
        cp_async_wait_all();
        __syncthreads();
        const float Ah = ms->A_next;
        float lam_u;
        {   // warp w scans chunks w and w + 4 (four positions per lane); chunk totals meet in smem
            constexpr int NR = (RMAX + NTHR / 32 - 1) / (NTHR / 32);
            const float bias = p.bias ? ms->bias_next : 0.f;
            float dt4[NR][4], cs4[NR][4], last[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int c = warp + r * (NTHR / 32);
                const bool wact = c < ui.nchunk;
                float run = 0.f, loc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int pos = c * QT + 4 * lane + i;
                    dt4[r][i] = (wact && pos >= ui.lo && pos < ui.len) ? softplus_f(dtn[pos] + bias) : 0.f;
                    run += dt4[r][i] * Ah;
                    loc[i] = run;
                }
                const float incl = warp_incl_sum(run);
                const float excl = incl - run;
#pragma unroll
                for (int i = 0; i < 4; ++i) cs4[r][i] = excl + loc[i];
                last[r] = __shfl_sync(0xffffffffu, cs4[r][3], lane | 7);   // cs at the 32-block's end
                const float ctot = __shfl_sync(0xffffffffu, incl, 31);
                if (lane == 0 && c < 8) ms->wsum[c] = wact ? ctot : 0.f;
            }
            __syncthreads();
            float tot = 0.f;
            for (int c = 0; c < ui.nchunk; ++c) tot += ms->wsum[c];
            lam_u = tot;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int c = warp + r * (NTHR / 32);
                if (c >= ui.nchunk) continue;
                float off = 0.f;
                for (int c2 = 0; c2 < c; ++c2) off += ms->wsum[c2];
                float pc[4], pw[4], pf[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float cs = cs4[r][i];
                    pc[i] = cs * LOG2E;
                    pw[i] = dt4[r][i] * ex2((lam_u - (off + cs)) * LOG2E);
                    pf[i] = dt4[r][i] * ex2((last[r] - cs) * LOG2E);
                }
                const int b4 = c * QT + 4 * lane;
                *reinterpret_cast<float4 *>(dtu + b4) = make_float4(dt4[r][0], dt4[r][1], dt4[r][2], dt4[r][3]);
                *reinterpret_cast<float4 *>(cs2u + b4) = make_float4(pc[0], pc[1], pc[2], pc[3]);
                *reinterpret_cast<float4 *>(wu + b4) = make_float4(pw[0], pw[1], pw[2], pw[3]);
                *reinterpret_cast<float4 *>(cfu + b4) = make_float4(pf[0], pf[1], pf[2], pf[3]);
            }
            __syncthreads();
        }

        // ---- phase 1: unit aggregate^T[n][p] = sum_l B[l][n] (w o x)[l][p], double-buffered.
        // States-only mode keeps every chunk's own state S_c^T (chunk-local weights) in TMEM
        // columns [64c, 64c+64) instead, and forms the aggregate from them.
        constexpr bool full = !kStatesOnly;
        for (int c = 0; c < ui.nchunk; ++c) {
            const int st = c & 1;
            uint8_t *xs = st ? Ws : Xs;
            wait_bar(st ? BAR_C : BAR_X);
            const float wl = full ? wu[c * QT + row]
                                  : dtu[c * QT + row] * ex2(cs2u[c * QT + QT - 1] - cs2u[c * QT + row]);
            scale_half(xs + row * 128, xs + row * 128, row, hf, wl);   // x -> w o x in place
            fence_proxy_async_smem();
            __syncthreads();
            if (ms->abort_) break;
            if (tid == 0) {
                tc_fence_after();
                const uint32_t sb_ = smem_u32(st ? Cs : Bs), sx_ = smem_u32(xs);
                const uint32_t dcol = full ? TM_SC : 64u * (uint32_t)c;
#pragma unroll
                for (int k = 0; k < QT / 16; ++k)
                    umma_bf16(tmem + dcol, mnmaj(sb_, k), mnmaj(sx_, k), idesc_sc,
                              (k > 0 || (full && c > 0)) ? 1u : 0u);
            }
            commit();
            wait_bar(BAR_MMA);   // stage st free again
            if (c + 2 < ui.nchunk)
                load_xb(st ? BAR_C : BAR_X, xs, st ? Cs : Bs, h, g, ui.t0 + (c + 2) * QT, ui.b);
        }
        if (ms->abort_) break;
        float s_run[32];   // row n, columns p = 32 hf + i: aggregate, then carried state
        if (full) {
            tmem_ld32(tmem + lane_base + TM_SC + 32 * hf, s_run);
            tmem_wait_ld();
        } else {   // aggregate = (..(S_0 a_1 + S_1) a_2 + ..) + S_last, a_c = the chunk's decay
#pragma unroll
            for (int i = 0; i < 32; ++i) s_run[i] = 0.f;
            for (int c = 0; c < ui.nchunk; ++c) {
                const float a_c = ex2(cs2u[c * QT + QT - 1]);
                float t32[32];
                tmem_ld32(tmem + lane_base + 64u * (uint32_t)c + 32 * hf, t32);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) s_run[i] = fmaf(a_c, s_run[i], t32[i]);
            }
        }
        const int64_t my = (int64_t)u * sh.H + h;
        const int64_t col0 = (int64_t)(32 * hf) * NT;   // this thread's first column p of a [P][N] state
        {   // aggregate^T row n -> agg[p][n]
            float *dst = p.agg + my * unit_stride + col0 + row;
#pragma unroll
            for (int i = 0; i < 32; ++i) __stcg(dst + (int64_t)i * NT, s_run[i]);
            if (tid == 0) __stcg(p.lam + my, lam_u);
        }
        __threadfence();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) st_release_u32(p.flags + my, 1u);

        if (full) {   // prefetch phase-2 chunk 0 while folding the carry-in (all phase-1 MMAs are done)
            load_x(h, ui.t0, ui.b);
            load_bc(BAR_B, &tmB, Bs, g, ui.t0, ui.b);
            load_bc(BAR_C, &tmC, Cs, g, ui.t0, ui.b);
        }

        {   // the next unit: its UnitInfo and dt inputs travel while this one folds and runs phase 2
            const int tn = ms->tnext;
            if (tn < total) {
                const UnitInfo un = p.units[tn / sh.H];
                if (tid == 0) ms->ui_next = un;
                fetch_unit_inputs(un, tn % sh.H);
            }
            ticket = tn;
        }
        // ---- carry-in state of the unit (row n, all 64 columns p)
        // P_j = sum_{i=b0}^{j-1} exp(lam_{i+1} + .. + lam_{j-1}) agg_i + exp(lam_{b0} + .. + lam_{j-1}) E,
        // E = end state of unit b0-1 (published by it) or the initial state when b0 = 0.
        float agg_keep[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) { agg_keep[i] = s_run[i]; s_run[i] = 0.f; }
        const int b0 = ui.j - (ui.j % KB);
        const int nfold = ui.j - b0;     // in-block predecessors: units u-1 .. u-nfold
        const int uprev_blk = (b0 > 0) ? (nfold > 0 ? p.units[u - nfold].prev : ui.prev) : -1;
        {   // wait for the flags: thread i < nfold polls unit u-1-i (aggregate), thread nfold the block end
            int need = 0;
            int64_t fi = 0;
            if (tid < nfold) { need = 1; fi = (int64_t)(u - 1 - tid) * sh.H + h; }
            else if (tid == nfold && uprev_blk >= 0) { need = 2; fi = (int64_t)uprev_blk * sh.H + h; }
            if (need) {
                uint32_t fl = ld_acquire_u32(p.flags + fi);
                if (fl < (uint32_t)need) {
                    const uint64_t t0 = globaltimer();
                    while ((fl = ld_acquire_u32(p.flags + fi)) < (uint32_t)need) {
                        if (globaltimer() - t0 > kWaitLimitNs) break;
                        __nanosleep(64);
                    }
                }
                if (fl < (uint32_t)need) fail();
            }
            __threadfence();
            __syncthreads();
            if (ms->abort_) break;
        }
        float logm = 0.f;
        for (int i = 1; i <= nfold; ++i) {   // units u-1, u-2, .. in that order
            const int64_t pi = (int64_t)(u - i) * sh.H + h;
            const float lam_i = __ldcg(p.lam + pi);
            fma_col32(s_run, p.agg + pi * unit_stride + col0 + row, ex2(logm * LOG2E));
            logm += lam_i;
        }
        if (uprev_blk >= 0) {
            const int64_t pi = (int64_t)uprev_blk * sh.H + h;
            fma_col32(s_run, p.incl + pi * unit_stride + col0 + row, ex2(logm * LOG2E));
        } else if (p.init) {
            const float sc = ex2(logm * LOG2E);
            const float *src = p.init + ((int64_t)ui.seq * sh.H + h) * PT * NT + col0 + row;
#pragma unroll
            for (int i = 0; i < 32; ++i) s_run[i] += sc * src[(int64_t)i * NT];
        }
        if ((ui.j % KB) == KB - 1 && !ui.last) {   // block end: publish the unit's end state
            const float dec = ex2(lam_u * LOG2E);
            float *dst = p.incl + my * unit_stride + col0 + row;
#pragma unroll
            for (int i = 0; i < 32; ++i) __stcg(dst + (int64_t)i * NT, agg_keep[i] + dec * s_run[i]);
            __threadfence();
            __syncthreads();
            if (tid == 0) st_release_u32(p.flags + my, 2u);
        }

        // ---- phase 2, states-only mode: the carried state entering every chunk, from the chunk
        // states kept in TMEM (no loads, no MMAs)
        if (!full) {
            const int64_t kfirst = (int64_t)p.seqs[ui.seq].chunk0 + ui.t0 / QT - p.seqs[ui.seq].t0 / QT;
            for (int c = 0; c < ui.nchunk; ++c) {
                store_state_half(state_tile_row(p.states_out, kfirst + c, sh.H, h, row), row, hf, s_run);
                const float a_c = ex2(cs2u[c * QT + QT - 1]);
                float t32[32];
                tmem_ld32(tmem + lane_base + 64u * (uint32_t)c + 32 * hf, t32);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) s_run[i] = fmaf(a_c, s_run[i], t32[i]);
            }
            tc_fence_before();
            __syncthreads();   // TMEM read: the next unit's phase 1 may overwrite it
            continue;
        }
        // ---- phase 2: outputs
        const float Dh = p.D ? p.D[h] : 0.f;
        const int64_t kfirst = (int64_t)p.seqs[ui.seq].chunk0 + ui.t0 / QT - p.seqs[ui.seq].t0 / QT;
        for (int c = 0; c < ui.nchunk; ++c) {
            const int tc0 = ui.t0 + c * QT;
            const int clen = min(QT, ui.len - c * QT);
            const int clo = c == 0 ? ui.lo : 0;   // rows [clo, clen) are this sequence's
            const bool more = c + 1 < ui.nchunk;
            const int64_t tok = (int64_t)tc0 + row;
            const bool has_z = p.z != nullptr;
            // chunk-local cumulative log-decay (computed at unit start)
            const float *cs2 = cs2u + c * QT;
            const float *dtc = dtu + c * QT;
            const float *cf = cfu + c * QT;
            const float a_c = ex2(cs2[QT - 1]);
            wait_bar(BAR_B);
            {   // CB = C B^T (K = state dim) runs while x is scaled; committed with S_c below
                wait_bar(BAR_C);
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < NT / 16; ++k)
                        umma_bf16(tmem + TM_CB, kmaj(sC, k, BC_BYTES / 2), kmaj(sB, k, BC_BYTES / 2), idesc_cb, k > 0);
                }
            }
            wait_bar(BAR_X);
            if (y_inflight) {   // the previous chunk's y tile is still being read out of W
                if (tid == 0) bulk_wait_read0();
                __syncthreads();
                y_inflight = false;
            }
            // W = w o x, w[l] = dt[l] exp(cs[Q-1] - cs[l])
            scale_half(Xs + row * 128, Ws + row * 128, row, hf, dtc[row] * ex2(cs2[QT - 1] - cs2[row]));
            fence_proxy_async_smem();
            __syncthreads();
            if (ms->abort_) {
                commit();   // the CB MMAs are in flight: the drain waits for them
                break;
            }
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < QT / 16; ++k)   // S_c^T = B^T (w o x) (K = tokens)
                    umma_bf16(tmem + TM_SC, mnmaj(sB, k), mnmaj(sW, k), idesc_sc, k > 0);
            }
            commit();   // one barrier phase per commit, waited before the next commit: a parity
            wait_bar(BAR_MMA);   // wait cannot tell a barrier two phases ahead from one behind
            if (full && more) load_bc(BAR_B, &tmB, Bs, g, tc0 + QT, ui.b);   // B is read by CB and S_c only
            if (full) {
                // S_in (bf16, MN-major [n][p]: row n = this thread's 64 columns) over the w o x
                // buffer, then Y_off = C S_in^T
                {   // (and the same bytes to the chunk-state tile when the caller keeps them)
                    uint8_t *rowp = Ws + row * 128;
                    uint8_t *grow = p.states_out ? state_tile_row(p.states_out, kfirst + c, sh.H, h, row) : nullptr;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 v =
                            make_uint4(pack_bf16(s_run[8 * q], s_run[8 * q + 1]), pack_bf16(s_run[8 * q + 2], s_run[8 * q + 3]),
                                       pack_bf16(s_run[8 * q + 4], s_run[8 * q + 5]), pack_bf16(s_run[8 * q + 6], s_run[8 * q + 7]));
                        const int pos = ((4 * hf + q) ^ (row & 7)) << 4;
                        *reinterpret_cast<uint4 *>(rowp + pos) = v;
                        if (grow) *reinterpret_cast<uint4 *>(grow + pos) = v;
                    }
                }
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < NT / 16; ++k)   // Y_off = C S_in^T (K = state dim)
                        umma_bf16(tmem + TM_YO, kmaj(sC, k, BC_BYTES / 2), mnmaj(sW, k), idesc_yo, k > 0);
                }
                commit();
                // M (bf16, [l][s], D on the diagonal) into TMEM while Y_off runs.  The two threads
                // of row l take two of its four 32-column blocks each (hf 0: blocks 0 and 3, hf 1:
                // blocks 1 and 2, so the causal work is split evenly).  M lives in CB's first 64
                // columns; each thread stores its two M blocks (16 columns each) over the CB block
                // it read first (hf 0 over CB block 0, hf 1 over CB block 1), which no other thread
                // reads, so no thread overwrites CB that another still needs.  M block sb thus sits
                // at column mcol(sb) = {0, 32, 48, 16}[sb]; Y_diag's K steps follow that order.
                const int l = row;
                const float cl = cs2[l];
#pragma unroll
                for (int bi = 0; bi < 2; ++bi) {
                    const int sb = hf == 0 ? (bi == 0 ? 0 : 3) : (bi == 0 ? 1 : 2);
                    uint32_t pk[16];
                    if (sb < quad) {
                        // strictly below the diagonal: exp(cs[l]-cs[s]) = exp(cs[l]-cs[e]) exp(cs[e]-cs[s]),
                        // e = last token of the block; both factors <= 1, so neither overflows
                        float cb[32];
                        tmem_ld32(tmem + lane_base + TM_CB + sb * 32, cb);
                        const float rl = ex2(cl - cs2[sb * 32 + 31]);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            pk[i >> 1] = pack_bf16(cb[i] * rl * cf[sb * 32 + i], cb[i + 1] * rl * cf[sb * 32 + i + 1]);
                    } else if (sb == quad) {   // diagonal block: causal mask, D on the diagonal
                        float cb[32];
                        tmem_ld32(tmem + lane_base + TM_CB + sb * 32, cb);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const int s0 = sb * 32 + i;
                            float m0 = (s0 <= l) ? cb[i] * ex2(cl - cs2[s0]) * dtc[s0] : 0.f;
                            float m1 = (s0 + 1 <= l) ? cb[i + 1] * ex2(cl - cs2[s0 + 1]) * dtc[s0 + 1] : 0.f;
                            if (s0 == l) m0 += Dh;
                            if (s0 + 1 == l) m1 += Dh;
                            pk[i >> 1] = pack_bf16(m0, m1);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = 0u;
                    }
                    // row l of M block sb: 16 packed pairs into this lane's TMEM, over CB columns
                    // this thread has already read
                    tmem_st16(tmem + lane_base + TM_M + mcol(sb), pk);
                }
            }
            {   // carried state update: S_in[c+1] = a_c S_in[c] + S_c (row n, this half's columns)
                float sc[32];
                tmem_ld32(tmem + lane_base + TM_SC + 32 * hf, sc);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) s_run[i] = a_c * s_run[i] + sc[i];
            }
            wait_bar(BAR_MMA);   // Y_off done: C and W free
            if (has_z) load_z(h, tc0, ui.b);
            if (more) load_bc(BAR_C, &tmC, Cs, g, tc0 + QT, ui.b);
            tmem_wait_st();
            tc_fence_before();
            __syncthreads();   // M in TMEM
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < QT / 16; ++k)   // Y_diag + D x = M x (K = source tokens), M from TMEM
                    umma_bf16_ta(tmem + TM_YD, tmem + TM_M + mcol(k >> 1) + 8 * (k & 1), mnmaj(sX, k), idesc_yd, k > 0);
            }
            commit();
            wait_bar(BAR_MMA);   // x free: next chunk's x
            if (more) load_x(h, tc0 + QT, ui.b);
            if (has_z) wait_bar(BAR_Z);
            // full chunks: y rows go into W (in place of the gate rows just read) and leave as
            // one TMA store; a chunk shared with another packed sequence stores its own rows
            // directly
            const bool tile_out = clen == QT && clo == 0;
            {   // epilogue: row l, this thread's half of the columns
                const int l = row;
                const float el = ex2(cs2[l]);
                __nv_bfloat16 *yrow = p.y + (int64_t)ui.b * p.syb + tok * p.syl + (int64_t)h * p.syh;
                const uint8_t *zrow = Ws + l * 128;
#pragma unroll
                for (int qq = 0; qq < 4; qq += 2) {   // two passes of 16 columns
                    const int q0 = 4 * hf + qq;       // first 16-byte piece (8 columns) of the pass
                    float yd[16], yo[16];
                    tmem_ld16(tmem + lane_base + TM_YD + 8 * q0, yd);
                    tmem_ld16(tmem + lane_base + TM_YO + 8 * q0, yo);
                    tmem_wait_ld();
                    if (l >= clo && l < clen) {
#pragma unroll
                        for (int qi = 0; qi < 2; ++qi) {
                            const int q = q0 + qi;
                            uint4 zq = make_uint4(0u, 0u, 0u, 0u);
                            if (has_z) zq = *reinterpret_cast<const uint4 *>(zrow + ((q ^ (l & 7)) << 4));
                            const __nv_bfloat162 *ze = reinterpret_cast<const __nv_bfloat162 *>(&zq);
                            uint32_t o[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int j = qi * 8 + 2 * i;
                                float v0 = yd[j] + el * yo[j];
                                float v1 = yd[j + 1] + el * yo[j + 1];
                                if (has_z) {
                                    const float2 zf = __bfloat1622float2(ze[i]);
                                    v0 *= silu_tanh(zf.x);
                                    v1 *= silu_tanh(zf.y);
                                }
                                o[i] = pack_bf16(v0, v1);
                            }
                            const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
                            if (tile_out)
                                *reinterpret_cast<uint4 *>(Ws + l * 128 + ((q ^ (l & 7)) << 4)) = ov;
                            else
                                *reinterpret_cast<uint4 *>(yrow + q * 8) = ov;
                        }
                    }
                }
            }
            if (tile_out) fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tile_out) {
                if (tid == 0) {
                    tma_store_4d(&tmY, Ws, 0, h, tc0, ui.b);
                    bulk_commit();
                }
                y_inflight = true;
            }
        }
        if (ms->abort_) break;
        if (ui.last && p.final_) {
            float *dst = p.final_ + ((int64_t)ui.seq * sh.H + h) * PT * NT + col0 + row;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[(int64_t)i * NT] = s_run[i];
        }
    }
    // Drain (only non-empty after an early stop): bounded waits for loads and
    // MMAs still in flight, so nothing lands in shared memory or TMEM after exit.
    cp_async_wait_all();
    if (tid == 0) bulk_wait0();   // y stores
    for (int b_ = 0; b_ < NBAR; ++b_)
        for (uint32_t q = 0; q < ((pend >> (4 * b_)) & 15u); ++q) mbar_wait(&ms->bar[b_], ((par >> b_) ^ q) & 1u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 4-D bf16 map over [B][L][H or G][64*k] with box {64, 1, 128, 1}, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int64_t inner, int64_t d1, int64_t L, int64_t B, int64_t s1,
              int64_t sL, int64_t sB) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)d1, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)(s1 * 2), (cuuint64_t)(sL * 2), (cuuint64_t)(sB * 2)};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)QT, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int fused_rmax() { return RMAX; }
int fused_rmax_states() { return RMAX_STATES; }
int fused_block_units() { return KB; }

cudaError_t launch_fused_fwd(const Shape &sh, int32_t *hdr, const UnitInfo *units, const void *x, const int64_t *sx,
                             const void *Bp, const int64_t *sb, const void *Cp, const int64_t *sc, const float *dt_raw,
                             int64_t sdb, int64_t sdl, const float *A, const float *D, const float *bias,
                             const void *z, const int64_t *sz, void *y, const int64_t *sy, const float *init,
                             float *final_, float *agg, float *incl, float *lam, uint32_t *flags, int grid,
                             __nv_bfloat16 *states_out, bool states_only, const SeqInfo *seqs, cudaStream_t st) {
    CUtensorMap mx, mb, mc, mz, my;
    if (!make_map(&mx, x, PT, sh.H, sh.L, sh.B, sx[2], sx[1], sx[0])) return cudaErrorInvalidValue;
    if (z != nullptr) {
        if (!make_map(&mz, z, PT, sh.H, sh.L, sh.B, sz[2], sz[1], sz[0])) return cudaErrorInvalidValue;
    } else {
        mz = mx;
    }
    if (!make_map(&mb, Bp, sh.Nio, sh.G, sh.L, sh.B, sb[2], sb[1], sb[0])) return cudaErrorInvalidValue;
    if (y != nullptr) {
        if (!make_map(&my, y, PT, sh.H, sh.L, sh.B, sy[2], sy[1], sy[0])) return cudaErrorInvalidValue;
    } else {
        my = mx;   // not written (states-only mode)
    }
    if (!make_map(&mc, Cp, sh.Nio, sh.G, sh.L, sh.B, sc[2], sc[1], sc[0])) return cudaErrorInvalidValue;
    FusedParams fp;
    fp.sh = sh; fp.hdr = hdr; fp.units = units; fp.dt_raw = dt_raw; fp.sdb = sdb; fp.sdl = sdl;
    fp.A = A; fp.D = D; fp.bias = bias;
    fp.z = (const __nv_bfloat16 *)z;
    fp.szb = sz ? sz[0] : 0; fp.szl = sz ? sz[1] : 0; fp.szh = sz ? sz[2] : 0;
    fp.y = (__nv_bfloat16 *)y; fp.syb = sy[0]; fp.syl = sy[1]; fp.syh = sy[2];
    fp.init = init; fp.final_ = final_; fp.agg = agg; fp.incl = incl; fp.lam = lam; fp.flags = flags;
    fp.states_out = states_out; fp.seqs = seqs;
    if (states_only) {
        if (states_out == nullptr) return cudaErrorInvalidValue;
        static int attr_done_s[64] = {0};
        cudaError_t e = ensure_smem_attr(k_fused_fwd<true>, (int)SMEM_BYTES, attr_done_s);
        if (e != cudaSuccess) return e;
        k_fused_fwd<true><<<grid, NTHR, SMEM_BYTES, st>>>(mx, mb, mc, mz, my, fp);
    } else {
        static int attr_done[64] = {0};
        cudaError_t e = ensure_smem_attr(k_fused_fwd<false>, (int)SMEM_BYTES, attr_done);
        if (e != cudaSuccess) return e;
        k_fused_fwd<false><<<grid, NTHR, SMEM_BYTES, st>>>(mx, mb, mc, mz, my, fp);
    }
    return cudaGetLastError();
}

}  // namespace ssd
