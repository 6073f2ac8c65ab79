// split_fwd.cu -- tensor-core forward of the SSD chunked scan in three launches with no
// waits between CTAs (bf16 inputs, fp32 state and accumulation; headdim 64, dstate 128,
// chunk 128).  The chunkwise decomposition of the Mamba-3-Lite "SSD Reference" page
// (section "ssd_complex_chunkwise -- the production scan"), one launch per stage:
//
//   k_split_states   per (chunk tile, group, subset of its heads): the chunk state
//                      S_c^T[n][p] = sum_l B[l][n] dt[l] exp(cs[Q-1] - cs[l]) x[l][p]
//                    on the tensor cores (section "Intra-chunk outputs and per-chunk
//                    states"), written as a bf16 [n][p] tile (128-byte swizzled rows), and
//                    the chunk's total log-decay cs[Q-1];
//   k_split_passing  per (sequence, head), over its chunks in order, in fp32 registers:
//                      S_in[first] = initial state,  S_in[c+1] = exp(cs_c[Q-1]) S_in[c] + S_c
//                    ("Inter-chunk propagation -- the fixed contract"), overwriting each
//                    tile's S_c with the S_in entering it, and the final state after the
//                    last chunk;
//   k_split_out      per (chunk tile, group, subset of its heads): CB = C B^T once, then
//                    per head Y_off = C S_in^T and Y_diag = M x with M = CB o exp(cs[l] -
//                    cs[s]) dt[s] 1[s<=l] (+ D on the diagonal), y = (Y_diag + exp(cs) Y_off)
//                    silu(z) ("Readout").  The heads of an item run two deep: head i's MMAs
//                    run while head i-1's outputs are formed, and one warp does nothing but
//                    issue the copies and the MMAs.
//
// The carried-state tiles are exactly the ones the backward reads (ssd_fwd_args.
// chunk_states): when the caller keeps them, the first two launches write them there.
// Every wait is bounded; on expiry a kernel records SSD_ERR_DEVICE_TIMEOUT, drains what
// it has in flight, frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <algorithm>

#include "tc_common.cuh"

namespace ssd {

namespace {

using namespace tc;

constexpr int QT = 128, PT = 64, NT = 128;
constexpr uint32_t X_BYTES = QT * PT * 2;    // 16 KB: a [token][p] tile, or a [n][p] state tile
constexpr uint32_t BC_BYTES = QT * NT * 2;   // 32 KB
constexpr int HSMAX = 8;                     // heads per work item at most
constexpr float LOG2E = 1.4426950408889634f;

struct SplitParams {
    Shape sh;
    int32_t *hdr;
    const ChunkInfo *chunks;
    const SeqInfo *seqs;
    int hs;                       // heads per work item (divides H/G, <= HSMAX)
    int n_items;                  // work items: (chunk tile, group, head subset), chunk-major
    const float *dt_raw;
    int64_t sdb, sdl;
    const float *A, *D, *bias;
    __nv_bfloat16 *y;
    int64_t syb, syl, syh;
    const float *init;
    float *final_;
    __nv_bfloat16 *states;        // one 16 KB tile per (chunk tile, head): S_c, then S_in
    float *lam;                   // [chunk tile][H] total log-decay of the tile
    bool z_present;
};

__device__ __forceinline__ uint64_t kmaj(uint32_t base, int k, uint32_t col_bytes) {
    return sdesc(base + (uint32_t)(k >> 2) * col_bytes + (uint32_t)(k & 3) * 32u, 16u, 1024u);
}
// MN-major SW128 operand: K rows of 128 B; 16-row K step = 2048 B; MN atoms 16 KB apart.
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int k) { return sdesc(base + (uint32_t)k * 2048u, 16384u, 1024u); }

__device__ __forceinline__ float silu_tanh(float z) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return 0.5f * z * (1.f + t);
}

// Row n of the 16 KB state tile of (chunk tile k, head h).
__device__ __forceinline__ uint8_t *tile_row(__nv_bfloat16 *base, int64_t k, int H, int h, int n) {
    return reinterpret_cast<uint8_t *>(base) + ((k * H + h) * (int64_t)(PT * NT) + (int64_t)n * PT) * 2;
}

// Decodes work item `it` into (chunk tile k, group g, first head h0).
__device__ __forceinline__ void item_of(int it, const Shape &sh, int hs, int &k, int &g, int &h0) {
    const int nsub = sh.hpg / hs, per_chunk = sh.G * nsub;
    k = it / per_chunk;
    const int r = it - k * per_chunk;
    g = r / nsub;
    h0 = g * sh.hpg + (r - g * nsub) * hs;
}

// Warp w < hs: the head h0 + w's in-chunk scan.  Lane j holds positions 4j .. 4j+3: dt :=
// softplus(dt_raw + bias) on the tile's rows [lo, len), 0 elsewhere; cs = inclusive cumsum
// of dt A.  Returns the chunk's total log-decay (all lanes).
__device__ __forceinline__ float head_scan(const SplitParams &p, const ChunkInfo &ci, int h, float (&dt4)[4],
                                           float (&cs4)[4]) {
    const int lane = threadIdx.x & 31;
    const float Ah = p.A[h], bias = p.bias ? p.bias[h] : 0.f;
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int pos = 4 * lane + i;
        float d = 0.f;
        if (pos >= ci.lo && pos < ci.len)
            d = softplus_f(p.dt_raw[(int64_t)ci.b * p.sdb + (int64_t)(ci.t0 + pos) * p.sdl + h] + bias);
        dt4[i] = d;
        run += d * Ah;
        cs4[i] = run;
    }
    const float incl = warp_incl_sum(run);
    const float excl = incl - run;
#pragma unroll
    for (int i = 0; i < 4; ++i) cs4[i] += excl;
    return __shfl_sync(0xffffffffu, incl, 31);
}

// ================================================================== chunk states
// Persistent, 288 threads: warps 0-7 scale x and read the states out (row r = tid & 127 of a
// tile, half hf = tid >> 7 of its head-dim columns); warp 8 lane 0 (the issuer) takes work
// items from a ticket and issues the copies and the MMAs.  The two sides meet on mbarriers
// only.  Shared memory: the B tile, two x stages, per-head weights w.  TMEM: two 64-column
// slots (a head's state S_c^T, row n per lane).
constexpr uint32_t ST_OFF_B = 0, ST_OFF_X = BC_BYTES, ST_OFF_W = ST_OFF_X + 2 * X_BYTES;
constexpr uint32_t ST_OFF_MISC = ST_OFF_W + HSMAX * QT * 4;
constexpr uint32_t ST_SMEM = ST_OFF_MISC + 256 + 1024;
constexpr int ST_THREADS = 288, ST_ISSUER = 256, NEW = 256;   // NEW: element-wise threads
constexpr int ST_CTAS_PER_SM = 3;
// barriers: B tile, x stages (2), w o x ready (2, NEW arrivals), MMA slots (2), slot read out (2, NEW arrivals)
enum { SB_B = 0, SB_X = 1, SB_W = 3, SB_MMA = 5, SB_DONE = 7, SB_N = 9 };
struct StMisc {
    uint64_t bar[SB_N];
    uint32_t tmem;
    int item, abort_;
};

__global__ void __launch_bounds__(ST_THREADS, 2)
k_split_states(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB, const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, hf = (tid >> 7) & 1;
    const Shape sh = p.sh;
    const int HS = p.hs;
    float *wt = reinterpret_cast<float *>(sm + ST_OFF_W);   // [HS][QT]
    StMisc *ms = reinterpret_cast<StMisc *>(sm + ST_OFF_MISC);
    uint64_t *bar = ms->bar;
    volatile int *abort_ = &ms->abort_;
    const bool issuer = tid == ST_ISSUER, ew = tid < NEW;
    if (issuer) {
        mbar_init(&bar[SB_B], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[SB_X + s], 1);
            mbar_init(&bar[SB_W + s], NEW);
            mbar_init(&bar[SB_MMA + s], 1);
            mbar_init(&bar[SB_DONE + s], NEW);
        }
        fence_mbar_init();
        ms->abort_ = 0;
    }
    if (warp == 0) tmem_alloc(&ms->tmem, 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t idesc = idesc_bf16(128, 64, 1, 1);
    const uint32_t sB = smem_u32(sm + ST_OFF_B);
    const int total = p.hdr[HDR_STATUS] != 0 ? 0 : p.n_items;
    // Phase parity of the next completion of each barrier a side waits on (bit b), and the
    // issuer's bookkeeping: stages whose x copy is issued and unwaited (xout), slots whose MMA
    // is issued and unwaited by it (mout), slots holding a state not yet read out (occ), a B
    // copy in flight.
    uint32_t ph = 0u, xout = 0u, mout = 0u, occ = 0u;
    uint32_t xiss = 0u, xlast = 0u;   // issuer: parity of the next / the last x copy's phase per stage
    bool bout = false;
    auto issue_x = [&](int s, int h, const ChunkInfo &c) {
        mbar_expect_tx(&bar[SB_X + s], X_BYTES);
        tma_load_4d(sm + ST_OFF_X + s * X_BYTES, &tmX, &bar[SB_X + s], 0, h, c.t0, c.b);
        xout |= 1u << s;
        xlast = (xlast & ~(1u << s)) | (xiss & (1u << s));
        xiss ^= 1u << s;
    };
    auto waitb = [&](int b) -> bool {
        const bool ok = mbar_wait_abort(&bar[b], (ph >> b) & 1u, abort_);
        ph ^= 1u << b;
        return ok;
    };
    for (;;) {
        if (issuer) ms->item = atomicAdd(&p.hdr[HDR_TICKET], 1);
        __syncthreads();
        const int it = ms->item;
        if (it >= total || *abort_) break;
        int k, g, h0;
        item_of(it, sh, HS, k, g, h0);
        if (k >= p.hdr[HDR_NCHUNKS]) continue;
        const ChunkInfo ci = p.chunks[k];
        if (issuer) {   // B once; x of the first two heads (each stage's last MMA must be done)
            for (int s = 0; s < 2; ++s)
                if (mout & (1u << s)) {
                    waitb(SB_MMA + s);
                    mout &= ~(1u << s);
                }
            mbar_expect_tx(&bar[SB_B], BC_BYTES);
            tma_load_4d(sm + ST_OFF_B, &tmB, &bar[SB_B], 0, g, ci.t0, ci.b);
            tma_load_4d(sm + ST_OFF_B + BC_BYTES / 2, &tmB, &bar[SB_B], 64, g, ci.t0, ci.b);
            bout = true;
            for (int s = 0; s < 2 && s < HS; ++s) issue_x(s, h0 + s, ci);
        }
        if (warp < HS) {   // per-head weights w = dt exp(cs[Q-1] - cs) and the tile's log-decay
            float dt4[4], cs4[4];
            const float tot = head_scan(p, ci, h0 + warp, dt4, cs4);
            const int lane = tid & 31;
#pragma unroll
            for (int i = 0; i < 4; ++i) wt[warp * QT + 4 * lane + i] = dt4[i] * ex2((tot - cs4[i]) * LOG2E);
            if (lane == 0) p.lam[(int64_t)k * sh.H + h0 + warp] = tot;
        }
        __syncthreads();
        if (ew) {
            // head i: x -> w o x in place; then head i-1's state (its MMA done) leaves TMEM for its tile
            auto readout = [&](int i) {
                float v[32];
                tmem_ld32(tmem + lane_base + 64u * (uint32_t)(i & 1) + 32u * hf, v);
                tmem_wait_ld();
                uint8_t *dst = tile_row(p.states, k, sh.H, h0 + i, row);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(dst + (((4 * hf + q) ^ (row & 7)) << 4)) =
                        make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                   pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
            };
            for (int i = 0; i <= HS; ++i) {
                const int st = i & 1;
                if (i < HS) {
                    if (waitb(SB_X + st)) {
                        const float wl = wt[i * QT + row];
                        uint4 *r4 = reinterpret_cast<uint4 *>(sm + ST_OFF_X + st * X_BYTES + row * 128);
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq) {
                            const int q = (4 * hf + qq) ^ (row & 7);
                            uint4 u = r4[q];
                            __nv_bfloat162 *e = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 f = __bfloat1622float2(e[j]);
                                e[j] = __floats2bfloat162_rn(f.x * wl, f.y * wl);
                            }
                            r4[q] = u;
                        }
                        fence_proxy_async_smem();
                    }
                    mbar_arrive(&bar[SB_W + st]);
                }
                if (i >= 1) {
                    const int so = st ^ 1;
                    if (waitb(SB_MMA + so)) {
                        tc_fence_after();
                        readout(i - 1);
                    }
                    tc_fence_before();
                    mbar_arrive(&bar[SB_DONE + so]);
                }
            }
        }
        if (issuer) {
            for (int i = 0; i < HS && !*abort_; ++i) {
                const int st = i & 1, so = st ^ 1;
                if (!waitb(SB_W + st)) break;   // w o x of head i in its stage
                xout &= ~(1u << st);
                if (occ & (1u << st)) {          // the slot's previous state has been read out
                    if (!waitb(SB_DONE + st)) break;
                    occ &= ~(1u << st);
                }
                if (bout) {
                    if (!waitb(SB_B)) break;
                    bout = false;
                }
                tc_fence_after();
                const uint32_t sx = smem_u32(sm + ST_OFF_X + st * X_BYTES);
#pragma unroll
                for (int kk = 0; kk < QT / 16; ++kk)   // S_c^T[n][p] = sum_l B[l][n] (w o x)[l][p]
                    umma_bf16(tmem + 64u * (uint32_t)st, mnmaj(sB, kk), mnmaj(sx, kk), idesc, kk > 0);
                umma_commit(&bar[SB_MMA + st]);
                mout |= 1u << st;
                occ |= 1u << st;
                if (i >= 1 && i + 1 < HS) {   // head i-1's MMA has read its stage: head i+1's x goes there
                    if (!waitb(SB_MMA + so)) break;
                    mout &= ~(1u << so);
                    issue_x(so, h0 + i + 1, ci);
                }
            }
        }
    }
    if (issuer) {   // every copy and MMA issued has landed before the CTA's memory goes
        if (bout) mbar_wait(&bar[SB_B], (ph >> SB_B) & 1u);
        for (int s = 0; s < 2; ++s) {
            if (xout & (1u << s)) mbar_wait(&bar[SB_X + s], (xlast >> s) & 1u);
            if (mout & (1u << s)) mbar_wait(&bar[SB_MMA + s], (ph >> (SB_MMA + s)) & 1u);
        }
        if (*abort_) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ================================================================== state passing
// grid (S * H, 4), 256 threads: thread = one 16-byte piece (8 bf16) of every tile of
// (sequence, head): piece j = 256 blockIdx.y + tid holds row n = j / 8, columns p = 8 q ..
// 8 q + 7 with q = (j % 8) ^ (n % 8).  Its eight fp32 carries walk the sequence's tiles in
// order, eight tiles' loads in flight at a time.
__global__ void __launch_bounds__(256)
k_split_passing(const SplitParams p) {
    constexpr int CB = 8;
    const Shape sh = p.sh;
    if (p.hdr[HDR_STATUS] != 0) return;
    const int s = blockIdx.x / sh.H, h = blockIdx.x % sh.H, lane = threadIdx.x & 31;
    const int j = blockIdx.y * 256 + threadIdx.x, n = j >> 3, q = (j & 7) ^ (n & 7);
    const SeqInfo si = p.seqs[s];
    const int nch = si.nch;
    const int64_t sbase = ((int64_t)s * sh.H + h) * PT * NT;
    float c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = p.init ? p.init[sbase + (int64_t)(8 * q + e) * NT + n] : 0.f;
    auto piece = [&](int pos) {
        return reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.states) +
                                         (((int64_t)(si.chunk0 + pos) * sh.H + h) * (PT * NT) + (int64_t)j * 8) * 2);
    };
    for (int c0 = 0; c0 < nch; c0 += CB) {
        const int nc = min(CB, nch - c0);
        const float mydec = lane < nc ? expf(p.lam[(int64_t)(si.chunk0 + c0 + lane) * sh.H + h]) : 0.f;
        uint4 v[CB];
#pragma unroll
        for (int t = 0; t < CB; ++t) v[t] = t < nc ? *piece(c0 + t) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int t = 0; t < CB; ++t) {
            const float d = __shfl_sync(0xffffffffu, mydec, t);
            if (t < nc) {
                *piece(c0 + t) = make_uint4(pack_bf16(c[0], c[1]), pack_bf16(c[2], c[3]), pack_bf16(c[4], c[5]),
                                            pack_bf16(c[6], c[7]));   // the state entering the tile
                const __nv_bfloat162 *e2 = reinterpret_cast<const __nv_bfloat162 *>(&v[t]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(e2[e]);
                    c[2 * e] = fmaf(d, c[2 * e], f.x);
                    c[2 * e + 1] = fmaf(d, c[2 * e + 1], f.y);
                }
            }
        }
    }
    if (p.final_ != nullptr && nch > 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) p.final_[sbase + (int64_t)(8 * q + e) * NT + n] = c[e];
    }
}

// ================================================================== outputs
// Persistent, one CTA per SM, 288 threads: warps 0-7 form M and the outputs (row r = tid &
// 127, half hf = (tid >> 7) & 1 of the head-dim columns); warp 8 lane 0 (the issuer) takes work
// items from a ticket and issues every copy, MMA and store.  The two sides meet on mbarriers
// only, so head i's MMAs run while head i-1's outputs are formed.  Shared memory: B, C; two
// slots of {x, z, S_in} (y is written over z, each thread over the z pieces it has just read,
// and leaves by one TMA store); per-head tables.  TMEM (512 columns): CB [0,128), slot s at
// 128 + 192 s: M (bf16 pairs) [+0,+64), Y_off [+64,+128), Y_diag [+128,+192).
constexpr int OUT_THREADS = 288, ISSUER = 256;
constexpr uint32_t O_B = 0, O_C = BC_BYTES, O_SLOT = 2 * BC_BYTES;
constexpr uint32_t SLOT_BYTES = 3 * X_BYTES;   // x, z (then y), S_in
constexpr uint32_t S_X = 0, S_Z = X_BYTES, S_S = 2 * X_BYTES;
constexpr uint32_t O_TAB = O_SLOT + 2 * SLOT_BYTES;
constexpr uint32_t TAB_FLOATS = 4 * QT;        // per head: dt, cs log2 e, block factors, exp(cs)
constexpr uint32_t O_MISC = O_TAB + HSMAX * TAB_FLOATS * 4;
constexpr uint32_t OUT_SMEM = O_MISC + 256 + 1024;
constexpr uint32_t TM_CB = 0, TM_SLOT0 = 128, TM_SLOT = 192;
// barriers: B/C tiles, CB MMA, slot inputs (2), slot MMAs (2), M ready (2, NEW arrivals),
// slot outputs formed (2, NEW arrivals)
enum { OB_BC = 0, OB_CB = 1, OB_IN = 2, OB_MMA = 4, OB_MRDY = 6, OB_FREE = 8, OB_N = 10 };
struct OutMisc {
    uint64_t bar[OB_N];
    uint32_t tmem;
    int item, abort_;
};

__global__ void __launch_bounds__(OUT_THREADS, 1)
k_split_out(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmZ,
            const __grid_constant__ CUtensorMap tmY, const SplitParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, row = tid & 127, hf = (tid >> 7) & 1;
    const Shape sh = p.sh;
    const int HS = p.hs;
    const bool has_z = p.z_present;
    float *tab = reinterpret_cast<float *>(sm + O_TAB);   // [HS][4][QT]
    OutMisc *ms = reinterpret_cast<OutMisc *>(sm + O_MISC);
    uint64_t *bar = ms->bar;
    volatile int *abort_ = &ms->abort_;
    const bool issuer = tid == ISSUER, ew = tid < NEW;
    if (issuer) {
        mbar_init(&bar[OB_BC], 1);
        mbar_init(&bar[OB_CB], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[OB_IN + s], 1);
            mbar_init(&bar[OB_MMA + s], 1);
            mbar_init(&bar[OB_MRDY + s], NEW);
            mbar_init(&bar[OB_FREE + s], NEW);
        }
        fence_mbar_init();
        ms->abort_ = 0;
    }
    if (warp == 0) tmem_alloc(&ms->tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t idesc_cb = idesc_bf16(128, 128, 0, 0), idesc_y = idesc_bf16(128, 64, 0, 1);
    const uint32_t sB = smem_u32(sm + O_B), sC = smem_u32(sm + O_C);
    const uint32_t in_bytes = (has_z ? 3u : 2u) * X_BYTES;
    const int total = p.hdr[HDR_STATUS] != 0 ? 0 : p.n_items;
    // Phase parity of the next completion of each barrier a side waits on (bit b); the issuer's
    // slots with an input copy issued and unwaited (inout) and the parity of its last phase.
    uint32_t ph = 0u, inout = 0u, iniss = 0u, inlast = 0u;
    bool bcout = false, stores = false;
    auto waitb = [&](int b) -> bool {
        const bool ok = mbar_wait_abort(&bar[b], (ph >> b) & 1u, abort_);
        ph ^= 1u << b;
        return ok;
    };
    for (;;) {
        if (issuer) ms->item = atomicAdd(&p.hdr[HDR_TICKET2], 1);
        tc_fence_before();
        __syncthreads();   // the previous item is over on both sides (TMEM reads of CB included)
        tc_fence_after();
        const int it = ms->item;
        if (it >= total || *abort_) break;
        int k, g, h0;
        item_of(it, sh, HS, k, g, h0);
        if (k >= p.hdr[HDR_NCHUNKS]) continue;
        const ChunkInfo ci = p.chunks[k];
        const bool tile_out = ci.lo == 0 && ci.len == QT;   // every row is this sequence's
        // issuer: x and S_in of head i into slot i & 1 (the phase also expects z's bytes), then z
        auto load_xs = [&](int i) {
            const int s = i & 1, h = h0 + i;
            uint8_t *sb = sm + O_SLOT + s * SLOT_BYTES;
            mbar_expect_tx(&bar[OB_IN + s], in_bytes);
            tma_load_4d(sb + S_X, &tmX, &bar[OB_IN + s], 0, h, ci.t0, ci.b);
            bulk_load(sb + S_S, tile_row(p.states, k, sh.H, h, 0), X_BYTES, &bar[OB_IN + s]);
            inout |= 1u << s;
            inlast = (inlast & ~(1u << s)) | (iniss & (1u << s));
            iniss ^= 1u << s;
        };
        auto load_z = [&](int i) {
            if (has_z)
                tma_load_4d(sm + O_SLOT + (i & 1) * SLOT_BYTES + S_Z, &tmZ, &bar[OB_IN + (i & 1)], 0, h0 + i, ci.t0,
                            ci.b);
        };
        if (issuer) {
            if (stores) {   // the previous item's y tiles have left the z buffers
                bulk_wait_read0();
                stores = false;
            }
            mbar_expect_tx(&bar[OB_BC], 2 * BC_BYTES);
            tma_load_4d(sm + O_B, &tmB, &bar[OB_BC], 0, g, ci.t0, ci.b);
            tma_load_4d(sm + O_B + BC_BYTES / 2, &tmB, &bar[OB_BC], 64, g, ci.t0, ci.b);
            tma_load_4d(sm + O_C, &tmC, &bar[OB_BC], 0, g, ci.t0, ci.b);
            tma_load_4d(sm + O_C + BC_BYTES / 2, &tmC, &bar[OB_BC], 64, g, ci.t0, ci.b);
            bcout = true;
            for (int i = 0; i < 2 && i < HS; ++i) {
                load_xs(i);
                load_z(i);
            }
        }
        if (warp < HS) {   // per-head tables: dt, cs log2 e, block factors dt exp(cs[a] - cs[s]), exp(cs)
            float dt4[4], cs4[4];
            head_scan(p, ci, h0 + warp, dt4, cs4);
            const int lane = tid & 31;
            float *T = tab + warp * TAB_FLOATS;
            float c2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) c2[i] = cs4[i] * LOG2E;
            const float c31 = __shfl_sync(0xffffffffu, c2[3], lane | 7);   // cs at the 32-block's last position
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pos = 4 * lane + i;
                T[pos] = dt4[i];
                T[QT + pos] = c2[i];
                T[2 * QT + pos] = dt4[i] * ex2(c31 - c2[i]);
                T[3 * QT + pos] = ex2(c2[i]);
            }
        }
        __syncthreads();   // tables written
        if (issuer) {   // CB = C B^T (K = state dim), once for the item's heads
            if (waitb(OB_BC)) {
                bcout = false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < NT / 16; ++kk)
                    umma_bf16(tmem + TM_CB, kmaj(sC, kk, BC_BYTES / 2), kmaj(sB, kk, BC_BYTES / 2), idesc_cb, kk > 0);
                umma_commit(&bar[OB_CB]);
                waitb(OB_CB);
                for (int i = 0; i < HS && !*abort_; ++i) {
                    const int st = i & 1, so = st ^ 1;
                    if (!waitb(OB_MRDY + st)) break;   // M of head i in its slot
                    if (!waitb(OB_IN + st)) break;     // x, z, S_in of head i
                    inout &= ~(1u << st);
                    tc_fence_after();
                    uint8_t *sb = sm + O_SLOT + st * SLOT_BYTES;
                    const uint32_t tsl = tmem + TM_SLOT0 + TM_SLOT * (uint32_t)st;
                    const uint32_t ss = smem_u32(sb + S_S), sx = smem_u32(sb + S_X);
#pragma unroll
                    for (int kk = 0; kk < NT / 16; ++kk)   // Y_off = C S_in^T (K = state dim)
                        umma_bf16(tsl + 64, kmaj(sC, kk, BC_BYTES / 2), mnmaj(ss, kk), idesc_y, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < QT / 16; ++kk)   // Y_diag + D x = M x (K = source tokens), M from TMEM
                        umma_bf16_ta(tsl + 128, tsl + 8 * kk, mnmaj(sx, kk), idesc_y, kk > 0);
                    umma_commit(&bar[OB_MMA + st]);
                    if (i >= 1) {   // head i-1's outputs are formed: its y leaves, its slot takes head i+1
                        if (!waitb(OB_FREE + so)) break;
                        if (tile_out) {
                            tma_store_4d(&tmY, sm + O_SLOT + so * SLOT_BYTES + S_Z, 0, h0 + i - 1, ci.t0, ci.b);
                            bulk_commit();
                            stores = true;
                        }
                        if (i + 1 < HS) {
                            load_xs(i + 1);
                            if (tile_out) bulk_wait_read0();   // before z of head i+1 lands over that y
                            load_z(i + 1);
                        }
                    }
                }
                if (!*abort_) {   // the last head's outputs
                    const int sl = (HS - 1) & 1;
                    if (waitb(OB_FREE + sl) && tile_out) {
                        tma_store_4d(&tmY, sm + O_SLOT + sl * SLOT_BYTES + S_Z, 0, h0 + HS - 1, ci.t0, ci.b);
                        bulk_commit();
                        stores = true;
                    }
                }
            }
        }
        if (ew) {
            bool live_ok = waitb(OB_CB);
            tc_fence_after();
            for (int i = 0; i <= HS; ++i) {
                const int st = i & 1;
                if (i < HS) {
                    if (live_ok && !*abort_) {
                        // M of head i (bf16, D on the diagonal) into its slot: the two threads of row l
                        // take blocks {0, 3} or {1, 2} of its four 32-column blocks (the causal work
                        // split evenly); CB is only read here
                        const float *T = tab + i * TAB_FLOATS;
                        const float Dh = p.D ? p.D[h0 + i] : 0.f;
                        const int l = row, quad = warp & 3;
                        const float cl = T[QT + l];
                        const uint32_t tm_m = tmem + lane_base + TM_SLOT0 + TM_SLOT * (uint32_t)st;
#pragma unroll
                        for (int bi = 0; bi < 2; ++bi) {
                            const int sbk = hf == 0 ? (bi == 0 ? 0 : 3) : (bi == 0 ? 1 : 2);
                            uint32_t pk[16];
                            if (sbk < quad) {   // below the diagonal: exp(cs[l]-cs[a]) exp(cs[a]-cs[s]) dt[s], both <= 1
                                float cb[32];
                                tmem_ld32(tmem + lane_base + TM_CB + sbk * 32, cb);
                                const float rl = ex2(cl - T[QT + sbk * 32 + 31]);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; e += 2)
                                    pk[e >> 1] = pack_bf16(cb[e] * rl * T[2 * QT + sbk * 32 + e],
                                                           cb[e + 1] * rl * T[2 * QT + sbk * 32 + e + 1]);
                            } else if (sbk == quad) {   // diagonal block: causal mask, D on the diagonal
                                float cb[32];
                                tmem_ld32(tmem + lane_base + TM_CB + sbk * 32, cb);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; e += 2) {
                                    const int s0 = sbk * 32 + e;
                                    float m0 = (s0 <= l) ? cb[e] * ex2(cl - T[QT + s0]) * T[s0] : 0.f;
                                    float m1 = (s0 + 1 <= l) ? cb[e + 1] * ex2(cl - T[QT + s0 + 1]) * T[s0 + 1] : 0.f;
                                    if (s0 == l) m0 += Dh;
                                    if (s0 + 1 == l) m1 += Dh;
                                    pk[e >> 1] = pack_bf16(m0, m1);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 16; ++e) pk[e] = 0u;
                            }
                            tmem_st16(tm_m + 16 * sbk, pk);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    mbar_arrive(&bar[OB_MRDY + st]);
                }
                if (i >= 1) {   // head i-1: its MMAs are done -> y = (Y_diag + exp(cs) Y_off) silu(z)
                    const int so = st ^ 1, hi = i - 1;
                    bool ok = waitb(OB_MMA + so);
                    if (has_z) ok = waitb(OB_IN + so) && ok;   // z of head i-1 (landed before its MMAs)
                    if (ok && live_ok && !*abort_) {
                        tc_fence_after();
                        const float *T = tab + hi * TAB_FLOATS;
                        uint8_t *zb = sm + O_SLOT + so * SLOT_BYTES + S_Z;
                        const uint32_t tsl = tmem + lane_base + TM_SLOT0 + TM_SLOT * (uint32_t)so;
                        const int l = row;
                        const float el = T[3 * QT + l];
                        const bool live = l >= ci.lo && l < ci.len;
                        __nv_bfloat16 *yrow =
                            p.y + (int64_t)ci.b * p.syb + (int64_t)(ci.t0 + l) * p.syl + (int64_t)(h0 + hi) * p.syh;
#pragma unroll
                        for (int qq = 0; qq < 4; qq += 2) {
                            const int q0 = 4 * hf + qq;
                            float yd[16], yo[16];
                            tmem_ld16(tsl + 128 + 8 * q0, yd);
                            tmem_ld16(tsl + 64 + 8 * q0, yo);
                            tmem_wait_ld();
                            if (live) {
#pragma unroll
                                for (int qi = 0; qi < 2; ++qi) {
                                    const int q = q0 + qi;
                                    uint4 *zp = reinterpret_cast<uint4 *>(zb + l * 128 + ((q ^ (l & 7)) << 4));
                                    uint4 zq = make_uint4(0u, 0u, 0u, 0u);
                                    if (has_z) zq = *zp;
                                    const __nv_bfloat162 *ze = reinterpret_cast<const __nv_bfloat162 *>(&zq);
                                    uint32_t o[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int jx = qi * 8 + 2 * e;
                                        float v0 = yd[jx] + el * yo[jx], v1 = yd[jx + 1] + el * yo[jx + 1];
                                        if (has_z) {
                                            const float2 zf = __bfloat1622float2(ze[e]);
                                            v0 *= silu_tanh(zf.x);
                                            v1 *= silu_tanh(zf.y);
                                        }
                                        o[e] = pack_bf16(v0, v1);
                                    }
                                    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
                                    if (tile_out)
                                        *zp = ov;   // y over the z piece just read
                                    else
                                        *reinterpret_cast<uint4 *>(yrow + q * 8) = ov;
                                }
                            }
                        }
                        if (tile_out) fence_proxy_async_smem();
                    }
                    tc_fence_before();
                    mbar_arrive(&bar[OB_FREE + so]);
                }
            }
        }
    }
    if (issuer) {   // every copy, MMA and store issued has completed before the CTA's memory goes
        if (bcout) mbar_wait(&bar[OB_BC], (ph >> OB_BC) & 1u);
        for (int s = 0; s < 2; ++s)
            if (inout & (1u << s)) mbar_wait(&bar[OB_IN + s], (inlast >> s) & 1u);
        umma_commit(&bar[OB_CB]);                    // all of this thread's MMAs
        mbar_wait(&bar[OB_CB], (ph >> OB_CB) & 1u);
        bulk_wait0();
        if (*abort_) set_status(p.hdr, SSD_ERR_DEVICE_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_s() {
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

// 4-D bf16 map over [B][L][H or G][64 k] with box {64, 1, 128, 1}, 128-byte swizzle.
bool map_s(CUtensorMap *m, const void *ptr, int64_t inner, int64_t d1, int64_t L, int64_t B, int64_t s1, int64_t sL,
           int64_t sB) {
    auto fn = encode_fn_s();
    if (fn == nullptr) return false;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)d1, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)(s1 * 2), (cuuint64_t)(sL * 2), (cuuint64_t)(sB * 2)};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)QT, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Heads per work item of the split kernels: the largest divisor of H/G up to 8.
int split_heads_per_item(int hpg) {
    for (int d = HSMAX; d > 1; --d)
        if (hpg % d == 0) return d;
    return 1;
}

// The carried-state tiles (S_in entering every chunk tile) and the final states: the first
// two launches.  `states` holds kmax * H tiles of 16 KB; `lam` kmax * H floats.
cudaError_t launch_split_states(const Shape &sh, int32_t *hdr, const ChunkInfo *chunks, const SeqInfo *seqs,
                                const void *x, const int64_t *sx, const void *Bp, const int64_t *sb,
                                const float *dt_raw, int64_t sdb, int64_t sdl, const float *A, const float *bias,
                                const float *init, float *final_, __nv_bfloat16 *states, float *lam, int sms,
                                cudaStream_t st) {
    CUtensorMap mx, mb;
    if (!map_s(&mx, x, PT, sh.H, sh.L, sh.B, sx[2], sx[1], sx[0])) return cudaErrorInvalidValue;
    if (!map_s(&mb, Bp, sh.Nio, sh.G, sh.L, sh.B, sb[2], sb[1], sb[0])) return cudaErrorInvalidValue;
    SplitParams p{};
    p.sh = sh; p.hdr = hdr; p.chunks = chunks; p.seqs = seqs;
    p.hs = split_heads_per_item(sh.hpg);
    p.n_items = sh.kmax * sh.G * (sh.hpg / p.hs);
    p.dt_raw = dt_raw; p.sdb = sdb; p.sdl = sdl; p.A = A; p.bias = bias;
    p.init = init; p.final_ = final_; p.states = states; p.lam = lam;
    if (p.n_items > 0) {
        static int attr[64] = {0};
        cudaError_t e = ensure_smem_attr(k_split_states, (int)ST_SMEM, attr);
        if (e != cudaSuccess) return e;
        const int grid = std::min(p.n_items, ST_CTAS_PER_SM * sms);
        k_split_states<<<grid, ST_THREADS, ST_SMEM, st>>>(mx, mb, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (sh.S > 0) {
        k_split_passing<<<dim3(sh.S * sh.H, (PT * NT / 8) / 256), 256, 0, st>>>(p);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

// The outputs y from the carried-state tiles (third launch).
cudaError_t launch_split_out(const Shape &sh, int32_t *hdr, const ChunkInfo *chunks, const void *x, const int64_t *sx,
                             const void *Bp, const int64_t *sb, const void *Cp, const int64_t *sc, const float *dt_raw,
                             int64_t sdb, int64_t sdl, const float *A, const float *D, const float *bias,
                             const void *z, const int64_t *sz, void *y, const int64_t *sy,
                             __nv_bfloat16 *states, int sms, cudaStream_t st) {
    CUtensorMap mx, mb, mc, mz, my;
    if (!map_s(&mx, x, PT, sh.H, sh.L, sh.B, sx[2], sx[1], sx[0])) return cudaErrorInvalidValue;
    if (!map_s(&mb, Bp, sh.Nio, sh.G, sh.L, sh.B, sb[2], sb[1], sb[0])) return cudaErrorInvalidValue;
    if (!map_s(&mc, Cp, sh.Nio, sh.G, sh.L, sh.B, sc[2], sc[1], sc[0])) return cudaErrorInvalidValue;
    if (!map_s(&my, y, PT, sh.H, sh.L, sh.B, sy[2], sy[1], sy[0])) return cudaErrorInvalidValue;
    if (z != nullptr) {
        if (!map_s(&mz, z, PT, sh.H, sh.L, sh.B, sz[2], sz[1], sz[0])) return cudaErrorInvalidValue;
    } else {
        mz = mx;   // not read
    }
    SplitParams p{};
    p.sh = sh; p.hdr = hdr; p.chunks = chunks;
    p.hs = split_heads_per_item(sh.hpg);
    p.n_items = sh.kmax * sh.G * (sh.hpg / p.hs);
    p.dt_raw = dt_raw; p.sdb = sdb; p.sdl = sdl; p.A = A; p.D = D; p.bias = bias;
    p.z_present = z != nullptr;
    p.y = (__nv_bfloat16 *)y; p.syb = sy[0]; p.syl = sy[1]; p.syh = sy[2];
    p.states = states;
    if (p.n_items == 0) return cudaSuccess;
    static int attr[64] = {0};
    cudaError_t e = ensure_smem_attr(k_split_out, (int)OUT_SMEM, attr);
    if (e != cudaSuccess) return e;
    k_split_out<<<std::min(p.n_items, sms), OUT_THREADS, OUT_SMEM, st>>>(mx, mb, mc, mz, my, p);
    return cudaGetLastError();
}

}  // namespace ssd
