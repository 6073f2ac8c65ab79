// api.cu -- the C ABI of libssd.so (declared in include/ssd.h): argument
// validation, workspace planning and launch sequencing on the caller's stream.
#include <string.h>

#include "common.cuh"

namespace ssd {
// meta.cu
cudaError_t launch_build_meta(const int32_t *cu, int B, int L, int S, int Q, int R, int num, int den, int KB, int kmax,
                              int umax, int32_t *hdr,
                              SeqInfo *seqs, ChunkInfo *chunks, UnitInfo *units, int32_t *last_unit,
                              uint32_t *zero_words, int64_t n_zero, cudaStream_t st);
cudaError_t launch_wait_probe(int32_t *hdr, int wait_ms, cudaStream_t st);
cudaError_t launch_varlen_metadata(const int32_t *cu, int S, int L, int Q, int32_t *status, int32_t *chunk_begin,
                                   int32_t *segments, int32_t *seq_idx, cudaStream_t st);
cudaError_t launch_states_cvt(const void *src, bool src_bf16, int src_n, void *dst, bool dst_bf16, int dst_n,
                              int64_t rows, cudaStream_t st);
cudaError_t launch_empty_seq_final(int S, int H, int PN, const SeqInfo *seqs, const int32_t *hdr, const float *init,
                                   float *final_, cudaStream_t st);
// simt_fwd.cu
cudaError_t launch_chunk_cumsum(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const float *dt_raw,
                                int64_t sdb, int64_t sdl, const float *A, const float *bias, float *dt_out,
                                float *cs_out, cudaStream_t st);
template <typename T>
cudaError_t launch_chunk_state(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 x, View3 Bm,
                               const float *dtw, const float *csw, float *states, cudaStream_t st);
cudaError_t launch_state_passing(const Shape &sh, const int32_t *hdr, const SeqInfo *seqs, const float *lamw,
                                 int lam_stride, float *states, const float *init, float *final_, int reverse,
                                 cudaStream_t st);
cudaError_t launch_state_passing(const Shape &sh, const int32_t *hdr, const SeqInfo *seqs, const float *lamw,
                                 int lam_stride, __nv_bfloat16 *states, const float *init, float *final_, int reverse,
                                 cudaStream_t st);
template <typename T>
cudaError_t launch_chunk_scan(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 x, View3 Bm,
                              View3 Cm, View3 z, const float *D, const float *dtw, const float *csw,
                              const float *states, MView3 y, cudaStream_t st);
// simt_bwd.cu
template <typename T>
cudaError_t launch_bwd_dstates(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 dy, View3 z,
                               View3 Cm, const float *csw, float *dstates, cudaStream_t st);
template <typename T>
cudaError_t launch_bwd_chunk(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, View3 x, View3 Bm,
                             View3 Cm, View3 z, View3 dy, const float *dt_raw, int64_t sdb, int64_t sdl,
                             const float *A, const float *D, const float *bias, const float *dtw, const float *csw,
                             const float *states, const float *dstates, MView3 dx, MView3 dz, float *ddt,
                             int64_t sddb, int64_t sddl, float *dBh, float *dCh, float *partials, cudaStream_t st);
template <typename T>
cudaError_t launch_reduce_group(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const float *srcB,
                                MView3 dstB, const float *srcC, MView3 dstC, cudaStream_t st);
cudaError_t launch_reduce_heads(const Shape &sh, const int32_t *hdr, const float *partials, float *dA, float *dD,
                                float *dbias, cudaStream_t st);
size_t bwd_chunk_smem(const Shape &sh);
size_t chunk_scan_smem(const Shape &sh);
// fused_fwd.cu
int fused_rmax();
int fused_rmax_states();
int fused_block_units();
// bwd_tc.cu
cudaError_t launch_bwd_dstates_tc(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a,
                                  cudaStream_t st);
cudaError_t launch_bwd_chunk_tc(const Shape &sh, const int32_t *hdr, const ChunkInfo *chunks, const BwdTcArgs &a,
                                cudaStream_t st);
// split_fwd.cu
cudaError_t launch_split_states(const Shape &sh, int32_t *hdr, const ChunkInfo *chunks, const SeqInfo *seqs,
                                const void *x, const int64_t *sx, const void *Bp, const int64_t *sb,
                                const float *dt_raw, int64_t sdb, int64_t sdl, const float *A, const float *bias,
                                const float *init, float *final_, __nv_bfloat16 *states, float *lam, int sms,
                                cudaStream_t st);
cudaError_t launch_split_out(const Shape &sh, int32_t *hdr, const ChunkInfo *chunks, const void *x, const int64_t *sx,
                             const void *Bp, const int64_t *sb, const void *Cp, const int64_t *sc, const float *dt_raw,
                             int64_t sdb, int64_t sdl, const float *A, const float *D, const float *bias,
                             const void *z, const int64_t *sz, void *y, const int64_t *sy,
                             __nv_bfloat16 *states, int sms, cudaStream_t st);
cudaError_t launch_fused_fwd(const Shape &sh, int32_t *hdr, const UnitInfo *units, const void *x, const int64_t *sx,
                             const void *Bp, const int64_t *sb, const void *Cp, const int64_t *sc, const float *dt_raw,
                             int64_t sdb, int64_t sdl, const float *A, const float *D, const float *bias,
                             const void *z, const int64_t *sz, void *y, const int64_t *sy, const float *init,
                             float *final_, float *agg, float *incl, float *lam, uint32_t *flags, int grid,
                             __nv_bfloat16 *states_out, bool states_only, const SeqInfo *seqs, cudaStream_t st);
}  // namespace ssd

using namespace ssd;

namespace {

constexpr int kSimtQmin = 32, kSimtQmax = 256, kSimtQbwd = 64;   // SIMT chunk lengths (powers of two)
constexpr int kTcQ = 128;
constexpr size_t kAlign = 256;

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool pow2_in(int64_t v, int64_t lo, int64_t hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

struct Plan {
    Shape sh;
    bool bf16 = false;
    bool varlen = false;
    int algo = SSD_ALGO_STAGED;
    int hs = 1;   // heads per work item of the tensor-core gradient kernel
    int k_pairs = 0, nsub_tail = 1, n_items = 0;   // its work items (see BwdTcArgs)
    size_t off_tpart = 0;
    size_t off_hdr = 0, off_seqs = 0, off_chunks = 0, off_lastunit = 0, off_units = 0;
    size_t off_dt = 0, off_cs = 0, off_states = 0, off_dstates = 0, off_dBh = 0, off_dCh = 0, off_part = 0;
    size_t off_agg = 0, off_incl = 0, off_lam = 0, off_flags = 0;
    size_t chunk_state_bytes = 0;   // tensor-core path: one bf16 [P][N] tile per (chunk, head)
    // fp32 [.., N] copies of state tensors stored otherwise (bf16, or dstate 64 on the tensor-core
    // path): initial, final, dfinal, dinitial
    size_t off_st32[4] = {0, 0, 0, 0};
    bool st_bf16[4] = {false, false, false, false};
    size_t total = 0;
};

// Heads per work item of the tensor-core gradient kernel: a divisor of H/G up to 32.  An
// item loads B and C of its chunk once for all its heads and writes final dB/dC when it
// covers the whole group; otherwise a reduction reads back fp32 shares of dB and dC for
// every head subset.  Groups of at most 8 heads are whole items; for larger groups the
// choice minimises the estimated time: whole rounds of items over the SMs, about 8 us per
// head, plus that reduction's traffic at about 5 TB/s.
int bwd_heads_per_cta(int64_t kmax, int64_t H, int hpg) {
    // groups of at most 8 heads: whole-group items (no dB/dC reduction; the persistent kernel
    // splits the pairs of its last partial wave itself)
    if (hpg <= 8) return hpg;
    const int64_t sms = num_sms();
    int best = 1;
    double best_us = 1e300;
    for (int d = 1; d <= 32 && d <= hpg; ++d) {
        if (hpg % d != 0) continue;
        const int64_t ctas = kmax * (H / d);
        const int64_t waves = (ctas + sms - 1) / sms;
        double us = 8.0 * (double)(waves * d);
        if (d < hpg) us += (double)ctas * 128.0 * 128.0 * 4.0 * 3.0 / 5.0e6;   // 2 reads + 1 write per subset tile
        if (us <= best_us) {   // ties go to more heads per CTA
            best_us = us;
            best = d;
        }
    }
    return best;
}

// Heads per CTA of the tensor-core dstates kernel (three CTAs per SM): the largest
// divisor of H/G up to 8 that still gives four full waves of CTAs (short CTAs keep the last
// wave's idle time small), else 1.
int dstates_heads_per_cta(int64_t kmax, int64_t H, int hpg) {
    const int64_t slots = 3LL * num_sms();
    for (int d = 8; d > 1; --d)
        if (hpg % d == 0 && kmax * (H / d) >= 4 * slots) return d;
    return 1;
}

struct Layout {
    size_t cur = 0;
    size_t take(size_t bytes) {
        size_t o = cur;
        cur = align_up(cur + bytes);
        return o;
    }
};

// Checks one tensor argument.  rank = number of meaningful strides; the
// innermost stride must be 1 and all strides non-negative.
ssd_status check_tensor(const ssd_tensor &t, int rank, int dtype_req, bool required) {
    if (t.ptr == nullptr) return required ? SSD_ERR_INVALID_ARGUMENT : SSD_OK;
    if (dtype_req >= 0 && t.dtype != dtype_req) return SSD_ERR_INVALID_ARGUMENT;
    if (t.dtype != SSD_F32 && t.dtype != SSD_BF16) return SSD_ERR_INVALID_ARGUMENT;
    if (rank > 0 && t.stride[rank - 1] != 1) return SSD_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < rank; ++i)
        if (t.stride[i] < 0) return SSD_ERR_INVALID_ARGUMENT;
    return SSD_OK;
}

// Contiguous [S, H, P, N] state tensors, fp32 or bf16.
ssd_status check_state(const ssd_tensor &t, int64_t H, int64_t P, int64_t N) {
    if (t.ptr == nullptr) return SSD_OK;
    if (t.dtype != SSD_F32 && t.dtype != SSD_BF16) return SSD_ERR_INVALID_ARGUMENT;
    if (t.stride[3] != 1 || t.stride[2] != N || t.stride[1] != P * N || t.stride[0] != H * P * N)
        return SSD_ERR_INVALID_ARGUMENT;
    return SSD_OK;
}

ssd_status check_vec(const ssd_tensor &t, bool required) {
    if (t.ptr == nullptr) return required ? SSD_ERR_INVALID_ARGUMENT : SSD_OK;
    if (t.dtype != SSD_F32 || t.stride[0] != 1) return SSD_ERR_INVALID_ARGUMENT;
    return SSD_OK;
}

#define SSD_TRY(expr)                      \
    do {                                   \
        ssd_status _s = (expr);            \
        if (_s != SSD_OK) return _s;       \
    } while (0)

ssd_status plan_common(const ssd_problem *p, const ssd_fwd_args *a, bool bwd, Plan *out,
                       const ssd_bwd_args *b = nullptr) {
    if (p == nullptr || a == nullptr || out == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    const int64_t B = p->batch, L = p->seqlen, H = p->nheads, P = p->headdim, G = p->ngroups, N = p->dstate;
    if (B < 1 || L < 0 || H < 1 || G < 1 || P < 1 || N < 1 || p->chunk_size < 1) return SSD_ERR_INVALID_ARGUMENT;
    if (H % G != 0) return SSD_ERR_INVALID_ARGUMENT;
    if (L > (int64_t)1 << 30 || B > (int64_t)1 << 20 || H > 65535) return SSD_ERR_UNSUPPORTED;
    if (!pow2_in(p->chunk_size, 16, 256)) return SSD_ERR_UNSUPPORTED;
    if (!pow2_in(P, 16, 128) || !pow2_in(N, 16, 128)) return SSD_ERR_UNSUPPORTED;
    if (p->algo < SSD_ALGO_AUTO || p->algo > SSD_ALGO_SPLIT) return SSD_ERR_INVALID_ARGUMENT;
    if (p->seg_chunks < 0 || p->seg_chunks > 8) return SSD_ERR_INVALID_ARGUMENT;
    if (p->bwd_heads < 0 || p->bwd_heads > 32 || p->reserved0 != 0) return SSD_ERR_INVALID_ARGUMENT;
    const bool varlen = a->cu_seqlens != nullptr;
    int64_t S = B;
    if (varlen) {
        if (B != 1 || p->nseqs < 1) return SSD_ERR_INVALID_ARGUMENT;
        S = p->nseqs;
        if (S > (int64_t)1 << 24) return SSD_ERR_UNSUPPORTED;
    } else if (p->nseqs != 0 && p->nseqs != B) {
        return SSD_ERR_INVALID_ARGUMENT;
    }
    // Token tensors of an empty sequence axis have no storage (NULL is allowed).
    const bool tok = L > 0;
    if (a->x.dtype != SSD_F32 && a->x.dtype != SSD_BF16) return SSD_ERR_INVALID_ARGUMENT;
    SSD_TRY(check_tensor(a->x, 4, -1, tok));
    const int dt_ = a->x.dtype;
    SSD_TRY(check_tensor(a->B, 4, dt_, tok));
    SSD_TRY(check_tensor(a->C, 4, dt_, tok));
    SSD_TRY(check_tensor(a->z, 4, dt_, false));
    SSD_TRY(check_tensor(a->dt, 3, SSD_F32, tok));
    SSD_TRY(check_vec(a->A, true));
    SSD_TRY(check_vec(a->D, false));
    SSD_TRY(check_vec(a->dt_bias, false));
    SSD_TRY(check_state(a->initial_states, H, P, N));
    if (!bwd) {
        SSD_TRY(check_tensor(a->y, 4, dt_, tok));
        SSD_TRY(check_state(a->final_states, H, P, N));
    }
    Plan pl;
    pl.bf16 = dt_ == SSD_BF16;
    pl.varlen = varlen;
    // Path choice.  The tensor-core forward covers bf16 inputs with headdim 64 and
    // dstate 128 whose x/B/C/z/y obey the 16-byte rule of TMA and vector access;
    // everything else (fp32 inputs in particular) runs the SIMT pipeline.  The
    // backward follows the same choice, with dy/dx/dz/dB/dC under the same rule.
    bool tc_ok = pl.bf16 && P == 64 && N <= 128;   // N < 128: the zero-extended tiles (below)
    bool aligned = true;
    {
        const ssd_tensor *ts[10] = {&a->x, &a->B, &a->C, &a->z, bwd ? nullptr : &a->y, b ? &b->dy : nullptr,
                                    b ? &b->dx : nullptr, b ? &b->dz : nullptr, b ? &b->dB : nullptr,
                                    b ? &b->dC : nullptr};
        for (const ssd_tensor *t : ts) {
            if (t == nullptr) continue;
            if (t->ptr == nullptr) continue;
            if (((uintptr_t)t->ptr) % 16 != 0) aligned = false;
            for (int i = 0; i < 3; ++i)
                if (t->stride[i] % 8 != 0) aligned = false;
        }
    }
    // The chunk length is the caller's, never replaced: the tensor-core path computes
    // 128-token chunks (one M = 128 tcgen05 tile per chunk); the SIMT path computes chunks of
    // 32, 64, 128 or 256 tokens in the forward and of 32 or 64 in the backward (whose per-chunk
    // tiles, Q x Q and Q x (P, N), live in shared memory).
    const bool simt_q = p->chunk_size >= kSimtQmin && p->chunk_size <= (bwd ? kSimtQbwd : kSimtQmax);
    bool fused = false;   // the tensor-core path (single-pass or split forward)
    if (p->algo == SSD_ALGO_FUSED || p->algo == SSD_ALGO_SPLIT) {
        if (!tc_ok || p->chunk_size != kTcQ) return SSD_ERR_UNSUPPORTED;
        if (!aligned) return SSD_ERR_MISALIGNED;
        fused = true;
    } else if (p->algo == SSD_ALGO_STAGED) {
        if (!simt_q) return SSD_ERR_UNSUPPORTED;
    } else if (p->chunk_size == kTcQ && tc_ok) {
        if (!aligned) return SSD_ERR_MISALIGNED;
        fused = true;
    } else if (!simt_q) {
        return SSD_ERR_UNSUPPORTED;
    }
    // AUTO takes the single-pass forward on the tensor-core path (measured faster than the
    // split forward at every benchmarked shape); SSD_ALGO_SPLIT selects the three-launch one.
    const bool split = fused && p->algo == SSD_ALGO_SPLIT;
    pl.algo = split ? SSD_ALGO_SPLIT : fused ? SSD_ALGO_FUSED : SSD_ALGO_STAGED;
    if (a->chunk_states != nullptr) {   // kept chunk states: the tensor-core path's tile format only
        if (!fused) return SSD_ERR_UNSUPPORTED;
        if (((uintptr_t)a->chunk_states) % 16 != 0) return SSD_ERR_MISALIGNED;
    }
    const int Q = fused ? kTcQ : (int)p->chunk_size;
    // dstate the kernels compute: the tensor-core tiles are N = 128; a smaller dstate runs as the
    // zero-extended tile (TMA fills the B/C columns past it with zeros; states are padded copies)
    const int64_t Nk = fused ? 128 : N;
    if (fused && bwd && b == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    int64_t kmax = varlen ? (L + Q - 1) / Q + S : B * ((L + Q - 1) / Q);
    if (kmax > (int64_t)1 << 30) return SSD_ERR_UNSUPPORTED;
    int R = 1, num = 1, den = 1;
    int64_t umax = 0;
    if (fused && !split) {
        R = p->seg_chunks;
        const int rmax = bwd ? fused_rmax_states() : fused_rmax();
        num = 1;   // units per chunk: 1/R, or the larger ratio num/den chosen below
        den = R;
        if (R == 0) {
            // Work units from a model of the persistent kernel: rounds of resident CTAs (two
            // per SM) times one unit's time, its chunks plus a fixed part (unit prologue and
            // carry-in fold).  Per-chunk cost: full forward about 9.3 us, states-only (the
            // backward's recompute) about 2.3 us; fixed part about 8 us.
            const int64_t slots = 2LL * num_sms();
            const double c_chunk = bwd ? 2.3 : 9.3, c_unit = 8.0;
            double best = 1e300;
            const int64_t n = (L + Q - 1) / Q;   // chunks per sequence of a fixed-length batch
            if (!varlen && n > 0) {
                // The number of units per sequence, U, is chosen rather than their length, so
                // that the units of the last round fill it: units of n/U chunks on average
                // (floor or ceil), B U H of them.  Units stay between rmax - 1 and rmax chunks
                // long: shorter ones measured slower (more carry-in folds and block ends in
                // the serial chain of a sequence).
                const int64_t U0 = (n + rmax - 1) / rmax;
                const int64_t U1 = rmax > 1 ? n / (rmax - 1) : n;   // n / U >= rmax - 1
                int64_t bestU = U0;
                for (int64_t U = U0; U <= U1 && U <= n; ++U) {
                    const int64_t rounds = (B * U * H + slots - 1) / slots;
                    const double cost = (double)rounds * ((double)n / (double)U * c_chunk + c_unit);
                    if (cost < best) {
                        best = cost;
                        bestU = U;
                    }
                }
                R = (int)((n + bestU - 1) / bestU);
                num = (int)bestU;
                den = (int)n;
            } else {
                for (int r = 1; r <= rmax; ++r) {
                    const int64_t units = varlen ? (kmax + r - 1) / r + S : B * ((n + r - 1) / r);
                    const int64_t rounds = (units * H + slots - 1) / slots;
                    const double cost = (double)rounds * (r * c_chunk + c_unit);
                    if (cost < best) {
                        best = cost;
                        R = r;
                    }
                }
                num = 1;
                den = R;
            }
        }
        if (R > rmax) return SSD_ERR_UNSUPPORTED;
        // units: sum over sequences of max(ceil(n/R), ceil(n num/den)) <= kmax max(1/R, num/den) + S
        const int64_t per = (int64_t)num * R > den ? (kmax * num + den - 1) / den : (kmax + R - 1) / R;
        umax = per + S;
    }
    Shape sh;
    sh.B = (int)B; sh.L = (int)L; sh.H = (int)H; sh.P = (int)P; sh.G = (int)G; sh.N = (int)Nk; sh.Nio = (int)N; sh.S = (int)S;
    sh.Q = Q; sh.hpg = (int)(H / G); sh.kmax = (int)kmax; sh.umax = (int)umax; sh.R = R; sh.useg_num = num; sh.useg_den = den;
    pl.sh = sh;
    Layout lay;
    pl.off_hdr = lay.take(HDR_WORDS * sizeof(int32_t));
    pl.off_seqs = lay.take(sizeof(SeqInfo) * (size_t)S);
    pl.off_chunks = lay.take(sizeof(ChunkInfo) * (size_t)kmax);
    pl.off_lastunit = lay.take(sizeof(int32_t) * (size_t)S);
    const size_t kh = (size_t)kmax * (size_t)H;
    if (fused) {
        if (!split) {   // the single-pass forward's work units and their exchange buffers
            const size_t uh = (size_t)umax * (size_t)H;
            pl.off_units = lay.take(sizeof(UnitInfo) * (size_t)umax);
            pl.off_agg = lay.take(sizeof(float) * uh * (size_t)(P * Nk));
            pl.off_incl = lay.take(sizeof(float) * uh * (size_t)(P * Nk));
            pl.off_lam = lay.take(sizeof(float) * uh);
            pl.off_flags = lay.take(sizeof(uint32_t) * uh);
        } else if (!bwd) {   // the split forward: carried-state tiles (unless kept) and tile log-decays
            if (a->chunk_states == nullptr) pl.off_states = lay.take(sizeof(__nv_bfloat16) * kh * (size_t)(P * Nk));
            pl.off_cs = lay.take(sizeof(float) * kh);
        }
        if (bwd) {
            pl.hs = p->bwd_heads > 0 ? p->bwd_heads : bwd_heads_per_cta(kmax, H, sh.hpg);
            if (sh.hpg % pl.hs != 0) return SSD_ERR_INVALID_ARGUMENT;
            // Work items of the persistent gradient kernel (one CTA per SM).  With whole-group
            // items, the pairs (chunk, group) that would form a last partial wave are split into
            // subsets of >= 2 heads, so the last wave is filled with smaller items; their dB/dC
            // shares are summed, in subset order, by a small kernel afterwards.
            const int64_t pairs = kmax * G;
            const int nsub_main = sh.hpg / pl.hs;
            pl.k_pairs = (int)pairs;
            pl.nsub_tail = nsub_main;
            if (p->bwd_heads == 0 && nsub_main == 1) {
                const int64_t sms = num_sms(), r = pairs % sms;
                // the fewest subsets (of at least 2 heads): halves measured faster than quarters
                // or single heads, whose per-item overhead (B/C loads, C B^T, dB/dC shares)
                // outweighs the finer fill of the last wave
                int f = 1;
                for (int d = 2; d <= pl.hs / 2; ++d)
                    if (pl.hs % d == 0) { f = d; break; }
                if (r > 0 && f > 1 && pairs > sms) {
                    pl.k_pairs = (int)(pairs - r);
                    pl.nsub_tail = f;
                }
            }
            pl.n_items = pl.k_pairs * nsub_main + (int)(pairs - pl.k_pairs) * pl.nsub_tail;
            const int64_t tail_items = nsub_main == 1 && pl.nsub_tail > 1 ? (pairs - pl.k_pairs) * pl.nsub_tail : 0;
            pl.off_tpart = lay.take(sizeof(float) * (size_t)tail_items * 2 * Q * (size_t)Nk);
            // dB/dC shares of head subsets, only when a CTA covers part of a group
            const size_t ksub = pl.hs < sh.hpg ? (size_t)kmax * (size_t)(H / pl.hs) : 0;
            if (a->chunk_states == nullptr)   // carried states, bf16, unless the forward kept them
                pl.off_states = lay.take(sizeof(__nv_bfloat16) * kh * (size_t)(P * Nk));
            pl.off_dstates = lay.take(sizeof(__nv_bfloat16) * kh * (size_t)(P * Nk));   // dS, bf16
            pl.off_cs = lay.take(sizeof(float) * kh);                                // chunk total log-decay
            pl.off_dBh = lay.take(sizeof(float) * ksub * Q * (size_t)Nk);
            pl.off_dCh = lay.take(sizeof(float) * ksub * Q * (size_t)Nk);
            pl.off_part = lay.take(sizeof(float) * kh * 4);
        }
    } else {
        pl.off_dt = lay.take(sizeof(float) * kh * Q);
        pl.off_cs = lay.take(sizeof(float) * kh * Q);
        pl.off_states = lay.take(sizeof(float) * kh * (size_t)(P * Nk));
    }
    if (bwd && !fused) {
        pl.off_dstates = lay.take(sizeof(float) * kh * (size_t)(P * Nk));
        pl.off_dBh = lay.take(sizeof(float) * kh * Q * (size_t)Nk);
        pl.off_dCh = lay.take(sizeof(float) * kh * Q * (size_t)Nk);
        pl.off_part = lay.take(sizeof(float) * kh * 4);
    }
    if (fused) pl.chunk_state_bytes = sizeof(__nv_bfloat16) * kh * (size_t)(P * Nk);
    const size_t st_bytes = sizeof(float) * (size_t)S * (size_t)H * (size_t)(P * Nk);
    const ssd_tensor *sts[4] = {&a->initial_states, bwd ? nullptr : &a->final_states,
                                b != nullptr ? &b->dfinal_states : nullptr, b != nullptr ? &b->dinitial_states : nullptr};
    for (int i = 0; i < 4; ++i)
        if (sts[i] != nullptr && sts[i]->ptr != nullptr && (sts[i]->dtype == SSD_BF16 || Nk != N)) {
            pl.st_bf16[i] = true;
            pl.off_st32[i] = lay.take(st_bytes);
        }
    pl.total = lay.cur;
    *out = pl;
    return SSD_OK;
}

ssd_status plan_bwd(const ssd_problem *p, const ssd_bwd_args *b, Plan *out) {
    if (b == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    SSD_TRY(plan_common(p, &b->fwd, true, out, b));
    const int dt_ = b->fwd.x.dtype;
    const int64_t H = p->nheads, P = p->headdim, N = p->dstate;
    const bool tok = p->seqlen > 0;
    SSD_TRY(check_tensor(b->dy, 4, dt_, tok));
    SSD_TRY(check_state(b->dfinal_states, H, P, N));
    SSD_TRY(check_tensor(b->dx, 4, dt_, tok));
    SSD_TRY(check_tensor(b->ddt, 3, SSD_F32, tok));
    SSD_TRY(check_vec(b->dA, true));
    SSD_TRY(check_tensor(b->dB, 4, dt_, tok));
    SSD_TRY(check_tensor(b->dC, 4, dt_, tok));
    SSD_TRY(check_vec(b->dD, b->fwd.D.ptr != nullptr));
    SSD_TRY(check_tensor(b->dz, 4, dt_, tok && b->fwd.z.ptr != nullptr));
    SSD_TRY(check_vec(b->ddt_bias, b->fwd.dt_bias.ptr != nullptr));
    SSD_TRY(check_state(b->dinitial_states, H, P, N));
    if (b->fwd.initial_states.ptr != nullptr && b->dinitial_states.ptr == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    return SSD_OK;
}

View3 view(const ssd_tensor &t) {
    View3 v;
    v.p = t.ptr; v.s0 = t.stride[0]; v.s1 = t.stride[1]; v.s2 = t.stride[2];
    return v;
}
MView3 mview(const ssd_tensor &t) {
    MView3 v;
    v.p = t.ptr; v.s0 = t.stride[0]; v.s1 = t.stride[1]; v.s2 = t.stride[2];
    return v;
}

template <typename Tp>
Tp *at(void *ws, size_t off) { return reinterpret_cast<Tp *>(static_cast<char *>(ws) + off); }

#define SSD_CUDA(expr)                               \
    do {                                             \
        if ((expr) != cudaSuccess) return SSD_ERR_CUDA; \
    } while (0)

// Metadata, dt/cs, carry-in states (and final states) -- shared by fwd and bwd.
ssd_status run_forward_states(const Plan &pl, const ssd_fwd_args *a, void *ws, float *final_, cudaStream_t st) {
    const Shape &sh = pl.sh;
    int32_t *hdr = at<int32_t>(ws, pl.off_hdr);
    SeqInfo *seqs = at<SeqInfo>(ws, pl.off_seqs);
    ChunkInfo *chunks = at<ChunkInfo>(ws, pl.off_chunks);
    float *dtw = at<float>(ws, pl.off_dt), *csw = at<float>(ws, pl.off_cs), *states = at<float>(ws, pl.off_states);
    SSD_CUDA(launch_build_meta(a->cu_seqlens, sh.B, sh.L, sh.S, sh.Q, 1, 1, 1, 1, sh.kmax, 0, hdr, seqs, chunks, nullptr,
                               at<int32_t>(ws, pl.off_lastunit), nullptr, 0, st));
    if (sh.kmax > 0) {
        SSD_CUDA(launch_chunk_cumsum(sh, hdr, chunks, (const float *)a->dt.ptr, a->dt.stride[0], a->dt.stride[1],
                                     (const float *)a->A.ptr, (const float *)a->dt_bias.ptr, dtw, csw, st));
        if (pl.bf16)
            SSD_CUDA(launch_chunk_state<__nv_bfloat16>(sh, hdr, chunks, view(a->x), view(a->B), dtw, csw, states, st));
        else
            SSD_CUDA(launch_chunk_state<float>(sh, hdr, chunks, view(a->x), view(a->B), dtw, csw, states, st));
    }
    SSD_CUDA(launch_state_passing(sh, hdr, seqs, csw + (sh.Q - 1), sh.Q, states, (const float *)a->initial_states.ptr,
                                  final_, 0, st));
    return SSD_OK;
}

}  // namespace

extern "C" {

const char *ssd_status_string(ssd_status s) {
    switch (s) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARGUMENT: return "SSD_ERR_INVALID_ARGUMENT";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED";
        case SSD_ERR_MISALIGNED: return "SSD_ERR_MISALIGNED";
        case SSD_ERR_WORKSPACE_TOO_SMALL: return "SSD_ERR_WORKSPACE_TOO_SMALL";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA";
        case SSD_ERR_DEVICE_TIMEOUT: return "SSD_ERR_DEVICE_TIMEOUT";
    }
    return "SSD_ERR_UNKNOWN";
}

int32_t ssd_abi_version(void) { return SSD_ABI_VERSION; }

ssd_status ssd_fwd_workspace_size(const ssd_problem *prob, const ssd_fwd_args *args, size_t *bytes) {
    if (bytes == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    Plan pl;
    SSD_TRY(plan_common(prob, args, false, &pl));
    *bytes = pl.total;
    return SSD_OK;
}

ssd_status ssd_fwd_debug_layout(const ssd_problem *prob, const ssd_fwd_args *args, ssd_debug_layout *out) {
    if (out == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    Plan pl;
    SSD_TRY(plan_common(prob, args, false, &pl));
    out->meta_counts = (int64_t)pl.off_hdr;
    out->chunk_info = (int64_t)pl.off_chunks;
    const bool staged = pl.algo == SSD_ALGO_STAGED;
    out->dt = staged ? (int64_t)pl.off_dt : -1;
    out->cs = staged ? (int64_t)pl.off_cs : -1;
    out->states = staged ? (int64_t)pl.off_states : -1;
    out->units = pl.algo == SSD_ALGO_FUSED ? (int64_t)pl.off_units : -1;
    out->qi = pl.sh.Q;
    return SSD_OK;
}

// A state tensor as the kernels take it: the caller's fp32 tensor, or the workspace's fp32
// copy of a bf16 one.
static ssd_tensor state32(const Plan &pl, int i, const ssd_tensor &t, void *ws) {
    ssd_tensor r = t;
    if (pl.st_bf16[i]) {
        r.ptr = at<float>(ws, pl.off_st32[i]);
        r.dtype = SSD_F32;
    }
    return r;
}
static int64_t state_rows(const Plan &pl) { return (int64_t)pl.sh.S * pl.sh.H * pl.sh.P; }
// caller's state tensor -> the kernels' fp32 rows of sh.N, and back
static cudaError_t state_in(const Plan &pl, const ssd_tensor &user, void *f32, cudaStream_t st) {
    return launch_states_cvt(user.ptr, user.dtype == SSD_BF16, pl.sh.Nio, f32, false, pl.sh.N, state_rows(pl), st);
}
static cudaError_t state_out(const Plan &pl, const void *f32, const ssd_tensor &user, cudaStream_t st) {
    return launch_states_cvt(f32, false, pl.sh.N, user.ptr, user.dtype == SSD_BF16, pl.sh.Nio, state_rows(pl), st);
}

static ssd_status fwd_impl(const Plan &pl, const ssd_fwd_args *a, void *ws, cudaStream_t st) {
    const Shape &sh = pl.sh;
    float *final_ = (float *)a->final_states.ptr;
    if (pl.algo == SSD_ALGO_SPLIT) {
        int32_t *hdr = at<int32_t>(ws, pl.off_hdr);
        SeqInfo *seqs = at<SeqInfo>(ws, pl.off_seqs);
        ChunkInfo *chunks = at<ChunkInfo>(ws, pl.off_chunks);
        __nv_bfloat16 *states = a->chunk_states ? static_cast<__nv_bfloat16 *>(a->chunk_states)
                                                : at<__nv_bfloat16>(ws, pl.off_states);
        float *lam = at<float>(ws, pl.off_cs);
        SSD_CUDA(launch_build_meta(a->cu_seqlens, sh.B, sh.L, sh.S, sh.Q, 1, 1, 1, 1, sh.kmax, 0, hdr, seqs, chunks,
                                   nullptr, at<int32_t>(ws, pl.off_lastunit), nullptr, 0, st));
        SSD_CUDA(launch_split_states(sh, hdr, chunks, seqs, a->x.ptr, a->x.stride, a->B.ptr, a->B.stride,
                                     (const float *)a->dt.ptr, a->dt.stride[0], a->dt.stride[1], (const float *)a->A.ptr,
                                     (const float *)a->dt_bias.ptr, (const float *)a->initial_states.ptr, final_, states,
                                     lam, num_sms(), st));
        if (sh.kmax > 0)
            SSD_CUDA(launch_split_out(sh, hdr, chunks, a->x.ptr, a->x.stride, a->B.ptr, a->B.stride, a->C.ptr,
                                      a->C.stride, (const float *)a->dt.ptr, a->dt.stride[0], a->dt.stride[1],
                                      (const float *)a->A.ptr, (const float *)a->D.ptr, (const float *)a->dt_bias.ptr,
                                      a->z.ptr, a->z.ptr ? a->z.stride : nullptr, a->y.ptr, a->y.stride, states,
                                      num_sms(), st));
        if (final_ != nullptr && (pl.varlen || sh.L == 0))
            SSD_CUDA(launch_empty_seq_final(sh.S, sh.H, sh.P * sh.N, seqs, hdr,
                                            (const float *)a->initial_states.ptr, final_, st));
        return SSD_OK;
    }
    if (pl.algo == SSD_ALGO_FUSED) {
        int32_t *hdr = at<int32_t>(ws, pl.off_hdr);
        SeqInfo *seqs = at<SeqInfo>(ws, pl.off_seqs);
        UnitInfo *units = at<UnitInfo>(ws, pl.off_units);
        uint32_t *flags = at<uint32_t>(ws, pl.off_flags);
        SSD_CUDA(launch_build_meta(a->cu_seqlens, sh.B, sh.L, sh.S, sh.Q, sh.R, sh.useg_num, sh.useg_den, fused_block_units(), sh.kmax,
                                   sh.umax, hdr, seqs,
                                   at<ChunkInfo>(ws, pl.off_chunks), units, at<int32_t>(ws, pl.off_lastunit), flags,
                                   (int64_t)sh.umax * sh.H, st));
        const int64_t tickets = (int64_t)sh.umax * sh.H;
        if (tickets > 0) {
            const int64_t slots = 2LL * num_sms();   // two CTAs per SM
            const int grid = (int)(tickets < slots ? tickets : slots);
            SSD_CUDA(launch_fused_fwd(sh, hdr, units, a->x.ptr, a->x.stride, a->B.ptr, a->B.stride, a->C.ptr,
                                      a->C.stride, (const float *)a->dt.ptr, a->dt.stride[0], a->dt.stride[1],
                                      (const float *)a->A.ptr, (const float *)a->D.ptr, (const float *)a->dt_bias.ptr,
                                      a->z.ptr, a->z.ptr ? a->z.stride : nullptr, a->y.ptr, a->y.stride,
                                      (const float *)a->initial_states.ptr, final_, at<float>(ws, pl.off_agg),
                                      at<float>(ws, pl.off_incl), at<float>(ws, pl.off_lam), flags, grid,
                                      static_cast<__nv_bfloat16 *>(a->chunk_states), false, seqs, st));
        }
        if (final_ != nullptr && (pl.varlen || sh.L == 0))
            SSD_CUDA(launch_empty_seq_final(sh.S, sh.H, sh.P * sh.N, seqs, hdr,
                                            (const float *)a->initial_states.ptr, final_, st));
        return SSD_OK;
    }
    SSD_TRY(run_forward_states(pl, a, ws, final_, st));
    if (sh.kmax > 0) {
        int32_t *hdr = at<int32_t>(ws, pl.off_hdr);
        ChunkInfo *chunks = at<ChunkInfo>(ws, pl.off_chunks);
        float *dtw = at<float>(ws, pl.off_dt), *csw = at<float>(ws, pl.off_cs), *states = at<float>(ws, pl.off_states);
        if (pl.bf16)
            SSD_CUDA(launch_chunk_scan<__nv_bfloat16>(sh, hdr, chunks, view(a->x), view(a->B), view(a->C), view(a->z),
                                                      (const float *)a->D.ptr, dtw, csw, states, mview(a->y), st));
        else
            SSD_CUDA(launch_chunk_scan<float>(sh, hdr, chunks, view(a->x), view(a->B), view(a->C), view(a->z),
                                              (const float *)a->D.ptr, dtw, csw, states, mview(a->y), st));
    }
    return SSD_OK;
}

ssd_status ssd_chunk_states_size(const ssd_problem *prob, const ssd_fwd_args *args, size_t *bytes) {
    if (bytes == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    Plan pl;
    SSD_TRY(plan_common(prob, args, false, &pl));
    if (pl.algo == SSD_ALGO_STAGED) return SSD_ERR_UNSUPPORTED;
    *bytes = pl.chunk_state_bytes;
    return SSD_OK;
}

ssd_status ssd_bwd_workspace_size(const ssd_problem *prob, const ssd_bwd_args *args, size_t *bytes) {
    if (bytes == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    Plan pl;
    SSD_TRY(plan_bwd(prob, args, &pl));
    *bytes = pl.total;
    return SSD_OK;
}

static ssd_status bwd_impl(const Plan &pl, const ssd_bwd_args *b, void *ws, cudaStream_t st) {
    const Shape &sh = pl.sh;
    const ssd_fwd_args *a = &b->fwd;
    if (pl.algo == SSD_ALGO_FUSED || pl.algo == SSD_ALGO_SPLIT) {
        const bool split = pl.algo == SSD_ALGO_SPLIT;
        int32_t *hdr = at<int32_t>(ws, pl.off_hdr);
        SeqInfo *seqs = at<SeqInfo>(ws, pl.off_seqs);
        ChunkInfo *chunks = at<ChunkInfo>(ws, pl.off_chunks);
        UnitInfo *units = split ? nullptr : at<UnitInfo>(ws, pl.off_units);
        uint32_t *flags = split ? nullptr : at<uint32_t>(ws, pl.off_flags);
        const bool kept = a->chunk_states != nullptr;   // the forward's chunk states, else recomputed
        __nv_bfloat16 *states = kept ? static_cast<__nv_bfloat16 *>(a->chunk_states) : at<__nv_bfloat16>(ws, pl.off_states);
        __nv_bfloat16 *dS = at<__nv_bfloat16>(ws, pl.off_dstates);
        float *clam = at<float>(ws, pl.off_cs);
        float *dBh = at<float>(ws, pl.off_dBh), *dCh = at<float>(ws, pl.off_dCh), *part = at<float>(ws, pl.off_part);
        const int64_t n_zero = (int64_t)sh.umax * sh.H;   // the unit flags
        SSD_CUDA(launch_build_meta(a->cu_seqlens, sh.B, sh.L, sh.S, sh.Q, sh.R, sh.useg_num, sh.useg_den,
                                   fused_block_units(), sh.kmax, sh.umax, hdr, seqs, chunks, units,
                                   at<int32_t>(ws, pl.off_lastunit), flags, n_zero, st));
        const int64_t tickets = (int64_t)sh.umax * sh.H;
        if (split && !kept) {   // carried state entering every chunk tile: the split forward's first two launches
            SSD_CUDA(launch_split_states(sh, hdr, chunks, seqs, a->x.ptr, a->x.stride, a->B.ptr, a->B.stride,
                                         (const float *)a->dt.ptr, a->dt.stride[0], a->dt.stride[1],
                                         (const float *)a->A.ptr, (const float *)a->dt_bias.ptr,
                                         (const float *)a->initial_states.ptr, nullptr, states, clam, num_sms(), st));
        } else if (tickets > 0 && !kept) {
            // carried state entering every chunk (forward recomputed in states-only mode)
            const int64_t slots = 2LL * num_sms();   // two CTAs per SM
            const int grid = (int)(tickets < slots ? tickets : slots);
            SSD_CUDA(launch_fused_fwd(sh, hdr, units, a->x.ptr, a->x.stride, a->B.ptr, a->B.stride, a->C.ptr,
                                      a->C.stride, (const float *)a->dt.ptr, a->dt.stride[0], a->dt.stride[1],
                                      (const float *)a->A.ptr, (const float *)a->D.ptr, (const float *)a->dt_bias.ptr,
                                      nullptr, nullptr, nullptr, a->x.stride, (const float *)a->initial_states.ptr,
                                      nullptr, at<float>(ws, pl.off_agg), at<float>(ws, pl.off_incl),
                                      at<float>(ws, pl.off_lam), flags, grid, states, true, seqs, st));
        }
        BwdTcArgs ta;
        ta.x = a->x.ptr; ta.Bp = a->B.ptr; ta.Cp = a->C.ptr;
        ta.sx = a->x.stride; ta.sb = a->B.stride; ta.sc = a->C.stride;
        ta.dt_raw = (const float *)a->dt.ptr; ta.sdb = a->dt.stride[0]; ta.sdl = a->dt.stride[1];
        ta.A = (const float *)a->A.ptr; ta.D = (const float *)a->D.ptr; ta.bias = (const float *)a->dt_bias.ptr;
        ta.dy = b->dy.ptr; ta.z = a->z.ptr; ta.sdy = b->dy.stride; ta.sz = a->z.ptr ? a->z.stride : nullptr;
        ta.dx = b->dx.ptr; ta.dz = b->dz.ptr; ta.sdx = b->dx.stride; ta.sdz = b->dz.ptr ? b->dz.stride : nullptr;
        ta.ddt = (float *)b->ddt.ptr; ta.sddb = b->ddt.stride[0]; ta.sddl = b->ddt.stride[1];
        ta.states = states; ta.dS = dS; ta.chunk_lam = clam; ta.dBh = dBh; ta.dCh = dCh; ta.partials = part;
        ta.hs = pl.hs; ta.hs_ds = dstates_heads_per_cta(sh.kmax, sh.H, sh.hpg);
        ta.dB = b->dB.ptr; ta.dC = b->dC.ptr; ta.sdB = b->dB.stride; ta.sdC = b->dC.stride;
        ta.k_pairs = pl.k_pairs; ta.nsub_tail = pl.nsub_tail; ta.n_items = pl.n_items;
        ta.grid = pl.n_items < num_sms() ? pl.n_items : num_sms();
        ta.tpart = at<float>(ws, pl.off_tpart);
        ta.dA = (float *)b->dA.ptr; ta.dD = (float *)b->dD.ptr; ta.dbias = (float *)b->ddt_bias.ptr;
        if (sh.kmax > 0) SSD_CUDA(launch_bwd_dstates_tc(sh, hdr, chunks, ta, st));
        SSD_CUDA(launch_state_passing(sh, hdr, seqs, clam, 1, dS, (const float *)b->dfinal_states.ptr,
                                      (float *)b->dinitial_states.ptr, 1, st));
        if (sh.kmax > 0) {
            SSD_CUDA(launch_bwd_chunk_tc(sh, hdr, chunks, ta, st));
            if (pl.hs < sh.hpg) {
                // sum the head subsets' shares: the same reduction over H/hs "heads", hpg/hs per group
                Shape ss = sh;
                ss.H = sh.H / pl.hs;
                ss.hpg = sh.hpg / pl.hs;
                SSD_CUDA(launch_reduce_group<__nv_bfloat16>(ss, hdr, chunks, dBh, mview(b->dB), dCh, mview(b->dC), st));
            }
        } else {   // no chunks: the per-head sums (zero) without the gradient kernel's finishing launch
            SSD_CUDA(launch_reduce_heads(sh, hdr, part, (float *)b->dA.ptr, (float *)b->dD.ptr,
                                         (float *)b->ddt_bias.ptr, st));
        }
        return SSD_OK;
    }
    SSD_TRY(run_forward_states(pl, a, ws, nullptr, st));
    int32_t *hdr = at<int32_t>(ws, pl.off_hdr);
    SeqInfo *seqs = at<SeqInfo>(ws, pl.off_seqs);
    ChunkInfo *chunks = at<ChunkInfo>(ws, pl.off_chunks);
    float *dtw = at<float>(ws, pl.off_dt), *csw = at<float>(ws, pl.off_cs), *states = at<float>(ws, pl.off_states);
    float *dstates = at<float>(ws, pl.off_dstates);
    float *dBh = at<float>(ws, pl.off_dBh), *dCh = at<float>(ws, pl.off_dCh), *part = at<float>(ws, pl.off_part);
    if (sh.kmax > 0) {
        if (pl.bf16)
            SSD_CUDA(launch_bwd_dstates<__nv_bfloat16>(sh, hdr, chunks, view(b->dy), view(a->z), view(a->C), csw,
                                                       dstates, st));
        else
            SSD_CUDA(launch_bwd_dstates<float>(sh, hdr, chunks, view(b->dy), view(a->z), view(a->C), csw, dstates, st));
    }
    SSD_CUDA(launch_state_passing(sh, hdr, seqs, csw + (sh.Q - 1), sh.Q, dstates, (const float *)b->dfinal_states.ptr,
                                  (float *)b->dinitial_states.ptr, 1, st));
    if (sh.kmax > 0) {
        if (pl.bf16) {
            SSD_CUDA(launch_bwd_chunk<__nv_bfloat16>(
                sh, hdr, chunks, view(a->x), view(a->B), view(a->C), view(a->z), view(b->dy), (const float *)a->dt.ptr,
                a->dt.stride[0], a->dt.stride[1], (const float *)a->A.ptr, (const float *)a->D.ptr,
                (const float *)a->dt_bias.ptr, dtw, csw, states, dstates, mview(b->dx), mview(b->dz),
                (float *)b->ddt.ptr, b->ddt.stride[0], b->ddt.stride[1], dBh, dCh, part, st));
            SSD_CUDA(launch_reduce_group<__nv_bfloat16>(sh, hdr, chunks, dBh, mview(b->dB), dCh, mview(b->dC), st));
        } else {
            SSD_CUDA(launch_bwd_chunk<float>(
                sh, hdr, chunks, view(a->x), view(a->B), view(a->C), view(a->z), view(b->dy), (const float *)a->dt.ptr,
                a->dt.stride[0], a->dt.stride[1], (const float *)a->A.ptr, (const float *)a->D.ptr,
                (const float *)a->dt_bias.ptr, dtw, csw, states, dstates, mview(b->dx), mview(b->dz),
                (float *)b->ddt.ptr, b->ddt.stride[0], b->ddt.stride[1], dBh, dCh, part, st));
            SSD_CUDA(launch_reduce_group<float>(sh, hdr, chunks, dBh, mview(b->dB), dCh, mview(b->dC), st));
        }
    }
    SSD_CUDA(launch_reduce_heads(sh, hdr, part, (float *)b->dA.ptr, (float *)b->dD.ptr, (float *)b->ddt_bias.ptr, st));
    return SSD_OK;
}

ssd_status ssd_fwd(const ssd_problem *prob, const ssd_fwd_args *a, void *ws, size_t ws_bytes, void *stream) {
    Plan pl;
    SSD_TRY(plan_common(prob, a, false, &pl));
    if (ws == nullptr || ws_bytes < pl.total) return SSD_ERR_WORKSPACE_TOO_SMALL;
    if (((uintptr_t)ws) % kAlign != 0) return SSD_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    ssd_fwd_args a32 = *a;
    a32.initial_states = state32(pl, 0, a->initial_states, ws);
    a32.final_states = state32(pl, 1, a->final_states, ws);
    if (pl.st_bf16[0]) SSD_CUDA(state_in(pl, a->initial_states, a32.initial_states.ptr, st));
    SSD_TRY(fwd_impl(pl, &a32, ws, st));
    if (pl.st_bf16[1]) SSD_CUDA(state_out(pl, a32.final_states.ptr, a->final_states, st));
    return SSD_OK;
}

ssd_status ssd_bwd(const ssd_problem *prob, const ssd_bwd_args *b, void *ws, size_t ws_bytes, void *stream) {
    Plan pl;
    SSD_TRY(plan_bwd(prob, b, &pl));
    if (ws == nullptr || ws_bytes < pl.total) return SSD_ERR_WORKSPACE_TOO_SMALL;
    if (((uintptr_t)ws) % kAlign != 0) return SSD_ERR_MISALIGNED;
    cudaStream_t st = (cudaStream_t)stream;
    ssd_bwd_args b32 = *b;
    b32.fwd.initial_states = state32(pl, 0, b->fwd.initial_states, ws);
    b32.dfinal_states = state32(pl, 2, b->dfinal_states, ws);
    b32.dinitial_states = state32(pl, 3, b->dinitial_states, ws);
    if (pl.st_bf16[0]) SSD_CUDA(state_in(pl, b->fwd.initial_states, b32.fwd.initial_states.ptr, st));
    if (pl.st_bf16[2]) SSD_CUDA(state_in(pl, b->dfinal_states, b32.dfinal_states.ptr, st));
    SSD_TRY(bwd_impl(pl, &b32, ws, st));
    if (pl.st_bf16[3]) SSD_CUDA(state_out(pl, b32.dinitial_states.ptr, b->dinitial_states, st));
    return SSD_OK;
}

ssd_status ssd_selftest_bounded_wait(void *ws, size_t ws_bytes, int32_t wait_ms, void *stream) {
    if (ws == nullptr || ws_bytes < HDR_WORDS * sizeof(int32_t) || wait_ms < 1 || wait_ms > 2000)
        return SSD_ERR_INVALID_ARGUMENT;
    if (launch_wait_probe(static_cast<int32_t *>(ws), wait_ms, (cudaStream_t)stream) != cudaSuccess) return SSD_ERR_CUDA;
    return SSD_OK;
}

ssd_status ssd_varlen_metadata(const int32_t *cu_seqlens, int64_t nseqs, int64_t seqlen, int64_t chunk_size,
                               int32_t *seq_idx, int32_t *chunk_begin, int32_t *segments, int32_t *status,
                               void *stream) {
    if (cu_seqlens == nullptr || chunk_begin == nullptr || segments == nullptr || status == nullptr)
        return SSD_ERR_INVALID_ARGUMENT;
    if (nseqs < 1 || seqlen < 0 || chunk_size < 1) return SSD_ERR_INVALID_ARGUMENT;
    if (nseqs > (int64_t)1 << 24 || seqlen > (int64_t)1 << 30 || chunk_size > 65536) return SSD_ERR_UNSUPPORTED;
    if (launch_varlen_metadata(cu_seqlens, (int)nseqs, (int)seqlen, (int)chunk_size, status, chunk_begin, segments,
                               seq_idx, (cudaStream_t)stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}

ssd_status ssd_query_status(const void *ws, void *stream) {
    if (ws == nullptr) return SSD_ERR_INVALID_ARGUMENT;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, static_cast<const int32_t *>(ws) + HDR_STATUS, sizeof(v), cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return SSD_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
    return (ssd_status)v;
}

}  // extern "C"
