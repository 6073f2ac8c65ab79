// meta.cu -- chunk-tile and work-unit lists for fixed-length batches and packed
// variable-length sequences (cu_seqlens), and the packed-sequence metadata entry
// point (sequence index of every token, segments of every physical chunk).
//
// The chunk grid runs over the token axis of each batch row: physical chunk c holds
// tokens [cQ, (c+1)Q).  With packed sequences a chunk may hold parts of several
// sequences, so chunk boundaries need not meet sequence starts; each part (segment) is
// one chunk tile (see ChunkInfo), and the carried state is reset to a sequence's initial
// state at its first tile.  A sequence's tiles are listed in order, sequences in order.
// Work units of the fused forward group consecutive tiles of one sequence (segment j of
// the sequence): a sequence of n tiles has m = max(ceil(n / R), min(n, ceil(n * num /
// den))) units of floor(n/m) or ceil(n/m) tiles, the larger ones first (the planner
// raises m above ceil(n/R) so that the units fill whole rounds of the resident CTAs);
// units are grouped in blocks of KB.  Units are listed by (block, sequence, segment), so
// a unit only ever depends on units listed before it and the units of one sequence inside
// one block are consecutive in the list.
#include <algorithm>

#include "common.cuh"

namespace ssd {

namespace {

constexpr int kMetaThreads = 1024;

__device__ int block_excl_scan(int v, int *total, int *sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += t;
    }
    if (lane == 31) sm[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = lane < nw ? sm[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += t;
        }
        sm[lane] = s;
    }
    __syncthreads();
    int excl = x - v + (w > 0 ? sm[w - 1] : 0);
    *total = sm[nw - 1];
    __syncthreads();
    return excl;
}

// Segment count of a sequence of n chunks (see the file comment).
__device__ __forceinline__ int seg_count(int n, int R, int num, int den) {
    if (n <= 0) return 0;
    const int lo = (n + R - 1) / R;
    const int64_t want = ((int64_t)n * num + den - 1) / den;
    const int m = (int)(want < n ? want : n);
    return m > lo ? m : lo;
}

__device__ int block_max(int v, int *sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sm[w] = v;
    __syncthreads();
    int m = 0;
    for (int i = 0; i < nw; ++i) m = max(m, sm[i]);
    __syncthreads();
    return m;
}

__global__ void __launch_bounds__(kMetaThreads)
k_build_meta(const int32_t *__restrict__ cu, int B, int L, int S, int Q, int R, int num, int den, int KB, int kmax,
             int umax,
             int32_t *hdr, SeqInfo *seqs, ChunkInfo *chunks, UnitInfo *units, int32_t *last_unit,
             uint32_t *zero_words, int64_t n_zero) {
    __shared__ int sm[32];
    __shared__ int bad;
    const int tid = threadIdx.x;
    for (int64_t i = tid; i < n_zero; i += blockDim.x) zero_words[i] = 0u;
    if (tid == 0) bad = 0;
    __syncthreads();
    if (tid < HDR_WORDS) hdr[tid] = 0;
    if (cu != nullptr) {
        for (int s = tid; s <= S; s += blockDim.x) {
            int c = cu[s];
            if (s == 0 && c != 0) bad = 1;
            if (s == S && c != L) bad = 1;
            if (s < S && cu[s + 1] < c) bad = 1;
        }
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) hdr[HDR_STATUS] = SSD_ERR_INVALID_ARGUMENT;
        return;
    }
    // pass 1: chunk offsets and the largest segment count
    int carry = 0, maxseg = 0;
    for (int base = 0; base < S; base += blockDim.x) {
        int s = base + tid;
        int len = 0, t0 = 0, b = 0;
        if (s < S) {
            if (cu) { t0 = cu[s]; len = cu[s + 1] - t0; }
            else { b = s; len = L; }
        }
        int nch = seq_nchunks(t0, len, Q);
        int tot;
        int off = block_excl_scan(s < S ? nch : 0, &tot, sm);
        if (s < S) {
            SeqInfo si;
            si.b = b; si.t0 = t0; si.len = len; si.chunk0 = carry + off;
            si.nch = nch; si.pad0 = si.pad1 = si.pad2 = 0;
            seqs[s] = si;
        }
        int nseg = seg_count(nch, R, num, den);
        maxseg = max(maxseg, block_max(s < S ? nseg : 0, sm));
        carry += tot;
    }
    const int nchunks = carry;
    if (nchunks > kmax) {
        if (tid == 0) hdr[HDR_STATUS] = SSD_ERR_INVALID_ARGUMENT;
        return;
    }
    __syncthreads();
    // pass 2: the chunk list, one thread per chunk; its sequence is the last one whose first
    // chunk is not after it (empty sequences share their successor's first chunk)
    for (int c = tid; c < nchunks; c += blockDim.x) {
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seqs[mid].chunk0 <= c) lo = mid; else hi = mid - 1;
        }
        const SeqInfo si = seqs[lo];
        const int j = c - si.chunk0;
        ChunkInfo ci;
        ci.seq = lo; ci.b = si.b; ci.t0 = (si.t0 / Q + j) * Q;
        ci.lo = (int16_t)max(si.t0 - ci.t0, 0);
        ci.len = (int16_t)min(Q, si.t0 + si.len - ci.t0);
        chunks[c] = ci;
    }
    // pass 3: work units ordered by (block of KB segments, sequence, segment)
    int nunits = 0;
    if (units != nullptr) {
        const int maxblk = (maxseg + KB - 1) / KB;
        for (int blk = 0; blk < maxblk; ++blk) {
            for (int base = 0; base < S; base += blockDim.x) {
                int s = base + tid;
                int cnt = 0, nch = 0, nseg = 0;
                SeqInfo si;
                if (s < S) {
                    si = seqs[s];
                    nch = si.nch;
                    nseg = seg_count(nch, R, num, den);
                    cnt = max(0, min(KB, nseg - blk * KB));
                }
                int tot;
                int off = block_excl_scan(cnt, &tot, sm);
                for (int i = 0; i < cnt; ++i) {
                    const int j = blk * KB + i;
                    const int u = nunits + off + i;
                    if (u < umax) {
                        UnitInfo ui;
                        ui.seq = s; ui.b = si.b;
                        const int base = nch / nseg, rem = nch % nseg;
                        const int c0 = j * base + min(j, rem);
                        ui.t0 = (si.t0 / Q + c0) * Q;
                        ui.nchunk = base + (j < rem ? 1 : 0);
                        ui.len = min(ui.nchunk * Q, si.t0 + si.len - ui.t0);
                        ui.lo = (int16_t)(c0 == 0 ? si.t0 - ui.t0 : 0);
                        ui.prev = (j == 0) ? -1 : (i > 0 ? u - 1 : last_unit[s]);
                        ui.last = (j == nseg - 1) ? 1 : 0;
                        ui.j = j;
                        units[u] = ui;
                        if (i == cnt - 1) last_unit[s] = u;
                    }
                }
                nunits += tot;
            }
            __syncthreads();
        }
        if (nunits > umax && tid == 0) hdr[HDR_STATUS] = SSD_ERR_INVALID_ARGUMENT;
    }
    __syncthreads();
    if (tid == 0) {
        hdr[HDR_NCHUNKS] = nchunks;
        hdr[HDR_NUNITS] = nunits > umax ? 0 : nunits;
        hdr[HDR_NSEQS] = S;
        hdr[HDR_MAXSEG] = maxseg;
    }
}

// Fixed-length batch (no cu_seqlens): every sequence has the same chunk and segment
// counts, so each list entry has a closed form -- the lists the general kernel builds,
// entry for entry, with one thread per entry and no block-wide steps.  Sequence s = row s;
// chunk c = (s, c mod nch); units of block blk (KB segments, cnt in the last) are listed
// sequence by sequence, so unit (s, j = blk KB + i) sits at B blk KB + s cnt + i.
__global__ void __launch_bounds__(kMetaThreads)
k_build_meta_fixed(int B, int L, int Q, int R, int num, int den, int KB, int kmax, int umax, int32_t *hdr,
                   SeqInfo *seqs, ChunkInfo *chunks, UnitInfo *units, uint32_t *zero_words, int64_t n_zero) {
    const int nch = (L + Q - 1) / Q;
    const int nseg = seg_count(nch, R, num, den);
    const int64_t nchunks = (int64_t)B * nch, nunits = units != nullptr ? (int64_t)B * nseg : 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool fits = nchunks <= kmax && nunits <= umax;
    if (t0 == 0) {
        for (int i = 0; i < HDR_WORDS; ++i) hdr[i] = 0;
        if (!fits) hdr[HDR_STATUS] = SSD_ERR_INVALID_ARGUMENT;
        hdr[HDR_NCHUNKS] = fits ? (int)nchunks : 0;
        hdr[HDR_NUNITS] = fits ? (int)nunits : 0;
        hdr[HDR_NSEQS] = B;
        hdr[HDR_MAXSEG] = nseg;
    }
    for (int64_t i = t0; i < n_zero; i += stride) zero_words[i] = 0u;
    if (!fits) return;
    for (int64_t s = t0; s < B; s += stride) {
        SeqInfo si;
        si.b = (int)s; si.t0 = 0; si.len = L; si.chunk0 = (int)(s * nch);
        si.nch = nch; si.pad0 = si.pad1 = si.pad2 = 0;
        seqs[s] = si;
    }
    for (int64_t c = t0; c < nchunks; c += stride) {
        const int s = (int)(c / nch), j = (int)(c % nch);
        ChunkInfo ci;
        ci.seq = s; ci.b = s; ci.t0 = j * Q; ci.len = (int16_t)min(Q, L - j * Q);
        ci.lo = 0;
        chunks[c] = ci;
    }
    const int base = nseg > 0 ? nch / nseg : 0, rem = nseg > 0 ? nch % nseg : 0;
    for (int64_t u = t0; u < nunits; u += stride) {
        const int64_t blk = u / ((int64_t)B * KB);          // full blocks before hold B KB units each
        const int cnt = min(KB, nseg - (int)blk * KB);
        const int64_t r = u - blk * B * KB;
        const int s = (int)(r / cnt), i = (int)(r % cnt);
        const int j = (int)blk * KB + i;
        UnitInfo ui;
        ui.seq = s; ui.b = s;
        const int c0 = j * base + min(j, rem);
        ui.t0 = c0 * Q;
        ui.nchunk = base + (j < rem ? 1 : 0);
        ui.len = min(ui.nchunk * Q, L - c0 * Q);
        ui.prev = j == 0 ? -1 : (i > 0 ? (int)u - 1 : (int)((blk - 1) * B * KB + (int64_t)s * KB + KB - 1));
        ui.last = j == nseg - 1 ? 1 : 0;
        ui.j = j;
        ui.lo = 0;
        units[u] = ui;
    }
}

// final_states[s] = initial_states[s] (or 0) for sequences with no tokens.
__global__ void k_empty_seq_final(int S, int H, int PN, const SeqInfo *seqs, const int32_t *hdr,
                                  const float *init, float *final_) {
    const int s = blockIdx.x, h = blockIdx.y;
    if (hdr[HDR_STATUS] != 0 || s >= S || seqs[s].len != 0) return;
    const int64_t base = ((int64_t)s * H + h) * PN;
    for (int i = threadIdx.x; i < PN; i += blockDim.x) final_[base + i] = init ? init[base + i] : 0.f;
}

// One block: clear the status word, then wait (bounded) for a header flag nothing sets.
__global__ void k_wait_probe(int32_t *hdr, uint64_t limit_ns) {
    if (threadIdx.x != 0) return;
    hdr[HDR_STATUS] = 0;
    hdr[HDR_PROBE] = 0;
    __threadfence();
    volatile int32_t *flag = hdr + HDR_PROBE;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (*flag != 0) return;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > limit_ns) break;
        __nanosleep(1000);
    }
    set_status(hdr, SSD_ERR_DEVICE_TIMEOUT);
}

// ---------------------------------------------------------------- packed-sequence metadata
// Largest s in [0, S] with cu[s] <= t (cu validated: cu[0] = 0 <= t, non-decreasing).
__device__ __forceinline__ int seq_of(const int32_t *cu, int S, int t) {
    int lo = 0, hi = S;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Walks the segments of physical chunk c (tokens [cQ, min((c+1)Q, L))): the sequence
// holding the current token runs to min(its end, the chunk's end), then the next token's
// sequence takes over.  Writes them at seg (when not null); returns their number.
__device__ int chunk_segments(const int32_t *cu, int S, int L, int Q, int c, int32_t *seg) {
    const int end = min((c + 1) * Q, L);
    int a = c * Q, n = 0;
    while (a < end) {
        const int s = seq_of(cu, S, a);
        const int e = min(cu[s + 1], end);
        if (seg != nullptr) {
            seg[3 * n] = s;
            seg[3 * n + 1] = a;
            seg[3 * n + 2] = e;
        }
        ++n;
        a = e;
    }
    return n;
}

// One block: validates cu (status), then the segment count of every physical chunk, their
// exclusive scan (chunk_begin) and the segments themselves.
__global__ void __launch_bounds__(kMetaThreads)
k_varlen_segments(const int32_t *__restrict__ cu, int S, int L, int Q, int32_t *status, int32_t *chunk_begin,
                  int32_t *segments) {
    __shared__ int sm[32];
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int s = tid; s <= S; s += blockDim.x) {
        const int c = cu[s];
        if ((s == 0 && c != 0) || (s == S && c != L) || (s < S && cu[s + 1] < c)) bad = 1;
    }
    __syncthreads();
    if (tid == 0) *status = bad ? SSD_ERR_INVALID_ARGUMENT : SSD_OK;
    if (bad) return;
    const int nch = (L + Q - 1) / Q;
    int carry = 0;
    for (int base = 0; base < nch; base += blockDim.x) {
        const int c = base + tid;
        const int n = c < nch ? chunk_segments(cu, S, L, Q, c, nullptr) : 0;
        int tot;
        const int off = block_excl_scan(n, &tot, sm);
        if (c < nch) {
            chunk_begin[c] = carry + off;
            chunk_segments(cu, S, L, Q, c, segments + 3 * (int64_t)(carry + off));
        }
        carry += tot;
    }
    if (tid == 0) chunk_begin[nch] = carry;
}

// seq_idx[t] for every token (after k_varlen_segments has validated cu).
__global__ void k_varlen_seq_idx(const int32_t *__restrict__ cu, int S, int L, const int32_t *status,
                                 int32_t *seq_idx) {
    if (*status != SSD_OK) return;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < L; t += (int64_t)gridDim.x * blockDim.x)
        seq_idx[t] = seq_of(cu, S, (int)t);
}

}  // namespace

cudaError_t launch_varlen_metadata(const int32_t *cu, int S, int L, int Q, int32_t *status, int32_t *chunk_begin,
                                   int32_t *segments, int32_t *seq_idx, cudaStream_t st) {
    k_varlen_segments<<<1, kMetaThreads, 0, st>>>(cu, S, L, Q, status, chunk_begin, segments);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || seq_idx == nullptr || L == 0) return e;
    const int blocks = (int)std::min<int64_t>(((int64_t)L + 255) / 256, 4096);
    k_varlen_seq_idx<<<blocks, 256, 0, st>>>(cu, S, L, status, seq_idx);
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(int32_t *hdr, int wait_ms, cudaStream_t st) {
    k_wait_probe<<<1, 32, 0, st>>>(hdr, (uint64_t)wait_ms * 1000000ull);
    return cudaGetLastError();
}

cudaError_t launch_build_meta(const int32_t *cu, int B, int L, int S, int Q, int R, int num, int den, int KB,
                              int kmax, int umax, int32_t *hdr, SeqInfo *seqs, ChunkInfo *chunks, UnitInfo *units,
                              int32_t *last_unit, uint32_t *zero_words, int64_t n_zero, cudaStream_t st) {
    if (cu == nullptr) {
        const int64_t work = std::max<int64_t>({(int64_t)B * ((L + Q - 1) / Q), n_zero, (int64_t)B, 1});
        const int blocks = (int)std::min<int64_t>((work + kMetaThreads - 1) / kMetaThreads, 256);
        k_build_meta_fixed<<<blocks, kMetaThreads, 0, st>>>(B, L, Q, R, num, den, KB, kmax, umax, hdr, seqs, chunks,
                                                            units, zero_words, n_zero);
    } else {
        k_build_meta<<<1, kMetaThreads, 0, st>>>(cu, B, L, S, Q, R, num, den, KB, kmax, umax, hdr, seqs, chunks, units,
                                                 last_unit, zero_words, n_zero);
    }
    return cudaGetLastError();
}

cudaError_t launch_empty_seq_final(int S, int H, int PN, const SeqInfo *seqs, const int32_t *hdr,
                                   const float *init, float *final_, cudaStream_t st) {
    if (S <= 0) return cudaSuccess;
    k_empty_seq_final<<<dim3(S, H), 256, 0, st>>>(S, H, PN, seqs, hdr, init, final_);
    return cudaGetLastError();
}

// State tensors at the boundary whose storage differs from the kernels' fp32 [.., N] rows: bf16
// storage, and/or dstate 64 on the tensor-core path (rows of 128, the upper half zero).  Copies
// rows of `src_n` columns into rows of `dst_n` columns (zero-filled past src_n), widening bf16
// or rounding to it (nearest even).
template <typename S, typename D>
__global__ void k_states_cvt(const S *src, int src_n, D *dst, int dst_n, int64_t rows) {
    const int64_t n = rows * dst_n;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / dst_n;
        const int c = (int)(i - r * dst_n);
        const float v = c < src_n ? (float)src[r * src_n + c] : 0.f;
        dst[i] = (D)v;
    }
}
cudaError_t launch_states_cvt(const void *src, bool src_bf16, int src_n, void *dst, bool dst_bf16, int dst_n,
                              int64_t rows, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>((rows * dst_n + 255) / 256, 4096);
    using bf = __nv_bfloat16;
    if (src_bf16)   // widen into the fp32 copy
        k_states_cvt<bf, float><<<blocks, 256, 0, st>>>(static_cast<const bf *>(src), src_n, static_cast<float *>(dst),
                                                         dst_n, rows);
    else if (dst_bf16)
        k_states_cvt<float, bf><<<blocks, 256, 0, st>>>(static_cast<const float *>(src), src_n, static_cast<bf *>(dst),
                                                         dst_n, rows);
    else
        k_states_cvt<float, float><<<blocks, 256, 0, st>>>(static_cast<const float *>(src), src_n,
                                                            static_cast<float *>(dst), dst_n, rows);
    return cudaGetLastError();
}

}  // namespace ssd
