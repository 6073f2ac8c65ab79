"""Sequence index and chunk segment lists of packed sequences -- TEST INFRASTRUCTURE ONLY.

The integer metadata of a packed (cu_seqlens) batch, written out by definition
with plain loops over tokens; it shares nothing with the CUDA path.

Definition (the continuous-batching workload of the source pages: the packed
THD path of the Helion pull request, section "Testing", and the cont-batch
tests of the vLLM pull request, section "Test Plan"; sequences are packed on
one token axis and the chunk grid runs over that axis, so chunk boundaries
need not fall on sequence starts):

* sequence s holds tokens [cu[s], cu[s+1]) of the packed axis (empty when
  cu[s] == cu[s+1]); cu[0] = 0, cu is non-decreasing, cu[S] = L;
* seq_idx[t] = the s with cu[s] <= t < cu[s+1], for every token t in [0, L);
* physical chunk c holds tokens [c Q, min((c+1) Q, L)), c = 0 .. ceil(L/Q) - 1;
* a segment of chunk c is a maximal run of its tokens with one seq_idx value:
  (seq, first token, one past the last token), in token order.

Every token lies in exactly one segment; a chunk that spans several sequences
has several segments.  ``segments`` lists them chunk by chunk (which is also
sequence by sequence), and ``chunk_begin[c]`` is the index of chunk c's first
segment (``chunk_begin[n_chunks]`` = the number of segments).

Parity: pinned by the hand-worked lists in ``tests/golden/varlen_segments.txt``
(a chunk covering three sequences, empty sequences at both ends and inside, a
sequence shorter than a chunk, sequences starting exactly on a chunk boundary),
checked in ``tests/test_varlen_meta_cpu.py``.
"""


def seq_idx(cu):
    """seq_idx[t] for t in [0, cu[-1]): walk the sequences, write each one's index
    over its tokens."""
    cu = [int(c) for c in cu]
    out = [None] * cu[-1]
    for s in range(len(cu) - 1):
        for t in range(cu[s], cu[s + 1]):
            out[t] = s
    assert all(v is not None for v in out), "cu_seqlens must cover every token"
    return out


def segments(cu, Q):
    """(segments, chunk_begin): the segments of every physical chunk of length Q."""
    idx = seq_idx(cu)
    L = len(idx)
    n_chunks = -(-L // Q)
    segs, begin = [], []
    for c in range(n_chunks):
        begin.append(len(segs))
        lo, hi = c * Q, min((c + 1) * Q, L)
        start = lo
        for t in range(lo + 1, hi + 1):
            if t == hi or idx[t] != idx[start]:
                segs.append((idx[start], start, t))
                start = t
    begin.append(len(segs))
    return segs, begin
