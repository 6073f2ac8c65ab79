"""The library's work lists restated in Python -- a SCHEDULER SELF-CONSISTENCY CHECK.

This module is not part of the oracle and defines nothing about the scan: it
restates, in plain Python, how the library lays its chunk tiles and fused-forward
work units out in the workspace, so that tests can compare the device-built lists
with a second implementation of the same scheduling rules.  What a chunk IS (the
sequence index of every token and each physical chunk's segments, by definition)
comes from ``oracle.varlen_meta``; this module only renumbers those segments into
the library's tile records and groups them into units.

Chunk tiles (one per segment of a physical chunk, sequence by sequence):
  (seq, batch row, first token of the physical chunk t0, end - t0, start - t0),
  i.e. tile rows [lo, len) of the Q-row tile starting at t0 belong to the segment.
  Fixed-length batch: row b is sequence b, its chunks [cQ, min((c+1)Q, L)).
Work units group consecutive tiles of one sequence: a sequence of n tiles has
m = max(ceil(n/R), min(n, ceil(n num/den))) units (num/den = 1/R unless given),
unit j holding floor(n/m) tiles plus one more for j < n mod m; units are grouped
in blocks of KB and listed by (block, sequence, j) -> rows (seq, batch row, t0 of
its first tile, end of the sequence's tokens - t0 capped at its tiles, tile count,
index of unit (s, j-1) or -1, j, 1 if last unit of s, leading rows lo of its first
tile).

decode_chunks / decode_units turn the library's raw records (16 and 32 bytes: the
last int32 word of each holds two int16 fields, low half first) into those tuples.
"""
import numpy as np


def decode_chunks(raw_bytes, n):
    a = np.frombuffer(raw_bytes[:16 * n].tobytes(), dtype=np.int32).reshape(n, 4)
    h = np.frombuffer(raw_bytes[:16 * n].tobytes(), dtype=np.int16).reshape(n, 8)
    return [(int(r[0]), int(r[1]), int(r[2]), int(q[6]), int(q[7])) for r, q in zip(a, h)]


def decode_units(raw_bytes, n):
    a = np.frombuffer(raw_bytes[:32 * n].tobytes(), dtype=np.int32).reshape(n, 8)
    h = np.frombuffer(raw_bytes[:32 * n].tobytes(), dtype=np.int16).reshape(n, 16)
    return [tuple(int(v) for v in r[:7]) + (int(q[14]), int(q[15])) for r, q in zip(a, h)]
from oracle import varlen_meta


def seg_count(n, R, num, den):
    if n <= 0:
        return 0
    return max(-(-n // R), min(n, -(-(n * num) // den)))


def build(cu=None, batch=1, seqlen=0, Q=64, R=1, KB=8, num=None, den=None):
    if num is None:
        num, den = 1, R
    chunks = []
    if cu is None:
        seqs = [(b, 0, seqlen) for b in range(batch)]
        for b in range(batch):
            for c in range(-(-seqlen // Q)):
                chunks.append((b, b, c * Q, min(Q, seqlen - c * Q), 0))
    else:
        cu = [int(c) for c in cu]
        seqs = [(0, cu[s], cu[s + 1] - cu[s]) for s in range(len(cu) - 1)]
        segs, _ = varlen_meta.segments(cu, Q)
        for (s, a, e) in segs:
            t0 = (a // Q) * Q
            chunks.append((s, 0, t0, e - t0, a - t0))
    nch = [sum(1 for ch in chunks if ch[0] == s) for s in range(len(seqs))]
    chunk0, k = [], 0
    for s in range(len(seqs)):
        chunk0.append(k)
        k += nch[s]
    units = []
    last = {}
    nseg = [seg_count(n, R, num, den) for n in nch]
    maxseg = max(nseg) if nseg else 0
    for blk in range(-(-maxseg // KB)):
        for s, (b, t0, n) in enumerate(seqs):
            for j in range(blk * KB, min((blk + 1) * KB, nseg[s])):
                base, rem = divmod(nch[s], nseg[s])
                c0 = j * base + min(j, rem)
                nc = base + (1 if j < rem else 0)
                first = chunks[chunk0[s] + c0]
                ut0 = first[2]
                units.append((s, b, ut0, min(nc * Q, t0 + n - ut0), nc,
                              last.get(s, -1) if j > 0 else -1, j, 1 if j == nseg[s] - 1 else 0, first[4]))
                last[s] = len(units) - 1
    return dict(seqs=[(b, t0, n, chunk0[s]) for s, (b, t0, n) in enumerate(seqs)], chunks=chunks, units=units)
