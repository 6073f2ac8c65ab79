"""Plain-Python builder of the chunk and work-unit lists -- TEST INFRASTRUCTURE ONLY.

The bit-exact reference for the library's metadata kernel.  Definition (the
reading of packed variable-length sequences used throughout: each sequence is
an independent scan from its own initial state; the chunk grid restarts at every
sequence's first token, so no chunk mixes two sequences):

* sequence s = tokens [t0, t0+len) of batch row b  (fixed-length batch: s = b,
  t0 = 0, len = L; packed: b = 0, t0 = cu[s], len = cu[s+1] - cu[s]);
* its chunks are [t0 + c Q, t0 + min((c+1) Q, len)) for c = 0 .. ceil(len/Q)-1,
  listed sequence by sequence -> rows (seq, b, first token, length);
* its work units group consecutive chunks: a sequence of n chunks has
  m = max(ceil(n/R), min(n, ceil(n num/den))) units (num/den = 1/R unless given),
  unit j holding floor(n/m) chunks plus one more for j < n mod m, so unit j starts
  at chunk j floor(n/m) + min(j, n mod m); segments j are grouped in blocks of KB;
  units are listed by (block, s, j) -> rows (seq, b, first token, token count,
  chunk count, index of unit (s, j-1) or -1, 1 if last unit of s, j).
"""


def seg_count(n, R, num, den):
    if n <= 0:
        return 0
    return max(-(-n // R), min(n, -(-(n * num) // den)))


def build(cu=None, batch=1, seqlen=0, Q=64, R=1, KB=8, num=None, den=None):
    if num is None:
        num, den = 1, R
    if cu is None:
        seqs = [(b, 0, seqlen) for b in range(batch)]
    else:
        cu = [int(c) for c in cu]
        seqs = [(0, cu[s], cu[s + 1] - cu[s]) for s in range(len(cu) - 1)]
    chunks, chunk0 = [], []
    for s, (b, t0, n) in enumerate(seqs):
        chunk0.append(len(chunks))
        nch = -(-n // Q)
        for c in range(nch):
            chunks.append((s, b, t0 + c * Q, min(Q, n - c * Q)))
    units = []
    last = {}
    nseg = [seg_count(-(-n // Q), R, num, den) for (_, _, n) in seqs]
    maxseg = max(nseg) if nseg else 0
    for blk in range(-(-maxseg // KB)):
        for s, (b, t0, n) in enumerate(seqs):
            nch = -(-n // Q)
            for j in range(blk * KB, min((blk + 1) * KB, nseg[s])):
                base, rem = divmod(nch, nseg[s])
                c0 = j * base + min(j, rem)
                nc = base + (1 if j < rem else 0)
                units.append((s, b, t0 + c0 * Q, min(nc * Q, n - c0 * Q), nc,
                              last.get(s, -1) if j > 0 else -1, 1 if j == nseg[s] - 1 else 0, j))
                last[s] = len(units) - 1
    return dict(seqs=[(b, t0, n, chunk0[s]) for s, (b, t0, n) in enumerate(seqs)], chunks=chunks, units=units)
