"""Pins of the packed-sequence metadata oracle (sequence index of every token and the
segments of every physical chunk), on the CPU: hand-worked lists, and invariants that
any correct segmentation satisfies whatever the lengths."""
import os

import numpy as np
import pytest

from oracle import varlen_meta

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "varlen_segments.txt")


def golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "Q":
            cur = {"Q": int(vals[0])}
            cases.append(cur)
        elif key == "segments":
            cur[key] = [tuple(int(v) for v in s.split(":")) for s in vals]
        else:
            cur[key] = [int(v) for v in vals]
    return cases


@pytest.mark.parametrize("case", golden_cases(), ids=lambda c: "Q%d_cu%s" % (c["Q"], "_".join(map(str, c["cu"]))))
def test_hand_worked_lists(case):
    assert varlen_meta.seq_idx(case["cu"]) == case["seq_idx"]
    segs, begin = varlen_meta.segments(case["cu"], case["Q"])
    assert segs == case["segments"]
    assert begin == case["chunk_begin"]


def random_cu(rng, S, maxlen, p_empty=0.2):
    lens = [0 if rng.random() < p_empty else int(rng.integers(1, maxlen + 1)) for _ in range(S)]
    return [0] + list(np.cumsum(lens)), lens


@pytest.mark.parametrize("seed", range(20))
def test_segmentation_invariants(seed):
    """Every token lies in exactly one segment of its own chunk; a segment's tokens share one
    sequence; the segment count is the chunk count plus one per non-empty sequence that
    starts off the chunk grid; seq_idx agrees with a search of cu."""
    rng = np.random.default_rng(seed)
    Q = int(rng.choice([1, 2, 4, 16, 64, 128]))
    cu, lens = random_cu(rng, int(rng.integers(1, 12)), int(rng.integers(1, 300)))
    L = cu[-1]
    if L == 0:
        return
    idx = varlen_meta.seq_idx(cu)
    assert idx == [int(np.searchsorted(cu, t, side="right")) - 1 for t in range(L)]
    segs, begin = varlen_meta.segments(cu, Q)
    cover = np.zeros(L, np.int64)
    for c in range(len(begin) - 1):
        for (s, a, e) in segs[begin[c]:begin[c + 1]]:
            assert c * Q <= a < e <= min((c + 1) * Q, L)
            assert cu[s] <= a and e <= cu[s + 1]
            cover[a:e] += 1
    assert (cover == 1).all()
    n_chunks = -(-L // Q)
    assert len(begin) == n_chunks + 1
    off_grid = sum(1 for s in range(len(lens)) if lens[s] > 0 and cu[s] % Q != 0)
    assert len(segs) == n_chunks + off_grid
    # consecutive segments of one chunk belong to different sequences (maximal runs)
    for c in range(n_chunks):
        ss = [s for (s, _, _) in segs[begin[c]:begin[c + 1]]]
        assert ss == sorted(set(ss))
