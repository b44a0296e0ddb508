"""A model, in plain Python, of the running top-k lists of the filtered
path's selection kernel, checked against a sort on rows that stress it.

The kernel's algorithm: each warp keeps its 64 best (logit, id) pairs, two
per lane (lane j holds entries 2j and 2j+1), ranked by larger logit, then
lower id.  Each lane offers one element at a time; the warp inserts, in lane
order, every offer that beats its k-th entry, by counting the entries that
beat the offer and shifting the rest one place.  The unaligned head and the
tail of a row go through warp 0 the same way, and warp 0 finally merges the
other warps' lists, each of which is sorted, so a merge stops at the first
entry that does not beat the k-th.

Rows: random, ascending (every id inserts), descending, all equal, a few
distinct values (long ties), mostly -inf; heads of 0 and 3 ids; a row
shorter than k.  This pins the algorithm the kernel implements; the kernel
itself is checked against the oracle on the GPU.
"""
import numpy as np
import pytest

INT_MAX = 2**31 - 1
LANES, VEC, WARPS = 32, 8, 8


def beats(av, ai, bv, bi):
    return av > bv or (av == bv and ai < bi)


class WarpList:
    def __init__(self):
        self.v = [[-np.inf, -np.inf] for _ in range(LANES)]
        self.i = [[INT_MAX, INT_MAX] for _ in range(LANES)]

    def get(self, j):
        return self.v[j >> 1][j & 1], self.i[j >> 1][j & 1]

    def insert(self, cv, ci):
        pos = sum(beats(self.v[lane][e], self.i[lane][e], cv, ci) for lane in range(LANES) for e in (0, 1))
        old_v = [pair[:] for pair in self.v]
        old_i = [pair[:] for pair in self.i]
        for lane in range(LANES):
            e0, e1 = 2 * lane, 2 * lane + 1
            prev_v = old_v[lane - 1][1] if lane > 0 else old_v[lane][1]   # entry 2j - 1
            prev_i = old_i[lane - 1][1] if lane > 0 else old_i[lane][1]
            nv1, ni1 = old_v[lane][1], old_i[lane][1]
            if e1 > pos:
                nv1, ni1 = old_v[lane][0], old_i[lane][0]
            elif e1 == pos:
                nv1, ni1 = cv, ci
            nv0, ni0 = old_v[lane][0], old_i[lane][0]
            if e0 > pos:
                nv0, ni0 = prev_v, prev_i
            elif e0 == pos:
                nv0, ni0 = cv, ci
            self.v[lane] = [nv0, nv1]
            self.i[lane] = [ni0, ni1]


def offer(wl, cands, k, bar):
    """One offer per lane (None: no element); returns the new k-th entry."""
    tv, ti = bar
    flagged = [c is not None and beats(c[0], c[1], tv, ti) for c in cands]
    for lane, flag in enumerate(flagged):
        if flag and beats(cands[lane][0], cands[lane][1], tv, ti):
            wl.insert(*cands[lane])
            tv, ti = wl.get(k - 1)
    return tv, ti


def topk(row, k, head=0):
    V = len(row)
    nvec = (V - head) // VEC
    tail0 = head + nvec * VEC
    lists, bars = [], []
    for w in range(WARPS):
        wl, bar = WarpList(), (-np.inf, INT_MAX)
        for g0 in range(w * LANES, nvec, LANES * WARPS):
            for j in range(VEC):
                cands = [(row[head + g * VEC + j], head + g * VEC + j) if g < nvec else None
                         for g in range(g0, g0 + LANES)]
                bar = offer(wl, cands, k, bar)
        if w == 0:  # the head and the tail
            cands = []
            for lane in range(LANES):
                e = lane if lane < head else tail0 + (lane - head)
                has = lane < head or lane - head < V - tail0
                cands.append((row[e], e) if has else None)
            bar = offer(wl, cands, k, bar)
        lists.append(wl)
        bars.append(bar)
    wl, bar = lists[0], bars[0]
    for w in range(1, WARPS):
        for j in range(k):
            cv, ci = lists[w].get(j)
            if not beats(cv, ci, *bar):
                break
            wl.insert(cv, ci)
            bar = wl.get(k - 1)
    return [wl.get(j) for j in range(k)]


def ref(row, k):
    order = sorted(range(len(row)), key=lambda v: (-row[v], v))
    out = [(row[v], v) for v in order[:k]]
    return out + [(-np.inf, INT_MAX)] * (k - len(out))


def _rows():
    rng = np.random.default_rng(0)
    V = 700
    masked = rng.normal(size=V).astype(np.float32)
    masked[rng.choice(V, 500, replace=False)] = -np.inf
    return [("random", rng.normal(size=V).astype(np.float32)),
            ("ascending", np.arange(V, dtype=np.float32)),
            ("descending", -np.arange(V, dtype=np.float32)),
            ("all equal", np.zeros(V, np.float32)),
            ("few values", rng.integers(0, 3, V).astype(np.float32)),
            ("many -inf", masked)]


@pytest.mark.parametrize("name,row", _rows(), ids=[r[0] for r in _rows()])
@pytest.mark.parametrize("k", [1, 50, 64])
def test_lists_give_the_exact_top_k(name, row, k):
    for head in (0, 3):
        assert topk(list(row), k, head=head) == ref(list(row), k)


def test_rows_shorter_than_k():
    small = list(np.random.default_rng(1).normal(size=40).astype(np.float32))
    assert topk(small, 40, head=5) == ref(small, 40)
