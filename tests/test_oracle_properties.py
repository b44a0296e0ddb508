"""Properties of the oracle's KV commit and sampling filters over generated
inputs (hypothesis), beyond the hand-worked pins:

- KV commit (Summary §3.3, kept prefix and next step from §3.2): on success
  every pool slot is free or referenced exactly once, each row is dense up to
  its in-flight entries, the kept count is 1 + a (1 for a proposal-only step,
  0 at admission) and the next in-flight count is 1 + L' + M; on refusal
  nothing changes.
- Filters (experiments §4.1): the filtered row is a distribution on at most
  top_k ids, those ids are the most probable ones, a larger top_p never
  keeps fewer ids, and top_p = 1 with top_k >= V is the plain softmax.
"""
import numpy as np
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st
from scipy.special import softmax as sp_softmax

import oracle
from speculative_verify_accept_02_b300.workloads import draw_accept_lengths, make_kv_state

SETTINGS = settings(max_examples=60, deadline=None, suppress_health_check=[HealthCheck.too_slow])


def _live(state):
    used = []
    for i in range(state.num_seqs):
        n = int(state.seq_len[i] + state.alloc[i])
        row = state.table[i]
        assert np.all(row[n:] == -1)
        used += list(row[:n])
    return used


@SETTINGS
@given(C=st.integers(1, 12), M=st.integers(0, 7), steps=st.integers(1, 8), alpha=st.floats(0.0, 1.0),
       seed=st.integers(0, 2**16), spare=st.integers(0, 40))
def test_kv_commit_invariants(C, M, steps, alpha, seed, spare):
    rng = np.random.default_rng(seed)
    committed = rng.integers(0, 4, C)
    ld = 4 + steps * (M + 1) + 2 * M + 2
    pool = int(committed.sum()) + C * (2 * M + 1) + spare   # may run short: refusals are checked too
    st_ = make_kv_state(C, ld, pool, committed, seed=seed)
    accept = np.zeros(C, np.int32)
    for _ in range(steps):
        before = st_.copy()
        status = oracle.kv_commit(st_, accept, M)
        if status:
            assert st_.equal(before)
            assert status in (8, 16, 24)  # POOL or CAPACITY: the inputs are otherwise well formed
            return
        for i in range(C):
            w, L = int(before.alloc[i]), int(before.pend[i])
            kept = 0 if w == 0 else 1 + (int(accept[i]) if L > 0 else 0)
            assert st_.seq_len[i] == before.seq_len[i] + kept
            assert st_.alloc[i] == 1 + st_.pend[i] + M
            assert np.array_equal(st_.table[i, :before.seq_len[i] + kept], before.table[i, :before.seq_len[i] + kept])
        free = list(st_.free_slots[:int(st_.free_top[0])])
        assert sorted(_live(st_) + free) == list(range(pool))
        accept = draw_accept_lengths(rng, st_.pend, alpha)


@SETTINGS
@given(V=st.integers(1, 60), k=st.integers(0, 70), top_p=st.floats(0.01, 1.0), T=st.floats(0.2, 3.0),
       seed=st.integers(0, 2**16))
def test_filter_properties(V, k, top_p, T, seed):
    z = np.random.default_rng(seed).normal(0, 2, V)
    w = oracle.filtered_probs(z, T, k, top_p)
    kept = np.flatnonzero(w > 0)
    assert abs(w.sum() - 1.0) < 1e-12
    assert kept.size <= (k if 0 < k < V else V)
    # the kept ids are the most probable ones
    if kept.size < V:
        assert z[kept].min() >= np.delete(z, kept).max()
    wider = oracle.filtered_probs(z, T, k, min(1.0, top_p + 0.1))
    assert np.count_nonzero(wider > 0) >= kept.size
    if k == 0 or k >= V:
        full = oracle.filtered_probs(z, T, k, 1.0)
        assert np.allclose(full, sp_softmax(z / T), atol=1e-14)


@SETTINGS
@given(C=st.integers(1, 6), V=st.integers(2, 40), Lmax=st.integers(1, 6), T=st.sampled_from([0.0, 0.5, 1.0, 2.0]),
       seed=st.integers(0, 2**16), same=st.booleans())
def test_verify_structure(C, V, Lmax, T, seed, same):
    """Per sequence: 0 <= a <= L; the emitted slots are x_1..x_a, one token,
    then -1; ratios in [0, 1] with alpha their mean; q == p accepts every
    proposal; at T = 0 a is the count of leading argmax proposals and the
    token is the argmax of p_{a+1}."""
    rng = np.random.default_rng(seed)
    Ls = rng.integers(1, Lmax + 1, C)
    offs = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    total = int(offs[-1])
    P = rng.normal(0, 2, (total + C, V)).astype(np.float32)
    Q = np.empty((total, V), np.float32)
    for i in range(C):
        for k in range(Ls[i]):
            Q[offs[i] + k] = P[offs[i] + i + k] if same else rng.normal(0, 2, V)
    toks = rng.integers(0, V, total).astype(np.int32)
    out = oracle.verify(P, Q, V, toks, offs, np.full(C, T, np.float32), seed, 3)
    for i in range(C):
        s, L = int(offs[i]), int(Ls[i])
        a = int(out["accept_len"][i])
        r = out["ratio"][s:s + L]
        slots = out["out_tokens"][s + i:s + i + L + 1]
        assert 0 <= a <= L
        assert np.array_equal(slots[:a], toks[s:s + a]) and 0 <= slots[a] < V and np.all(slots[a + 1:] == -1)
        assert np.all((r >= 0) & (r <= 1)) and abs(out["alpha"][i] - r.mean()) < 1e-12
        if same and T > 0:
            assert a == L
        if T == 0.0:
            hits = [toks[s + k] == int(np.argmax(P[s + i + k])) for k in range(L)]
            want_a = hits.index(False) if False in hits else L
            assert a == want_a and slots[a] == int(np.argmax(P[s + i + a]))
