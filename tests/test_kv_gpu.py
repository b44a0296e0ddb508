"""isd_kv_commit (include/isd_kv.h) on the GPU against the oracle's KV commit.

The commit is integer bookkeeping, so the bar is bit-exactness: after every
commit the table, lengths, pending counts, in-flight counts, free stack, its
top and the status must equal the oracle's.  Both sides start from the same
seeded state and take the same accept lengths each step.  Cases: the
hand-worked commits of tests/golden/handworked_kv_commit.json, multi-step
runs over one tile and several tiles of 256 sequences (with a ragged last
tile), no masks (stride 1) and the largest stride, an empty batch, a large
batch, and refused commits (each error bit, the state left unchanged).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_verify_accept_02_b300 import isd_kv_commit
from speculative_verify_accept_02_b300.workloads import KVState, draw_accept_lengths, make_kv_state

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "handworked_kv_commit.json")


def _dev(state: KVState) -> dict:
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    return state.to_torch("cuda")


def _commit(dev: dict, accept, M: int) -> int:
    acc = torch.as_tensor(np.asarray(accept, np.int32), device="cuda")
    return int(isd_kv_commit(dev, acc, M).item())


def _both(ref: KVState, dev: dict, accept, M: int):
    want = oracle.kv_commit(ref, accept, M)
    got = _commit(dev, accept, M)
    assert got == want
    assert KVState.from_torch(dev).equal(ref)
    return got


def _state(d):
    a = lambda x: np.array(x, np.int32)
    return KVState(a(d["table"]), a(d["seq_len"]), a(d["pend"]), a(d["alloc"]), a(d["free_slots"]),
                   a([d["free_top"]]))


def test_handworked_commits():
    with open(GOLDEN) as f:
        g = json.load(f)
    st = _state(g["initial"])
    dev = _dev(st)
    for c in g["commits"]:
        before = KVState.from_torch(dev)
        assert _commit(dev, c["accept_len"], g["num_masks"]) == c["status"], c["name"]
        now = KVState.from_torch(dev)
        assert now.equal(before if c.get("unchanged") else _state(c)), c["name"]
    pc = g["pool_case"]
    dev = _dev(_state(pc))
    assert _commit(dev, pc["accept_len"], pc["num_masks"]) == pc["status"]
    assert KVState.from_torch(dev).equal(_state(pc))


def _run(C, M, steps, alpha, seed, start_max=8):
    rng = np.random.default_rng(seed)
    ld = start_max + steps * (M + 1) + 2 * M + 2
    ref = make_kv_state(C, ld, C * ld, rng.integers(0, start_max + 1, C), seed=seed)
    dev = _dev(ref)
    accept = np.zeros(C, np.int32)
    for _ in range(steps):
        assert _both(ref, dev, accept, M) == 0
        accept = draw_accept_lengths(rng, ref.pend, alpha)
    return ref, dev


@pytest.mark.parametrize("C,M,steps,alpha", [
    (64, 7, 30, 0.7),      # the c64 batch at stride 8
    (600, 3, 20, 0.5),     # three tiles of 256, the last one ragged
    (1, 0, 12, 0.5),       # stride 1: no masks, nothing ever pending
    (257, 31, 8, 0.9),     # the largest stride, one sequence past a tile
])
def test_random_runs(C, M, steps, alpha):
    _run(C, M, steps, alpha, seed=C * 100 + M)


def test_large_batch():
    """100,000 sequences in one launch (391 tiles), two commits."""
    _run(100_000, 7, 2, 0.6, seed=3, start_max=4)


def test_empty_batch():
    ref = make_kv_state(0, 16, 32, [], seed=1)
    dev = _dev(ref)
    assert _both(ref, dev, np.zeros(0, np.int32), 3) == 0
    assert int(KVState.from_torch(dev).free_top[0]) == 32


def test_refused_commits_change_nothing():
    """Each error bit, alone and combined, on a state mid-run: the status
    equals the oracle's and neither side changes anything."""
    ref, _ = _run(40, 3, 6, 0.6, seed=9)
    rng = np.random.default_rng(4)
    pend = ref.pend.copy()
    fused = np.flatnonzero(pend > 0)
    assert fused.size >= 2
    base_accept = draw_accept_lengths(rng, pend, 0.6)

    def check(mutate, accept=base_accept, expect=None):
        st = ref.copy()
        mutate(st)
        before = st.copy()
        dev = _dev(st)
        status = _both(st, dev, accept, 3)
        if status != 0:
            assert st.equal(before)
        if expect is not None:
            assert status == expect, status

    bad = base_accept.copy()
    bad[fused[0]] = pend[fused[0]] + 1
    check(lambda s: None, bad, expect=2)                                   # ACCEPT
    bad[fused[1]] = -1
    check(lambda s: None, bad, expect=2)

    def slot(s, v):
        i = int(fused[0])
        s.table[i, s.seq_len[i] + s.alloc[i] - 1] = v                         # a mask entry: always trimmed
    check(lambda s: slot(s, s.pool_size), expect=4)                       # SLOT
    check(lambda s: slot(s, -3), expect=4)

    def alloc_off(s):
        s.alloc[0] += 1
    check(alloc_off, expect=1)                                            # STATE
    check(lambda s: s.seq_len.__setitem__(1, -1), expect=1)

    def top_high(s):
        s.free_top[0] = s.pool_size + 1
    check(top_high, expect=1)

    def top_zero(s):
        s.free_top[0] = 0
    check(top_zero)                                      # POOL unless the trims cover the batch

    combo = base_accept.copy()
    combo[fused[0]] = -4
    check(lambda s: slot(s, s.pool_size + 7), combo, expect=2)            # ACCEPT stops that sequence's checks


def test_capacity_refusal():
    """Rows one entry short of the next allocation: CAPACITY, nothing changes."""
    M = 3
    ref = make_kv_state(3, 1 + 2 * M, 64, [0, 0, 0], seed=2)   # ld = 7
    dev = _dev(ref)
    assert _both(ref, dev, np.zeros(3, np.int32), M) == 0     # admission: 1 + 0 + 3 entries each
    before = ref.copy()
    # kept 1 -> length 1, then 1 + 3 + 3 = 7 entries -> 8 > 7
    assert _both(ref, dev, np.zeros(3, np.int32), M) == 16
    assert ref.equal(before)


@pytest.mark.parametrize("short", [1, 0])
def test_pool_refusal_across_tiles(short):
    """300 admitted sequences (two tiles) want 1 + 0 + 3 slots each: a pool
    one slot short is refused (POOL), an exact fit empties the stack."""
    M, C = 3, 300
    ref = make_kv_state(C, 16, C * (1 + M) - short, np.zeros(C), seed=6)
    before = ref.copy()
    dev = _dev(ref)
    status = _both(ref, dev, np.zeros(C, np.int32), M)
    if short:
        assert status == 8 and ref.equal(before)
    else:
        assert status == 0 and int(ref.free_top[0]) == 0
