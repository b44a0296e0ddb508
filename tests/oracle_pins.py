"""Pins of the fp64 oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  tests/test_oracle_pins.py runs them on the oracle; the mutation
tests run them on builds of the oracle with a planted mistake and require
that some pin fails for every mistake.

Sources: "Introspective Diffusion Language Models | Summary" — §2 (alpha),
§3.2 (strict acceptance, residual correction, bonus token, and the claim
that acceptance plus correction keeps the anchor distribution), §3.3 (argmax
proposals with strict verification), §3.1 (next-token shift).  Philox4x64-10
from Salmon et al., SC'11, checked against numpy's implementation.
"""
import itertools
import json
import math
import os

import numpy as np
from scipy.special import log_softmax as sp_log_softmax
from scipy.special import softmax as sp_softmax
from scipy.stats import chi2

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")

TAG_ACCEPT, TAG_CORRECT, TAG_BONUS, TAG_PROPOSE = 0, 1, 2, 3


def _bf16_bits(x):
    """float32 -> bfloat16 bit patterns (round to nearest even) via torch."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _bf16_values(bits):
    import torch
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def _chi2_ok(counts, probs, alpha=1e-6):
    """Pearson goodness of fit; passes unless the p-value is below alpha."""
    counts = np.asarray(counts, np.float64)
    n = counts.sum()
    exp = n * np.asarray(probs, np.float64)
    keep = exp > 0
    assert np.all(counts[~keep] == 0), "mass on an impossible outcome"
    stat = np.sum((counts[keep] - exp[keep]) ** 2 / exp[keep])
    dof = max(int(keep.sum()) - 1, 1)
    return chi2.sf(stat, dof) > alpha


# ---------------------------------------------------------------------------
# Generator
# ---------------------------------------------------------------------------

def pin_philox_numpy(orc):
    """Philox4x64-10 equals numpy.random.Philox, which increments the
    256-bit counter before each block: set it to c - 1 to get block c."""
    rng = np.random.default_rng(7)
    for _ in range(24):
        ctr = rng.integers(1, 2**63, size=4, dtype=np.uint64)
        key = rng.integers(0, 2**63, size=2, dtype=np.uint64)
        ref = np.random.Philox(counter=np.array([ctr[0] - np.uint64(1), ctr[1], ctr[2], ctr[3]],
                                                dtype=np.uint64), key=key).random_raw(4)
        got = orc.philox4x64_10(ctr, key)
        assert np.array_equal(ref.astype(np.uint64), got), (ctr, key, ref, got)
    # Small counters, the ones the library uses.
    for ctr in ([1, 0, 0, 0], [1, 3, 5, 2], [9, 63, 1, 3]):
        c = np.array(ctr, dtype=np.uint64)
        ref = np.random.Philox(counter=np.array([c[0] - 1, c[1], c[2], c[3]], np.uint64),
                               key=np.array([0, 0], np.uint64)).random_raw(4)
        assert np.array_equal(ref.astype(np.uint64), orc.philox4x64_10(c, [0, 0]))


def pin_uniform_layout(orc):
    """u(seed, offset, i, k, tag) is the top 24 bits of word 0 of the block at
    counter (offset, i, k, tag) under key (seed, 0), scaled by 2^-24."""
    rng = np.random.default_rng(11)
    for _ in range(16):
        seed, offset = (int(v) for v in rng.integers(0, 2**40, size=2))
        i, k, tag = int(rng.integers(0, 4096)), int(rng.integers(1, 33)), int(rng.integers(0, 4))
        offset += 1
        word0 = np.random.Philox(counter=np.array([offset - 1, i, k, tag], np.uint64),
                                 key=np.array([seed, 0], np.uint64)).random_raw(1)[0]
        expect = float(int(word0) >> 40) / 2.0**24
        assert orc.uniform(seed, offset, i, k, tag) == expect
    # Uniformity and the grid: 65536 draws over 64 equal bins.
    us = np.array([orc.uniform(3, off, 1, 2, TAG_ACCEPT) for off in range(65536)])
    assert us.min() >= 0.0 and us.max() < 1.0
    assert np.all(us * 2**24 == np.floor(us * 2**24))
    counts = np.bincount((us * 64).astype(int), minlength=64)
    assert _chi2_ok(counts, np.full(64, 1 / 64))


# ---------------------------------------------------------------------------
# Row-level definitions
# ---------------------------------------------------------------------------

def pin_softmax_library(orc):
    """softmax and log-softmax of logits/T equal scipy's routines."""
    rng = np.random.default_rng(5)
    for V, T in ((7, 1.0), (300, 0.6), (1000, 2.5), (64, 0.05)):
        z = rng.normal(0, 3, V)
        ref = sp_softmax(z / T)
        assert np.allclose(orc.softmax(z, T), ref, rtol=1e-13, atol=1e-300)
        lref = sp_log_softmax(z / T)
        for x in (0, V // 2, V - 1, int(np.argmin(z))):
            assert abs(orc.log_softmax_at(z, T, x) - lref[x]) <= 1e-12 * max(1, abs(lref[x]))


def pin_temperature_ratio(orc):
    """With logits T*log(pi), softmax(logits/T) = pi, so the ratio of x is
    min(1, pi_p(x)/pi_q(x)) at every temperature (§3.2)."""
    rng = np.random.default_rng(6)
    for T in (0.3, 0.7, 1.0, 1.9):
        for _ in range(10):
            V = int(rng.integers(2, 40))
            pp = rng.dirichlet(np.ones(V))
            qq = rng.dirichlet(np.ones(V))
            x = int(rng.integers(0, V))
            want = min(1.0, pp[x] / qq[x])
            got = orc.ratio(T * np.log(pp), T * np.log(qq), T, x)
            assert abs(got - want) <= 1e-12 * max(want, 1e-300) + 1e-15, (T, got, want)


def pin_tv_identity(orc):
    """E_{x~q}[min(1, p(x)/q(x))] = sum_v min(p_v, q_v) = 1 - TV(p, q)."""
    rng = np.random.default_rng(8)
    for T in (0.5, 1.0, 2.0):
        V = 50
        P, Q = rng.normal(0, 2, V), rng.normal(0, 2, V)
        p, q = sp_softmax(P / T), sp_softmax(Q / T)
        lhs = sum(q[x] * orc.ratio(P, Q, T, x) for x in range(V))
        rhs = np.minimum(p, q).sum()
        assert abs(lhs - rhs) < 1e-12, (T, lhs, rhs)


def pin_residual_known(orc):
    """w = max(0, p - q) (§3.2) on hand-picked distributions; all-zero w
    (q == p) falls back to p."""
    p = np.array([0.1, 0.4, 0.2, 0.3])
    q = np.array([0.3, 0.1, 0.5, 0.1])
    w = orc.residual(np.log(p), np.log(q), 1.0)
    assert np.allclose(w, [0.0, 0.3, 0.0, 0.2], atol=1e-15)
    w = orc.residual(1.5 * np.log(p), 1.5 * np.log(q), 1.5)
    assert np.allclose(w, [0.0, 0.3, 0.0, 0.2], atol=1e-15)
    w = orc.residual(np.log(p), np.log(p), 1.0)
    assert np.allclose(w, p, atol=1e-15)


def pin_icdf_grid(orc):
    """Inverse CDF over the grid u = n/2^16 with dyadic weights: each id is
    hit exactly 2^16 * w_v / S times; zero weights never; ties at interval
    ends go up (smallest v with C(v) > t)."""
    w = np.array([1, 3, 0, 4, 0, 8], dtype=np.float64) / 16.0
    n = 1 << 16
    counts = np.zeros(w.size, dtype=np.int64)
    for j in range(n):
        v, m = orc.icdf(w, j / n)
        counts[v] += 1
        assert m >= 0.0
    assert np.array_equal(counts, (w / w.sum() * n).astype(np.int64)), counts
    assert orc.icdf(w, 1 / 16)[0] == 1          # t = C(0) -> next id
    assert orc.icdf(w, 1 / 16)[1] == 0.0
    assert orc.icdf(w, 0.0)[0] == 0
    assert orc.icdf(np.array([0.0, 0.0, 2.0]), 0.0)[0] == 2
    v, m = orc.icdf(w, 0.25 + 1 / 64)            # inside id 3's interval [4/16, 8/16)
    assert v == 3 and abs(m - 1 / 64) < 1e-15


def pin_handworked(orc):
    """The worked cases in tests/golden/handworked_verify.json."""
    with open(os.path.join(GOLDEN, "handworked_verify.json")) as f:
        g = json.load(f)
    pp, qq = np.array(g["probs_p"]), np.array(g["probs_q"])
    for case in g["cases"]:
        T = case["T"]
        scale = T if T > 0 else 1.0
        r = orc.verify_one(scale * np.log(pp), scale * np.log(qq), T, case["x"], case["u_accept"],
                           case["u_correct"], case["u_bonus"])
        assert r["accept_len"] == case["accept_len"], (case["name"], r)
        assert list(r["out_tokens"]) == case["out_tokens"], (case["name"], r)
        assert np.allclose(r["ratio"], case["ratio"], rtol=1e-12, atol=1e-15), (case["name"], r)
        assert abs(r["alpha"] - case["alpha"]) < 1e-12, (case["name"], r)
        if "accept_margin" in case:
            assert np.allclose(r["accept_margin"], case["accept_margin"], atol=1e-12)


def pin_greedy_planted(orc):
    """T = 0 (§3.3): a = number of leading positions whose token is the
    lowest-id argmax of p_k; the next token is the argmax of p_{a+1} (or of
    the final anchor).  Planted maxima, with ties, across a packed batch, so
    the next-token-shifted row layout is pinned too."""
    rng = np.random.default_rng(12)
    V = 97
    Ls = [3, 1, 5, 2, 4]
    C = len(Ls)
    offs = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    total = int(offs[-1])
    P = rng.normal(0, 1, (total + C, V)).astype(np.float32)
    Q = rng.normal(0, 1, (total, V)).astype(np.float32)
    planted = rng.integers(0, V - 1, total + C)
    for r, v in enumerate(planted):
        P[r, v] = 9.0
        P[r, v + 1] = 9.0 if r % 2 else 8.5   # ties on odd rows: lowest id wins
    tokens = np.zeros(total, np.int32)
    expect_a = []
    for i, L in enumerate(Ls):
        reject_at = [None, 1, 4, None, 2][i]  # 1-based position that is wrong, or None
        for k in range(1, L + 1):
            prow = offs[i] + i + k - 1
            good = planted[prow]
            tokens[offs[i] + k - 1] = good if (reject_at is None or k < reject_at) else (good + 1)
        expect_a.append(L if reject_at is None else reject_at - 1)
    out = orc.verify(P, Q, V, tokens, offs, np.zeros(C, np.float32), 0, 0)
    assert list(out["accept_len"]) == expect_a, (out["accept_len"], expect_a)
    for i, L in enumerate(Ls):
        a = expect_a[i]
        slots = out["out_tokens"][offs[i] + i: offs[i] + i + L + 1]
        assert list(slots[:a]) == list(tokens[offs[i]: offs[i] + a])
        assert slots[a] == planted[offs[i] + i + a]       # argmax of p_{a+1}
        assert all(s == -1 for s in slots[a + 1:])
        assert abs(out["alpha"][i] - sum(out["ratio"][offs[i]:offs[i] + L]) / L) < 1e-15


def pin_p_equals_q(orc):
    """q bitwise equal to p gives ratio 1 exactly, so every proposal is
    accepted for every uniform (the all-accept invariant of §3.2)."""
    rng = np.random.default_rng(13)
    V, Ls = 300, [4, 8, 1, 16, 3]
    C = len(Ls)
    offs = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    total = int(offs[-1])
    P = _bf16_bits(rng.normal(0, 1, (total + C, V)))
    Q = np.empty((total, V), np.uint16)
    for i, L in enumerate(Ls):
        Q[offs[i]:offs[i] + L] = P[offs[i] + i: offs[i] + i + L]
    tokens = rng.integers(0, V, total).astype(np.int32)
    for T in (0.6, 1.0, 1.7):
        for off in range(5):
            out = orc.verify(P, Q, V, tokens, offs, np.full(C, T, np.float32), 9, off)
            assert np.all(out["ratio"] == 1.0)
            assert list(out["accept_len"]) == Ls
            assert np.all(out["alpha"] == 1.0)


def pin_lossless_enumeration(orc):
    """§3.2: acceptance plus correction keeps the anchor distribution.  Exact
    enumeration over every proposal tuple and accept/reject branch with
    prefix-dependent tables p(.|prefix), q(.|prefix): the k-th emitted token,
    given the emitted prefix and that at least k tokens are emitted, follows
    p(.|prefix) (speculative sampling, Leviathan et al. 2022; Chen et al. 2023)."""
    rng = np.random.default_rng(14)
    for V, L, T in ((4, 3, 1.0), (3, 2, 0.7), (5, 2, 1.4)):
        Pt, Qt = {}, {}
        for n in range(L + 1):
            for pre in itertools.product(range(V), repeat=n):
                Pt[pre] = rng.normal(0, 1.5, V)
                if n < L:
                    Qt[pre] = rng.normal(0, 1.5, V)
        law = {}
        for xs in itertools.product(range(V), repeat=L):
            wq = 1.0
            for k in range(L):
                wq *= sp_softmax(Qt[xs[:k]] / T)[xs[k]]
            ratios = [orc.ratio(Pt[xs[:k]], Qt[xs[:k]], T, xs[k]) for k in range(L)]
            reach = 1.0
            for a in range(L + 1):
                if a < L:
                    pa = reach * (1.0 - ratios[a])
                    w = orc.residual(Pt[xs[:a]], Qt[xs[:a]], T)
                else:
                    pa = reach
                    w = orc.softmax(Pt[xs], T)
                w = w / w.sum()
                for v in range(V):
                    key = xs[:a] + (v,)
                    law[key] = law.get(key, 0.0) + wq * pa * w[v]
                if a < L:
                    reach *= ratios[a]
        # Conditional law of the k-th emitted token.
        for pre, ptab in Pt.items():
            p = sp_softmax(ptab / T)
            mass = np.array([sum(m for e, m in law.items()
                                 if len(e) > len(pre) and e[:len(pre) + 1] == pre + (v,))
                             for v in range(V)])
            if mass.sum() <= 1e-14:
                continue
            assert np.allclose(mass / mass.sum(), p, atol=1e-12), (V, L, T, pre)
        first = np.array([sum(m for e, m in law.items() if e[0] == v) for v in range(V)])
        assert np.allclose(first, sp_softmax(Pt[()] / T), atol=1e-12)


# ---------------------------------------------------------------------------
# Batched, Philox-driven entry points
# ---------------------------------------------------------------------------

def pin_mc_verify_law(orc):
    """The batched verify draws its uniforms per sequence: many copies of one
    tiny sequence give accept lengths and emitted tokens with the exact law
    (chi-square), including the correction and bonus draws."""
    V, L, T = 3, 2, 1.0
    pp = [np.array([0.5, 0.3, 0.2]), np.array([0.2, 0.2, 0.6]), np.array([0.1, 0.6, 0.3])]
    qq = [np.array([0.2, 0.5, 0.3]), np.array([0.5, 0.1, 0.4])]
    x = [1, 0]
    C = 40000
    P = np.tile(np.log(np.stack(pp)).astype(np.float32), (C, 1))
    Q = np.tile(np.log(np.stack(qq)).astype(np.float32), (C, 1))
    offs = (np.arange(C + 1) * L).astype(np.int32)
    tokens = np.tile(np.array(x, np.int32), C)
    pf = np.log(np.stack(pp)).astype(np.float32).astype(np.float64)
    qf = np.log(np.stack(qq)).astype(np.float32).astype(np.float64)
    pr = [sp_softmax(r) for r in pf]
    qr = [sp_softmax(r) for r in qf]
    r1 = min(1, pr[0][1] / qr[0][1])
    r2 = min(1, pr[1][0] / qr[1][0])
    out = orc.verify(P, Q, V, tokens, offs, np.full(C, T, np.float32), 1234, 5)
    a = out["accept_len"]
    last = out["out_tokens"].reshape(C, L + 1)[np.arange(C), a]
    w1 = np.maximum(pr[0] - qr[0], 0); w1 /= w1.sum()
    w2 = np.maximum(pr[1] - qr[1], 0); w2 /= w2.sum()
    # Joint law of (a, emitted token) over 3 x V outcomes.
    probs = np.concatenate([(1 - r1) * w1, r1 * (1 - r2) * w2, r1 * r2 * pr[2]])
    counts = np.bincount(a * V + last, minlength=3 * V)
    assert _chi2_ok(counts, probs), (counts, probs * C)
    # With the proposals drawn from q, the first emitted token follows p_1
    # (the losslessness claim, sampled).
    rng = np.random.default_rng(16)
    xs = np.stack([rng.choice(V, size=C, p=qr[0]), rng.choice(V, size=C, p=qr[1])], axis=1)
    out = orc.verify(P, Q, V, xs.reshape(-1).astype(np.int32), offs, np.full(C, T, np.float32),
                     99, 0)
    first = out["out_tokens"].reshape(C, L + 1)[:, 0]
    assert _chi2_ok(np.bincount(first, minlength=V), pr[0])


def pin_relaxed_law(orc):
    """Relaxed acceptance (the pages' Table 4 ablation: the ratio multiplied by
    1 + tau): many copies of one tiny sequence give (accept length, emitted
    token) with the exact law when every accept test uses
    min(1, (1 + tau) p/q) and the correction stays normalize(max(0, p - q));
    the reported ratios stay min(1, p/q).  The first ratio is below 1 even
    relaxed, the second is clipped to 1 by the relaxation."""
    V, L, T, tau = 3, 2, 1.0, 0.5
    pp = [np.array([0.5, 0.3, 0.2]), np.array([0.4, 0.2, 0.4]), np.array([0.1, 0.6, 0.3])]
    qq = [np.array([0.2, 0.5, 0.3]), np.array([0.5, 0.1, 0.4])]
    x = [1, 0]
    C = 40000
    P = np.tile(np.log(np.stack(pp)).astype(np.float32), (C, 1))
    Q = np.tile(np.log(np.stack(qq)).astype(np.float32), (C, 1))
    offs = (np.arange(C + 1) * L).astype(np.int32)
    tokens = np.tile(np.array(x, np.int32), C)
    pr = [sp_softmax(r) for r in np.log(np.stack(pp)).astype(np.float32).astype(np.float64)]
    qr = [sp_softmax(r) for r in np.log(np.stack(qq)).astype(np.float32).astype(np.float64)]
    s1, s2 = pr[0][1] / qr[0][1], pr[1][0] / qr[1][0]
    r1, r2 = min(1, (1 + tau) * s1), min(1, (1 + tau) * s2)
    assert r1 < 1 and r2 == 1 and s2 < 1
    out = orc.verify(P, Q, V, tokens, offs, np.full(C, T, np.float32), 77, 2, tau=tau)
    a = out["accept_len"]
    last = out["out_tokens"].reshape(C, L + 1)[np.arange(C), a]
    w1 = np.maximum(pr[0] - qr[0], 0); w1 /= w1.sum()
    w2 = np.maximum(pr[1] - qr[1], 0); w2 /= w2.sum()
    probs = np.concatenate([(1 - r1) * w1, r1 * (1 - r2) * w2, r1 * r2 * pr[2]])
    counts = np.bincount(a * V + last, minlength=3 * V)
    assert _chi2_ok(counts, probs), (counts, probs * C)
    assert np.allclose(out["ratio"].reshape(C, L)[0], [s1, s2], rtol=1e-6)
    # tau = 0 is the strict step, bit for bit.
    strict = orc.verify(P[:200 * (L + 1)], Q[:200 * L], V, tokens[:200 * L], offs[:201],
                        np.full(200, T, np.float32), 77, 2)
    relaxed0 = orc.verify(P[:200 * (L + 1)], Q[:200 * L], V, tokens[:200 * L], offs[:201],
                          np.full(200, T, np.float32), 77, 2, tau=0.0)
    for k in ("accept_len", "out_tokens", "ratio", "alpha"):
        assert np.array_equal(strict[k], relaxed0[k])
    # The relaxed ratio of one row pair, and the argmax indicator at T = 0.
    assert math.isclose(orc.ratio_relaxed(np.log(pp[0]), np.log(qq[0]), 1.0, 1, tau),
                        (1 + tau) * pp[0][1] / qq[0][1], rel_tol=1e-12)
    assert orc.ratio_relaxed(np.log(pp[0]), np.log(qq[0]), 0.0, 0, 9.0) == 1.0
    assert orc.ratio_relaxed(np.log(pp[0]), np.log(qq[0]), 0.0, 1, 9.0) == 0.0


def pin_filter_known(orc):
    """The sampling filters of the pages' evaluation setting (experiments,
    §4.1: top-k, then top-p, renormalised) on hand-worked rows; no filter is
    plain softmax; top-k 1 is the lowest-id argmax; the temperature applies
    before the filters."""
    pr = np.array([0.5, 0.3, 0.15, 0.05])
    lg = np.log(pr)
    cases = [((0, 0.75), [0.625, 0.375, 0, 0]), ((0, 0.45), [1, 0, 0, 0]),
             ((3, 1.0), [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0]), ((2, 0.9), [0.625, 0.375, 0, 0]),
             ((0, 0.9), [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0]),
             ((3, 0.82), [0.625, 0.375, 0, 0])]  # top-p measured within the top 3
    for (k, tp), want in cases:
        assert np.allclose(orc.filtered_probs(lg, 1.0, k, tp), want, atol=1e-12), (k, tp)
    # Equal probabilities: the lower ids are kept.
    assert np.allclose(orc.filtered_probs(np.zeros(4), 1.0, 2, 1.0), [0.5, 0.5, 0, 0], atol=1e-12)
    rng = np.random.default_rng(21)
    z = rng.normal(0, 2, 50)
    assert np.allclose(orc.filtered_probs(z, 0.7, 0, 1.0), sp_softmax(z / 0.7), atol=1e-14)
    assert np.allclose(orc.filtered_probs(z, 0.7, 50, 1.0), sp_softmax(z / 0.7), atol=1e-14)
    onehot = np.zeros(50)
    onehot[int(np.argmax(z))] = 1.0
    assert np.array_equal(orc.filtered_probs(z, 1.3, 1, 1.0), onehot)
    # T = 2 turns p into sqrt(p) renormalised, before the top-2 filter.
    sq = np.sqrt(pr)
    assert np.allclose(orc.filtered_probs(lg, 2.0, 2, 1.0), [sq[0] / (sq[0] + sq[1]), sq[1] / (sq[0] + sq[1]), 0, 0],
                       atol=1e-12)
    # The cut's margin: shares 0.5, 0.8 of the whole row at top-p 0.75 -> min(0.05, 0.25);
    # within the top 3 (mass 0.95) at top-p 0.82: shares 0.5/0.95, 0.8/0.95 -> min(0.8/0.95 - 0.82, 0.82 - 0.5/0.95).
    assert abs(orc.filtered_probs(lg, 1.0, 0, 0.75, with_margin=True)[1] - 0.05) < 1e-12
    assert abs(orc.filtered_probs(lg, 1.0, 3, 0.82, with_margin=True)[1] - (0.8 / 0.95 - 0.82)) < 1e-12
    assert orc.filtered_probs(lg, 1.0, 3, 1.0, with_margin=True)[1] == np.inf


def pin_filtered_verify_law(orc):
    """Verification on filtered distributions (both p and q filtered, then
    §3.2's strict acceptance and residual correction): many copies of one
    sequence give (accept length, emitted token) with the exact law built
    from the hand-worked filtered rows, and the emitted first token follows
    the filtered p (the lossless property carries over to any pair of
    distributions).  With no filter it is the plain verify step."""
    V, L, T = 4, 1, 1.0
    p1 = np.array([0.5, 0.3, 0.15, 0.05])
    q1 = np.array([0.1, 0.4, 0.3, 0.2])
    p2 = np.array([0.1, 0.2, 0.3, 0.4])
    k, tp = 3, 0.9
    # Filtered by hand: p1 -> top-3 {0, 1, 2} renormalised, cumulative 0.526,
    # 0.842, 1.0 -> all three; q1 -> top-3 {1, 2, 3}: 0.444, 0.778, 1.0 -> all
    # three; p2 -> top-3 {3, 2, 1}: 0.444, 0.778, 1.0 -> all three.
    pt = np.array([0.5, 0.3, 0.15, 0]) / 0.95
    qt = np.array([0, 0.4, 0.3, 0.2]) / 0.9
    bt = np.array([0, 0.2, 0.3, 0.4]) / 0.9
    C = 20000
    P = np.tile(np.log(np.stack([p1, p2])).astype(np.float32), (C, 1))
    Q = np.tile(np.log(q1[None]).astype(np.float32), (C, 1))
    offs = (np.arange(C + 1) * L).astype(np.int32)
    rng = np.random.default_rng(31)
    xs = rng.choice(V, size=C, p=qt).astype(np.int32)  # proposals from the filtered q
    out = orc.verify_filtered(P, Q, V, xs, offs, np.full(C, T, np.float32), 5, 1, k, tp)
    a = out["accept_len"]
    tok = out["out_tokens"].reshape(C, L + 1)[np.arange(C), a]
    first = out["out_tokens"].reshape(C, L + 1)[:, 0]
    assert _chi2_ok(np.bincount(first, minlength=V), pt), np.bincount(first, minlength=V)
    ratio = np.where(qt > 0, np.minimum(1.0, pt / np.where(qt > 0, qt, 1.0)), 1.0)
    w = np.maximum(pt - qt, 0.0)
    w /= w.sum()
    law = np.concatenate([np.array([qt[x] * (1 - ratio[x]) for x in range(V)]).sum() * w,
                          np.zeros(V)])
    for x in range(V):  # accepted: token x itself in slot 0, then the bonus
        law[V:] += qt[x] * ratio[x] * bt
    counts = np.bincount(a * V + tok, minlength=2 * V)
    assert _chi2_ok(counts, law), (counts, law * C)
    # No filter: the plain step.
    Pn = P[:400 * (L + 1)]
    Qn = Q[:400 * L]
    xn = xs[:400]
    plain = orc.verify(Pn, Qn, V, xn, offs[:401], np.full(400, T, np.float32), 5, 1)
    filt = orc.verify_filtered(Pn, Qn, V, xn, offs[:401], np.full(400, T, np.float32), 5, 1, 0, 1.0)
    assert np.array_equal(plain["accept_len"], filt["accept_len"])
    assert np.array_equal(plain["out_tokens"], filt["out_tokens"])
    assert np.allclose(plain["ratio"], filt["ratio"], rtol=1e-12)


def pin_mc_propose_law(orc):
    """Proposals follow softmax(qnew/T) (inverse CDF with the PROPOSE
    uniforms); T = 0 gives the lowest-id argmax; accept_len < L gives no
    proposals."""
    V = 5
    probs = np.array([0.05, 0.4, 0.15, 0.3, 0.1])
    for T in (1.0, 0.5):
        C = 30000
        row = (T * np.log(probs)).astype(np.float32)
        pr = sp_softmax(row.astype(np.float64) / T)
        Qn = np.tile(row, (C, 1))
        offs = np.arange(C + 1, dtype=np.int32)
        out = orc.propose(Qn, V, offs, np.full(C, T, np.float32), 77, 3)
        assert np.all(out["valid"] == 1)
        assert _chi2_ok(np.bincount(out["proposals"], minlength=V), pr)
    Qn = np.array([[0.0, 2.0, 2.0, 1.0, -1.0]] * 4, np.float32)
    offs = np.array([0, 2, 4], np.int32)
    out = orc.propose(Qn, V, offs, np.zeros(2, np.float32), 0, 0, accept_len=np.array([2, 1], np.int32))
    assert list(out["valid"]) == [1, 0]
    assert list(out["proposals"]) == [1, 1, -1, -1]


def pin_mc_step_independence(orc):
    """Every decision of a step draws its own uniform: conditioned on all
    proposals passing (u_k < ratio_k), the next proposals still follow
    softmax(qnew/T), so the propose draws do not reuse the accept draws."""
    V, L, T = 4, 2, 1.0
    C = 40000
    prow = np.log(np.array([[0.4, 0.3, 0.2, 0.1], [0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]]))
    qrow = np.log(np.array([[0.1, 0.2, 0.3, 0.4], [0.4, 0.3, 0.2, 0.1]]))
    P = np.tile(prow.astype(np.float32), (C, 1))
    Q = np.tile(qrow.astype(np.float32), (C, 1))
    offs = (np.arange(C + 1) * L).astype(np.int32)
    tokens = np.tile(np.array([2, 1], np.int32), C)    # ratios 2/3 and 2/3
    temps = np.full(C, T, np.float32)
    ver = orc.verify(P, Q, V, tokens, offs, temps, 21, 4)
    qn = np.log(np.array([[0.1, 0.2, 0.3, 0.4], [0.4, 0.3, 0.2, 0.1]])).astype(np.float32)
    Qn = np.tile(qn, (C, 1))
    pro = orc.propose(Qn, V, offs, temps, 21, 4, accept_len=ver["accept_len"])
    ok = pro["valid"].astype(bool)
    assert ok.sum() > C // 5
    props = pro["proposals"].reshape(C, L)[ok]
    pn = [sp_softmax(r.astype(np.float64)) for r in qn]
    for m in range(L):
        assert _chi2_ok(np.bincount(props[:, m], minlength=V), pn[m]), m


def pin_alpha_mean(orc):
    """alpha_i is the mean of the sequence's ratios over all its positions
    (§2, no truncation at the first rejection); the batch value is the mean
    over sequences."""
    r = np.array([1.0, 0.5, 0.25, 1.0, 0.0, 0.75], np.float32)
    offs = np.array([0, 3, 4, 6], np.int32)
    per, mean = orc.alpha(r, offs)
    assert np.allclose(per, [1.75 / 3, 1.0, 0.375], atol=1e-15)
    assert abs(mean - (1.75 / 3 + 1.0 + 0.375) / 3) < 1e-15


def pin_bf16_decoding(orc):
    """bf16 logits (as bit patterns, padded rows) decode to the values torch
    gives them: the batched verify equals verify_one on torch's decoding."""
    rng = np.random.default_rng(15)
    V, ld, Ls, T = 41, 48, [3, 2], 0.8
    C = len(Ls)
    offs = np.array([0, 3, 5], np.int32)
    Pb = np.zeros((5 + C, ld), np.uint16)
    Qb = np.zeros((5, ld), np.uint16)
    Pb[:, :V] = _bf16_bits(rng.normal(0, 2, (5 + C, V)))
    Qb[:, :V] = _bf16_bits(rng.normal(0, 2, (5, V)))
    tokens = rng.integers(0, V, 5).astype(np.int32)
    out = orc.verify(Pb, Qb, V, tokens, offs, np.full(C, T, np.float32), 4, 2)
    for i, L in enumerate(Ls):
        Pd = _bf16_values(Pb[offs[i] + i: offs[i] + i + L + 1, :V].copy())
        Qd = _bf16_values(Qb[offs[i]: offs[i] + L, :V].copy())
        ua = [orc.uniform(4, 2, i, k, TAG_ACCEPT) for k in range(1, L + 1)]
        uc = [orc.uniform(4, 2, i, k, TAG_CORRECT) for k in range(1, L + 1)]
        ub = orc.uniform(4, 2, i, L + 1, TAG_BONUS)
        # The batched entry takes T as float32, as the library does.
        ref = orc.verify_one(Pd, Qd, float(np.float32(T)), tokens[offs[i]: offs[i] + L], ua, uc, ub)
        assert ref["accept_len"] == out["accept_len"][i]
        assert np.array_equal(ref["ratio"], out["ratio"][offs[i]: offs[i] + L])
        assert list(ref["out_tokens"]) == list(out["out_tokens"][offs[i] + i: offs[i] + i + L + 1])


def pin_invalid_inputs(orc):
    """Bad sequences are flagged, not computed: stride outside [1, 32], a
    negative or non-finite temperature, a token outside [0, V)."""
    V = 8
    Ls = [2, 0, 33, 2, 2, 2, 1]
    temps = np.array([1.0, 1.0, 1.0, -0.5, np.nan, 1.0, 0.0], np.float32)
    C = len(Ls)
    offs = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    total = int(offs[-1])
    P = np.zeros((total + C, V), np.float32)
    Q = np.zeros((total, V), np.float32)
    tokens = np.zeros(total, np.int32)
    tokens[offs[5] + 1] = V           # out of range in sequence 5
    tokens[offs[6]] = -1              # out of range in sequence 6
    out = orc.verify(P, Q, V, tokens, offs, temps, 0, 0)
    assert list(out["accept_len"]) == [2, -1, -1, -1, -1, -1, -1]
    for i in range(1, C):
        assert np.isnan(out["alpha"][i])
        assert np.all(out["out_tokens"][offs[i] + i: offs[i + 1] + i + 1] == -1)
        assert np.all(np.isnan(out["ratio"][offs[i]: offs[i + 1]]))
    assert not math.isnan(out["alpha"][0])


# ---------------------------------------------------------------------------
# Gumbel-max draws (the pages' sampler, Summary §3.3)
# ---------------------------------------------------------------------------

def pin_gumbel_uniform_layout(orc):
    """The uniform of id v is the top 23 bits (plus one half) of word v % 4 of
    the block at counter (offset, i, k, 16 + tag + 256 (v // 4)), key
    (seed, 0), scaled by 2^-23 (numpy's Philox as the reference)."""
    rng = np.random.default_rng(31)
    for _ in range(12):
        seed, offset = (int(x) for x in rng.integers(0, 2**40, size=2))
        offset += 1
        i, k, tag = int(rng.integers(0, 4096)), int(rng.integers(1, 33)), int(rng.integers(1, 4))
        for v in (0, 1, 2, 3, 4, 7, 8, 151935, int(rng.integers(0, 151936))):
            words = np.random.Philox(counter=np.array([offset - 1, i, k, 16 + tag + 256 * (v // 4)], np.uint64),
                                     key=np.array([seed, 0], np.uint64)).random_raw(4)
            expect = (float(int(words[v % 4]) >> 41) + 0.5) / 2.0**23
            assert orc.gumbel_uniform(seed, offset, i, k, tag, v) == expect, (v, tag)
    us = np.array([orc.gumbel_uniform(5, 3, 2, 1, TAG_CORRECT, v) for v in range(65536)])
    assert us.min() > 0.0 and us.max() < 1.0
    assert _chi2_ok(np.bincount((us * 64).astype(int), minlength=64), np.full(64, 1 / 64))


def pin_gumbel_law(orc):
    """Gumbel-max property: the draw over weights w follows w / sum(w)
    (chi-square over 20,000 draws); ids of weight 0 never come out; one
    positive weight always wins; scaling w by a power of two changes no
    draw whose score gap is not a rounding tie."""
    w = np.array([0.1, 0.0, 0.5, 0.25, 0.15, 0.0])
    draws = [orc.gumbel_draw(w, 7, off, 3, 2, TAG_BONUS) for off in range(20000)]
    toks = np.array([d[0] for d in draws])
    assert _chi2_ok(np.bincount(toks, minlength=w.size), w / w.sum())
    one = np.zeros(9)
    one[6] = 0.3
    assert all(orc.gumbel_draw(one, 1, off, 0, 1, TAG_CORRECT)[0] == 6 for off in range(50))
    assert orc.gumbel_draw(np.zeros(4), 1, 0, 0, 1, TAG_CORRECT)[0] == -1
    for off in range(200):
        t1, gap = orc.gumbel_draw(w, 7, off, 3, 2, TAG_BONUS)
        if gap > 1e-9:
            assert orc.gumbel_draw(w * 8.0, 7, off, 3, 2, TAG_BONUS)[0] == t1


def pin_gumbel_verify_law(orc):
    """Verify with Gumbel-max correction and bonus draws has the exact law of
    (accept length, emitted token), as with inverse-CDF draws, and the first
    emitted token follows p_1 when the proposals come from q; Gumbel
    proposals follow softmax(qnew / T)."""
    V, L, T = 3, 2, 1.0
    pp = [np.array([0.5, 0.3, 0.2]), np.array([0.2, 0.2, 0.6]), np.array([0.1, 0.6, 0.3])]
    qq = [np.array([0.2, 0.5, 0.3]), np.array([0.5, 0.1, 0.4])]
    C = 12000
    P = np.tile(np.log(np.stack(pp)).astype(np.float32), (C, 1))
    Q = np.tile(np.log(np.stack(qq)).astype(np.float32), (C, 1))
    offs = (np.arange(C + 1) * L).astype(np.int32)
    pr = [sp_softmax(r) for r in np.log(np.stack(pp)).astype(np.float32).astype(np.float64)]
    qr = [sp_softmax(r) for r in np.log(np.stack(qq)).astype(np.float32).astype(np.float64)]
    r1, r2 = min(1, pr[0][1] / qr[0][1]), min(1, pr[1][0] / qr[1][0])
    out = orc.verify_gumbel(P, Q, V, np.tile(np.array([1, 0], np.int32), C), offs, np.full(C, T, np.float32),
                            77, 1)
    a = out["accept_len"]
    last = out["out_tokens"].reshape(C, L + 1)[np.arange(C), a]
    w1 = np.maximum(pr[0] - qr[0], 0); w1 /= w1.sum()
    w2 = np.maximum(pr[1] - qr[1], 0); w2 /= w2.sum()
    probs = np.concatenate([(1 - r1) * w1, r1 * (1 - r2) * w2, r1 * r2 * pr[2]])
    assert _chi2_ok(np.bincount(a * V + last, minlength=3 * V), probs)
    rng = np.random.default_rng(18)
    xs = np.stack([rng.choice(V, size=C, p=qr[0]), rng.choice(V, size=C, p=qr[1])], axis=1)
    out = orc.verify_gumbel(P, Q, V, xs.reshape(-1).astype(np.int32), offs, np.full(C, T, np.float32), 99, 0)
    assert _chi2_ok(np.bincount(out["out_tokens"].reshape(C, L + 1)[:, 0], minlength=V), pr[0])
    # proposals: softmax(qnew / 0.5)
    Qn = np.tile(np.log(qq[0]).astype(np.float32), (C, 1))
    prop = orc.propose_gumbel(Qn, V, np.arange(C + 1, dtype=np.int32), np.full(C, 0.5, np.float32), 4, 2)
    qn = sp_softmax(np.log(qq[0]).astype(np.float32).astype(np.float64) / 0.5)
    assert _chi2_ok(np.bincount(prop["proposals"], minlength=V), qn)


# ---------------------------------------------------------------------------
# KV-slot bookkeeping of the stationary-batch loop (Summary §3.3)
# ---------------------------------------------------------------------------

def _kv_state(d):
    from speculative_verify_accept_02_b300.workloads import KVState
    a = lambda x: np.array(x, np.int32)
    return KVState(a(d["table"]), a(d["seq_len"]), a(d["pend"]), a(d["alloc"]), a(d["free_slots"]),
                   a([d["free_top"]]))


def pin_kv_handworked(orc):
    """Commits worked by hand (tests/golden/handworked_kv_commit.json): the
    kept prefix, the trimmed slots pushed in order, the batch's block taken
    from the stack top, and refusals that change nothing."""
    with open(os.path.join(GOLDEN, "handworked_kv_commit.json")) as f:
        g = json.load(f)
    st = _kv_state(dict(g["initial"]))
    for c in g["commits"]:
        before = st.copy()
        status = orc.kv_commit(st, c["accept_len"], g["num_masks"])
        assert status == c["status"], (c["name"], status)
        if c.get("unchanged"):
            assert st.equal(before), c["name"]
        else:
            assert st.equal(_kv_state(c)), c["name"]
    pc = g["pool_case"]
    st = _kv_state(pc)
    before = st.copy()
    assert orc.kv_commit(st, pc["accept_len"], pc["num_masks"]) == pc["status"]
    assert st.equal(before)


def pin_kv_refusals_and_exact_fits(orc):
    """Hand-derived edge cases: an inconsistent in-flight count (STATE = 1),
    a trimmed entry that is not a pool slot (SLOT = 4), and allocations that
    use the last free slot and the last table column (accepted)."""
    from speculative_verify_accept_02_b300.workloads import KVState
    a = lambda x: np.array(x, np.int32)
    # After the admission of the worked example: seq 0 at positions 2..4, seq 1 at 1..3.
    admitted = dict(table=[[0, 1, 14, 15, 16, -1, -1, -1, -1, -1], [2, 17, 18, 19, -1, -1, -1, -1, -1, -1]],
                    seq_len=[2, 1], pend=[0, 0], alloc=[3, 3],
                    free_slots=list(range(3, 20)) + [-1, -1, -1], free_top=11)
    st = _kv_state(admitted)
    st.alloc[0] = 4                      # not 1 + L + M = 3
    before = st.copy()
    assert orc.kv_commit(st, [0, 0], 2) == 1 and st.equal(before)
    st = _kv_state(admitted)
    st.table[1, 3] = 20                  # trimmed in this commit; the pool has slots 0..19
    before = st.copy()
    assert orc.kv_commit(st, [0, 0], 2) == 4 and st.equal(before)
    st = _kv_state(admitted)
    st.pend[1] = 1                       # then alloc 3 != 1 + 1 + 2
    assert orc.kv_commit(st, [0, 0], 2) == 1
    # Exact fits: one admitted sequence takes all 4 free slots and fills its row.
    st = KVState(a([[7, 6, -1, -1, -1, -1]]), a([2]), a([0]), a([0]), a([3, 2, 1, 0, 5, 4, 6, 7]), a([4]))
    assert orc.kv_commit(st, [0], 3) == 0
    assert list(st.table[0]) == [7, 6, 3, 2, 1, 0] and int(st.free_top[0]) == 0
    assert list(st.alloc) == [4] and list(st.pend) == [0] and list(st.seq_len) == [2]


def pin_kv_cache_holds_token_stream(orc):
    """A stationary batch run for many steps with random accept lengths: a
    synthetic forward writes each query token's id into its slot (x_last,
    the pending proposals, a mask id at the mask positions), verification is
    simulated from §3.2 (accept a prefix, then a correction or bonus token;
    the masks' proposals are verified next only after a full acceptance or a
    proposal-only step).  After every commit the cache must hold exactly the
    committed token stream minus its newest token (x_last), and every pool
    slot must be either free or referenced once."""
    from speculative_verify_accept_02_b300.workloads import draw_accept_lengths, make_kv_state
    rng = np.random.default_rng(11)
    C, M, steps, MASK = 5, 3, 40, -7
    prompts = [list(rng.integers(0, 1000, int(n))) for n in rng.integers(1, 9, C)]
    ld = 9 + steps * (M + 1) + 2 * M + 1
    st = make_kv_state(C, ld, C * ld, [len(pr) - 1 for pr in prompts], seed=5)
    content = np.full(C * ld, -1, np.int64)
    for i, pr in enumerate(prompts):
        content[st.table[i, :len(pr) - 1]] = pr[:-1]
    stream = [list(pr) for pr in prompts]
    pending = [[] for _ in range(C)]
    accept = np.zeros(C, np.int32)
    for step in range(steps):
        assert orc.kv_commit(st, accept, M) == 0, step
        used = []
        for i in range(C):
            n = int(st.seq_len[i])
            assert n == len(stream[i]) - 1, (step, i)
            assert list(content[st.table[i, :n]]) == stream[i][:-1], (step, i)
            assert int(st.pend[i]) == len(pending[i]) and int(st.alloc[i]) == 1 + len(pending[i]) + M
            live = n + int(st.alloc[i])
            assert np.all(st.table[i, live:] == -1)
            used += list(st.table[i, :live])
        free = list(st.free_slots[:int(st.free_top[0])])
        assert sorted(used + free) == list(range(st.pool_size)), step
        # the forward writes its query tokens into the allocated slots
        for i in range(C):
            n, L = int(st.seq_len[i]), len(pending[i])
            toks = [stream[i][-1]] + pending[i] + [MASK] * M
            content[st.table[i, n:n + len(toks)]] = toks
        accept = draw_accept_lengths(rng, st.pend, 0.7)
        for i in range(C):
            L = len(pending[i])
            if L == 0:                                   # proposal-only step
                stream[i].append(int(rng.integers(0, 1000)))
                pending[i] = list(rng.integers(0, 1000, M))
                continue
            k = int(accept[i])
            stream[i] += pending[i][:k] + [int(rng.integers(0, 1000))]
            pending[i] = list(rng.integers(0, 1000, M)) if k == L else []


ALL_PINS = [
    pin_philox_numpy, pin_uniform_layout, pin_softmax_library, pin_temperature_ratio,
    pin_tv_identity, pin_residual_known, pin_icdf_grid, pin_handworked, pin_greedy_planted,
    pin_p_equals_q, pin_lossless_enumeration, pin_mc_verify_law, pin_mc_propose_law,
    pin_mc_step_independence, pin_alpha_mean, pin_bf16_decoding, pin_invalid_inputs, pin_relaxed_law,
    pin_filter_known, pin_filtered_verify_law, pin_kv_handworked, pin_kv_refusals_and_exact_fits,
    pin_kv_cache_holds_token_stream, pin_gumbel_uniform_layout, pin_gumbel_law, pin_gumbel_verify_law,
]
