"""GPU-vs-oracle comparison of one verify / propose step.

The bar: accept lengths, emitted tokens and proposals bit-exact, except at a
decision whose oracle margin (|u - ratio| for an accept test, the inverse-CDF
distance for a draw) is below 1e-5 — those are counted and reported, and
nothing downstream of them in that sequence is compared.  Greedy (T = 0)
decisions compare exact logits and have no exemption.  Per-position ratios
and alpha agree within 1e-4 relative.
"""
from dataclasses import dataclass, field

import numpy as np

MARGIN = 1e-5
RTOL = 1e-4


@dataclass
class Report:
    """What a comparison covered: the sequences compared, the decisions
    exempted for an oracle margin below MARGIN (accept tests, draws), and the
    sequences left out of a filtered comparison because the oracle's top-p
    cut lies within its own rounding of moving (cut_skips)."""
    sequences: int = 0
    exempt_accept: int = 0
    exempt_token: int = 0
    cut_skips: int = 0
    failures: list = field(default_factory=list)

    def fail(self, msg):
        self.failures.append(msg)

    def check(self):
        assert not self.failures, "\n".join(self.failures[:20])

    def summary(self):
        return {"compared": self.sequences, "exempt_accept": self.exempt_accept,
                "exempt_token": self.exempt_token, "cut_skips": self.cut_skips}

    def merge(self, other):
        self.sequences += other.sequences
        self.exempt_accept += other.exempt_accept
        self.exempt_token += other.exempt_token
        self.cut_skips += other.cut_skips
        self.failures += other.failures
        return self


def _close(a, b, rtol=RTOL):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    ok = np.abs(a - b) <= rtol * np.abs(b) + 1e-30
    return ok | both_nan


def compare_verify(ora, gpu, offsets, seqs=None, report=None):
    """ora: dict from oracle.verify; gpu: dict of numpy arrays (accept_len,
    out_tokens, ratio, alpha).  Compares the sequences in `seqs` (all if None)."""
    rep = report or Report()
    offs = np.asarray(offsets)
    C = offs.size - 1
    for i in (range(C) if seqs is None else seqs):
        rep.sequences += 1
        s, e = int(offs[i]), int(offs[i + 1])
        L = e - s
        a_o, a_g = int(ora["accept_len"][i]), int(gpu["accept_len"][i])
        r_o, r_g = ora["ratio"][s:e], gpu["ratio"][s:e]
        if not np.all(_close(r_g, r_o)):
            bad = np.where(~_close(r_g, r_o))[0]
            rep.fail(f"seq {i}: ratio mismatch at {bad[:4]}: gpu {r_g[bad[:4]]} oracle {r_o[bad[:4]]}")
        if not _close([gpu["alpha"][i]], [ora["alpha"][i]])[0]:
            rep.fail(f"seq {i}: alpha gpu {gpu['alpha'][i]} oracle {ora['alpha'][i]}")
        if a_o < 0 or a_g < 0:
            if a_o != a_g:
                rep.fail(f"seq {i}: validity differs (gpu {a_g}, oracle {a_o})")
            continue
        if a_o != a_g:
            k = min(a_o, a_g)              # first decision that differs (0-based)
            m = ora["accept_margin"][s + k]
            if m < MARGIN:
                rep.exempt_accept += 1
            else:
                rep.fail(f"seq {i}: accept_len gpu {a_g} oracle {a_o} (margin {m:.3g})")
            continue
        slots_o = ora["out_tokens"][s + i: e + i + 1]
        slots_g = gpu["out_tokens"][s + i: e + i + 1]
        if not np.array_equal(slots_o[:a_o], slots_g[:a_o]) or not np.all(slots_g[a_o + 1:] == -1):
            rep.fail(f"seq {i}: emitted prefix differs gpu {slots_g} oracle {slots_o}")
            continue
        if slots_o[a_o] != slots_g[a_o]:
            m = ora["token_margin"][i]
            if m < MARGIN:
                rep.exempt_token += 1
            else:
                rep.fail(f"seq {i}: token gpu {slots_g[a_o]} oracle {slots_o[a_o]} (margin {m:.3g}, "
                         f"a={a_o}, L={L})")
    return rep


def compare_propose(ora, gpu, offsets, seqs=None, report=None):
    rep = report or Report()
    offs = np.asarray(offsets)
    C = offs.size - 1
    for i in (range(C) if seqs is None else seqs):
        rep.sequences += 1
        s, e = int(offs[i]), int(offs[i + 1])
        if int(ora["valid"][i]) != int(gpu["valid"][i]):
            rep.fail(f"seq {i}: valid gpu {gpu['valid'][i]} oracle {ora['valid'][i]}")
            continue
        for r in range(s, e):
            po, pg = int(ora["proposals"][r]), int(gpu["proposals"][r])
            if po != pg:
                m = ora["margin"][r]
                if m < MARGIN:
                    rep.exempt_token += 1
                else:
                    rep.fail(f"seq {i} row {r}: proposal gpu {pg} oracle {po} (margin {m:.3g})")
    return rep
