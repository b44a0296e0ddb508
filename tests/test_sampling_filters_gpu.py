"""isd_verify_filtered and isd_propose_filtered (include/isd_filter.h) against
the oracle's filtered step (top-k, then top-p, on p and q alike: the pages'
evaluation setting), element by element on the same seeded inputs.

The bar is parity.py's: accept lengths, emitted tokens and proposals exact,
ratios and alpha within 1e-4 relative, except at a decision whose oracle
margin is below 1e-5.  A sequence one of whose rows has its top-p cut within
CUT_MARGIN of moving is not compared at all (the kept set itself is then a
rounding decision); such sequences are counted and must stay rare.  The
kernels do the list arithmetic in double precision (weights within a few
ulp, sums of at most 64 terms), so their running shares agree with the
oracle's to about 1e-14: CUT_MARGIN = 1e-9.  The oracle gets top_p as the
float32 the C ABI receives.  Cases:
the evaluation setting on full-size rows, ragged strides with mixed
temperatures and q == p, padded rows whose first ids are not 16-byte
aligned (both dtypes), top-k above the vocabulary, top-1, a tight top-p,
the largest stride, greedy batches, invalid sequences, and rows that
stress the top-k lists (runs of equal logits, ascending logits, all-equal
and mostly -inf rows).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import MARGIN, Report, compare_propose, compare_verify
from speculative_verify_accept_02_b300 import build, isd_propose_filtered, isd_verify_filtered, workloads

pytestmark = pytest.mark.gpu

CUT_MARGIN = 1e-9


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def f32(x):
    """x as the float32 the C ABI receives."""
    return float(np.float32(x))


def host(batch):
    return dict(p=workloads.host_logits(batch.p), q=workloads.host_logits(batch.q),
                qnew=workloads.host_logits(batch.qnew), tokens=batch.tokens.cpu().numpy(),
                offs=batch.seq_offsets.cpu().numpy(), temp=batch.temperature.cpu().numpy())


def gpu_verify(batch, seed, offset, top_k, top_p):
    b = batch.to("cuda")
    v = isd_verify_filtered(b.p, b.q, b.tokens, b.seq_offsets, b.temperature, seed, offset, top_k=top_k,
                            top_p=top_p, vocab=b.vocab, total=b.total)
    torch.cuda.synchronize()
    return dict(accept_len=v.accept_len.cpu().numpy(), out_tokens=v.out_tokens.cpu().numpy(),
                ratio=v.ratio.cpu().numpy(), alpha=v.alpha.cpu().numpy())


def gpu_propose(batch, seed, offset, top_k, top_p, accept_len):
    b = batch.to("cuda")
    acc = None if accept_len is None else torch.as_tensor(accept_len, dtype=torch.int32, device="cuda")
    pr = isd_propose_filtered(b.qnew, b.seq_offsets, b.temperature, seed, offset, acc, top_k=top_k,
                              top_p=top_p, vocab=b.vocab, total=b.total)
    torch.cuda.synchronize()
    return dict(proposals=pr.proposals.cpu().numpy(), valid=pr.valid.cpu().numpy())


def compare_step(batch, seed, offset, top_k, top_p, rep):
    """Verify, then propose with the GPU's accept lengths; returns the number
    of sequences left out for a top-p cut on the edge."""
    h = host(batch)
    V = batch.vocab
    gv = gpu_verify(batch, seed, offset, top_k, top_p)
    tp = f32(top_p)
    ov = oracle.verify_filtered(h["p"], h["q"], V, h["tokens"], h["offs"], h["temp"], seed, offset, top_k, tp)
    keep = [i for i in range(batch.num_seqs) if ov["cut_margin"][i] >= CUT_MARGIN]
    rep.cut_skips += batch.num_seqs - len(keep)
    compare_verify(ov, gv, h["offs"], seqs=keep, report=rep)
    op = oracle.propose_filtered(h["qnew"], V, h["offs"], h["temp"], seed, offset, top_k, tp,
                                 accept_len=gv["accept_len"])
    gp = gpu_propose(batch, seed, offset, top_k, top_p, gv["accept_len"])
    compare_propose(op, gp, h["offs"], report=rep)
    return batch.num_seqs - len(keep)


CASES = [
    ("tiny", dict(), 50, 0.95),
    ("c64", dict(num_seqs=3), 50, 0.95),                                  # the evaluation setting, full V
    ("c64", dict(num_seqs=5, vocab=20003), 50, 0.95),                     # V not a multiple of the vector
    ("c64", dict(num_seqs=4, vocab=5000, ld=5003), 50, 0.9),              # rows start off 16-byte boundaries
    ("ragged", dict(num_seqs=12, vocab=4099), 50, 0.95),                  # T in {0, 0.6, 1}; q == p on even i
    ("ragged", dict(num_seqs=10, vocab=777, ld=781, dtype=torch.float32), 64, 0.8),
    ("highconc", dict(num_seqs=4, vocab=8191), 20, 0.95),
    ("tiny", dict(num_seqs=5, vocab=40), 64, 1.0),                        # top_k above V: every id kept
    ("tiny", dict(num_seqs=4, vocab=300), 1, 0.95),                       # top-1
    ("c64", dict(num_seqs=3, stride=32, vocab=4099), 50, 0.5),            # the largest stride, tight top-p
    ("greedy", dict(num_seqs=6, vocab=3001), 50, 0.95),                   # T = 0: filters change nothing
]


@pytest.mark.parametrize("name,kw,top_k,top_p", CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_filtered_parity(name, kw, top_k, top_p):
    batch = workloads.make(name, **kw)
    rep = Report()
    skipped = 0
    for seed, offset in ((0, 0), (5, 2)):
        skipped += compare_step(batch, seed, offset, top_k, top_p, rep)
    rep.check()
    assert skipped <= max(1, batch.num_seqs // 10), skipped
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 10)


def _pattern_rows(kind, rows, V, g):
    if kind == "ties":        # a ramp in bf16: long runs of equal logits, broken by id
        base = torch.linspace(-8.0, 8.0, V)
        return (base + 0.0 * torch.randn(rows, V, generator=g)).to(torch.bfloat16).float()
    if kind == "ascending":   # every id beats the list: the worst case for the running lists
        return torch.linspace(-4.0, 4.0, V).repeat(rows, 1) + 0.01 * torch.randn(rows, V, generator=g)
    if kind == "equal":       # all logits equal: the lowest ids are kept
        return torch.zeros(rows, V)
    z = torch.randn(rows, V, generator=g)   # "masked": most logits -inf, a few finite
    keep = torch.rand(rows, V, generator=g) < 0.01
    keep[:, 0] = True
    return torch.where(keep, z, torch.full_like(z, -float("inf")))


@pytest.mark.parametrize("kind", ["ties", "ascending", "equal", "masked"])
def test_filtered_adversarial_rows(kind):
    """Rows that stress the top-k lists: runs of equal logits, ascending
    logits (every id a candidate), all-equal rows, and rows that are mostly
    -inf; bf16, rows not 16-byte aligned."""
    g = torch.Generator().manual_seed(11)
    C, L, V, ld = 3, 4, 4099, 4103
    total = C * L
    offs = torch.arange(C + 1, dtype=torch.int32) * L
    P = _pattern_rows(kind, total + C, V, g)
    Q = _pattern_rows(kind, total, V, g) + (0.0 if kind == "equal" else 0.5 * torch.randn(total, V, generator=g))
    Q = torch.where(torch.isfinite(P[:total]) | (kind != "masked"), Q, torch.full_like(Q, -float("inf")))
    Q[:, 0] = torch.where(torch.isfinite(Q[:, 0]), Q[:, 0], torch.zeros(total))
    toks = torch.stack([torch.multinomial(torch.softmax(Q[r], 0), 1, generator=g)[0] for r in range(total)])
    pad = lambda x: torch.nn.functional.pad(x, (0, ld - V)).to(torch.bfloat16)
    batch = workloads.Batch(kind, V, ld, torch.bfloat16, offs, torch.ones(C), toks.to(torch.int32),
                            pad(P), pad(Q), pad(_pattern_rows(kind, total, V, g)))
    rep = Report()
    skipped = compare_step(batch, 3, 1, 50, 0.95, rep)
    rep.check()
    assert skipped <= 1


def test_filtered_invalid_sequences():
    """Strides outside [1, 32], bad temperatures and out-of-range tokens are
    flagged as isd_verify flags them: accept_len -1, slots -1, NaN ratios."""
    V = 64
    Ls = [2, 0, 33, 2, 2, 2, 1]
    temps = torch.tensor([1.0, 1.0, 1.0, -0.5, float("nan"), 1.0, 0.0])
    C = len(Ls)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(Ls)]), dtype=torch.int32)
    total = int(offs[-1])
    g = torch.Generator().manual_seed(3)
    P = torch.randn(total + C, V, generator=g)
    Q = torch.randn(total, V, generator=g)
    toks = torch.randint(0, V, (total,), generator=g, dtype=torch.int32)
    toks[int(offs[5]) + 1] = V
    toks[int(offs[6])] = -1
    batch = workloads.Batch("invalid", V, V, torch.float32, offs, temps, toks, P, Q, Q.clone())
    gv = gpu_verify(batch, 0, 0, 50, 0.95)
    h = host(batch)
    ov = oracle.verify_filtered(h["p"], h["q"], V, h["tokens"], h["offs"], h["temp"], 0, 0, 50, f32(0.95))
    assert list(gv["accept_len"]) == list(ov["accept_len"])
    assert gv["accept_len"][0] >= 0 and np.all(gv["accept_len"][1:] == -1)
    for i in range(1, C):
        s, e = int(offs[i]), int(offs[i + 1])
        if 0 <= s <= e <= total:
            assert np.all(gv["out_tokens"][s + i:e + i + 1] == -1)
            assert np.all(np.isnan(gv["ratio"][s:e]))
    gp = gpu_propose(batch, 0, 0, 50, 0.95, None)
    assert list(gp["valid"]) == [1, 0, 0, 0, 0, 1, 1]


def test_filters_at_full_size():
    """The evaluation setting on the c64 batch shape (C=64, L=8, V=151936
    bf16) in one call: every accept length in [0, L], and sampled sequences
    equal to the oracle's run of the same sequence."""
    batch = workloads.make("c64")
    gv = gpu_verify(batch, 0, 0, 50, 0.95)
    assert np.all((gv["accept_len"] >= 0) & (gv["accept_len"] <= 8))
    o = batch.seq_offsets.tolist()
    h = host(batch)
    rep = Report()
    for i in (0, 17, 63):
        ov = _oracle_one_sequence(batch, h, i)
        if ov["cut_margin"][0] < CUT_MARGIN:
            continue
        g = dict(accept_len=gv["accept_len"][i:i + 1], out_tokens=gv["out_tokens"][o[i] + i:o[i + 1] + i + 1],
                 ratio=gv["ratio"][o[i]:o[i + 1]], alpha=gv["alpha"][i:i + 1])
        compare_verify(ov, g, [0, o[i + 1] - o[i]], report=rep)
    rep.check()


def _oracle_one_sequence(batch, h, i):
    """The oracle's filtered verify of sequence i alone, with its own
    uniforms: its rows placed at batch index i of a batch whose first i
    sequences are empty (stride 0: invalid, not computed).  Returned as a
    one-sequence result."""
    o = batch.seq_offsets.tolist()
    L = o[i + 1] - o[i]
    P = h["p"][o[i] + i:o[i] + i + L + 1]
    P = np.concatenate([np.zeros((i,) + P.shape[1:], P.dtype), P])
    Q = h["q"][o[i]:o[i] + L]
    offs = np.array([0] * (i + 1) + [L], np.int32)
    temp = np.concatenate([np.ones(i, np.float32), h["temp"][i:i + 1]]).astype(np.float32)
    ov = oracle.verify_filtered(P, Q, batch.vocab, h["tokens"][o[i]:o[i] + L], offs, temp, 0, 0, 50, f32(0.95))
    return dict(accept_len=ov["accept_len"][i:i + 1], out_tokens=ov["out_tokens"][i:i + L + 1],
                ratio=ov["ratio"][:L], alpha=ov["alpha"][i:i + 1], accept_margin=ov["accept_margin"][:L],
                token_margin=ov["token_margin"][i:i + 1], cut_margin=ov["cut_margin"][i:i + 1])
