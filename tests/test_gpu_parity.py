"""CUDA path (through the C ABI) against the fp64 oracle, element by element,
on the same seeded inputs: small batches of every workload at sizes the
oracle finishes in seconds (several chunks, ragged tails, padded rows, both
dtypes), the full-size workloads on sampled sequences, and edge cases."""
import numpy as np
import pytest
import torch

import oracle
from parity import Report, compare_propose, compare_verify
from speculative_verify_accept_02_b300 import build, isd_alpha, isd_propose, isd_verify, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def host(batch):
    return dict(p=workloads.host_logits(batch.p), q=workloads.host_logits(batch.q),
                qnew=workloads.host_logits(batch.qnew), tokens=batch.tokens.cpu().numpy(),
                offs=batch.seq_offsets.cpu().numpy(), temp=batch.temperature.cpu().numpy())


def gpu_step(batch, seed=0, offset=0, skip_rejected=True):
    b = batch.to("cuda")
    v = isd_verify(b.p, b.q, b.tokens, b.seq_offsets, b.temperature, seed, offset, vocab=b.vocab,
                   total=b.total)
    pr = isd_propose(b.qnew, b.seq_offsets, b.temperature, seed, offset,
                     accept_len=v.accept_len if skip_rejected else None, vocab=b.vocab, total=b.total)
    torch.cuda.synchronize()
    ver = dict(accept_len=v.accept_len.cpu().numpy(), out_tokens=v.out_tokens.cpu().numpy(),
               ratio=v.ratio.cpu().numpy(), alpha=v.alpha.cpu().numpy())
    pro = dict(proposals=pr.proposals.cpu().numpy(), valid=pr.valid.cpu().numpy())
    return ver, pro


def oracle_step(h, vocab, seed=0, offset=0, seqs=None, accept_len=None):
    ver = oracle.verify(h["p"], h["q"], vocab, h["tokens"], h["offs"], h["temp"], seed, offset, seqs=seqs)
    acc = ver["accept_len"] if accept_len is None else accept_len
    pro = oracle.propose(h["qnew"], vocab, h["offs"], h["temp"], seed, offset, accept_len=acc, seqs=seqs)
    return ver, pro


SMALL = [
    ("tiny", dict()),
    ("c64", dict(num_seqs=5)),                                   # full V: 19 chunks, short last chunk
    ("c64", dict(num_seqs=7, vocab=20003)),                      # V not a multiple of the vector width
    ("c64", dict(num_seqs=4, vocab=5000, ld=5003)),              # padded, 16-byte-misaligned rows
    ("c64", dict(num_seqs=3, stride=32, vocab=4099)),            # the largest stride
    ("greedy", dict(num_seqs=9)),
    ("greedy", dict(num_seqs=6, vocab=3001, ld=3005)),
    ("highconc", dict(num_seqs=5)),
    ("highconc", dict(num_seqs=8, vocab=8191)),
    ("ragged", dict(num_seqs=16)),
    ("ragged", dict(num_seqs=24, vocab=1537, dtype=torch.float32)),
    ("ragged", dict(num_seqs=12, vocab=777, ld=781, dtype=torch.float32)),
    ("tiny", dict(num_seqs=6, vocab=5)),
    ("tiny", dict(num_seqs=4, vocab=1)),
    ("tiny", dict(num_seqs=5, vocab=17, dtype=torch.bfloat16)),
    ("ragged", dict(num_seqs=600, vocab=300)),                  # layout and tokens beyond shared memory
]


@pytest.mark.parametrize("name,kw", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_small_parity(name, kw):
    batch = workloads.make(name, **kw)
    h = host(batch)
    rep = Report()
    for seed, offset in ((0, 0), (7, 3)):
        gv, gp = gpu_step(batch, seed, offset)
        ov, op = oracle_step(h, batch.vocab, seed, offset)
        compare_verify(ov, gv, h["offs"], report=rep)
        # Proposals are compared for the sequences whose accept lengths agree.
        agree = [i for i in range(batch.num_seqs) if ov["accept_len"][i] == gv["accept_len"][i]]
        op = oracle.propose(h["qnew"], batch.vocab, h["offs"], h["temp"], seed, offset,
                            accept_len=gv["accept_len"])
        compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep


@pytest.mark.parametrize("name,kw", [("c64", dict(num_seqs=6)), ("ragged", dict(num_seqs=6)), ("tiny", {}),
                                     ("ragged", dict(num_seqs=600, vocab=300))])
def test_propose_without_skip(name, kw):
    batch = workloads.make(name, **kw)
    h = host(batch)
    _, gp = gpu_step(batch, 5, 11, skip_rejected=False)
    op = oracle.propose(h["qnew"], batch.vocab, h["offs"], h["temp"], 5, 11)
    rep = compare_propose(op, gp, h["offs"])
    rep.check()
    assert np.all(gp["valid"] == 1)


def test_alpha_entry_point():
    batch = workloads.make("ragged", num_seqs=20, vocab=3000)
    gv, _ = gpu_step(batch)
    offs = batch.seq_offsets
    ratio = torch.from_numpy(gv["ratio"]).cuda()
    per, mean = isd_alpha(ratio, offs.cuda(), total=batch.total)
    o_per, o_mean = oracle.alpha(gv["ratio"].astype(np.float32), offs.numpy())
    assert np.allclose(per.cpu().numpy(), o_per, rtol=1e-5)
    assert abs(mean.item() - o_mean) <= 1e-5 * abs(o_mean)
    # The verify step's own alpha is the same quantity.
    assert np.allclose(gv["alpha"], o_per, rtol=1e-4)


FULL = ["c64", "greedy", "highconc", "ragged"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """The full workload in the configuration the benchmark times; the oracle
    checks a sample of sequences one by one."""
    batch = workloads.make(name, device="cuda")
    gv, gp = gpu_step(batch)
    C = batch.num_seqs
    rng = np.random.default_rng(3)
    seqs = sorted(set([0, C - 1] + list(rng.choice(C, size=min(C, 10), replace=False))))
    h = host(batch)
    ov, op = oracle_step(h, batch.vocab, seqs=seqs, accept_len=gv["accept_len"])
    rep = compare_verify(ov, gv, h["offs"], seqs=seqs)
    compare_propose(op, gp, h["offs"], seqs=[i for i in seqs if ov["accept_len"][i] == gv["accept_len"][i]],
                    report=rep)
    rep.check()
    # Properties that hold at any size, on every sequence.
    acc = gv["accept_len"]
    L = np.diff(h["offs"])
    assert np.all((acc >= 0) & (acc <= L))
    for i in range(C):
        s = h["offs"][i]
        slots = gv["out_tokens"][s + i: s + i + L[i] + 1]
        assert np.array_equal(slots[:acc[i]], h["tokens"][s: s + acc[i]])
        assert 0 <= slots[acc[i]] < batch.vocab and np.all(slots[acc[i] + 1:] == -1)
    assert np.all((gv["ratio"] >= 0) & (gv["ratio"] <= 1))
    if name == "ragged":
        even = np.arange(0, C, 2)
        assert np.all(acc[even] == L[even])                 # q == p accepts everything
    if name == "greedy":
        assert np.all(np.isin(gv["ratio"], [0.0, 1.0]))


def test_repeatable_and_seeded():
    batch = workloads.make("c64", num_seqs=8, vocab=30000)
    a1, p1 = gpu_step(batch, 1, 2)
    a2, p2 = gpu_step(batch, 1, 2)
    for k in a1:
        assert np.array_equal(a1[k], a2[k], equal_nan=True), k
    assert np.array_equal(p1["proposals"], p2["proposals"])
    b1, _ = gpu_step(batch, 1, 3)
    assert not np.array_equal(a1["out_tokens"], b1["out_tokens"])


def test_invalid_sequences_and_empty_batch():
    V = 300
    Ls = [2, 0, 33, 2, 2, 2, 1, 3]
    temps = np.array([1.0, 1.0, 1.0, -0.5, np.nan, 1.0, 1e-40, 0.0], np.float32)
    C = len(Ls)
    offs = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    total = int(offs[-1])
    g = torch.Generator().manual_seed(1)
    P = torch.randn(total + C, V, generator=g).to(torch.bfloat16)
    Q = torch.randn(total, V, generator=g).to(torch.bfloat16)
    tokens = torch.randint(0, V, (total,), generator=g, dtype=torch.int32)
    tokens[offs[5] + 1] = V
    d = "cuda"
    out = isd_verify(P.to(d), Q.to(d), tokens.to(d), torch.from_numpy(offs).to(d),
                     torch.from_numpy(temps).to(d), 0, 0, total=total)
    torch.cuda.synchronize()
    ov = oracle.verify(workloads.host_logits(P), workloads.host_logits(Q), V, tokens.numpy(), offs, temps, 0, 0)
    gv = dict(accept_len=out.accept_len.cpu().numpy(), out_tokens=out.out_tokens.cpu().numpy(),
              ratio=out.ratio.cpu().numpy(), alpha=out.alpha.cpu().numpy())
    assert list(gv["accept_len"][1:7]) == [-1] * 6
    compare_verify(ov, gv, offs).check()
    # Empty batch: nothing launched, nothing written.
    e = torch.zeros(1, dtype=torch.int32, device=d)
    r = isd_verify(P.to(d), Q.to(d), tokens.to(d), e, torch.zeros(0, device=d), total=0)
    assert r.accept_len.numel() == 0


def test_greedy_ties_lowest_id():
    """bf16 ties at the maximum: the lowest id is the argmax everywhere."""
    V, L, C = 4099, 3, 4
    offs = torch.arange(C + 1, dtype=torch.int32) * L
    P = torch.zeros(C * (L + 1), V)
    for r in range(P.shape[0]):
        P[r, (37 * r + 5) % V] = 3.0
        P[r, (37 * r + 900) % V] = 3.0
        P[r, V - 1] = 3.0
    Q = torch.zeros(C * L, V)
    lo = torch.tensor([min((37 * r + 5) % V, (37 * r + 900) % V) for r in range(P.shape[0])])
    tokens = torch.empty(C * L, dtype=torch.int32)
    for i in range(C):
        for k in range(L):
            tokens[i * L + k] = lo[i * L + i + k] if k != i else (lo[i * L + i + k] + 1) % V
    temps = torch.zeros(C)
    d = "cuda"
    Pb, Qb = P.to(torch.bfloat16), Q.to(torch.bfloat16)
    out = isd_verify(Pb.to(d), Qb.to(d), tokens.to(d), offs.to(d), temps.to(d), total=C * L)
    torch.cuda.synchronize()
    acc = out.accept_len.cpu().tolist()
    assert acc == [0, 1, 2, 3]
    ov = oracle.verify(workloads.host_logits(Pb), workloads.host_logits(Qb), V, tokens.numpy(),
                       offs.numpy(), temps.numpy(), 0, 0)
    assert np.array_equal(ov["out_tokens"], out.out_tokens.cpu().numpy())


def test_all_accepted_largest_stride():
    """q identical to p accepts every proposal (Summary §3.2), here at the
    largest stride: the bonus token comes from the final anchor p_{L+1}, by a
    softmax draw at T > 0 and as its argmax at T = 0."""
    V, L = 4099, 32
    temps = np.array([1.0, 0.0, 0.6, 0.0], np.float32)
    C = len(temps)
    offs = (np.arange(C + 1) * L).astype(np.int32)
    total = C * L
    g = torch.Generator().manual_seed(11)
    P = torch.randn(total + C, V, generator=g).to(torch.bfloat16)
    prow = [int(offs[i]) + i + k for i in range(C) for k in range(L)]
    Q = P[prow].clone()
    tokens = torch.argmax(P[prow].float(), dim=1).to(torch.int32)  # accepted at T = 0 too
    d = "cuda"
    for seed, offset in ((0, 0), (3, 9)):
        out = isd_verify(P.to(d), Q.to(d), tokens.to(d), torch.from_numpy(offs).to(d),
                         torch.from_numpy(temps).to(d), seed, offset, total=total)
        torch.cuda.synchronize()
        gv = dict(accept_len=out.accept_len.cpu().numpy(), out_tokens=out.out_tokens.cpu().numpy(),
                  ratio=out.ratio.cpu().numpy(), alpha=out.alpha.cpu().numpy())
        assert list(gv["accept_len"]) == [L] * C
        ov = oracle.verify(workloads.host_logits(P), workloads.host_logits(Q), V, tokens.numpy(), offs, temps,
                           seed, offset)
        compare_verify(ov, gv, offs).check()


@pytest.mark.parametrize("name,kw,tau", [("c64", dict(num_seqs=6), 0.5), ("highconc", dict(num_seqs=5), 1.0),
                                          ("ragged", dict(num_seqs=12, vocab=3001), 0.25)])
def test_relaxed_acceptance_parity(name, kw, tau):
    """isd_verify_relaxed (the pages' relaxed-acceptance ablation, ratio x
    (1 + tau)) against the oracle with the same tau; with the same uniforms a
    relaxed accept length is never shorter than the strict one."""
    batch = workloads.make(name, **kw)
    h = host(batch)
    b = batch.to("cuda")
    rep = Report()
    for seed, offset in ((0, 0), (7, 3)):
        outs = {}
        for t in (0.0, tau):
            v = isd_verify(b.p, b.q, b.tokens, b.seq_offsets, b.temperature, seed, offset, vocab=b.vocab,
                           total=b.total, tau=t)
            torch.cuda.synchronize()
            outs[t] = dict(accept_len=v.accept_len.cpu().numpy(), out_tokens=v.out_tokens.cpu().numpy(),
                           ratio=v.ratio.cpu().numpy(), alpha=v.alpha.cpu().numpy())
        ov = oracle.verify(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], seed, offset, tau=tau)
        compare_verify(ov, outs[tau], h["offs"], report=rep)
        assert np.all(outs[tau]["accept_len"] >= outs[0.0]["accept_len"])
        assert np.array_equal(outs[tau]["ratio"], outs[0.0]["ratio"])
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep


FUSED = [("c64", dict(num_seqs=5)), ("greedy", dict(num_seqs=9)), ("highconc", dict(num_seqs=5)),
         ("ragged", dict(num_seqs=16)), ("ragged", dict(num_seqs=24, vocab=1537, dtype=torch.float32)),
         ("tiny", dict(num_seqs=6, vocab=5)), ("c64", dict(num_seqs=3, stride=32, vocab=4099))]


@pytest.mark.parametrize("name,kw", FUSED, ids=[f"{n}-{i}" for i, (n, _) in enumerate(FUSED)])
def test_fused_verify_propose_parity(name, kw):
    """isd_verify_propose (the fused step of Summary §3.2) against the oracle's
    verify and its propose with the same accept lengths."""
    from speculative_verify_accept_02_b300 import isd_verify_propose
    batch = workloads.make(name, **kw)
    h = host(batch)
    b = batch.to("cuda")
    rep = Report()
    for seed, offset in ((0, 0), (7, 3)):
        v, pr = isd_verify_propose(b.p, b.q, b.tokens, b.qnew, b.seq_offsets, b.temperature, seed, offset,
                                   vocab=b.vocab, total=b.total)
        torch.cuda.synchronize()
        gv = dict(accept_len=v.accept_len.cpu().numpy(), out_tokens=v.out_tokens.cpu().numpy(),
                  ratio=v.ratio.cpu().numpy(), alpha=v.alpha.cpu().numpy())
        gp = dict(proposals=pr.proposals.cpu().numpy(), valid=pr.valid.cpu().numpy())
        ov = oracle.verify(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], seed, offset)
        compare_verify(ov, gv, h["offs"], report=rep)
        agree = [i for i in range(batch.num_seqs) if ov["accept_len"][i] == gv["accept_len"][i]]
        op = oracle.propose(h["qnew"], batch.vocab, h["offs"], h["temp"], seed, offset,
                            accept_len=gv["accept_len"])
        compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
        assert np.array_equal(gp["valid"], (gv["accept_len"] == np.diff(h["offs"])).astype(np.uint8))
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep


def test_fused_invalid_sequences_and_relaxed():
    """The fused call on a batch with invalid sequences (strides out of range,
    bad temperatures, a token out of range): those get accept length -1,
    valid 0 and proposals -1; the valid ones match the oracle, also relaxed."""
    from speculative_verify_accept_02_b300 import isd_verify_propose
    V = 300
    Ls = [2, 0, 33, 2, 2, 2, 1, 3, 4]
    temps = np.array([1.0, 1.0, 1.0, -0.5, np.nan, 1.0, 1e-40, 0.0, 0.7], np.float32)
    C = len(Ls)
    offs = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    total = int(offs[-1])
    g = torch.Generator().manual_seed(5)
    P = torch.randn(total + C, V, generator=g).to(torch.bfloat16)
    Q = P[[int(offs[i]) + i + k for i in range(C) for k in range(Ls[i])]].clone()  # q == p: all accept
    Qn = torch.randn(total, V, generator=g).to(torch.bfloat16)
    tokens = torch.empty(total, dtype=torch.int32)
    for i in range(C):
        for k in range(Ls[i]):
            tokens[offs[i] + k] = int(torch.argmax(P[offs[i] + i + k].float()))  # accepted at T = 0 too
    tokens[offs[5] + 1] = V
    d = "cuda"
    hp, hq, hn = workloads.host_logits(P), workloads.host_logits(Q), workloads.host_logits(Qn)
    for tau in (0.0, 0.5):
        v, pr = isd_verify_propose(P.to(d), Q.to(d), tokens.to(d), Qn.to(d), torch.from_numpy(offs).to(d),
                                   torch.from_numpy(temps).to(d), 2, 9, total=total, tau=tau)
        torch.cuda.synchronize()
        gv = dict(accept_len=v.accept_len.cpu().numpy(), out_tokens=v.out_tokens.cpu().numpy(),
                  ratio=v.ratio.cpu().numpy(), alpha=v.alpha.cpu().numpy())
        gp = dict(proposals=pr.proposals.cpu().numpy(), valid=pr.valid.cpu().numpy())
        assert list(gv["accept_len"][1:7]) == [-1] * 6
        assert list(gp["valid"]) == [1, 0, 0, 0, 0, 0, 0, 1, 1]
        assert np.all(gp["proposals"][offs[1]:offs[7]] == -1)
        ov = oracle.verify(hp, hq, V, tokens.numpy(), offs, temps, 2, 9, tau=tau)
        compare_verify(ov, gv, offs).check()
        op = oracle.propose(hn, V, offs, temps, 2, 9, accept_len=gv["accept_len"])
        compare_propose(op, gp, offs, seqs=[0, 7, 8]).check()
    # Empty batch: nothing launched, nothing written.
    e = torch.zeros(1, dtype=torch.int32, device=d)
    r, rp = isd_verify_propose(P.to(d), Q.to(d), tokens.to(d), Qn.to(d), e, torch.zeros(0, device=d), total=0)
    assert r.accept_len.numel() == 0 and rp.valid.numel() == 0
