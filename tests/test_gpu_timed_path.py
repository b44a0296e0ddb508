"""The call the benchmark times, isd_verify_propose (the fused step of
"Introspective Diffusion Language Models | Summary", §3.2: one forward
verifies the stride and proposes the next), against the fp64 oracle at the
benchmark's own sizes; its Gumbel-max sampler mode (§3.3: the fused kernel
draws by Gumbel-max); and the bounded-wait failure path.

Full-size comparisons check a sample of sequences one by one; the sample
always holds the last four sequences of the batch, whose decisions, tail
pieces and draws come last in the stream.  The bar is parity.py's (bit-exact
accept lengths, emitted tokens and proposals; ratios and alpha within 1e-4
relative; decisions with an oracle margin below 1e-5 exempted, counted and
printed).  For the Gumbel-max sampler the margin of a draw is the gap between
the two best Gumbel scores.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import Report, compare_propose, compare_verify
from speculative_verify_accept_02_b300 import build, isd_verify_propose, isd_verify_propose_workspace_bytes, workloads
from speculative_verify_accept_02_b300.api import isd_debug_verify_stall, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()


def host(batch):
    return dict(p=workloads.host_logits(batch.p), q=workloads.host_logits(batch.q),
                qnew=workloads.host_logits(batch.qnew), tokens=batch.tokens.cpu().numpy(),
                offs=batch.seq_offsets.cpu().numpy(), temp=batch.temperature.cpu().numpy())


def fused(b, seed, offset, tau=0.0, sampler="icdf", ws=None):
    v, pr = isd_verify_propose(b.p, b.q, b.tokens, b.qnew, b.seq_offsets, b.temperature, seed, offset,
                               vocab=b.vocab, total=b.total, tau=tau, sampler=sampler, ws=ws)
    torch.cuda.synchronize()
    gv = dict(accept_len=v.accept_len.cpu().numpy(), out_tokens=v.out_tokens.cpu().numpy(),
              ratio=v.ratio.cpu().numpy(), alpha=v.alpha.cpu().numpy())
    gp = dict(proposals=pr.proposals.cpu().numpy(), valid=pr.valid.cpu().numpy())
    return gv, gp


def sample(C, n=8, seed=11):
    """The first sequence, the last four, and n more at random."""
    rng = np.random.default_rng(seed)
    return sorted(set([0] + list(range(max(0, C - 4), C)) + list(rng.choice(C, size=min(C, n), replace=False))))


def check_layout(gv, gp, h, vocab):
    """Properties of the fused outputs that hold at any size, on every sequence."""
    acc = gv["accept_len"]
    L = np.diff(h["offs"])
    assert np.all((acc >= 0) & (acc <= L))
    assert np.array_equal(gp["valid"], (acc == L).astype(np.uint8))
    for i in range(L.size):
        s, e = h["offs"][i], h["offs"][i + 1]
        slots = gv["out_tokens"][s + i: e + i + 1]
        assert np.array_equal(slots[:acc[i]], h["tokens"][s: s + acc[i]])
        assert 0 <= slots[acc[i]] < vocab and np.all(slots[acc[i] + 1:] == -1)
        props = gp["proposals"][s:e]
        assert np.all((props >= 0) & (props < vocab)) if gp["valid"][i] else np.all(props == -1)


@pytest.mark.parametrize("name,tau", [("c64", 0.0), ("c64", 0.5), ("highconc", 0.0)])
def test_timed_call_full_size(name, tau):
    """isd_verify_propose on the full batch the benchmark times (c64: C=64;
    highconc: C=256), strict and relaxed (tau = 0.5), against oracle.verify
    and oracle.propose with the GPU's accept lengths."""
    batch = workloads.make(name, device="cuda")
    h = host(batch)
    rep = Report()
    for seed, offset in ((0, 0), (7, 3)):
        gv, gp = fused(batch, seed, offset, tau=tau)
        check_layout(gv, gp, h, batch.vocab)
        seqs = sample(batch.num_seqs, seed=seed + 11)
        ov = oracle.verify(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], seed, offset,
                           seqs=seqs, tau=tau)
        compare_verify(ov, gv, h["offs"], seqs=seqs, report=rep)
        agree = [i for i in seqs if ov["accept_len"][i] == gv["accept_len"][i]]
        op = oracle.propose(h["qnew"], batch.vocab, h["offs"], h["temp"], seed, offset,
                            accept_len=gv["accept_len"], seqs=agree)
        compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
    print(f"\n{name} tau={tau}: {rep.summary()}")
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep.summary()


GUMBEL = [("c64", dict(num_seqs=5)), ("greedy", dict(num_seqs=6)), ("highconc", dict(num_seqs=4)),
          ("ragged", dict(num_seqs=16)), ("ragged", dict(num_seqs=12, vocab=1537, dtype=torch.float32)),
          ("tiny", dict(num_seqs=6, vocab=5)), ("c64", dict(num_seqs=3, stride=32, vocab=4099)),
          ("c64", dict(num_seqs=4, vocab=5000, ld=5003))]


def compare_gumbel(batch, seed, offset, rep):
    h = host(batch)
    gv, gp = fused(batch.to("cuda"), seed, offset, sampler="gumbel")
    ov = oracle.verify_gumbel(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], seed, offset)
    compare_verify(ov, gv, h["offs"], report=rep)
    agree = [i for i in range(batch.num_seqs) if ov["accept_len"][i] == gv["accept_len"][i]]
    op = oracle.propose_gumbel(h["qnew"], batch.vocab, h["offs"], h["temp"], seed, offset,
                               accept_len=gv["accept_len"])
    compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
    return gv, gp, h


@pytest.mark.parametrize("name,kw", GUMBEL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(GUMBEL)])
def test_gumbel_sampler_parity(name, kw):
    """isd_verify_propose_gumbel: acceptance as the inverse-CDF call, the
    correction, bonus and proposal draws by Gumbel-max over the residual,
    p_{L+1} and softmax(qnew / T), against Oracle.verify_gumbel and
    propose_gumbel."""
    batch = workloads.make(name, **kw)
    rep = Report()
    for seed, offset in ((0, 0), (7, 3)):
        compare_gumbel(batch, seed, offset, rep)
    print(f"\n{name} gumbel: {rep.summary()}")
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep.summary()


def test_gumbel_sampler_full_size():
    """The Gumbel-max mode on the full c64 batch, every sequence compared;
    its ratios are the inverse-CDF call's (up to the rounding of partials
    merged in another order: the stream kernel deals its chunks dynamically)."""
    batch = workloads.make("c64", device="cuda")
    rep = Report()
    gv, gp, h = compare_gumbel(batch, 0, 0, rep)
    check_layout(gv, gp, h, batch.vocab)
    iv, _ = fused(batch, 0, 0)
    assert np.allclose(iv["ratio"], gv["ratio"], rtol=1e-5, atol=0.0)
    print(f"\nc64 gumbel full: {rep.summary()}")
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep.summary()


def test_bounded_wait_runs_out_then_recovers():
    """Failure detection without a GPU fault: the check hook holds back one
    sequence's correction draw, the workers that take its pieces poll for a
    descriptor that never comes, and their bound (200 us here) runs out.  The
    call then reports a timeout (every accept length -2, every valid flag 0,
    the workspace's error word set); after the workspace is zero-filled the
    next ordinary call equals the oracle."""
    batch = workloads.make("c64", num_seqs=12, vocab=20000, device="cuda")
    b = batch
    C, total, V = b.num_seqs, b.total, b.vocab
    ws = workspace(isd_verify_propose_workspace_bytes(C, total, V, b.dtype), torch.device("cuda"))
    stall = 5
    assert float(b.temperature[stall]) > 0.0
    v, pr = isd_debug_verify_stall(b.p, b.q, b.tokens, b.qnew, b.seq_offsets, b.temperature, 0, 0, stall,
                                   200_000, total=total, ws=ws)
    torch.cuda.synchronize()
    assert np.all(v.accept_len.cpu().numpy() == -2)
    assert np.all(pr.valid.cpu().numpy() == 0)
    assert int(ws[:4].view(torch.int32)[0]) != 0  # the control block's error word leads the workspace
    ws.zero_()
    gv, gp = fused(b, 0, 0, ws=ws)
    h = host(batch)
    ov = oracle.verify(h["p"], h["q"], V, h["tokens"], h["offs"], h["temp"], 0, 0)
    rep = compare_verify(ov, gv, h["offs"])
    agree = [i for i in range(C) if ov["accept_len"][i] == gv["accept_len"][i]]
    op = oracle.propose(h["qnew"], V, h["offs"], h["temp"], 0, 0, accept_len=gv["accept_len"])
    compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
    rep.check()
    # The same hook with no sequence held back is an ordinary call.
    ws.zero_()
    v2, pr2 = isd_debug_verify_stall(b.p, b.q, b.tokens, b.qnew, b.seq_offsets, b.temperature, 0, 0, -1,
                                     4_000_000_000, total=total, ws=ws)
    torch.cuda.synchronize()
    assert np.array_equal(v2.accept_len.cpu().numpy(), gv["accept_len"])
    assert np.array_equal(v2.out_tokens.cpu().numpy(), gv["out_tokens"])


def test_fused_step_replays_from_a_cuda_graph():
    """isd_verify_propose captured once in a CUDA graph (both launches and the
    programmatic dependency between them) and replayed on new inputs copied
    into the captured buffers: the call allocates nothing and never
    synchronises, and every call leaves the workspace ready for the next (its
    counters, queue and tail words re-zeroed; its partials rewritten by the
    next stream), so every replay equals the oracle on the inputs it saw."""
    from speculative_verify_accept_02_b300.api import ProposeOut, VerifyOut
    a = workloads.make("c64", num_seqs=6, vocab=20000, seed=1)
    b = workloads.make("c64", num_seqs=6, vocab=20000, seed=2)
    assert torch.equal(a.seq_offsets, b.seq_offsets) and torch.equal(a.temperature, b.temperature)
    assert not torch.equal(a.p, b.p)
    x = a.to("cuda")  # the buffers the graph reads
    dev = x.p.device
    C, total, V = x.num_seqs, x.total, x.vocab
    i32 = torch.int32
    out = VerifyOut(torch.empty(C, dtype=i32, device=dev), torch.empty(total + C, dtype=i32, device=dev),
                    torch.empty(total, dtype=torch.float32, device=dev), torch.empty(C, dtype=torch.float32, device=dev))
    pout = ProposeOut(torch.empty(total, dtype=i32, device=dev), torch.empty(C, dtype=torch.uint8, device=dev))
    ws = workspace(isd_verify_propose_workspace_bytes(C, total, V, x.dtype), dev)
    seed, offset = 3, 5

    def step():
        isd_verify_propose(x.p, x.q, x.tokens, x.qnew, x.seq_offsets, x.temperature, seed, offset,
                           vocab=V, total=total, out=out, pout=pout, ws=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # one ordinary call first, outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    rep = Report()
    for batch in (b, a, b):
        for dst, src in ((x.p, batch.p), (x.q, batch.q), (x.qnew, batch.qnew), (x.tokens, batch.tokens)):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        gv = dict(accept_len=out.accept_len.cpu().numpy(), out_tokens=out.out_tokens.cpu().numpy(),
                  ratio=out.ratio.cpu().numpy(), alpha=out.alpha.cpu().numpy())
        gp = dict(proposals=pout.proposals.cpu().numpy(), valid=pout.valid.cpu().numpy())
        h = host(batch)
        check_layout(gv, gp, h, V)
        ov = oracle.verify(h["p"], h["q"], V, h["tokens"], h["offs"], h["temp"], seed, offset)
        compare_verify(ov, gv, h["offs"], report=rep)
        agree = [i for i in range(C) if ov["accept_len"][i] == gv["accept_len"][i]]
        op = oracle.propose(h["qnew"], V, h["offs"], h["temp"], seed, offset, accept_len=gv["accept_len"])
        compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
        assert int(ws[:4].view(torch.int32)[0]) == 0  # no wait ran out (the error word leads the workspace)
    print(f"\ngraph replays: {rep.summary()}")
    rep.check()
    assert rep.exempt_accept + rep.exempt_token <= max(1, rep.sequences // 20), rep.summary()
