"""The decode loop of Introspective Strided Decoding around the verify and
propose calls, over a table-driven synthetic model, and its tokens per
forward (TPF).

"Introspective Diffusion Language Models | Summary", §3.2 and Appendix B.1:
  - a proposal-only step (after prefill, and after every rejection) yields
    one token from the causal anchor and N-1 proposals from mask positions;
  - a fused step verifies the N-1 pending proposals against their anchors
    and proposes the next N-1: all accepted -> N tokens (the proposals and a
    bonus token from the final anchor) and the new proposals stand; a
    rejection after a accepted -> a+1 tokens (the correction last) and the
    next step is proposal-only;
  - under a uniform acceptance probability p the renewal argument gives
    TPF_N = (2 + p + ... + p^(N-2)) / (2 - p^(N-1)).

The synthetic model stands in for the forward pass.  Its anchor and proposal
distributions at absolute position t of sequence i are fixed table entries
(chosen by a hash of (i, t)), built so that every proposal is accepted with
probability exactly ``alpha``: the proposal distribution q is uniform on a
support S of size s, the anchor p puts mass alpha uniformly on S and 1-alpha
uniformly on a disjoint support S', hence sum_v min(p_v, q_v) = alpha.  The
logits are what a forward would hand to the step; everything the method
computes on them runs in the library's kernels.

The loop itself is host orchestration: it gathers each step's rows, calls
``isd_verify`` for the sequences with pending proposals and ``isd_propose``
for every sequence that proposes, reads back the accept lengths and
proposals, and advances per-sequence state.  The Philox offset advances by
one per step.

With ``kv_len`` set, the loop also keeps the batch's KV-slot state and runs
``isd_kv_commit`` after every step (§3.3: the stationary-batch loop's batched
slot scatter and trim of rejected and masked entries): each sequence starts
with one prompt token (x_last) and nothing cached, so after every step its
cache holds exactly the tokens it has emitted (all but the newest, plus the
prompt token).
"""
from dataclasses import dataclass, field
from typing import List

import numpy as np
import torch


def tpf_isd(n: int, p: float) -> float:
    """Tokens per forward of ISD at stride n under uniform acceptance p
    (Summary, Appendix B.1)."""
    num = 2.0 + sum(p ** k for k in range(1, n - 1))
    return num / (2.0 - p ** (n - 1))


class TableModel:
    """Anchor and proposal logits of a synthetic model with uniform
    acceptance probability ``alpha`` (at temperature 1).

    entries: number of table entries; each entry has its own random supports.
    The tables live on ``device`` in float32 (logits -inf off the supports).
    """

    def __init__(self, vocab: int, alpha: float, entries: int = 64, support: int = 64, seed: int = 0,
                 device="cpu"):
        if not 0.0 <= alpha <= 1.0:
            raise ValueError("alpha must lie in [0, 1]")
        if 2 * support > vocab:
            raise ValueError("vocab must hold two disjoint supports")
        self.vocab, self.alpha, self.entries, self.seed = vocab, float(alpha), entries, seed
        g = torch.Generator().manual_seed(seed)
        P = torch.full((entries, vocab), -float("inf"), dtype=torch.float64)
        Q = torch.full((entries, vocab), -float("inf"), dtype=torch.float64)
        for e in range(entries):
            perm = torch.randperm(vocab, generator=g)
            S, S2 = perm[:support], perm[support:2 * support]
            Q[e, S] = 0.0
            if alpha > 0.0:
                P[e, S] = np.log(alpha / support)
            if alpha < 1.0:
                P[e, S2] = np.log((1.0 - alpha) / support)
        self.P = P.to(torch.float32).to(device)
        self.Q = Q.to(torch.float32).to(device)

    def entry(self, seq: np.ndarray, pos: np.ndarray) -> np.ndarray:
        """Table entry of (sequence, absolute position): a fixed integer hash."""
        h = (seq.astype(np.int64) * 1000003 + pos.astype(np.int64) * 10007 + self.seed * 7919) % 2147483647
        h = (h * 48271) % 2147483647
        return (h % self.entries).astype(np.int64)

    def anchor_rows(self, seq, pos) -> torch.Tensor:
        idx = torch.as_tensor(self.entry(np.asarray(seq), np.asarray(pos)), device=self.P.device)
        return self.P.index_select(0, idx)

    def proposal_rows(self, seq, pos) -> torch.Tensor:
        idx = torch.as_tensor(self.entry(np.asarray(seq), np.asarray(pos)), device=self.Q.device)
        return self.Q.index_select(0, idx)


class CudaBackend:
    """The library's entry points (isd_verify, isd_propose, isd_kv_commit)
    on CUDA tensors."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)

    def kv_state(self, state):
        return state.to_torch(self.device)

    def kv_commit(self, handle, accept, num_masks) -> int:
        from .api import isd_kv_commit
        acc = torch.as_tensor(np.asarray(accept, np.int32), device=self.device)
        return int(isd_kv_commit(handle, acc, num_masks).item())

    def kv_read(self, handle):
        from .workloads import KVState
        return KVState.from_torch(handle)

    def verify(self, p, q, tokens, offs, temp, seed, offset, filters=None):
        from .api import isd_verify, isd_verify_filtered
        d = self.device
        args = (p.to(d), q.to(d), torch.as_tensor(tokens, dtype=torch.int32, device=d),
                torch.as_tensor(offs, dtype=torch.int32, device=d),
                torch.as_tensor(temp, dtype=torch.float32, device=d), seed, offset)
        if filters is None:
            out = isd_verify(*args, total=int(offs[-1]))
        else:
            out = isd_verify_filtered(*args, top_k=filters[0], top_p=filters[1], total=int(offs[-1]))
        return out.accept_len.cpu().numpy(), out.out_tokens.cpu().numpy()

    def propose(self, qnew, offs, temp, seed, offset, filters=None):
        from .api import isd_propose, isd_propose_filtered
        d = self.device
        args = (qnew.to(d), torch.as_tensor(offs, dtype=torch.int32, device=d),
                torch.as_tensor(temp, dtype=torch.float32, device=d), seed, offset)
        if filters is None:
            out = isd_propose(*args, total=int(offs[-1]))
        else:
            out = isd_propose_filtered(*args, top_k=filters[0], top_p=filters[1], total=int(offs[-1]))
        return out.proposals.cpu().numpy(), out.valid.cpu().numpy()


@dataclass
class LoopStats:
    steps: int = 0
    forwards: int = 0           # one per active sequence per step
    tokens: int = 0             # emitted tokens
    verify_steps: int = 0       # forwards that verified proposals
    accepted: int = 0           # accepted proposals
    rejected: int = 0           # rejected proposals (at most one per fused step)
    verified: int = 0           # proposals pending at fused steps
    per_seq_tokens: List[int] = field(default_factory=list)

    @property
    def tpf(self) -> float:
        return self.tokens / self.forwards if self.forwards else float("nan")

    @property
    def acceptance(self) -> float:
        """Accepted over tested proposals: the per-proposal acceptance rate."""
        tested = self.accepted + self.rejected
        return self.accepted / tested if tested else float("nan")


class ISDLoop:
    """C sequences decoded with stride n (n-1 proposals per step) by ISD.

    backend: an object with verify(p, q, tokens, offs, temp, seed, offset,
    filters) -> (accept_len, out_tokens) and propose(qnew, offs, temp, seed,
    offset, filters) -> (proposals, valid), over the library's layout
    (include/isd.h).  filters: (top_k, top_p) to decode under the evaluation
    setting's sampling filters (include/isd_filter.h), or None.
    """

    def __init__(self, model: TableModel, num_seqs: int, stride: int, backend, seed: int = 0,
                 kv_len: int = 0, filters=None):
        if not 2 <= stride <= 32:
            raise ValueError("stride n must lie in [2, 32] (n - 1 proposals, one anchor row more)")
        self.model, self.C, self.n, self.backend, self.seed = model, num_seqs, stride, backend, seed
        self.pos = np.zeros(num_seqs, np.int64)        # tokens emitted so far
        self.pending = [None] * num_seqs              # proposals awaiting verification
        self.tokens: List[List[int]] = [[] for _ in range(num_seqs)]
        self.stats = LoopStats(per_seq_tokens=[0] * num_seqs)
        self.offset = 0
        self.filters = filters  # (top_k, top_p) of the evaluation setting, or None
        self.kv = None
        if kv_len:
            # every row holds the cache of kv_len positions; the pool backs all rows
            from .workloads import make_kv_state
            self.kv = backend.kv_state(make_kv_state(num_seqs, kv_len, num_seqs * kv_len, 0, seed=seed))
            self._kv_commit(np.zeros(num_seqs, np.int32))  # admission: the first forward's slots

    def _kv_commit(self, accept):
        status = self.backend.kv_commit(self.kv, accept, self.n - 1)
        if status != 0:
            raise RuntimeError(f"isd_kv_commit refused the step (status {status})")

    def _propose(self, jobs):
        """One isd_propose call for every proposing sequence of the step, so
        that each draws from its own Philox counters.  jobs: (sequence, first
        position, with_anchor) -- with_anchor: the anchor token at the first
        position comes first (a proposal-only step), then n-1 proposals for
        the positions after it."""
        L = self.n - 1
        seq_ids, pos_ids, is_anchor, offs = [], [], [], [0]
        for i, t, anchor in jobs:
            m = L + 1 if anchor else L
            seq_ids += [i] * m
            pos_ids += [t + k for k in range(m)]
            is_anchor += [anchor and k == 0 for k in range(m)]
            offs.append(offs[-1] + m)
        seq_ids, pos_ids = np.asarray(seq_ids), np.asarray(pos_ids)
        A = self.model.anchor_rows(seq_ids, pos_ids)
        Qr = self.model.proposal_rows(seq_ids, pos_ids)
        rows = torch.where(torch.as_tensor(is_anchor, device=A.device)[:, None], A, Qr)
        offs = np.asarray(offs, dtype=np.int32)
        temp = np.ones(len(jobs), np.float32)
        props, valid = self.backend.propose(rows, offs, temp, self.seed, self.offset, filters=self.filters)
        assert np.all(valid == 1)
        return [props[offs[j]:offs[j + 1]] for j in range(len(jobs))]

    def step(self):
        L = self.n - 1
        st = self.stats
        kv_accept = np.zeros(self.C, np.int32)         # by batch position, read where proposals were pending
        ver = [i for i in range(self.C) if self.pending[i] is not None]
        jobs = [(i, int(self.pos[i]), True) for i in range(self.C) if self.pending[i] is None]
        if ver:  # fused steps: verify the pending proposals
            seq_ids = np.repeat(ver, L + 1)
            pos_ids = np.concatenate([self.pos[i] + np.arange(L + 1) for i in ver])
            p = self.model.anchor_rows(seq_ids, pos_ids)
            qseq = np.repeat(ver, L)
            qpos = np.concatenate([self.pos[i] + np.arange(L) for i in ver])
            q = self.model.proposal_rows(qseq, qpos)
            toks = np.concatenate([self.pending[i] for i in ver]).astype(np.int32)
            offs = np.arange(len(ver) + 1, dtype=np.int32) * L
            temp = np.ones(len(ver), np.float32)
            acc, out = self.backend.verify(p, q, toks, offs, temp, self.seed, self.offset, filters=self.filters)
            assert np.all(acc >= 0), acc
            for j, i in enumerate(ver):
                a = int(acc[j])
                kv_accept[i] = a
                emitted = out[j * (L + 1): j * (L + 1) + a + 1]
                self.tokens[i].extend(int(x) for x in emitted)
                st.tokens += a + 1
                st.per_seq_tokens[i] += a + 1
                st.accepted += a
                st.rejected += 1 if a < L else 0
                st.verified += L
                self.pos[i] += a + 1
                self.pending[i] = None
                if a == L:  # the fused step's mask positions propose the next stride
                    jobs.append((i, int(self.pos[i]), False))
            st.verify_steps += len(ver)
        if jobs:
            for (i, _, anchor), props in zip(jobs, self._propose(jobs)):
                if anchor:  # proposal-only step: the anchor token is emitted
                    self.tokens[i].append(int(props[0]))
                    st.tokens += 1
                    st.per_seq_tokens[i] += 1
                    self.pos[i] += 1
                    props = props[1:]
                self.pending[i] = np.asarray(props, dtype=np.int32)
        if self.kv is not None:
            self._kv_commit(kv_accept)
        st.forwards += self.C
        st.steps += 1
        self.offset += 1
        return st

    def run(self, steps: int) -> LoopStats:
        for _ in range(steps):
            self.step()
        return self.stats


def main():
    import argparse
    import json
    import time
    ap = argparse.ArgumentParser(description="ISD decode loop on the library: measured TPF against "
                                             "the closed form, and time per step")
    ap.add_argument("--stride", type=int, default=4)
    ap.add_argument("--alpha", type=float, default=0.6)
    ap.add_argument("--num-seqs", type=int, default=64)
    ap.add_argument("--vocab", type=int, default=151936)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--kv", action="store_true", help="keep the batch's KV-slot state with isd_kv_commit")
    args = ap.parse_args()
    model = TableModel(args.vocab, args.alpha, device="cuda")
    kv_len = 1 + (args.steps + 3) * args.stride + 2 * args.stride if args.kv else 0
    loop = ISDLoop(model, args.num_seqs, args.stride, CudaBackend(), kv_len=kv_len)
    loop.run(3)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    loop.run(args.steps)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    st = loop.stats
    per = np.asarray(st.per_seq_tokens) / st.steps
    print(json.dumps({"stride": args.stride, "alpha": args.alpha, "num_seqs": args.num_seqs,
                      "steps": st.steps, "tpf": st.tpf, "tpf_closed_form": tpf_isd(args.stride, args.alpha),
                      "tpf_stderr": float(per.std(ddof=1) / np.sqrt(len(per))),
                      "acceptance": st.acceptance, "kv_commit": bool(args.kv),
                      "host_loop_ms_per_step": 1e3 * dt / args.steps}))


if __name__ == "__main__":
    main()
