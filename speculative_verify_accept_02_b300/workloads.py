"""Seeded synthetic inputs for the verify-and-propose step.

This module only makes inputs; it holds none of the step's arithmetic (no
ratios, no acceptance, no residuals, no KV-slot bookkeeping).  Both the CUDA
path and the fp64 oracle consume what it makes.  Random draws use torch's own generators (CPU or CUDA)
seeded per workload; proposed tokens are drawn with ``torch.multinomial`` /
``torch.argmax`` as a stand-in for the forward pass that produced them.

The shapes follow the configurations the step is measured on.  The pages
measure on serving runs over MATH-500 / MBPP / LMSYS-Chat / GSM8K with a
trained model; neither is available, so these distributions of LM-head logits
stand in for them.

Layout (shared with the library, see include/isd.h):
  seq_offsets[C+1]  exclusive prefix sum of the per-sequence strides L_i
  p  [sum L + C, ld] anchor logits; position k (1..L_i+1) of sequence i is
                     row seq_offsets[i] + i + k - 1
  q  [sum L, ld]     proposal logits; position k (1..L_i) is row
                     seq_offsets[i] + k - 1 (also the token index)
  qnew [sum L, ld]   this forward's mask-position logits (next proposals)
  tokens [sum L]     previously proposed x_k
  temperature [C]
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

VOCAB = 151936

# name -> (data seed, description)
CONFIGS = {
    "tiny": (1000, "C=1, L=4, V=1024, fp32; p ~ N(0, 2^2); q = p + N(0, 0.5^2); x ~ softmax(q); T=1"),
    "c64": (1001, "C=64, L=8, V=151936, bf16; p ~ N(0,1) with +8 on 5 random ids per row; "
                  "q = p + N(0,1); x ~ softmax(q); T=1"),
    "greedy": (1002, "C=32, L=4, V=151936, bf16, T=0; p as c64; q = p + N(0, 0.3^2); x = argmax q, "
                     "10% replaced by a uniform id other than argmax p"),
    "highconc": (1003, "C=256, L=16, V=151936, bf16, T=0.7; p rank-r logit -1.1 ln r + N(0, 0.5^2) "
                       "under a per-row random permutation; q = p + N(0, 1.5^2); x ~ softmax(q/0.7)"),
    "ragged": (1004, "C=64, L_i ~ U{1..16}, T_i in {0, 0.6, 1.0}, V=151936, bf16; p as c64; "
                     "even i: q == p bitwise, odd i: q = p + N(0,1); x ~ softmax(q/T) (argmax at T=0)"),
}

DEFAULT_SIZES = {
    "tiny": dict(num_seqs=1, stride=4, vocab=1024),
    "c64": dict(num_seqs=64, stride=8, vocab=VOCAB),
    "greedy": dict(num_seqs=32, stride=4, vocab=VOCAB),
    "highconc": dict(num_seqs=256, stride=16, vocab=VOCAB),
    "ragged": dict(num_seqs=64, stride=16, vocab=VOCAB),  # stride = max of U{1..stride}
}


@dataclass
class Batch:
    name: str
    vocab: int
    ld: int
    dtype: torch.dtype
    seq_offsets: torch.Tensor   # int32 [C+1]
    temperature: torch.Tensor   # float32 [C]
    tokens: torch.Tensor        # int32 [sum L]
    p: torch.Tensor             # [sum L + C, ld]
    q: torch.Tensor             # [sum L, ld]
    qnew: torch.Tensor          # [sum L, ld]
    seed: int = 0
    offset: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return self.seq_offsets.numel() - 1

    @property
    def total(self) -> int:
        return int(self.seq_offsets[-1])

    def strides(self):
        o = self.seq_offsets.cpu().tolist()
        return [o[i + 1] - o[i] for i in range(len(o) - 1)]

    def to(self, device):
        f = lambda t: t.to(device)
        return Batch(self.name, self.vocab, self.ld, self.dtype, f(self.seq_offsets),
                     f(self.temperature), f(self.tokens), f(self.p), f(self.q), f(self.qnew),
                     self.seed, self.offset, dict(self.meta))


def _peaked(g, rows, V, device):
    """N(0,1) logits with +8 added on 5 random ids per row."""
    x = torch.randn(rows, V, generator=g, device=device)
    if rows:
        ids = torch.randint(0, V, (rows, 5), generator=g, device=device)
        x.scatter_add_(1, ids, torch.full((rows, 5), 8.0, device=device))
    return x


def _zipf(g, rows, V, device):
    """Rank-r logit -1.1 ln r + N(0, 0.5^2), ids permuted at random per row."""
    ranks = torch.arange(1, V + 1, device=device, dtype=torch.float32)
    base = -1.1 * torch.log(ranks)
    out = torch.empty(rows, V, device=device)
    chunk = 256
    for s in range(0, rows, chunk):
        n = min(chunk, rows - s)
        vals = base.expand(n, V) + 0.5 * torch.randn(n, V, generator=g, device=device)
        perm = torch.argsort(torch.rand(n, V, generator=g, device=device), dim=1)
        out[s:s + n].scatter_(1, perm, vals)
    return out


def _sample(g, logits, T):
    """Stand-in for the proposal mechanism of the previous forward."""
    if T == 0:
        return torch.argmax(logits, dim=1)
    probs = torch.softmax(logits.double() / T, dim=1)
    return torch.multinomial(probs, 1, generator=g).squeeze(1)


def _pad(x: torch.Tensor, ld: int, dtype):
    rows, V = x.shape
    buf = torch.zeros(rows, ld, dtype=dtype, device=x.device)
    buf[:, :V] = x.to(dtype)
    return buf


def make(name: str, device="cpu", num_seqs: Optional[int] = None, stride: Optional[int] = None,
         vocab: Optional[int] = None, ld: Optional[int] = None, seed: Optional[int] = None,
         dtype: Optional[torch.dtype] = None) -> Batch:
    """Build one named workload, optionally at other sizes (tests use smaller
    batches of the same distributions).  ``ld`` > vocab pads every row."""
    if name not in CONFIGS:
        raise KeyError(name)
    sizes = dict(DEFAULT_SIZES[name])
    if num_seqs is not None:
        sizes["num_seqs"] = num_seqs
    if stride is not None:
        sizes["stride"] = stride
    if vocab is not None:
        sizes["vocab"] = vocab
    C, Lmax, V = sizes["num_seqs"], sizes["stride"], sizes["vocab"]
    data_seed = CONFIGS[name][0] if seed is None else seed
    if dtype is None:
        dtype = torch.float32 if name == "tiny" else torch.bfloat16
    ld = V if ld is None else ld
    if ld < V:
        raise ValueError("ld must be >= vocab")
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(data_seed)

    # Strides and temperatures.
    if name == "ragged":
        L = torch.randint(1, Lmax + 1, (C,), generator=g, device=device).cpu()
        T = torch.tensor([0.0, 0.6, 1.0])[torch.randint(0, 3, (C,), generator=g, device=device).cpu()]
    else:
        L = torch.full((C,), Lmax, dtype=torch.int64)
        T = torch.full((C,), {"greedy": 0.0, "highconc": 0.7}.get(name, 1.0))
    offs = torch.zeros(C + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(L, 0)
    total = int(offs[-1])
    Ls = L.tolist()

    # Anchor logits, all L_i + 1 rows per sequence.
    rows_p = total + C
    if name == "tiny":
        p32 = 2.0 * torch.randn(rows_p, V, generator=g, device=device)
    elif name == "highconc":
        p32 = _zipf(g, rows_p, V, device)
    else:
        p32 = _peaked(g, rows_p, V, device)
    p = p32.to(dtype)

    # Proposal logits: q_k = p_k + noise (p_k = the anchor row of position k).
    prow = torch.cat([torch.arange(int(offs[i]) + i, int(offs[i]) + i + Ls[i]) for i in range(C)]) \
        if C else torch.zeros(0, dtype=torch.int64)
    prow = prow.to(device)
    base = p[prow].float()
    sigma = {"tiny": 0.5, "c64": 1.0, "greedy": 0.3, "highconc": 1.5, "ragged": 1.0}[name]
    q32 = base + sigma * torch.randn(total, V, generator=g, device=device)
    q = q32.to(dtype)
    if name == "ragged":
        # Even sequences: q is a bit copy of p (the all-accept invariant).
        for i in range(0, C, 2):
            s = int(offs[i])
            q[s:s + Ls[i]] = p[s + i:s + i + Ls[i]]

    # Proposed tokens, drawn from the proposal distribution that made them.
    toks = torch.empty(total, dtype=torch.int64, device=device)
    for i in range(C):
        s, n = int(offs[i]), Ls[i]
        toks[s:s + n] = _sample(g, q[s:s + n].float(), float(T[i]))
    if name == "greedy" and total:
        # 10% of the proposals become a uniformly drawn id that is not argmax p.
        pick = torch.rand(total, generator=g, device=device) < 0.10
        amax = torch.argmax(p[prow].float(), dim=1)
        other = torch.randint(0, V - 1, (total,), generator=g, device=device)
        other = other + (other >= amax).to(other.dtype)
        toks = torch.where(pick, other, toks)

    # This forward's mask-position logits for the next stride (same recipe as q).
    if name == "tiny":
        qn32 = 2.0 * torch.randn(total, V, generator=g, device=device)
    elif name == "highconc":
        qn32 = _zipf(g, total, V, device)
    else:
        qn32 = _peaked(g, total, V, device)
    qn32 = qn32 + sigma * torch.randn(total, V, generator=g, device=device)

    return Batch(name=name, vocab=V, ld=ld, dtype=dtype,
                 seq_offsets=offs.to(torch.int32).to(device),
                 temperature=T.to(torch.float32).to(device),
                 tokens=toks.to(torch.int32),
                 p=_pad(p.float(), ld, dtype) if ld != V else p,
                 q=_pad(q.float(), ld, dtype) if ld != V else q,
                 qnew=_pad(qn32, ld, dtype),
                 seed=0, offset=0, meta=dict(data_seed=data_seed, description=CONFIGS[name][1]))


def host_logits(t: torch.Tensor):
    """A host numpy view of a logit tensor in the form the oracle takes:
    bf16 as uint16 bit patterns, fp32 as float32 (row padding kept)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


# ---------------------------------------------------------------------------
# KV-slot state of a stationary batch (inputs of isd_kv_commit)
# ---------------------------------------------------------------------------

KV_FIELDS = ("table", "seq_len", "pend", "alloc", "free_slots", "free_top")


@dataclass
class KVState:
    """KV-slot state of a stationary batch, as int32 host arrays (layout of
    isd_kv_commit in include/isd.h):

    table      [C, ld]  slot id of each cached position, -1 where empty
    seq_len    [C]      committed positions per sequence
    pend       [C]      proposals the forward in flight verifies
    alloc      [C]      entries the forward in flight writes (0: none yet)
    free_slots [pool]   stack of free slots; free_slots[:free_top] are free
    free_top   [1]
    """
    table: np.ndarray
    seq_len: np.ndarray
    pend: np.ndarray
    alloc: np.ndarray
    free_slots: np.ndarray
    free_top: np.ndarray

    @property
    def num_seqs(self) -> int:
        return self.table.shape[0]

    @property
    def ld(self) -> int:
        return self.table.shape[1]

    @property
    def pool_size(self) -> int:
        return self.free_slots.size

    def copy(self) -> "KVState":
        return KVState(*(getattr(self, f).copy() for f in KV_FIELDS))

    def equal(self, other) -> bool:
        return all(np.array_equal(getattr(self, f), getattr(other, f)) for f in KV_FIELDS)

    def to_torch(self, device) -> dict:
        return {f: torch.from_numpy(getattr(self, f).copy()).to(device) for f in KV_FIELDS}

    @staticmethod
    def from_torch(tensors: dict) -> "KVState":
        return KVState(*(tensors[f].detach().cpu().numpy().astype(np.int32, copy=True) for f in KV_FIELDS))


def make_kv_state(num_seqs: int, max_len: int, pool_size: int, committed, seed: int = 0) -> KVState:
    """Admitted sequences with `committed[i]` cached positions each (the
    prompt, already prefilled) on slots drawn from a seeded permutation of
    the pool; the remaining slots form the free stack in that permuted order.
    Nothing is in flight (pend = alloc = 0)."""
    committed = np.broadcast_to(np.asarray(committed, np.int64), (num_seqs,))
    if np.any(committed < 0) or np.any(committed > max_len) or committed.sum() > pool_size:
        raise ValueError("committed lengths do not fit the rows or the pool")
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pool_size).astype(np.int32)
    table = np.full((num_seqs, max_len), -1, np.int32)
    at = 0
    for i in range(num_seqs):
        n = int(committed[i])
        table[i, :n] = perm[at:at + n]
        at += n
    free = np.full(pool_size, -1, np.int32)
    rest = perm[at:]
    free[:rest.size] = rest
    return KVState(table, committed.astype(np.int32), np.zeros(num_seqs, np.int32),
                   np.zeros(num_seqs, np.int32), free, np.array([rest.size], np.int32))


def draw_accept_lengths(rng: np.random.Generator, pend: np.ndarray, alpha: float) -> np.ndarray:
    """Stand-in for a verify call's accept lengths: each of the pend[i]
    proposals passes with probability alpha until the first failure.
    Entries of sequences with nothing pending hold arbitrary values (the
    commit ignores them)."""
    pend = np.asarray(pend)
    a = np.zeros(pend.size, np.int32)
    for i, L in enumerate(pend):
        if L == 0:
            a[i] = rng.integers(-100, 100)
            continue
        k = 0
        while k < L and rng.random() < alpha:
            k += 1
        a[i] = k
    return a
