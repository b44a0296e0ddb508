"""Python binding of libisd: the entry points declared under include/
(isd.h, isd_filter.h, isd_kv.h, isd_debug.h) over torch CUDA tensors.  Argument marshalling only — every step of the computation runs
in the library's kernels; torch supplies device memory and the stream.

Tensors:
  p [sum L + C, ld_p], q [sum L, ld_q], qnew [sum L, ld]: torch.bfloat16 or
      torch.float32 on one CUDA device, unit stride along the vocabulary
      (row padding allowed), base pointer 16-byte aligned;
  tokens [sum L] int32, seq_offsets [C+1] int32, temperature [C] float32.
``total`` (= seq_offsets[-1]) must be passed to avoid a device->host read.
"""
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

_DTYPES = {torch.bfloat16: _lib.ISD_DTYPE_BF16, torch.float32: _lib.ISD_DTYPE_F32}


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"logits must be bfloat16 or float32, not {t.dtype}") from None


def _rows(t: torch.Tensor, name: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit stride along the vocabulary")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr(), t.stride(0)


def _int32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    return t.data_ptr()


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    return t.data_ptr()


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _total(seq_offsets: torch.Tensor, total: Optional[int]) -> int:
    return int(seq_offsets[-1].item()) if total is None else int(total)


def isd_verify_workspace_bytes(num_seqs: int, total: int, vocab: int, dtype: torch.dtype) -> int:
    return int(_lib.load().isd_verify_workspace_bytes(num_seqs, total, vocab, _DTYPES[dtype]))


def isd_propose_workspace_bytes(num_seqs: int, total: int, vocab: int, dtype: torch.dtype) -> int:
    return int(_lib.load().isd_propose_workspace_bytes(num_seqs, total, vocab, _DTYPES[dtype]))


def workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace (torch's allocator aligns to 512)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)


@dataclass
class VerifyOut:
    accept_len: torch.Tensor   # [C] int32
    out_tokens: torch.Tensor   # [sum L + C] int32
    ratio: torch.Tensor        # [sum L] float32
    alpha: torch.Tensor        # [C] float32


@dataclass
class ProposeOut:
    proposals: torch.Tensor    # [sum L] int32
    valid: torch.Tensor        # [C] uint8


def isd_verify(p: torch.Tensor, q: torch.Tensor, tokens: torch.Tensor, seq_offsets: torch.Tensor,
               temperature: torch.Tensor, seed: int = 0, offset: int = 0, *, vocab: Optional[int] = None,
               total: Optional[int] = None, out: Optional[VerifyOut] = None,
               ws: Optional[torch.Tensor] = None, stream=None, tau: float = 0.0) -> VerifyOut:
    """isd_verify; tau > 0 calls isd_verify_relaxed (accept tests use
    min(1, (1 + tau) p/q))."""
    device = p.device
    C = seq_offsets.numel() - 1
    total = _total(seq_offsets, total)
    V = p.shape[1] if vocab is None else int(vocab)
    if p.dtype != q.dtype:
        raise TypeError("p and q must share a dtype")
    pp, ldp = _rows(p, "p")
    qp, ldq = _rows(q, "q")
    if out is None:
        out = VerifyOut(torch.empty(C, dtype=torch.int32, device=device),
                        torch.empty(total + C, dtype=torch.int32, device=device),
                        torch.empty(total, dtype=torch.float32, device=device),
                        torch.empty(C, dtype=torch.float32, device=device))
    need = isd_verify_workspace_bytes(C, total, V, p.dtype)
    if ws is None:
        ws = workspace(need, device)
    head = (pp, ldp, qp, ldq, _dtype_code(p), V, _int32(tokens, "tokens"), _int32(seq_offsets, "seq_offsets"),
            C, total, _f32(temperature, "temperature"), int(seed), int(offset))
    tail = (out.accept_len.data_ptr(), out.out_tokens.data_ptr(), out.ratio.data_ptr(), out.alpha.data_ptr(),
            ws.data_ptr(), ws.numel() * ws.element_size(), _stream(device, stream))
    if tau == 0.0:
        status = _lib.load().isd_verify(*head, *tail)
        _lib.check("isd_verify", status)
    else:
        status = _lib.load().isd_verify_relaxed(*head, float(tau), *tail)
        _lib.check("isd_verify_relaxed", status)
    return out


def isd_verify_propose_workspace_bytes(num_seqs: int, total: int, vocab: int, dtype: torch.dtype) -> int:
    return int(_lib.load().isd_verify_propose_workspace_bytes(num_seqs, total, vocab, _DTYPES[dtype]))


def isd_verify_propose(p: torch.Tensor, q: torch.Tensor, tokens: torch.Tensor, qnew: torch.Tensor,
                       seq_offsets: torch.Tensor, temperature: torch.Tensor, seed: int = 0, offset: int = 0, *,
                       vocab: Optional[int] = None, total: Optional[int] = None, tau: float = 0.0,
                       out: Optional[VerifyOut] = None, pout: Optional[ProposeOut] = None,
                       ws: Optional[torch.Tensor] = None, stream=None, sampler: str = "icdf"):
    """isd_verify_propose: verify and the next stride's proposals in one
    launch; sampler="gumbel" calls isd_verify_propose_gumbel (Gumbel-max
    draws in place of inverse-CDF draws).  Returns (VerifyOut, ProposeOut)."""
    if sampler not in ("icdf", "gumbel"):
        raise ValueError(f"sampler must be 'icdf' or 'gumbel', not {sampler!r}")
    device = p.device
    C = seq_offsets.numel() - 1
    total = _total(seq_offsets, total)
    V = p.shape[1] if vocab is None else int(vocab)
    if p.dtype != q.dtype or qnew.dtype != p.dtype:
        raise TypeError("p, q and qnew must share a dtype")
    pp, ldp = _rows(p, "p")
    qp, ldq = _rows(q, "q")
    np_, ldn = _rows(qnew, "qnew")
    if out is None:
        out = VerifyOut(torch.empty(C, dtype=torch.int32, device=device),
                        torch.empty(total + C, dtype=torch.int32, device=device),
                        torch.empty(total, dtype=torch.float32, device=device),
                        torch.empty(C, dtype=torch.float32, device=device))
    if pout is None:
        pout = ProposeOut(torch.empty(total, dtype=torch.int32, device=device),
                          torch.empty(C, dtype=torch.uint8, device=device))
    need = isd_verify_propose_workspace_bytes(C, total, V, p.dtype)
    if ws is None:
        ws = workspace(need, device)
    name = "isd_verify_propose_gumbel" if sampler == "gumbel" else "isd_verify_propose"
    status = getattr(_lib.load(), name)(
        pp, ldp, qp, ldq, _dtype_code(p), V, _int32(tokens, "tokens"), _int32(seq_offsets, "seq_offsets"),
        C, total, _f32(temperature, "temperature"), int(seed), int(offset), float(tau),
        out.accept_len.data_ptr(), out.out_tokens.data_ptr(), out.ratio.data_ptr(), out.alpha.data_ptr(),
        np_, ldn, pout.proposals.data_ptr(), pout.valid.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), _stream(device, stream))
    _lib.check(name, status)
    return out, pout


def isd_debug_verify_stall(p: torch.Tensor, q: torch.Tensor, tokens: torch.Tensor, qnew: torch.Tensor,
                           seq_offsets: torch.Tensor, temperature: torch.Tensor, seed: int, offset: int,
                           stall_seq: int, wait_ns: int, *, total: int, ws: torch.Tensor,
                           out: Optional[VerifyOut] = None, pout: Optional[ProposeOut] = None, stream=None):
    """isd_debug_verify_stall (include/isd_debug.h): isd_verify_propose with
    the decision of sequence ``stall_seq`` held back and the kernel's waits on
    other CTAs bounded by ``wait_ns``.  Returns (VerifyOut, ProposeOut)."""
    device = p.device
    C = seq_offsets.numel() - 1
    V = p.shape[1]
    pp, ldp = _rows(p, "p")
    qp, ldq = _rows(q, "q")
    np_, ldn = _rows(qnew, "qnew")
    if out is None:
        out = VerifyOut(torch.empty(C, dtype=torch.int32, device=device),
                        torch.empty(total + C, dtype=torch.int32, device=device),
                        torch.empty(total, dtype=torch.float32, device=device),
                        torch.empty(C, dtype=torch.float32, device=device))
    if pout is None:
        pout = ProposeOut(torch.empty(total, dtype=torch.int32, device=device),
                          torch.empty(C, dtype=torch.uint8, device=device))
    status = _lib.load().isd_debug_verify_stall(
        pp, ldp, qp, ldq, _dtype_code(p), V, _int32(tokens, "tokens"), _int32(seq_offsets, "seq_offsets"),
        C, int(total), _f32(temperature, "temperature"), int(seed), int(offset),
        out.accept_len.data_ptr(), out.out_tokens.data_ptr(), out.ratio.data_ptr(), out.alpha.data_ptr(),
        np_, ldn, pout.proposals.data_ptr(), pout.valid.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), int(stall_seq), int(wait_ns), _stream(device, stream))
    _lib.check("isd_debug_verify_stall", status)
    return out, pout


def isd_propose(qnew: torch.Tensor, seq_offsets: torch.Tensor, temperature: torch.Tensor,
                seed: int = 0, offset: int = 0, accept_len: Optional[torch.Tensor] = None, *,
                vocab: Optional[int] = None, total: Optional[int] = None,
                out: Optional[ProposeOut] = None, ws: Optional[torch.Tensor] = None,
                stream=None) -> ProposeOut:
    device = qnew.device
    C = seq_offsets.numel() - 1
    total = _total(seq_offsets, total)
    V = qnew.shape[1] if vocab is None else int(vocab)
    qp, ld = _rows(qnew, "qnew")
    if out is None:
        out = ProposeOut(torch.empty(total, dtype=torch.int32, device=device),
                         torch.empty(C, dtype=torch.uint8, device=device))
    need = isd_propose_workspace_bytes(C, total, V, qnew.dtype)
    if ws is None:
        ws = workspace(need, device)
    acc = None if accept_len is None else _int32(accept_len, "accept_len")
    status = _lib.load().isd_propose(
        qp, ld, _dtype_code(qnew), V, _int32(seq_offsets, "seq_offsets"), C, total,
        _f32(temperature, "temperature"), int(seed), int(offset), acc, out.proposals.data_ptr(),
        out.valid.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(device, stream))
    _lib.check("isd_propose", status)
    return out


def isd_verify_filtered_workspace_bytes(num_seqs: int, total: int, top_k: int) -> int:
    return int(_lib.load().isd_verify_filtered_workspace_bytes(num_seqs, total, top_k))


def isd_propose_filtered_workspace_bytes(num_seqs: int, total: int, top_k: int) -> int:
    return int(_lib.load().isd_propose_filtered_workspace_bytes(num_seqs, total, top_k))


def isd_verify_filtered(p: torch.Tensor, q: torch.Tensor, tokens: torch.Tensor, seq_offsets: torch.Tensor,
                        temperature: torch.Tensor, seed: int = 0, offset: int = 0, *, top_k: int = 50,
                        top_p: float = 0.95, vocab: Optional[int] = None, total: Optional[int] = None,
                        out: Optional[VerifyOut] = None, ws: Optional[torch.Tensor] = None,
                        stream=None) -> VerifyOut:
    """isd_verify_filtered: isd_verify with p and q under the top-k, then
    top-p filters (include/isd_filter.h)."""
    device = p.device
    C = seq_offsets.numel() - 1
    total = _total(seq_offsets, total)
    V = p.shape[1] if vocab is None else int(vocab)
    if p.dtype != q.dtype:
        raise TypeError("p and q must share a dtype")
    pp, ldp = _rows(p, "p")
    qp, ldq = _rows(q, "q")
    if out is None:
        out = VerifyOut(torch.empty(C, dtype=torch.int32, device=device),
                        torch.empty(total + C, dtype=torch.int32, device=device),
                        torch.empty(total, dtype=torch.float32, device=device),
                        torch.empty(C, dtype=torch.float32, device=device))
    if ws is None:
        ws = workspace(isd_verify_filtered_workspace_bytes(C, total, top_k), device)
    status = _lib.load().isd_verify_filtered(
        pp, ldp, qp, ldq, _dtype_code(p), V, _int32(tokens, "tokens"), _int32(seq_offsets, "seq_offsets"),
        C, total, _f32(temperature, "temperature"), int(seed), int(offset), int(top_k), float(top_p),
        out.accept_len.data_ptr(), out.out_tokens.data_ptr(), out.ratio.data_ptr(), out.alpha.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), _stream(device, stream))
    _lib.check("isd_verify_filtered", status)
    return out


def isd_propose_filtered(qnew: torch.Tensor, seq_offsets: torch.Tensor, temperature: torch.Tensor,
                         seed: int = 0, offset: int = 0, accept_len: Optional[torch.Tensor] = None, *,
                         top_k: int = 50, top_p: float = 0.95, vocab: Optional[int] = None,
                         total: Optional[int] = None, out: Optional[ProposeOut] = None,
                         ws: Optional[torch.Tensor] = None, stream=None) -> ProposeOut:
    """isd_propose_filtered: proposals drawn from the filtered softmax(qnew/T)."""
    device = qnew.device
    C = seq_offsets.numel() - 1
    total = _total(seq_offsets, total)
    V = qnew.shape[1] if vocab is None else int(vocab)
    qp, ld = _rows(qnew, "qnew")
    if out is None:
        out = ProposeOut(torch.empty(total, dtype=torch.int32, device=device),
                         torch.empty(C, dtype=torch.uint8, device=device))
    if ws is None:
        ws = workspace(isd_propose_filtered_workspace_bytes(C, total, top_k), device)
    acc = None if accept_len is None else _int32(accept_len, "accept_len")
    status = _lib.load().isd_propose_filtered(
        qp, ld, _dtype_code(qnew), V, _int32(seq_offsets, "seq_offsets"), C, total,
        _f32(temperature, "temperature"), int(seed), int(offset), int(top_k), float(top_p), acc,
        out.proposals.data_ptr(), out.valid.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
        _stream(device, stream))
    _lib.check("isd_propose_filtered", status)
    return out


def isd_alpha(ratio: torch.Tensor, seq_offsets: torch.Tensor, *, total: Optional[int] = None,
              stream=None):
    """Returns (alpha_per_seq [C] float32, alpha_mean [1] float32)."""
    device = ratio.device
    C = seq_offsets.numel() - 1
    total = _total(seq_offsets, total)
    per = torch.empty(C, dtype=torch.float32, device=device)
    mean = torch.empty(1, dtype=torch.float32, device=device)
    status = _lib.load().isd_alpha(_f32(ratio, "ratio"), _int32(seq_offsets, "seq_offsets"), C, total,
                                   per.data_ptr(), mean.data_ptr(), _stream(device, stream))
    _lib.check("isd_alpha", status)
    return per, mean


KV_FIELDS = ("table", "seq_len", "pend", "alloc", "free_slots", "free_top")


def isd_kv_commit(state: dict, accept_len: torch.Tensor, num_masks: int, *,
                  status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One KV-slot commit of the stationary batch (include/isd_kv.h).

    state: int32 CUDA tensors under the keys table [C, ld] (row-major),
    seq_len, pend, alloc [C], free_slots [pool], free_top [1]; updated in
    place when the commit succeeds.  accept_len [C] int32: the step's accept
    lengths by batch position (read where pend > 0).  Returns the status
    tensor [1] int32 on the device (0 = committed, else the OR of the
    ISD_KV_ERR_* bits and nothing changed); reading it is a device->host
    sync the caller may defer."""
    t = state["table"]
    if t.dim() != 2:
        raise ValueError("table must be 2-D [num_seqs, ld]")
    ptrs = {k: _int32(state[k], k) for k in KV_FIELDS}
    C, ld = t.shape
    for k in ("seq_len", "pend", "alloc"):
        if state[k].numel() != C:
            raise ValueError(f"{k} must have one entry per sequence")
    if state["free_top"].numel() != 1 or accept_len.numel() != C:
        raise ValueError("free_top must hold one entry and accept_len one per sequence")
    device = t.device
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=device)
    rc = _lib.load().isd_kv_commit(ptrs["table"], ld, ptrs["seq_len"], ptrs["pend"], ptrs["alloc"],
                                   ptrs["free_slots"], ptrs["free_top"], state["free_slots"].numel(),
                                   _int32(accept_len, "accept_len"), C, int(num_masks),
                                   _int32(status, "status"), _stream(device, stream))
    _lib.check("isd_kv_commit", rc)
    return status


def isd_decision_uniforms(seed: int, offset: int, counters: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """isd_decision_uniforms (include/isd_debug.h): the decision uniform of
    each (sequence, position, purpose) row of ``counters`` ([n, 3] int64 on
    a CUDA device, non-negative) under (seed, offset).  Returns [n] float32."""
    if counters.dtype != torch.int64 or counters.dim() != 2 or counters.shape[1] != 3 or \
            not counters.is_contiguous() or not counters.is_cuda:
        raise ValueError("counters must be a contiguous [n, 3] int64 CUDA tensor")
    n = counters.shape[0]
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=counters.device)
    status = _lib.load().isd_decision_uniforms(int(seed), int(offset), counters.data_ptr(), n,
                                               _f32(out, "out"), _stream(counters.device, stream))
    _lib.check("isd_decision_uniforms", status)
    return out
