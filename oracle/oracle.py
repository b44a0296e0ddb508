"""ctypes wrapper over the fp64 C oracle (oracle/isd_oracle.c).

TEST INFRASTRUCTURE ONLY: used by tests/, the smoke entry point and the
benchmark's CPU-baseline leg.  Arrays are numpy, on the host.  Argument
meaning follows the library's C ABI (see include/isd.h) with host memory.

Source of every definition: "Introspective Diffusion Language Models |
Summary" — §2 (alpha), §3.2 (acceptance, residual correction, bonus token),
§3.3 (argmax proposals with strict verification), §3.1 (next-token shift).
"""
import ctypes as C
import math

import numpy as np

from . import build as _build

DTYPE_BF16 = 0
DTYPE_F32 = 1
TAG_ACCEPT, TAG_CORRECT, TAG_BONUS, TAG_PROPOSE = 0, 1, 2, 3

_dp = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_fp = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_ip = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_up = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
_bp = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def _declare(L):
    L.oracle_philox4x64_10.argtypes = [_up, _up, _up]
    L.oracle_philox4x64_10.restype = None
    L.oracle_uniform.argtypes = [C.c_uint64] * 5
    L.oracle_uniform.restype = C.c_double
    L.oracle_argmax.argtypes = [_dp, C.c_int]
    L.oracle_argmax.restype = C.c_int
    L.oracle_softmax.argtypes = [_dp, C.c_int, C.c_double, _dp]
    L.oracle_softmax.restype = None
    L.oracle_log_softmax_at.argtypes = [_dp, C.c_int, C.c_double, C.c_int]
    L.oracle_log_softmax_at.restype = C.c_double
    L.oracle_ratio.argtypes = [_dp, _dp, C.c_int, C.c_double, C.c_int]
    L.oracle_ratio.restype = C.c_double
    L.oracle_residual.argtypes = [_dp, _dp, C.c_int, C.c_double, _dp]
    L.oracle_residual.restype = None
    L.oracle_icdf.argtypes = [_dp, C.c_int, C.c_double, C.POINTER(C.c_double)]
    L.oracle_icdf.restype = C.c_int
    L.oracle_verify_one.argtypes = [_dp, _dp, C.c_int, C.c_int, C.c_double, _ip, _dp, _dp,
                                    C.c_double, C.POINTER(C.c_int32), _ip, _dp,
                                    C.POINTER(C.c_double), _dp, C.POINTER(C.c_double), C.c_double]
    L.oracle_verify_one.restype = None
    L.oracle_filtered_probs.argtypes = [_dp, C.c_int, C.c_double, C.c_int, C.c_double, _dp,
                                        C.POINTER(C.c_double)]
    L.oracle_filtered_probs.restype = None
    L.oracle_ratio_relaxed.argtypes = [_dp, _dp, C.c_int, C.c_double, C.c_int, C.c_double]
    L.oracle_ratio_relaxed.restype = C.c_double
    L.oracle_verify.argtypes = [C.c_void_p, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_int,
                                _ip, _ip, C.c_int, _fp, C.c_uint64, C.c_uint64,
                                _ip, _ip, _dp, _dp, _dp, _dp, C.c_void_p, C.c_int, C.c_int, C.c_double]
    L.oracle_verify.restype = None
    L.oracle_propose.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_int, _ip, C.c_int, _fp,
                                 C.c_uint64, C.c_uint64, C.c_void_p, _ip, _bp, _dp,
                                 C.c_void_p, C.c_int, C.c_int]
    L.oracle_propose.restype = None
    L.oracle_alpha.argtypes = [_fp, _ip, C.c_int, _dp, C.POINTER(C.c_double)]
    L.oracle_alpha.restype = None
    L.oracle_gumbel_uniform.argtypes = [C.c_uint64] * 6
    L.oracle_gumbel_uniform.restype = C.c_double
    L.oracle_gumbel_draw.argtypes = [_dp, C.c_int, C.c_uint64, C.c_uint64, C.c_uint64, C.c_uint64, C.c_uint64,
                                     C.POINTER(C.c_double)]
    L.oracle_gumbel_draw.restype = C.c_int
    L.oracle_kv_commit.argtypes = [_ip, C.c_int64, _ip, _ip, _ip, _ip, _ip, C.c_int, _ip, C.c_int, C.c_int]
    L.oracle_kv_commit.restype = C.c_int
    L.oracle_max_threads.argtypes = [C.c_int]
    L.oracle_max_threads.restype = C.c_int


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _logit_buffer(logits):
    """(pointer-owner array, dtype code, row stride) of a 2-D host array.

    bf16 logits are passed as uint16 bit patterns (or int16), fp32 as float32.
    Rows may be padded: the row stride is taken from the array's strides."""
    a = logits
    if a.ndim != 2:
        raise ValueError("logits must be 2-D")
    if a.dtype in (np.uint16, np.int16):
        code = DTYPE_BF16
    elif a.dtype == np.float32:
        code = DTYPE_F32
    else:
        raise TypeError(f"unsupported logit dtype {a.dtype}")
    if a.strides[1] != a.itemsize or a.strides[0] % a.itemsize:
        raise ValueError("rows must be contiguous")
    return a, code, a.strides[0] // a.itemsize


def _decode(logits, vocab):
    """Rows of a host logit buffer (bf16 bit patterns or float32) as float64."""
    a = np.asarray(logits)
    if a.dtype in (np.uint16, np.int16):
        a = (a.view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return a[:, :vocab].astype(np.float64)


def _sel(seqs):
    if seqs is None:
        return None, 0, None
    s = np.ascontiguousarray(seqs, dtype=np.int32)
    return s.ctypes.data, s.size, s


class Oracle:
    """The oracle library loaded from one path (tests may load other builds)."""

    def __init__(self, path=None):
        self.path = path or _build.build()
        self.lib = C.CDLL(self.path)
        _declare(self.lib)

    def philox4x64_10(self, counter, key):
        """Philox4x64-10 of a 4-word counter under a 2-word key (Salmon et al.)."""
        out = np.zeros(4, dtype=np.uint64)
        self.lib.oracle_philox4x64_10(np.asarray(counter, dtype=np.uint64),
                                      np.asarray(key, dtype=np.uint64), out)
        return out

    def uniform(self, seed, offset, seq, pos, tag):
        return self.lib.oracle_uniform(seed, offset, seq, pos, tag)

    def argmax(self, logits):
        x = _d(logits)
        return self.lib.oracle_argmax(x, x.size)

    def softmax(self, logits, T):
        x = _d(logits)
        out = np.empty_like(x)
        self.lib.oracle_softmax(x, x.size, float(T), out)
        return out

    def log_softmax_at(self, logits, T, x):
        z = _d(logits)
        return self.lib.oracle_log_softmax_at(z, z.size, float(T), int(x))

    def ratio(self, P, Q, T, x):
        p, q = _d(P), _d(Q)
        return self.lib.oracle_ratio(p, q, p.size, float(T), int(x))

    def residual(self, P, Q, T):
        p, q = _d(P), _d(Q)
        w = np.empty_like(p)
        self.lib.oracle_residual(p, q, p.size, float(T), w)
        return w

    def icdf(self, w, u):
        """Returns (token, margin)."""
        ww = _d(w)
        m = C.c_double()
        v = self.lib.oracle_icdf(ww, ww.size, float(u), C.byref(m))
        return v, m.value

    def filtered_probs(self, logits, T, top_k, top_p, with_margin=False):
        """softmax(logits/T) after the top-k, then top-p filter, renormalised
        (the pages' evaluation sampling setting).  with_margin: also return
        the distance of the top-p cut from moving."""
        z = _d(logits)
        out = np.empty(z.size, dtype=np.float64)
        m = C.c_double()
        self.lib.oracle_filtered_probs(z, z.size, float(T), int(top_k), float(top_p), out, C.byref(m))
        return (out, m.value) if with_margin else out

    def verify_filtered(self, p_logits, q_logits, vocab, tokens, seq_offsets, temperature, seed, offset,
                        top_k, top_p):
        """The verify step with the sampling filters applied to both p and q
        (p~, q~): ratio min(1, p~(x)/q~(x)) (1 where q~(x) = 0), strict
        acceptance, correction from normalize(max(0, p~_j - q~_j)) (p~_j if that
        is all zero), bonus from p~_{L+1}.  T = 0 sequences are unaffected by
        the filters and follow verify().  Same outputs as verify(), with the
        margins of the decisions: accept_margin [sum L] (|u - ratio| of each
        tested position, +inf for the rest), token_margin [C] (inverse-CDF
        margin of the correction or bonus draw) and cut_margin [C] (the
        smallest top-p cut margin of the sequence's rows)."""
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        C_ = offs.size - 1
        total = int(offs[-1])
        temp = np.ascontiguousarray(temperature, dtype=np.float32)
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        P, Q = _decode(p_logits, vocab), _decode(q_logits, vocab)
        out = dict(accept_len=np.full(C_, -2, np.int32), out_tokens=np.full(total + C_, -2, np.int32),
                   ratio=np.full(total, np.nan), alpha=np.full(C_, np.nan),
                   accept_margin=np.full(total, np.inf), token_margin=np.full(C_, np.inf),
                   cut_margin=np.full(C_, np.inf))
        for i in range(C_):
            s, L, T = int(offs[i]), int(offs[i + 1] - offs[i]), float(temp[i])
            if T == 0.0 or not (1 <= L <= 32) or not math.isfinite(T) or T < 0 or (0 < T < 1.17549435e-38) \
                    or np.any((toks[s:s + L] < 0) | (toks[s:s + L] >= vocab)):
                one = self.verify(p_logits, q_logits, vocab, tokens, seq_offsets, temperature, seed, offset,
                                  seqs=[i])
                for k in out:
                    if k in ("accept_len", "alpha", "token_margin"):
                        out[k][i] = one[k][i]
                    elif k in ("ratio", "accept_margin"):
                        out[k][s:s + max(L, 0)] = one[k][s:s + max(L, 0)]
                    elif k == "out_tokens":
                        out[k][s + i: s + i + max(L, 0) + 1] = one[k][s + i: s + i + max(L, 0) + 1]
                continue
            pm = [self.filtered_probs(P[s + i + k], T, top_k, top_p, with_margin=True) for k in range(L + 1)]
            qm = [self.filtered_probs(Q[s + k], T, top_k, top_p, with_margin=True) for k in range(L)]
            pt, qt = [m[0] for m in pm], [m[0] for m in qm]
            out["cut_margin"][i] = min(m[1] for m in pm + qm)
            x = toks[s:s + L]
            ratio = np.array([1.0 if qt[k][x[k]] == 0.0 else min(1.0, pt[k][x[k]] / qt[k][x[k]])
                              for k in range(L)])
            a = 0
            while a < L:
                u = self.uniform(seed, offset, i, a + 1, TAG_ACCEPT)
                out["accept_margin"][s + a] = abs(u - ratio[a])
                if not u < ratio[a]:
                    break
                a += 1
            if a < L:
                w = np.maximum(pt[a] - qt[a], 0.0)
                if not w.sum() > 0.0:
                    w = pt[a]
                tok, tm = self.icdf(w, self.uniform(seed, offset, i, a + 1, TAG_CORRECT))
            else:
                tok, tm = self.icdf(pt[L], self.uniform(seed, offset, i, L + 1, TAG_BONUS))
            out["token_margin"][i] = tm
            out["accept_len"][i] = a
            out["ratio"][s:s + L] = ratio
            out["alpha"][i] = ratio.mean()
            slots = out["out_tokens"][s + i: s + i + L + 1]
            slots[:] = -1
            slots[:a] = x[:a]
            slots[a] = tok
        return out

    def propose_filtered(self, qnew_logits, vocab, seq_offsets, temperature, seed, offset, top_k, top_p,
                         accept_len=None):
        """Proposals drawn from the filtered softmax(qnew/T) (argmax at T = 0),
        with propose()'s validity rules; margin [sum L] is the smaller of the
        draw's inverse-CDF margin and its row's top-p cut margin."""
        base = self.propose(qnew_logits, vocab, seq_offsets, temperature, seed, offset, accept_len=accept_len)
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        temp = np.ascontiguousarray(temperature, dtype=np.float32)
        Qn = _decode(qnew_logits, vocab)
        for i in range(offs.size - 1):
            if not base["valid"][i] or temp[i] == 0.0:
                continue
            for m in range(1, int(offs[i + 1] - offs[i]) + 1):
                r = int(offs[i]) + m - 1
                w, cm = self.filtered_probs(Qn[r], float(temp[i]), top_k, top_p, with_margin=True)
                base["proposals"][r], tm = self.icdf(w, self.uniform(seed, offset, i, m, TAG_PROPOSE))
                base["margin"][r] = min(tm, cm)
        return base

    def gumbel_uniform(self, seed, offset, seq, pos, tag, v):
        """The uniform of vocabulary id v in one Gumbel-max draw, in (0, 1)."""
        return self.lib.oracle_gumbel_uniform(seed, offset, seq, pos, tag, v)

    def gumbel_draw(self, w, seed, offset, seq, pos, tag):
        """Gumbel-max draw over weights w: (token, margin)."""
        ww = _d(w)
        m = C.c_double()
        v = self.lib.oracle_gumbel_draw(ww, ww.size, seed, offset, seq, pos, tag, C.byref(m))
        return v, m.value

    def verify_gumbel(self, p_logits, q_logits, vocab, tokens, seq_offsets, temperature, seed, offset):
        """The verify step with Gumbel-max draws for the correction and the
        bonus token (the sampler of the pages' fused kernel) in place of
        inverse-CDF draws; ratios, acceptance and alpha as verify().  T = 0
        sequences and invalid ones follow verify().  Returns verify()'s
        outputs; token_margin is the Gumbel score gap of the draw."""
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        temp = np.ascontiguousarray(temperature, dtype=np.float32)
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        out = self.verify(p_logits, q_logits, vocab, tokens, seq_offsets, temperature, seed, offset)
        P, Q = _decode(p_logits, vocab), _decode(q_logits, vocab)
        for i in range(offs.size - 1):
            s, L, T = int(offs[i]), int(offs[i + 1] - offs[i]), float(temp[i])
            a = int(out["accept_len"][i])
            if a < 0 or T == 0.0:
                continue
            if a < L:
                w = self.residual(P[s + i + a], Q[s + a], T)
                tok, gap = self.gumbel_draw(w, seed, offset, i, a + 1, TAG_CORRECT)
            else:
                tok, gap = self.gumbel_draw(self.softmax(P[s + i + L], T), seed, offset, i, L + 1, TAG_BONUS)
            out["out_tokens"][s + i + a] = tok
            out["token_margin"][i] = gap
        return out

    def propose_gumbel(self, qnew_logits, vocab, seq_offsets, temperature, seed, offset, accept_len=None):
        """Proposals by Gumbel-max draws from softmax(qnew/T) (argmax at
        T = 0), with propose()'s validity rules; margin is the score gap."""
        base = self.propose(qnew_logits, vocab, seq_offsets, temperature, seed, offset, accept_len=accept_len)
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        temp = np.ascontiguousarray(temperature, dtype=np.float32)
        Qn = _decode(qnew_logits, vocab)
        for i in range(offs.size - 1):
            if not base["valid"][i] or temp[i] == 0.0:
                continue
            for m in range(1, int(offs[i + 1] - offs[i]) + 1):
                r = int(offs[i]) + m - 1
                w = self.softmax(Qn[r], float(temp[i]))
                base["proposals"][r], base["margin"][r] = self.gumbel_draw(w, seed, offset, i, m, TAG_PROPOSE)
        return base

    def ratio_relaxed(self, P, Q, T, x, tau):
        """min(1, (1 + tau) p(x)/q(x)) of one row pair (argmax indicator at T = 0)."""
        P, Q = _d(P), _d(Q)
        return self.lib.oracle_ratio_relaxed(P, Q, P.size, float(T), int(x), float(tau))

    def verify_one(self, P, Q, T, x, u_accept, u_correct, u_bonus, tau=0.0):
        """One sequence with explicit uniforms. P: (L+1, V), Q: (L, V).  tau:
        the accept test uses min(1, (1 + tau) p/q) (relaxed acceptance)."""
        P, Q = _d(P), _d(Q)
        L, V = Q.shape
        assert P.shape == (L + 1, V)
        x = np.ascontiguousarray(x, dtype=np.int32)
        a = C.c_int32()
        out = np.empty(L + 1, dtype=np.int32)
        r = np.empty(L, dtype=np.float64)
        alpha = C.c_double()
        am = np.empty(L, dtype=np.float64)
        tm = C.c_double()
        self.lib.oracle_verify_one(P, Q, V, L, float(T), x, _d(u_accept), _d(u_correct),
                                   float(u_bonus), C.byref(a), out, r, C.byref(alpha), am,
                                   C.byref(tm), float(tau))
        return dict(accept_len=a.value, out_tokens=out, ratio=r, alpha=alpha.value,
                    accept_margin=am, token_margin=tm.value)

    def verify(self, p_logits, q_logits, vocab, tokens, seq_offsets, temperature, seed, offset,
               seqs=None, nthreads=0, tau=0.0):
        """All (or the selected) sequences of one verify step.  tau > 0: the
        accept test uses the relaxed ratio min(1, (1 + tau) p/q); the reported
        ratios and alpha stay the strict ones.

        Returns a dict of accept_len [C], out_tokens [sum L + C], ratio [sum L],
        alpha [C], accept_margin [sum L], token_margin [C]; entries of unselected
        sequences are left at their fill values (-2 / NaN)."""
        pa, code_p, ld_p = _logit_buffer(p_logits)
        qa, code_q, ld_q = _logit_buffer(q_logits)
        if code_p != code_q:
            raise TypeError("p and q must share a dtype")
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        C_ = offs.size - 1
        total = int(offs[-1])
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        temp = np.ascontiguousarray(temperature, dtype=np.float32)
        out = dict(accept_len=np.full(C_, -2, np.int32), out_tokens=np.full(total + C_, -2, np.int32),
                   ratio=np.full(total, np.nan), alpha=np.full(C_, np.nan),
                   accept_margin=np.full(total, np.inf), token_margin=np.full(C_, np.inf))
        sp, sn, _keep = _sel(seqs)
        self.lib.oracle_verify(pa.ctypes.data, ld_p, qa.ctypes.data, ld_q, code_p, int(vocab),
                               toks, offs, C_, temp, int(seed), int(offset), out["accept_len"],
                               out["out_tokens"], out["ratio"], out["alpha"],
                               out["accept_margin"], out["token_margin"], sp, sn, int(nthreads),
                               float(tau))
        return out

    def propose(self, qnew_logits, vocab, seq_offsets, temperature, seed, offset, accept_len=None,
                seqs=None, nthreads=0):
        """Proposals for the next stride. Returns proposals [sum L], valid [C], margin [sum L]."""
        qa, code, ld = _logit_buffer(qnew_logits)
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        C_ = offs.size - 1
        total = int(offs[-1])
        temp = np.ascontiguousarray(temperature, dtype=np.float32)
        acc = None if accept_len is None else np.ascontiguousarray(accept_len, dtype=np.int32)
        out = dict(proposals=np.full(total, -2, np.int32), valid=np.zeros(C_, np.uint8),
                   margin=np.full(total, np.inf))
        sp, sn, _keep = _sel(seqs)
        self.lib.oracle_propose(qa.ctypes.data, ld, code, int(vocab), offs, C_, temp, int(seed),
                                int(offset), None if acc is None else acc.ctypes.data,
                                out["proposals"], out["valid"], out["margin"], sp, sn,
                                int(nthreads))
        return out

    def alpha(self, ratio_f32, seq_offsets):
        r = np.ascontiguousarray(ratio_f32, dtype=np.float32)
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int32)
        C_ = offs.size - 1
        per = np.empty(C_, dtype=np.float64)
        mean = C.c_double()
        self.lib.oracle_alpha(r, offs, C_, per, C.byref(mean))
        return per, mean.value

    def kv_commit(self, state, accept_len, num_masks):
        """One commit of the stationary batch's KV-slot bookkeeping (Summary
        §3.3: batched slot scatter, trim of rejected and masked entries).

        state: a KVState (speculative_verify_accept_02_b300.kv) or any object
        with int32 numpy arrays table [C, ld], seq_len, pend, alloc [C],
        free_slots [pool] and free_top [1]; updated in place on success.
        Returns the status: 0, or the OR of the KV error bits (state
        unchanged)."""
        arrs = [state.table, state.seq_len, state.pend, state.alloc, state.free_slots, state.free_top]
        for a in arrs:
            if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
                raise TypeError("KV state arrays must be C-contiguous int32 numpy arrays")
        C_, ld = state.table.shape
        acc = np.ascontiguousarray(np.broadcast_to(np.asarray(accept_len, np.int32), (C_,)))
        return self.lib.oracle_kv_commit(state.table, ld, state.seq_len, state.pend, state.alloc,
                                         state.free_slots, state.free_top, state.free_slots.size, acc, C_,
                                         int(num_masks))

    def threads(self, nthreads=0):
        """Number of threads the batched oracle calls use."""
        return self.lib.oracle_max_threads(int(nthreads))


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def __getattr__(name):
    # Module-level access (oracle.ratio(...)) goes to the default build.
    if name.startswith("__"):
        raise AttributeError(name)
    return getattr(default(), name)
