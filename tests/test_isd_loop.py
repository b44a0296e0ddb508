"""The ISD decode loop over the table-driven synthetic model
(speculative_verify_accept_02_b300/isd_loop.py) and its tokens per forward
against "Introspective Diffusion Language Models | Summary", Appendix B.1:
TPF_N = (2 + p + ... + p^(N-2)) / (2 - p^(N-1)) under uniform acceptance p,
TPF = N at perfect acceptance and TPF = 1 at zero acceptance (§ B.1 prose).

The closed form is pinned against the stationary law of the step chain
(proposal-only step / fused step) solved as a linear system; the loop runs
on the fp64 oracle here and on the CUDA path in the GPU tests."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_accept_02_b300 import workloads
from speculative_verify_accept_02_b300.isd_loop import CudaBackend, ISDLoop, TableModel, tpf_isd


class OracleBackend:
    def verify(self, p, q, tokens, offs, temp, seed, offset, filters=None):
        V = p.shape[1]
        hp, hq = workloads.host_logits(p), workloads.host_logits(q)
        if filters is None:
            ov = oracle.verify(hp, hq, V, tokens, offs, temp, seed, offset)
        else:
            ov = oracle.verify_filtered(hp, hq, V, tokens, offs, temp, seed, offset, filters[0], filters[1])
        return ov["accept_len"], ov["out_tokens"]

    def propose(self, qnew, offs, temp, seed, offset, filters=None):
        V = qnew.shape[1]
        hq = workloads.host_logits(qnew)
        if filters is None:
            op = oracle.propose(hq, V, offs, temp, seed, offset)
        else:
            op = oracle.propose_filtered(hq, V, offs, temp, seed, offset, filters[0], filters[1])
        return op["proposals"], op["valid"]

    def kv_state(self, state):
        return state.copy()

    def kv_commit(self, handle, accept, num_masks):
        return oracle.kv_commit(handle, accept, num_masks)

    def kv_read(self, handle):
        return handle.copy()


def chain_tpf(n, p):
    """Tokens per forward from the stationary law of the two-state step chain:
    proposal-only (1 token, then a fused step) and fused (a accepted of n-1
    with probability p^a (1-p), a+1 tokens, then proposal-only; all n-1
    accepted with probability p^(n-1), n tokens, fused again)."""
    stay = p ** (n - 1)
    # pi = pi T over states (proposal-only, fused)
    T = np.array([[0.0, 1.0], [1.0 - stay, stay]])
    A = np.vstack([T.T - np.eye(2), np.ones(2)])
    pi = np.linalg.lstsq(A, np.array([0.0, 0.0, 1.0]), rcond=None)[0]
    emit_fused = sum((a + 1) * p ** a * (1 - p) for a in range(n - 1)) + n * stay
    return pi[0] * 1.0 + pi[1] * emit_fused


@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 32])
@pytest.mark.parametrize("p", [0.0, 0.3, 0.6, 0.9, 1.0])
def test_closed_form_matches_step_chain(n, p):
    assert tpf_isd(n, p) == pytest.approx(chain_tpf(n, p), rel=1e-12)


def test_closed_form_end_points():
    for n in range(2, 33):
        assert tpf_isd(n, 1.0) == pytest.approx(n)
        assert tpf_isd(n, 0.0) == pytest.approx(1.0)


def test_table_model_acceptance_is_alpha():
    """sum_v min(p_v, q_v) = alpha in every table entry (the TV identity of
    the acceptance probability, Summary §3.2)."""
    for alpha in (0.0, 0.25, 0.6, 1.0):
        m = TableModel(300, alpha, entries=5, support=40, seed=3)
        p = torch.softmax(m.P.double(), dim=1)
        q = torch.softmax(m.Q.double(), dim=1)
        acc = torch.minimum(p, q).sum(dim=1)
        assert torch.allclose(acc, torch.full_like(acc, alpha), atol=1e-6)


def _extremes(backend, vocab, device):
    n, C, S = 4, 3, 9
    full = ISDLoop(TableModel(vocab, 1.0, entries=7, support=32, seed=1, device=device), C, n, backend).run(S)
    assert full.per_seq_tokens == [1 + n * (S - 1)] * C  # proposal-only once, then n per fused step
    none = ISDLoop(TableModel(vocab, 0.0, entries=7, support=32, seed=1, device=device), C, n, backend).run(S)
    assert none.per_seq_tokens == [S] * C and none.tpf == 1.0
    assert none.accepted == 0 and full.accepted == full.verified


def _law(backend, vocab, device, C, S):
    n, alpha = 4, 0.6
    st = ISDLoop(TableModel(vocab, alpha, entries=31, support=32, seed=2, device=device), C, n, backend).run(S)
    per = np.asarray(st.per_seq_tokens) / S
    se = per.std(ddof=1) / np.sqrt(C)
    # The first step is always proposal-only: at most (n - 1) / S tokens per forward of start-up bias.
    assert abs(st.tpf - tpf_isd(n, alpha)) < 4 * se + (n - 1) / S, (st.tpf, tpf_isd(n, alpha), se)
    tested = st.accepted + st.rejected
    assert abs(st.acceptance - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / tested), st.acceptance


def test_loop_on_oracle_extremes():
    _extremes(OracleBackend(), 256, "cpu")


def test_loop_on_oracle_tpf_law():
    _law(OracleBackend(), 256, "cpu", C=24, S=120)


@pytest.mark.gpu
def test_loop_on_cuda_extremes():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    _extremes(CudaBackend(), 4096, "cuda")


@pytest.mark.gpu
def test_loop_on_cuda_tpf_law():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    _law(CudaBackend(), 4096, "cuda", C=64, S=200)


def _kv_loop(backend, vocab, device):
    """The loop with its KV-slot state (Summary §3.3): after every step each
    sequence caches exactly as many entries as it has emitted tokens (the
    prompt token plus all emitted but the newest), its next forward verifies
    exactly its pending proposals, and every pool slot is free or cached
    once."""
    n, C, S = 4, 6, 25
    loop = ISDLoop(TableModel(vocab, 0.6, entries=9, support=32, seed=4, device=device), C, n, backend,
                   kv_len=2 + S * n + 2 * n)
    for _ in range(S):
        st = loop.step()
        kv = backend.kv_read(loop.kv)
        assert list(kv.seq_len) == st.per_seq_tokens
        assert list(kv.pend) == [0 if p is None else len(p) for p in loop.pending]
        assert list(kv.alloc) == [1 + int(p) + n - 1 for p in kv.pend]
        live = [kv.table[i, :kv.seq_len[i] + kv.alloc[i]] for i in range(C)]
        used = np.concatenate(live + [kv.free_slots[:kv.free_top[0]]])
        assert np.array_equal(np.sort(used), np.arange(kv.pool_size))


def test_loop_kv_on_oracle():
    _kv_loop(OracleBackend(), 256, "cpu")


@pytest.mark.gpu
def test_loop_kv_on_cuda():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    _kv_loop(CudaBackend(), 4096, "cuda")


def _filtered_extremes(backend, device):
    """Closed forms of the loop under the evaluation setting's filters (see
    test_loop_under_filters_on_oracle): top-10 of a 32-id support, and top-50
    then top-p 0.95 of a 64-id support (both filtered rows uniform on the
    same 48 ids, the cut 0.01 from moving).  Returns the loop statistics."""
    n, C, S = 4, 3, 7
    out = []
    for filters, support in (((10, 1.0), 32), ((50, 0.95), 64)):
        for alpha, all_pass in ((0.6, True), (0.4, False)):
            model = TableModel(256, alpha, entries=5, support=support, seed=8, device=device)
            st = ISDLoop(model, C, n, backend, filters=filters).run(S)
            if all_pass:
                assert st.per_seq_tokens == [1 + n * (S - 1)] * C and st.accepted == st.verified
            else:
                assert st.per_seq_tokens == [S] * C and st.accepted == 0
            out.append((st.per_seq_tokens, st.accepted, st.rejected, st.verified, st.forwards))
    return out


@pytest.mark.gpu
def test_loop_under_filters_on_cuda():
    """The decode loop on the CUDA backend under top-k / top-p (Summary §4.1:
    top-k 50, top-p 0.95), through isd_verify_filtered and
    isd_propose_filtered: the closed forms hold, and the step statistics equal
    the oracle backend's."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    assert _filtered_extremes(CudaBackend(), "cuda") == _filtered_extremes(OracleBackend(), "cpu")


def test_loop_under_filters_on_oracle():
    """The evaluation setting's filters change what the table model accepts,
    exactly: q is uniform on a support S and p puts alpha/s on S, (1-alpha)/s
    on a disjoint S'.  Top-10 of 32 keeps the 10 lowest ids of the larger
    block: for alpha > 1/2 both filtered p and q are uniform on the same 10
    ids of S, so every proposal passes (TPF = n after the first step); for
    alpha < 1/2 filtered p lives on S' and nothing passes (TPF = 1)."""
    n, C, S = 4, 3, 7
    for alpha, all_pass in ((0.6, True), (0.4, False)):
        model = TableModel(256, alpha, entries=5, support=32, seed=8)
        st = ISDLoop(model, C, n, OracleBackend(), filters=(10, 1.0)).run(S)
        if all_pass:
            assert st.per_seq_tokens == [1 + n * (S - 1)] * C and st.accepted == st.verified
        else:
            assert st.per_seq_tokens == [S] * C and st.accepted == 0
