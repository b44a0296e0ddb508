"""isd_verify_noalloc: the verify entry point for callers that cannot allocate
device memory (a plug-in living inside another engine's memory pool, code
running while that pool is locked).  It keeps its scratch in an array inside
the library instead of a caller-provided workspace.

Its results must equal isd_verify's on the same inputs, call after call: the
array keeps what the previous call left, so two different batches run back
to back here.  The file is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from speculative_verify_accept_02_b300 import _lib, build, isd_verify, workloads

RTOL = 1e-4  # the tolerance of the parity tests for ratios and alpha


def _noalloc(lib, b, seed, offset, out):
    dtype = _lib.ISD_DTYPE_BF16 if b.p.dtype == torch.bfloat16 else _lib.ISD_DTYPE_F32
    stream = torch.cuda.current_stream().cuda_stream
    return lib.isd_verify_noalloc(
        b.p.data_ptr(), b.p.stride(0), b.q.data_ptr(), b.q.stride(0), dtype, b.vocab,
        b.tokens.data_ptr(), b.seq_offsets.data_ptr(), b.num_seqs, b.total, b.temperature.data_ptr(),
        seed, offset, out["accept_len"].data_ptr(), out["out_tokens"].data_ptr(), out["ratio"].data_ptr(),
        out["alpha"].data_ptr(), stream)


def test_rejects_a_batch_larger_than_its_array():
    build.build()
    lib = _lib.load()
    fake = 0x10000  # never dereferenced: the size check returns first
    V, C_, total = 151936, 8192, 65536
    assert lib.isd_verify_workspace_bytes(C_, total, V, 0) > _lib.NOALLOC_SCRATCH_BYTES
    status = lib.isd_verify_noalloc(fake, V, fake, V, 0, V, fake, fake, C_, total, fake, 0, 0,
                                    fake, fake, fake, fake, None)
    assert status == _lib.ISD_ERR_WORKSPACE
    assert lib.isd_verify_noalloc(fake, V, fake, V, 0, V, fake, fake, 0, 0, fake, 0, 0,
                                  fake, fake, fake, fake, None) == _lib.ISD_OK
    # Every argument check comes before the array is touched: a refused call
    # returns its status and queues nothing (here no CUDA call is made at all).
    C_, total = 4, 16
    args = [fake, V, fake, V, 0, V, fake, fake, C_, total, fake, 0, 0, fake, fake, fake, fake, None]
    for i in (0, 2, 6, 7, 10, 13, 14, 15, 16):  # p, q, tokens, offsets, temperature and the four outputs
        bad = list(args)
        bad[i] = None
        assert lib.isd_verify_noalloc(*bad) == _lib.ISD_ERR_INVALID_ARG, i
    bad = list(args)
    bad[1] = V - 1                                 # ld_p below the vocabulary
    assert lib.isd_verify_noalloc(*bad) == _lib.ISD_ERR_INVALID_ARG
    bad = list(args)
    bad[0] = fake + 2                              # p not on a 16-byte boundary
    assert lib.isd_verify_noalloc(*bad) == _lib.ISD_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_matches_isd_verify_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    build.build()
    lib = _lib.load()
    cases = [(workloads.make("ragged", num_seqs=12), 3, 5),
             (workloads.make("c64", num_seqs=6), 0, 1)]
    for batch, seed, offset in cases:
        b = batch.to("cuda")
        want = isd_verify(b.p, b.q, b.tokens, b.seq_offsets, b.temperature, seed, offset,
                          vocab=b.vocab, total=b.total)
        C_, total = b.num_seqs, b.total
        got = {"accept_len": torch.full((C_,), -7, dtype=torch.int32, device="cuda"),
               "out_tokens": torch.full((total + C_,), -7, dtype=torch.int32, device="cuda"),
               "ratio": torch.full((total,), -7.0, device="cuda"),
               "alpha": torch.full((C_,), -7.0, device="cuda")}
        status = _noalloc(lib, b, seed, offset, got)
        assert status == _lib.ISD_OK, lib.isd_status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(got["accept_len"], want.accept_len)
        assert torch.equal(got["out_tokens"], want.out_tokens)
        for k, ref in (("ratio", want.ratio), ("alpha", want.alpha)):
            g, w = got[k].cpu().numpy(), ref.cpu().numpy()
            assert np.allclose(g, w, rtol=RTOL, atol=0.0, equal_nan=True), k
        assert (want.accept_len >= 0).all()
