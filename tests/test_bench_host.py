"""Host-side arithmetic of bench.py: the algorithmic bytes of a step (the
roofline's numerator) and the code-only hash that keys profiled traffic."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_verify_accept_02_b300 import workloads  # noqa: E402


def test_algorithmic_bytes_counts_rows_read():
    """Per sequence: 2 L rows at T > 0 and L at T = 0 (greedy reads no q), the
    final anchor row only when every proposal was accepted; the propose pass
    adds L qnew rows for each sequence whose proposals are drawn."""
    b = workloads.make("ragged", num_seqs=6, vocab=1000)
    Ls = b.strides()
    temps = b.temperature.tolist()
    acc = [Ls[0], 0, Ls[2], 1, 0, Ls[5]]
    valid = [1, 0, 1, 0, 0, 1]
    row = 2 * 1000  # bf16
    want_v = sum(row * ((2 * L if t > 0 else L) + (1 if a == L else 0)) for L, t, a in zip(Ls, temps, acc))
    want_p = sum(row * L for L, ok in zip(Ls, valid) if ok)
    assert bench.algorithmic_bytes(b, acc, valid) == (want_v, want_p)
    f = workloads.make("tiny", num_seqs=2, vocab=100)  # fp32 rows: 4 bytes per id
    v, p = bench.algorithmic_bytes(f, [0, 0], [0, 0])
    assert v == 4 * 100 * sum(2 * L for L in f.strides()) and p == 0


def test_c64_algorithmic_bytes_match_the_recorded_figure():
    """c64 (C=64, L=8, V=151936 bf16, T=1) reads 1024 rows of 303,872 bytes,
    plus one final anchor row per sequence that accepts all 8."""
    b = workloads.make("c64", num_seqs=2, vocab=151936)  # the per-sequence arithmetic
    v, _ = bench.algorithmic_bytes(b, [3, 8], [0, 1])
    assert v == 303872 * (16 + 16 + 1)


def test_source_hash_ignores_comments_only():
    src = "int a = 1; // note\n/* block\n comment */ const char* s = \"x//y\";\nint b;\n"
    assert bench._strip_comments(src) == bench._strip_comments(src.replace("note", "other"))
    assert bench._strip_comments(src) != bench._strip_comments(src.replace("int b", "int c"))
    assert '"x//y"' in bench._strip_comments(src)


def test_profiled_sources_are_the_verify_kernels():
    """The traffic key covers the verify kernel's translation unit, the host
    file that launches it and every local header they include, and nothing
    else (another kernel's source may change without voiding the counters)."""
    names = {os.path.relpath(p, ROOT) for p in bench.profiled_source_files()}
    csrc = "speculative_verify_accept_02_b300/csrc/"
    assert {csrc + "isd_verify.cu", csrc + "isd_api.cu", csrc + "isd_device.cuh", csrc + "isd_internal.h",
            "include/isd.h"} <= names
    assert csrc + "isd_kv.cu" not in names and csrc + "isd_propose.cu" not in names


def test_filtered_bytes_count_every_row_once():
    """The filtered verify streams all sum L + C anchor rows and sum L
    proposal rows once: c64 reads 1088 rows of 303,872 bytes."""
    b = workloads.make("c64", num_seqs=2, vocab=151936)
    assert bench.filtered_verify_bytes(b) == (2 * 16 + 2) * 303872
    f = workloads.make("tiny", num_seqs=3, vocab=100)
    assert bench.filtered_verify_bytes(f) == (2 * f.total + 3) * 100 * 4


def test_bench_rows_parse(monkeypatch):
    for row in ("step", "kv", "filtered"):
        monkeypatch.setattr("sys.argv", ["bench.py", "--row", row, "--steps", "5"])
        a = bench.parse()
        assert a.row == row and a.steps == 5


def test_time_oracle_all_cores_and_one():
    """The CPU baseline's timer on a small batch: the rate counts the sampled
    positions, and a single-core run reports one thread."""
    import oracle
    b = workloads.make("tiny", num_seqs=3, vocab=64)
    rate, threads, reps, el, pos = bench.time_oracle(b, 0.05)
    assert pos == sum(b.strides()) and reps >= 1 and rate == pytest.approx(pos * reps / el)
    rate1, threads1, reps1, el1, pos1 = bench.time_oracle(b, 0.05, nthreads=1, seqs=[0])
    assert threads1 == 1 and pos1 == b.strides()[0]
    assert oracle.threads() == threads  # the single-core run put the thread count back


def test_reread_bytes_count_rejecting_sampled_sequences():
    """Two rows (p_j, q_j) per T > 0 sequence that rejects; greedy, invalid
    and all-accepting sequences re-read nothing."""
    b = workloads.make("ragged", num_seqs=6, vocab=1000)
    Ls, temps = b.strides(), b.temperature.tolist()
    acc = [0, Ls[1], 0, -1, 0, 0]
    want = sum(2 * 2000 for i in range(6) if temps[i] > 0 and 0 <= acc[i] < Ls[i])
    assert bench.reread_bytes(b, acc) == want


def test_accepted_share():
    b = workloads.make("ragged", num_seqs=4, vocab=1000)
    Ls = b.strides()
    assert bench.accepted_share(b, [Ls[0], 0, -1, 1]) == (Ls[0] + 1) / sum(Ls)
