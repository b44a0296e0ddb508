"""The C-ABI library: builds for sm_103a, loads, exports every declared entry
point, and rejects bad arguments on the host before touching the device.
No compute call runs here (no GPU needed)."""
import os
import re

import pytest

from speculative_verify_accept_02_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_symbols():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"ISD_API\s+[\w\s\*]+?\b(isd_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("isd_verify", "isd_verify_relaxed", "isd_verify_propose", "isd_propose", "isd_alpha",
              "isd_verify_workspace_bytes", "isd_verify_propose_workspace_bytes",
              "isd_propose_workspace_bytes", "isd_status_string", "isd_kv_commit", "isd_verify_filtered",
              "isd_propose_filtered"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_build_targets_sm103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in range(5):
        assert lib.isd_status_string(code)
    assert lib.isd_status_string(99) == b"unknown status"


def test_workspace_sizes(lib):
    # Grows with the batch, 256-byte granular, 0 for bad shapes.
    a = lib.isd_verify_workspace_bytes(64, 512, 151936, 0)
    b = lib.isd_verify_workspace_bytes(128, 1024, 151936, 0)
    assert 0 < a < b and a % 256 == 0
    assert lib.isd_verify_workspace_bytes(-1, 0, 10, 0) == 0
    assert lib.isd_verify_workspace_bytes(1, 1, 0, 0) == 0
    assert lib.isd_verify_workspace_bytes(1, 1, 10, 7) == 0
    assert lib.isd_propose_workspace_bytes(64, 512, 151936, 1) > 0


def test_noalloc_figures_in_the_header(lib):
    """The sizes include/isd.h quotes for isd_verify_noalloc's array are the
    library's own: ISD_NOALLOC_SCRATCH_BYTES equals the binding's constant,
    and the bf16 and fp32 needs it gives for V = 151936, C = 256, L = 16 (and
    their shares of the array) equal isd_verify_workspace_bytes."""
    text = open(os.path.join(ROOT, "include", "isd.h")).read()
    m = re.search(r"#define ISD_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m, "ISD_NOALLOC_SCRATCH_BYTES definition"
    array = int(m.group(1)) << int(m.group(2))
    assert array == _lib.NOALLOC_SCRATCH_BYTES
    flat = " ".join(line.strip(" *") for line in text.splitlines())
    m = re.search(r"V = 151936 at C = 256, L = 16 need ([\d,]+) bytes in bf16, about (\d+) % "
                  r"of the array, and ([\d,]+) bytes in fp32, about (\d+) %", flat)
    assert m, "the quoted figures"
    for (nbytes, pct), dtype in (((m.group(1), m.group(2)), 0), ((m.group(3), m.group(4)), 1)):
        need = lib.isd_verify_workspace_bytes(256, 256 * 16, 151936, dtype)
        assert int(nbytes.replace(",", "")) == need
        assert int(pct) == round(100 * need / array)


# A 16-byte aligned address that is never dereferenced: every call below has
# at least one bad argument (or an empty batch), so it returns on the host
# before any launch.
FAKE = 0x10000


def _verify(lib, **kw):
    args = dict(p=FAKE, ldp=1024, q=FAKE, ldq=1024, dtype=0, vocab=1024, tokens=FAKE, offs=FAKE,
                C=2, total=4, temp=FAKE, seed=0, offset=0, acc=FAKE, out=FAKE, ratio=FAKE, alpha=FAKE,
                ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.isd_verify(*args.values())


def test_verify_host_checks(lib):
    assert _verify(lib, C=0) == _lib.ISD_OK                          # empty batch: nothing to do
    assert _verify(lib, C=-1) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, total=-1) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, vocab=0) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, dtype=5) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, p=None) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, tokens=None) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, ws=None) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, ldq=1000) == _lib.ISD_ERR_INVALID_ARG
    assert _verify(lib, p=FAKE + 2) == _lib.ISD_ERR_UNSUPPORTED
    assert _verify(lib, q=FAKE + 8) == _lib.ISD_ERR_UNSUPPORTED
    assert _verify(lib, wsb=16) == _lib.ISD_ERR_WORKSPACE
    assert _verify(lib, ws=FAKE + 16) == _lib.ISD_ERR_WORKSPACE


def _verify_relaxed(lib, tau, **kw):
    args = dict(p=FAKE, ldp=1024, q=FAKE, ldq=1024, dtype=0, vocab=1024, tokens=FAKE, offs=FAKE,
                C=2, total=4, temp=FAKE, seed=0, offset=0, tau=tau, acc=FAKE, out=FAKE, ratio=FAKE,
                alpha=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.isd_verify_relaxed(*args.values())


def test_verify_vocabulary_limit(lib):
    """The verify calls refuse, on the host, a vocabulary past the most tail
    pieces a row may have (524,288 bf16 or 262,144 fp32 ids, as isd.h
    states): UNSUPPORTED, nothing launched.  The largest vocabulary passes
    that check and stops at the next one, a workspace too small (also on
    the host, before any CUDA call)."""
    for dtype, vmax in ((0, 524288), (1, 262144)):
        v = vmax + 1
        assert _verify(lib, dtype=dtype, vocab=v, ldp=v, ldq=v) == _lib.ISD_ERR_UNSUPPORTED
        assert _verify(lib, dtype=dtype, vocab=vmax, ldp=vmax, ldq=vmax, wsb=1) == _lib.ISD_ERR_WORKSPACE
        assert lib.isd_verify_workspace_bytes(64, 512, vmax, dtype) > 0


def test_verify_relaxed_host_checks(lib):
    """tau must be finite and >= 0; the other checks are isd_verify's."""
    for bad in (-0.5, float("nan"), float("inf")):
        assert _verify_relaxed(lib, bad) == _lib.ISD_ERR_INVALID_ARG
    assert _verify_relaxed(lib, 0.5, C=0) == _lib.ISD_OK
    assert _verify_relaxed(lib, 0.5, p=FAKE + 2) == _lib.ISD_ERR_UNSUPPORTED
    assert _verify_relaxed(lib, 0.5, wsb=16) == _lib.ISD_ERR_WORKSPACE


def _verify_propose(lib, **kw):
    args = dict(p=FAKE, ldp=1024, q=FAKE, ldq=1024, dtype=0, vocab=1024, tokens=FAKE, offs=FAKE,
                C=2, total=4, temp=FAKE, seed=0, offset=0, tau=0.0, acc=FAKE, out=FAKE, ratio=FAKE,
                alpha=FAKE, qnew=FAKE, ldn=1024, props=FAKE, valid=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.isd_verify_propose(*args.values())


def test_verify_propose_host_checks(lib):
    """The fused call needs its qnew rows and proposal outputs, except for an
    empty batch; qnew's base must be 16-byte aligned like p's and q's."""
    assert _verify_propose(lib, C=0, qnew=None, props=None, valid=None) == _lib.ISD_OK
    for k in ("qnew", "props", "valid"):
        assert _verify_propose(lib, **{k: None}) == _lib.ISD_ERR_INVALID_ARG
    assert _verify_propose(lib, ldn=1000) == _lib.ISD_ERR_INVALID_ARG
    assert _verify_propose(lib, qnew=FAKE + 4) == _lib.ISD_ERR_UNSUPPORTED
    assert _verify_propose(lib, tau=-1.0) == _lib.ISD_ERR_INVALID_ARG
    assert lib.isd_verify_propose_workspace_bytes(64, 512, 151936, 0) > lib.isd_verify_workspace_bytes(64, 512, 151936, 0)
    # The fused call's workspace check uses its own, larger size.
    small = lib.isd_verify_workspace_bytes(64, 512, 151936, 0)
    assert _verify_propose(lib, C=64, total=512, vocab=151936, ldp=151936, ldq=151936, ldn=151936,
                           wsb=small) == _lib.ISD_ERR_WORKSPACE


def test_propose_and_alpha_host_checks(lib):
    base = [FAKE, 1024, 0, 1024, FAKE, 2, 4, FAKE, 0, 0, None, FAKE, FAKE, FAKE, 1 << 30, None]
    bad = list(base); bad[1] = 10
    assert lib.isd_propose(*bad) == _lib.ISD_ERR_INVALID_ARG
    bad = list(base); bad[0] = FAKE + 4
    assert lib.isd_propose(*bad) == _lib.ISD_ERR_UNSUPPORTED
    bad = list(base); bad[14] = 8
    assert lib.isd_propose(*bad) == _lib.ISD_ERR_WORKSPACE
    bad = list(base); bad[5] = 0
    assert lib.isd_propose(*bad) == _lib.ISD_OK
    assert lib.isd_alpha(FAKE, FAKE, 0, 0, FAKE, FAKE, None) == _lib.ISD_OK
    assert lib.isd_alpha(None, FAKE, 3, 4, FAKE, FAKE, None) == _lib.ISD_ERR_INVALID_ARG
    assert lib.isd_alpha(FAKE, FAKE, -3, 4, FAKE, FAKE, None) == _lib.ISD_ERR_INVALID_ARG


def _verify_filtered(lib, **kw):
    args = dict(p=FAKE, ldp=1024, q=FAKE, ldq=1024, dtype=0, vocab=1024, tokens=FAKE, offs=FAKE,
                C=2, total=4, temp=FAKE, seed=0, offset=0, top_k=50, top_p=0.95, acc=FAKE, out=FAKE,
                ratio=FAKE, alpha=FAKE, ws=FAKE, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.isd_verify_filtered(*args.values())


def _propose_filtered(lib, **kw):
    args = dict(qnew=FAKE, ld=1024, dtype=0, vocab=1024, offs=FAKE, C=2, total=4, temp=FAKE, seed=0,
                offset=0, top_k=50, top_p=0.95, acc=None, props=FAKE, valid=FAKE, ws=FAKE, wsb=1 << 30,
                stream=None)
    args.update(kw)
    return lib.isd_propose_filtered(*args.values())


def test_filtered_host_checks(lib):
    """top_k in [1, 64] and top_p in (0, 1]; the rest as isd_verify and
    isd_propose; every refusal happens before a launch."""
    for fn in (_verify_filtered, _propose_filtered):
        assert fn(lib, C=0) == _lib.ISD_OK
        for kw in (dict(top_k=0), dict(top_k=65), dict(top_p=0.0), dict(top_p=-0.5), dict(top_p=1.5),
                   dict(top_p=float("nan")), dict(C=-1), dict(vocab=0), dict(dtype=3), dict(ws=None)):
            assert fn(lib, **kw) == _lib.ISD_ERR_INVALID_ARG, (fn.__name__, kw)
        assert fn(lib, wsb=16) == _lib.ISD_ERR_WORKSPACE
        assert fn(lib, ws=FAKE + 16) == _lib.ISD_ERR_WORKSPACE
    assert _verify_filtered(lib, p=FAKE + 2) == _lib.ISD_ERR_UNSUPPORTED
    assert _verify_filtered(lib, ldq=1000) == _lib.ISD_ERR_INVALID_ARG
    assert _propose_filtered(lib, qnew=FAKE + 4) == _lib.ISD_ERR_UNSUPPORTED
    assert _propose_filtered(lib, ld=10) == _lib.ISD_ERR_INVALID_ARG
    # 8 bytes per kept entry of every row read, 256-byte granular; 0 for a bad top_k.
    a = lib.isd_verify_filtered_workspace_bytes(64, 512, 50)
    assert a >= 8 * 50 * (2 * 512 + 64) and a % 256 == 0
    assert lib.isd_propose_filtered_workspace_bytes(64, 512, 50) >= 8 * 50 * 512
    assert lib.isd_verify_filtered_workspace_bytes(64, 512, 0) == 0
    assert lib.isd_propose_filtered_workspace_bytes(64, 512, 65) == 0


def _kv_commit(lib, **kw):
    args = dict(table=FAKE, ld=64, seq_len=FAKE, pend=FAKE, alloc=FAKE, free_slots=FAKE, free_top=FAKE,
                pool=1024, accept=FAKE, C=4, M=7, status=FAKE, stream=None)
    args.update(kw)
    return lib.isd_kv_commit(*args.values())


def test_kv_commit_host_checks(lib):
    """Bad sizes and missing pointers are refused before any launch (a
    valid call always launches: even an empty batch writes its status)."""
    for kw in (dict(C=-1), dict(ld=0), dict(pool=-1), dict(M=-1), dict(M=32), dict(status=None),
               dict(free_top=None), dict(free_slots=None), dict(table=None), dict(seq_len=None),
               dict(pend=None), dict(alloc=None), dict(accept=None)):
        assert _kv_commit(lib, **kw) == _lib.ISD_ERR_INVALID_ARG, kw
    assert _kv_commit(lib, C=_lib.ISD_KV_MAX_SEQS + 1) == _lib.ISD_ERR_UNSUPPORTED
    # Pool and batch pointers are only required when there is something behind them.
    assert _kv_commit(lib, C=-1, table=None, seq_len=None) == _lib.ISD_ERR_INVALID_ARG


def test_decision_uniforms_host_checks(lib):
    assert lib.isd_decision_uniforms(0, 0, None, 0, None, None) == _lib.ISD_OK   # nothing to do
    assert lib.isd_decision_uniforms(0, 0, FAKE, -1, FAKE, None) == _lib.ISD_ERR_INVALID_ARG
    assert lib.isd_decision_uniforms(0, 0, None, 4, FAKE, None) == _lib.ISD_ERR_INVALID_ARG
    assert lib.isd_decision_uniforms(0, 0, FAKE, 4, None, None) == _lib.ISD_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIBRARY", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()
