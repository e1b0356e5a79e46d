"""The C ABI without a GPU: the library loads, exports every entry point that
include/dsa.h declares, and refuses bad arguments on the host (before any
CUDA call) with a status and a message listing every reason."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    from dsa_sparse_mla_query_gb300 import _binding as B
    from dsa_sparse_mla_query_gb300 import build
    build.build()
    return B.load()


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("dsa_workspace_size", "dsa_index_scores", "dsa_topk", "sparse_mla_decode", "dsa_decode_layer",
              "dsa_last_error_string", "dsa_status_string", "dsa_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"libdsa.so does not export {n}"


def test_version_and_status_names(lib):
    assert lib.dsa_version().decode().count(".") == 2
    assert lib.dsa_status_string(0) == b"DSA_OK"
    assert lib.dsa_status_string(6) == b"DSA_ERR_BAD_INPUT"


def _seqs(B, **kw):
    base = dict(num_seqs=1, max_ctx=4096, max_q_per_seq=1, page_size=0, max_pages=0, reserved=0, num_rows=4096,
                ctx_len=0x1000, q_start=0x2000, q_pos=0x3000, page_table=None, seq_base=0x4000)
    base.update(kw)
    return B.DsaSeqsC(**base)


def test_host_validation_lists_every_reason(lib):
    from dsa_sparse_mla_query_gb300 import _binding as B
    s = _seqs(B, num_seqs=0, q_pos=None)
    rc = lib.dsa_index_scores(None, None, 0x10, 0x10, None, 0x10, None, 7, ctypes.byref(s), 1, 0x10, 3, None, 0,
                              None, None)
    assert rc == B.DSA_ERR_INVALID_ARG
    msg = lib.dsa_last_error_string().decode()
    for part in ("num_seqs 0", "seqs.q_pos is NULL", "q_idx is NULL", "w is NULL", "dtype 7", "ld 3"):
        assert part in msg, (part, msg)


def test_workspace_size_and_refusals(lib):
    from dsa_sparse_mla_query_gb300 import _binding as B
    s = _seqs(B)
    n = ctypes.c_size_t()
    assert lib.dsa_workspace_size(ctypes.byref(s), 4, 2048, ctypes.byref(n)) == 0
    assert n.value > 4 * 4096 * 4
    assert lib.dsa_workspace_size(ctypes.byref(s), 4, 4096, ctypes.byref(n)) == B.DSA_ERR_UNSUPPORTED
    assert "k 4096" in lib.dsa_last_error_string().decode()
    # too-small workspace is refused before anything is enqueued
    rc = lib.sparse_mla_decode(0x100, 0x100, 0, ctypes.byref(s), 4, 0x100, 0x100, 2048, ctypes.c_float(0.07), 0x100,
                               None, 0x100, 16, None, None)
    assert rc == B.DSA_ERR_WORKSPACE
    assert "workspace has 16 bytes" in lib.dsa_last_error_string().decode()
    # misaligned pointer and bad page size
    s2 = _seqs(B, page_table=0x5000, page_size=10, max_pages=4)
    rc = lib.dsa_topk(0x104, 4096, ctypes.byref(s2), 1, 2048, 0x200, 0x300, None, 0, None, None)
    assert rc != 0
    msg = lib.dsa_last_error_string().decode()
    assert "scores is not 16-byte aligned" in msg and "page_size 10 is not a power of two" in msg


def test_zero_queries_is_a_no_op(lib):
    from dsa_sparse_mla_query_gb300 import _binding as B
    s = _seqs(B)
    rc = lib.dsa_topk(0x100, 4096, ctypes.byref(s), 0, 2048, 0x200, 0x300, None, 0, None, None)
    assert rc == 0


def test_binding_fails_loudly_without_library(tmp_path):
    from dsa_sparse_mla_query_gb300 import _binding as B
    with pytest.raises(RuntimeError, match="not built"):
        B._lib_saved = B._lib
        try:
            B._lib = None
            B.load(str(tmp_path / "missing.so"))
        finally:
            B._lib = B._lib_saved


def test_dcp_calls_refuse_bad_arguments(lib):
    """The DCP calls refuse, on the host and with every reason listed, what
    they cannot serve; nothing is enqueued (no GPU needed)."""
    from dsa_sparse_mla_query_gb300 import _binding as B
    P = ctypes.c_void_p

    def msg():
        return lib.dsa_last_error_string().decode()

    many = (P * 17)(*([0x100] * 17))
    assert lib.dsa_topk_merge(ctypes.cast(many, P), 17, 64, 1, 2048, 0x200, 0x300, None, None) == \
        B.DSA_ERR_UNSUPPORTED
    assert "num_lists 17" in msg()
    eight = (P * 8)(*([0x100] * 8))
    assert lib.dsa_topk_merge(ctypes.cast(eight, P), 8, 4096, 1, 2048, 0x200, 0x300, None, None) == \
        B.DSA_ERR_UNSUPPORTED
    assert "exceeds 16384" in msg()
    bad = (P * 3)(0x100, None, 0x104)
    assert lib.dsa_topk_merge(ctypes.cast(bad, P), 3, 64, 1, 2048, 0x200, 0x300, None, None) == \
        B.DSA_ERR_INVALID_ARG
    assert "lists[r] is NULL" in msg() and "lists[r] is not 8-byte aligned" in msg()
    assert lib.dsa_topk_merge(None, 2, 64, 1, 2048, 0x200, 0x300, None, None) == B.DSA_ERR_INVALID_ARG
    assert "lists (host array) is NULL" in msg()

    sh = B.DcpShard(4, 4, 0)
    assert lib.dsa_topk_compact(0x100, 0x200, 1, 2048, ctypes.byref(sh), 0x300, 0x400, None, None) == \
        B.DSA_ERR_INVALID_ARG
    assert "shard rank 4" in msg() and "shard interleave 0" in msg()
    assert lib.dsa_topk_compact(0x100, 0x200, 1, 2048, None, 0x300, 0x400, None, None) == B.DSA_ERR_INVALID_ARG
    assert "shard is NULL" in msg()

    s = _seqs(B)
    big = B.DcpShard(17, 0, 1)
    rc = lib.dsa_topk_candidates(0x100, 4096, ctypes.byref(s), 1, 2048, ctypes.byref(big), 0x200, 0x300, 0x404, None,
                                 0, None, None)
    assert rc != 0 and "shard world 17" in msg() and "cand is not 8-byte aligned" in msg()

    assert lib.dsa_lse_combine(ctypes.cast(eight, P), ctypes.cast(eight, P), 0, 1, 0x100, None, None) == \
        B.DSA_ERR_UNSUPPORTED
    assert "num_parts 0" in msg()
    assert lib.dsa_lse_combine(None, None, 2, 1, 0x100, None, None) == B.DSA_ERR_INVALID_ARG


def test_dcp_calls_with_zero_queries_are_no_ops(lib):
    from dsa_sparse_mla_query_gb300 import _binding as B
    P = ctypes.c_void_p
    two = (P * 2)(0x100, 0x200)
    sh = B.DcpShard(2, 1, 64)
    assert lib.dsa_topk_merge(ctypes.cast(two, P), 2, 64, 0, 2048, None, None, None, None) == 0
    assert lib.dsa_topk_compact(None, None, 0, 2048, ctypes.byref(sh), None, None, None, None) == 0
    assert lib.dsa_lse_combine(ctypes.cast(two, P), ctypes.cast(two, P), 2, 0, None, None, None) == 0


def test_block_topk_refuses_what_it_cannot_serve(lib):
    """Block selection: sizes past the selection width, too many blocks for one
    CTA, bad counts and pointers are refused on the host (no GPU needed)."""
    from dsa_sparse_mla_query_gb300 import _binding as B
    s = _seqs(B)

    def call(block, nsel, seqs=s, scores=0x100, idx=0x200):
        return lib.dsa_block_topk(scores, 4096, ctypes.byref(seqs), 1, block, nsel, idx, 0x300, None, None)

    assert call(128, 17) == B.DSA_ERR_UNSUPPORTED and "exceeds 2048" in lib.dsa_last_error_string().decode()
    assert call(0, 16) == B.DSA_ERR_UNSUPPORTED
    assert call(32, 65) == B.DSA_ERR_UNSUPPORTED
    big = _seqs(B, max_ctx=1 << 30)
    rc = lib.dsa_block_topk(0x100, 1 << 30, ctypes.byref(big), 1, 128, 16, 0x200, 0x300, None, None)
    assert rc == B.DSA_ERR_UNSUPPORTED and "too many blocks" in lib.dsa_last_error_string().decode()
    assert call(128, 16, scores=None, idx=0x202) == B.DSA_ERR_INVALID_ARG
    msg = lib.dsa_last_error_string().decode()
    assert "scores is NULL" in msg and "idx is not 4-byte aligned" in msg
    assert lib.dsa_block_topk(0x100, 4096, ctypes.byref(s), 0, 128, 16, 0x200, 0x300, None, None) == 0


def _declared_arities():
    """Parameter count of every function include/dsa.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.M | re.S):
        name, params = m.group(1), m.group(2).strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argtypes_match_the_header(lib):
    """Every entry point the binding declares argument types for takes as many
    arguments as the header says (a drift would shift arguments silently)."""
    ar = _declared_arities()
    assert set(ar) == set(declared_functions()), "every declaration parsed"
    checked = 0
    for name, n in ar.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == n, f"{name}: binding has {len(fn.argtypes)} argument types, header {n}"
        checked += 1
    assert checked >= len(ar) - 3  # all but the argument-free ones
