"""ctypes binding of ``libdsa.so`` (include/dsa.h): argument marshalling only.

Every compute step runs in the library's CUDA kernels.  If the library is not
built, the first call raises; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA = 0, 1, 2, 3
DSA_ERR_WORKSPACE, DSA_ERR_TIMEOUT, DSA_ERR_BAD_INPUT = 4, 5, 6
DSA_BF16, DSA_FP8_E4M3_ROWSCALE, DSA_FP8_DS_MLA, DSA_NVFP4 = 0, 1, 2, 3
EXPORTS = ("dsa_workspace_size", "dsa_index_scores", "dsa_topk", "sparse_mla_decode", "dsa_decode_layer",
           "dsa_decode_layer_launches", "dsa_decode_layer_launches_for", "sparse_mla_decode_noalloc",
           "dsa_last_error_string", "dsa_status_string", "dsa_version")


class DcpShard(ctypes.Structure):
    """dsa_dcp_shard: token t lives on rank (t // interleave) % world."""
    _fields_ = [("world", ctypes.c_int32), ("rank", ctypes.c_int32), ("interleave", ctypes.c_int32)]


class DsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


class DsaSeqsC(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("max_ctx", ctypes.c_int32), ("max_q_per_seq", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("num_rows", ctypes.c_int64), ("ctx_len", ctypes.c_void_p), ("q_start", ctypes.c_void_p),
                ("q_pos", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("seq_base", ctypes.c_void_p),
                ("q_rope_pos", ctypes.c_void_p)]


class DsaLayerArgsC(ctypes.Structure):
    _fields_ = [("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("ssmax_s", ctypes.c_void_p),
                ("ssmax_b", ctypes.c_void_p), ("inv_freq", ctypes.c_void_p), ("k_idx", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("k_dtype", ctypes.c_int), ("reuse_idx", ctypes.c_int32),
                ("k", ctypes.c_int32), ("select_block", ctypes.c_int32), ("idx", ctypes.c_void_p),
                ("topk_len", ctypes.c_void_p), ("q_mla", ctypes.c_void_p), ("latent", ctypes.c_void_p),
                ("latent_dtype", ctypes.c_int), ("sm_scale", ctypes.c_float), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("events", ctypes.c_void_p), ("latent_scales", ctypes.c_void_p),
                ("latent_global", ctypes.c_float), ("k_global", ctypes.c_float), ("k_block_scales", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load and type the library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is not built: run __graft_entry__.build() "
                               "(nvcc, sm_103a); there is no CPU fallback")
        L = ctypes.CDLL(path)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        S = ctypes.POINTER(DsaSeqsC)
        L.dsa_workspace_size.argtypes = [S, I32, I32, ctypes.POINTER(SZ)]
        L.dsa_index_scores.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, S, I32, P, I64, P, SZ, P, P]
        L.dsa_index_scores_nvfp4.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, S, I32, P, I64, P, SZ, P, P]
        L.dsa_index_scores_nvfp4.restype = ctypes.c_int
        L.dsa_topk.argtypes = [P, I64, S, I32, I32, P, P, P, SZ, P, P]
        L.sparse_mla_decode.argtypes = [P, P, ctypes.c_int, S, I32, P, P, I32, ctypes.c_float, P, P, P, SZ, P, P]
        L.dsa_decode_layer.argtypes = [ctypes.POINTER(DsaLayerArgsC), S, I32, P, SZ, P, P]
        L.sparse_mla_decode_noalloc.argtypes = [P, P, ctypes.c_int, S, I32, P, P, I32, ctypes.c_float, P, P, P, P]
        L.sparse_mla_decode_noalloc.restype = ctypes.c_int
        L.sparse_mla_decode_nvfp4.argtypes = [P, P, P, ctypes.c_float, S, I32, P, P, I32, ctypes.c_float, P, P, P, SZ,
                                              P, P]
        L.sparse_mla_decode_nvfp4.restype = ctypes.c_int
        L.dsa_decode_layer_launches.argtypes = [S, I32, I32, I32, ctypes.c_int]
        L.dsa_decode_layer_launches_for.argtypes = [ctypes.POINTER(DsaLayerArgsC), S, I32]
        L.dsa_decode_layer_launches_for.restype = ctypes.c_int32
        F = ctypes.c_float
        L.dsa_index_k_insert.argtypes = [P, P, P, F, P, P, P, I32, P, P, ctypes.c_int, I64, P, P]
        L.dsa_latent_insert.argtypes = [P, P, P, P, P, I32, P, ctypes.c_int, I64, P, P]
        L.dsa_mla_q_prep.argtypes = [P, P, P, P, P, I32, P, P, P]
        SH = ctypes.POINTER(DcpShard)
        L.dsa_topk_candidates.argtypes = [P, I64, S, I32, I32, SH, P, P, P, P, SZ, P, P]
        L.dsa_topk_merge.argtypes = [P, I32, I32, I32, I32, P, P, P, P]
        L.dsa_topk_compact.argtypes = [P, P, I32, I32, SH, P, P, P, P]
        L.dsa_lse_combine.argtypes = [P, P, I32, I32, P, P, P]
        L.dsa_dcp_shard_seqs.argtypes = [S, I32, SH, P, P, P, I32, ctypes.POINTER(I32), P, P]
        L.dsa_block_topk.argtypes = [P, I64, S, I32, I32, I32, P, P, P, P]
        L.dsa_decode_layer_launches.restype = ctypes.c_int32
        for f in ("dsa_workspace_size", "dsa_index_scores", "dsa_topk", "sparse_mla_decode", "dsa_decode_layer"):
            getattr(L, f).restype = ctypes.c_int
        L.dsa_last_error_string.restype = ctypes.c_char_p
        L.dsa_status_string.restype = ctypes.c_char_p
        L.dsa_status_string.argtypes = [ctypes.c_int]
        L.dsa_version.restype = ctypes.c_char_p
        _lib = L
        return L


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != DSA_OK:
        L = load()
        raise DsaError(rc, L.dsa_last_error_string().decode())


class Seqs:
    """Where tokens live (include/dsa.h, dsa_seqs): device tensors plus the
    host-side bounds.  Keeps the tensors alive while calls are enqueued."""

    def __init__(self, ctx_len, q_start, q_pos, *, max_ctx: int, max_q_per_seq: int, num_rows: int,
                 page_table=None, page_size: int = 0, seq_base=None, q_rope_pos=None):
        self.ctx_len, self.q_start, self.q_pos = ctx_len, q_start, q_pos
        self.q_rope_pos = q_rope_pos
        self.page_table, self.seq_base = page_table, seq_base
        self.num_seqs = int(ctx_len.shape[0])
        self.num_q = int(q_pos.shape[0])
        self.max_ctx, self.max_q_per_seq, self.num_rows = int(max_ctx), int(max_q_per_seq), int(num_rows)
        self.page_size = int(page_size)
        self.max_pages = int(page_table.shape[1]) if page_table is not None else 0

    def c(self) -> DsaSeqsC:
        return DsaSeqsC(self.num_seqs, self.max_ctx, self.max_q_per_seq, self.page_size, self.max_pages, 0,
                        self.num_rows, _p(self.ctx_len), _p(self.q_start), _p(self.q_pos), _p(self.page_table),
                        _p(self.seq_base), _p(self.q_rope_pos))


def dsa_workspace_size(seqs: Seqs, num_q: int, k: int) -> int:
    n = ctypes.c_size_t()
    sc = seqs.c()
    _check(load().dsa_workspace_size(ctypes.byref(sc), num_q, k, ctypes.byref(n)))
    return int(n.value)


def dsa_index_scores(q_idx, w, ssmax_s, ssmax_b, inv_freq, k_idx, k_scale, k_dtype: int, seqs: Seqs, num_q: int,
                     scores, ld: int, workspace, workspace_bytes: int, d_status=None, stream=None):
    sc = seqs.c()
    _check(load().dsa_index_scores(_p(q_idx), _p(w), _p(ssmax_s), _p(ssmax_b), _p(inv_freq), _p(k_idx), _p(k_scale),
                                   k_dtype, ctypes.byref(sc), num_q, _p(scores), ld, _p(workspace), workspace_bytes,
                                   _p(d_status), _stream(stream)))


def dsa_index_scores_nvfp4(q_idx, w, ssmax_s, ssmax_b, inv_freq, k_codes, k_block_scales, k_global: float,
                           seqs: Seqs, num_q: int, scores, ld: int, workspace, workspace_bytes: int, d_status=None,
                           stream=None):
    sc = seqs.c()
    _check(load().dsa_index_scores_nvfp4(_p(q_idx), _p(w), _p(ssmax_s), _p(ssmax_b), _p(inv_freq), _p(k_codes),
                                         _p(k_block_scales), float(k_global), ctypes.byref(sc), num_q, _p(scores), ld,
                                         _p(workspace), workspace_bytes, _p(d_status), _stream(stream)))


def dsa_topk(scores, ld: int, seqs: Seqs, num_q: int, k: int, idx, topk_len, workspace=None,
             workspace_bytes: int = 0, d_status=None, stream=None):
    sc = seqs.c()
    _check(load().dsa_topk(_p(scores), ld, ctypes.byref(sc), num_q, k, _p(idx), _p(topk_len), _p(workspace),
                           workspace_bytes, _p(d_status), _stream(stream)))


def sparse_mla_decode(q, latent, latent_dtype: int, seqs: Seqs, num_q: int, idx, topk_len, k: int, sm_scale: float,
                      out, lse, workspace, workspace_bytes: int, d_status=None, stream=None):
    sc = seqs.c()
    _check(load().sparse_mla_decode(_p(q), _p(latent), latent_dtype, ctypes.byref(sc), num_q, _p(idx), _p(topk_len),
                                    k, float(sm_scale), _p(out), _p(lse), _p(workspace), workspace_bytes,
                                    _p(d_status), _stream(stream)))


def sparse_mla_decode_nvfp4(q, codes, block_scales, g: float, seqs: Seqs, num_q: int, idx, topk_len, k: int,
                            sm_scale: float, out, lse=None, workspace=None, workspace_bytes: int = 0, d_status=None,
                            stream=None):
    sc = seqs.c()
    _check(load().sparse_mla_decode_nvfp4(_p(q), _p(codes), _p(block_scales), float(g), ctypes.byref(sc), num_q,
                                          _p(idx), _p(topk_len), k, float(sm_scale), _p(out), _p(lse), _p(workspace),
                                          workspace_bytes, _p(d_status), _stream(stream)))


def sparse_mla_decode_noalloc(q, latent, latent_dtype: int, seqs: Seqs, num_q: int, idx, topk_len, k: int,
                              sm_scale: float, out, lse, d_status=None, stream=None):
    """sparse_mla_decode for callers that cannot allocate: no workspace, the
    partials live in the library's static device scratch (see include/dsa.h)."""
    sc = seqs.c()
    _check(load().sparse_mla_decode_noalloc(_p(q), _p(latent), latent_dtype, ctypes.byref(sc), num_q, _p(idx),
                                            _p(topk_len), k, float(sm_scale), _p(out), _p(lse), _p(d_status),
                                            _stream(stream)))


def dsa_decode_layer_launches(seqs: Seqs, num_q: int, k: int, reuse_idx: int = 0, latent_dtype: int = 0) -> int:
    sc = seqs.c()
    return int(load().dsa_decode_layer_launches(ctypes.byref(sc), num_q, k, reuse_idx, latent_dtype))


def _layer_args(args: dict):
    """dsa_layer_args from fields by name (tensors or None); returns the struct
    and what must stay alive while it is used."""
    a = DsaLayerArgsC()
    keep = None
    for name, ctype in DsaLayerArgsC._fields_:
        v = args.get(name)
        if v is None:
            continue
        if name == "events":
            keep = (ctypes.c_void_p * 4)(*[e.cuda_event for e in v])
            a.events = ctypes.cast(keep, ctypes.c_void_p)
            continue
        if ctype is ctypes.c_void_p:
            setattr(a, name, _p(v))
        elif ctype is ctypes.c_float:
            setattr(a, name, float(v))
        else:
            setattr(a, name, int(v))
    return a, keep


def dsa_decode_layer(args: dict, seqs: Seqs, num_q: int, workspace, workspace_bytes: int, d_status=None,
                     stream=None):
    """``args`` holds the dsa_layer_args fields by name (tensors or None);
    ``events`` may be a list of 4 recorded torch.cuda.Event objects."""
    a, keep = _layer_args(args)
    sc = seqs.c()
    _check(load().dsa_decode_layer(ctypes.byref(a), ctypes.byref(sc), num_q, _p(workspace), workspace_bytes,
                                   _p(d_status), _stream(stream)))
    del keep


def dsa_decode_layer_launches_for(args: dict, seqs: Seqs, num_q: int) -> int:
    a, _ = _layer_args({k: v for k, v in args.items() if k != "events"})
    sc = seqs.c()
    return int(load().dsa_decode_layer_launches_for(ctypes.byref(a), ctypes.byref(sc), num_q))


def version() -> str:
    return load().dsa_version().decode()


# ---- the cache-write side (include/dsa.h)
def dsa_index_k_insert(x, ln_gamma, ln_beta, ln_eps: float, pos, inv_freq, slot, n: int, k_cache, k_scale,
                       k_dtype: int, num_rows: int, d_status=None, stream=None):
    _check(load().dsa_index_k_insert(_p(x), _p(ln_gamma), _p(ln_beta), float(ln_eps), _p(pos), _p(inv_freq), _p(slot),
                                     n, _p(k_cache), _p(k_scale), k_dtype, num_rows, _p(d_status), _stream(stream)))


def dsa_latent_insert(c_kv, k_pe, pos, inv_freq, slot, n: int, latent, latent_dtype: int, num_rows: int,
                      d_status=None, stream=None):
    _check(load().dsa_latent_insert(_p(c_kv), _p(k_pe), _p(pos), _p(inv_freq), _p(slot), n, _p(latent), latent_dtype,
                                    num_rows, _p(d_status), _stream(stream)))


def dsa_mla_q_prep(q, ssmax_s, ssmax_b, inv_freq, q_pos, num_q: int, q_out, d_status=None, stream=None):
    _check(load().dsa_mla_q_prep(_p(q), _p(ssmax_s), _p(ssmax_b), _p(inv_freq), _p(q_pos), num_q, _p(q_out),
                                 _p(d_status), _stream(stream)))


# ---- DCP: one rank's compute steps (include/dsa.h)
def _ptr_array(tensors):
    """Host array of device pointers (kept alive by the caller's reference)."""
    arr = (ctypes.c_void_p * len(tensors))(*[_p(t) for t in tensors])
    return arr


def dsa_topk_candidates(scores, ld: int, seqs: Seqs, num_q: int, k: int, shard: DcpShard, idx, topk_len, cand,
                        workspace=None, workspace_bytes: int = 0, d_status=None, stream=None):
    sc = seqs.c()
    _check(load().dsa_topk_candidates(_p(scores), ld, ctypes.byref(sc), num_q, k, ctypes.byref(shard), _p(idx),
                                      _p(topk_len), _p(cand), _p(workspace), workspace_bytes, _p(d_status),
                                      _stream(stream)))


def dsa_topk_merge(lists, list_len: int, num_q: int, k: int, idx, topk_len, d_status=None, stream=None):
    arr = _ptr_array(lists)
    _check(load().dsa_topk_merge(ctypes.cast(arr, ctypes.c_void_p), len(lists), list_len, num_q, k, _p(idx),
                                 _p(topk_len), _p(d_status), _stream(stream)))


def dsa_topk_compact(idx, topk_len, num_q: int, k: int, shard: DcpShard, local_idx, local_len, d_status=None,
                     stream=None):
    _check(load().dsa_topk_compact(_p(idx), _p(topk_len), num_q, k, ctypes.byref(shard), _p(local_idx),
                                   _p(local_len), _p(d_status), _stream(stream)))


def dsa_dcp_shard_seqs(seqs: Seqs, num_q: int, shard: DcpShard, local_ctx_len, local_q_pos, local_page_table=None,
                       local_max_pages: int = 0, d_status=None, stream=None) -> int:
    """Fills one rank's local context lengths, causal bounds and (optionally)
    page table; returns the rank's local max_ctx (host)."""
    sc = seqs.c()
    out = ctypes.c_int32(0)
    _check(load().dsa_dcp_shard_seqs(ctypes.byref(sc), num_q, ctypes.byref(shard), _p(local_ctx_len), _p(local_q_pos),
                                     _p(local_page_table), int(local_max_pages), ctypes.byref(out), _p(d_status),
                                     _stream(stream)))
    return int(out.value)


def dsa_lse_combine(o_parts, lse_parts, num_q: int, out, lse=None, stream=None):
    if len(o_parts) != len(lse_parts):
        raise ValueError("o_parts and lse_parts differ in length")
    oa, la = _ptr_array(o_parts), _ptr_array(lse_parts)
    _check(load().dsa_lse_combine(ctypes.cast(oa, ctypes.c_void_p), ctypes.cast(la, ctypes.c_void_p), len(o_parts),
                                  num_q, _p(out), _p(lse), _stream(stream)))


# ---- block-sparse selection (include/dsa.h)
def dsa_block_topk(scores, ld: int, seqs: Seqs, num_q: int, block: int, nsel: int, idx, topk_len, d_status=None,
                   stream=None):
    sc = seqs.c()
    _check(load().dsa_block_topk(_p(scores), ld, ctypes.byref(sc), num_q, block, nsel, _p(idx), _p(topk_len),
                                 _p(d_status), _stream(stream)))
