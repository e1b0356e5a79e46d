"""CPU oracle for the DSA decode path -- TEST INFRASTRUCTURE ONLY.

Python marshalling for ``dsa_oracle.c`` (plain single-threaded fp64 C).  Only
the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package; the product path never does.

Functions take numpy arrays (or CPU torch tensors) and return numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

KEYS_BF16, KEYS_E4M3_ROW, KEYS_NVFP4 = 0, 1, 2
LATENT_BF16, LATENT_DS_MLA, LATENT_NVFP4 = 0, 2, 3
ERRORS = {-1: "bad argument", -2: "query position outside the context", -3: "page or row outside the cache",
          -4: "selected index outside the context", -5: "out of memory"}


def compile_oracle(src: str, out: str) -> str:
    """gcc, fp64, no FMA contraction (so x86 and Arm round the same way)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-shared", "-fPIC",
                           "-I", _HERE, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def _foreign(path: str) -> bool:
    import platform
    want = {"x86_64": 0x3E, "AMD64": 0x3E, "aarch64": 0xB7, "arm64": 0xB7}.get(platform.machine())
    with open(path, "rb") as f:
        head = f.read(20)
    return len(head) < 20 or head[:4] != b"\x7fELF" or int.from_bytes(head[18:20], "little") != want


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or _foreign(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "dsa_oracle.h"))):
        compile_oracle(_SRC, _LIB)
    return _LIB


def load(path: str):
    """A handle on another build of the oracle (e.g. a deliberately broken
    copy in a test); pass it as ``L=`` to the functions below."""
    return _bind(path)


class Seqs(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("ctx_len", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("seq_base", ctypes.c_void_p),
                ("num_rows", ctypes.c_int64)]


def _bind(path: str):
    L = ctypes.CDLL(path)
    P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    L.oracle_bf16_value.argtypes, L.oracle_bf16_value.restype = [ctypes.c_uint16], D
    L.oracle_e4m3_value.argtypes, L.oracle_e4m3_value.restype = [ctypes.c_uint8], D
    L.oracle_ds_mla_row.argtypes, L.oracle_ds_mla_row.restype = [P, P], ctypes.c_int
    L.oracle_index_scores.argtypes = [I32, P, P, P, P, P, P, P, I32, P, P, ctypes.POINTER(Seqs), P, I64]
    L.oracle_index_scores.restype = ctypes.c_int
    L.oracle_topk.argtypes, L.oracle_topk.restype = [P, I32, I32, P, ctypes.POINTER(I32)], ctypes.c_int
    L.oracle_sparse_mla.argtypes = [P, I32, P, ctypes.POINTER(Seqs), I32, P, I32, D, P, P, P]
    L.oracle_sparse_mla.restype = ctypes.c_int
    L.oracle_latent_row_bytes.argtypes, L.oracle_latent_row_bytes.restype = [I32], I64
    L.oracle_index_row_bytes.argtypes, L.oracle_index_row_bytes.restype = [I32], I64
    L.oracle_bf16_encode.argtypes, L.oracle_bf16_encode.restype = [D], ctypes.c_uint16
    L.oracle_e4m3_encode.argtypes, L.oracle_e4m3_encode.restype = [D], ctypes.c_uint8
    L.oracle_index_k.argtypes, L.oracle_index_k.restype = [I32, P, P, P, D, P, P, P], ctypes.c_int
    L.oracle_latent_k.argtypes, L.oracle_latent_k.restype = [I32, P, P, P, P, P], ctypes.c_int
    L.oracle_mla_q.argtypes, L.oracle_mla_q.restype = [I32, P, P, P, P, P, P], ctypes.c_int
    L.oracle_dcp_owner.argtypes, L.oracle_dcp_owner.restype = [I32, I32, I32], I32
    L.oracle_dcp_local.argtypes, L.oracle_dcp_local.restype = [I32, I32, I32], I32
    L.oracle_dcp_global.argtypes, L.oracle_dcp_global.restype = [I32, I32, I32, I32], I32
    L.oracle_dcp_pack.argtypes, L.oracle_dcp_pack.restype = [ctypes.c_float, I32], ctypes.c_uint64
    L.oracle_dcp_unpack.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(I32)]
    L.oracle_dcp_unpack.restype = ctypes.c_int
    L.oracle_topk_merge.argtypes = [I32, I32, P, I32, P, ctypes.POINTER(I32)]
    L.oracle_topk_merge.restype = ctypes.c_int
    L.oracle_topk_compact.argtypes = [I32, P, I32, I32, I32, I32, P, ctypes.POINTER(I32)]
    L.oracle_topk_compact.restype = ctypes.c_int
    L.oracle_lse_combine.argtypes, L.oracle_lse_combine.restype = [I32, I64, I32, P, P, P, P], ctypes.c_int
    L.oracle_e2m1_value.argtypes, L.oracle_e2m1_value.restype = [ctypes.c_uint8], D
    L.oracle_e2m1_encode.argtypes, L.oracle_e2m1_encode.restype = [D], ctypes.c_uint8
    L.oracle_nvfp4_quantize.argtypes, L.oracle_nvfp4_quantize.restype = [I32, P, D, P, P], ctypes.c_int
    L.oracle_nvfp4_dequantize.argtypes, L.oracle_nvfp4_dequantize.restype = [I32, P, P, D, P], ctypes.c_int
    L.oracle_block_topk.argtypes = [P, I32, I32, I32, P, ctypes.POINTER(I32)]
    L.oracle_block_topk.restype = ctypes.c_int
    L.oracle_index_scores_nvfp4.argtypes = [I32, P, P, P, P, P, P, P, P, P, D, ctypes.POINTER(Seqs), P, I64]
    L.oracle_index_scores_nvfp4.restype = ctypes.c_int
    L.oracle_sparse_mla_nvfp4.argtypes = [P, P, P, D, ctypes.POINTER(Seqs), I32, P, I32, D, P, P, P]
    L.oracle_sparse_mla_nvfp4.restype = ctypes.c_int
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def _np(x, dtype=None):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().cpu()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.numpy()
    a = np.ascontiguousarray(x)
    if dtype is not None:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype != dtype else a.astype(dtype, copy=False)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc):
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")


class Layout:
    """Host copy of where tokens live; keeps the arrays alive for the call."""

    def __init__(self, ctx_len, num_rows, page_table=None, page_size=0, seq_base=None):
        self.ctx_len = _np(ctx_len, np.int32)
        self.page_table = None if page_table is None else _np(page_table, np.int32)
        self.seq_base = None if seq_base is None else _np(seq_base, np.int64)
        self.page_size = int(page_size)
        self.max_pages = 0 if self.page_table is None else int(self.page_table.shape[-1])
        self.num_rows = int(num_rows)
        if self.page_table is None and self.seq_base is None:
            raise ValueError("need page_table or seq_base")

    def struct(self):
        return Seqs(len(self.ctx_len), _ptr(self.ctx_len), _ptr(self.page_table), self.page_size, self.max_pages,
                    _ptr(self.seq_base), self.num_rows)


def bf16_value(bits: int, L=None) -> float:
    return (L or lib()).oracle_bf16_value(bits & 0xFFFF)


def e4m3_value(code: int, L=None) -> float:
    return (L or lib()).oracle_e4m3_value(code & 0xFF)


def ds_mla_row(row656, L=None) -> np.ndarray:
    r = _np(row656, np.uint8)
    assert r.size == 656
    out = np.empty(576, np.float64)
    _check((L or lib()).oracle_ds_mla_row(_ptr(r), _ptr(out)))
    return out


def latent_row_bytes(kind: int, L=None) -> int:
    return (L or lib()).oracle_latent_row_bytes(kind)


def index_row_bytes(kind: int, L=None) -> int:
    return (L or lib()).oracle_index_row_bytes(kind)


def index_scores(q, w, ssmax_s, ssmax_b, inv_freq, q_seq, q_pos, keys, layout: Layout, key_scale=None,
                 ld=None, L=None) -> np.ndarray:
    """fp64 scores [nq, ld]; -inf after each query's position."""
    q = _np(q, np.uint16)
    w = _np(w, np.float32)
    ss, sb = _np(ssmax_s, np.float32), _np(ssmax_b, np.float32)
    fr = None if inv_freq is None else _np(inv_freq, np.float32)
    qs, qp = _np(q_seq, np.int32), _np(q_pos, np.int32)
    if key_scale is None:
        k, kind, ks = _np(keys, np.uint16), KEYS_BF16, None
    else:
        k, kind, ks = _np(keys, np.uint8), KEYS_E4M3_ROW, _np(key_scale, np.float32)
    nq = qp.shape[0]
    ld = int(layout.ctx_len.max()) if ld is None else int(ld)
    out = np.full((nq, ld), -np.inf, np.float64)
    st = layout.struct()
    _check((L or lib()).oracle_index_scores(nq, _ptr(q), _ptr(w), _ptr(ss), _ptr(sb), _ptr(fr), _ptr(qs), _ptr(qp), kind,
                                     _ptr(k), _ptr(ks), ctypes.byref(st), _ptr(out), ld))
    return out


def topk(scores, k: int, L=None):
    """(idx int32 [k] in selection order, -1 padded; length)."""
    s = _np(scores, np.float64)
    idx = np.empty(k, np.int32)
    n = ctypes.c_int32()
    _check((L or lib()).oracle_topk(_ptr(s), s.shape[0], k, _ptr(idx), ctypes.byref(n)))
    return idx, int(n.value)


def sparse_mla(q, latent, layout: Layout, seq: int, idx, topk_len: int, sm_scale: float, fp8: bool = False,
               want_probs: bool = False, L=None):
    """(out fp64 [64,512], lse fp64 [64], probs [64, topk_len] or None)."""
    qq = _np(q, np.uint16)
    lat = _np(latent, np.uint8 if fp8 else np.uint16)
    ii = _np(idx, np.int32)
    out = np.empty((64, 512), np.float64)
    lse = np.empty(64, np.float64)
    probs = np.empty((64, max(topk_len, 1)), np.float64) if want_probs else None
    st = layout.struct()
    _check((L or lib()).oracle_sparse_mla(_ptr(qq), LATENT_DS_MLA if fp8 else LATENT_BF16, _ptr(lat), ctypes.byref(st),
                                   seq, _ptr(ii), topk_len, sm_scale, _ptr(out), _ptr(lse), _ptr(probs)))
    return out, lse, (probs[:, :topk_len] if want_probs else None)


# ---- the cache-write side
def bf16_encode(v: float, L=None) -> int:
    return int((L or lib()).oracle_bf16_encode(float(v)))


def e4m3_encode(v: float, L=None) -> int:
    return int((L or lib()).oracle_e4m3_encode(float(v)))


def index_k(x, gamma, beta, eps: float, pos, inv_freq=None, L=None) -> np.ndarray:
    """LayerNorm + RoPE of new indexer keys: fp64 [n,128] before storage rounding."""
    xx = _np(x, np.uint16).reshape(-1, 128)
    g, b = _np(gamma, np.float32), _np(beta, np.float32)
    pp = _np(pos, np.int32)
    fr = None if inv_freq is None else _np(inv_freq, np.float32)
    out = np.empty((xx.shape[0], 128), np.float64)
    _check((L or lib()).oracle_index_k(xx.shape[0], _ptr(xx), _ptr(g), _ptr(b), float(eps), _ptr(pp), _ptr(fr),
                                       _ptr(out)))
    return out


def latent_k(c_kv, k_pe, pos, inv_freq=None, L=None) -> np.ndarray:
    """New latent rows: fp64 [n,576] (512 copied, 64 rotated) before storage rounding."""
    c = _np(c_kv, np.uint16).reshape(-1, 512)
    k = _np(k_pe, np.uint16).reshape(-1, 64)
    pp = _np(pos, np.int32)
    fr = None if inv_freq is None else _np(inv_freq, np.float32)
    out = np.empty((c.shape[0], 576), np.float64)
    _check((L or lib()).oracle_latent_k(c.shape[0], _ptr(c), _ptr(k), _ptr(pp), _ptr(fr), _ptr(out)))
    return out


def mla_q(q, ssmax_s, ssmax_b, pos, inv_freq=None, L=None) -> np.ndarray:
    """Attention queries after RoPE + SSMax: fp64 [nq,64,576] before rounding."""
    qq = _np(q, np.uint16).reshape(-1, 64, 576)
    ss, sb = _np(ssmax_s, np.float32), _np(ssmax_b, np.float32)
    pp = _np(pos, np.int32)
    fr = None if inv_freq is None else _np(inv_freq, np.float32)
    out = np.empty(qq.shape, np.float64)
    _check((L or lib()).oracle_mla_q(qq.shape[0], _ptr(qq), _ptr(ss), _ptr(sb), _ptr(fr), _ptr(pp), _ptr(out)))
    return out


def quantize_rows_e4m3(v, group: int, L=None):
    """Per-group e4m3 quantisation of fp64 rows v [n, d] (groups of `group`
    consecutive values): scale = amax / 448 (1 when amax is 0), codes =
    e4m3_encode(v / scale).  Returns (codes uint8 [n, d], scales fp64 [n, d / group])."""
    v = np.asarray(v, np.float64)
    n, d = v.shape
    g = v.reshape(n, d // group, group)
    amax = np.abs(g).max(axis=2)
    scale = np.where(amax > 0, amax / 448.0, 1.0)
    enc = np.vectorize(lambda x: e4m3_encode(x, L), otypes=[np.uint8])
    codes = enc(g / scale[:, :, None]).reshape(n, d)
    return codes, scale


# ---- DCP: the per-rank steps of decode context parallelism ----

def dcp_owner(t: int, world: int, interleave: int, L=None) -> int:
    return int((L or lib()).oracle_dcp_owner(int(t), int(world), int(interleave)))


def dcp_local(t: int, world: int, interleave: int, L=None) -> int:
    return int((L or lib()).oracle_dcp_local(int(t), int(world), int(interleave)))


def dcp_global(local: int, rank: int, world: int, interleave: int, L=None) -> int:
    return int((L or lib()).oracle_dcp_global(int(local), int(rank), int(world), int(interleave)))


def dcp_pack(scores, ids, L=None) -> np.ndarray:
    """Packed candidates (uint64) of fp32 scores and ids, element by element."""
    L = L or lib()
    sc = np.asarray(_np(scores, np.float32), np.float32).ravel()
    ii = np.asarray(ids, np.int64).ravel()
    out = np.empty(sc.shape[0], np.uint64)
    for n in range(sc.shape[0]):
        out[n] = L.oracle_dcp_pack(float(sc[n]), int(ii[n]))
    return out.reshape(np.shape(scores))


def dcp_unpack(c: int, L=None):
    """(score, id) of a packed candidate, or None for an empty slot."""
    sc, i = ctypes.c_float(), ctypes.c_int32()
    if not (L or lib()).oracle_dcp_unpack(ctypes.c_uint64(int(c)), ctypes.byref(sc), ctypes.byref(i)):
        return None
    return float(sc.value), int(i.value)


def topk_merge(lists, k: int, L=None):
    """lists uint64 [R, Q, list_len] -> (ids int32 [Q, k] ascending then -1, len int32 [Q]).
    Raises on an id present twice among a query's candidates."""
    L = L or lib()
    a = np.asarray(_np(lists, np.uint64), np.uint64)
    R, Q, n = a.shape
    ids = np.empty((Q, k), np.int32)
    lens = np.empty(Q, np.int32)
    for q in range(Q):
        per = np.ascontiguousarray(a[:, q, :])
        m = ctypes.c_int32()
        _check(L.oracle_topk_merge(R, n, _ptr(per), k, _ptr(ids[q]), ctypes.byref(m)))
        lens[q] = m.value
    return ids, lens


def topk_compact(idx, lens, rank: int, world: int, interleave: int, L=None):
    """idx int32 [Q, k], lens [Q] -> (local idx int32 [Q, k], local len [Q]) of one rank."""
    L = L or lib()
    ii = np.ascontiguousarray(_np(idx, np.int32))
    ll = _np(lens, np.int32)
    Q, k = ii.shape
    out = np.empty((Q, k), np.int32)
    ol = np.empty(Q, np.int32)
    for q in range(Q):
        m = ctypes.c_int32()
        _check(L.oracle_topk_compact(k, _ptr(ii[q]), int(ll[q]), rank, world, interleave, _ptr(out[q]),
                                     ctypes.byref(m)))
        ol[q] = m.value
    return out, ol


def lse_combine(o_parts, lse_parts, L=None):
    """o_parts [R, ..., dim] (fp64 values), lse_parts [R, ...] -> (out [..., dim], lse [...])."""
    o = np.ascontiguousarray(np.asarray(o_parts, np.float64))
    ls = np.ascontiguousarray(np.asarray(lse_parts, np.float64))
    R, dim = o.shape[0], o.shape[-1]
    rows = int(np.prod(o.shape[1:-1]))
    out = np.empty(o.shape[1:], np.float64)
    lse = np.empty(ls.shape[1:], np.float64)
    _check((L or lib()).oracle_lse_combine(R, rows, dim, _ptr(o), _ptr(ls), _ptr(out), _ptr(lse)))
    return out, lse


# ---- NVFP4 (4.5-bit cache values)
def e2m1_value(nibble: int, L=None) -> float:
    return float((L or lib()).oracle_e2m1_value(nibble & 15))


def e2m1_encode(v: float, L=None) -> int:
    return int((L or lib()).oracle_e2m1_encode(float(v)))


def nvfp4_quantize(v, g: float, L=None):
    """fp64 values [..., n] (n % 16 == 0) -> (codes uint8 [..., n/2], scales uint8 [..., n/16])."""
    a = np.ascontiguousarray(np.asarray(v, np.float64))
    n = a.shape[-1]
    flat = a.reshape(-1)
    codes = np.empty(flat.size // 2, np.uint8)
    scales = np.empty(flat.size // 16, np.uint8)
    _check((L or lib()).oracle_nvfp4_quantize(flat.size, _ptr(flat), float(g), _ptr(codes), _ptr(scales)))
    return codes.reshape(a.shape[:-1] + (n // 2,)), scales.reshape(a.shape[:-1] + (n // 16,))


def nvfp4_dequantize(codes, scales, g: float, L=None) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, np.uint8))
    s = np.ascontiguousarray(np.asarray(scales, np.uint8))
    n = c.shape[-1] * 2
    out = np.empty(c.shape[:-1] + (n,), np.float64)
    _check((L or lib()).oracle_nvfp4_dequantize(c.size * 2, _ptr(c.reshape(-1)), _ptr(s.reshape(-1)), float(g),
                                                _ptr(out.reshape(-1))))
    return out


# ---- block-sparse selection (MiniMax Sparse Attention)
def block_topk(scores, block: int = 128, nsel: int = 16, L=None):
    """Causal scores [n] (the query at n-1) -> (idx int32 [nsel*block], len)."""
    sc = np.ascontiguousarray(np.asarray(scores, np.float64))
    idx = np.empty(nsel * block, np.int32)
    m = ctypes.c_int32()
    _check((L or lib()).oracle_block_topk(_ptr(sc), sc.shape[0], block, nsel, _ptr(idx), ctypes.byref(m)))
    return idx, int(m.value)


def index_scores_nvfp4(q, w, ssmax_s, ssmax_b, inv_freq, q_seq, q_pos, codes, block_scales, g: float,
                       layout: Layout, ld=None, L=None) -> np.ndarray:
    """Scores [nq, ld] over NVFP4 index keys (codes [rows,64], E4M3 scales [rows,8], tensor scale g)."""
    qq = _np(q, np.uint16)
    ww = _np(w, np.float32)
    ss, sb = _np(ssmax_s, np.float32), _np(ssmax_b, np.float32)
    fr = None if inv_freq is None else _np(inv_freq, np.float32)
    qs, qp = _np(q_seq, np.int32), _np(q_pos, np.int32)
    cc, bs = _np(codes, np.uint8), _np(block_scales, np.uint8)
    nq = qp.shape[0]
    ld = int(layout.ctx_len.max()) if ld is None else int(ld)
    out = np.full((nq, ld), -np.inf, np.float64)
    st = layout.struct()
    _check((L or lib()).oracle_index_scores_nvfp4(nq, _ptr(qq), _ptr(ww), _ptr(ss), _ptr(sb), _ptr(fr), _ptr(qs),
                                                  _ptr(qp), _ptr(cc), _ptr(bs), float(g), ctypes.byref(st),
                                                  _ptr(out), ld))
    return out


def sparse_mla_nvfp4(q, codes, block_scales, g: float, layout: Layout, seq: int, idx, topk_len: int,
                     sm_scale: float, L=None):
    """(out fp64 [64,512], lse fp64 [64]) over NVFP4 latent rows (codes [rows,288], scales [rows,36])."""
    qq = _np(q, np.uint16)
    cc, bs = _np(codes, np.uint8), _np(block_scales, np.uint8)
    ii = _np(idx, np.int32)
    out = np.empty((64, 512), np.float64)
    lse = np.empty(64, np.float64)
    st = layout.struct()
    _check((L or lib()).oracle_sparse_mla_nvfp4(_ptr(qq), _ptr(cc), _ptr(bs), float(g), ctypes.byref(st), seq,
                                                _ptr(ii), topk_len, sm_scale, _ptr(out), _ptr(lse), None))
    return out, lse
