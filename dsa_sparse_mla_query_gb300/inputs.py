"""Seeded synthetic inputs for the DSA decode path.

This module is the only code that the CUDA path and the CPU oracle share.  It
holds none of the method's arithmetic (no SSMax, rotation, scoring, selection
or attention): only a counter-based random source, the value distributions of
the workloads, and the storage encodings of the caches (bf16 rounding, e4m3
with an fp32 scale per group), so that both sides read the same bytes.

Random source.  SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator: element ``i`` of stream ``key`` is ``mix(key + (i + 1) * GAMMA)``,
where ``mix`` is the generator's 64-bit finaliser.  A stream key is derived
from ``(seed, tensor id)``, so every tensor element is a pure function of
``(seed, tensor id, element index)``; the order and the device of generation do
not matter, and any subset (one sequence's rows) can be generated alone.
Uniforms take the top 53 bits; normals use the Box-Muller transform in fp64.

Workloads (Mistral Large 4 decode layer, "Day 0 support for Mistral Large 4",
Implementation details / Model architecture table: 32 index heads of dim 128,
top-k 2048, MLA with KV LoRA rank 512 and RoPE dim 64, 64 heads):

* ``tiny``     1 sequence x 4096 keys, 4 queries at 4092..4095, RoPE layer.
* ``paged``    64 sequences x 32768 keys, 1 query each, 64-token pages with a
               random permutation over all pages, LeRoPE divisor exp(alpha)
               with alpha ~ U(-0.5, 0.5) per pair.
* ``specv``    128 sequences with contexts ~ U{8192..131072}, 4 causal
               queries each, NoPE layer, plus a shared-indexer layer with its
               own query and latent cache.
* ``long_fp8`` 32 sequences x 524288 keys, 1 query each, e4m3 indexer keys
               with one fp32 scale per row (132 B/token) and the fp8_ds_mla
               latent row (656 B/token).
* ``prefill``  1 sequence, 4096 queries at 126976..131071 over 131072 keys.
* ``block_fp8`` as ``long_fp8``, with block-sparse selection (16 blocks of
               128 keys, "vLLM adds NVFP4 serving for MiniMax M3.1 Flash",
               MiniMax Sparse Attention).
* ``long_nvfp4`` as ``long_fp8``, with NVFP4 caches ("vLLM adds NVFP4
               serving for MiniMax M3.1 Flash": 4.5 bits per value): index
               keys of 72 B/token and latent rows of 324 B/token.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

# ---------------------------------------------------------------------------
# fixed shapes of the path
INDEX_HEADS = 32
INDEX_DIM = 128
ROPE_PAIRS = 32
MLA_HEADS = 64
MLA_DIM = 576
MLA_VDIM = 512
MLA_ROPE_DIM = 64
DS_MLA_ROW_BYTES = 656      # 512 e4m3 + 4 fp32 scales + 64 bf16
FP8_GROUP = 128
E4M3_MAX = 448.0
NVFP4_BLOCK = 16
# Tensor scale of the synthetic NVFP4 caches: their values are N(0, 1), so a
# block maximum above 8 (probability ~1e-15 per value) is the only case whose
# E4M3 block scale amax / (6 g) would pass 448 (it saturates there).
NVFP4_GLOBAL = 8.0 / (6.0 * E4M3_MAX)

# tensor ids of the counter streams
T_Q_IDX, T_W, T_SSMAX_S, T_SSMAX_B, T_ALPHA = 1, 2, 3, 4, 5
T_K_IDX, T_LATENT, T_Q_MLA, T_CTX, T_PAGES = 6, 7, 8, 9, 10
T_LATENT2, T_Q_MLA2 = 11, 12
# new tokens for the cache-write side
T_NEW_X, T_NEW_GAMMA, T_NEW_BETA, T_NEW_CKV, T_NEW_KPE, T_NEW_Q, T_NEW_SS, T_NEW_SB, T_NEW_SLOT = range(13, 22)

# ---------------------------------------------------------------------------
# SplitMix64, counter based
_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_MUL1 = 0xBF58476D1CE4E5B9
_MUL2 = 0x94D049BB133111EB


def _signed(c: int) -> int:
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (reference for the tensor form)."""
    z &= _M64
    z = ((z ^ (z >> 30)) * _MUL1) & _M64
    z = ((z ^ (z >> 27)) * _MUL2) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    return mix64_int(mix64_int(seed * _GAMMA + 0x632BE59BD9B4E019) ^ (tensor_id * _GAMMA))


def bits_int(key: int, counter: int) -> int:
    """Element ``counter`` of stream ``key`` (Python int form)."""
    return mix64_int(key + (counter + 1) * _GAMMA)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _signed(_MUL1)
    z = (z ^ _lsr(z, 27)) * _signed(_MUL2)
    return z ^ _lsr(z, 31)


def bits(key: int, counters: torch.Tensor) -> torch.Tensor:
    """int64 tensor of stream elements (two's complement view of the uint64)."""
    return _mix64(counters * _signed(_GAMMA) + _signed(key + _GAMMA))


def uniform(key: int, counters: torch.Tensor) -> torch.Tensor:
    """fp64 uniforms in [0, 1) from the top 53 bits."""
    return _lsr(bits(key, counters), 11).to(torch.float64) * (2.0 ** -53)


def normal(key: int, counters: torch.Tensor) -> torch.Tensor:
    """fp64 N(0,1) by Box-Muller on the uniforms at 2c and 2c+1."""
    u1 = uniform(key, 2 * counters)
    u2 = uniform(key, 2 * counters + 1)
    return torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos((2.0 * math.pi) * u2)


def _counters(start: int, n: int, device) -> torch.Tensor:
    return torch.arange(start, start + n, dtype=torch.int64, device=device)


# ---------------------------------------------------------------------------
# storage encodings
def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """fp64 -> fp32 (round to nearest) -> bf16 (round to nearest even)."""
    return x.to(torch.float32).to(torch.bfloat16)


def quantize_e4m3_groups(v: torch.Tensor, group: int):
    """Quantise the last dim of fp32 ``v`` in groups: scale = amax / 448,
    code = e4m3(round-nearest-even(v / scale)), saturating; a group of zeros
    gets scale 0 and zero codes.  Returns (uint8 codes, fp32 scales)."""
    shp = v.shape
    g = v.reshape(*shp[:-1], shp[-1] // group, group)
    amax = g.abs().amax(dim=-1, keepdim=True)
    scale = amax / E4M3_MAX
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    q = torch.where(scale > 0, g / safe, torch.zeros_like(g)).clamp(-E4M3_MAX, E4M3_MAX)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(shp)
    return codes, scale.squeeze(-1)


def quantize_nvfp4(v: torch.Tensor, g: float):
    """NVFP4 encoding of the last dim of ``v`` (a multiple of 16): per block of
    16 values the E4M3 scale s = e4m3(amax / (6 g)) (nearest, at most 448),
    then each value's E2M1 code of v / (g s): the nearest of 0, 0.5, 1, 1.5,
    2, 3, 4, 6, a tie to the code with mantissa bit 0, beyond 6 the largest;
    a block with s = 0 gets zero codes.  Value 2i in the low nibble of byte i.
    Returns (uint8 codes [..., n/2], uint8 scale codes [..., n/16])."""
    shp = v.shape
    n = shp[-1]
    x = v.to(torch.float64).reshape(*shp[:-1], n // NVFP4_BLOCK, NVFP4_BLOCK)
    amax = x.abs().amax(dim=-1, keepdim=True)
    sc = (amax / (6.0 * g)).clamp(max=E4M3_MAX).to(torch.float8_e4m3fn)
    s = sc.to(torch.float64)
    live = s > 0
    y = torch.where(live, x / (g * torch.where(live, s, torch.ones_like(s))), torch.zeros_like(x))
    a = y.abs()
    code = ((a > 0.25).to(torch.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5) + (a >= 3.5) + (a > 5))
    code = code + torch.where(torch.signbit(y) & live, 8, 0).to(torch.uint8)
    code = code.reshape(*shp[:-1], n // 2, 2)
    codes = (code[..., 0] | (code[..., 1] << 4)).to(torch.uint8)
    return codes, sc.view(torch.uint8).reshape(*shp[:-1], n // NVFP4_BLOCK)


# ---------------------------------------------------------------------------
# workloads
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    queries_per_seq: int
    ctx: Optional[int] = None              # fixed context per sequence
    ctx_range: Optional[tuple] = None      # (lo, hi) inclusive, uniform integer
    ctx_list: Optional[tuple] = None       # explicit context per sequence
    rope: bool = True
    alpha_range: Optional[tuple] = None    # LeRoPE alpha ~ U(lo, hi) per pair
    page_size: int = 0                     # 0 = contiguous rows per sequence
    index_fp8: bool = False
    latent_fp8: bool = False
    index_nvfp4: bool = False
    latent_nvfp4: bool = False
    shared_layer: bool = False
    topk: int = 2048
    select_block: int = 0                  # 0: exact top-k; > 0: block-sparse selection, blocks of this size
    seed: int = 0

    @property
    def num_queries(self) -> int:
        return self.num_seqs * self.queries_per_seq

    def describe(self) -> str:
        c = (f"{self.ctx}" if self.ctx else f"U{{{self.ctx_range[0]}..{self.ctx_range[1]}}}" if self.ctx_range
             else f"{list(self.ctx_list)}")
        return (f"{self.name}: {self.num_seqs} seq x ctx {c}, {self.queries_per_seq} q/seq, "
                f"{'RoPE' if self.rope else 'NoPE'}, index "
                f"{'e4m3+rowscale' if self.index_fp8 else 'nvfp4' if self.index_nvfp4 else 'bf16'}, "
                f"latent {'fp8_ds_mla' if self.latent_fp8 else 'nvfp4' if self.latent_nvfp4 else 'bf16'}"
                f"{', pages of %d' % self.page_size if self.page_size else ''}"
                f"{', + shared-indexer layer' if self.shared_layer else ''}, "
                + (f"{self.topk // self.select_block} blocks of {self.select_block}" if self.select_block
                   else f"top-{self.topk}"))


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 4, ctx=4096),
    "paged": Workload("paged", 64, 1, ctx=32768, alpha_range=(-0.5, 0.5), page_size=64),
    "specv": Workload("specv", 128, 4, ctx_range=(8192, 131072), rope=False, shared_layer=True),
    "long_fp8": Workload("long_fp8", 32, 1, ctx=524288, index_fp8=True, latent_fp8=True),
    "prefill": Workload("prefill", 1, 4096, ctx=131072),
    # block-sparse selection as the MiniMax M3.1 page describes it: 128-token
    # blocks, 16 selected (2,048 keys) at long context; caches as long_fp8
    "block_fp8": Workload("block_fp8", 32, 1, ctx=524288, index_fp8=True, latent_fp8=True, select_block=128),
    # NVFP4 caches as the MiniMax M3.1 page describes them (72 B index keys,
    # 324 B latent rows), at the long_fp8 shape
    "long_nvfp4": Workload("long_nvfp4", 32, 1, ctx=524288, index_nvfp4=True, latent_nvfp4=True),
}


def context_lengths(wl: Workload) -> List[int]:
    if wl.ctx_list is not None:
        assert len(wl.ctx_list) == wl.num_seqs
        return [int(c) for c in wl.ctx_list]
    if wl.ctx is not None:
        return [wl.ctx] * wl.num_seqs
    lo, hi = wl.ctx_range
    u = uniform(stream_key(wl.seed, T_CTX), _counters(0, wl.num_seqs, "cpu"))
    return [lo + int(math.floor(x * (hi - lo + 1))) for x in u.tolist()]


@dataclasses.dataclass
class Layout:
    """Where each sequence's tokens live (host copies)."""
    ctx_len: List[int]
    q_start: List[int]
    q_pos: List[int]
    q_seq: List[int]
    page_size: int
    max_pages: int
    page_table: Optional[torch.Tensor]   # int32 [B, max_pages]
    seq_base: Optional[torch.Tensor]     # int64 [B]
    num_rows: int

    def phys_rows(self, b: int, n: Optional[int] = None) -> torch.Tensor:
        """Physical cache rows of sequence b's first n tokens, in logical order."""
        n = self.ctx_len[b] if n is None else n
        j = torch.arange(n, dtype=torch.int64)
        if self.page_table is not None:
            return self.page_table[b].to(torch.int64)[j // self.page_size] * self.page_size + j % self.page_size
        return self.seq_base[b] + j


def make_layout(wl: Workload) -> Layout:
    ctx = context_lengths(wl)
    B, T = wl.num_seqs, wl.queries_per_seq
    q_start = [b * T for b in range(B + 1)]
    q_pos = [ctx[b] - T + i for b in range(B) for i in range(T)]
    q_seq = [b for b in range(B) for _ in range(T)]
    if wl.page_size:
        ps = wl.page_size
        pages = [(c + ps - 1) // ps for c in ctx]
        total = sum(pages)
        # a uniformly random permutation of all physical pages: argsort of
        # 64-bit stream values (ties have probability ~2^-64; argsort is stable)
        perm = torch.argsort(bits(stream_key(wl.seed, T_PAGES), _counters(0, total, "cpu")), stable=True)
        max_pages = max(pages)
        table = torch.zeros(B, max_pages, dtype=torch.int32)
        o = 0
        for b in range(B):
            table[b, :pages[b]] = perm[o:o + pages[b]].to(torch.int32)
            o += pages[b]
        return Layout(ctx, q_start, q_pos, q_seq, ps, max_pages, table, None, total * ps)
    base = [0]
    for c in ctx[:-1]:
        base.append(base[-1] + c)
    return Layout(ctx, q_start, q_pos, q_seq, 0, 0, None,
                  torch.tensor(base, dtype=torch.int64), sum(ctx))


# ---------------------------------------------------------------------------
# tensor generators (element counter = flat index in the physical tensor)
_CHUNK_ROWS_ELEMS = 1 << 24


def _fill_rows(out_fn, rows: torch.Tensor, width: int, key: int, device, make):
    """Generate rows ``rows`` (physical row ids) of a [*, width] stream in
    chunks; ``make(normals_fp64[nrows, width]) -> encoded chunk`` and
    ``out_fn(slice, chunk)`` stores it."""
    step = max(1, _CHUNK_ROWS_ELEMS // width)
    col = torch.arange(width, dtype=torch.int64, device=device)
    for s in range(0, rows.numel(), step):
        r = rows[s:s + step].to(device)
        cnt = r[:, None] * width + col[None, :]
        out_fn(slice(s, s + r.numel()), make(normal(key, cnt)))


def gen_bf16_rows(key: int, rows: torch.Tensor, width: int, device, zero_from: Optional[int] = None):
    out = torch.empty(rows.numel(), width, dtype=torch.bfloat16, device=device)

    def make(x):
        y = to_bf16(x)
        if zero_from is not None:
            y[:, zero_from:] = 0
        return y

    def store(sl, chunk):
        out[sl] = chunk
    _fill_rows(store, rows, width, key, device, make)
    return out


def gen_e4m3_rowscale_rows(key: int, rows: torch.Tensor, device):
    """Indexer keys, 132 B/token: 128 e4m3 codes + one fp32 scale per row."""
    codes = torch.empty(rows.numel(), INDEX_DIM, dtype=torch.uint8, device=device)
    scale = torch.empty(rows.numel(), dtype=torch.float32, device=device)

    def make(x):
        return quantize_e4m3_groups(x.to(torch.float32), INDEX_DIM)

    def store(sl, chunk):
        codes[sl] = chunk[0]
        scale[sl] = chunk[1][:, 0]
    _fill_rows(store, rows, INDEX_DIM, key, device, make)
    return codes, scale


def gen_ds_mla_rows(key: int, rows: torch.Tensor, device):
    """fp8_ds_mla latent rows, 656 B/token: [0,512) e4m3 latent codes,
    [512,528) four fp32 scales (one per 128 latent dims), [528,656) the 64
    RoPE dims as bf16.  Values are the same N(0,1) stream as a bf16 latent."""
    out = torch.empty(rows.numel(), DS_MLA_ROW_BYTES, dtype=torch.uint8, device=device)

    def make(x):
        codes, scale = quantize_e4m3_groups(x[:, :MLA_VDIM].to(torch.float32), FP8_GROUP)
        rope = to_bf16(x[:, MLA_VDIM:]).contiguous().view(torch.uint8)
        return torch.cat([codes, scale.contiguous().view(torch.uint8), rope], dim=1)

    def store(sl, chunk):
        out[sl] = chunk
    _fill_rows(store, rows, MLA_DIM, key, device, make)
    return out


def gen_nvfp4_rows(key: int, rows: torch.Tensor, width: int, device, zero_from: Optional[int] = None):
    """NVFP4 rows of the same N(0,1) stream as gen_bf16_rows (rounded to bf16
    first, as a bf16 cache quantised to NVFP4): codes [n, width/2] and E4M3
    block scales [n, width/16], tensor scale NVFP4_GLOBAL."""
    codes = torch.empty(rows.numel(), width // 2, dtype=torch.uint8, device=device)
    scales = torch.empty(rows.numel(), width // NVFP4_BLOCK, dtype=torch.uint8, device=device)

    def make(x):
        y = to_bf16(x)
        if zero_from is not None:
            y[:, zero_from:] = 0
        return quantize_nvfp4(y, NVFP4_GLOBAL)

    def store(sl, chunk):
        codes[sl] = chunk[0]
        scales[sl] = chunk[1]
    _fill_rows(store, rows, width, key, device, make)
    return codes, scales


def _params(wl: Workload):
    s = (0.05 + 0.10 * uniform(stream_key(wl.seed, T_SSMAX_S), _counters(0, INDEX_HEADS, "cpu"))).to(torch.float32)
    b = (0.9 + 0.2 * uniform(stream_key(wl.seed, T_SSMAX_B), _counters(0, INDEX_HEADS, "cpu"))).to(torch.float32)
    inv_freq = None
    if wl.rope:
        i = torch.arange(ROPE_PAIRS, dtype=torch.float64)
        base = 10000.0 ** (-2.0 * i / (2 * ROPE_PAIRS))
        alpha = torch.zeros(ROPE_PAIRS, dtype=torch.float64)
        if wl.alpha_range is not None:
            lo, hi = wl.alpha_range
            alpha = lo + (hi - lo) * uniform(stream_key(wl.seed, T_ALPHA), _counters(0, ROPE_PAIRS, "cpu"))
        # LeRoPE: each pair's frequency divided by its learned factor exp(alpha)
        inv_freq = (base / torch.exp(alpha)).to(torch.float32)
    return s, b, inv_freq


def _query_rows(key, q0, nq, width, device, make):
    rows = torch.arange(q0, q0 + nq, dtype=torch.int64)
    out = []
    _fill_rows(lambda sl, c: out.append(c), rows, width, key, device, make)
    return torch.cat(out, 0)


def make_queries(wl: Workload, device, q0: int = 0, nq: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Query-side tensors for query rows q0..q0+nq-1."""
    nq = wl.num_queries - q0 if nq is None else nq
    out = {}
    out["q_idx"] = _query_rows(stream_key(wl.seed, T_Q_IDX), q0, nq, INDEX_HEADS * INDEX_DIM, device,
                               to_bf16).view(nq, INDEX_HEADS, INDEX_DIM)
    out["w"] = _query_rows(stream_key(wl.seed, T_W), q0, nq, INDEX_HEADS, device,
                           lambda x: x.to(torch.float32))
    zero = MLA_VDIM if not wl.rope else None

    def mla(x):
        y = to_bf16(x)
        if zero is not None:
            y[:, zero:] = 0
        return y
    out["q_mla"] = _query_rows(stream_key(wl.seed, T_Q_MLA), q0, nq, MLA_HEADS * MLA_DIM, device,
                               mla).view(nq, MLA_HEADS, MLA_DIM)
    if wl.shared_layer:
        out["q_mla2"] = _query_rows(stream_key(wl.seed, T_Q_MLA2), q0, nq, MLA_HEADS * MLA_DIM, device,
                                    mla).view(nq, MLA_HEADS, MLA_DIM)
    return out


def make_cache_rows(wl: Workload, rows: torch.Tensor, device, which: str = "all") -> Dict[str, torch.Tensor]:
    """Cache rows ``rows`` (physical ids) of the index keys and latent caches."""
    out = {}
    zero = None if wl.rope else MLA_VDIM
    if which in ("all", "index"):
        if wl.index_fp8:
            out["k_idx"], out["k_scale"] = gen_e4m3_rowscale_rows(stream_key(wl.seed, T_K_IDX), rows, device)
        elif wl.index_nvfp4:
            out["k_idx"], out["k_bscale"] = gen_nvfp4_rows(stream_key(wl.seed, T_K_IDX), rows, INDEX_DIM, device)
            out["k_global"] = NVFP4_GLOBAL
        else:
            out["k_idx"] = gen_bf16_rows(stream_key(wl.seed, T_K_IDX), rows, INDEX_DIM, device)
    if which in ("all", "latent"):
        if wl.latent_fp8:
            out["latent"] = gen_ds_mla_rows(stream_key(wl.seed, T_LATENT), rows, device)
        elif wl.latent_nvfp4:
            out["latent"], out["lat_bscale"] = gen_nvfp4_rows(stream_key(wl.seed, T_LATENT), rows, MLA_DIM, device,
                                                              zero)
            out["lat_global"] = NVFP4_GLOBAL
        else:
            out["latent"] = gen_bf16_rows(stream_key(wl.seed, T_LATENT), rows, MLA_DIM, device, zero)
        if wl.shared_layer:
            if wl.latent_nvfp4:
                raise ValueError("the shared-indexer layer's second latent cache has no NVFP4 form here")
            if wl.latent_fp8:
                out["latent2"] = gen_ds_mla_rows(stream_key(wl.seed, T_LATENT2), rows, device)
            else:
                out["latent2"] = gen_bf16_rows(stream_key(wl.seed, T_LATENT2), rows, MLA_DIM, device, zero)
    return out


def make_inputs(wl: Workload, device) -> Dict[str, object]:
    """Every tensor of the workload on ``device`` (full size)."""
    lay = make_layout(wl)
    s, b, inv_freq = _params(wl)
    d = dict(layout=lay, ssmax_s=s.to(device), ssmax_b=b.to(device),
             inv_freq=None if inv_freq is None else inv_freq.to(device),
             sm_scale=1.0 / math.sqrt(192.0), topk=wl.topk)
    d.update(make_queries(wl, device))
    d.update(make_cache_rows(wl, torch.arange(lay.num_rows, dtype=torch.int64), device))
    d["ctx_len"] = torch.tensor(lay.ctx_len, dtype=torch.int32, device=device)
    d["q_start"] = torch.tensor(lay.q_start, dtype=torch.int32, device=device)
    d["q_pos"] = torch.tensor(lay.q_pos, dtype=torch.int32, device=device)
    d["page_table"] = None if lay.page_table is None else lay.page_table.to(device)
    d["seq_base"] = None if lay.seq_base is None else lay.seq_base.to(device)
    return d


def params(wl: Workload):
    """(ssmax_s, ssmax_b, inv_freq or None) as fp32 CPU tensors."""
    return _params(wl)


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (small test cases)."""
    return dataclasses.replace(wl, **kw)


def make_insert_inputs(n: int, nq: int, num_rows: int, device, seed: int = 0, rope: bool = True,
                       page_size: int = 0) -> Dict[str, object]:
    """New tokens for the cache-write side: indexer-key projections x bf16
    [n,128] ~ N(0.3, 2); LayerNorm gamma ~ U(0.5, 1.5), beta ~ U(-0.2, 0.2)
    [128]; latent c_kv bf16 [n,512] and k_pe [n,64] ~ N(0,1); attention queries
    q bf16 [nq,64,576] ~ N(0,1) with SSMax s ~ U(0.05, 0.15), b ~ U(0.9, 1.1)
    per head; positions 0..n-1 (queries at the last nq); distinct physical rows:
    a random permutation of the cache rows, or with page_size consecutive
    tokens filling pages taken in a random order; the workloads' RoPE table."""
    c = lambda k: _counters(0, k, device)  # noqa: E731
    out: Dict[str, object] = {}
    out["x"] = to_bf16(normal(stream_key(seed, T_NEW_X), c(n * INDEX_DIM)) * 2.0 + 0.3).view(n, INDEX_DIM)
    out["gamma"] = (0.5 + uniform(stream_key(seed, T_NEW_GAMMA), c(INDEX_DIM))).to(torch.float32)
    out["beta"] = (uniform(stream_key(seed, T_NEW_BETA), c(INDEX_DIM)) * 0.4 - 0.2).to(torch.float32)
    out["c_kv"] = to_bf16(normal(stream_key(seed, T_NEW_CKV), c(n * MLA_VDIM))).view(n, MLA_VDIM)
    out["k_pe"] = to_bf16(normal(stream_key(seed, T_NEW_KPE), c(n * MLA_ROPE_DIM))).view(n, MLA_ROPE_DIM)
    out["q"] = to_bf16(normal(stream_key(seed, T_NEW_Q), c(nq * MLA_HEADS * MLA_DIM))).view(nq, MLA_HEADS, MLA_DIM)
    out["ssmax_s"] = (0.05 + 0.1 * uniform(stream_key(seed, T_NEW_SS), c(MLA_HEADS))).to(torch.float32)
    out["ssmax_b"] = (0.9 + 0.2 * uniform(stream_key(seed, T_NEW_SB), c(MLA_HEADS))).to(torch.float32)
    out["pos"] = torch.arange(n, dtype=torch.int32, device=device)
    out["q_pos"] = torch.arange(n - nq, n, dtype=torch.int32, device=device)
    if page_size:
        pages = torch.argsort(bits(stream_key(seed, T_NEW_SLOT), c(num_rows // page_size)))
        t = torch.arange(n, dtype=torch.int64, device=device)
        out["slot"] = pages[t // page_size].to(torch.int64) * page_size + t % page_size
    else:
        perm = torch.argsort(bits(stream_key(seed, T_NEW_SLOT), c(num_rows)))
        out["slot"] = perm[:n].to(torch.int64)
    out["inv_freq"] = (1.0 / 10000.0 ** (torch.arange(ROPE_PAIRS, dtype=torch.float64, device=device) / ROPE_PAIRS)
                       ).to(torch.float32) if rope else None
    return out
