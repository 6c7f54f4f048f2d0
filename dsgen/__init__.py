"""Seeded synthetic inputs for decode-step top-k sparse attention.

This module is shared by the tests, the benchmark and the oracle's callers. It
only draws numbers and lays them out in the cache formats the library consumes;
it holds none of the method's arithmetic (no scoring, no selection, no softmax,
no merge, no FP8 decoding).

Random numbers come from a counter-based generator: element ``i`` of stream
``key`` is ``fmix32(lo32(i) ^ fmix32(hi32(i) ^ key))`` where ``fmix32`` is the
32-bit MurmurHash3 finaliser. It is written with int64 torch ops whose
intermediate products stay below 2**63, so it gives the same integers on the
CPU and on a GPU and any chunk of a tensor can be drawn independently.

Workload shapes follow the pages:
* "Support double sparsity" (sglang PR #1459), section "Speedup Evaluation":
  longchat-7b batch 3 x 20000 tokens, 16 heavy channels, 1024 heavy tokens;
  Llama-3.1-8B batch 3 x 60000 tokens, 32 K-type channels, 3000 heavy tokens.
* "QSA HiSparse - SGLang plugin", section "Supported versions": FP8 E4M3 KV
  cache, page size 64, up to 262,144 tokens per request, up to 8 requests.
* sglang PR #43527 "QSA cache sharding", section "Performance": 1M-token
  requests, shard size 4; sglang PR #43533, "Speed Tests and Profiling":
  top_k = 2048.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

_M32 = 0xFFFFFFFF
PAGE_SIZE = 64


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 ``x`` in [0, 2**32) without int64 overflow."""
    lo = c & 0xFFFF
    hi = (c >> 16) & 0xFFFF
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def _fmix32_int(h: int) -> int:
    h &= _M32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & _M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & _M32
    h ^= h >> 16
    return h


def stream_key(seed: int, tensor_id: int) -> int:
    """Key of one named random stream (one per tensor and seed)."""
    return _fmix32_int(_fmix32_int(seed * 0x9E3779B9 + 0x7F4A7C15) ^ (tensor_id * 0x632BE5AB + 0x1B873593))


def hash_u32(key: int, start: int, n: int, device) -> torch.Tensor:
    """``n`` uint32 draws (as int64) of stream ``key`` at counters start..start+n-1."""
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    lo = i & _M32
    hi = (i >> 32) & _M32
    return _fmix32(lo ^ _fmix32(hi ^ key))


_CHUNK = 1 << 24


def _fill(out_flat: torch.Tensor, key: int, draw):
    n = out_flat.numel()
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        out_flat[s:s + m] = draw(key, s, m, out_flat.device)


def uniform_int(shape, lo: int, hi: int, seed: int, tensor_id: int, device="cpu",
                dtype=torch.bfloat16) -> torch.Tensor:
    """Integers uniform in [lo, hi], stored as ``dtype``."""
    out = torch.empty(shape, dtype=dtype, device=device)
    span = hi - lo + 1

    def draw(key, s, m, dev):
        return (hash_u32(key, s, m, dev) % span + lo).to(dtype)

    _fill(out.view(-1), stream_key(seed, tensor_id), draw)
    return out


def normal(shape, seed: int, tensor_id: int, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, 1) draws by the Box-Muller transform, rounded to ``dtype`` (RNE)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    k1 = stream_key(seed, tensor_id)
    k2 = stream_key(seed, tensor_id + 0x10000)

    def draw(_key, s, m, dev):
        u1 = (hash_u32(k1, s, m, dev).to(torch.float32) + 0.5) * (1.0 / 4294967296.0)
        u2 = hash_u32(k2, s, m, dev).to(torch.float32) * (1.0 / 4294967296.0)
        z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        return z.to(dtype)

    _fill(out.view(-1), k1, draw)
    return out


def uniform_float(shape, lo: float, hi: float, seed: int, tensor_id: int, device="cpu") -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.float32, device=device)

    def draw(key, s, m, dev):
        u = hash_u32(key, s, m, dev).to(torch.float64) * (1.0 / 4294967296.0)
        return (lo + (hi - lo) * u).to(torch.float32)

    _fill(out.view(-1), stream_key(seed, tensor_id), draw)
    return out


def permutation(n: int, seed: int, tensor_id: int) -> torch.Tensor:
    """A seeded random permutation of 0..n-1 (Fisher-Yates via torch.randperm on CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(stream_key(seed, tensor_id))
    return torch.randperm(n, generator=g, dtype=torch.int64).to(torch.int32)


@dataclasses.dataclass
class Workload:
    """One decode-step configuration.

    ``label_heads`` is the number of proxy-key heads in the cache: equal to
    ``num_kv_heads`` for a Double-Sparsity label cache (one label row per KV
    head), 1 for QSA-style index keys (one key per token shared by all heads).
    """
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_lens: List[int]
    proxy_dim: int
    label_heads: int
    top_k: int
    kv_dtype: str                 # "bf16" or "fp8_e4m3"
    shuffle_pages: bool
    seed: int
    splits: List[int] = dataclasses.field(default_factory=lambda: [1])
    proxy_from_query: bool = True  # DS: qp = q at the heavy channels; QSA: own index query
    page_size: int = PAGE_SIZE

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens) if self.seq_lens else 0

    @property
    def max_pages_per_req(self) -> int:
        return max(1, -(-self.max_seq_len // self.page_size))

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _w(name, B, Hq, Hkv, T, C, HL, K, kvd, shuffle, seed, splits=(1,), from_q=True):
    return Workload(name=name, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                    seq_lens=[T] * B, proxy_dim=C, label_heads=HL, top_k=K, kv_dtype=kvd,
                    shuffle_pages=shuffle, seed=seed, splits=list(splits), proxy_from_query=from_q)


# The five decode workloads (seed = 1000 + index).
WORKLOADS = [
    _w("tiny_ds_b1_h4_t4096_c16_k256", 1, 4, 1, 4096, 16, 1, 256, "bf16", False, 1000),
    _w("llama8b_ds_b3_h32kv8_t60000_c32_k3000", 3, 32, 8, 60000, 32, 8, 3000, "bf16", False, 1001),
    _w("longchat7b_ds_b3_h32kv32_t20000_c16_k1024", 3, 32, 32, 20000, 16, 32, 1024, "bf16", False, 1002),
    _w("qsa_b8_h32kv4_t262144_idx64_k2048_fp8", 8, 32, 4, 262144, 64, 1, 2048, "fp8_e4m3", True, 1003,
       from_q=False),
    _w("qsa_1m_b1_h32kv4_t1048576_idx64_k2048_fp8", 1, 32, 4, 1048576, 64, 1, 2048, "fp8_e4m3", True, 1004,
       splits=(1, 4, 16), from_q=False),
]

# Stream ids, one per generated tensor.
_ID_Q, _ID_CH, _ID_QP, _ID_LABEL, _ID_K, _ID_V, _ID_KS, _ID_VS, _ID_PERM = range(1, 10)


@dataclasses.dataclass
class Inputs:
    """Tensors of one decode step, all on one device, in the library's layouts.

    q          bf16  [B, Hq, D]            decode query (integer-valued in [-4, 4])
    qp         bf16  [B, Hq, C]            proxy query (heavy channels of q, or an index query)
    label      bf16  [num_slots, HL, C]    label cache / index keys, integer-valued in [-8, 8]
    k_cache    bf16 or uint8 (e4m3 bytes) [num_slots, Hkv, D]
    v_cache    same as k_cache
    k_scale    fp32  [num_pages] per-page dequantisation scale (FP8 only, else None)
    v_scale    fp32  [num_pages]
    page_table int32 [B, max_pages_per_req]  physical page of each logical page
    seq_lens   int32 [B]
    """
    w: Workload
    q: torch.Tensor
    qp: torch.Tensor
    label: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor]
    v_scale: Optional[torch.Tensor]
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    num_pages: int

    def to(self, device) -> "Inputs":
        f = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, q=f(self.q), qp=f(self.qp), label=f(self.label),
                                   k_cache=f(self.k_cache), v_cache=f(self.v_cache),
                                   k_scale=f(self.k_scale), v_scale=f(self.v_scale),
                                   page_table=f(self.page_table), seq_lens=f(self.seq_lens))


def page_table_for(w: Workload, seed: int):
    """Pages of request b: its own ceil(T_b/64) pages, contiguous or shuffled over the pool.

    Unused entries hold -1 (consumers must stop at the request's length).
    """
    P = w.page_size
    counts = [-(-t // P) for t in w.seq_lens]
    total = max(1, sum(counts))
    order = permutation(total, seed, _ID_PERM) if w.shuffle_pages else torch.arange(total, dtype=torch.int32)
    pt = torch.full((w.batch, w.max_pages_per_req), -1, dtype=torch.int32)
    o = 0
    for b, c in enumerate(counts):
        pt[b, :c] = order[o:o + c]
        o += c
    return pt, total


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> Inputs:
    """Draw every input of one decode step of workload ``w`` on ``device``."""
    seed = w.seed if seed is None else seed
    B, Hq, Hkv, D, C, HL = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.proxy_dim, w.label_heads
    pt, num_pages = page_table_for(w, seed)
    slots = num_pages * w.page_size
    q = uniform_int((B, Hq, D), -4, 4, seed, _ID_Q, device)
    if w.proxy_from_query:
        # Heavy channels: C distinct channels of D per KV head (seeded), gathered from q.
        ch = torch.stack([permutation(D, seed, _ID_CH * 1000 + g)[:C] for g in range(Hkv)]).long()
        ch_per_q = ch.repeat_interleave(w.group, dim=0).to(device)          # [Hq, C]
        qp = torch.gather(q, 2, ch_per_q.unsqueeze(0).expand(B, Hq, C)).contiguous()
    else:
        qp = uniform_int((B, Hq, C), -4, 4, seed, _ID_QP, device)
    label = uniform_int((slots, HL, C), -8, 8, seed, _ID_LABEL, device)
    if w.kv_dtype == "bf16":
        k_cache = normal((slots, Hkv, D), seed, _ID_K, device)
        v_cache = normal((slots, Hkv, D), seed, _ID_V, device)
        k_scale = v_scale = None
    elif w.kv_dtype == "fp8_e4m3":
        k_scale = uniform_float((num_pages,), 0.25, 4.0, seed, _ID_KS, device)
        v_scale = uniform_float((num_pages,), 0.25, 4.0, seed, _ID_VS, device)
        k_cache = _fp8_pages(slots, Hkv, D, k_scale, seed, _ID_K, device, w.page_size)
        v_cache = _fp8_pages(slots, Hkv, D, v_scale, seed, _ID_V, device, w.page_size)
    else:
        raise ValueError(w.kv_dtype)
    seq = torch.tensor(w.seq_lens, dtype=torch.int32)
    return Inputs(w, q, qp, label, k_cache, v_cache, k_scale, v_scale, pt.to(device), seq.to(device), num_pages)


def _fp8_pages(slots, H, D, scale, seed, tid, device, P):
    """x ~ N(0,1) stored as e4m3 bytes of x / scale[page] (RNE, clamped to +-448)."""
    out = torch.empty((slots, H, D), dtype=torch.uint8, device=device)
    rows_per_chunk = max(P, (_CHUNK // (H * D)) // P * P)
    for s in range(0, slots, rows_per_chunk):
        e = min(slots, s + rows_per_chunk)
        x = _normal_at(seed, tid, s * H * D, (e - s, H, D), device)
        sc = scale[torch.arange(s, e, device=device) // P].view(-1, 1, 1)
        y = torch.clamp(x / sc, -448.0, 448.0)
        out[s:e] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def _normal_at(seed, tensor_id, start, shape, device):
    """Same stream as ``normal(..., torch.float32)`` but starting at counter ``start``."""
    n = math.prod(shape)
    k1 = stream_key(seed, tensor_id)
    k2 = stream_key(seed, tensor_id + 0x10000)
    u1 = (hash_u32(k1, start, n, device).to(torch.float32) + 0.5) * (1.0 / 4294967296.0)
    u2 = hash_u32(k2, start, n, device).to(torch.float32) * (1.0 / 4294967296.0)
    return (torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)).view(shape)


def shape_kwargs(inp: Inputs) -> dict:
    """Sizes of ``inp`` as keyword arguments of the library's ds_shape."""
    w = inp.w
    return dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                page_size=w.page_size, max_pages_per_req=int(inp.page_table.shape[1]), num_pages=int(inp.num_pages),
                max_seq_len=w.max_seq_len)
