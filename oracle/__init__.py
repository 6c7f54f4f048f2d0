"""Loader for the C++ oracle. TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The library never does, and the oracle shares no
code with it. ``build()`` compiles ``oracle.cpp`` with the host C++ compiler;
the wrappers below only marshal torch CPU tensors to the C functions.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional

import torch

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "oracle.cpp")
_LIB_PATH = os.path.join(_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (no CUDA involved).

    With ``DS_ORACLE_LIB`` set, that prebuilt library is used instead: the
    planted-mistake tests load a deliberately altered copy of the oracle this
    way to show that the pins reject it.
    """
    override = os.environ.get("DS_ORACLE_LIB")
    if override:
        return override
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cxx = os.environ.get("CXX", "g++")
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([cxx, "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        _lib.oracle_bf16_value.restype = ctypes.c_double
        _lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        _lib.oracle_e4m3_value.restype = ctypes.c_double
        _lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        _lib.oracle_index_score.restype = I
        _lib.oracle_index_score.argtypes = [I] * 8 + [P] * 6
        _lib.oracle_topk.restype = I
        _lib.oracle_topk.argtypes = [I, I, I, P, P, I, P, P]
        _lib.oracle_sparse_attn.restype = I
        _lib.oracle_sparse_attn.argtypes = ([I] * 7 + [P] * 8 + [I, ctypes.c_double, I, I, P, P, P])
        _lib.oracle_lse_merge.restype = I
        _lib.oracle_lse_merge.argtypes = [I, ctypes.c_longlong, I, P, P, P, P]
        _lib.oracle_topk_sharded.restype = I
        _lib.oracle_topk_sharded.argtypes = [I, I, I, P, P, I, I, I, P]
        _lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        _lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        _lib.oracle_cache_append.restype = I
        _lib.oracle_cache_append.argtypes = [I] * 7 + [P] * 8 + [I, I, P, P, P]
        _lib.oracle_block_compress.restype = I
        _lib.oracle_block_compress.argtypes = [I] * 5 + [P] * 4
        _lib.oracle_block_score.restype = I
        _lib.oracle_block_score.argtypes = [I] * 7 + [P] * 5
        _lib.oracle_block_expand.restype = I
        _lib.oracle_block_expand.argtypes = [I] * 4 + [P] * 3
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous()
    return ctypes.c_void_p(t.data_ptr())


def _bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> its uint16 bit pattern (as int16 storage), CPU, contiguous."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16)


def _mask(row_mask):
    return None if row_mask is None else row_mask.to(torch.uint8).cpu().contiguous()


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(bits)


def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(byte)


def e4m3_encode(x: float) -> int:
    """E4M3 code of x: nearest finite value, ties to even, saturated to +-448."""
    return lib().oracle_e4m3_encode(float(x))


def cache_append(k_new, v_new, k_cache, v_cache, k_scale, v_scale, page_table, positions, label,
                 channels=None, index_key=None, page_size: int = 64):
    """The cache-append step on CPU copies: returns (k_cache, v_cache, label) after writing the new tokens.

    k_new, v_new bf16 [B, Hkv, D]; caches bf16 or uint8 (e4m3) [slots, Hkv, D]; label bf16 [slots, HL, C];
    channels int32 [Hkv, C] (per-head label) or index_key bf16 [B, C] (shared key); positions int32 [B].
    """
    B, Hkv, D = k_new.shape
    fp8 = k_cache.dtype == torch.uint8
    kc = k_cache.cpu().contiguous().clone() if fp8 else _bits(k_cache).clone()
    vc = v_cache.cpu().contiguous().clone() if fp8 else _bits(v_cache).clone()
    ks = k_scale.float().cpu().contiguous() if fp8 else None
    vs = v_scale.float().cpu().contiguous() if fp8 else None
    pt = page_table.to(torch.int32).cpu().contiguous()
    pos = positions.to(torch.int32).cpu().contiguous()
    lb = _bits(label).clone()
    HL, C = label.shape[1], label.shape[2]
    ch = channels.to(torch.int32).cpu().contiguous() if channels is not None else None
    ik = _bits(index_key) if index_key is not None else None
    num_pages = kc.shape[0] // page_size
    rc = lib().oracle_cache_append(B, Hkv, D, page_size, pt.shape[1], num_pages, int(fp8), _ptr(_bits(k_new)),
                                   _ptr(_bits(v_new)), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(pt),
                                   _ptr(pos), HL, C, _ptr(ch), _ptr(ik), _ptr(lb))
    if rc != 0:
        raise ValueError("oracle_cache_append: argument outside the definition")
    if not fp8:
        kc, vc = kc.view(torch.bfloat16), vc.view(torch.bfloat16)
    return kc, vc, lb.view(torch.bfloat16)


def index_score(qp, label, page_table, seq_lens, num_kv_heads: int, max_seq_len: int,
                page_size: int = 64, row_mask=None) -> torch.Tensor:
    """Proxy scores float32 [B, Hkv, max_seq_len]; positions t >= seq_lens[b] hold NaN."""
    B, Hq, C = qp.shape
    HL = label.shape[1]
    pt = page_table.to(torch.int32).cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    out = torch.full((B, num_kv_heads, max_seq_len), float("nan"), dtype=torch.float32)
    qb, lb, m = _bits(qp), _bits(label), _mask(row_mask)
    rc = lib().oracle_index_score(B, Hq, num_kv_heads, HL, C, page_size, pt.shape[1], max_seq_len,
                                  _ptr(qb), _ptr(lb), _ptr(pt), _ptr(sl), _ptr(m), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_index_score: argument outside the definition")
    return out


def topk(scores, seq_lens, k: int, row_mask=None) -> torch.Tensor:
    """Top-k token indices int32 [B, Hkv, k], ascending, -1 padded."""
    B, Hkv, Tmax = scores.shape
    s = scores.to(torch.float32).cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    out = torch.full((B, Hkv, max(k, 0)), -1, dtype=torch.int32)
    m = _mask(row_mask)
    rc = lib().oracle_topk(B, Hkv, Tmax, _ptr(s), _ptr(sl), k, _ptr(m), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_topk: argument outside the definition")
    return out


def block_compress(keys, page_table, seq_lens, num_pages: int, page_size: int = 64) -> torch.Tensor:
    """Compressed block keys bf16 [num_pages, C] (readings R15, R16); pages no request uses stay zero."""
    C = keys.shape[-1]
    kb = _bits(keys.reshape(-1, C))
    pt = page_table.to(torch.int32).cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    out = torch.zeros((num_pages, C), dtype=torch.int16)
    if lib().oracle_block_compress(pt.shape[0], C, page_size, pt.shape[1], num_pages, _ptr(kb), _ptr(pt), _ptr(sl),
                                   _ptr(out)) != 0:
        raise ValueError("oracle_block_compress: argument outside the definition")
    return out.view(torch.bfloat16)


def block_score(qp, block_keys, page_table, seq_lens, num_kv_heads: int, page_size: int = 64) -> torch.Tensor:
    """Block scores float32 [B, Hkv, max_pages]; blocks past ceil(T_b / 64) hold NaN."""
    B, Hq, C = qp.shape
    pt = page_table.to(torch.int32).cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    nbm = pt.shape[1]
    out = torch.full((B, num_kv_heads, nbm), float("nan"), dtype=torch.float32)
    if lib().oracle_block_score(B, Hq, num_kv_heads, C, page_size, pt.shape[1], nbm, _ptr(_bits(qp)),
                                _ptr(_bits(block_keys)), _ptr(pt), _ptr(sl), _ptr(out)) != 0:
        raise ValueError("oracle_block_score: argument outside the definition")
    return out


def block_expand(blocks, seq_lens, page_size: int = 64) -> torch.Tensor:
    """Tokens of the kept blocks int32 [B, Hkv, kb * 64], ascending, -1 padded (reading R17)."""
    B, Hkv, kb = blocks.shape
    bl = blocks.to(torch.int32).cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    out = torch.empty((B, Hkv, kb * page_size), dtype=torch.int32)
    if lib().oracle_block_expand(B, Hkv, kb, page_size, _ptr(bl), _ptr(sl), _ptr(out)) != 0:
        raise ValueError("oracle_block_expand: argument outside the definition")
    return out


def topk_sharded(scores, seq_lens, k: int, num_shards: int, page_size: int = 64) -> torch.Tensor:
    """Top-k by shard-local selection and a global merge (int32 [B, Hkv, k]); equals topk() by construction."""
    B, Hkv, Tmax = scores.shape
    sc = scores.float().cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    idx = torch.empty((B, Hkv, k), dtype=torch.int32)
    if lib().oracle_topk_sharded(B, Hkv, Tmax, _ptr(sc), _ptr(sl), k, num_shards, page_size, _ptr(idx)) != 0:
        raise ValueError("oracle_topk_sharded: argument outside the definition")
    return idx


def sparse_attn(q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, idx,
                sm_scale: Optional[float] = None, num_splits: int = 1, split_mode: int = 0,
                page_size: int = 64, row_mask=None):
    """Split partials (o_part float64 [S, B, Hq, D], lse_part float64 [S, B, Hq])."""
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    k = idx.shape[2]
    fp8 = k_cache.dtype == torch.uint8
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    kc = k_cache.cpu().contiguous() if fp8 else _bits(k_cache)
    vc = v_cache.cpu().contiguous() if fp8 else _bits(v_cache)
    ks = k_scale.float().cpu().contiguous() if fp8 else None
    vs = v_scale.float().cpu().contiguous() if fp8 else None
    pt = page_table.to(torch.int32).cpu().contiguous()
    sl = seq_lens.to(torch.int32).cpu().contiguous()
    ix = idx.to(torch.int32).cpu().contiguous()
    o = torch.zeros((num_splits, B, Hq, D), dtype=torch.float64)
    lse = torch.zeros((num_splits, B, Hq), dtype=torch.float64)
    qb, m = _bits(q), _mask(row_mask)
    rc = lib().oracle_sparse_attn(B, Hq, Hkv, D, page_size, pt.shape[1], int(fp8),
                                  _ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(pt), _ptr(sl),
                                  _ptr(ix), k, float(sm_scale), num_splits, split_mode, _ptr(m),
                                  _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_sparse_attn: argument outside the definition")
    return o, lse


def lse_merge(o_part: torch.Tensor, lse_part: torch.Tensor):
    """Merge partials [S, ..., D] / [S, ...] -> (out [..., D], lse [...]) in float64."""
    S = o_part.shape[0]
    D = o_part.shape[-1]
    rows = lse_part[0].numel()
    o = o_part.to(torch.float64).cpu().contiguous()
    l = lse_part.to(torch.float64).cpu().contiguous()
    out = torch.zeros(o.shape[1:], dtype=torch.float64)
    lse = torch.zeros(l.shape[1:], dtype=torch.float64)
    rc = lib().oracle_lse_merge(S, rows, D, _ptr(o), _ptr(l), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_lse_merge: argument outside the definition")
    return out, lse


def decode(inp, k: Optional[int] = None, sm_scale: Optional[float] = None, num_splits: int = 1,
           split_mode: int = 0, row_mask=None):
    """The four stages chained on one ``dsgen.Inputs``: (scores, idx, out, lse)."""
    w = inp.w
    k = w.top_k if k is None else k
    scores = index_score(inp.qp, inp.label, inp.page_table, inp.seq_lens, w.num_kv_heads,
                         w.max_seq_len, w.page_size, row_mask)
    idx = topk(scores, inp.seq_lens, k, row_mask)
    o, l = sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                       inp.seq_lens, idx, sm_scale, num_splits, split_mode, w.page_size, row_mask)
    out, lse = lse_merge(o, l)
    return scores, idx, out, lse
