"""Python binding of libdssparse: decode-step top-k sparse attention on one GPU.

Argument marshalling only. Every function takes torch CUDA tensors (device
memory) and passes their pointers, with the current torch stream, to the C
entry point of the same name declared in ``include/ds_sparse.h``; every step of
the computation runs in the library's CUDA kernels. There is no fallback: if
``libdssparse.so`` has not been built, importing the binding raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "Shape", "DsError", "ds_index_score", "ds_topk_select", "ds_topk_select_static", "ds_topk_workspace_bytes",
    "ds_sparse_decode_attn", "ds_lse_merge", "ds_sparse_decode", "ds_decode_workspace_bytes", "ds_cache_append",
    "ds_topk_select_sharded", "ds_topk_sharded_workspace_bytes", "ds_block_compress",
    "ds_block_decode_workspace_bytes", "ds_sparse_decode_blocks",
    "ds_device_errors", "ds_decode_kernel_launches", "ds_decode_num_splits", "lib", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdssparse.so")

DS_KV_BF16, DS_KV_FP8_E4M3 = 0, 1
DS_SPLIT_CONTIGUOUS, DS_SPLIT_PAGE_INTERLEAVED = 0, 1


class Shape(ctypes.Structure):
    """ds_shape: sizes shared by all entry points."""
    _fields_ = [("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("page_size", ctypes.c_int), ("max_pages_per_req", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("max_seq_len", ctypes.c_int)]


class DecodeArgs(ctypes.Structure):
    """ds_decode_args: the chained call's tensors."""
    _fields_ = [("q", ctypes.c_void_p), ("qp", ctypes.c_void_p), ("proxy_dim", ctypes.c_int),
                ("label", ctypes.c_void_p), ("label_heads", ctypes.c_int), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("k", ctypes.c_int), ("sm_scale", ctypes.c_float), ("idx", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class BlockDecodeArgs(ctypes.Structure):
    """ds_block_decode_args: the block-level decode step's tensors."""
    _fields_ = [("q", ctypes.c_void_p), ("qp", ctypes.c_void_p), ("proxy_dim", ctypes.c_int),
                ("block_keys", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("kb", ctypes.c_int),
                ("sm_scale", ctypes.c_float), ("blocks", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p)]


class DsError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().ds_error_string(status).decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


_lib = None


def lib():
    """The loaded libdssparse (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                              f"g.build()\"` (nvcc for sm_103a). There is no non-CUDA fallback.")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        SP = ctypes.POINTER(Shape)
        L.ds_index_score.argtypes = [SP, P, I, P, I, P, P, P, P]
        L.ds_topk_workspace_bytes.argtypes = [SP, I]
        L.ds_topk_workspace_bytes.restype = Z
        L.ds_topk_select.argtypes = [SP, P, P, I, P, P, Z, P]
        L.ds_topk_select_static.argtypes = [SP, P, P, I, P, P]
        L.ds_topk_select_static.restype = I
        L.ds_sparse_decode_attn.argtypes = [SP, P, P, P, I, P, P, P, P, P, I, ctypes.c_float, I, I, P, P, P, P, P]
        L.ds_lse_merge.argtypes = [I, I, I, P, P, P, P, P]
        L.ds_cache_append.argtypes = [SP, P, P, I, P, P, P, P, P, P, I, I, P, P, P, P]
        L.ds_topk_sharded_workspace_bytes.argtypes = [SP, I, I]
        L.ds_topk_sharded_workspace_bytes.restype = Z
        L.ds_topk_select_sharded.argtypes = [SP, P, P, I, I, P, P, Z, P]
        L.ds_decode_workspace_bytes.argtypes = [SP, I, I]
        L.ds_decode_workspace_bytes.restype = Z
        L.ds_sparse_decode.argtypes = [SP, ctypes.POINTER(DecodeArgs), P, Z, P]
        L.ds_sparse_decode_profiled.argtypes = [SP, ctypes.POINTER(DecodeArgs), P, Z, P, ctypes.POINTER(P)]
        L.ds_sparse_decode_profiled.restype = ctypes.c_int
        L.ds_decode_num_splits.argtypes = [SP, I]
        L.ds_decode_num_splits.restype = I
        L.ds_decode_kernel_launches.argtypes = [SP, I]
        L.ds_decode_kernel_launches.restype = I
        L.ds_block_compress.argtypes = [SP, P, I, P, P, I, P, P]
        L.ds_block_decode_workspace_bytes.argtypes = [SP, I]
        L.ds_block_decode_workspace_bytes.restype = Z
        L.ds_sparse_decode_blocks.argtypes = [SP, ctypes.POINTER(BlockDecodeArgs), P, Z, P]
        L.ds_error_string.argtypes = [I]
        L.ds_error_string.restype = ctypes.c_char_p
        L.ds_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        for name in ("ds_index_score", "ds_topk_select", "ds_sparse_decode_attn", "ds_lse_merge",
                     "ds_sparse_decode", "ds_device_errors", "ds_cache_append", "ds_topk_select_sharded",
                     "ds_block_compress", "ds_sparse_decode_blocks"):
            getattr(L, name).restype = I
        _lib = L
    return _lib


# Load eagerly so that a missing library fails at import time.
lib()


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libdssparse takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libdssparse takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != 0:
        raise DsError(status, where)


def _kv_dtype(cache: torch.Tensor) -> int:
    if cache.dtype == torch.bfloat16:
        return DS_KV_BF16
    if cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        return DS_KV_FP8_E4M3
    raise ValueError(f"unsupported KV dtype {cache.dtype}")


def ds_index_score(shape: Shape, qp, label, page_table, seq_lens, scores, stream=None) -> None:
    """Stage 1 (ds_index_score): proxy scores into ``scores`` [B, Hkv, max_seq_len] fp32."""
    _check(lib().ds_index_score(ctypes.byref(shape), _p(qp), qp.shape[-1], _p(label), label.shape[1],
                                _p(page_table), _p(seq_lens), _p(scores), _stream(stream)), "ds_index_score")


def ds_topk_workspace_bytes(shape: Shape, k: int) -> int:
    return lib().ds_topk_workspace_bytes(ctypes.byref(shape), k)


def ds_topk_select(shape: Shape, scores, seq_lens, k: int, idx, workspace, stream=None) -> None:
    """Stage 2 (ds_topk_select): exact top-k token indices into ``idx`` [B, Hkv, k] int32."""
    _check(lib().ds_topk_select(ctypes.byref(shape), _p(scores), _p(seq_lens), k, _p(idx), _p(workspace),
                                workspace.numel() * workspace.element_size() if workspace is not None else 0,
                                _stream(stream)), "ds_topk_select")


def ds_topk_select_static(shape: Shape, scores, seq_lens, k: int, idx, stream=None) -> None:
    """ds_topk_select with the library's fixed 16 MiB device scratch instead of a workspace.

    For callers that cannot allocate device memory. Calls that overlap on the
    GPU share the scratch and race; the first call on a device should come
    before any stream capture.
    """
    _check(lib().ds_topk_select_static(ctypes.byref(shape), _p(scores), _p(seq_lens), k, _p(idx), _stream(stream)),
           "ds_topk_select_static")


def ds_sparse_decode_attn(shape: Shape, q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, idx,
                          sm_scale: Optional[float] = None, num_splits: int = 1, split_mode: int = 0,
                          o_part=None, lse_part=None, out=None, lse=None, stream=None) -> None:
    """Stage 3 (ds_sparse_decode_attn): out/lse (one split) or o_part/lse_part (several)."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(shape.head_dim)
    k = idx.shape[-1]
    _check(lib().ds_sparse_decode_attn(ctypes.byref(shape), _p(q), _p(k_cache), _p(v_cache), _kv_dtype(k_cache),
                                       _p(k_scale), _p(v_scale), _p(page_table), _p(seq_lens), _p(idx), k,
                                       float(sm_scale), num_splits, split_mode, _p(o_part), _p(lse_part), _p(out),
                                       _p(lse), _stream(stream)), "ds_sparse_decode_attn")


def ds_lse_merge(o_part, lse_part, out, lse=None, stream=None) -> None:
    """Stage 4 (ds_lse_merge): o_part [S, rows..., D], lse_part [S, rows...] -> out bf16, lse fp32."""
    S = o_part.shape[0]
    D = o_part.shape[-1]
    rows = lse_part[0].numel()
    _check(lib().ds_lse_merge(S, rows, D, _p(o_part), _p(lse_part), _p(out), _p(lse), _stream(stream)),
           "ds_lse_merge")


def ds_topk_sharded_workspace_bytes(shape: Shape, k: int, num_shards: int) -> int:
    return lib().ds_topk_sharded_workspace_bytes(ctypes.byref(shape), k, num_shards)


def ds_topk_select_sharded(shape: Shape, scores, seq_lens, k: int, num_shards: int, idx, workspace,
                           stream=None) -> None:
    """ds_topk_select by page-interleaved shards and an exact merge (ds_topk_select_sharded); same result."""
    _check(lib().ds_topk_select_sharded(ctypes.byref(shape), _p(scores), _p(seq_lens), k, num_shards, _p(idx),
                                        _p(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "ds_topk_select_sharded")


def ds_cache_append(shape: Shape, k_new, v_new, k_cache, v_cache, k_scale, v_scale, page_table, positions,
                    label=None, channels=None, index_key=None, stream=None) -> None:
    """The step before the path (ds_cache_append): each request's new token into its slot, K/V and label."""
    fp8 = k_cache.dtype == torch.uint8
    proxy_dim = label.shape[-1] if label is not None else 0
    label_heads = label.shape[1] if label is not None else 0
    _check(lib().ds_cache_append(ctypes.byref(shape), _p(k_new), _p(v_new), DS_KV_FP8_E4M3 if fp8 else DS_KV_BF16,
                                 _p(k_cache), _p(v_cache), _p(k_scale) if fp8 else None,
                                 _p(v_scale) if fp8 else None, _p(page_table), _p(positions), proxy_dim,
                                 label_heads, _p(channels), _p(index_key), _p(label), _stream(stream)),
           "ds_cache_append")


def ds_decode_workspace_bytes(shape: Shape, proxy_dim: int, k: int) -> int:
    return lib().ds_decode_workspace_bytes(ctypes.byref(shape), proxy_dim, k)


def ds_sparse_decode(shape: Shape, q, qp, label, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens,
                     k: int, idx, out, lse=None, workspace=None, sm_scale: Optional[float] = None,
                     stream=None, events=None) -> None:
    """The chained decode step (ds_sparse_decode): idx, out and lse from the caches and queries.

    ``workspace`` (ds_decode_workspace_bytes bytes) must be zero-filled before
    its first use (torch.zeros); every call leaves it reusable without
    clearing. With ``events`` (four torch.cuda.Event
    objects with timing enabled) the instrumented entry point records them
    before scoring and after scoring, top-k and attention.
    """
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(shape.head_dim)
    a = DecodeArgs(q=_p(q), qp=_p(qp), proxy_dim=qp.shape[-1], label=_p(label), label_heads=label.shape[1],
                   k_cache=_p(k_cache), v_cache=_p(v_cache), kv_dtype=_kv_dtype(k_cache), k_scale=_p(k_scale),
                   v_scale=_p(v_scale), page_table=_p(page_table), seq_lens=_p(seq_lens), k=k,
                   sm_scale=float(sm_scale), idx=_p(idx), out=_p(out), lse=_p(lse))
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if events is None:
        st = lib().ds_sparse_decode(ctypes.byref(shape), ctypes.byref(a), _p(workspace), nbytes, _stream(stream))
    else:
        if len(events) != 4:
            raise ValueError("events: four torch.cuda.Event objects")
        for e in events:
            if not e.cuda_event:   # torch creates the handle on the first record
                e.record(stream if stream is not None else torch.cuda.current_stream())
        handles = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        st = lib().ds_sparse_decode_profiled(ctypes.byref(shape), ctypes.byref(a), _p(workspace), nbytes,
                                             _stream(stream), handles)
    _check(st, "ds_sparse_decode")


def ds_block_compress(shape: Shape, index_key, page_table, seq_lens, block_keys, last_page_only: bool = False,
                      stream=None) -> None:
    """Compressed block keys (ds_block_compress): bf16 [num_pages, C] from the index keys [slots, 1, C]."""
    _check(lib().ds_block_compress(ctypes.byref(shape), _p(index_key), index_key.shape[-1], _p(page_table),
                                   _p(seq_lens), 1 if last_page_only else 0, _p(block_keys), _stream(stream)),
           "ds_block_compress")


def ds_block_decode_workspace_bytes(shape: Shape, kb: int) -> int:
    return lib().ds_block_decode_workspace_bytes(ctypes.byref(shape), kb)


def ds_sparse_decode_blocks(shape: Shape, q, qp, block_keys, k_cache, v_cache, k_scale, v_scale, page_table,
                            seq_lens, kb: int, blocks, out, lse=None, workspace=None,
                            sm_scale: Optional[float] = None, stream=None) -> None:
    """The block-level decode step (ds_sparse_decode_blocks): kept blocks, out and lse."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(shape.head_dim)
    a = BlockDecodeArgs(q=_p(q), qp=_p(qp), proxy_dim=qp.shape[-1], block_keys=_p(block_keys), k_cache=_p(k_cache),
                        v_cache=_p(v_cache), kv_dtype=_kv_dtype(k_cache), k_scale=_p(k_scale),
                        v_scale=_p(v_scale), page_table=_p(page_table), seq_lens=_p(seq_lens), kb=kb,
                        sm_scale=float(sm_scale), blocks=_p(blocks), out=_p(out), lse=_p(lse))
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().ds_sparse_decode_blocks(ctypes.byref(shape), ctypes.byref(a), _p(workspace), nbytes,
                                         _stream(stream)), "ds_sparse_decode_blocks")


def ds_decode_kernel_launches(shape: Shape, k: int) -> int:
    """Kernel launches one chained call makes (host-only query)."""
    return lib().ds_decode_kernel_launches(ctypes.byref(shape), k)


def ds_decode_num_splits(shape: Shape, k: int) -> int:
    """Split-KV count the chained call uses internally (host-only query)."""
    return lib().ds_decode_num_splits(ctypes.byref(shape), k)


def ds_device_errors() -> int:
    """Synchronises, returns and clears the sticky device error word (DS_DEVERR_* bits)."""
    flags = ctypes.c_uint(0)
    st = lib().ds_device_errors(ctypes.byref(flags))
    if st not in (0, -5):
        raise DsError(st, "ds_device_errors")
    return flags.value
