"""Thin Python binding over the libpagedkv C ABI (include/pagedkv.h).

Every function here only checks dtypes/devices, reads pointers, sizes and
strides off torch tensors, allocates outputs/workspace with torch when the
caller did not pass them, and calls the C entry point of the same name on the
current CUDA stream.  All computation runs in the library's CUDA kernels.
There is no fallback: if libpagedkv.so is missing or was built for another
architecture the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from pathlib import Path
from typing import Optional

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libpagedkv.so"

PKV_STATUS_BAD_SLOT = 1
PKV_STATUS_BAD_BLOCK = 2
PKV_STATUS_BAD_LENGTH = 4
PKV_STATUS_TIMEOUT = 8
PKV_STATUS_DUP_SLOT = 16

_ERRNAMES = {1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_WORKSPACE",
             4: "PKV_ERR_CUDA", 5: "PKV_ERR_DEVICE_CHECK", 6: "PKV_ERR_DEVICE_TIMEOUT"}


class PagedKVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRNAMES.get(code, code)}: {msg}")
        self.code = code


_P, _I32, _I64, _F32, _SZ, _INT = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_float, ctypes.c_size_t, ctypes.c_int)

SIGNATURES = {
    "pkv_last_error": ([], ctypes.c_char_p),
    "pkv_version": ([], _INT),
    "pkv_set_validate": ([_INT], None),
    "pkv_device_status": ([_P, _P, _INT], _INT),
    "pkv_set_decode_chunk_tiles": ([_INT], _INT),
    "kv_build_slot_mapping": ([_P, _I64, _I32, _P, _P, _I32, _I32, _P, _I32, _P], _INT),
    "kv_build_decode_slots": ([_P, _I64, _I32, _P, _I32, _I32, _P, _P], _INT),
    "kv_store": ([_P, _I64, _P, _I64, _P, _P, _P, _I32, _I32, _I32, _I64, _P], _INT),
    "qk_norm_rope_store": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _F32, _F32, _P, _I64, _P,
                            _I64, _P, _P, _P, _I32, _I32, _I32, _I32, _I64, _P], _INT),
    "paged_attn_prefill": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I32, _P, _P,
                            _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _I64,
                            _P, _P, _SZ, _P], _INT),
    "paged_attn_prefill_workspace_size": ([_I32, _I32, _I32, _I32], _SZ),
    "paged_attn_decode": ([_P, _I64, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32, _I32, _I32,
                           _I32, _I32, _F32, _P, _I64, _P, _P, _SZ, _P], _INT),
    "paged_attn_decode_store": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I32, _P,
                                 _I32, _I32, _I32, _I32, _I32, _I32, _F32, _P, _I64, _P, _P, _SZ,
                                 _P], _INT),
    "paged_attn_decode_workspace_size": ([_I32, _I32, _I32, _I32, _I32], _SZ),
    "paged_attn_decode_noalloc": ([_P, _I64, _P, _P, _I64, _P, _I64, _I32, _P, _I32, _I32, _I32,
                                   _I32, _I32, _I32, _F32, _P, _I64, _P, _P], _INT),
}

_lib = None


def library_path() -> Path:
    return _LIB_PATH


def lib():
    """The loaded libpagedkv (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_303_gb300.build` (nvcc, sm_103a)")
        l = ctypes.CDLL(str(_LIB_PATH))
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        _lib = l
    return _lib


def _check(rc: int):
    if rc != 0:
        raise PagedKVError(rc, lib().pkv_last_error().decode(errors="replace"))


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _cuda(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _rows(t: torch.Tensor, name: str):
    """[rows, heads, head_dim] with heads and head_dim contiguous; returns row stride."""
    _cuda(t, torch.bfloat16, name)
    if t.dim() != 3:
        raise ValueError(f"{name} must be [rows, heads, head_dim]")
    if t.stride(2) != 1 or (t.shape[1] > 1 and t.stride(1) != t.shape[2]):
        raise ValueError(f"{name}: heads and head_dim must be contiguous within a row")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1] * t.shape[2]


def _i32(t: torch.Tensor, name: str):
    _cuda(t, torch.int32, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _table(bt: torch.Tensor):
    _cuda(bt, torch.int32, "block_tables")
    if bt.dim() != 2 or bt.stride(1) != 1:
        raise ValueError("block_tables must be [num_seqs, max_blocks] with unit column stride")
    return bt.stride(0) if bt.shape[0] > 1 else bt.shape[1], bt.shape[1]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def set_validate(on: bool):
    lib().pkv_set_validate(1 if on else 0)


def set_decode_chunk_tiles(tiles: int):
    """Force decode chunks of tiles*32 keys (0 restores the automatic plan)."""
    _check(lib().pkv_set_decode_chunk_tiles(int(tiles)))


def device_status(clear: bool = True, device=None) -> int:
    dev = torch.device(device or torch.cuda.current_device())
    st = ctypes.c_uint32(0)
    _check(lib().pkv_device_status(_stream(dev), ctypes.byref(st), 1 if clear else 0))
    return st.value


def kv_build_slot_mapping(block_tables, start, cu_seqlens_q, block_size: int,
                          num_tokens: Optional[int] = None, out: Optional[torch.Tensor] = None):
    """slot_mapping for a prefill / chunked-prefill step (int32 [num_tokens])."""
    bt_stride, width = _table(block_tables)
    start = _i32(start, "start")
    cu = _i32(cu_seqlens_q, "cu_seqlens_q")
    num_seqs = cu.numel() - 1
    if out is None:
        if num_tokens is None:
            num_tokens = int(cu[-1].item())
        out = torch.empty(num_tokens, dtype=torch.int32, device=cu.device)
    _i32(out, "slot_mapping")
    _check(lib().kv_build_slot_mapping(_ptr(block_tables), bt_stride, width, _ptr(start), _ptr(cu),
                                       num_seqs, block_size, _ptr(out), out.numel(),
                                       _stream(cu.device)))
    return out


def kv_build_decode_slots(block_tables, context_lens, block_size: int,
                          out: Optional[torch.Tensor] = None):
    """The slot of each decode row's new token; -1 for padding rows (context 0)."""
    bt_stride, width = _table(block_tables)
    ctx = _i32(context_lens, "context_lens")
    if out is None:
        out = torch.empty(ctx.numel(), dtype=torch.int32, device=ctx.device)
    _i32(out, "slot_mapping")
    _check(lib().kv_build_decode_slots(_ptr(block_tables), bt_stride, width, _ptr(ctx), ctx.numel(),
                                       block_size, _ptr(out), _stream(ctx.device)))
    return out


def kv_store(key, value, k_cache, v_cache, slot_mapping):
    """store_kvcache: k_cache[slot] = key[n], v_cache[slot] = value[n] for slot != -1."""
    krs = _rows(key, "key")
    vrs = _rows(value, "value")
    for c, name in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda(c, torch.bfloat16, name)
        if not c.is_contiguous():
            raise ValueError(f"{name} must be contiguous [num_blocks, block_size, Hkv, d]")
    n, hkv, d = key.shape
    if value.shape != key.shape:
        raise ValueError("key and value shapes differ")
    slots = _i32(slot_mapping, "slot_mapping")
    if slots.numel() != n:
        raise ValueError("slot_mapping must have one entry per token")
    D = hkv * d
    num_slots = k_cache.numel() // D
    if k_cache.numel() != v_cache.numel() or k_cache.numel() % D:
        raise ValueError("cache sizes do not match num_kv_heads * head_dim")
    _check(lib().kv_store(_ptr(key), krs, _ptr(value), vrs, _ptr(k_cache), _ptr(v_cache),
                          _ptr(slots), n, hkv, d, num_slots, _stream(key.device)))


def qk_norm_rope_store(q, k, v, positions, q_norm_weight, k_norm_weight, k_cache, v_cache,
                       slot_mapping, eps: float = 1e-6, theta: float = 1e6,
                       q_out: Optional[torch.Tensor] = None, k_out: Optional[torch.Tensor] = None):
    """QK-Norm then RoPE on q [N, Hq, d] and k [N, Hkv, d], fused with the
    store of the rotated k and of v [N, Hkv, d] into the paged caches.
    Returns (q_out, k_out); q_out=q (and k_out=k) rotate in place; k_out None
    writes rotated k only to the cache."""
    qrs, krs, vrs = _rows(q, "q"), _rows(k, "k"), _rows(v, "v")
    n, hq, d = q.shape
    hkv = k.shape[1]
    if tuple(k.shape) != (n, hkv, d) or tuple(v.shape) != (n, hkv, d):
        raise ValueError("q, k, v must be [N, heads, head_dim] with the same N and head_dim")
    _cuda(k_cache, torch.bfloat16, "k_cache")
    _cuda(v_cache, torch.bfloat16, "v_cache")
    if k_cache.shape != v_cache.shape or k_cache.shape[2:] != (hkv, d) or not k_cache.is_contiguous() \
            or not v_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, d]")
    pos = positions
    if pos.dtype != torch.int64 or pos.device != q.device or not pos.is_contiguous() or pos.numel() != n:
        raise ValueError("positions must be a contiguous int64 CUDA tensor with one entry per token")
    for w, name in ((q_norm_weight, "q_norm_weight"), (k_norm_weight, "k_norm_weight")):
        _cuda(w, torch.bfloat16, name)
        if w.numel() != d or not w.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [head_dim] bf16 tensor")
    slots = _i32(slot_mapping, "slot_mapping")
    if slots.numel() != n:
        raise ValueError("slot_mapping must have one entry per token")
    if q_out is None:
        q_out = torch.empty((n, hq, d), dtype=torch.bfloat16, device=q.device)
    qors = _rows(q_out, "q_out")
    kors = _rows(k_out, "k_out") if k_out is not None else 0
    num_slots = k_cache.shape[0] * k_cache.shape[1]
    _check(lib().qk_norm_rope_store(_ptr(q), qrs, _ptr(k), krs, _ptr(v), vrs, _ptr(pos),
                                    _ptr(q_norm_weight), _ptr(k_norm_weight), float(eps),
                                    float(theta), _ptr(q_out), qors, _ptr(k_out), kors,
                                    _ptr(k_cache), _ptr(v_cache), _ptr(slots), n, hq, hkv, d,
                                    num_slots, _stream(q.device)))
    return q_out, k_out


def decode_workspace_size(batch, num_heads, num_kv_heads, head_dim, max_context_len) -> int:
    return int(lib().paged_attn_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                                      max_context_len))


def prefill_workspace_size(num_seqs, total_q, max_seqlen_q, num_heads) -> int:
    return int(lib().paged_attn_prefill_workspace_size(num_seqs, total_q, max_seqlen_q, num_heads))


def _workspace(nbytes: int, device, ws: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    return ws, ws.numel() * ws.element_size()


def paged_attn_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                      softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      return_lse: bool = False):
    """Single-token paged decode: q [B, Hq, d] -> out [B, Hq, d] (bf16)."""
    qrs = _rows(q, "q")
    b, hq, d = q.shape
    _cuda(k_cache, torch.bfloat16, "k_cache")
    _cuda(v_cache, torch.bfloat16, "v_cache")
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    bt_stride, width = _table(block_tables)
    ctx = _i32(context_lens, "context_lens")
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=q.device)
    ors = _rows(out, "out")
    if return_lse and lse is None:
        lse = torch.empty((b, hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _cuda(lse, torch.float32, "lse")
    need = decode_workspace_size(b, hq, hkv, d, max_context_len)
    workspace, wbytes = _workspace(need, q.device, workspace)
    _check(lib().paged_attn_decode(_ptr(q), qrs, _ptr(k_cache), _ptr(v_cache), nb,
                                   _ptr(block_tables), bt_stride, width, _ptr(ctx), b, hq, hkv, d, bs,
                                   max_context_len, float(scale), _ptr(out), ors, _ptr(lse),
                                   _ptr(workspace), wbytes, _stream(q.device)))
    return (out, lse) if return_lse else out


def paged_attn_decode_store(q, key, value, k_cache, v_cache, block_tables, context_lens,
                            max_context_len: int, softmax_scale: Optional[float] = None,
                            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, return_lse: bool = False):
    """Writes this step's key/value [B, Hkv, d] to each row's decode slot and
    attends over the context (new token included) in one launch."""
    qrs = _rows(q, "q")
    krs, vrs = _rows(key, "key"), _rows(value, "value")
    b, hq, d = q.shape
    _cuda(k_cache, torch.bfloat16, "k_cache")
    _cuda(v_cache, torch.bfloat16, "v_cache")
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    if tuple(key.shape) != (b, hkv, d) or tuple(value.shape) != (b, hkv, d):
        raise ValueError("key/value must be [batch, num_kv_heads, head_dim]")
    bt_stride, width = _table(block_tables)
    ctx = _i32(context_lens, "context_lens")
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=q.device)
    ors = _rows(out, "out")
    if return_lse and lse is None:
        lse = torch.empty((b, hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _cuda(lse, torch.float32, "lse")
    need = decode_workspace_size(b, hq, hkv, d, max_context_len)
    workspace, wbytes = _workspace(need, q.device, workspace)
    _check(lib().paged_attn_decode_store(_ptr(q), qrs, _ptr(key), krs, _ptr(value), vrs,
                                         _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables),
                                         bt_stride, width, _ptr(ctx), b, hq, hkv, d, bs,
                                         max_context_len, float(scale), _ptr(out), ors, _ptr(lse),
                                         _ptr(workspace), wbytes, _stream(q.device)))
    return (out, lse) if return_lse else out


def paged_attn_prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                       softmax_scale: Optional[float] = None, *, k_cache=None, v_cache=None,
                       block_tables=None, out: Optional[torch.Tensor] = None,
                       lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                       return_lse: bool = False):
    """Varlen causal prefill.  Without block_tables keys come from the packed
    k/v [total_k, Hkv, d]; with block_tables from the paged caches."""
    qrs = _rows(q, "q")
    total_q, hq, d = q.shape
    cu_q = _i32(cu_seqlens_q, "cu_seqlens_q")
    cu_k = _i32(cu_seqlens_k, "cu_seqlens_k")
    num_seqs = cu_q.numel() - 1
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d)
    if block_tables is None:
        krs, vrs = _rows(k, "k"), _rows(v, "v")
        total_k, hkv = k.shape[0], k.shape[1]
        nb, bs, bt_stride, width = 0, 0, 0, 0
        kc = vc = None
    else:
        krs = vrs = 0
        k = v = None
        _cuda(k_cache, torch.bfloat16, "k_cache")
        _cuda(v_cache, torch.bfloat16, "v_cache")
        nb, bs, hkv, _ = k_cache.shape
        bt_stride, width = _table(block_tables)
        total_k = 0
        kc, vc = k_cache, v_cache
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=torch.bfloat16, device=q.device)
    ors = _rows(out, "out")
    if return_lse and lse is None:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    need = prefill_workspace_size(num_seqs, total_q, max_seqlen_q, hq)
    workspace, wbytes = _workspace(need, q.device, workspace)
    _check(lib().paged_attn_prefill(_ptr(q), qrs, _ptr(k), krs, _ptr(v), vrs, _ptr(kc), _ptr(vc), nb,
                                    _ptr(block_tables), bt_stride, width, _ptr(cu_q), _ptr(cu_k),
                                    max_seqlen_q, max_seqlen_k, num_seqs, total_q, total_k, hq, hkv,
                                    d, bs, float(scale), _ptr(out), ors, _ptr(lse), _ptr(workspace),
                                    wbytes, _stream(q.device)))
    return (out, lse) if return_lse else out
