"""CPU oracle for the paged KV cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``paged_kv_cache_303_gb300``)
never imports, links or calls it, and this package imports nothing from the
product: the two share no code.  The arithmetic lives in ``oracle.c`` (plain
C loops, fp64 accumulation); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

bf16 tensors are passed as ``numpy.uint16`` arrays holding the raw bf16 bits.

What each function follows (page title + section):

* ``slot_mapping_blockwalk`` / ``slot_mapping_per_token`` -- "Lesson 04:
  where exactly does the KV go", §2 (slot_mapping construction) and §7
  (Exercise A).  Pinned by the worked answers of Exercise A.
* ``decode_slots`` -- same page, §9 item 1; "L17: Qwen3 attention
  sub-layer" §7 (context length counts the token just written).
* ``kv_store`` -- "L17: Qwen3 attention sub-layer" §5.1 (scatter_kernel and
  store_kvcache examples, both pinned by their printed outputs).
* ``prefill`` / ``decode`` -- "L17: Qwen3 attention sub-layer" §5.2 (naive
  definition) and §5.3 (prefill / prefix-cache / decode calls); pinned by
  closed forms, invariants and torch's scaled_dot_product_attention on
  special cases.
* ``online_softmax`` / ``decode_split`` -- §5.2 online-softmax rescaling;
  pinned by the worked example printed there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_DIR = Path(__file__).resolve().parent
_SRC = _DIR / "oracle.c"
# ORACLE_PLANT names one ORC_PLANT_* macro of oracle.c to compile in (used only
# by the test that checks the pins catch planted mistakes)
_PLANT = os.environ.get("ORACLE_PLANT", "")
_LIB = _DIR / (f"liboracle_{_PLANT.lower()}.so" if _PLANT else "liboracle.so")

ERRORS = {
    -1: "invalid argument",
    -2: "slot out of range",
    -3: "duplicate slot",
    -4: "block table entry missing or out of range",
    -5: "inconsistent lengths",
    -6: "out of memory",
}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what}: {ERRORS.get(code, code)} ({code})")
        self.code = code


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so (plain gcc, OpenMP for timing only)."""
    if force or not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               *([f"-D{_PLANT}"] if _PLANT else []), "-o", str(tmp), str(_SRC), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_D = ctypes.c_double
_INT = ctypes.c_int


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        sig = {
            "orc_version": ([], _INT),
            "orc_num_threads": ([_INT], _INT),
            "orc_slot_mapping_blockwalk": ([_P, _I64, _I32, _P, _P, _I32, _I32, _P, _I64], _INT),
            "orc_slot_mapping_per_token": ([_P, _I64, _I32, _P, _P, _I32, _I32, _P, _I64], _INT),
            "orc_decode_slots": ([_P, _I64, _I32, _P, _I32, _I32, _P], _INT),
            "orc_kv_store": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I64, _I64], _INT),
            "orc_prefill": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I32,
                             _P, _P, _I32, _I32, _I32, _I32, _I32, _D, _P, _P, _INT], _INT),
            "orc_decode": ([_P, _I64, _P, _P, _I64, _P, _I64, _I32, _P, _I32,
                            _I32, _I32, _I32, _I32, _D, _P, _P, _INT], _INT),
            "orc_online_softmax": ([_P, _P, _I64, _I64, _I64, _P, _P, _P, _P], _INT),
            "orc_prefill_rows": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _I64, _P, _I64, _I32,
                                  _P, _P, _I32, _I32, _I32, _I32, _I32, _D, _P, _I64, _P, _P,
                                  _INT], _INT),
            "orc_decode_split": ([_P, _I64, _P, _P, _I64, _P, _I64, _I32, _P, _I32,
                                  _I32, _I32, _I32, _I32, _D, _I64, _P, _P], _INT),
            "orc_round_bf16": ([_D], ctypes.c_uint16),
            "orc_qk_norm_rope": ([_P, _I64, _P, _I64, _P, _P, _P, _D, _D, _I64, _I32, _I32,
                                  _I32, _P, _P], _INT),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _u16(a):
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as uint16 bit patterns")
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(rc, what)


def num_threads(n: int = 0) -> int:
    """Threads the oracle's OpenMP loops use (n <= 0: the runtime default)."""
    return _load().orc_num_threads(n)


def _table(block_tables):
    bt = _i32(block_tables)
    if bt.ndim != 2:
        raise ValueError("block_tables must be 2-D [num_seqs, max_blocks]")
    return bt, bt.shape[1], bt.shape[1]


def slot_mapping_blockwalk(block_tables, start, cu_seqlens_q, block_size):
    bt, stride, width = _table(block_tables)
    start, cu = _i32(start), _i32(cu_seqlens_q)
    n = int(cu[-1])
    out = np.full(n, -7, dtype=np.int32)
    _check(_load().orc_slot_mapping_blockwalk(_ptr(bt), stride, width, _ptr(start), _ptr(cu),
                                              len(cu) - 1, block_size, _ptr(out), n),
           "slot_mapping_blockwalk")
    return out


def slot_mapping_per_token(block_tables, start, cu_seqlens_q, block_size):
    bt, stride, width = _table(block_tables)
    start, cu = _i32(start), _i32(cu_seqlens_q)
    n = int(cu[-1])
    out = np.full(n, -7, dtype=np.int32)
    _check(_load().orc_slot_mapping_per_token(_ptr(bt), stride, width, _ptr(start), _ptr(cu),
                                              len(cu) - 1, block_size, _ptr(out), n),
           "slot_mapping_per_token")
    return out


def slot_mapping(block_tables, start, cu_seqlens_q, block_size):
    """Both statements of the prefill slot mapping; they must agree."""
    a = slot_mapping_blockwalk(block_tables, start, cu_seqlens_q, block_size)
    b = slot_mapping_per_token(block_tables, start, cu_seqlens_q, block_size)
    if not np.array_equal(a, b):
        raise AssertionError("the two statements of slot_mapping disagree")
    return a


def decode_slots(block_tables, context_lens, block_size):
    bt, stride, width = _table(block_tables)
    ctx = _i32(context_lens)
    out = np.full(len(ctx), -7, dtype=np.int32)
    _check(_load().orc_decode_slots(_ptr(bt), stride, width, _ptr(ctx), len(ctx), block_size,
                                    _ptr(out)), "decode_slots")
    return out


def kv_store(key, value, k_cache, v_cache, slot_mapping):
    """In-place scatter.  key/value: uint16 [N, Hkv, d] views whose last two
    dims are contiguous (row stride free); caches: uint16
    [num_blocks, block_size, Hkv, d] contiguous."""
    key, value = _u16(key), _u16(value)
    for c in (k_cache, v_cache):
        if _u16(c).flags["C_CONTIGUOUS"] is False:
            raise ValueError("caches must be contiguous")
    n = key.shape[0]
    D = key.shape[1] * key.shape[2]
    item = key.itemsize
    for t in (key, value):
        if t.strides[2] != item or t.strides[1] != key.shape[2] * item:
            raise ValueError("key/value rows must be contiguous within a token")
    slots = _i32(slot_mapping)
    if slots.size != n:
        raise ValueError("slot_mapping must have one entry per token")
    num_slots = k_cache.size // D
    _check(_load().orc_kv_store(_ptr(key), key.strides[0] // item, _ptr(value),
                                value.strides[0] // item, _ptr(k_cache), _ptr(v_cache),
                                _ptr(slots), n, D, num_slots), "kv_store")


def _rows(t):
    t = _u16(t)
    item = t.itemsize
    if t.strides[-1] != item or t.strides[-2] != t.shape[-1] * item:
        raise ValueError("heads and head_dim must be contiguous within a row")
    return t, t.strides[0] // item


def prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, scale, *, k_cache=None, v_cache=None,
            block_tables=None, nthreads=0):
    """Varlen causal prefill.  q [Nq, Hq, d]; when block_tables is None, k/v are
    packed [Nk, Hkv, d]; otherwise keys come from the caches
    [num_blocks, block_size, Hkv, d].  Returns (out fp64 [Nq, Hq, d],
    lse fp64 [Nq, Hq])."""
    q, q_rs = _rows(q)
    nq, hq, d = q.shape
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    out = np.zeros((nq, hq, d), dtype=np.float64)
    lse = np.zeros((nq, hq), dtype=np.float64)
    if block_tables is None:
        k, k_rs = _rows(k)
        v, v_rs = _rows(v)
        hkv = k.shape[1]
        rc = _load().orc_prefill(_ptr(q), q_rs, _ptr(k), k_rs, _ptr(v), v_rs, None, None, 0,
                                 None, 0, 0, _ptr(cu_q), _ptr(cu_k), len(cu_q) - 1, hq, hkv, d,
                                 1, float(scale), _ptr(out), _ptr(lse), nthreads)
    else:
        k_cache, v_cache = _u16(k_cache), _u16(v_cache)
        nb, bs, hkv, _ = k_cache.shape
        bt, stride, width = _table(block_tables)
        rc = _load().orc_prefill(_ptr(q), q_rs, None, 0, None, 0, _ptr(k_cache), _ptr(v_cache),
                                 nb, _ptr(bt), stride, width, _ptr(cu_q), _ptr(cu_k),
                                 len(cu_q) - 1, hq, hkv, d, bs, float(scale), _ptr(out),
                                 _ptr(lse), nthreads)
    _check(rc, "prefill")
    return out, lse


def prefill_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, scale, rows, *, k_cache=None,
                 v_cache=None, block_tables=None, nthreads=0):
    """prefill() restricted to the given global query rows; returns
    (out fp64 [len(rows), Hq, d], lse fp64 [len(rows), Hq])."""
    q, q_rs = _rows(q)
    nq, hq, d = q.shape
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(rows), hq, d), dtype=np.float64)
    lse = np.zeros((len(rows), hq), dtype=np.float64)
    if block_tables is None:
        k, k_rs = _rows(k)
        v, v_rs = _rows(v)
        rc = _load().orc_prefill_rows(_ptr(q), q_rs, _ptr(k), k_rs, _ptr(v), v_rs, None, None, 0,
                                      None, 0, 0, _ptr(cu_q), _ptr(cu_k), len(cu_q) - 1, hq,
                                      k.shape[1], d, 1, float(scale), _ptr(rows), len(rows),
                                      _ptr(out), _ptr(lse), nthreads)
    else:
        k_cache, v_cache = _u16(k_cache), _u16(v_cache)
        nb, bs, hkv, _ = k_cache.shape
        bt, stride, width = _table(block_tables)
        rc = _load().orc_prefill_rows(_ptr(q), q_rs, None, 0, None, 0, _ptr(k_cache),
                                      _ptr(v_cache), nb, _ptr(bt), stride, width, _ptr(cu_q),
                                      _ptr(cu_k), len(cu_q) - 1, hq, hkv, d, bs, float(scale),
                                      _ptr(rows), len(rows), _ptr(out), _ptr(lse), nthreads)
    _check(rc, "prefill_rows")
    return out, lse


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, nthreads=0):
    """Single-token paged decode.  q [B, Hq, d]; returns (out fp64 [B, Hq, d],
    lse fp64 [B, Hq])."""
    q, q_rs = _rows(q)
    b, hq, d = q.shape
    k_cache, v_cache = _u16(k_cache), _u16(v_cache)
    nb, bs, hkv, _ = k_cache.shape
    bt, stride, width = _table(block_tables)
    ctx = _i32(context_lens)
    out = np.zeros((b, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq), dtype=np.float64)
    _check(_load().orc_decode(_ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), nb, _ptr(bt), stride,
                              width, _ptr(ctx), b, hq, hkv, d, bs, float(scale), _ptr(out),
                              _ptr(lse), nthreads), "decode")
    return out, lse


def decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, split):
    """Split-K decode merged by the rescaling identity; equals decode()."""
    q, q_rs = _rows(q)
    b, hq, d = q.shape
    k_cache, v_cache = _u16(k_cache), _u16(v_cache)
    nb, bs, hkv, _ = k_cache.shape
    bt, stride, width = _table(block_tables)
    ctx = _i32(context_lens)
    out = np.zeros((b, hq, d), dtype=np.float64)
    lse = np.zeros((b, hq), dtype=np.float64)
    _check(_load().orc_decode_split(_ptr(q), q_rs, _ptr(k_cache), _ptr(v_cache), nb, _ptr(bt),
                                    stride, width, _ptr(ctx), b, hq, hkv, d, bs, float(scale),
                                    int(split), _ptr(out), _ptr(lse)), "decode_split")
    return out, lse


def online_softmax(s, v, block):
    """Blocked online softmax of one row of scaled scores s[n] with values
    v[n, w].  Returns (out[w], m, l, trace) where trace[b] holds
    (m, l_rescaled, acc_rescaled[w], l_after, acc_after[w]) for block b."""
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float64))
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    if v.ndim == 1:
        v = v[:, None]
    n, w = v.shape
    nb = (n + block - 1) // block
    out = np.zeros(w)
    m = np.zeros(1)
    l = np.zeros(1)
    trace = np.zeros((nb, 3 + 2 * w))
    _check(_load().orc_online_softmax(_ptr(s), _ptr(v), n, w, block, _ptr(out), _ptr(m), _ptr(l),
                                      _ptr(trace)), "online_softmax")
    return out, float(m[0]), float(l[0]), trace


def round_bf16(x: float) -> int:
    """Nearest bf16 (ties to even) of a double, as its bit pattern."""
    return int(_load().orc_round_bf16(float(x)))


def qk_norm_rope(q, k, positions, q_weight, k_weight, eps=1e-6, theta=1e6):
    """QK-Norm then RoPE.  q: uint16 [N, Hq, d], k: uint16 [N, Hkv, d] (rows
    may be strided, heads contiguous), positions [N] int, weights uint16 [d].
    Returns (q_out, k_out) as contiguous uint16 arrays of the same shapes."""
    q, k = _u16(q), _u16(k)
    n, hq, d = q.shape
    hkv = k.shape[1]
    item = q.itemsize
    for t in (q, k):
        if t.strides[2] != item or t.strides[1] != d * item or t.shape[0] != n or t.shape[2] != d:
            raise ValueError("q/k must be [N, heads, d] with heads and d contiguous")
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    qw = np.ascontiguousarray(_u16(q_weight))
    kw = np.ascontiguousarray(_u16(k_weight))
    if pos.size != n or qw.size != d or kw.size != d:
        raise ValueError("positions must have N entries, weights d entries")
    qo = np.empty((n, hq, d), np.uint16)
    ko = np.empty((n, hkv, d), np.uint16)
    q_rs = q.strides[0] // item if n > 1 else hq * d
    k_rs = k.strides[0] // item if n > 1 else hkv * d
    _check(_load().orc_qk_norm_rope(_ptr(q), q_rs, _ptr(k), k_rs, _ptr(pos), _ptr(qw), _ptr(kw),
                                    float(eps), float(theta), n, hq, hkv, d, _ptr(qo), _ptr(ko)),
           "qk_norm_rope")
    return qo, ko
