"""Small helpers shared by the tests (no method arithmetic)."""
import contextlib
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device, any strides) -> numpy uint16 bit patterns with
    the same shape and the same element strides."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def f64(a_bits: np.ndarray) -> np.ndarray:
    """exact bf16 bits -> float64"""
    return (np.asarray(a_bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_of(values) -> np.ndarray:
    """float values that are exactly representable in bf16 -> bit patterns"""
    t = torch.as_tensor(np.asarray(values, dtype=np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float32), t), "value not exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


@contextlib.contextmanager
def decode_chunk_tiles(tiles):
    """Force decode chunks of tiles*32 keys inside the block (None or 0: the
    library's automatic plan), restoring the automatic plan afterwards."""
    from paged_kv_cache_303_gb300 import ops
    ops.set_decode_chunk_tiles(int(tiles or 0))
    try:
        yield
    finally:
        ops.set_decode_chunk_tiles(0)
