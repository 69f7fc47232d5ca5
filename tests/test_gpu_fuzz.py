"""Seeded random cases for the attention paths, each against the oracle.

The hand-picked parity cases pin one mechanism each; these draw the
combinations at random: head shapes with GQA groups 1 to 8, 12 and 16,
head_dim 64 and 128, every power-of-two block size from 1 to 256, length
mixes that hit the tile edges (0, 1, 63-65, 127-129 rows or keys) beside
uniform draws, cached prefixes aligned or not to the block size, and decode
batches with padding rows (context 0), for the decode call and the fused
store + decode step, and chunked-prefill mixed batches (decode rows among
prompt chunks in one prefill call).  Unused cache slots hold NaN, so a
masked key that reached a sum would show.  Every case is fixed by its seed.
"""
import random

import pytest

from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from test_gpu_fused import _decode_store_case
from test_gpu_parity import _decode_case, _prefill_packed, _prefill_paged

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_303_gb300 import build
    build.build()
    ops.device_status(clear=True)
    yield
    assert ops.device_status(clear=True) == 0, "a kernel flagged its input"

# (query heads, kv heads): groups 1 to 8, 12 and 16
HEAD_SHAPES = [(8, 8), (16, 8), (12, 4), (10, 2), (16, 4), (32, 4), (5, 1), (12, 2), (7, 1), (24, 2),
               (32, 2)]
BLOCK_SIZES = [1, 2, 4, 8, 16, 32, 64, 128, 256]
EDGE_LENGTHS = [0, 1, 63, 64, 65, 127, 128, 129]


def _length(rng: random.Random, top: int) -> int:
    return rng.choice(EDGE_LENGTHS) if rng.random() < 0.4 else rng.randint(1, top)


def _heads(rng: random.Random, block_size: int, tokens_per_seq, shape=None) -> W.Heads:
    hq, hkv = rng.choice(HEAD_SHAPES) if shape is None else shape
    d = rng.choice([64, 128])
    blocks = sum((t + block_size - 1) // block_size for t in tokens_per_seq)
    return W.Heads(hq, hkv, d, block_size, blocks + 8)


@pytest.mark.parametrize("seed", range(24))
def test_random_packed_prefill(seed):
    rng = random.Random(20000 + seed)
    lens = [_length(rng, 400) for _ in range(rng.randint(1, 5))]
    if not any(lens):
        lens[0] = 1
    heads = _heads(rng, 16, lens)
    _prefill_packed(heads, lens, seed=21000 + seed, growing=rng.random() < 0.3)


@pytest.mark.parametrize("seed", range(36))
def test_random_paged_prefill(seed):
    rng = random.Random(22000 + seed)
    bs = BLOCK_SIZES[seed % len(BLOCK_SIZES)]
    n = rng.randint(1, 4)
    q_lens = [_length(rng, 300) for _ in range(n)]
    if not any(q_lens):
        q_lens[0] = 1
    prefix = [rng.choice([0, bs, 3 * bs]) if rng.random() < 0.4 else rng.randint(1, 700)
              for _ in range(n)]
    heads = _heads(rng, bs, [q + p for q, p in zip(q_lens, prefix)])
    _prefill_paged(heads, q_lens, prefix, seed=23000 + seed, growing=rng.random() < 0.3)


@pytest.mark.parametrize("seed", range(18))
def test_random_mixed_prefill(seed):
    """Chunked-prefill mixed batches: decode rows (one new token behind a
    cached context) interleaved with prompt chunks (cached prefix or none)
    in one paged prefill call."""
    rng = random.Random(29000 + seed)
    bs = BLOCK_SIZES[seed % len(BLOCK_SIZES)]
    q_lens, prefix = [], []
    for _ in range(rng.randint(2, 8)):
        if rng.random() < 0.5:
            q_lens.append(1)
            prefix.append(rng.choice([0, bs - 1, bs, 127, 128]) if rng.random() < 0.3
                          else rng.randint(1, 2500))
        else:
            q_lens.append(_length(rng, 400) or 1)
            prefix.append(0 if rng.random() < 0.3 else rng.randint(1, 1500))
    heads = _heads(rng, bs, [q + p for q, p in zip(q_lens, prefix)],
                   HEAD_SHAPES[seed % len(HEAD_SHAPES)])
    _prefill_paged(heads, q_lens, prefix, seed=30000 + seed)


def _decode_draw(rng: random.Random, seed: int):
    bs = BLOCK_SIZES[seed % len(BLOCK_SIZES)]
    ctx = [rng.choice([0, 1, bs, bs + 1]) if rng.random() < 0.3 else _length(rng, 3000)
           for _ in range(rng.randint(1, 9))]
    if not any(ctx):
        ctx[0] = 1
    # the head shapes in turn, so that every group size meets the decode kernel
    return _heads(rng, bs, ctx, HEAD_SHAPES[seed % len(HEAD_SHAPES)]), ctx


@pytest.mark.parametrize("seed", range(27))
def test_random_decode(seed):
    heads, ctx = _decode_draw(random.Random(24000 + seed), seed)
    _decode_case(heads, ctx, seed=25000 + seed)


@pytest.mark.parametrize("seed", range(27))
def test_random_decode_store(seed):
    """The fused step (decode slot, K/V store and decode in one launch):
    oracle, cache bits and the unfused sequence."""
    heads, ctx = _decode_draw(random.Random(26000 + seed), seed)
    _decode_store_case(heads, ctx, seed=27000 + seed, cache_seed=28000 + seed)
