"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact for slot mapping and the cache scatter; for attention every output
element must satisfy |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| (bf16 inputs,
fp32 accumulation on the GPU, fp64 in the oracle, bf16 output).  Inputs are
the seeded workloads; the oracle never sees a value the CUDA path produced:
each side builds its own slot mapping and its own cache from the same inputs.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits, bf16_bits_of, decode_chunk_tiles, f64, from_bits, golden

pytestmark = pytest.mark.gpu

TOL = 1e-2
NAN_BITS = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_303_gb300 import build
    build.build()
    ops.device_status(clear=True)
    yield
    assert ops.device_status(clear=True) == 0, "a kernel flagged its input"


def dev(t):
    return t.to("cuda")


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what: str, tol=TOL):
    g = gpu.detach().float().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    bound = tol + tol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance, "
                             f"max abs {np.nanmax(err):.3e}, first bad {idx}")


# ---------------------------------------------------------------------------
# slot mapping (bit-exact)
# ---------------------------------------------------------------------------
def test_slot_mapping_exercise():
    g = golden("t3_slot_mapping.json")
    bt = dev(torch.tensor([g["block_table"]], dtype=torch.int32))
    for case in g["cases"]:
        start = dev(torch.tensor([case["cached"]], dtype=torch.int32))
        cu = dev(torch.tensor([0, case["new_tokens"]], dtype=torch.int32))
        got = ops.kv_build_slot_mapping(bt, start, cu, g["block_size"])
        assert got.cpu().tolist() == case["slot_mapping"]


@pytest.mark.parametrize("bs", [1, 4, 16, 256])
def test_slot_mapping_random(bs):
    rng = np.random.default_rng(100 + bs)
    for _ in range(10):
        n = int(rng.integers(1, 40))
        start = rng.integers(0, 4 * bs + 3, n).astype(np.int32)
        lens = rng.integers(0, 4 * bs + 3, n).astype(np.int32)
        width = int(((start + lens + bs - 1) // bs).max()) + 2
        bt = rng.permutation(n * width * 2)[: n * width].reshape(n, width).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        ref = oracle.slot_mapping(bt, start, cu, bs)
        got = ops.kv_build_slot_mapping(dev(torch.from_numpy(bt)), dev(torch.from_numpy(start)),
                                        dev(torch.from_numpy(cu)), bs)
        assert np.array_equal(got.cpu().numpy(), ref)


def test_decode_slots_with_padding():
    work = W.large_decode(batch=40, pads=8, num_blocks=8000)
    ref = oracle.decode_slots(work.block_tables, work.context_lens, work.heads.block_size)
    got = ops.kv_build_decode_slots(dev(work.block_tables), dev(work.context_lens),
                                    work.heads.block_size)
    assert np.array_equal(got.cpu().numpy(), ref)
    assert (ref[-8:] == -1).all()


def test_missing_table_entry_is_flagged_not_written():
    bt = dev(torch.tensor([[3, -1]], dtype=torch.int32))
    got = ops.kv_build_slot_mapping(bt, dev(torch.tensor([0], dtype=torch.int32)),
                                    dev(torch.tensor([0, 6], dtype=torch.int32)), 4)
    assert got.cpu().tolist() == [12, 13, 14, 15, -1, -1]
    assert ops.device_status(clear=True) & ops.PKV_STATUS_BAD_BLOCK


# ---------------------------------------------------------------------------
# kv_store (bit-exact)
# ---------------------------------------------------------------------------
def test_store_scatter_toy():
    g = golden("t1_scatter_toy.json")
    src = from_bits(bf16_bits_of(g["src"]).reshape(3, 1, 4))
    kc = torch.zeros(3, 1, 1, 4, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ops.kv_store(dev(src), dev(src), kc, vc, dev(torch.tensor(g["slot"], dtype=torch.int32)))
    assert np.array_equal(kc.view(3, 4).float().cpu().numpy(), np.array(g["dst"], np.float32))


def test_store_kvcache_example_with_skip():
    g = golden("t2_store_kvcache.json")
    key = from_bits(bf16_bits_of(g["key"]))
    value = from_bits(bf16_bits_of(np.array(g["key"]) + g["value_offset"]))
    kc = torch.full((1, 4, 2, 2), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full((1, 4, 2, 2), float("nan"), dtype=torch.bfloat16, device="cuda")
    ops.kv_store(dev(key), dev(value), kc, vc, dev(torch.tensor(g["slot_mapping"], dtype=torch.int32)))
    rows = kc.view(4, 4).float().cpu().numpy()
    assert np.array_equal(rows[:3], np.array(g["k_cache_rows"][:3], np.float32))
    assert np.isnan(rows[3]).all()                       # no token maps to slot 3
    assert np.array_equal(vc.view(4, 4)[0].float().cpu().numpy(),
                          np.array(g["v_cache_slot0"], np.float32))


@pytest.mark.parametrize("fused,hkv,d", [(False, 8, 128), (True, 8, 128), (False, 2, 64),
                                         (True, 3, 20)])
def test_store_random_vs_oracle(fused, hkv, d):
    heads = W.Heads(2 * hkv, hkv, d, 16, 64)
    rng = np.random.default_rng(7)
    n = 300
    work = W.prefill_work(heads, [n], seed=200)
    if fused:   # k/v as views of one fused projection output (row stride > Hkv*d)
        qkv = torch.cat([work.q.flatten(1), work.k.flatten(1), work.v.flatten(1)], 1)
        qw = heads.num_heads * d
        key = qkv[:, qw:qw + hkv * d].view(n, hkv, d)
        value = qkv[:, qw + hkv * d:].view(n, hkv, d)
    else:
        key, value = work.k, work.v
    slots = rng.permutation(heads.num_blocks * heads.block_size)[:n].astype(np.int32)
    slots[rng.random(n) < 0.1] = -1
    kc, vc = W.history_cache(heads, 201)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    oracle.kv_store(bits(key), bits(value), kref, vref, slots)
    gk, gv = dev(kc), dev(vc)
    if fused:
        dq = dev(qkv)
        dkey = dq[:, qw:qw + hkv * d].view(n, hkv, d)
        dval = dq[:, qw + hkv * d:].view(n, hkv, d)
    else:
        dkey, dval = dev(key), dev(value)
    ops.kv_store(dkey, dval, gk, gv, dev(torch.from_numpy(slots)))
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)


def test_store_bad_slot_is_skipped_and_flagged():
    kc = torch.zeros(2, 4, 1, 8, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    x = torch.ones(3, 1, 8, dtype=torch.bfloat16, device="cuda")
    ops.kv_store(x, x, kc, vc, dev(torch.tensor([1, 8, -5], dtype=torch.int32)))
    assert ops.device_status(clear=True) & ops.PKV_STATUS_BAD_SLOT
    assert kc.view(8, 8)[1].eq(1).all() and kc.view(8, 8)[[0, 2, 3, 4, 5, 6, 7]].eq(0).all()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
def _poison_unused(kc: torch.Tensor, vc: torch.Tensor, block_tables, lens):
    """NaN every cache slot that no row reads (positions >= its length)."""
    nb, bs = kc.shape[0], kc.shape[1]
    used = torch.zeros(nb * bs, dtype=torch.bool)
    for row, n in zip(block_tables.tolist(), lens.tolist()):
        for j in range(int(n)):
            used[row[j // bs] * bs + j % bs] = True
    flat_k, flat_v = kc.view(nb * bs, -1), vc.view(nb * bs, -1)
    flat_k[~used] = float("nan")
    flat_v[~used] = float("nan")


def _decode_case(heads, ctx, seed, poison=True, lse=True):
    work = W.decode_work(heads, ctx, seed=seed)
    kc, vc = W.history_cache(heads, seed + 1)
    if poison:
        _poison_unused(kc, vc, work.block_tables, work.context_lens)
    # oracle side: write the new token with its own slot mapping, then decode
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, heads.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, ref_lse = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens,
                                 heads.scale, nthreads=0)
    # GPU side through the C ABI
    gk, gv = dev(kc), dev(vc)
    bt, ctxd = dev(work.block_tables), dev(work.context_lens)
    gslots = ops.kv_build_decode_slots(bt, ctxd, heads.block_size)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, gslots)
    out, out_lse = ops.paged_attn_decode(dev(work.q), gk, gv, bt, ctxd, max(1, work.max_context_len),
                                         heads.scale, return_lse=True)
    torch.cuda.synchronize()
    assert np.array_equal(gslots.cpu().numpy(), slots)
    assert_close(out, ref, "decode out")
    fin = np.isfinite(ref_lse)
    got_lse = out_lse.cpu().double().numpy()
    assert np.array_equal(np.isfinite(got_lse), fin)
    if lse:
        assert np.allclose(got_lse[fin], ref_lse[fin], atol=2e-3, rtol=1e-4)
    return work


DECODE_SHAPES = [
    # Hq, Hkv, d, bs, contexts
    (16, 8, 128, 256, [1, 63, 64, 65, 255, 256, 257, 1000, 2047]),
    (4, 2, 64, 4, [7, 4, 1, 13, 64, 100]),
    (32, 8, 128, 256, [1500, 0, 3000, 0, 129]),
    (8, 8, 128, 16, [33, 200, 511]),
    (16, 2, 128, 64, [65, 640, 1]),
    (8, 1, 64, 32, [300, 31, 32]),
    (16, 8, 128, 16, [0, 5, 0, 200, 1]),      # one chunk per row, padding rows
    # GQA groups 3, 5, 6, 7 (odd groups and a group that is not a power of two)
    (12, 4, 128, 256, [700, 1, 256, 2500]),
    (10, 2, 64, 16, [90, 333, 0]),
    (12, 2, 128, 32, [64, 1025]),
    (14, 2, 128, 256, [513, 7]),
    # groups above 8, run as sub-groups of 6, 8, 3 and 1 heads (12, 16, 9, 11)
    (24, 2, 128, 16, [300, 0, 1000, 1]),
    (32, 2, 64, 64, [257, 2000]),
    (9, 1, 128, 8, [100, 33]),
    (11, 1, 64, 256, [700, 0, 5]),
]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d_bs{s[3]}")
@pytest.mark.parametrize("chunk_tiles", [None, 1, 3])
def test_decode_vs_oracle(shape, chunk_tiles):
    hq, hkv, d, bs, ctx = shape
    need = sum((c + bs - 1) // bs for c in ctx) + 3
    heads = W.Heads(hq, hkv, d, bs, need)
    with decode_chunk_tiles(chunk_tiles):
        _decode_case(heads, ctx, seed=300 + hq + d + bs)


@pytest.mark.parametrize("bs", [1, 2, 8, 128])
def test_decode_other_block_sizes(bs):
    """Block sizes the decode shapes above leave out: one or two slots per
    TMA box (no swizzle), 8 (the smallest swizzled box) and 128."""
    ctx = [1, bs, bs + 1, 3 * bs + 5, 97, 0]
    need = sum((c + bs - 1) // bs for c in ctx) + 3
    _decode_case(W.Heads(16, 4, 128, bs, need), ctx, seed=340 + bs)


@pytest.mark.parametrize("bs", [512, 1024])
def test_blocks_larger_than_a_tile(bs):
    """Block sizes above the 256 of the pages' engine: a block spans several
    128-key prefill tiles and several decode boxes.  Decode, the fused store +
    decode step and prefix-cache prefill (prefixes ending inside a block and
    on a block edge) against the oracle."""
    from test_gpu_fused import _decode_store_case
    ctx = [1, bs - 1, bs, bs + 1, 2 * bs + 77, 0]
    need = sum((c + bs - 1) // bs for c in ctx) + 2
    _decode_case(W.Heads(16, 8, 128, bs, need), ctx, seed=380 + bs)
    _decode_store_case(W.Heads(16, 4, 64, bs, need), ctx, seed=381 + bs, cache_seed=382 + bs)
    q_lens, prefix = [200, 1, 129, 64], [bs, 3, bs + 300, 0]
    need = sum((q + p + bs - 1) // bs for q, p in zip(q_lens, prefix)) + 2
    _prefill_paged(W.Heads(16, 8, 128, bs, need), q_lens, prefix, seed=383 + bs)


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 128])
def test_prefill_prefix_cache_other_block_sizes(bs):
    """Block sizes 1, 2 and 4 (shorter than the 8-row swizzle atom: tiles
    gathered row by row) next to 8 and 128 (TMA boxes per block), with
    prefixes that end mid-block and NaN in every slot no row reads."""
    heads = W.Heads(16, 8, 128, bs, 96 * 256 // bs)
    _prefill_paged(heads, [100, 257, 7], [bs + 5, 3, 2 * bs], seed=790 + bs)


@pytest.mark.parametrize("bs", [1, 2, 4])
def test_prefill_small_blocks_d64_group4_growing_scores(bs):
    heads = W.Heads(16, 4, 64, bs, 64 * 64 // bs)
    _prefill_paged(heads, [300, 129, 1], [77, 0, 130], seed=820 + bs)
    heads = W.Heads(16, 8, 128, bs, 96 * 64 // bs)
    _prefill_paged(heads, [400, 60], [3 * 128 + 1, 5], seed=830 + bs, growing=True)


def test_decode_tiny_pipeline():
    """Config 'tiny': slot mapping + store of the two prompts, then one decode
    step per sequence (new tokens at positions 6 and 3)."""
    pre, dec = W.tiny()
    h = pre.heads
    kc, vc = W.empty_cache(h)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(pre.block_tables, pre.prefix_lens, pre.cu_seqlens_q, h.block_size)
    oracle.kv_store(bits(pre.k), bits(pre.v), kref, vref, slots)
    dslots = oracle.decode_slots(dec.block_tables, dec.context_lens, h.block_size)
    assert dslots[0] == 38
    oracle.kv_store(bits(dec.k), bits(dec.v), kref, vref, dslots)
    ref, _ = oracle.decode(bits(dec.q), kref, vref, dec.block_tables, dec.context_lens, h.scale)
    ref_pre, _ = oracle.prefill(bits(pre.q), bits(pre.k), bits(pre.v), pre.cu_seqlens_q,
                                pre.cu_seqlens_k, h.scale)

    gk, gv = dev(kc), dev(vc)
    bt = dev(pre.block_tables)
    gs = ops.kv_build_slot_mapping(bt, dev(pre.prefix_lens), dev(pre.cu_seqlens_q), h.block_size)
    ops.kv_store(dev(pre.k), dev(pre.v), gk, gv, gs)
    out_pre = ops.paged_attn_prefill(dev(pre.q), dev(pre.k), dev(pre.v), dev(pre.cu_seqlens_q),
                                     dev(pre.cu_seqlens_k), pre.max_seqlen_q, pre.max_seqlen_k, h.scale)
    gds = ops.kv_build_decode_slots(bt, dev(dec.context_lens), h.block_size)
    ops.kv_store(dev(dec.k), dev(dec.v), gk, gv, gds)
    out = ops.paged_attn_decode(dev(dec.q), gk, gv, bt, dev(dec.context_lens), 7, h.scale)
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy(), slots)
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)
    assert_close(out_pre, ref_pre, "tiny prefill")
    assert_close(out, ref, "tiny decode")


def test_decode_qwen3_full_size():
    """Qwen3-shaped decode, batch 64, contexts U[512, 4096]: every output."""
    work = W.qwen3_decode()
    h = work.heads
    kc, vc = W.history_cache(h, 401)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, h.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, _ = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens, h.scale)
    gk, gv = dev(kc), dev(vc)
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, ops.kv_build_decode_slots(bt, ctx, h.block_size))
    out = ops.paged_attn_decode(dev(work.q), gk, gv, bt, ctx, work.max_context_len, h.scale)
    assert_close(out, ref, "qwen3 decode")


def _compact_blocks(block_tables, rows, lens):
    """For the given rows, the physical blocks they read and a table remapped to
    a compact cache holding only those blocks."""
    bs_rows = block_tables[rows]
    used = sorted({int(b) for r, n in zip(bs_rows.tolist(), lens) for b in r[:n] if b >= 0})
    remap = {b: i for i, b in enumerate(used)}
    table = np.full(bs_rows.shape, -1, np.int32)
    for i, (r, n) in enumerate(zip(bs_rows.tolist(), lens)):
        for j in range(n):
            table[i, j] = remap[r[j]]
    return used, table


def test_decode_large_padded_full_size():
    """Batch 256 + 32 padding rows, GQA group 4, lognormal contexts up to 32k,
    40000-block pool (40 GiB of K/V on the device), in the launch the
    benchmark times: every row and every head against the oracle, on a
    compacted copy of all the blocks the live rows read."""
    work = W.large_decode()
    h = work.heads
    lens = work.context_lens.numpy()
    rows = list(range(work.batch))
    nblk = [int((lens[r] + h.block_size - 1) // h.block_size) for r in rows]
    used, table = _compact_blocks(work.block_tables.numpy(), rows, nblk)
    shape = (h.num_blocks, h.block_size, h.num_kv_heads, h.head_dim)
    gk = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    gv = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    W.fill_normal_(gk, 501)
    W.fill_normal_(gv, 502)
    # the oracle's copy of the history: the seeded values, taken before the
    # CUDA path writes anything
    idx = torch.tensor(used, dtype=torch.long, device="cuda")
    kref, vref = bits(gk[idx]).copy(), bits(gv[idx]).copy()
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    gslots = ops.kv_build_decode_slots(bt, ctx, h.block_size)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, gslots)
    out, lse = ops.paged_attn_decode(dev(work.q), gk, gv, bt, ctx, work.max_context_len, h.scale,
                                     return_lse=True)
    torch.cuda.synchronize()
    del gk, gv, idx
    torch.cuda.empty_cache()
    slots = oracle.decode_slots(table, lens, h.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, ref_lse = oracle.decode(bits(work.q), kref, vref, table, lens, h.scale)
    assert_close(out, ref, "large decode (all rows)")
    got = lse.cpu().double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.allclose(got[fin], ref_lse[fin], atol=2e-3, rtol=1e-4)
    assert out[256:].eq(0).all()


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
def _growing_scores(work, heads, rate=12.0):
    """Make a row's scores rise along the keys: q[..., 0] is 0, 4 or 8 by row
    (all three kinds in every warp) and k[..., 0] grows with the key's position
    among the step's new tokens, so that rows with q[..., 0] = 8 see their
    scores (log2 units of the softmax) rise by about `rate` per 128 keys and
    move the running maximum past any lazy-rescale threshold on most tiles,
    rows with 4 on some tiles, rows with 0 never."""
    per_key = rate / 128 / (8 * heads.scale * math.log2(math.e))
    pos = torch.cat([torch.arange(n) for n in work.q_lens.tolist()]).double()
    work.k[:, :, 0] = (pos * per_key).to(torch.bfloat16)[:, None]
    a = torch.tensor([0.0, 4.0, 8.0], dtype=torch.bfloat16)
    work.q[:, :, 0] = a[torch.arange(work.q.shape[0]) % 3][:, None]


def _prefill_packed(heads, lens, seed, fused=False, growing=False):
    work = W.prefill_work(heads, lens, seed=seed)
    if growing:
        _growing_scores(work, heads)
    ref, ref_lse = oracle.prefill(bits(work.q), bits(work.k), bits(work.v), work.cu_seqlens_q,
                                  work.cu_seqlens_k, heads.scale)
    if fused:
        qkv = dev(torch.cat([work.q.flatten(1), work.k.flatten(1), work.v.flatten(1)], 1))
        qw, kw = heads.num_heads * heads.head_dim, heads.num_kv_heads * heads.head_dim
        n = work.total_q
        q = qkv[:, :qw].view(n, heads.num_heads, heads.head_dim)
        k = qkv[:, qw:qw + kw].view(n, heads.num_kv_heads, heads.head_dim)
        v = qkv[:, qw + kw:].view(n, heads.num_kv_heads, heads.head_dim)
    else:
        q, k, v = dev(work.q), dev(work.k), dev(work.v)
    out, lse = ops.paged_attn_prefill(q, k, v, dev(work.cu_seqlens_q), dev(work.cu_seqlens_k),
                                      work.max_seqlen_q, work.max_seqlen_k, heads.scale,
                                      return_lse=True)
    torch.cuda.synchronize()
    assert_close(out, ref, "prefill out")
    got = lse.cpu().double().numpy()
    assert np.allclose(got, ref_lse, atol=2e-3, rtol=1e-4)


PREFILL_SHAPES = [
    (16, 8, 128, [1, 127, 128, 129, 300, 0, 17]),
    (16, 8, 128, [512]),
    (8, 8, 128, [200, 5]),
    (16, 4, 128, [130, 64]),
    (8, 2, 64, [250, 1, 129]),
]


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d")
def test_prefill_packed_vs_oracle(shape):
    hq, hkv, d, lens = shape
    _prefill_packed(W.Heads(hq, hkv, d, 16, 256), lens, seed=600 + hq + d + len(lens))


def test_prefill_many_sequences():
    """More sequences than the planning kernel keeps on chip (1024): the
    lengths of the rest are read again from cu_seqlens in its second pass;
    short sequences, empty ones among them."""
    g = W.generator(9100)
    lens = torch.randint(0, 6, (1300,), generator=g).tolist()
    lens[1100] = 300
    _prefill_packed(W.Heads(4, 2, 64, 16, 4096), lens, seed=9101)


def test_prefill_fused_qkv_views():
    _prefill_packed(W.Heads(16, 8, 128, 16, 256), [300, 77], seed=650, fused=True)


def _prefill_paged(heads, q_lens, prefix, seed, poison=True, growing=False):
    work = W.prefill_work(heads, q_lens, prefix, seed=seed)
    if growing:
        _growing_scores(work, heads)
    kc, vc = W.history_cache(heads, seed + 1)
    if poison:
        _poison_unused(kc, vc, work.block_tables, work.prefix_lens)   # the chunk is written below
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q,
                                heads.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, ref_lse = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q, work.cu_seqlens_k,
                                  heads.scale, k_cache=kref, v_cache=vref,
                                  block_tables=work.block_tables)
    gk, gv = dev(kc), dev(vc)
    bt = dev(work.block_tables)
    gs = ops.kv_build_slot_mapping(bt, dev(work.prefix_lens), dev(work.cu_seqlens_q),
                                   heads.block_size)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, gs)
    out, lse = ops.paged_attn_prefill(dev(work.q), None, None, dev(work.cu_seqlens_q),
                                      dev(work.cu_seqlens_k), work.max_seqlen_q, work.max_seqlen_k,
                                      heads.scale, k_cache=gk, v_cache=gv, block_tables=bt,
                                      return_lse=True)
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy(), slots)
    assert_close(out, ref, "paged prefill out")
    assert np.allclose(lse.cpu().double().numpy(), ref_lse, atol=2e-3, rtol=1e-4)


def test_prefill_growing_scores_move_the_running_maximum():
    _prefill_packed(W.Heads(16, 8, 128, 16, 256), [700, 300, 129], seed=660, growing=True)


def test_prefill_prefix_cache_growing_scores():
    heads = W.Heads(16, 8, 128, 64, 96 * 4)
    _prefill_paged(heads, [600, 200], [3 * 64, 64 + 5], seed=670, growing=True)


@pytest.mark.parametrize("bs", [16, 64, 256])
def test_prefill_prefix_cache_aligned(bs):
    heads = W.Heads(16, 8, 128, bs, 96 * 256 // bs)
    _prefill_paged(heads, [100, 300, 1, 64], [2 * bs, 0, 3 * bs, bs], seed=700 + bs)


@pytest.mark.parametrize("bs", [4, 16, 256])
def test_prefill_prefix_cache_unaligned(bs):
    heads = W.Heads(16, 8, 128, bs, 96 * 256 // bs)
    _prefill_paged(heads, [100, 257, 7], [bs + 5, 3, 2 * bs + bs - 1], seed=750 + bs)


@pytest.mark.parametrize("hq,hkv,d", [(12, 4, 128), (10, 2, 64), (7, 1, 128)])
def test_prefill_odd_groups(hq, hkv, d):
    """GQA groups 3, 5 and 7: one head per CTA; packed and prefix-cache
    prefill both against the oracle."""
    _prefill_packed(W.Heads(hq, hkv, d, 16, 256), [1, 129, 300, 77], seed=640 + hq)
    heads = W.Heads(hq, hkv, d, 32, 64)
    _prefill_paged(heads, [150, 40], [64 + 3, 0], seed=650 + hq)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (6, 2, 64)])
def test_prefill_one_head_units_long(hq, hkv, d):
    """Groups 1 and 3 (one head per work unit) on long sequences with odd and
    even key-tile counts, packed and prefix-cache, and scores that grow
    along the keys (the running maximum moves late)."""
    _prefill_packed(W.Heads(hq, hkv, d, 16, 256), [1000, 513, 64, 1], seed=680 + hq)
    heads = W.Heads(hq, hkv, d, 64, 96)
    _prefill_paged(heads, [300, 65, 640], [1000, 7, 129], seed=690 + hq)
    _prefill_paged(heads, [200, 640], [900, 0], seed=695 + hq, growing=True)


def test_prefill_packed_blocks_long_prefix():
    """Blocks of at most 64 rows (both heads of a pair in one tile) behind a
    long cached prefix: many key tiles for one packed tile stream."""
    heads = W.Heads(16, 8, 128, 256, 48)
    _prefill_paged(heads, [60, 7, 192 + 33], [2048 + 100, 777, 1500], seed=710)


def test_prefill_paged_group4_d64():
    heads = W.Heads(16, 4, 64, 32, 64)
    _prefill_paged(heads, [90, 200], [40, 0], seed=780)


def _check_lse(lse, ref_lse, what):
    got = lse.cpu().double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got), fin), what
    assert np.allclose(got[fin], ref_lse[fin], atol=2e-3, rtol=1e-4), what


def test_prefill_varlen_full_size():
    """8 prompts of U[128, 4096] tokens (about 19.6k), packed, as the
    benchmark runs them: every output element and every lse against the
    oracle."""
    work = W.varlen_prefill()
    h = work.heads
    out, lse = ops.paged_attn_prefill(dev(work.q), dev(work.k), dev(work.v),
                                      dev(work.cu_seqlens_q), dev(work.cu_seqlens_k),
                                      work.max_seqlen_q, work.max_seqlen_k, h.scale,
                                      return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.prefill(bits(work.q), bits(work.k), bits(work.v), work.cu_seqlens_q,
                                  work.cu_seqlens_k, h.scale)
    assert_close(out, ref, "varlen prefill (all rows)")
    _check_lse(lse, ref_lse, "varlen prefill lse")


def _prefix_full_size(work, seed):
    h = work.heads
    kc, vc = W.history_cache(h, seed)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q,
                                h.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    gk, gv = dev(kc), dev(vc)
    bt = dev(work.block_tables)
    gs = ops.kv_build_slot_mapping(bt, dev(work.prefix_lens), dev(work.cu_seqlens_q), h.block_size)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, gs)
    out, lse = ops.paged_attn_prefill(dev(work.q), None, None, dev(work.cu_seqlens_q),
                                      dev(work.cu_seqlens_k), work.max_seqlen_q, work.max_seqlen_k,
                                      h.scale, k_cache=gk, v_cache=gv, block_tables=bt,
                                      return_lse=True)
    torch.cuda.synchronize()
    assert np.array_equal(gs.cpu().numpy(), slots)
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)
    ref, ref_lse = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q, work.cu_seqlens_k,
                                  h.scale, k_cache=kref, v_cache=vref,
                                  block_tables=work.block_tables)
    return out, lse, ref, ref_lse


def test_prefill_prefix_full_size():
    """16 sequences, cached prefix of U{0..12} blocks of 256 plus a chunk of
    U[64, 1024] tokens read through block_tables, as the benchmark runs
    them: every output element and every lse against the oracle."""
    out, lse, ref, ref_lse = _prefix_full_size(W.prefix_prefill(), 801)
    assert_close(out, ref, "prefix prefill (all rows)")
    _check_lse(lse, ref_lse, "prefix prefill lse")


def test_prefill_unaligned_prefix_full_size():
    """The same with prefixes that end mid-block (256 p + U[1, 255]), so every
    chunk starts mid-block: every output element and every lse."""
    out, lse, ref, ref_lse = _prefix_full_size(W.prefix_prefill(unaligned=True), 811)
    assert_close(out, ref, "unaligned prefix prefill (all rows)")
    _check_lse(lse, ref_lse, "unaligned prefix prefill lse")


def test_prefill_mixed_chunked_full_size():
    """The chunked-prefill mixed batch the benchmark times: 64 decode rows
    (contexts U[512, 4096]) and 4 chunks of 496 tokens behind cached
    prefixes of 512 x U{0..7} in one paged call: every output element and
    every lse against the oracle."""
    out, lse, ref, ref_lse = _prefix_full_size(W.mixed_chunked(), 821)
    assert_close(out, ref, "mixed chunked prefill (all rows)")
    _check_lse(lse, ref_lse, "mixed chunked prefill lse")


def test_empty_inputs_are_no_ops():
    """Zero tokens, zero sequences and a zero batch through every entry point:
    each call returns without error, writes nothing (the caches keep their
    canary bits) and leaves no device status."""
    ops.device_status(clear=True)
    h = W.Heads(16, 8, 128, 16, 8)
    kc = W.fill_normal_(torch.empty((8, 16, 8, 128), dtype=torch.bfloat16, device="cuda"), 990)
    vc = W.fill_normal_(torch.empty_like(kc), 991)
    k0, v0 = kc.clone(), vc.clone()
    bt = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    none_i = torch.zeros(0, dtype=torch.int32, device="cuda")
    rows = lambda n, heads: torch.zeros((n, heads, 128), dtype=torch.bfloat16, device="cuda")
    # slot mapping: no sequences, and sequences with no new tokens
    assert ops.kv_build_slot_mapping(bt, none_i, dev(torch.zeros(1, dtype=torch.int32)), 16).numel() == 0
    bt2 = dev(torch.tensor([[0, 1], [2, 3]], dtype=torch.int32))
    assert ops.kv_build_slot_mapping(bt2, dev(torch.tensor([5, 0], dtype=torch.int32)),
                                     dev(torch.zeros(3, dtype=torch.int32)), 16).numel() == 0
    assert ops.kv_build_decode_slots(bt, none_i, 16).numel() == 0
    ops.kv_store(rows(0, 8), rows(0, 8), kc, vc, none_i)
    pos = torch.zeros(0, dtype=torch.int64, device="cuda")
    w = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    q_out, _ = ops.qk_norm_rope_store(rows(0, 16), rows(0, 8), rows(0, 8), pos, w, w, kc, vc, none_i)
    assert q_out.shape == (0, 16, 128)
    assert ops.paged_attn_decode(rows(0, 16), kc, vc, bt, none_i, 1, h.scale).shape == (0, 16, 128)
    assert ops.paged_attn_decode_store(rows(0, 16), rows(0, 8), rows(0, 8), kc, vc, bt, none_i, 1,
                                       h.scale).shape == (0, 16, 128)
    cu0 = dev(torch.zeros(2, dtype=torch.int32))
    assert ops.paged_attn_prefill(rows(0, 16), rows(0, 8), rows(0, 8), cu0, cu0, 0, 0,
                                  h.scale).shape == (0, 16, 128)
    # cached prefixes and no new tokens, through the block tables
    cuk = dev(torch.tensor([0, 20, 40], dtype=torch.int32))
    assert ops.paged_attn_prefill(rows(0, 16), None, None, dev(torch.zeros(3, dtype=torch.int32)), cuk,
                                  0, 20, h.scale, k_cache=kc, v_cache=vc,
                                  block_tables=bt2).shape == (0, 16, 128)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), v0.view(torch.int16))
    assert ops.device_status(clear=True) == 0


def test_decode_batch_of_padding_rows_only():
    """A CUDA-graph batch whose rows are all padding (context 0, table rows of
    -1): the output is zero, lse is -inf, and the fused step writes nothing."""
    ops.device_status(clear=True)
    kc = W.fill_normal_(torch.empty((8, 16, 8, 128), dtype=torch.bfloat16, device="cuda"), 992)
    vc = W.fill_normal_(torch.empty_like(kc), 993)
    k0, v0 = kc.clone(), vc.clone()
    b = 5
    bt = torch.full((b, 4), -1, dtype=torch.int32, device="cuda")
    ctx = torch.zeros(b, dtype=torch.int32, device="cuda")
    q = W.fill_normal_(torch.empty((b, 16, 128), dtype=torch.bfloat16, device="cuda"), 994)
    kn = W.fill_normal_(torch.empty((b, 8, 128), dtype=torch.bfloat16, device="cuda"), 995)
    for fused in (False, True):
        if fused:
            out, lse = ops.paged_attn_decode_store(q, kn, kn, kc, vc, bt, ctx, 64, 0.125,
                                                   return_lse=True)
        else:
            out, lse = ops.paged_attn_decode(q, kc, vc, bt, ctx, 64, 0.125, return_lse=True)
        torch.cuda.synchronize()
        assert torch.equal(out.float(), torch.zeros_like(out.float()))
        assert bool(torch.isneginf(lse).all())
    assert torch.equal(ops.kv_build_decode_slots(bt, ctx, 16).cpu(), torch.full((b,), -1, dtype=torch.int32))
    assert torch.equal(kc.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), v0.view(torch.int16))
    assert ops.device_status(clear=True) == 0


def test_decode_equals_last_prefill_row_on_gpu():
    """The invariant of the pages (decode step t sees position t) on the CUDA
    path itself: decode over ctx tokens equals the last row of a causal
    prefill over the same tokens, within tolerance."""
    heads = W.Heads(16, 8, 128, 256, 8)
    n = 700
    work = W.prefill_work(heads, [n], seed=900)
    gk, gv = (t.to("cuda") for t in W.empty_cache(heads))
    bt = dev(work.block_tables)
    gs = ops.kv_build_slot_mapping(bt, dev(work.prefix_lens), dev(work.cu_seqlens_q), 256)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, gs)
    full = ops.paged_attn_prefill(dev(work.q), dev(work.k), dev(work.v), dev(work.cu_seqlens_q),
                                  dev(work.cu_seqlens_k), n, n, heads.scale)
    dec = ops.paged_attn_decode(dev(work.q[n - 1:n]), gk, gv, bt, dev(torch.tensor([n], dtype=torch.int32)),
                                n, heads.scale)
    torch.cuda.synchronize()
    assert_close(dec[0], full[n - 1].float().cpu().double().numpy(), "decode vs last prefill row")


def test_validate_mode_reports_bad_table():
    ops.set_validate(True)
    try:
        bt = dev(torch.tensor([[0, -1]], dtype=torch.int32))
        with pytest.raises(ops.PagedKVError) as e:
            ops.kv_build_decode_slots(bt, dev(torch.tensor([6], dtype=torch.int32)), 4)
        assert e.value.code == 5
    finally:
        ops.set_validate(False)


def test_validate_mode_flags_duplicate_slots():
    """Two tokens of one store that write the same slot race (a -1 slot writes
    nothing and is never a duplicate).  Validate mode flags the race with
    PKV_STATUS_DUP_SLOT in kv_store, qk_norm_rope_store and the fused decode
    store, and passes the same calls once the slots are distinct."""
    hkv, d, bs = 2, 128, 4
    g = torch.Generator().manual_seed(77)
    kc = torch.zeros((8, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    key = torch.randn((5, hkv, d), generator=g).to(torch.bfloat16).cuda()
    val = torch.randn((5, hkv, d), generator=g).to(torch.bfloat16).cuda()
    q = torch.randn((5, 4, d), generator=g).to(torch.bfloat16).cuda()
    pos = torch.arange(5, dtype=torch.int64, device="cuda")
    w = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    dup = dev(torch.tensor([3, 9, -1, 3, -1], dtype=torch.int32))
    distinct = dev(torch.tensor([3, 9, -1, 4, -1], dtype=torch.int32))
    ops.set_validate(True)
    try:
        for call in (lambda s: ops.kv_store(key, val, kc, vc, s),
                     lambda s: ops.qk_norm_rope_store(q, key, val, pos, w, w, kc, vc, s)):
            with pytest.raises(ops.PagedKVError) as e:
                call(dup)
            assert e.value.code == 5 and "0x10" in str(e.value), str(e.value)
            call(distinct)
        # decode rows 0 and 2 share a table row and a context length, so
        # their new tokens map to the same slot; row 1 is a padding row
        bt = dev(torch.tensor([[1, 2], [-1, -1], [1, 2]], dtype=torch.int32))
        qd = torch.randn((3, 4, d), generator=g).to(torch.bfloat16).cuda()
        kd, vd = key[:3].contiguous(), val[:3].contiguous()
        ctx = dev(torch.tensor([6, 0, 6], dtype=torch.int32))
        with pytest.raises(ops.PagedKVError) as e:
            ops.paged_attn_decode_store(qd, kd, vd, kc, vc, bt, ctx, 8)
        assert e.value.code == 5 and "0x10" in str(e.value), str(e.value)
        ops.paged_attn_decode_store(qd, kd, vd, kc, vc, bt, dev(torch.tensor([6, 0, 5], dtype=torch.int32)), 8)
    finally:
        ops.set_validate(False)
    assert ops.device_status(clear=True) == 0


def test_decode_step_replayed_as_cuda_graph():
    """The padded decode step (decode slots, kv_store, decode) captured once
    in a CUDA graph and replayed on new inputs gives the eager result."""
    heads = W.Heads(16, 8, 128, 256, 64)
    work = W.decode_work(heads, [300, 0, 1000, 17], seed=950)
    kc, vc = W.history_cache(heads, 951)
    gk, gv = dev(kc), dev(vc)
    q, k, v = dev(work.q), dev(work.k), dev(work.v)
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    slots = torch.empty(work.batch, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(max(1, ops.decode_workspace_size(work.batch, 16, 8, 128, 1000)),
                     dtype=torch.uint8, device="cuda")

    def step():
        ops.kv_build_decode_slots(bt, ctx, 256, out=slots)
        ops.kv_store(k, v, gk, gv, slots)
        ops.paged_attn_decode(q, gk, gv, bt, ctx, 1000, heads.scale, out=out, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    new_q = W.normal_bf16(tuple(q.shape), W.generator(952)).cuda()
    q.copy_(new_q)
    graph.replay()
    torch.cuda.synchronize()
    got = out.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(got, out)
    assert got[1].eq(0).all()


def test_prefill_step_replayed_as_cuda_graph():
    """A prefix-cache step (slot mapping, K/V store, paged prefill: planning
    kernel and prefill kernel, the latter a programmatic dependent) captured
    once in a CUDA graph and replayed twice on new chunks; each replay's
    output against the oracle.  The work list and the claim counter are
    rebuilt by every replay's planning kernel."""
    heads = W.Heads(16, 8, 128, 64, 160)
    q_lens, prefix = [300, 77, 129, 1], [128, 5, 0, 640]
    work = W.prefill_work(heads, q_lens, prefix, seed=970)
    kc, vc = W.history_cache(heads, 971)
    gk, gv = dev(kc), dev(vc)
    q, k, v = dev(work.q), dev(work.k), dev(work.v)
    bt, start = dev(work.block_tables), dev(work.prefix_lens)
    cu_q, cu_k = dev(work.cu_seqlens_q), dev(work.cu_seqlens_k)
    slots = torch.empty(work.total_q, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(ops.prefill_workspace_size(len(q_lens), work.total_q, work.max_seqlen_q, 16),
                     dtype=torch.uint8, device="cuda")

    def step():
        ops.kv_build_slot_mapping(bt, start, cu_q, heads.block_size, out=slots)
        ops.kv_store(k, v, gk, gv, slots)
        ops.paged_attn_prefill(q, None, None, cu_q, cu_k, work.max_seqlen_q, work.max_seqlen_k,
                               heads.scale, k_cache=gk, v_cache=gv, block_tables=bt, out=out,
                               workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    kref, vref = bits(kc).copy(), bits(vc).copy()
    ref_slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q, 64)
    for rep in range(2):
        g = W.generator(980 + rep)
        nq, nk, nv = (W.normal_bf16(tuple(t.shape), g) for t in (work.q, work.k, work.v))
        q.copy_(nq.cuda())
        k.copy_(nk.cuda())
        v.copy_(nv.cuda())
        graph.replay()
        torch.cuda.synchronize()
        oracle.kv_store(bits(nk), bits(nv), kref, vref, ref_slots)
        ref, _ = oracle.prefill(bits(nq), None, None, work.cu_seqlens_q, work.cu_seqlens_k,
                                heads.scale, k_cache=kref, v_cache=vref,
                                block_tables=work.block_tables)
        assert_close(out, ref, f"prefill graph replay {rep}")
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)


def test_mixed_batch_chunks_and_decode_rows_in_one_prefill():
    """Chunked-prefill mixed batch: sequences with a cached prefix and a new
    chunk, and decode rows (one new token over their whole cache), run as one
    paged prefill launch.  A decode row is the Lq = 1 case of the
    bottom-right causal mask, so it must equal the decode kernel too."""
    heads = W.Heads(16, 8, 128, 256, 160)
    q_lens = [200, 1, 77, 1, 1]
    prefix = [512, 999, 0, 3000, 255]
    work = W.prefill_work(heads, q_lens, prefix, seed=960)
    kc, vc = W.history_cache(heads, 961)
    _poison_unused(kc, vc, work.block_tables, work.prefix_lens)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q, 256)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, _ = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q, work.cu_seqlens_k,
                            heads.scale, k_cache=kref, v_cache=vref, block_tables=work.block_tables)
    gk, gv = dev(kc), dev(vc)
    bt = dev(work.block_tables)
    gs = ops.kv_build_slot_mapping(bt, dev(work.prefix_lens), dev(work.cu_seqlens_q), 256)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, gs)
    out = ops.paged_attn_prefill(dev(work.q), None, None, dev(work.cu_seqlens_q),
                                 dev(work.cu_seqlens_k), work.max_seqlen_q, work.max_seqlen_k,
                                 heads.scale, k_cache=gk, v_cache=gv, block_tables=bt)
    torch.cuda.synchronize()
    assert_close(out, ref, "mixed batch")
    # the decode rows through the decode kernel give the same rows
    cu = work.cu_seqlens_q.tolist()
    rows = [cu[i] for i in range(len(q_lens)) if q_lens[i] == 1]
    seqs = [i for i in range(len(q_lens)) if q_lens[i] == 1]
    ctx = torch.tensor([prefix[i] + 1 for i in seqs], dtype=torch.int32)
    dec = ops.paged_attn_decode(dev(work.q[rows]), gk, gv, dev(work.block_tables[seqs].contiguous()),
                                dev(ctx), int(ctx.max()), heads.scale)
    torch.cuda.synchronize()
    assert_close(dec, ref[rows], "decode rows of the mixed batch")
