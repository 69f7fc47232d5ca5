"""Guard bands around the attention outputs, and device-side length checks.

Every output is written through a strided view into a larger buffer filled
with a NaN canary: a row of padding before and after the rows, and 64 extra
elements after each row.  After the call the canary must be intact, and the
rows themselves must match the oracle.  The lse outputs get canary elements
past their end.  Lengths that only the device can see (a context length
above the declared maximum, fewer keys than queries) must never cause an
out-of-bounds access: they are clamped or skipped and flagged, which
validate mode reports as PKV_ERR_DEVICE_CHECK.
"""
import re

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits
from test_gpu_parity import _poison_unused, assert_close, dev

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FC1
PAD = 64            # extra elements after each output row


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_303_gb300 import build
    build.build()
    ops.device_status(clear=True)
    yield
    ops.device_status(clear=True)


def _guarded_out(rows, heads, d, shift=0):
    """(buffer, view): the view is [rows, heads, d] at row 1 of a canary-filled
    buffer whose rows are heads*d + PAD elements long, starting `shift`
    elements into the row (8: rows 16-byte but not 32-byte aligned)."""
    width = heads * d + PAD
    buf = torch.full((rows + 2, width), NAN_BITS, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    view = buf[1:rows + 1, shift:shift + heads * d].view(rows, heads, d)
    assert view.stride(0) == width
    return buf, view


def _guarded_lse(rows, heads):
    buf = torch.full((rows * heads + PAD,), float("nan"), dtype=torch.float32, device="cuda")
    return buf, buf[:rows * heads].view(rows, heads)


def _canary_intact(buf, rows, heads, d, shift=0):
    b = buf.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(b[0] == NAN_BITS) and np.all(b[rows + 1] == NAN_BITS), "pad rows written"
    assert np.all(b[1:rows + 1, :shift] == NAN_BITS), "row gaps written"
    assert np.all(b[1:rows + 1, shift + heads * d:] == NAN_BITS), "row gaps written"


def _status_of(err) -> int:
    m = re.search(r"status 0x([0-9a-f]+)", str(err))
    assert m, str(err)
    return int(m.group(1), 16)


def _lse_canary_intact(buf, rows, heads):
    assert torch.isnan(buf[rows * heads:]).all(), "elements past the lse written"


@pytest.mark.parametrize("shift", [0, 8], ids=["aligned32", "aligned16"])
@pytest.mark.parametrize("paged", [False, True])
def test_prefill_writes_only_its_rows(paged, shift):
    """Output rows 32-byte aligned (32-byte stores) and only 16-byte aligned
    (16-byte stores)."""
    heads = W.Heads(16, 8, 128, 64, 96)
    lens, prefix = [1, 129, 300, 64], ([0, 70, 128, 5] if paged else None)
    work = W.prefill_work(heads, lens, prefix, seed=910 + paged)
    n = work.total_q
    obuf, out = _guarded_out(n, heads.num_heads, heads.head_dim, shift)
    lbuf, lse = _guarded_lse(n, heads.num_heads)
    if paged:
        kc, vc = W.history_cache(heads, 911)
        _poison_unused(kc, vc, work.block_tables, work.prefix_lens)
        kref, vref = bits(kc).copy(), bits(vc).copy()
        slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q,
                                    heads.block_size)
        oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
        ref, ref_lse = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q,
                                      work.cu_seqlens_k, heads.scale, k_cache=kref, v_cache=vref,
                                      block_tables=work.block_tables)
        gk, gv = dev(kc), dev(vc)
        bt = dev(work.block_tables)
        gs = ops.kv_build_slot_mapping(bt, dev(work.prefix_lens), dev(work.cu_seqlens_q),
                                       heads.block_size)
        ops.kv_store(dev(work.k), dev(work.v), gk, gv, gs)
        ops.paged_attn_prefill(dev(work.q), None, None, dev(work.cu_seqlens_q),
                               dev(work.cu_seqlens_k), work.max_seqlen_q, work.max_seqlen_k,
                               heads.scale, k_cache=gk, v_cache=gv, block_tables=bt, out=out,
                               lse=lse)
    else:
        ref, ref_lse = oracle.prefill(bits(work.q), bits(work.k), bits(work.v), work.cu_seqlens_q,
                                      work.cu_seqlens_k, heads.scale)
        ops.paged_attn_prefill(dev(work.q), dev(work.k), dev(work.v), dev(work.cu_seqlens_q),
                               dev(work.cu_seqlens_k), work.max_seqlen_q, work.max_seqlen_k,
                               heads.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    _canary_intact(obuf, n, heads.num_heads, heads.head_dim, shift)
    _lse_canary_intact(lbuf, n, heads.num_heads)
    assert_close(out, ref, "prefill rows inside the guard bands")
    assert np.allclose(lse.cpu().double().numpy(), ref_lse, atol=2e-3, rtol=1e-4)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("ctx", [[5, 0, 700, 3000], [40, 7, 1]], ids=["split", "one-chunk"])
def test_decode_writes_only_its_rows(fused, ctx):
    heads = W.Heads(16, 8, 128, 64, 64)
    work = W.decode_work(heads, ctx, seed=920 + len(ctx) + fused)
    kc, vc = W.history_cache(heads, 921)
    _poison_unused(kc, vc, work.block_tables, work.context_lens)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, heads.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, ref_lse = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens,
                                 heads.scale)
    b = work.batch
    obuf, out = _guarded_out(b, heads.num_heads, heads.head_dim)
    lbuf, lse = _guarded_lse(b, heads.num_heads)
    gk, gv = dev(kc), dev(vc)
    bt, gctx = dev(work.block_tables), dev(work.context_lens)
    max_ctx = max(1, work.max_context_len)
    if fused:
        ops.paged_attn_decode_store(dev(work.q), dev(work.k), dev(work.v), gk, gv, bt, gctx,
                                    max_ctx, heads.scale, out=out, lse=lse)
    else:
        ops.kv_store(dev(work.k), dev(work.v), gk, gv,
                     ops.kv_build_decode_slots(bt, gctx, heads.block_size))
        ops.paged_attn_decode(dev(work.q), gk, gv, bt, gctx, max_ctx, heads.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    _canary_intact(obuf, b, heads.num_heads, heads.head_dim)
    _lse_canary_intact(lbuf, b, heads.num_heads)
    assert_close(out, ref, "decode rows inside the guard bands")
    fin = np.isfinite(ref_lse)
    got = lse.cpu().double().numpy()
    assert np.array_equal(np.isfinite(got), fin)
    assert np.allclose(got[fin], ref_lse[fin], atol=2e-3, rtol=1e-4)
    # the caches: exactly the oracle's bytes (the new rows, and NaN elsewhere)
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)


def test_context_above_the_declared_maximum_is_flagged():
    """A context length above max_context_len is clamped to it (no read past
    the table the host sized) and flagged."""
    heads = W.Heads(8, 4, 128, 64, 16)
    work = W.decode_work(heads, [100, 64], seed=930)
    kc, vc = W.history_cache(heads, 931)
    gk, gv = dev(kc), dev(vc)
    bt = dev(work.block_tables)
    ctx = dev(torch.tensor([100, 5000], dtype=torch.int32))      # row 1 claims 5000 tokens
    ops.set_validate(True)
    try:
        with pytest.raises(ops.PagedKVError) as e:
            ops.paged_attn_decode(dev(work.q), gk, gv, bt, ctx, 128, heads.scale)
        # BAD_LENGTH; the clamped range also reaches the row's missing second
        # block (BAD_BLOCK)
        assert e.value.code == 5 and _status_of(e.value) & ops.PKV_STATUS_BAD_LENGTH, str(e.value)
    finally:
        ops.set_validate(False)
    assert ops.device_status(clear=True) == 0


def test_fewer_keys_than_queries_is_flagged():
    """cu_seqlens_k giving a sequence fewer keys than queries is invalid: the
    planner skips the sequence and flags it."""
    heads = W.Heads(8, 4, 128, 16, 64)
    work = W.prefill_work(heads, [50, 20], seed=940)
    cu_k = dev(torch.tensor([0, 50, 60], dtype=torch.int32))       # sequence 1: 10 keys, 20 queries
    ops.set_validate(True)
    try:
        with pytest.raises(ops.PagedKVError) as e:
            ops.paged_attn_prefill(dev(work.q), dev(work.k), dev(work.v), dev(work.cu_seqlens_q),
                                   cu_k, work.max_seqlen_q, 50, heads.scale)
        assert e.value.code == 5 and _status_of(e.value) & ops.PKV_STATUS_BAD_LENGTH, str(e.value)
    finally:
        ops.set_validate(False)
    assert ops.device_status(clear=True) == 0
