"""A bounded device wait that runs out ends the kernel with an error status,
and the CUDA context stays usable.

Every mbarrier wait in the library's kernels gives up after a bounded number
of cycles, raises PKV_STATUS_TIMEOUT in the device status word and lets the
kernel's roles leave (each role polls a shared abort flag while it waits, and
the TMA producer waits for its own copies in flight before it leaves).  The
product bound is about a second; this test uses a test-only build of the
library (never the product library) with a bound of 2^22 cycles and a hook
that makes every decode CTA's producer withhold its arrival on the first
item's "ready" barrier.  Only that barrier is starved, and no bulk copy is
ever pending on it: the producer's tile copies of the item are issued and
land as usual, and it drains them before the CTA ends.  So the wait runs
out, the call reports PKV_ERR_DEVICE_TIMEOUT in validate mode, and the next
call on the same context, with the hook off, matches the oracle.

The persistent prefill kernel has a second hook: the scheduler of CTA 0
publishes no unit, so that CTA's producer, MMA issuer and softmax
warpgroups wait on the first unit record until the bound runs out (one of
them raises the CTA's abort flag, the others see it and leave).  Nothing
was issued in that CTA, so nothing is in flight when it releases its tensor
memory; the other CTAs claim and finish the remaining units as usual.  It
is run for each producer: TMA from packed keys, TMA through block tables,
and the cp.async row copy of blocks shorter than 8 rows.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits, from_bits
from test_gpu_parity import assert_close, dev

pytestmark = pytest.mark.gpu

PKV_ERR_DEVICE_TIMEOUT = 6


@pytest.fixture(scope="module")
def shortwait():
    from paged_kv_cache_303_gb300 import build
    path = build.build_test_variant("shortwait", ["PKV_TEST_HOOKS=1", "PKV_WAIT_CYCLES=(1ll<<22)"])
    lib = ctypes.CDLL(str(path))
    for name, (args, res) in ops.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    for hook in ("pkv_test_withhold_decode_ready", "pkv_test_withhold_prefill_unit"):
        getattr(lib, hook).argtypes = [ctypes.c_int]
        getattr(lib, hook).restype = ctypes.c_int
    yield lib
    lib.pkv_test_withhold_decode_ready(0)
    lib.pkv_test_withhold_prefill_unit(0)
    lib.pkv_set_validate(0)


def _decode(lib, q, kc, vc, bt, ctx, max_ctx, scale, out, ws):
    b, hq, d = q.shape
    nb, bs, hkv, _ = kc.shape
    rc = lib.paged_attn_decode(q.data_ptr(), q.stride(0), kc.data_ptr(), vc.data_ptr(), nb,
                               bt.data_ptr(), bt.stride(0), bt.shape[1], ctx.data_ptr(), b, hq, hkv,
                               d, bs, max_ctx, scale, out.data_ptr(), out.stride(0), None,
                               ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    return rc, lib.pkv_last_error().decode()


def test_decode_wait_that_runs_out_reports_timeout_and_leaves(shortwait):
    lib = shortwait
    heads = W.Heads(16, 8, 128, 256, 64)
    ctx = [1000, 2000, 700, 3000]
    work = W.decode_work(heads, ctx, seed=990)
    kc, vc = W.history_cache(heads, 991)
    ref, _ = oracle.decode(bits(work.q), bits(kc), bits(vc), work.block_tables, work.context_lens,
                           heads.scale)
    q, gk, gv = dev(work.q), dev(kc), dev(vc)
    bt, gctx = dev(work.block_tables), dev(work.context_lens)
    max_ctx = work.max_context_len
    need = lib.paged_attn_decode_workspace_size(work.batch, heads.num_heads, heads.num_kv_heads,
                                                heads.head_dim, max_ctx)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    lib.pkv_set_validate(1)
    try:
        assert lib.pkv_test_withhold_decode_ready(1) == 0
        t0 = time.perf_counter()
        rc, msg = _decode(lib, q, gk, gv, bt, gctx, max_ctx, heads.scale, out, ws)
        took = time.perf_counter() - t0
        assert rc == PKV_ERR_DEVICE_TIMEOUT, (rc, msg)
        assert "bounded device wait" in msg, msg
        assert took < 30.0, took
        # the context is still usable: the same call without the hook is right
        assert lib.pkv_test_withhold_decode_ready(0) == 0
        rc, msg = _decode(lib, q, gk, gv, bt, gctx, max_ctx, heads.scale, out, ws)
        assert rc == 0, msg
    finally:
        lib.pkv_test_withhold_decode_ready(0)
        lib.pkv_set_validate(0)
    torch.cuda.synchronize()
    assert_close(out, ref, "decode after a timed-out call")
    st = ctypes.c_uint32(0)
    assert lib.pkv_device_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(st), 1) == 0
    assert st.value == 0


def _prefill(lib, work, heads, q, k, v, kc, vc, bt, out):
    """paged_attn_prefill through the given library (k/v packed, or None
    with kc/vc/bt paged)."""
    total_q = work.total_q
    hq, hkv, d = heads.num_heads, heads.num_kv_heads, heads.head_dim
    num_seqs = len(work.cu_seqlens_q) - 1
    cu_q, cu_k = dev(work.cu_seqlens_q), dev(work.cu_seqlens_k)
    need = lib.paged_attn_prefill_workspace_size(num_seqs, total_q, work.max_seqlen_q, hq)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    if bt is None:
        args = (q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0), v.data_ptr(), v.stride(0),
                None, None, 0, None, 0, 0)
        total_k, bs = k.shape[0], 0
    else:
        args = (q.data_ptr(), q.stride(0), None, 0, None, 0, kc.data_ptr(), vc.data_ptr(),
                kc.shape[0], bt.data_ptr(), bt.stride(0), bt.shape[1])
        total_k, bs = 0, kc.shape[1]
    rc = lib.paged_attn_prefill(*args, cu_q.data_ptr(), cu_k.data_ptr(), work.max_seqlen_q,
                                work.max_seqlen_k, num_seqs, total_q, total_k, hq, hkv, d, bs,
                                heads.scale, out.data_ptr(), out.stride(0), None, ws.data_ptr(),
                                ws.numel(), torch.cuda.current_stream().cuda_stream)
    return rc, lib.pkv_last_error().decode()


@pytest.mark.parametrize("mode", ["packed", "paged16", "paged4"])
def test_prefill_wait_that_runs_out_reports_timeout_and_leaves(shortwait, mode):
    lib = shortwait
    bs = {"packed": 16, "paged16": 16, "paged4": 4}[mode]
    heads = W.Heads(16, 8, 128, bs, 512)
    q_lens, prefix = [300, 129, 64, 500], [0, 200, 37, 0]
    if mode == "packed":
        work = W.prefill_work(heads, q_lens, seed=992)
        ref, _ = oracle.prefill(bits(work.q), bits(work.k), bits(work.v), work.cu_seqlens_q,
                                work.cu_seqlens_k, heads.scale)
        q, k, v = dev(work.q), dev(work.k), dev(work.v)
        kc = vc = bt = None
    else:
        work = W.prefill_work(heads, q_lens, prefix, seed=993)
        kc_h, vc_h = W.history_cache(heads, 994)
        kref, vref = bits(kc_h).copy(), bits(vc_h).copy()
        slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q, bs)
        oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
        ref, _ = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q, work.cu_seqlens_k,
                                heads.scale, k_cache=kref, v_cache=vref,
                                block_tables=work.block_tables)
        q, k, v = dev(work.q), None, None
        kc, vc = dev(from_bits(kref)), dev(from_bits(vref))
        bt = dev(work.block_tables)
    out = torch.empty_like(q)
    lib.pkv_set_validate(1)
    try:
        assert lib.pkv_test_withhold_prefill_unit(1) == 0
        t0 = time.perf_counter()
        rc, msg = _prefill(lib, work, heads, q, k, v, kc, vc, bt, out)
        took = time.perf_counter() - t0
        assert rc == PKV_ERR_DEVICE_TIMEOUT, (rc, msg)
        assert "bounded device wait" in msg, msg
        assert took < 30.0, took
        assert lib.pkv_test_withhold_prefill_unit(0) == 0
        rc, msg = _prefill(lib, work, heads, q, k, v, kc, vc, bt, out)
        assert rc == 0, msg
    finally:
        lib.pkv_test_withhold_prefill_unit(0)
        lib.pkv_set_validate(0)
    torch.cuda.synchronize()
    assert_close(out, ref, f"prefill ({mode}) after a timed-out call")
    st = ctypes.c_uint32(0)
    assert lib.pkv_device_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(st), 1) == 0
    assert st.value == 0
