"""Parity of paged_attn_decode_store (the step's K/V write and the decode in
one launch) with the oracle, and with the unfused kv_build_decode_slots ->
kv_store -> paged_attn_decode sequence: the caches must end bit-identical and
the outputs equal bit for bit (the attention arithmetic is the same kernel's).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits
from test_gpu_parity import DECODE_SHAPES, _poison_unused, assert_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_303_gb300 import build
    build.build()
    ops.device_status(clear=True)
    yield
    assert ops.device_status(clear=True) == 0, "a kernel flagged its input"


def _unfused(work, gk, gv, max_ctx):
    h = work.heads
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    ops.kv_store(dev(work.k), dev(work.v), gk, gv, ops.kv_build_decode_slots(bt, ctx, h.block_size))
    return ops.paged_attn_decode(dev(work.q), gk, gv, bt, ctx, max_ctx, h.scale, return_lse=True)


def _fused(work, gk, gv, max_ctx):
    h = work.heads
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    return ops.paged_attn_decode_store(dev(work.q), dev(work.k), dev(work.v), gk, gv, bt, ctx,
                                       max_ctx, h.scale, return_lse=True)


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d_bs{s[3]}")
@pytest.mark.parametrize("chunk_tiles", [None, 1])
def test_decode_store_vs_oracle_and_unfused(shape, chunk_tiles, request):
    hq, hkv, d, bs, ctx = shape
    if chunk_tiles:
        ops.set_decode_chunk_tiles(chunk_tiles)
        request.addfinalizer(lambda: ops.set_decode_chunk_tiles(0))
    need = sum((c + bs - 1) // bs for c in ctx) + 3
    _decode_store_case(W.Heads(hq, hkv, d, bs, need), ctx, seed=700 + hq + d + bs, cache_seed=701 + bs)


def _decode_store_case(heads, ctx, seed, cache_seed):
    """paged_attn_decode_store against the oracle (outputs, and the cache bit
    for bit with NaN canaries in the unused slots) and against the unfused
    four-launch sequence (outputs bit for bit)."""
    work = W.decode_work(heads, ctx, seed=seed)
    kc, vc = W.history_cache(heads, cache_seed)
    _poison_unused(kc, vc, work.block_tables, work.context_lens)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, heads.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, ref_lse = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens,
                                 heads.scale, nthreads=0)
    max_ctx = max(1, work.max_context_len)
    gk1, gv1 = dev(kc), dev(vc)
    out1, lse1 = _unfused(work, gk1, gv1, max_ctx)
    gk2, gv2 = dev(kc), dev(vc)
    out2, lse2 = _fused(work, gk2, gv2, max_ctx)
    torch.cuda.synchronize()
    # the cache: what the oracle's scatter wrote, NaN canaries untouched
    assert np.array_equal(bits(gk2), kref) and np.array_equal(bits(gv2), vref)
    assert_close(out2, ref, "fused decode out")
    fin = np.isfinite(ref_lse)
    got = lse2.cpu().double().numpy()
    assert np.array_equal(np.isfinite(got), fin)
    assert np.allclose(got[fin], ref_lse[fin], atol=2e-3, rtol=1e-4)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_decode_store_qwen3_full_size():
    """Batch 64, contexts U[512, 4096], 2048-block pool: every output against
    the oracle, cache and outputs against the unfused sequence."""
    work = W.qwen3_decode()
    h = work.heads
    kc, vc = W.history_cache(h, 401)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, h.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, _ = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens, h.scale)
    gk1, gv1 = dev(kc), dev(vc)
    out1, lse1 = _unfused(work, gk1, gv1, work.max_context_len)
    del gk1, gv1
    gk2, gv2 = dev(kc), dev(vc)
    out2, lse2 = _fused(work, gk2, gv2, work.max_context_len)
    torch.cuda.synchronize()
    assert np.array_equal(bits(gk2), kref) and np.array_equal(bits(gv2), vref)
    assert_close(out2, ref, "qwen3 fused decode")
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_decode_store_large_padded():
    """Batch 256 + 32 padding rows, GQA group 4, contexts up to 32k, 40000-block
    pool.  The unfused sequence runs first; the new tokens' slots are then
    overwritten with NaN and the fused call must write them back and return
    the same outputs bit for bit (padding rows: zero output)."""
    work = W.large_decode()
    h = work.heads
    shape = (h.num_blocks, h.block_size, h.num_kv_heads, h.head_dim)
    gk = W.fill_normal_(torch.empty(shape, dtype=torch.bfloat16, device="cuda"), 601)
    gv = W.fill_normal_(torch.empty(shape, dtype=torch.bfloat16, device="cuda"), 602)
    out1, lse1 = _unfused(work, gk, gv, work.max_context_len)
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    slots = ops.kv_build_decode_slots(bt, ctx, h.block_size).long()
    live = slots[slots >= 0]
    fk, fv = gk.view(-1, h.num_kv_heads, h.head_dim), gv.view(-1, h.num_kv_heads, h.head_dim)
    fk[live] = float("nan")
    fv[live] = float("nan")
    out2, lse2 = _fused(work, gk, gv, work.max_context_len)
    torch.cuda.synchronize()
    rows = (slots >= 0).nonzero().flatten()
    assert torch.equal(fk[live].view(torch.int16), dev(work.k)[rows].view(torch.int16))
    assert torch.equal(fv[live].view(torch.int16), dev(work.v)[rows].view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    assert out2[256:].eq(0).all()
    del gk, gv, fk, fv
    torch.cuda.empty_cache()


def test_decode_store_consecutive_steps():
    """Three decode steps in a row, each fused call writing position ctx-1 and
    attending over it; the oracle replays the same steps with its own scatter."""
    heads = W.Heads(16, 8, 128, 16, 64)
    ctx0 = [5, 16, 31, 100]
    kc, vc = W.history_cache(heads, 77)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    gk, gv = dev(kc), dev(vc)
    base = W.decode_work(heads, [c + 3 for c in ctx0], seed=78)
    for step in range(3):
        lens = torch.tensor([c + step for c in ctx0], dtype=torch.int32)
        work = W.decode_work(heads, lens.tolist(), seed=80 + step)
        work = W.DecodeWork(heads, lens, base.block_tables, work.q, work.k, work.v, work.seed, "")
        slots = oracle.decode_slots(work.block_tables, lens, heads.block_size)
        oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
        ref, _ = oracle.decode(bits(work.q), kref, vref, work.block_tables, lens, heads.scale)
        out, _ = _fused(work, gk, gv, max(lens.tolist()))
        torch.cuda.synchronize()
        assert_close(out, ref, f"step {step}")
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)


def test_decode_store_step_replayed_as_cuda_graph():
    """The fused step (one decode launch plus the chunk merge) captured once and
    replayed over new inputs copied into the same buffers."""
    work = W.qwen3_decode()
    h = work.heads
    kc, vc = W.history_cache(h, 411)
    gk, gv = dev(kc), dev(vc)
    q, k, v = dev(work.q), dev(work.k), dev(work.v)
    bt, ctx = dev(work.block_tables), dev(work.context_lens)
    out = torch.empty_like(q)
    ws = torch.empty(max(1, ops.decode_workspace_size(work.batch, h.num_heads, h.num_kv_heads,
                                                      h.head_dim, work.max_context_len)),
                     dtype=torch.uint8, device="cuda")

    def step():
        ops.paged_attn_decode_store(q, k, v, gk, gv, bt, ctx, work.max_context_len, h.scale,
                                    out=out, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    g = W.generator(412)
    nq = W.normal_bf16(tuple(q.shape), g)
    nk = W.normal_bf16(tuple(k.shape), g)
    nv = W.normal_bf16(tuple(v.shape), g)
    q.copy_(nq)
    k.copy_(nk)
    v.copy_(nv)
    graph.replay()
    torch.cuda.synchronize()
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, h.block_size)
    oracle.kv_store(bits(nk), bits(nv), kref, vref, slots)
    ref, _ = oracle.decode(bits(nq), kref, vref, work.block_tables, work.context_lens, h.scale)
    assert_close(out, ref, "graph-replayed fused decode")
    assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)


@pytest.mark.parametrize("fused", [False, True])
def test_chunk_merge_with_dirty_workspace_twice(fused, request):
    """Chunks of 32 keys (up to 64 per sequence), a workspace full of 0xFF
    bytes and two calls in a row on it: the chunk counters and partials must
    not depend on what the workspace held before."""
    ops.set_decode_chunk_tiles(1)
    request.addfinalizer(lambda: ops.set_decode_chunk_tiles(0))
    heads = W.Heads(16, 8, 128, 64, 128)
    ctx = [1, 31, 32, 33, 64, 65, 1000, 2047, 2048, 0, 7]
    work = W.decode_work(heads, ctx, seed=880)
    kc, vc = W.history_cache(heads, 881)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.decode_slots(work.block_tables, work.context_lens, heads.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, ref_lse = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens,
                                 heads.scale)
    gk, gv = dev(kc), dev(vc)
    bt, gctx = dev(work.block_tables), dev(work.context_lens)
    max_ctx = work.max_context_len
    need = ops.decode_workspace_size(work.batch, heads.num_heads, heads.num_kv_heads,
                                     heads.head_dim, max_ctx)
    assert need > 0
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        if fused:
            out, lse = ops.paged_attn_decode_store(dev(work.q), dev(work.k), dev(work.v), gk, gv, bt,
                                                   gctx, max_ctx, heads.scale, workspace=ws,
                                                   return_lse=True)
        else:
            ops.kv_store(dev(work.k), dev(work.v), gk, gv,
                         ops.kv_build_decode_slots(bt, gctx, heads.block_size))
            out, lse = ops.paged_attn_decode(dev(work.q), gk, gv, bt, gctx, max_ctx, heads.scale,
                                             workspace=ws, return_lse=True)
        torch.cuda.synchronize()
        assert_close(out, ref, "decode with 1-tile chunks")
        fin = np.isfinite(ref_lse)
        got = lse.cpu().double().numpy()
        assert np.array_equal(np.isfinite(got), fin)
        assert np.allclose(got[fin], ref_lse[fin], atol=2e-3, rtol=1e-4)
        outs.append(out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_pipelined_end_to_end_steps_read_back_the_decode_output():
    """The benchmark's end-to-end decode: two buffer sets on one cache, with
    the host-to-device copies, the graph replays and the read-backs on three
    streams.  Every step has the same inputs (the same new row is rewritten),
    so each read-back must hold the oracle's output for the cache the step
    read; the second buffer set shares the cache and not the inputs."""
    import bench
    work = W.decode_work(W.Heads(16, 8, 128, 16, 256), [40, 0, 300, 17, 129], seed=431)
    h = work.heads
    st = bench.DecodeStep(work, cache_seed=432, fused=True)
    kref, vref = bits(st.kc.cpu()).copy(), bits(st.vc.cpu()).copy()   # before any step
    slots = oracle.decode_slots(work.block_tables, work.context_lens, h.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kref, vref, slots)
    ref, _ = oracle.decode(bits(work.q), kref, vref, work.block_tables, work.context_lens, h.scale)
    graph = st.capture()
    _, h2d, d2h, out_host = bench.e2e_decode(st, graph, steps=5, warmup=2, world=1)
    torch.cuda.synchronize()
    assert h2d == st.inputs_host.numel() and d2h == st.out.numel() * st.out.element_size()
    for b, oh in enumerate(out_host):
        assert_close(oh, ref, f"read-back of buffer set {b}")
        assert torch.equal(oh, st.out.cpu())
    tw = st.twin()
    assert tw.kc.data_ptr() == st.kc.data_ptr() and tw.inputs.data_ptr() != st.inputs.data_ptr()


def test_prefill_and_decode_store_on_two_streams_at_once():
    """A packed prefill and a fused decode step launched on two streams,
    where they can run at the same time, three rounds: when both persistent
    grids share the SMs, each claims only its own work, and both outputs
    match the oracle."""
    from paged_kv_cache_303_gb300 import workloads as W
    ph = W.Heads(16, 8, 128, 16, 256)
    pw = W.prefill_work(ph, [700, 129, 64, 1000], seed=990)
    pref, _ = oracle.prefill(bits(pw.q), bits(pw.k), bits(pw.v), pw.cu_seqlens_q, pw.cu_seqlens_k,
                             ph.scale)
    dh = W.Heads(16, 8, 128, 64, 256)
    dw = W.decode_work(dh, [3000, 1, 0, 2000, 777, 4000], seed=991)
    kc, vc = W.history_cache(dh, 992)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    dslots = oracle.decode_slots(dw.block_tables, dw.context_lens, dh.block_size)
    oracle.kv_store(bits(dw.k), bits(dw.v), kref, vref, dslots)
    dref, _ = oracle.decode(bits(dw.q), kref, vref, dw.block_tables, dw.context_lens, dh.scale,
                            nthreads=0)
    pq, pk, pv = dev(pw.q), dev(pw.k), dev(pw.v)
    cu_q, cu_k = dev(pw.cu_seqlens_q), dev(pw.cu_seqlens_k)
    dq, dk, dv = dev(dw.q), dev(dw.k), dev(dw.v)
    bt, ctx = dev(dw.block_tables), dev(dw.context_lens)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        gk, gv = dev(kc), dev(vc)
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            pout = ops.paged_attn_prefill(pq, pk, pv, cu_q, cu_k, pw.max_seqlen_q, pw.max_seqlen_k,
                                          ph.scale)
        with torch.cuda.stream(s2):
            dout = ops.paged_attn_decode_store(dq, dk, dv, gk, gv, bt, ctx, dw.max_context_len,
                                               dh.scale)
        torch.cuda.synchronize()
        assert_close(pout, pref, "prefill beside a decode")
        assert_close(dout, dref, "decode beside a prefill")
        assert np.array_equal(bits(gk), kref) and np.array_equal(bits(gv), vref)
