"""paged_attn_decode_noalloc: decode for callers that cannot allocate device
memory (for example a plugin inside a host framework that owns every device
allocation, or a runtime that forbids allocations after start-up).  Its split
partials live in a static device array owned by the library instead of a
caller workspace.

The test calls the entry point directly through the C ABI, twice in a row on
different inputs, and compares each result with the regular
paged_attn_decode (caller workspace) and with the CPU oracle, within the
tolerance the other decode tests use.  It also checks that a launch needing more scratch than the array
holds is refused with PKV_ERR_WORKSPACE before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _noalloc(q, kc, vc, bt, ctx, max_ctx, scale, out, lse):
    lib = ops.lib()
    b, hq, d = q.shape
    nb, bs, hkv, _ = kc.shape
    rc = lib.paged_attn_decode_noalloc(
        q.data_ptr(), q.stride(0), kc.data_ptr(), vc.data_ptr(), nb, bt.data_ptr(), bt.stride(0),
        bt.shape[1], ctx.data_ptr(), b, hq, hkv, d, bs, max_ctx, ctypes.c_float(scale),
        out.data_ptr(), out.stride(0), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc, lib.pkv_last_error().decode()


def _close(got: torch.Tensor, ref):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref, np.float64)
    bad = ~(np.abs(g - r) <= TOL + TOL * np.abs(r))
    assert not bad.any(), f"{int(bad.sum())} elements outside tolerance"


def test_noalloc_matches_workspace_decode_twice():
    from paged_kv_cache_303_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    h = W.Heads(16, 8, 128, 256, 512)
    ws_needed = []
    for call, seed in enumerate((1201, 1202)):
        work = W.qwen3_decode(seed=seed, batch=16, num_blocks=512)
        # a padding row rides along, as in a padded decode batch
        ctx = work.context_lens.clone()
        ctx[-1] = 0
        kc = W.fill_normal_(torch.empty((h.num_blocks, 256, 8, 128), dtype=torch.bfloat16,
                                        device="cuda"), seed)
        vc = W.fill_normal_(torch.empty_like(kc), seed + 1)
        q = work.q.cuda()
        bt, dctx = work.block_tables.cuda(), ctx.cuda()
        max_ctx = int(ctx.max())
        need = ops.decode_workspace_size(16, 16, 8, 128, max_ctx)
        # 256 bytes is the chunk counter alone (one split, no partials); more
        # means the split partials, and so the static array, are in use
        assert 256 < need <= 16 << 20
        ws_needed.append(need)
        ref, ref_lse = ops.paged_attn_decode(q, kc, vc, bt, dctx, max_ctx, h.scale, return_lse=True)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((16, 16), float("nan"), dtype=torch.float32, device="cuda")
        rc, msg = _noalloc(q, kc, vc, bt, dctx, max_ctx, h.scale, out, lse)
        torch.cuda.synchronize()
        assert rc == 0, msg
        _close(out, ref)
        oref, _ = oracle.decode(bits(work.q), bits(kc), bits(vc), work.block_tables, ctx, h.scale)
        _close(out, oref)
        fin = torch.isfinite(ref_lse)
        assert torch.equal(torch.isfinite(lse), fin)
        _close(lse[fin], ref_lse[fin])
        assert out[-1].eq(0).all()
    assert ops.device_status(clear=True) == 0


def test_noalloc_refuses_launches_beyond_its_scratch():
    torch.cuda.set_device(0)
    # 288 rows x 32 heads with contexts up to 32k need more split scratch than
    # the static array holds
    b, hq, hkv, d, bs, max_ctx = 288, 32, 8, 128, 256, 32768
    need = ops.decode_workspace_size(b, hq, hkv, d, max_ctx)
    assert need > 16 << 20
    q = torch.zeros((b, hq, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((b, max_ctx // bs), dtype=torch.int32, device="cuda")
    ctx = torch.zeros(b, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((b, hq), dtype=torch.float32, device="cuda")
    rc, msg = _noalloc(q, kc, kc, bt, ctx, max_ctx, 0.1, out, lse)
    assert rc == 3 and "static array" in msg, (rc, msg)
