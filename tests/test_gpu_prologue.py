"""Parity of qk_norm_rope_store (QK-Norm, RoPE and the K/V store in one
launch; L17 §4 then §5.1) with the oracle.

Tolerance, derived from the arithmetic: the RMSNorm of "Nano-VLLM full-code
notes (5)" rounds to bf16 twice (the normalised value, then its product with
the weight) from fp32 values.  The GPU and the oracle (fp64) agree on those
roundings except where the exact value sits within a few fp32 ulps of a bf16
rounding boundary; there one side may land one bf16 ulp away, and RoPE mixes
that input of the pair into both outputs.  So element e of a pair with
magnitude r = sqrt(out_e^2 + out_partner^2) must satisfy
    |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| + 2 * ulp_bf16(r),
and at least 97% of all elements must be bit-identical.  The cache must
hold exactly the k the kernel returned and exactly the input v at every
stored slot, and nothing anywhere else.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_303_gb300 import ops
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits, f64
from test_gpu_parity import assert_close, dev

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_303_gb300 import build
    build.build()
    ops.device_status(clear=True)
    yield
    assert ops.device_status(clear=True) == 0, "a kernel flagged its input"


def _inputs(n, hq, hkv, d, seed, num_slots, pad_every=0, max_pos=32767):
    """Projected q/k/v as views of one fused [N, Hq + 2 Hkv, d] buffer (raw
    projections: N(0, 1) times a per-head scale, not normalised), positions,
    norm weights and a slot mapping (a permutation prefix, some -1)."""
    g = W.generator(seed)
    qkv = (torch.randn((n, hq + 2 * hkv, d), generator=g) *
           torch.empty((1, hq + 2 * hkv, 1)).uniform_(0.2, 4.0, generator=g)).to(torch.bfloat16)
    pos = torch.randint(0, max_pos + 1, (n,), generator=g, dtype=torch.int64)
    if n:
        pos[0] = 0
    qw = torch.empty(d).uniform_(0.5, 1.5, generator=g).to(torch.bfloat16)
    kw = torch.empty(d).uniform_(0.5, 1.5, generator=g).to(torch.bfloat16)
    slots = torch.randperm(num_slots, generator=g)[:n].to(torch.int32)
    if pad_every:
        slots[::pad_every] = -1
    return qkv, pos, qw, kw, slots


def _ulp_bf16(x):
    """spacing of bf16 numbers at magnitude x (8 significant bits)"""
    x = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(x)) - 7)


def assert_rotated_close(gpu: torch.Tensor, ref_bits: np.ndarray, what: str):
    g = gpu.detach().float().cpu().double().numpy()
    ref = f64(ref_bits)
    assert g.shape == ref.shape
    h = ref.shape[-1] // 2
    partner = np.concatenate([ref[..., h:], ref[..., :h]], axis=-1)
    bound = 1e-2 + 1e-2 * np.abs(ref) + 2 * _ulp_bf16(np.hypot(ref, partner))
    err = np.abs(g - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance, "
                             f"max abs {np.nanmax(err):.3e}, first bad {idx}")
    same = float((bits(gpu) == ref_bits).mean())
    print(f"{what}: bit-identical fraction {same:.6f}, max abs {err.max():.3e}")
    assert same > 0.97, same


def _oracle(qkv, pos, qw, kw, hq, hkv, eps, theta):
    q, k = bits(qkv[:, :hq]), bits(qkv[:, hq:hq + hkv])
    return oracle.qk_norm_rope(q, k, pos.numpy(), bits(qw), bits(kw), eps, theta)


def _check_cache(gk, gv, slots, k_rot_bits, v_bits, num_slots):
    """Stored slots hold the rotated k / input v bit for bit; all others
    still hold the NaN canary."""
    hkv, d = gk.shape[2], gk.shape[3]
    ck = bits(gk).reshape(num_slots, hkv, d)
    cv = bits(gv).reshape(num_slots, hkv, d)
    s = slots.numpy()
    live = s >= 0
    assert np.array_equal(ck[s[live]], k_rot_bits[live])
    assert np.array_equal(cv[s[live]], v_bits[live])
    mask = np.ones(num_slots, bool)
    mask[s[live]] = False
    assert np.all(ck[mask] == NAN_BITS) and np.all(cv[mask] == NAN_BITS)


def _canary_cache(num_blocks, bs, hkv, d):
    shape = (num_blocks, bs, hkv, d)
    c = torch.full(shape, 0, dtype=torch.int16, device="cuda")
    c.fill_(NAN_BITS)
    return c.view(torch.bfloat16), c.clone().view(torch.bfloat16)


@pytest.mark.parametrize("hq,hkv,d,n,theta", [(16, 8, 128, 300, 1e6), (4, 2, 64, 77, 1e4),
                                              (32, 8, 128, 129, 1e6), (8, 1, 64, 33, 5e5),
                                              (16, 16, 128, 1, 1e4)])
def test_prologue_vs_oracle(hq, hkv, d, n, theta):
    bs, nb = 16, (n + 40) // 16 + 2
    num_slots = nb * bs
    qkv, pos, qw, kw, slots = _inputs(n, hq, hkv, d, seed=900 + n, num_slots=num_slots, pad_every=7)
    ref_q, ref_k = _oracle(qkv, pos, qw, kw, hq, hkv, 1e-6, theta)
    g = dev(qkv)
    gk, gv = _canary_cache(nb, bs, hkv, d)
    q_out, k_out = ops.qk_norm_rope_store(g[:, :hq], g[:, hq:hq + hkv], g[:, hq + hkv:], dev(pos),
                                          dev(qw), dev(kw), gk, gv, dev(slots), 1e-6, theta,
                                          k_out=torch.empty((n, hkv, d), dtype=torch.bfloat16,
                                                            device="cuda"))
    torch.cuda.synchronize()
    assert_rotated_close(q_out, ref_q, "rotated q")
    assert_rotated_close(k_out, ref_k, "rotated k")
    _check_cache(gk, gv, slots, bits(k_out), bits(qkv[:, hq + hkv:]), num_slots)


@pytest.mark.parametrize("hq,hkv,d,theta", [(16, 8, 128, 1e6), (4, 2, 64, 1e4)])
def test_prologue_large_positions(hq, hkv, d, theta):
    """Positions up to 2^24 - 1 (the largest the fp32 position is exact for):
    angles of up to 1.7e7 rad must still be reduced accurately."""
    n, bs = 200, 16
    nb = (n + 40) // bs + 2
    num_slots = nb * bs
    qkv, pos, qw, kw, slots = _inputs(n, hq, hkv, d, seed=950 + d, num_slots=num_slots,
                                      max_pos=2 ** 24 - 1)
    pos[1] = 2 ** 24 - 1
    ref_q, ref_k = _oracle(qkv, pos, qw, kw, hq, hkv, 1e-6, theta)
    g = dev(qkv)
    gk, gv = _canary_cache(nb, bs, hkv, d)
    q_out, k_out = ops.qk_norm_rope_store(g[:, :hq], g[:, hq:hq + hkv], g[:, hq + hkv:], dev(pos),
                                          dev(qw), dev(kw), gk, gv, dev(slots), 1e-6, theta,
                                          k_out=torch.empty((n, hkv, d), dtype=torch.bfloat16,
                                                            device="cuda"))
    torch.cuda.synchronize()
    assert_rotated_close(q_out, ref_q, "rotated q, large positions")
    assert_rotated_close(k_out, ref_k, "rotated k, large positions")


def test_prologue_in_place_equals_out_of_place():
    hq, hkv, d, n = 16, 8, 128, 200
    num_slots = 16 * 16
    qkv, pos, qw, kw, slots = _inputs(n, hq, hkv, d, seed=950, num_slots=num_slots)
    a = dev(qkv)
    k1, v1 = _canary_cache(16, 16, hkv, d)
    q_out, k_out = ops.qk_norm_rope_store(a[:, :hq], a[:, hq:hq + hkv], a[:, hq + hkv:], dev(pos),
                                          dev(qw), dev(kw), k1, v1, dev(slots),
                                          k_out=torch.empty((n, hkv, d), dtype=torch.bfloat16,
                                                            device="cuda"))
    b = dev(qkv)
    k2, v2 = _canary_cache(16, 16, hkv, d)
    ops.qk_norm_rope_store(b[:, :hq], b[:, hq:hq + hkv], b[:, hq + hkv:], dev(pos), dev(qw), dev(kw),
                           k2, v2, dev(slots), q_out=b[:, :hq], k_out=b[:, hq:hq + hkv])
    torch.cuda.synchronize()
    assert torch.equal(b[:, :hq].view(torch.int16), q_out.view(torch.int16))
    assert torch.equal(b[:, hq:hq + hkv].view(torch.int16), k_out.view(torch.int16))
    assert torch.equal(b[:, hq + hkv:].view(torch.int16), a[:, hq + hkv:].view(torch.int16))
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))


def test_prologue_full_size_varlen_step():
    """The varlen-prefill step's 19576 tokens, Qwen3 heads, positions 0..L-1
    of each prompt: every element against the oracle."""
    work = W.varlen_prefill()
    h = work.heads
    n = work.total_q
    lens = (work.cu_seqlens_q[1:] - work.cu_seqlens_q[:-1]).tolist()
    pos = torch.cat([torch.arange(L, dtype=torch.int64) for L in lens])
    g = W.generator(961)
    qkv = (torch.randn((n, h.num_heads + 2 * h.num_kv_heads, h.head_dim), generator=g) * 2
           ).to(torch.bfloat16)
    qw = torch.empty(h.head_dim).uniform_(0.5, 1.5, generator=g).to(torch.bfloat16)
    kw = torch.empty(h.head_dim).uniform_(0.5, 1.5, generator=g).to(torch.bfloat16)
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q, h.block_size)
    ref_q, ref_k = _oracle(qkv, pos, qw, kw, h.num_heads, h.num_kv_heads, 1e-6, 1e6)
    gq = dev(qkv)
    num_slots = h.num_blocks * h.block_size
    gk, gv = _canary_cache(h.num_blocks, h.block_size, h.num_kv_heads, h.head_dim)
    hq, hkv = h.num_heads, h.num_kv_heads
    q_out, _ = ops.qk_norm_rope_store(gq[:, :hq], gq[:, hq:hq + hkv], gq[:, hq + hkv:], dev(pos),
                                      dev(qw), dev(kw), gk, gv, dev(torch.from_numpy(slots)))
    torch.cuda.synchronize()
    assert_rotated_close(q_out, ref_q, "rotated q, full size")
    cached_k = bits(gk).reshape(num_slots, hkv, h.head_dim)[slots]
    assert_rotated_close(torch.from_numpy(cached_k.view(np.int16)).view(torch.bfloat16), ref_k,
                         "rotated k in the cache, full size")
    _check_cache(gk, gv, torch.from_numpy(slots), cached_k, bits(qkv[:, hq + hkv:]), num_slots)


def test_prologue_then_prefix_prefill_and_decode():
    """Chunked prefill with a cached prefix, then one decode step: the
    prologue writes the chunk's rotated k / v into the cache (positions
    prefix + t), paged prefill and decode read them back; the oracle runs its
    own prologue, scatter and attention on the same raw projections."""
    heads = W.Heads(16, 8, 128, 64, 64)
    q_lens, prefix = [100, 37, 64], [128, 0, 300]
    work = W.prefill_work(heads, q_lens, prefix, seed=970)
    hq, hkv, d = heads.num_heads, heads.num_kv_heads, heads.head_dim
    n = work.total_q
    g = W.generator(971)
    qkv = (torch.randn((n, hq + 2 * hkv, d), generator=g) * 1.5).to(torch.bfloat16)
    qw = torch.empty(d).uniform_(0.5, 1.5, generator=g).to(torch.bfloat16)
    kw = torch.empty(d).uniform_(0.5, 1.5, generator=g).to(torch.bfloat16)
    pos = torch.cat([torch.arange(p, p + c, dtype=torch.int64) for p, c in zip(prefix, q_lens)])
    kc, vc = W.history_cache(heads, 972)
    # oracle: prologue, scatter, paged prefill
    rq, rk = _oracle(qkv, pos, qw, kw, hq, hkv, 1e-6, 1e6)
    kref, vref = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q,
                                heads.block_size)
    oracle.kv_store(rk, bits(qkv[:, hq + hkv:]), kref, vref, slots)
    ref, _ = oracle.prefill(rq, None, None, work.cu_seqlens_q, work.cu_seqlens_k, heads.scale,
                            k_cache=kref, v_cache=vref, block_tables=work.block_tables)
    # GPU: prologue + store in one launch, then paged prefill
    gq = dev(qkv)
    gk, gv = dev(kc), dev(vc)
    bt = dev(work.block_tables)
    gslots = ops.kv_build_slot_mapping(bt, dev(work.prefix_lens), dev(work.cu_seqlens_q),
                                       heads.block_size)
    q_rot, _ = ops.qk_norm_rope_store(gq[:, :hq], gq[:, hq:hq + hkv], gq[:, hq + hkv:], dev(pos),
                                      dev(qw), dev(kw), gk, gv, gslots)
    out = ops.paged_attn_prefill(q_rot, None, None, dev(work.cu_seqlens_q), dev(work.cu_seqlens_k),
                                 work.max_seqlen_q, work.max_seqlen_k, heads.scale,
                                 k_cache=gk, v_cache=gv, block_tables=bt)
    torch.cuda.synchronize()
    assert_close(out, ref, "prologue + prefix prefill")
    # one decode step per sequence at position prefix + q_len
    ctx = torch.tensor([p + c + 1 for p, c in zip(prefix, q_lens)], dtype=torch.int32)
    dq = (torch.randn((3, hq + 2 * hkv, d), generator=g) * 1.5).to(torch.bfloat16)
    dpos = (ctx - 1).to(torch.int64)
    drq, drk = _oracle(dq, dpos, qw, kw, hq, hkv, 1e-6, 1e6)
    dslots = oracle.decode_slots(work.block_tables, ctx, heads.block_size)
    oracle.kv_store(drk, bits(dq[:, hq + hkv:]), kref, vref, dslots)
    dref, _ = oracle.decode(drq, kref, vref, work.block_tables, ctx, heads.scale)
    gd = dev(dq)
    gctx = dev(ctx)
    gds = ops.kv_build_decode_slots(bt, gctx, heads.block_size)
    dq_rot, _ = ops.qk_norm_rope_store(gd[:, :hq], gd[:, hq:hq + hkv], gd[:, hq + hkv:], dev(dpos),
                                       dev(qw), dev(kw), gk, gv, gds)
    dout = ops.paged_attn_decode(dq_rot, gk, gv, bt, gctx, int(ctx.max()), heads.scale)
    torch.cuda.synchronize()
    assert_close(dout, dref, "prologue + decode")


def test_prologue_bad_slot_is_skipped_and_flagged():
    hq, hkv, d, n = 4, 2, 64, 8
    qkv, pos, qw, kw, slots = _inputs(n, hq, hkv, d, seed=980, num_slots=32)
    slots[3] = 32                       # one past the end
    g = dev(qkv)
    gk, gv = _canary_cache(2, 16, hkv, d)
    ops.qk_norm_rope_store(g[:, :hq], g[:, hq:hq + hkv], g[:, hq + hkv:], dev(pos), dev(qw),
                           dev(kw), gk, gv, dev(slots))
    torch.cuda.synchronize()
    assert ops.device_status(clear=True) & 1
    live = torch.cat([slots[:3], slots[4:]]).long()
    mask = torch.ones(32, dtype=torch.bool)
    mask[live] = False
    assert (gk.view(torch.int16).view(32, -1)[mask.cuda()] == NAN_BITS).all()
