"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here touches the CUDA path.  Each pin is chosen so that a plausible
slip in the oracle (a dropped term, a wrong sign or index, a transposed
operand, an off-by-one in the causal bound, the wrong GQA grouping) fails at
least one of them:

* values the pages print (golden fixtures, each with its citation);
* closed forms (single key, identical keys, zero query, dominant key);
* special cases that reduce to a library routine (torch's fp64
  scaled_dot_product_attention on contiguous, unpaged inputs);
* invariants (two statements of slot_mapping agree; physical block order is
  irrelevant; decode equals the last prefill row; prefix prefill equals the
  tail of a full prefill; GQA equals MHA with repeated kv heads; split-K
  merging equals the unsplit result).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_303_gb300 import workloads as W
from _util import bits, bf16_bits_of, f64, golden

pytestmark = pytest.mark.filterwarnings("ignore")


# ---------------------------------------------------------------------------
# printed worked examples
# ---------------------------------------------------------------------------
def test_t1_scatter_toy():
    g = golden("t1_scatter_toy.json")
    src = bf16_bits_of(g["src"]).reshape(3, 1, 4)
    kc = np.zeros((3, 1, 1, 4), dtype=np.uint16)
    vc = np.zeros_like(kc)
    oracle.kv_store(src, src, kc, vc, g["slot"])
    assert np.array_equal(f64(kc.reshape(3, 4)), np.array(g["dst"], dtype=np.float64))


def test_t2_store_kvcache_with_skip():
    g = golden("t2_store_kvcache.json")
    key = bf16_bits_of(g["key"])
    value = bf16_bits_of(np.array(g["key"]) + g["value_offset"])
    kc = np.zeros((1, 4, 2, 2), dtype=np.uint16)
    vc = np.zeros_like(kc)
    oracle.kv_store(key, value, kc, vc, g["slot_mapping"])
    assert np.array_equal(f64(kc.reshape(4, 4)), np.array(g["k_cache_rows"], dtype=np.float64))
    assert np.array_equal(f64(vc.reshape(4, 4)[0]), np.array(g["v_cache_slot0"], dtype=np.float64))
    # slot 3 receives no token and stays zero; every v row is k row + 100 where written
    assert np.all(vc.reshape(4, 4)[3] == 0)


def test_t2_untouched_slots_keep_any_content():
    """A -1 slot writes nothing: every byte outside the written slots is
    unchanged (canary pattern instead of zeros)."""
    g = golden("t2_store_kvcache.json")
    key = bf16_bits_of(g["key"])
    value = bf16_bits_of(np.array(g["key"]) + g["value_offset"])
    canary = np.uint16(0x7FC1)                # a NaN bit pattern
    kc = np.full((1, 4, 2, 2), canary, dtype=np.uint16)
    vc = np.full((1, 4, 2, 2), canary, dtype=np.uint16)
    oracle.kv_store(key, value, kc, vc, g["slot_mapping"])
    assert np.all(kc.reshape(4, 4)[3] == canary) and np.all(vc.reshape(4, 4)[3] == canary)


def test_kv_store_rejects_bad_slots():
    key = bf16_bits_of(np.arange(8).reshape(2, 1, 4))
    kc = np.zeros((1, 4, 1, 4), dtype=np.uint16)
    vc = np.zeros_like(kc)
    with pytest.raises(oracle.OracleError) as e:
        oracle.kv_store(key, key, kc, vc, [1, 1])
    assert e.value.code == -3
    with pytest.raises(oracle.OracleError) as e:
        oracle.kv_store(key, key, kc, vc, [0, 4])
    assert e.value.code == -2
    with pytest.raises(oracle.OracleError) as e:
        oracle.kv_store(key, key, kc, vc, [0, -2])
    assert e.value.code == -2
    assert np.all(kc == 0)                    # rejected before anything is written


def test_t3_t4_slot_mapping_exercise():
    g = golden("t3_slot_mapping.json")
    for case in g["cases"]:
        cu = [0, case["new_tokens"]]
        for fn in (oracle.slot_mapping_blockwalk, oracle.slot_mapping_per_token):
            got = fn([g["block_table"]], [case["cached"]], cu, g["block_size"])
            assert got.tolist() == case["slot_mapping"], fn.__name__


def test_t5_online_softmax_printed_values():
    g = golden("t5_online_softmax.json")
    tol = g["printed_tolerance"]
    out, m, l, _ = oracle.online_softmax(g["s"], g["v"], block=len(g["s"]))
    assert m == g["whole"]["m"]
    assert abs(l - g["whole"]["l"]) < tol and abs(out[0] - g["whole"]["O"]) < tol
    b = g["blocked"]
    out, m, l, tr = oracle.online_softmax(g["s"], g["v"], block=b["block"])
    # trace row: m, l_rescaled, acc_rescaled, l_after, acc_after
    a_row, b_row = tr
    assert a_row[0] == b["after_A"]["m"]
    assert abs(a_row[3] - b["after_A"]["l"]) < tol and abs(a_row[4] - b["after_A"]["acc"]) < tol
    assert b_row[0] == b["after_B"]["m"]
    assert abs(b_row[1] - b["rescaled"]["l"]) < tol and abs(b_row[2] - b["rescaled"]["acc"]) < tol
    assert abs(b_row[1] / a_row[3] - b["rescale_factor"]) < tol
    assert abs(b_row[3] - b["after_B"]["l"]) < tol and abs(b_row[4] - b["after_B"]["acc"]) < tol
    assert abs(out[0] - b["O"]) < tol
    # every blocking gives the same answer
    ref, _, _, _ = oracle.online_softmax(g["s"], g["v"], block=4)
    for blk in (1, 2, 3):
        o, _, _, _ = oracle.online_softmax(g["s"], g["v"], block=blk)
        assert abs(o[0] - ref[0]) < 1e-12


def _t5_attention_problem():
    """The §5.2 row as a real attention problem: one head, head_dim 8,
    scale 1; q = e0, key j = s_j e0, value j = v_j e0 + e_{1+j}.  Then
    out[0] is O and out[1:5] are the softmax weights."""
    g = golden("t5_online_softmax.json")
    s, v = g["s"], g["v"]
    n, d = len(s), 8
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1
    k = np.zeros((n, 1, d)); v_ = np.zeros((n, 1, d))
    for j in range(n):
        k[j, 0, 0] = s[j]
        v_[j, 0, 0] = v[j]
        v_[j, 0, 1 + j] = 1
    return g, bf16_bits_of(q), bf16_bits_of(k), bf16_bits_of(v_)


def test_t5_through_decode_and_prefill():
    g, q, k, v = _t5_attention_problem()
    tol = g["printed_tolerance"]
    # decode: one block of 4 slots, context 4
    kc, vc = k.reshape(1, 4, 1, 8).copy(), v.reshape(1, 4, 1, 8).copy()
    out, lse = oracle.decode(q, kc, vc, [[0]], [4], 1.0)
    assert abs(out[0, 0, 0] - g["whole"]["O"]) < tol
    assert np.all(np.abs(out[0, 0, 1:5] - np.array(g["whole"]["weights"])) < tol)
    assert abs(lse[0, 0] - (g["whole"]["m"] + math.log(g["whole"]["l"]))) < tol
    # prefill: the last of 4 causal rows is the same row
    qq = np.repeat(q, 4, axis=0)
    out_p, _ = oracle.prefill(qq, k, v, [0, 4], [0, 4], 1.0)
    assert np.array_equal(out_p[3], out[0])
    # row 0 sees only key 0: weight 1 on it
    assert np.allclose(out_p[0, 0, :5], [g["v"][0], 1, 0, 0, 0], atol=0, rtol=0)


def test_t6_decode_after_prefill_slots():
    g = golden("t6_decode_after_prefill.json")
    bs = g["block_size"]
    pre = oracle.slot_mapping(g["decode_block_tables"], [0], [0, g["prefill_tokens"]], bs)
    assert pre.tolist() == g["prefill_slot_mapping"]
    dec = oracle.decode_slots(g["decode_block_tables"], g["decode_context_lens"], bs)
    assert dec.tolist() == [g["decode_slot"]]


def test_t6_decode_sees_its_own_token():
    """§7 shape: prefill 5 tokens, then decode token 6 with context 6 equals the
    last row of a 6-token causal prefill; shapes flatten to [*, Hq*d]."""
    g = golden("t6_decode_after_prefill.json")
    heads = W.Heads(g["num_heads"], g["num_kv_heads"], g["head_dim"], g["block_size"], 2)
    work = W.prefill_work(heads, [6], seed=11)
    q, k, v = bits(work.q), bits(work.k), bits(work.v)
    kc = np.zeros((2, heads.block_size, heads.num_kv_heads, heads.head_dim), np.uint16)
    vc = np.zeros_like(kc)
    slots = oracle.slot_mapping(g["decode_block_tables"], [0], [0, 5], heads.block_size)
    oracle.kv_store(k[:5], v[:5], kc, vc, slots)
    out_pre, _ = oracle.prefill(q[:5], k[:5], v[:5], [0, 5], [0, 5], heads.scale)
    assert out_pre.reshape(5, -1).shape == tuple(g["prefill_output_shape_flat"])
    dslot = oracle.decode_slots(g["decode_block_tables"], g["decode_context_lens"], heads.block_size)
    oracle.kv_store(k[5:6], v[5:6], kc, vc, dslot)
    out_dec, _ = oracle.decode(q[5:6], kc, vc, g["decode_block_tables"], g["decode_context_lens"],
                               heads.scale)
    assert out_dec.reshape(1, -1).shape == tuple(g["decode_output_shape_flat"])
    full, _ = oracle.prefill(q, k, v, [0, 6], [0, 6], heads.scale)
    assert np.array_equal(out_dec[0], full[5])
    assert np.array_equal(out_pre, full[:5])


def test_t7_gqa_widths():
    g = golden("t7_gqa_widths.json")
    heads = W.Heads(g["num_heads"], g["num_kv_heads"], g["head_dim"], 256, 4)
    work = W.prefill_work(heads, [3], seed=5)
    assert work.q[0].numel() == g["q_size"]
    assert work.k[0].numel() == g["kv_size"]
    assert work.q[0].numel() + 2 * work.k[0].numel() == g["qkv_size"]
    assert heads.num_heads // heads.num_kv_heads == g["group"]


# ---------------------------------------------------------------------------
# slot mapping invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bs", [1, 4, 16, 256])
def test_slot_mapping_two_statements_agree(bs):
    rng = np.random.default_rng(bs)
    for _ in range(20):
        n = int(rng.integers(1, 6))
        start = rng.integers(0, 3 * bs + 2, n)
        lens = rng.integers(0, 3 * bs + 2, n)
        width = int(((start + lens + bs - 1) // bs).max()) + 1
        bt = rng.permutation(n * width * 2)[: n * width].reshape(n, width).astype(np.int32)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        a = oracle.slot_mapping_blockwalk(bt, start, cu, bs)
        b = oracle.slot_mapping_per_token(bt, start, cu, bs)
        assert np.array_equal(a, b)
        # decode slot of a sequence equals the per-token slot of position ctx-1
        ctx = start + 1
        d = oracle.decode_slots(bt, ctx, bs)
        one = oracle.slot_mapping_per_token(bt, ctx - 1, np.arange(n + 1), bs)
        assert np.array_equal(d, one)


def test_slot_mapping_errors_and_padding():
    with pytest.raises(oracle.OracleError) as e:
        oracle.slot_mapping_blockwalk([[3, -1]], [0], [0, 6], 4)
    assert e.value.code == -4
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping_per_token([[3]], [2], [0, 3], 4)
    # padding rows: context 0 -> slot -1
    assert oracle.decode_slots([[5, 6], [-1, -1]], [5, 0], 4).tolist() == [24, -1]


# ---------------------------------------------------------------------------
# attention: closed forms
# ---------------------------------------------------------------------------
def _rand_bits(rng, shape, scale=1.0):
    return bf16_bits_of(torch.tensor(rng.normal(size=shape) * scale, dtype=torch.float32)
                        .to(torch.bfloat16).float().numpy())


def test_single_key_returns_its_value():
    rng = np.random.default_rng(1)
    q = _rand_bits(rng, (1, 2, 16))
    kc = _rand_bits(rng, (1, 4, 1, 16))
    vc = _rand_bits(rng, (1, 4, 1, 16))
    out, lse = oracle.decode(q, kc, vc, [[0]], [1], 0.25)
    assert np.array_equal(out[0, 0], f64(vc[0, 0, 0])) and np.array_equal(out[0, 1], f64(vc[0, 0, 0]))
    s = 0.25 * float(f64(q[0, 0]) @ f64(kc[0, 0, 0]))
    assert abs(lse[0, 0] - s) < 1e-12


def test_identical_keys_average_values():
    rng = np.random.default_rng(2)
    n = 7
    q = _rand_bits(rng, (1, 1, 8))
    k1 = _rand_bits(rng, (1, 8))
    kc = np.repeat(k1[None, :, None, :], 1, 0).repeat(n, 1).reshape(1, n, 1, 8).copy()
    vc = _rand_bits(rng, (1, n, 1, 8))
    out, lse = oracle.decode(q, kc, vc, [[0]], [n], 0.5)
    assert np.allclose(out[0, 0], f64(vc[0, :, 0]).mean(0), rtol=0, atol=1e-12)
    s = 0.5 * float(f64(q[0, 0]) @ f64(k1[0]))
    assert abs(lse[0, 0] - (s + math.log(n))) < 1e-12


def test_zero_query_is_causal_prefix_mean_with_prefix():
    """q = 0 makes every admitted key equally likely, so row t of a sequence
    with prefix P must be the mean of values 0..P+t -- pins the causal bound
    and its bottom-right alignment."""
    rng = np.random.default_rng(3)
    hq, hkv, d, bs = 4, 2, 8, 4
    P, C = 6, 5
    q = np.zeros((C, hq, d), np.uint16)
    kc = _rand_bits(rng, (4, bs, hkv, d))
    vc = _rand_bits(rng, (4, bs, hkv, d))
    bt = [[2, 0, 3]]
    out, _ = oracle.prefill(q, None, None, [0, C], [0, P + C], 1.0, k_cache=kc, v_cache=vc,
                            block_tables=bt)
    vals = f64(vc)
    for t in range(C):
        keys = [(bt[0][j // bs], j % bs) for j in range(P + t + 1)]
        for h in range(hq):
            mean = np.mean([vals[b, o, h // (hq // hkv)] for b, o in keys], axis=0)
            assert np.allclose(out[t, h], mean, atol=1e-12, rtol=0)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    d, n = 8, 9
    q = np.zeros((1, 1, d)); q[0, 0, 3] = 8
    k = np.zeros((1, n, 1, d)); k[0, 5, 0, 3] = 8
    v = rng.normal(size=(1, n, 1, d))
    qb, kb, vb = bf16_bits_of(q), bf16_bits_of(k), bits(torch.tensor(v).to(torch.bfloat16))
    out, _ = oracle.decode(qb, kb, vb, [[0]], [n], 1.0)
    # weight of key 5 is 1 / (1 + 8 e^-64): equal to its value to 1e-20
    assert np.allclose(out[0, 0], f64(vb[0, 5, 0]), atol=1e-20, rtol=0)


# ---------------------------------------------------------------------------
# attention: special cases that reduce to a library routine
# ---------------------------------------------------------------------------
def _sdpa(q, k, v, scale, mask=None, causal=False):
    """torch fp64 SDPA for one sequence: q [Lq, Hq, d], k/v [Lk, Hq, d]."""
    qt = torch.from_numpy(q).transpose(0, 1)[None]
    kt = torch.from_numpy(k).transpose(0, 1)[None]
    vt = torch.from_numpy(v).transpose(0, 1)[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, is_causal=causal, scale=scale)
    return o[0].transpose(0, 1).numpy()


def test_varlen_prefill_matches_library_sdpa():
    heads = W.Heads(8, 2, 32, 16, 64)
    work = W.prefill_work(heads, [1, 17, 40, 5], seed=21)
    q, k, v = bits(work.q), bits(work.k), bits(work.v)
    out, lse = oracle.prefill(q, k, v, work.cu_seqlens_q, work.cu_seqlens_k, heads.scale)
    g = heads.num_heads // heads.num_kv_heads
    cu = work.cu_seqlens_q.tolist()
    for i in range(work.num_seqs):
        a, b = cu[i], cu[i + 1]
        kk = np.repeat(f64(k[a:b]), g, axis=1)          # GQA: kv head h serves q heads h*g..h*g+g-1
        vv = np.repeat(f64(v[a:b]), g, axis=1)
        ref = _sdpa(f64(q[a:b]), kk, vv, heads.scale, causal=True)
        assert np.allclose(out[a:b], ref, atol=1e-12, rtol=1e-12)


def test_prefix_prefill_matches_library_sdpa_bottom_right():
    heads = W.Heads(4, 4, 16, 4, 32)
    rng = np.random.default_rng(5)
    P, C = 9, 6
    work = W.prefill_work(heads, [C], [P], seed=22)
    kc, vc = W.history_cache(heads, 23)
    kcb, vcb = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q,
                                heads.block_size)
    oracle.kv_store(bits(work.k), bits(work.v), kcb, vcb, slots)
    out, _ = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q, work.cu_seqlens_k,
                            heads.scale, k_cache=kcb, v_cache=vcb, block_tables=work.block_tables)
    bt = work.block_tables[0].tolist()
    kk = np.stack([f64(kcb[bt[j // 4], j % 4]) for j in range(P + C)])
    vv = np.stack([f64(vcb[bt[j // 4], j % 4]) for j in range(P + C)])
    mask = torch.ones(C, P + C, dtype=torch.bool).tril(diagonal=P)
    ref = _sdpa(f64(bits(work.q)), kk, vv, heads.scale, mask=mask)
    assert np.allclose(out, ref, atol=1e-12, rtol=1e-12)
    del rng


def test_decode_matches_library_sdpa():
    heads = W.Heads(8, 4, 16, 8, 40)
    work = W.decode_work(heads, [1, 9, 30, 64, 0], seed=24)
    kc, vc = W.history_cache(heads, 25)
    kcb, vcb = bits(kc).copy(), bits(vc).copy()
    out, lse = oracle.decode(bits(work.q), kcb, vcb, work.block_tables, work.context_lens,
                             heads.scale)
    g = 2
    for b, ctx in enumerate(work.context_lens.tolist()):
        if ctx == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        bt = work.block_tables[b].tolist()
        kk = np.stack([f64(kcb[bt[j // 8], j % 8]) for j in range(ctx)]).repeat(g, axis=1)
        vv = np.stack([f64(vcb[bt[j // 8], j % 8]) for j in range(ctx)]).repeat(g, axis=1)
        ref = _sdpa(f64(bits(work.q[b:b + 1])), kk, vv, heads.scale)
        assert np.allclose(out[b:b + 1], ref, atol=1e-12, rtol=1e-12)
        s = heads.scale * np.einsum("hd,jhd->hj", f64(bits(work.q[b])), kk)
        ref_lse = torch.logsumexp(torch.from_numpy(s), dim=1).numpy()
        assert np.allclose(lse[b], ref_lse, atol=1e-12, rtol=0)


# ---------------------------------------------------------------------------
# attention: invariants
# ---------------------------------------------------------------------------
def test_physical_block_order_is_irrelevant():
    heads = W.Heads(4, 2, 16, 4, 24)
    work = W.decode_work(heads, [13, 5, 22], seed=31)
    kc, vc = W.history_cache(heads, 32)
    kcb, vcb = bits(kc), bits(vc)
    out, lse = oracle.decode(bits(work.q), kcb, vcb, work.block_tables, work.context_lens,
                             heads.scale)
    perm = np.random.default_rng(0).permutation(heads.num_blocks)   # new position of block b
    kc2 = np.empty_like(kcb); vc2 = np.empty_like(vcb)
    kc2[perm] = kcb; vc2[perm] = vcb
    bt = work.block_tables.numpy()
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.decode(bits(work.q), kc2, vc2, bt2, work.context_lens, heads.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_prefix_prefill_equals_tail_of_full_prefill():
    heads = W.Heads(4, 2, 16, 4, 32)
    P, C = 10, 7
    full = W.prefill_work(heads, [P + C], seed=41)
    q, k, v = bits(full.q), bits(full.k), bits(full.v)
    kc = np.zeros((heads.num_blocks, 4, 2, 16), np.uint16); vc = np.zeros_like(kc)
    slots = oracle.slot_mapping(full.block_tables, [0], [0, P + C], 4)
    oracle.kv_store(k, v, kc, vc, slots)
    ref, ref_lse = oracle.prefill(q, k, v, [0, P + C], [0, P + C], heads.scale)
    out, lse = oracle.prefill(q[P:], None, None, [0, C], [0, P + C], heads.scale, k_cache=kc,
                              v_cache=vc, block_tables=full.block_tables)
    assert np.array_equal(out, ref[P:]) and np.array_equal(lse, ref_lse[P:])


def test_gqa_equals_mha_with_repeated_kv():
    heads = W.Heads(6, 2, 16, 4, 8)
    work = W.prefill_work(heads, [5, 8], seed=51)
    q, k, v = bits(work.q), bits(work.k), bits(work.v)
    out, _ = oracle.prefill(q, k, v, work.cu_seqlens_q, work.cu_seqlens_k, heads.scale)
    k3 = np.ascontiguousarray(np.repeat(k, 3, axis=1))
    v3 = np.ascontiguousarray(np.repeat(v, 3, axis=1))
    out3, _ = oracle.prefill(q, k3, v3, work.cu_seqlens_q, work.cu_seqlens_k, heads.scale)
    assert np.array_equal(out, out3)


def test_strided_rows_equal_contiguous_rows():
    """k/v views of a fused qkv row (row stride > Hkv*d) give the same result."""
    heads = W.Heads(4, 2, 8, 4, 8)
    work = W.prefill_work(heads, [6, 3], seed=61)
    qkv = torch.cat([work.q.flatten(1), work.k.flatten(1), work.v.flatten(1)], dim=1)
    q = qkv[:, :32].view(-1, 4, 8); k = qkv[:, 32:48].view(-1, 2, 8); v = qkv[:, 48:].view(-1, 2, 8)
    a, _ = oracle.prefill(bits(q), bits(k), bits(v), work.cu_seqlens_q, work.cu_seqlens_k, 0.3)
    b, _ = oracle.prefill(bits(work.q), bits(work.k), bits(work.v), work.cu_seqlens_q,
                          work.cu_seqlens_k, 0.3)
    assert bits(k).strides[0] == 64 * 2 and np.array_equal(a, b)


@pytest.mark.parametrize("split", [1, 3, 16, 64, 1000])
def test_split_k_merge_equals_unsplit(split):
    heads = W.Heads(8, 2, 16, 16, 24)
    work = W.decode_work(heads, [1, 17, 100, 0, 64], seed=71)
    kc, vc = W.history_cache(heads, 72)
    args = (bits(work.q), bits(kc), bits(vc), work.block_tables, work.context_lens, heads.scale)
    ref, ref_lse = oracle.decode(*args)
    out, lse = oracle.decode_split(*args, split=split)
    assert np.allclose(out, ref, atol=1e-13, rtol=1e-12)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)) and np.allclose(lse[fin], ref_lse[fin], atol=1e-12)


def test_attention_rejects_holes_in_block_table():
    heads = W.Heads(2, 1, 8, 4, 4)
    kc, vc = W.history_cache(heads, 3)
    q = bits(W.normal_bf16((1, 2, 8), W.generator(1)))
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(q, bits(kc), bits(vc), [[1, -1]], [6], 0.3)
    assert e.value.code == -4
    with pytest.raises(oracle.OracleError) as e:
        oracle.prefill(q, None, None, [0, 1], [0, 0], 0.3, k_cache=bits(kc), v_cache=bits(vc),
                       block_tables=[[0]])
    assert e.value.code == -5


def test_tiny_workload_shape():
    pre, dec = W.tiny()
    assert pre.block_tables[0].tolist() == [7, 9]
    assert pre.total_q == 9 and dec.context_lens.tolist() == [7, 4]
    # decode slot of seq 0: position 6 lives in block 9 at offset 2
    assert oracle.decode_slots(dec.block_tables, dec.context_lens, 4)[0] == 38


def test_prefill_rows_equal_full_prefill_rows():
    heads = W.Heads(4, 2, 16, 4, 32)
    work = W.prefill_work(heads, [5, 0, 11], [3, 0, 6], seed=81)
    kc, vc = W.history_cache(heads, 82)
    kcb, vcb = bits(kc).copy(), bits(vc).copy()
    slots = oracle.slot_mapping(work.block_tables, work.prefix_lens, work.cu_seqlens_q, 4)
    oracle.kv_store(bits(work.k), bits(work.v), kcb, vcb, slots)
    kw = dict(k_cache=kcb, v_cache=vcb, block_tables=work.block_tables)
    full, full_lse = oracle.prefill(bits(work.q), None, None, work.cu_seqlens_q,
                                    work.cu_seqlens_k, heads.scale, **kw)
    rows = [15, 0, 7, 4]
    part, part_lse = oracle.prefill_rows(bits(work.q), None, None, work.cu_seqlens_q,
                                         work.cu_seqlens_k, heads.scale, rows, **kw)
    assert np.array_equal(part, full[rows]) and np.array_equal(part_lse, full_lse[rows])


# ---------------------------------------------------------------------------
# QK-Norm + RoPE prologue (L17 §4; RMSNorm module of "Nano-VLLM full-code
# notes (5)"; rotary embedding as read: split-halves pairing, e with e + d/2,
# which the pages apply but do not print)
# ---------------------------------------------------------------------------
def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _ones(d):
    return _bf16_bits(np.ones(d))


def test_round_bf16_matches_library_and_breaks_ties_to_even():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-30,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle.round_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(lib, mine)
    one = 0x3F80
    assert oracle.round_bf16(1 + 2.0 ** -8) == one               # tie -> even (1.0)
    assert oracle.round_bf16(1 + 3 * 2.0 ** -8) == one + 2       # tie -> even (1 + 2^-6)
    assert oracle.round_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == one + 1   # just above the tie


def _prologue(rows, pos, w=None, eps=1e-6, theta=1e6):
    """rows: float array [n, d] (bf16-exact) used as one q head per token."""
    rows = np.asarray(rows, np.float64)
    n, d = rows.shape
    q = _bf16_bits(rows).reshape(n, 1, d)
    k = q.copy()
    w = _ones(d) if w is None else w
    qo, ko = oracle.qk_norm_rope(q, k, np.broadcast_to(np.asarray(pos, np.int64), (n,)), w, w,
                                 eps, theta)
    assert np.array_equal(qo, ko)
    return f64(qo.reshape(n, d))


def test_rmsnorm_of_a_constant_row():
    # every element equal: x / sqrt(mean(x^2) + eps) = sign(x) / sqrt(1 + eps/x^2)
    out = _prologue([[0.5] * 64, [3.0] * 64, [-2.0] * 64], 0)
    assert np.array_equal(out, np.array([[1.0] * 64, [1.0] * 64, [-1.0] * 64]))
    # eps sits inside the square root: x = 1e-3, eps = 1e-6 -> 1/sqrt(2)
    x = float(torch.tensor(1e-3).to(torch.bfloat16))
    out = _prologue([[x] * 64], 0, eps=x * x)
    assert np.all(out == float(torch.tensor(2 ** -0.5).to(torch.bfloat16)))


def test_rmsnorm_output_has_unit_rms_and_ignores_scale():
    rng = np.random.default_rng(12)
    rows = f64(_bf16_bits(rng.standard_normal((16, 128)) * 3))
    out = _prologue(rows, 0)
    assert np.allclose(np.sqrt((out ** 2).mean(axis=1)), 1.0, atol=2e-3)
    # with eps = 0, scaling a row by a power of two changes nothing
    a = _prologue(rows, 0, eps=0.0)
    b = _prologue(rows * 8.0, 0, eps=0.0)
    assert np.array_equal(a, b)


def test_rmsnorm_weight_scales_each_element():
    rng = np.random.default_rng(13)
    rows = f64(_bf16_bits(rng.standard_normal((4, 128))))
    base = _prologue(rows, 0)
    assert np.array_equal(_prologue(rows, 0, w=_bf16_bits(np.full(128, 2.0))), 2 * base)
    w = np.ones(128)
    w[37] = 0.0
    w[100] = -1.0
    got = _prologue(rows, 0, w=_bf16_bits(w))
    assert np.all(got[:, 37] == 0) and np.array_equal(got[:, 100], -base[:, 100])
    keep = [e for e in range(128) if e not in (37, 100)]
    assert np.array_equal(got[:, keep], base[:, keep])


@pytest.mark.parametrize("d,theta", [(128, 1e6), (128, 1e4), (64, 1e4)])
def test_rope_turns_pairs_by_closed_form_angles(d, theta):
    """Pair i = (e, e + d/2) is the complex number x_e + j x_{e+d/2}, turned by
    pos * theta^(-2i/d): pair 0 by pos radians, pair d/4 by pos / sqrt(theta)."""
    rng = np.random.default_rng(14)
    rows = f64(_bf16_bits(rng.standard_normal((8, d))))
    base = _prologue(rows, 0, theta=theta)                 # position 0: no rotation
    h = d // 2
    for pos in (1, 7, 300, 4095, 32767):
        out = _prologue(rows, pos, theta=theta)
        for i, angle in ((0, pos), (d // 4, pos / math.sqrt(theta))):
            z = (base[:, i] + 1j * base[:, i + h]) * np.exp(1j * angle)
            tol = 2.0 ** -7 * np.abs(z) + 1e-6
            assert np.all(np.abs(out[:, i] - z.real) <= tol), (pos, i)
            assert np.all(np.abs(out[:, i + h] - z.imag) <= tol), (pos, i)


def test_rope_keeps_pair_norms_and_depends_on_relative_position():
    rng = np.random.default_rng(15)
    d = 128
    rows = f64(_bf16_bits(rng.standard_normal((2, d))))
    base = _prologue(rows, 0)
    out = _prologue(rows, 1234)
    nb = base[:, :64] ** 2 + base[:, 64:] ** 2
    no = out[:, :64] ** 2 + out[:, 64:] ** 2
    assert np.allclose(no, nb, rtol=2e-2, atol=1e-3)
    # <R(p) q, R(p') k> depends on p - p' only
    def dot(p, pk):
        return float((_prologue(rows[:1], p) * _prologue(rows[1:], pk)).sum())
    for p, pk, s in ((10, 3, 500), (4000, 100, -50), (7, 7, 31000)):
        assert abs(dot(p, pk) - dot(p + s, pk + s)) <= 0.05 * (1 + abs(dot(p, pk)))


def test_prologue_reads_each_tokens_position_and_strided_rows():
    rng = np.random.default_rng(16)
    n, hq, hkv, d = 5, 4, 2, 64
    big = _bf16_bits(rng.standard_normal((n, hq + 2 * hkv, d)))      # fused qkv rows
    q, k = big[:, :hq], big[:, hq:hq + hkv]
    pos = [0, 9, 9, 100, 3]
    qw, kw = _bf16_bits(rng.uniform(0.5, 1.5, d)), _bf16_bits(rng.uniform(0.5, 1.5, d))
    qo, ko = oracle.qk_norm_rope(q, k, pos, qw, kw)
    qc, kc = oracle.qk_norm_rope(np.ascontiguousarray(q), np.ascontiguousarray(k), pos, qw, kw)
    assert np.array_equal(qo, qc) and np.array_equal(ko, kc)
    for t in range(n):                      # token by token gives the same rows
        a, b = oracle.qk_norm_rope(q[t:t + 1], k[t:t + 1], pos[t:t + 1], qw, kw)
        assert np.array_equal(a[0], qo[t]) and np.array_equal(b[0], ko[t])
    # the two tokens at position 9 differ only through their inputs: swap them
    q2, k2 = q[[0, 2, 1, 3, 4]], k[[0, 2, 1, 3, 4]]
    a, b = oracle.qk_norm_rope(q2, k2, pos, qw, kw)
    assert np.array_equal(a[[0, 2, 1, 3, 4]], qo) and np.array_equal(b[[0, 2, 1, 3, 4]], ko)
    # q and k use their own weights
    a, b = oracle.qk_norm_rope(q, k, pos, kw, qw)
    assert not np.array_equal(a, qo)


def _check_tables(work, nblk):
    """Each sequence owns ceil(len / bs) distinct pool blocks, no block is
    shared, and the rest of its row is -1."""
    bt = work.block_tables
    seen = []
    for i, n in enumerate(nblk):
        row = bt[i].tolist()
        assert all(0 <= b < work.heads.num_blocks for b in row[:n]), i
        assert all(b == -1 for b in row[n:]), i
        seen += row[:n]
    assert len(seen) == len(set(seen))


def test_benchmark_workloads_follow_the_recipe():
    """The seeded inputs have the shapes, ranges and table structure the
    input recipe states, and the same seed gives the same inputs."""
    bs = 256
    dec = W.qwen3_decode()
    h = dec.heads
    assert (h.num_heads, h.num_kv_heads, h.head_dim, h.block_size, h.num_blocks) == (16, 8, 128, bs, 2048)
    ctx = dec.context_lens
    assert dec.batch == 64 and int(ctx.min()) >= 512 and int(ctx.max()) <= 4096
    _check_tables(dec, [(c + bs - 1) // bs for c in ctx.tolist()])
    again = W.qwen3_decode()
    assert torch.equal(again.context_lens, ctx) and torch.equal(again.q, dec.q)

    pre = W.varlen_prefill()
    lens = pre.q_lens.tolist()
    assert len(lens) == 8 and all(128 <= n <= 4096 for n in lens) and pre.total_q == 19576
    assert torch.equal(pre.cu_seqlens_q, pre.cu_seqlens_k) and int(pre.prefix_lens.sum()) == 0

    px = W.prefix_prefill()
    assert px.num_seqs == 16
    assert all(p % bs == 0 and 0 <= p <= 12 * bs for p in px.prefix_lens.tolist())
    assert all(64 <= c <= 1024 for c in px.q_lens.tolist())
    tot = (px.prefix_lens + px.q_lens).tolist()
    assert (px.cu_seqlens_k[1:] - px.cu_seqlens_k[:-1]).tolist() == tot
    _check_tables(px, [(t + bs - 1) // bs for t in tot])
    pu = W.prefix_prefill(unaligned=True)
    assert all(p % bs != 0 for p in pu.prefix_lens.tolist())

    lg = W.large_decode()
    assert (lg.heads.num_heads, lg.heads.num_kv_heads, lg.heads.num_blocks) == (32, 8, 40000)
    c = lg.context_lens.tolist()
    assert len(c) == 288 and all(v == 0 for v in c[256:])
    assert all(1024 <= v <= 32768 for v in c[:256])
    _check_tables(lg, [(v + bs - 1) // bs for v in c])
