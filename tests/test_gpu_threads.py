"""First use of the library from several host threads at once.

Each entry point sets up per-device state on its first call (kernel
attributes, occupancy, SM counts).  A fresh process starts four threads
behind a barrier; each makes its first kv_store, decode and prefill calls at
the same moment on its own stream.  The results must equal, bit for bit,
the same calls made afterwards from one thread, and no kernel may flag its
input.  The kernels are deterministic (every output element is computed by
one CTA in a fixed order), so equality is exact.
"""
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent

SCRIPT = textwrap.dedent("""
    import sys, threading
    import torch
    sys.path.insert(0, {root!r})
    from paged_kv_cache_303_gb300 import ops, workloads as W

    dh = W.Heads(16, 8, 128, 16, 512)
    dw = W.decode_work(dh, [900, 0, 33, 2500, 1], seed=1201)
    ph = W.Heads(16, 8, 128, 16, 64)
    pw = W.prefill_work(ph, [300, 1, 129], seed=1202)
    kc0, vc0 = W.history_cache(dh, 1203, device="cuda")
    args = dict(
        dq=dw.q.cuda(), dk=dw.k.cuda(), dv=dw.v.cuda(), bt=dw.block_tables.cuda(),
        ctx=dw.context_lens.cuda(), pq=pw.q.cuda(), pk=pw.k.cuda(), pv=pw.v.cuda(),
        cu_q=pw.cu_seqlens_q.cuda(), cu_k=pw.cu_seqlens_k.cuda())
    torch.cuda.synchronize()

    def work(a):
        kc, vc = kc0.clone(), vc0.clone()
        slots = ops.kv_build_decode_slots(a["bt"], a["ctx"], dh.block_size)
        ops.kv_store(a["dk"], a["dv"], kc, vc, slots)
        dout = ops.paged_attn_decode(a["dq"], kc, vc, a["bt"], a["ctx"], dw.max_context_len, dh.scale)
        pout = ops.paged_attn_prefill(a["pq"], a["pk"], a["pv"], a["cu_q"], a["cu_k"],
                                      pw.max_seqlen_q, pw.max_seqlen_k, ph.scale)
        return kc, dout, pout

    n = 4
    barrier = threading.Barrier(n)
    results, errors = [None] * n, []

    def run(i):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.default_stream())
            barrier.wait()
            with torch.cuda.stream(s):
                results[i] = work(args)
            s.synchronize()
        except Exception as e:          # reported by the parent
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    ref = work(args)
    torch.cuda.synchronize()
    for kc, dout, pout in results:
        assert torch.equal(kc, ref[0])
        assert torch.equal(dout.view(torch.int16), ref[1].view(torch.int16))
        assert torch.equal(pout.view(torch.int16), ref[2].view(torch.int16))
    assert ops.device_status(clear=True) == 0
    print("threads ok")
""")


def test_first_calls_from_four_threads_at_once():
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=str(ROOT))], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout + r.stderr
