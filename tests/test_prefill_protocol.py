"""Model check of the persistent prefill kernel's barrier protocol (CPU only).

One CTA of the prefill kernel runs work units one after another. A scheduler
lane publishes each unit in one of two shared-memory records. A producer
lane loads Q and streams the unit's K/V tiles through a ring of kSlots
stages. The MMA lane issues S = Q K^T and O += P V per tile and head. Two
softmax warpgroups turn S into P and write the output. They synchronise
through mbarriers:

  * unit_full / unit_empty: the unit records;
  * loads_done: the producer has issued a unit's last load;
  * q_full / q_free: the Q buffer;
  * slot_full / slot_free: the ring;
  * s_full / p_full / o_done: the S, P and O hand-offs per head.

The tensor-core products run in issue order, and a commit arrives once
every earlier product has completed; bulk copies land in any order.

The model runs the protocol as the kernel writes it under random schedules,
with the mbarrier semantics of PTX: a phase completes when its pending
arrivals and transaction bytes reach zero, and `try_wait.parity P` succeeds
when the open phase's parity is not P. It checks that:

  * every product reads a K, V or Q tile that has fully landed and is the one
    it expects;
  * no stage or Q buffer is refilled while a product still reads it;
  * the softmax reads the S of the tile it waits for;
  * the epilogue reads O after all of the unit's P V products;
  * the zeroing of a paged unit's last V tile hits that tile after it has
    landed and before its P V;
  * nothing deadlocks;
  * when the CTA ends, no copy is landing and no product or commit is
    pending.

Every wait of a role but the teardown's gives up once the CTA's abort flag
is raised (the kernel raises it when a bounded wait runs out).  Runs that
raise it at a random step check that each role leaves by its own exit path
and that the teardown still waits for every copy and product it issued.

Five planted mistakes are caught. The first is a separate warp that zeroes
the V tail without the softmax's ordering. The second is a softmax whose S
parity restarts with every unit instead of running on across units. The
third has the producer skip the wait for the previous unit's last S
products before reloading Q. The fourth and fifth leave after an abort
without the teardown: a producer that does not wait for its copies and an
MMA thread that does not wait for its products.
"""
import random

import pytest

K_SLOTS = 5


class Bar:
    def __init__(self, count, log, name):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0
        self.log, self.name = log, name

    def _settle(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        if self.pending == 0:
            self.log.append(f"{self.name}: arrival beyond the phase's count")
            return
        self.pending -= 1
        self._settle()

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._settle()

    def try_wait_parity(self, parity):
        return (self.phase & 1) != parity


class W:
    """A wait that gives up when the CTA's abort flag is raised (the kernel's
    wait_or_abort): the role receives True if the phase completed, False if
    it gave up."""

    def __init__(self, pred):
        self.pred = pred


class P:
    """A plain wait (bounded only by time): the teardown waits for copies and
    products that are already issued."""

    def __init__(self, pred):
        self.pred = pred


def simulate(units, rng, plant=None, units_per_tile=2, abort_at=None):
    """units: list of (n_kv, ntile, tail); tail: paged unit whose last V tile
    has rows past the last key.  abort_at: scheduling step at which the CTA's
    abort flag is raised (as when some wait of the CTA ran out of time).
    Returns the list of violations."""
    log = []
    B = lambda n, c=1: Bar(c, log, n)
    q_full, q_free, loads_done = B("q_full"), B("q_free"), B("loads_done")
    drain = B("drain")
    slot_full = [B(f"slot_full{s}") for s in range(K_SLOTS)]
    slot_free = [B(f"slot_free{s}") for s in range(K_SLOTS)]
    s_full = [B(f"s_full{t}") for t in range(2)]
    p_full = [B(f"p_full{t}") for t in range(2)]
    o_done = [B(f"o_done{t}") for t in range(2)]
    unit_full = [B(f"unit_full{i}") for i in range(2)]
    unit_empty = [B(f"unit_empty{i}", 4) for i in range(2)]   # producer, MMA, two softmax groups
    records = [None, None]
    total_units = len(units)
    abort = [False]

    slot = [None] * K_SLOTS            # [load index, landed units, zeroed] in the stage
    q_buf = [None]                     # [unit, landed units]
    readers = [0] * K_SLOTS            # products issued and not yet run that read the stage
    q_readers = [0]
    inflight = []                      # copy units: ("kv", stage, load) / ("q", unit)
    pipe = []                          # tensor-core products and commits, in issue order
    s_tile = [None, None]              # (unit, tile) whose S the head's S columns hold
    o_count = [[None, 0], [None, 0]]   # [unit, P V products completed] per head

    def scheduler():
        for u in range(total_units + 1):
            if u >= 1:
                if not (yield W(lambda u=u: loads_done.try_wait_parity((u - 1) & 1))):
                    return
            if u >= 2:
                if not (yield W(lambda u=u: unit_empty[u % 2].try_wait_parity(((u // 2) - 1) & 1))):
                    return
            records[u % 2] = units[u] if u < total_units else None
            unit_full[u % 2].arrive()
            yield None

    def producer():
        n, nq = 0, 0
        live = True
        for u in range(total_units + 1):
            if not (yield W(lambda u=u: unit_full[u % 2].try_wait_parity((u // 2) & 1))):
                break
            rec = records[u % 2]
            if rec is None:
                break
            n_kv = rec[0]
            q_at = 0 if u == 0 else min(2, 2 * n_kv - 1)
            for i in range(2 * n_kv):
                if i == q_at:
                    if u > 0 and plant != "no_q_free_wait":
                        if not (yield W(lambda u=u: q_free.try_wait_parity((u - 1) & 1))):
                            live = False
                            break
                    if q_readers[0]:
                        log.append(f"Q of unit {u} loaded while a product still reads unit {q_buf[0][0]}'s")
                    q_full.arrive_expect_tx(units_per_tile)
                    q_buf[0] = [u, 0]
                    inflight.extend([("q", u)] * units_per_tile)
                    nq += 1
                    yield None
                s = n % K_SLOTS
                if n >= K_SLOTS:
                    if not (yield W(lambda s=s, n=n: slot_free[s].try_wait_parity(((n // K_SLOTS) - 1) & 1))):
                        live = False
                        break
                if readers[s]:
                    log.append(f"stage {s} refilled with load {n} while a product reads it")
                if any(c[0] == "kv" and c[1] == s for c in inflight):
                    log.append(f"stage {s} refilled with load {n} while an earlier copy lands")
                slot_full[s].arrive_expect_tx(units_per_tile)
                slot[s] = [n, 0, False]
                inflight.extend([("kv", s, n)] * units_per_tile)
                n += 1
                yield None
            if not live:
                break
            loads_done.arrive()
            unit_empty[u % 2].arrive()
        if plant == "no_copy_drain":
            return
        # no copy may still be landing when the CTA leaves
        for m in range(max(0, n - K_SLOTS), n):
            yield P(lambda m=m: slot_full[m % K_SLOTS].try_wait_parity((m // K_SLOTS) & 1))
        if nq:
            yield P(lambda: q_full.try_wait_parity((nq - 1) & 1))

    def use_slot(n, what):
        s = n % K_SLOTS
        if slot[s] is None or slot[s][0] != n or slot[s][1] != units_per_tile:
            log.append(f"{what} issued on stage {s} holding {slot[s]}, expected load {n}")
        readers[s] += 1
        return s

    def mma():
        n0 = 0
        ppar = [0, 0]
        for u in range(total_units + 1):
            if not (yield W(lambda u=u: unit_full[u % 2].try_wait_parity((u // 2) & 1))):
                break
            rec = records[u % 2]
            if rec is None:
                break
            n_kv, ntile, tail = rec
            if not (yield W(lambda u=u: q_full.try_wait_parity(u & 1))):
                break
            if not (yield W(lambda n0=n0: slot_full[n0 % K_SLOTS].try_wait_parity((n0 // K_SLOTS) & 1))):
                break
            if q_buf[0] is None or q_buf[0] != [u, units_per_tile]:
                log.append(f"S of unit {u} issued on Q buffer {q_buf[0]}")
            for t in range(ntile):
                s = use_slot(n0, "S")
                q_readers[0] += 1
                pipe.append(("S", t, u, 0, s))
                pipe.append(("commit", s_full[t]))
            if n_kv == 1:
                pipe.append(("commit", q_free))
            pipe.append(("commit", slot_free[n0 % K_SLOTS]))
            yield None
            live = True
            for j in range(n_kv):
                nv, nxt, nk = n0 + 2 * j + 1, j + 1 < n_kv, n0 + 2 * j + 2
                live = yield W(lambda nv=nv: slot_full[nv % K_SLOTS].try_wait_parity((nv // K_SLOTS) & 1))
                if live and nxt:
                    live = yield W(lambda nk=nk: slot_full[nk % K_SLOTS].try_wait_parity((nk // K_SLOTS) & 1))
                for t in range(ntile):
                    if not live:
                        break
                    live = yield W(lambda t=t: p_full[t].try_wait_parity(ppar[t]))
                    if not live:
                        break
                    ppar[t] ^= 1
                    if tail and not nxt and t == 0:
                        st = slot[nv % K_SLOTS]
                        if st is None or st[0] != nv or not st[2]:
                            log.append(f"last P V of unit {u} issued before its V tail was zeroed")
                    s = use_slot(nv, "P V")
                    pipe.append(("PV", t, u, j, s))
                    pipe.append(("commit", o_done[t]))
                    if nxt:
                        s = use_slot(nk, "S")
                        q_readers[0] += 1
                        pipe.append(("S", t, u, j + 1, s))
                        pipe.append(("commit", s_full[t]))
                if not live:
                    break
                if j + 2 == n_kv:
                    pipe.append(("commit", q_free))
                pipe.append(("commit", slot_free[nv % K_SLOTS]))
                if nxt:
                    pipe.append(("commit", slot_free[nk % K_SLOTS]))
                yield None
            if not live:
                break
            n0 += 2 * n_kv
            unit_empty[u % 2].arrive()
        if plant == "no_mma_drain":
            return
        # every product has completed before tensor memory is released
        pipe.append(("commit", drain))
        yield P(lambda: drain.try_wait_parity(0))

    def softmax(t):
        n0 = 0
        jpar = 0
        for u in range(total_units + 1):
            if not (yield W(lambda u=u: unit_full[u % 2].try_wait_parity((u // 2) & 1))):
                return
            rec = records[u % 2]
            if rec is None:
                return
            n_kv, ntile, tail = rec
            if plant == "jpar_per_unit":
                jpar = 0            # wrong: the barrier's phases run on across units
            if t < ntile:
                for j in range(n_kv):
                    if not (yield W(lambda jp=jpar: s_full[t].try_wait_parity(jp))):
                        return
                    jpar ^= 1
                    if s_tile[t] != (u, j):
                        log.append(f"head {t} read S {s_tile[t]} as unit {u} tile {j}")
                    if j + 1 == n_kv and tail and t == 0 and plant != "fixer_warp":
                        nv = n0 + 2 * n_kv - 1
                        if not (yield W(lambda nv=nv: slot_full[nv % K_SLOTS].try_wait_parity((nv // K_SLOTS) & 1))):
                            return
                        st = slot[nv % K_SLOTS]
                        if st is None or st[0] != nv or st[1] != units_per_tile:
                            log.append(f"V tail of unit {u} zeroed on stage holding {st}")
                        else:
                            st[2] = True
                    p_full[t].arrive()
                    yield None
                if not (yield W(lambda jp=jpar: o_done[t].try_wait_parity(jp ^ 1))):
                    return
                if o_count[t] != [u, n_kv]:
                    log.append(f"epilogue of head {t} unit {u} read O after {o_count[t]}")
            n0 += 2 * n_kv
            unit_empty[u % 2].arrive()

    def fixer():
        # planted: a separate warp zeroes the V tail as soon as the unit is
        # published, waiting on the stage by parity alone
        n0 = 0
        for u in range(total_units + 1):
            if not (yield W(lambda u=u: unit_full[u % 2].try_wait_parity((u // 2) & 1))):
                return
            rec = records[u % 2]
            if rec is None:
                return
            n_kv, ntile, tail = rec
            if tail:
                nv = n0 + 2 * n_kv - 1
                if not (yield W(lambda nv=nv: slot_full[nv % K_SLOTS].try_wait_parity((nv // K_SLOTS) & 1))):
                    return
                st = slot[nv % K_SLOTS]
                if st is None or st[0] != nv or st[1] != units_per_tile:
                    log.append(f"V tail of unit {u} zeroed on stage holding {st}")
                else:
                    st[2] = True
            n0 += 2 * n_kv

    procs = [scheduler(), producer(), mma(), softmax(0), softmax(1)]
    if plant == "fixer_warp":
        procs.append(fixer())
    waits = [None] * len(procs)
    done = [False] * len(procs)

    def ready(k):
        w = waits[k]
        if w is None:
            return True
        if isinstance(w, W):
            return w.pred() or abort[0]
        return w.pred()

    def advance(k, first=False):
        w = waits[k]
        try:
            if first:
                waits[k] = next(procs[k])
            else:
                waits[k] = procs[k].send(True if w is None else bool(w.pred()))
        except StopIteration:
            done[k] = True

    def run_pipe():
        op = pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, t, u, j, s = op
        readers[s] -= 1
        if kind == "S":
            q_readers[0] -= 1
            s_tile[t] = (u, j)
        else:
            if j == 0:
                o_count[t] = [u, 1]
            elif o_count[t][0] == u:
                o_count[t][1] += 1

    for k in range(len(procs)):
        advance(k, first=True)
    for step in range(400000):
        if log:
            break
        if all(done):
            # the CTA releases tensor memory and ends
            if inflight:
                log.append(f"{len(inflight)} copies still landing when the CTA ends")
            if pipe:
                log.append(f"{len(pipe)} tensor-core products or commits still pending when the CTA "
                           "releases tensor memory")
            break
        if step == abort_at:
            abort[0] = True
        rdy = [k for k in range(len(procs)) if not done[k] and ready(k)]
        choices = [("r", k) for k in rdy] + [("c", i) for i in range(len(inflight))]
        if pipe:
            choices.append(("m", 0))
        if not choices:
            log.append("deadlock: every wait would time out")
            break
        kind, k = rng.choice(choices)
        if kind == "r":
            advance(k)
        elif kind == "m":
            run_pipe()
        else:
            c = inflight.pop(k)
            if c[0] == "q":
                if q_buf[0] is not None and q_buf[0][0] == c[1]:
                    q_buf[0][1] += 1
                q_full.complete_tx(1)
            else:
                _, s, n = c
                if slot[s] is not None and slot[s][0] == n:
                    slot[s][1] += 1
                slot_full[s].complete_tx(1)
    return log


def random_units(rng, tails=True):
    out = []
    for _ in range(rng.randint(1, 6)):
        n_kv = rng.choice([1, 1, 2, 3, 4, 6])
        out.append((n_kv, rng.choice([1, 2, 2]), tails and rng.random() < 0.5))
    return out


def run_many(runs, seed, plant=None, aborts=False):
    rng = random.Random(seed)
    bad = []
    for _ in range(runs):
        abort_at = rng.randrange(0, 400) if aborts else None
        log = simulate(random_units(rng), rng, plant, abort_at=abort_at)
        if log:
            bad.append(log[0])
    return bad


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_prefill_protocol_is_race_free(seed):
    bad = run_many(300, 5000 + seed)
    assert not bad, bad[:3]


def test_separate_zeroing_warp_races():
    bad = run_many(300, 17, plant="fixer_warp")
    assert any("V tail" in b for b in bad), bad[:3]


def test_s_parity_restarting_per_unit_is_caught():
    bad = run_many(300, 19, plant="jpar_per_unit")
    assert bad, "the model should catch a parity that restarts with every unit"



def test_q_reload_without_q_free_races():
    bad = run_many(300, 23, plant="no_q_free_wait")
    assert any("Q of unit" in b or "issued on Q buffer" in b for b in bad), bad[:3]


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_abort_at_any_moment_leaves_cleanly(seed):
    """The abort flag raised at a random step (some wait of the CTA ran out):
    every role leaves, nothing deadlocks, the tiles that are still used are
    the right ones, and when the CTA ends no copy is landing and no product
    or commit is pending."""
    bad = run_many(400, 7000 + seed, aborts=True)
    assert not bad, bad[:3]


def test_producer_leaving_without_its_copies_is_caught():
    bad = run_many(400, 29, plant="no_copy_drain", aborts=True)
    assert any("copies still landing" in b for b in bad), bad[:3]


def test_mma_leaving_without_drain_is_caught():
    bad = run_many(400, 31, plant="no_mma_drain", aborts=True)
    assert any("still pending" in b for b in bad), bad[:3]
