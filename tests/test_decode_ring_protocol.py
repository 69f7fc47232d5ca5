"""Model check of the decode kernel's tile-ring protocol (CPU only).

The decode split kernel streams K/V tiles through a ring of kStages shared-
memory stages: one producer (a TMA-issuing lane) and kConsumers consumer
warps, a `full` and an `empty` mbarrier per stage, tiles of an item dealt
round-robin to the warps, the ring running on across items.  Parity tests
cannot catch a synchronisation race, so this file simulates the protocol under
random schedules -- random interleaving of the producer and the warps, and
bulk copies that complete in any order -- with the mbarrier semantics of PTX:

  * a phase completes when its pending arrival count and its transaction
    count are both zero;
  * `try_wait.parity P` succeeds when the barrier's current (open) phase has a
    parity other than P, i.e. whenever the phase before the open one has P.

It checks that every consumer reads a stage only after the tile it waits for
has fully landed there, that the producer never refills a stage that is
being read or still landing, that no phase gets more arrivals than its count,
that nothing deadlocks, and that no copy is in flight when the CTA ends.

The kernel's protocol (a consumer first waits for the release of the stage's
previous tile, then for its own tile's phase) passes for every (consumers,
stages) pair the kernel's static assertion admits; the parity-only wait that
an earlier version of the kernel used, and the fixed wait on a ring that the
assertion rejects, are both caught.
"""
import random

import pytest


class Bar:
    """An mbarrier: expected arrivals per phase, pending arrivals and
    transaction bytes of the open phase, and the number of completed phases."""

    def __init__(self, count, log):
        self.count, self.pending, self.tx, self.phase, self.log = count, count, 0, 0, log

    def _settle(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        if self.pending == 0:
            self.log.append("arrival beyond the phase's count")
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


def simulate(items, consumers, stages, fixed, rng, units_per_tile=2, queue=2):
    """Run one random schedule; returns the list of violations (empty: clean)."""
    log = []
    full = [Bar(1, log) for _ in range(stages)]
    empty = [Bar(1, log) for _ in range(stages)]
    content = [None] * stages          # (tile, landed units) the stage holds
    reader = [None] * stages           # warp reading the stage
    inflight = []                      # (stage, tile) per copy unit
    state = {"published": 0, "merged": 0, "at_merge": 0}

    def producer():
        g = 0
        for seq, n in enumerate(items):
            if seq >= queue:           # the item queue entry was used two items ago
                yield lambda s=seq: state["merged"] > s - queue
            state["published"] = seq + 1
            for _ in range(n):
                s = g % stages
                if g >= stages:
                    yield lambda s=s, g=g: empty[s].try_wait_parity(((g // stages) - 1) & 1)
                if reader[s] is not None:
                    log.append(f"stage {s} refilled with tile {g} while warp {reader[s]} reads it")
                if any(st == s for st, _ in inflight):
                    log.append(f"stage {s} refilled with tile {g} while an earlier copy lands")
                full[s].arrive_expect_tx(units_per_tile)
                content[s] = [g, 0]
                inflight.extend([(s, g)] * units_per_tile)
                g += 1
                yield None
        # drain: the last stages' copies have landed before the CTA leaves
        for j in range(max(0, g - stages), g):
            yield lambda j=j: full[j % stages].try_wait_parity((j // stages) & 1)

    def consumer(w):
        g0 = 0
        for seq, n in enumerate(items):
            yield lambda s=seq: state["published"] > s
            for i in range(w, n, consumers):
                gt = g0 + i
                s = gt % stages
                if fixed and gt >= stages:
                    yield lambda s=s, gt=gt: empty[s].try_wait_parity(((gt // stages) - 1) & 1)
                yield lambda s=s, gt=gt: full[s].try_wait_parity((gt // stages) & 1)
                if content[s] != [gt, units_per_tile]:
                    log.append(f"warp {w} read stage {s} as tile {gt} holding {content[s]}")
                reader[s] = w
                yield None
                if content[s] is None or content[s][0] != gt:
                    log.append(f"stage {s} changed under warp {w} reading tile {gt}")
                reader[s] = None
                empty[s].arrive()
                yield None
            # merge barrier of the consumer warps
            state["at_merge"] += 1
            yield lambda s=seq: state["at_merge"] >= consumers * (s + 1)
            if w == 0:
                state["merged"] = seq + 1
            g0 += n

    procs = [producer()] + [consumer(w) for w in range(consumers)]
    waits = [None] * len(procs)
    done = [False] * len(procs)

    def advance(k):
        try:
            waits[k] = next(procs[k])
        except StopIteration:
            done[k] = True

    for k in range(len(procs)):
        advance(k)
    for _ in range(200000):
        if log:
            break
        ready = [k for k in range(len(procs))
                 if not done[k] and (waits[k] is None or waits[k]())]
        choices = [("p", k) for k in ready] + [("c", i) for i in range(len(inflight))]
        if not choices:
            if not all(done):
                log.append("deadlock: every wait would time out")
            break
        kind, k = rng.choice(choices)
        if kind == "p":
            advance(k)
        else:
            s, g = inflight.pop(k)
            if content[s] is not None and content[s][0] == g:
                content[s][1] += 1
            full[s].complete_tx(1)
    if not log and inflight:
        log.append(f"{len(inflight)} copies still landing when the CTA ends")
    return log


def random_items(rng):
    # items of 1..9 tiles (empty items never reach the ring), with many
    # one-tile items so that a warp can sit out whole items
    return [rng.choice([1, 1, 2, 3, 4, 5, 7, 9]) for _ in range(rng.randint(1, 7))]


def run_many(consumers, stages, fixed, runs, seed):
    rng = random.Random(seed)
    bad = []
    for _ in range(runs):
        log = simulate(random_items(rng), consumers, stages, fixed, rng)
        if log:
            bad.append(log[0])
    return bad


@pytest.mark.parametrize("consumers,stages", [(2, 3), (1, 2), (1, 3), (2, 2), (2, 4), (3, 3), (3, 6)])
def test_ring_protocol_is_race_free(consumers, stages):
    assert (2 * stages) % consumers == 0       # the kernel's static assertion
    bad = run_many(consumers, stages, fixed=True, runs=400, seed=1000 + 10 * consumers + stages)
    assert not bad, bad[:3]


def test_parity_only_wait_reads_unlanded_tiles():
    # the earlier protocol: each warp waited on full[stage] by parity alone
    bad = run_many(2, 3, fixed=False, runs=400, seed=7)
    assert any("read stage" in b for b in bad), bad[:3]


def test_ring_rejected_by_the_static_assertion_races():
    # 4 warps on 3 stages: 2*3 % 4 != 0, so even the release wait can pass on
    # a stale phase
    assert (2 * 3) % 4 != 0
    bad = run_many(4, 3, fixed=True, runs=400, seed=11)
    assert bad, "the model should find a race on a ring the kernel refuses"
