"""Model check of the split-K slot handshake of the GEMM kernel's epilogue.

The split-K reduce-scatter in `fp8_gemm_kernel` (csrc/dg_gemm_kernel.cuh, epilogue, `split > 1`)
moves partial accumulator rows between the CTAs of a cluster.  Which warps send and receive
changes from unit to unit (ownership follows the unit's valid rows V), so the kernel guards the
single-buffered receive slots with:

* per CTA and per peer CTA o, a slot-free barrier: one arrival from o once o has read all of a
  unit's data, plus one local arrival from each epilogue warp made after its own wait;
* before sending unit k, every epilogue warp waits for the unit k - 1 phase of all its slot-free
  barriers;
* per TMEM lane quadrant, a receive barrier: the receiving warp arrives with the expected byte
  count, the peers' copies complete it;
* after its unit, each epilogue warp arrives on a unit-done barrier and waits for all of them;
  then one thread arrives on every peer's slot-free barrier for this CTA;
* a CTA's last unit is different: its rows travel as whole padded rows by bulk copy, every
  epilogue warp waits (unit-done barrier) until all of them have staged their rows, then waits
  for the receive barriers of every quadrant holding rows this CTA owns, arrives on the
  cluster-wide exit barrier and adds and stores a share of those rows; nothing is sent
  afterwards, so the handshake is skipped;
* a CTA's first unit skips the slot-free waits (they are for the phase before the barriers'
  first, which counts as complete).

Copies are asynchronous: a send is issued by its warp and lands later, in any order, through a
separate process.  This test runs the protocol under random interleavings with the mbarrier
semantics (phase, pending arrivals, transaction count, parity waits) and checks that no receive
slot is overwritten while it is read, that every read sees the current unit's data, that no
copy is still in flight when the exit barrier completes (a CTA may leave then, and a copy
landing in or reading from its shared memory afterwards would be lost), and that nothing
deadlocks.  Three planted mistakes (no unit-done wait; no local arrivals; an exit arrival made
before the receive waits) must be caught, which shows that the checker can see each failure
kind.
"""
import random

import pytest


class Bar:
    """One mbarrier: phase counter, pending arrivals, transaction bytes."""

    completions = 0   # phases completed by any barrier (the scheduler's progress measure)

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.phase = 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count
            Bar.completions += 1

    def arrive(self, expect_tx=0):
        self.tx += expect_tx
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def try_wait(self, parity):
        # waiting on `parity` succeeds once the phase with that parity has completed
        return (self.phase & 1) != parity


class Deadlock(AssertionError):
    pass


class DataRace(AssertionError):
    pass


class LostCopy(AssertionError):
    pass


def run_protocol(split, units, seed, *, unit_done_wait=True, local_arrivals=True, early_exit_arrive=False,
                 bn=4, recv_row=5):
    """units: V per unit (0 = a zero unit, skipped by every CTA).  Returns the step count."""
    rng = random.Random(seed)
    in_flight = []                 # issued copies that have not landed: (dest CTA, quadrant, key, unit, bytes)
    exit_bar = {"arrived": 0, "done": False}
    n_epi = split * 4
    W, ACC = 4, 2
    ctas = [dict(free=[Bar(1 + (W if local_arrivals else 0)) for _ in range(split)], done=Bar(W),
                 recv=[Bar(1) for _ in range(4)], tfull=[Bar(1) for _ in range(ACC)],
                 tempty=[Bar(W) for _ in range(ACC)], slots={}) for _ in range(split)]
    live_units = [u for u, v in enumerate(units) if v > 0]
    last = live_units[-1] if live_units else -1
    last_any = len(units) - 1          # the kernel's `u + u_step >= total_units`

    def exit_arrive():
        exit_bar["arrived"] += 1
        if exit_bar["arrived"] == n_epi:
            exit_bar["done"] = True
            if in_flight:
                raise LostCopy(f"exit barrier complete with {len(in_flight)} copies in flight (split {split})")

    def lander():
        # lands the issued copies one at a time, in random order
        while True:
            if in_flight:
                o, q, key, u, nbytes = in_flight.pop(rng.randrange(len(in_flight)))
                prev = ctas[o]["slots"].get(key)
                if prev is not None and prev[1] == "reading":
                    raise DataRace(f"CTA {o} slot {key} overwritten while read (unit {u})")
                ctas[o]["slots"][key] = (u, "written")
                ctas[o]["recv"][q].complete_tx(nbytes)
            elif all_epilogues_done[0]:
                return
            yield

    all_epilogues_done = [False]

    def mma(c):
        X = ctas[c]
        acc, ph = 0, 0
        for u in live_units:
            while not X["tempty"][acc].try_wait(ph ^ 1):
                yield
            for _ in range(rng.randint(0, 3)):
                yield
            X["tfull"][acc].arrive()
            acc += 1
            if acc == ACC:
                acc, ph = 0, ph ^ 1

    def epilogue(c, q):
        X = ctas[c]
        acc, acc_ph, free_ph, done_ph, recv_mask = 0, 0, 0, 0, 0
        for u in live_units:
            V = units[u]
            last_unit = u == last_any
            row_bytes = recv_row if last_unit else bn
            rpo = (V + split - 1) // split
            cap = (128 + split - 1) // split
            q0 = 32 * q
            own0 = min(V, c * rpo)
            own1 = min(V, own0 + rpo)
            ro0, ro1 = max(own0, q0), min(own1, q0 + 32)
            sends = [r for r in range(q0, q0 + 32) if r < V and r // rpo != c]
            while not X["tfull"][acc].try_wait(acc_ph):
                yield
            if u != live_units[0]:
                for o in range(split):
                    if o != c:
                        while not X["free"][o].try_wait(free_ph ^ 1):
                            yield
            free_ph ^= 1
            if local_arrivals:
                for o in range(split):
                    if o != c:
                        X["free"][o].arrive()
            for r in sends:                     # st.async rows, or bulk runs of rows: issued here, landing later
                o = r // rpo
                key = (c if c < o else c - 1, r - o * rpo)
                assert key[1] < cap
                in_flight.append((o, q, key, u, row_bytes))
                yield
            qr0 = own0 // 32
            qr1 = (own1 - 1) // 32 + 1 if own1 > own0 else qr0
            if last_unit:
                if ro0 < ro1:
                    X["recv"][q].arrive((split - 1) * (ro1 - ro0) * row_bytes)
                X["tempty"][acc].arrive()
                X["done"].arrive()
                if unit_done_wait:
                    while not X["done"].try_wait(done_ph):
                        yield
                done_ph ^= 1
                if early_exit_arrive:
                    exit_arrive()
                for qq in range(qr0, qr1):
                    while not X["recv"][qq].try_wait((recv_mask >> qq) & 1):
                        yield
                for qq in range(qr0, qr1):
                    recv_mask ^= 1 << qq
                if not early_exit_arrive:
                    exit_arrive()
                # this warp's share of the owned rows, every partial of each
                keys = [(sl, r - own0) for r in range(own0, own1) if (r - own0) % W == q for sl in range(split - 1)]
                for k in keys:
                    got = X["slots"].get(k, (None,))[0]   # (None: nothing has landed there yet)
                    if got != u:
                        raise DataRace(f"CTA {c} read unit {got} data in unit {u}")
                for _ in range(rng.randint(0, 4)):
                    yield
                continue
            if ro0 < ro1:
                X["recv"][q].arrive((split - 1) * (ro1 - ro0) * row_bytes)
                while not X["recv"][q].try_wait((recv_mask >> q) & 1):
                    yield
                keys = [(sl, r - own0) for r in range(ro0, ro1) for sl in range(split - 1)]
                for k in keys:
                    got = X["slots"].get(k, (None,))[0]   # (None: nothing has landed there yet)
                    if got != u:
                        raise DataRace(f"CTA {c} read unit {got} data in unit {u}")
                    X["slots"][k] = (u, "reading")
                for _ in range(rng.randint(0, 4)):
                    yield
                for k in keys:
                    X["slots"][k] = (u, "read")
            for qq in range(qr0, qr1):
                recv_mask ^= 1 << qq
            X["tempty"][acc].arrive()
            acc += 1
            if acc == ACC:
                acc, acc_ph = 0, acc_ph ^ 1
            X["done"].arrive()
            if unit_done_wait:
                while not X["done"].try_wait(done_ph):
                    yield
            done_ph ^= 1
            if q == 0:
                for rk in range(split):
                    if rk != c:
                        ctas[rk]["free"][c].arrive()
                        yield

    procs = []
    for c in range(split):
        procs.append(mma(c))
        procs += [epilogue(c, q) for q in range(W)]
    epi_ids = {i for i in range(len(procs)) if i % (W + 1) != 0}
    procs.append(lander())
    live = list(range(len(procs)))
    steps = stalled = 0
    seen = Bar.completions
    while live:
        i = rng.choice(live)
        if Bar.completions != seen:      # a barrier phase completed: progress
            seen = Bar.completions
            stalled = 0
        try:
            next(procs[i])
        except StopIteration:
            live.remove(i)
            if not (epi_ids & set(live)):
                all_epilogues_done[0] = True
            stalled = 0
            continue
        steps += 1
        stalled += 1
        if stalled > 50000:
            raise Deadlock(f"no progress (split {split}, units {units})")
    return steps


def _cases(n, seed0):
    rng = random.Random(seed0)
    for i in range(n):
        split = rng.randint(2, 8)
        units = [rng.choice([0, 1, 2, 17, 31, 32, 33, 64, 71, 100, 127, 128, rng.randint(1, 128)])
                 for _ in range(rng.randint(1, 7))]
        yield i, split, units


def test_handshake_holds_under_random_interleavings():
    for i, split, units in _cases(120, 0):
        run_protocol(split, units, seed=i)


@pytest.mark.parametrize("mutation", ["no_unit_done_wait", "no_local_arrivals", "early_exit_arrive"])
def test_checker_catches_planted_mistakes(mutation):
    kw = {"no_unit_done_wait": {"unit_done_wait": False}, "no_local_arrivals": {"local_arrivals": False},
          "early_exit_arrive": {"early_exit_arrive": True}}[mutation]
    caught = 0
    for i, split, units in _cases(120, 1):
        try:
            run_protocol(split, units, seed=i, **kw)
        except (Deadlock, DataRace, LostCopy, AssertionError):
            caught += 1
    assert caught > 0, f"the checker did not see the planted mistake ({mutation})"
