"""The Q/dO barriers of the d = 256 dK/dV kernel (fa_bwd_d256.cu), checked on
a model under random interleavings (host only, no GPU).

At d = 256 a 128-row Q or dO tile is 64 KB and the kernel holds one stage
of each.  Each is handled as two halves of d (128 columns), with a full and
an empty barrier per half.  Per step s (one query tile): dP = dO V^T reads
dO half 0 (k-steps 0-7) then half 1 (k-steps 8-15); S = Q K^T reads Q the
same way; once the row threads have written P, dV^T[h] += dO^T[h] P reads
dO half h and a commit releases that half; once they have written dS,
dK^T[h] += Q^T[h] dS does the same for Q.  The producer refills a half for
step s + 1 as soon as its empty barrier completes.

The model runs the TMA producer, the MMA issuer, the tensor pipe (which
executes the issued products in order, each reading its operand when it
runs), the copies in flight (which land in any order) and the row threads
as coroutines scheduled in random order.  It checks that nothing deadlocks
and that every product reads the half of the step it belongs to: a copy
that overwrote a half still to be read, or a product that ran before its
half landed, fails.  The same model with one barrier pair for all of dO,
committed after the first dV^T half instead of after both, finds the
overwrite.
"""

import random

import pytest


class _Violation(Exception):
    """A product read a half of another step."""


class _Barrier:
    """An mbarrier with one arrival per phase, waited for by phase parity."""

    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(n_steps, rng, split=True):
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    # Which step's data each half of the Q and dO buffers holds (None: empty).
    held = {("dO", 0): None, ("dO", 1): None, ("Q", 0): None, ("Q", 1): None}
    in_flight = []  # copies issued, not landed: (tensor, half, step)
    pipe = []       # products and commits issued, not yet run
    n_written = {"P": 0, "dS": 0}

    def full(t, h):
        return (t + "FULL", h if split else 0)

    def empty(t, h):
        return (t + "EMPTY", h if split else 0)

    def issue_load(t, h, s):
        in_flight.append((t, h, s))

    def producer():
        for t in ("dO", "Q"):
            for h in (0, 1):
                issue_load(t, h, 0)
        for s in range(1, n_steps):
            for t in ("dO", "Q"):
                for h in (0, 1):
                    if split or h == 0:
                        yield empty(t, h), (s - 1) & 1
                    issue_load(t, h, s)

    def copies():
        # A landed copy completes its half's full barrier; with one barrier
        # pair the barrier completes once both halves of the step landed.
        landed = {}
        while True:
            if not in_flight:
                yield None
                continue
            t, h, s = in_flight.pop(rng.randrange(len(in_flight)))
            held[(t, h)] = s
            if split:
                bar(full(t, h)).arrive()
            else:
                landed[(t, s)] = landed.get((t, s), 0) + 1
                if landed[(t, s)] == 2:
                    bar(full(t, 0)).arrive()
            yield None

    def read(t, h, s):
        if held[(t, h)] != s:
            raise _Violation(f"{t} half {h} read at step {s} held step {held[(t, h)]}")

    def tensor_pipe():
        while True:
            if not pipe:
                yield None
                continue
            op = pipe.pop(0)
            if op[0] == "read":
                read(*op[1:])
            else:
                bar(op[1]).arrive()
            yield None

    def issuer():
        for s in range(n_steps):
            ph = s & 1
            for t, done in (("dO", "DP"), ("Q", "S")):
                for h in (0, 1):
                    if split or h == 0:
                        yield full(t, h), ph
                    pipe.append(("read", t, h, s))
                pipe.append(("commit", done))
            for t, waited in (("dO", "P"), ("Q", "DS")):
                yield waited, ph
                for h in (0, 1):
                    pipe.append(("read", t, h, s))
                    if split or h == 0:
                        pipe.append(("commit", empty(t, h)))
        pipe.append(("commit", "FINAL"))

    def threads():
        for s in range(n_steps):
            yield "S", s & 1
            n_written["P"] += 1
            bar("P").arrive()
            yield "DP", s & 1
            n_written["dS"] += 1
            bar("DS").arrive()
        yield "FINAL", 0

    finite = {"producer": producer(), "issuer": issuer(), "threads": threads()}
    endless = {"copies": copies(), "pipe": tensor_pipe()}
    waiting = dict.fromkeys(finite)
    alive = set(finite)
    while alive:
        ready = [r for r in alive
                 if waiting[r] is None or bar(waiting[r][0]).passed(waiting[r][1])]
        helpers = [r for r in endless if (r == "copies" and in_flight) or (r == "pipe" and pipe)]
        if not ready and not helpers:
            return "deadlock"
        r = rng.choice(sorted(ready) + sorted(helpers))
        if r in endless:
            next(endless[r])
            continue
        try:
            waiting[r] = next(finite[r])
        except StopIteration:
            alive.discard(r)
    return "ok"


def _outcomes(split, seed, tries=40):
    rng = random.Random(seed)
    seen = {}
    for n_steps in range(1, 7):
        for _ in range(tries):
            try:
                r = _run(n_steps, rng, split)
            except _Violation as e:
                r = "overwrite: " + str(e).split(" read")[0]
            seen[r] = seen.get(r, 0) + 1
    return seen


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_halves_of_d_are_safe_under_any_interleaving(seed):
    assert _outcomes(True, seed) == {"ok": 6 * 40}


def test_one_barrier_pair_released_early_fails_in_the_model():
    """With one empty barrier per tensor, committed after the first half's
    product only, a refill lands over the second half before it is read."""
    seen = _outcomes(False, seed=4)
    assert any(k.startswith("overwrite") for k in seen), seen
