"""The barrier protocols of the two-tile forward (fa_fwd.cu), checked on a
model under random interleavings (host only, no GPU).

At d = 64 three S buffers of tensor memory rotate between the CTA's two
query tiles A and B (the n-th S issued goes to buffer n % 3, P is written
over its own S), and one thread issues the products in the order
S_A(0) S_B(0) S_A(1), then per key tile j: O_A += P_A V_j, S_B(j+1),
O_B += P_B V_j, S_A(j+2).  The kernel's roles meet only on mbarriers waited
for by phase parity, which cannot tell phase k from phase k + 2.  So every
barrier must be at most one phase from each of its waiters whatever the
timing: a softmax warpgroup may run ahead of the MMA issuer (say while the
issuer waits for a late V tile), and the tensor pipe may lag the issuer.

The model runs the four roles (the TMA producer's K/V ring, the MMA issuer,
the two softmax warpgroups) as coroutines scheduled in random order.  An
issued product completes at once, the earliest the tensor pipe could.  It
checks that nothing deadlocks and that every role sees what it waits for:
the softmax the right S, the issuer the right P, the rescale and the
epilogue every product before them.  The same model with the former
per-tile P barrier and per-tile epilogue wait finds both failures, which
is why the kernel has one P barrier per S buffer and a barrier committed
once after each tile's last P V.

At d = 96 and 128 (and in the FP8 forward) each tile has its own S
buffer and the order is S_A(0) S_B(0), then per key tile j: O_A += P_A V_j,
S_A(j+1), O_B += P_B V_j, S_B(j+1).  There a tile's next S follows its own
P V, so per-tile barriers suffice; the second model checks that too.
"""

import random

import pytest


class _Violation(Exception):
    """A role saw something other than what it waited for."""


def _check(cond, what):
    if not cond:
        raise _Violation(what)


class _Barrier:
    """An mbarrier with one arrival per phase: wait(parity) returns once the
    phase of that parity has completed, i.e. the current phase's parity
    differs."""

    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(nA, nB, rng, per_buffer_p=True, final_barrier=True, stages=4):
    n_kv = max(nA, nB)
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    def snum(x, j):  # S_x(j) is the n-th S issued
        return min(j + x, nA) + min(j, nB)

    issued_s = []     # (tile, key tile) of each S issued, in order
    p_written = {}    # buffer or tile -> P arrivals
    pv_done = [0, 0]  # completed O += P V per tile

    def producer():
        for j in range(n_kv):
            st, ph = j % stages, ((j // stages) - 1) & 1
            if j >= stages:
                yield ("KEMPTY", st), ph
            bar(("KFULL", st)).arrive()
            if j >= stages:
                yield ("VEMPTY", st), ph
            bar(("VFULL", st)).arrive()

    def issuer():
        k_waited = [0]

        def s(x, j):
            if j >= k_waited[0]:
                yield ("KFULL", j % stages), (j // stages) & 1
                k_waited[0] = j + 1
            issued_s.append((x, j))
            bar(("SFULL", snum(x, j) % 3)).arrive()
            if x == 1 or j >= nB:
                bar(("KEMPTY", j % stages)).arrive()

        def pv(x, j):
            st = j % stages
            if x == 0 or j >= nA:
                yield ("VFULL", st), (j // stages) & 1
            n = snum(x, j)
            if per_buffer_p:
                yield ("PFULL", n % 3), (n // 3) & 1
                _check(p_written.get(n % 3, 0) == n // 3 + 1, "P of another S")
            else:
                yield ("PFULL", x), j & 1
                _check(p_written.get(x, 0) == j + 1, "P of another step")
            pv_done[x] += 1
            bar(("ODONE", x)).arrive()
            if j == (nA, nB)[x] - 1:
                bar(("OFIN", x)).arrive()
            if x == 1 or j >= nB:
                bar(("VEMPTY", st)).arrive()

        if nA > 0:
            yield from s(0, 0)
        if nB > 0:
            yield from s(1, 0)
        if nA > 1:
            yield from s(0, 1)
        for j in range(n_kv):
            if j < nA:
                yield from pv(0, j)
            if j + 1 < nB:
                yield from s(1, j + 1)
            if j < nB:
                yield from pv(1, j)
            if j + 2 < nA:
                yield from s(0, j + 2)

    def softmax(x):
        nt = (nA, nB)[x]
        for j in range(nt):
            n = snum(x, j)
            yield ("SFULL", n % 3), (n // 3) & 1
            _check(issued_s[n] == (x, j), "softmax read another tile's S")
            if j > 0 and rng.random() < 0.5:  # the row maximum grew: rescale O
                yield ("ODONE", x), (j - 1) & 1
                _check(pv_done[x] >= j, "O rescaled before its last P V")
            key = n % 3 if per_buffer_p else x
            p_written[key] = p_written.get(key, 0) + 1
            bar(("PFULL", key)).arrive()
        if nt > 0:
            if final_barrier:
                yield ("OFIN", x), 0
            else:
                yield ("ODONE", x), (nt - 1) & 1
            _check(pv_done[x] == nt, "epilogue before the last P V")

    roles = {"producer": producer(), "issuer": issuer(), "A": softmax(0), "B": softmax(1)}
    waiting = dict.fromkeys(roles)
    alive = set(roles)
    while alive:
        ready = [r for r in alive if waiting[r] is None or bar(waiting[r][0]).passed(waiting[r][1])]
        if not ready:
            return "deadlock"
        r = rng.choice(sorted(ready))
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.discard(r)
    return "ok"


def _outcomes(per_buffer_p, final_barrier, seed, tries=60):
    rng = random.Random(seed)
    seen = {}
    for nA in range(8):
        for nB in range(8):
            for _ in range(tries):
                try:
                    r = _run(nA, nB, rng, per_buffer_p, final_barrier)
                except _Violation as e:
                    r = str(e)
                seen[r] = seen.get(r, 0) + 1
    return seen


def _run_ping_pong(nA, nB, rng, stages=2):
    """The d = 96 / 128 order: per-tile S buffer, P barrier and P V barrier."""
    n_kv = max(nA, nB)
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    issued_s = {0: 0, 1: 0}
    p_written = [0, 0]
    pv_done = [0, 0]

    def producer():
        for j in range(n_kv):
            st, ph = j % stages, ((j // stages) - 1) & 1
            if j >= stages:
                yield ("KEMPTY", st), ph
            bar(("KFULL", st)).arrive()
            if j >= stages:
                yield ("VEMPTY", st), ph
            bar(("VFULL", st)).arrive()

    def issuer():
        def s(x, j):
            issued_s[x] += 1
            bar(("SFULL", x)).arrive()

        if n_kv > 0:
            yield ("KFULL", 0), 0
            if nA > 0:
                s(0, 0)
            if nB > 0:
                s(1, 0)
            bar(("KEMPTY", 0)).arrive()
        for j in range(n_kv):
            st = j % stages
            yield ("VFULL", st), (j // stages) & 1
            k_ready = False
            for x in (0, 1):
                if j >= (nA, nB)[x]:
                    continue
                yield ("PFULL", x), j & 1
                _check(p_written[x] == j + 1, "P of another step")
                pv_done[x] += 1
                bar(("ODONE", x)).arrive()
                if j + 1 < n_kv and j + 1 < (nA, nB)[x]:
                    if not k_ready:
                        yield ("KFULL", (j + 1) % stages), ((j + 1) // stages) & 1
                        k_ready = True
                    s(x, j + 1)
            bar(("VEMPTY", st)).arrive()
            if k_ready:
                bar(("KEMPTY", (j + 1) % stages)).arrive()

    def softmax(x):
        nt = (nA, nB)[x]
        for j in range(nt):
            yield ("SFULL", x), j & 1
            _check(issued_s[x] == j + 1, "softmax read another step's S")
            if j > 0 and rng.random() < 0.5:
                yield ("ODONE", x), (j - 1) & 1
                _check(pv_done[x] >= j, "O rescaled before its last P V")
            p_written[x] += 1
            bar(("PFULL", x)).arrive()
        if nt > 0:
            yield ("ODONE", x), (nt - 1) & 1
            _check(pv_done[x] == nt, "epilogue before the last P V")

    roles = {"producer": producer(), "issuer": issuer(), "A": softmax(0), "B": softmax(1)}
    waiting = dict.fromkeys(roles)
    alive = set(roles)
    while alive:
        ready = [r for r in alive if waiting[r] is None or bar(waiting[r][0]).passed(waiting[r][1])]
        if not ready:
            return "deadlock"
        r = rng.choice(sorted(ready))
        try:
            waiting[r] = next(roles[r])
        except StopIteration:
            alive.discard(r)
    return "ok"


@pytest.mark.parametrize("seed", [5, 6])
def test_ping_pong_order_is_safe_under_any_interleaving(seed):
    rng = random.Random(seed)
    for nA in range(8):
        for nB in range(8):
            for _ in range(60):
                try:
                    r = _run_ping_pong(nA, nB, rng)
                except _Violation as e:
                    r = str(e)
                assert r == "ok", (nA, nB, r)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_protocol_is_safe_under_any_interleaving(seed):
    assert _outcomes(True, True, seed) == {"ok": 8 * 8 * 60}


def test_per_tile_p_barrier_and_epilogue_wait_fail_in_the_model():
    """The model can tell: the earlier barriers deadlock or read O early."""
    seen = _outcomes(False, False, seed=4)
    assert seen.get("deadlock", 0) > 0
    assert seen.get("epilogue before the last P V", 0) > 0
