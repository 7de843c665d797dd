"""The barrier protocol of the one-tile forward (fa_fwd_tile1.cu: the forward
at d = 256, and at 128 query rows per CTA for the other head dimensions),
checked on a model under random interleavings (host only, no GPU).

One CTA owns one query tile.  Key tiles j = 0, 1, ... stream through K and
V ring stages j % NS; S_j goes into tensor-memory buffer j % 3 and P_j is
written over it.  The roles meet only on mbarriers waited for by phase
parity:

  producer    K_j and V_j once the products of tile j - NS have read their
              stages;
  issuer      S_0, S_1; then per key tile: once the softmax has written P_j,
              O += P_j V_j, then S_{j+2} into buffer (j + 2) % 3, whose P_{j-1}
              the previous product read;
  softmax     per key tile: read S_j, write P_j over it; when the running
              maximum grows, rescale O, which first waits for every product
              before it (the per-tile barrier, waited for at phase j - 1);
              at the end, wait for a barrier committed once after the last
              product;
  tensor pipe runs the issued products in issue order, each reading its
              operands when it runs; a commit arrives once everything issued
              before it has run.

The rescale's wait is unambiguous only because S_j, which the softmax has
waited for, was issued after O += P_{j-2} V_{j-2}: the per-tile barrier is
then at most one phase behind.  The model checks every read and the O
contributions seen at each rescale and at the epilogue; it fails as it
should when S_{j+2} is issued before O += P_j V_j (the rescale can then see
O two products short), or when the epilogue waits on the per-tile barrier
instead of the final one.
"""

import random

import pytest


class _Violation(Exception):
    """A role or product saw data of another key tile."""


class _Barrier:
    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1

    def passed(self, parity):
        return (self.phase & 1) != parity


NB = 3


def _run(n_kv, ns, rng, s_after_pv=True, final_barrier=True):
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    buf = dict.fromkeys(range(NB))   # ("S", j) or ("P", j)
    k_stage = dict.fromkeys(range(ns))
    v_stage = dict.fromkeys(range(ns))
    o_done = [0]                     # products O += P V that have run
    in_flight = []
    pipe = []

    def expect(cond, what):
        if not cond:
            raise _Violation(what)

    def producer():
        for j in range(n_kv):
            if j >= ns:
                yield ("KEMPTY", j % ns), ((j // ns) - 1) & 1
            in_flight.append(("K", j % ns, j))
            if j >= ns:
                yield ("VEMPTY", j % ns), ((j // ns) - 1) & 1
            in_flight.append(("V", j % ns, j))

    def copies():
        while True:
            if in_flight:
                t, st, j = in_flight.pop(rng.randrange(len(in_flight)))
                (k_stage if t == "K" else v_stage)[st] = j
                bar((t + "FULL", st)).arrive()
            yield None

    def tensor_pipe():
        while True:
            if pipe:
                op = pipe.pop(0)
                kind, j = op[0], op[1]
                if kind == "S":
                    expect(k_stage[j % ns] == j, f"S_{j} read K of {k_stage[j % ns]}")
                    buf[j % NB] = ("S", j)
                elif kind == "PV":
                    expect(buf[j % NB] == ("P", j), f"PV_{j} read {buf[j % NB]}")
                    expect(v_stage[j % ns] == j, f"PV_{j} read V of {v_stage[j % ns]}")
                    o_done[0] += 1
                elif kind == "commit":
                    bar(j).arrive()
            yield None

    def issuer():
        def issue_s(j):
            yield ("KFULL", j % ns), (j // ns) & 1
            pipe.append(("S", j))
            pipe.append(("commit", ("SFULL", j % NB)))
            pipe.append(("commit", ("KEMPTY", j % ns)))

        yield "QFULL", 0
        for j in range(min(n_kv, 2)):
            yield from issue_s(j)
        for j in range(n_kv):
            if not s_after_pv and j + 2 < n_kv:
                yield from issue_s(j + 2)  # mutation: before O += P_j V_j
            yield ("VFULL", j % ns), (j // ns) & 1
            yield ("PFULL", j % NB), (j // NB) & 1
            pipe.append(("PV", j))
            pipe.append(("commit", "ODONE"))
            pipe.append(("commit", ("VEMPTY", j % ns)))
            if j == n_kv - 1:
                pipe.append(("commit", "FINAL"))
            if s_after_pv and j + 2 < n_kv:
                yield from issue_s(j + 2)

    def softmax():
        for j in range(n_kv):
            yield ("SFULL", j % NB), (j // NB) & 1
            expect(buf[j % NB] == ("S", j), f"softmax read {buf[j % NB]} as S_{j}")
            buf[j % NB] = ("P", j)
            if j > 0 and rng.random() < 0.5:  # the running maximum grew
                yield "ODONE", (j - 1) & 1
                expect(o_done[0] == j, f"rescale at tile {j} saw {o_done[0]} products")
            bar(("PFULL", j % NB)).arrive()
        if n_kv:
            if final_barrier:
                yield "FINAL", 0
            else:
                yield "ODONE", (n_kv - 1) & 1
            expect(o_done[0] == n_kv, f"epilogue saw {o_done[0]} of {n_kv} products")

    bar("QFULL").arrive()
    finite = {"producer": producer(), "issuer": issuer(), "softmax": softmax()}
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


def _outcomes(ns, seed, tries=40, **kw):
    rng = random.Random(seed)
    seen = {}
    for n_kv in range(1, 10):
        for _ in range(tries):
            try:
                r = _run(n_kv, ns, rng, **kw)
            except _Violation as e:
                r = str(e).split(" ")[0] + " violation"
            seen[r] = seen.get(r, 0) + 1
    return seen


@pytest.mark.parametrize("ns", [2, 4])
@pytest.mark.parametrize("seed", [1, 2])
def test_protocol_is_safe_under_any_interleaving(ns, seed):
    assert _outcomes(ns, seed) == {"ok": 9 * 40}


@pytest.mark.parametrize("ns", [2, 4])
def test_next_s_before_the_product_fails_in_the_model(ns):
    seen = _outcomes(ns, 3, s_after_pv=False)
    assert any(k != "ok" for k in seen), seen


@pytest.mark.parametrize("ns", [2, 4])
def test_epilogue_on_the_per_tile_barrier_fails_in_the_model(ns):
    seen = _outcomes(ns, 4, final_barrier=False)
    assert any(k != "ok" for k in seen), seen
