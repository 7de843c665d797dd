"""The barrier protocol of the dQ kernel (fa_bwd_dq.cu: the deterministic
backward's dQ, and dQ at d = 256), checked on a model under random
interleavings (host only, no GPU).

One CTA owns a query tile and walks key tiles j = 0, 1, ...  Q and dO are
loaded once; K_j goes into stage j % NSK, V_j into stage j % NSV.  Tensor
memory holds two S buffers (S_j in buffer j % 2, dS_j written over it) and
one dP buffer.  The roles meet only on mbarriers waited for by phase
parity:

  producer    K_j once dQ_{j - NSK} has read its stage, V_j once
              dP_{j - NSV} has;
  issuer      S_0, dP_0, S_1; then per key tile: dP_{j+1} once the row
              warps hold dP_j in registers; once they have written dS_j,
              dQ += dS_j K_j, then S_{j+2} over dS_j;
  row warps   per key tile: read S_j and dP_j (releasing the dP buffer),
              write dS_j over S_j, hand it back;
  tensor pipe runs the issued products in issue order, each reading its
              operands when it runs; a commit arrives once everything issued
              before it has run.

S_{j+2} overwriting dS_j rests on the issue order alone (it follows dQ_j).
The model checks every read for each stage count the kernel uses (4 and 4
stages at d = 64, 3 and 2 at d = 96/128, 2 and 1 at d = 256), and finds
S_{j+2} issued before dQ_j, dP_{j+1} issued before the row warps released
the dP buffer, and a K stage released before dQ_j has read it.
"""

import random

import pytest


class _Violation(Exception):
    """A product or the row warps read data of another key tile."""


class _Barrier:
    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(n_kv, nsk, nsv, rng, s_after_dq=True, dp_free_wait=True, k_empty_after_dq=True):
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    s_buf = {0: None, 1: None}   # ("S", j) or ("dS", j)
    dp_buf = [None]              # j of dP
    k_stage = dict.fromkeys(range(nsk))
    v_stage = dict.fromkeys(range(nsv))
    in_flight = []
    pipe = []

    def expect(cond, what):
        if not cond:
            raise _Violation(what)

    def producer():
        for j in range(n_kv):
            if j >= nsk:
                yield ("KEMPTY", j % nsk), ((j // nsk) - 1) & 1
            in_flight.append(("K", j % nsk, j))
            if j >= nsv:
                yield ("VEMPTY", j % nsv), ((j // nsv) - 1) & 1
            in_flight.append(("V", j % nsv, j))

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
                    expect(k_stage[j % nsk] == j, f"S_{j} read K of {k_stage[j % nsk]}")
                    s_buf[j % 2] = ("S", j)
                elif kind == "dP":
                    expect(v_stage[j % nsv] == j, f"dP_{j} read V of {v_stage[j % nsv]}")
                    dp_buf[0] = j
                elif kind == "dQ":
                    expect(s_buf[j % 2] == ("dS", j), f"dQ_{j} read {s_buf[j % 2]}")
                    expect(k_stage[j % nsk] == j, f"dQ_{j} read K of {k_stage[j % nsk]}")
                elif kind == "commit":
                    bar(j).arrive()
            yield None

    def issuer():
        def issue_s(j):
            yield ("KFULL", j % nsk), (j // nsk) & 1
            pipe.append(("S", j))
            pipe.append(("commit", ("SFULL", j % 2)))
            if not k_empty_after_dq:
                pipe.append(("commit", ("KEMPTY", j % nsk)))  # mutation: before dQ_j

        def issue_dp(j):
            yield ("VFULL", j % nsv), (j // nsv) & 1
            pipe.append(("dP", j))
            pipe.append(("commit", "DPFULL"))
            pipe.append(("commit", ("VEMPTY", j % nsv)))

        yield "QD", 0
        yield from issue_s(0)
        yield from issue_dp(0)
        if n_kv > 1:
            yield from issue_s(1)
        for j in range(n_kv):
            if j + 1 < n_kv:
                if dp_free_wait:
                    yield "DPFREE", j & 1
                yield from issue_dp(j + 1)
            yield ("DSREADY", j % 2), (j >> 1) & 1
            if not s_after_dq and j + 2 < n_kv:
                yield from issue_s(j + 2)  # mutation: before dQ_j
            pipe.append(("dQ", j))
            if k_empty_after_dq:
                pipe.append(("commit", ("KEMPTY", j % nsk)))
            if s_after_dq and j + 2 < n_kv:
                yield from issue_s(j + 2)
            if j == n_kv - 1:
                pipe.append(("commit", "DQDONE"))

    def rows():
        for j in range(n_kv):
            yield ("SFULL", j % 2), (j >> 1) & 1
            expect(s_buf[j % 2] == ("S", j), f"rows read {s_buf[j % 2]} as S_{j}")
            yield "DPFULL", j & 1
            expect(dp_buf[0] == j, f"rows read dP of {dp_buf[0]} as dP_{j}")
            bar("DPFREE").arrive()
            s_buf[j % 2] = ("dS", j)
            bar(("DSREADY", j % 2)).arrive()
        yield "DQDONE", 0

    bar("QD").arrive()  # Q and dO are loaded once, before the walk
    finite = {"producer": producer(), "issuer": issuer(), "rows": rows()}
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


STAGES = [(4, 4), (3, 2), (2, 1)]


def _outcomes(stages, seed, tries=30, **kw):
    rng = random.Random(seed)
    seen = {}
    for n_kv in range(1, 10):
        for _ in range(tries):
            try:
                r = _run(n_kv, *stages, rng, **kw)
            except _Violation as e:
                r = str(e).split(" ")[0] + " violation"
            seen[r] = seen.get(r, 0) + 1
    return seen


@pytest.mark.parametrize("stages", STAGES)
@pytest.mark.parametrize("seed", [1, 2])
def test_protocol_is_safe_under_any_interleaving(stages, seed):
    assert _outcomes(stages, seed) == {"ok": 9 * 30}


@pytest.mark.parametrize("stages", STAGES)
def test_s_before_dq_fails_in_the_model(stages):
    seen = _outcomes(stages, 3, s_after_dq=False)
    assert any(k != "ok" for k in seen), seen


@pytest.mark.parametrize("stages", STAGES)
def test_dp_before_the_rows_release_it_fails_in_the_model(stages):
    seen = _outcomes(stages, 4, dp_free_wait=False)
    assert any(k != "ok" for k in seen), seen


def test_k_stage_released_before_dq_fails_in_the_model():
    """With two K stages (d = 256) the refill can land before dQ_j runs."""
    seen = _outcomes((2, 1), 5, k_empty_after_dq=False)
    assert any(k != "ok" for k in seen), seen
