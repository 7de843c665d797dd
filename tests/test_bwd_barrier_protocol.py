"""The barrier protocol of the d = 96/128 backward kernel (fa_bwd.cu), checked
on a model under random interleavings (host only, no GPU).

One CTA walks query tiles (steps) s = 0, 1, ... of its key tile.  Tensor
memory holds S^T (then P^T over it) and dP^T, whose columns also take dQ of
the step; shared memory holds Q in two stages, dO and the dS^T tile in one
each.  The roles meet only on mbarriers waited for by phase parity:

  producer    Q of step s into stage s % 2 once dK of step s - 2 has read
              it, dO of step s once dV of step s - 1 has;
  issuer      S^T(0), dP^T(0); then per step: once the key-row threads have
              written P^T, dV (reading P^T and dO), S^T(s + 1) over P^T;
              once they have written dS^T, dQ (reading dS^T, into dP^T's
              columns), dK (reading dS^T and Q), then dP^T(s + 1) once the
              drain has taken dQ out of those columns;
  key rows    per step: read S^T, write P^T over it, hand it back; read
              dP^T, write dS^T into shared memory, hand it back;
  drain       per step: read dQ out of tensor memory and release the columns;
  tensor pipe runs the issued products in issue order, each reading its
              operands when it runs; a commit arrives once everything issued
              before it has run.

Three hazards have no barrier of their own and rest on the issue order:
S^T(s + 1) overwrites P^T(s) after dV(s) read it; dQ(s) overwrites dP^T(s)
after the key rows read it (dQ waits for their dS^T); and the key rows
write dS^T(s + 1) over dS^T(s) once dP^T(s + 1) is in, which was issued
after dQ(s) and dK(s).  L and D enter S^T and dP^T as one more k-step whose
B operand the key rows write for the next step: -L/scale once S^T(s) has
completed and before they hand back P^T(s) (after which S^T(s + 1) is
issued), -D once dP^T(s) has completed and before they hand back dS^T(s).
The model checks every read, and finds the slips it should: dP^T(s + 1)
issued without waiting for the drain, dK(s) issued after dP^T(s + 1), dO
released before dV has run, and the next step's -L/scale written before
S^T(s) has read the slot.
"""

import random

import pytest


class _Violation(Exception):
    """A role or product read data of another step."""


class _Barrier:
    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1

    def passed(self, parity):
        return (self.phase & 1) != parity


NQ = 2


def _run(n_steps, rng, dq_free_wait=True, dk_before_dp=True, do_empty_after_dv=True,
         aug_early=False):
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    col_s = [None]      # ("S", s) or ("P", s)
    col_dp = [None]     # ("dP", s) or ("dQ", s)
    ds_smem = [None]    # step of the dS^T tile
    q_stage = dict.fromkeys(range(NQ))
    do_stage = [None]
    aug_l = [None]      # step whose -L/scale rows are in slot 1 of the extra k-step's tile
    aug_d = [None]      # step whose -D rows are in slot 2
    in_flight = []      # ("Q", stage, s) or ("dO", 0, s)
    pipe = []

    def expect(cond, what):
        if not cond:
            raise _Violation(what)

    def producer():
        for s in range(n_steps):
            if s >= NQ:
                yield ("QEMPTY", s % NQ), ((s // NQ) - 1) & 1
            in_flight.append(("Q", s % NQ, s))
            if s >= 1:
                yield "DOEMPTY", (s - 1) & 1
            in_flight.append(("dO", 0, s))

    def copies():
        while True:
            if in_flight:
                t, st, s = in_flight.pop(rng.randrange(len(in_flight)))
                if t == "Q":
                    q_stage[st] = s
                    bar(("QFULL", st)).arrive()
                else:
                    do_stage[0] = s
                    bar("DOFULL").arrive()
            yield None

    def tensor_pipe():
        while True:
            if pipe:
                op = pipe.pop(0)
                kind, s = op[0], op[1]
                if kind == "S":
                    expect(q_stage[s % NQ] == s, f"S^T({s}) read Q of {q_stage[s % NQ]}")
                    expect(aug_l[0] == s, f"S^T({s}) read -L/scale of {aug_l[0]}")
                    col_s[0] = ("S", s)
                elif kind == "dP":
                    expect(do_stage[0] == s, f"dP^T({s}) read dO of {do_stage[0]}")
                    expect(aug_d[0] == s, f"dP^T({s}) read -D of {aug_d[0]}")
                    col_dp[0] = ("dP", s)
                elif kind == "dV":
                    expect(col_s[0] == ("P", s), f"dV({s}) read {col_s[0]}")
                    expect(do_stage[0] == s, f"dV({s}) read dO of {do_stage[0]}")
                elif kind == "dQ":
                    expect(ds_smem[0] == s, f"dQ({s}) read dS^T of {ds_smem[0]}")
                    col_dp[0] = ("dQ", s)
                elif kind == "dK":
                    expect(ds_smem[0] == s, f"dK({s}) read dS^T of {ds_smem[0]}")
                    expect(q_stage[s % NQ] == s, f"dK({s}) read Q of {q_stage[s % NQ]}")
                elif kind == "commit":
                    bar(s).arrive()
            yield None

    def issuer():
        def issue_s(s):
            yield ("QFULL", s % NQ), (s // NQ) & 1
            pipe.append(("S", s))
            pipe.append(("commit", "S"))

        def issue_dp(s):
            if s > 0 and dq_free_wait:
                yield "DQFREE", (s - 1) & 1
            yield "DOFULL", s & 1
            pipe.append(("dP", s))
            pipe.append(("commit", "DP"))

        if n_steps == 0:
            return
        yield "AUG0", 0
        yield from issue_s(0)
        yield from issue_dp(0)
        for s in range(n_steps):
            yield "P", s & 1
            if not do_empty_after_dv:
                bar("DOEMPTY").arrive()  # mutation: released before dV has run
            pipe.append(("dV", s))
            if do_empty_after_dv:
                pipe.append(("commit", "DOEMPTY"))
            if s + 1 < n_steps:
                yield from issue_s(s + 1)
            yield "DS", s & 1
            pipe.append(("dQ", s))
            pipe.append(("commit", "DQFULL"))
            if dk_before_dp:
                pipe.append(("dK", s))
                pipe.append(("commit", ("QEMPTY", s % NQ)))
                if s == n_steps - 1:
                    pipe.append(("commit", "FINAL"))
                if s + 1 < n_steps:
                    yield from issue_dp(s + 1)
            else:
                # mutation: dK after the next dP^T
                if s + 1 < n_steps:
                    yield from issue_dp(s + 1)
                pipe.append(("dK", s))
                pipe.append(("commit", ("QEMPTY", s % NQ)))
                if s == n_steps - 1:
                    pipe.append(("commit", "FINAL"))

    def key_rows():
        if n_steps:
            aug_l[0] = aug_d[0] = 0
            bar("AUG0").arrive()
        for s in range(n_steps):
            if aug_early and s + 1 < n_steps:
                aug_l[0] = s + 1  # mutation: before S^T(s) has read the slot
            yield "S", s & 1
            expect(col_s[0] == ("S", s), f"key rows read {col_s[0]} as S^T({s})")
            col_s[0] = ("P", s)
            if s + 1 < n_steps:
                aug_l[0] = s + 1  # the next step's -L/scale, before P(s) is handed back
            bar("P").arrive()
            yield "DP", s & 1
            expect(col_dp[0] == ("dP", s), f"key rows read {col_dp[0]} as dP^T({s})")
            ds_smem[0] = s
            if s + 1 < n_steps:
                aug_d[0] = s + 1  # the next step's -D, before dS^T(s) is handed back
            bar("DS").arrive()
        if n_steps:
            yield "FINAL", 0

    def drain():
        for s in range(n_steps):
            yield "DQFULL", s & 1
            expect(col_dp[0] == ("dQ", s), f"drain read {col_dp[0]} as dQ({s})")
            bar("DQFREE").arrive()

    finite = {"producer": producer(), "issuer": issuer(), "key_rows": key_rows(),
              "drain": drain()}
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


def _outcomes(seed, tries=40, **kw):
    rng = random.Random(seed)
    seen = {}
    for n_steps in range(1, 8):
        for _ in range(tries):
            try:
                r = _run(n_steps, rng, **kw)
            except _Violation as e:
                r = str(e).split("(")[0] + " violation"
            seen[r] = seen.get(r, 0) + 1
    return seen


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_protocol_is_safe_under_any_interleaving(seed):
    assert _outcomes(seed) == {"ok": 7 * 40}


def test_next_dp_without_waiting_for_the_drain_fails_in_the_model():
    seen = _outcomes(4, dq_free_wait=False)
    assert any(k != "ok" for k in seen), seen


def test_dk_after_the_next_dp_fails_in_the_model():
    """The key rows may overwrite dS^T(s) once dP^T(s + 1) is in only
    because dK(s) was issued before it."""
    seen = _outcomes(5, dk_before_dp=False)
    assert any(k != "ok" for k in seen), seen


def test_do_released_before_dv_fails_in_the_model():
    seen = _outcomes(6, do_empty_after_dv=False)
    assert any(k != "ok" for k in seen), seen


def test_next_steps_l_rows_written_before_s_was_read_fails_in_the_model():
    """The key rows write the next step's -L/scale rows only after the S^T
    they wait for has completed; written at the top of the step instead,
    S^T can read them."""
    seen = _outcomes(7, aug_early=True)
    assert any(k != "ok" for k in seen), seen
