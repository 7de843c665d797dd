"""The barrier protocol of the d = 64 backward kernel (fa_bwd_d64.cu),
checked on a model under random interleavings (host only, no GPU).

One CTA walks query tiles s = 0, 1, ... of its key tile, each as two
64-query halves h = 2s and 2s + 1.  Its roles meet only on mbarriers waited
for by phase parity:

  producer    Q/dO of step s into ring stage s % 3, once the dV/dK products
              of step s - 3 have released it;
  issuer      S^T/dP^T of half h into TMEM buffer h % 2 (the first half of a
              step waits for its Q/dO); once the compute warps hand half h
              back: dV/dK of half h (reading its P^T/dS^T and Q/dO), then
              S^T/dP^T of half h + 2 into the same buffer, then, after a
              step's second half, dQ of step s (reading the dS^T tile of
              shared-memory buffer s % 2) once the drain has taken dQ of
              step s - 1 out of TMEM;
  compute     per half: wait for its S^T/dP^T and its L/D ring slot, write
              P^T/dS^T over the buffer and dS^T into shared-memory buffer
              s % 2, hand the half back and release the slot;
  drain       fills the six-slot L/D ring, and per step takes dQ out of TMEM
              (releasing the columns) and refills the slots of step s with
              step s + 3;
  tensor pipe runs the issued products in issue order, each reading its
              operands when it runs; a commit arrives once everything issued
              before it has run.

The model checks that nothing deadlocks and that every read sees the data
of its own half or step: the compute warps their S^T/dP^T and L/D, each
product its Q/dO, P^T/dS^T and dS^T tile, the drain its dQ.  In particular
the compute warps write the dS^T buffer of step s without waiting for the
dQ product of step s - 2 that read it: that product was issued before the
S^T/dP^T they wait for, so it has run.  Dropping the drain's release of the
dQ columns, letting the producer refill a stage before its dV/dK products
ran, or issuing a step's dQ after the next step's first S^T/dP^T fails in
the model.
"""

import random

import pytest


class _Violation(Exception):
    """A role read data of another half or step."""


class _Barrier:
    def __init__(self):
        self.phase = 0

    def arrive(self):
        self.phase += 1

    def passed(self, parity):
        return (self.phase & 1) != parity


NSQ, NLD = 3, 6


def _run(n_steps, rng, dq_free_wait=True, qd_empty_after_dvdk=True, dq_late=False):
    n_half = 2 * n_steps
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Barrier())

    # What each buffer holds: tags of the half or step written last.
    tmem_buf = {0: None, 1: None}       # ("S", h) after S^T/dP^T, ("P", h) after the compute warps
    ds_smem = {0: None, 1: None}        # step whose dS^T tile is there
    dq_cols = [None]                    # step whose dQ is in TMEM
    qd_stage = dict.fromkeys(range(NSQ))  # step whose Q/dO is there
    ld_slot = dict.fromkeys(range(NLD))   # half whose L/D is there
    in_flight = []                      # Q/dO copies issued: (stage, step)
    pipe = []

    def expect(cond, what):
        if not cond:
            raise _Violation(what)

    def producer():
        for s in range(n_steps):
            st = s % NSQ
            if s >= NSQ:
                yield ("QDEMPTY", st), ((s // NSQ) - 1) & 1
            in_flight.append((st, s))

    def copies():
        while True:
            if in_flight:
                st, s = in_flight.pop(rng.randrange(len(in_flight)))
                qd_stage[st] = s
                bar(("QDFULL", st)).arrive()
            yield None

    def tensor_pipe():
        while True:
            if pipe:
                op = pipe.pop(0)
                kind = op[0]
                if kind == "sdp":
                    h = op[1]
                    s = h // 2
                    expect(qd_stage[s % NSQ] == s, f"S^T/dP^T of half {h} read another step's Q/dO")
                    tmem_buf[h % 2] = ("S", h)
                elif kind == "dvdk":
                    h = op[1]
                    s = h // 2
                    expect(tmem_buf[h % 2] == ("P", h), f"dV/dK of half {h} read {tmem_buf[h % 2]}")
                    expect(qd_stage[s % NSQ] == s, f"dV/dK of half {h} read another step's Q/dO")
                elif kind == "dq":
                    s = op[1]
                    expect(ds_smem[s % 2] == s, f"dQ of step {s} read dS^T of {ds_smem[s % 2]}")
                    dq_cols[0] = s
                elif kind == "commit":
                    bar(op[1]).arrive()
            yield None

    def issuer():
        yield "KVT", 0

        def issue_sdp(h):
            if h % 2 == 0:
                yield ("QDFULL", (h // 2) % NSQ), ((h // 2) // NSQ) & 1
            pipe.append(("sdp", h))
            pipe.append(("commit", ("SDP", h % 2)))

        def issue_dq(s):
            if s > 0 and dq_free_wait:
                yield "DQFREE", (s - 1) & 1
            pipe.append(("dq", s))
            pipe.append(("commit", "DQFULL"))

        yield from issue_sdp(0)
        if n_half > 1:
            yield from issue_sdp(1)
        for h in range(n_half):
            s, a = h // 2, h % 2
            yield ("PDS", a), (h // 2) & 1
            pipe.append(("dvdk", h))
            if a == 1 and qd_empty_after_dvdk:
                pipe.append(("commit", ("QDEMPTY", s % NSQ)))
            if a == 1 and not qd_empty_after_dvdk and h + 2 < n_half:
                # mutation: the stage released before its products have run
                bar(("QDEMPTY", s % NSQ)).arrive()
            if h + 2 < n_half:
                yield from issue_sdp(h + 2)
            if dq_late:
                # mutation: dQ of step s - 1 only after the next step's first
                # S^T/dP^T, which the compute warps wait for before writing
                # dS^T into the buffer that dQ still has to read
                if a == 0 and s > 0:
                    yield from issue_dq(s - 1)
                if h == n_half - 1:
                    yield from issue_dq(s)
            elif a == 1:
                yield from issue_dq(s)
            if h == n_half - 1:
                pipe.append(("commit", "FINAL"))

    def compute():
        for h in range(n_half):
            s, a = h // 2, h % 2
            yield ("SDP", a), (h // 2) & 1
            yield ("LDFULL", h % NLD), (h // NLD) & 1
            expect(tmem_buf[a] == ("S", h), f"compute read {tmem_buf[a]} for half {h}")
            expect(ld_slot[h % NLD] == h, f"compute read L/D of {ld_slot[h % NLD]} for half {h}")
            tmem_buf[a] = ("P", h)
            # dS^T of step s into shared-memory buffer s % 2 (written per half;
            # the model writes the tag at the first half, checked by dQ)
            ds_smem[s % 2] = s
            bar(("PDS", a)).arrive()
            bar(("LDEMPTY", h % NLD)).arrive()
        yield "FINAL", 0

    def drain():
        bar("KVT").arrive()  # K and V copied into TMEM
        for h in range(min(NLD, n_half)):
            ld_slot[h] = h
            bar(("LDFULL", h)).arrive()
        for s in range(n_steps):
            yield "DQFULL", s & 1
            expect(dq_cols[0] == s, f"drain read dQ of {dq_cols[0]} for step {s}")
            bar("DQFREE").arrive()
            for x in range(2):
                h_new = 2 * (s + 3) + x
                if h_new >= n_half:
                    break
                h = 2 * s + x
                yield ("LDEMPTY", h % NLD), (h // NLD) & 1
                ld_slot[h_new % NLD] = h_new
                bar(("LDFULL", h_new % NLD)).arrive()

    finite = {"producer": producer(), "issuer": issuer(), "compute": compute(), "drain": drain()}
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


def _outcomes(seed, tries=30, **kw):
    rng = random.Random(seed)
    seen = {}
    for n_steps in range(1, 9):
        for _ in range(tries):
            try:
                r = _run(n_steps, rng, **kw)
            except _Violation as e:
                r = str(e).split(" ")[0] + " violation"
            seen[r] = seen.get(r, 0) + 1
    return seen


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_protocol_is_safe_under_any_interleaving(seed):
    assert _outcomes(seed) == {"ok": 8 * 30}


def test_dropping_the_drains_release_wait_fails_in_the_model():
    """Without the issuer's wait for the drain, a dQ product overwrites the
    columns the drain has not yet read."""
    seen = _outcomes(4, dq_free_wait=False)
    assert any(k != "ok" for k in seen), seen


def test_releasing_a_qdo_stage_before_its_products_run_fails_in_the_model():
    seen = _outcomes(5, qd_empty_after_dvdk=False)
    assert any(k != "ok" for k in seen), seen


def test_issuing_dq_after_the_next_steps_products_fails_in_the_model():
    """The compute warps may write a step's dS^T without a barrier of its own
    only because the dQ product that read the buffer two steps before was
    issued ahead of the S^T/dP^T they wait for; issued later, it can read
    the next tile's dS^T."""
    seen = _outcomes(6, dq_late=True)
    assert any(k != "ok" for k in seen), seen
