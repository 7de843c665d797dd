"""The barrier protocol of the pair-of-CTAs forward (fa_fwd_pair.cu, d = 128,
opted into with fa_set_forward_tile_rows(512)), checked on a model under
random interleavings (host only, no GPU).

Two CTAs of a cluster run every product as one M = 256 MMA.  Each holds
two query tiles (A and B, one softmax warpgroup each) and half of every K
and V tile (stage j % NS).  Per CTA:

  producer    its Q once, its halves of K_j and V_j once the pair's
              products of tile j - NS have released the stage;
  relay       forwards "this CTA's Q / K half / V half landed" to CTA 0;
  softmax x   per key tile: wait for S_x(j) (a commit that arrives in both
              CTAs), write P over it, rescale O when the maximum grew (after
              waiting for the previous O += P V), then arrive on CTA 0's P
              barrier of tile x; at the end wait for the last O += P V.

CTA 0's issuer waits for both CTAs' halves (two relay arrivals each),
issues S_A(0) and S_B(0), then per key tile: once both CTAs' P_x(j) are in,
O_x += P_x(j) V_j and S_x(j + 1); after both tiles, it releases the V and
K stages in both CTAs.  The tensor pipe runs the products in issue order,
each reading both CTAs' operands when it runs.

The model checks every read (each product sees both halves of its own key
tile; each softmax its S; O at each rescale and at the epilogue holds
exactly the products before it) and fails as it should when the issuer
takes one relay for both halves, or when S_x(j + 1) is issued before
O += P_x(j) V (the rescale can then see O one product short).
"""

import random

import pytest


class _Violation(Exception):
    """A role or product saw data of another key tile."""


class _Barrier:
    def __init__(self, count=1):
        self.count = count
        self.pending = count
        self.phase = 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.phase & 1) != parity


def _run(nA, nB, ns, rng, relays=2, s_after_pv=True):
    n_kv = max(nA, nB)
    nx = (nA, nB)
    counts = {"QREADY": relays, "PFULL": 2}  # CTA 0's: relays; both CTAs' softmax x
    bars = {}

    def bar(cta, name):
        key = (cta, name)
        if key not in bars:
            base = name[0] if isinstance(name, tuple) else name
            bars[key] = _Barrier(counts.get(base, relays if base in ("KREADY", "VREADY") else 1))
        return bars[key]

    k_half = {(r, st): None for r in (0, 1) for st in range(ns)}
    v_half = {(r, st): None for r in (0, 1) for st in range(ns)}
    q_in = {0: False, 1: False}
    s_buf = {(r, x): None for r in (0, 1) for x in (0, 1)}  # ("S", j) or ("P", j)
    o_done = {0: 0, 1: 0}
    in_flight = []
    pipe = []

    def expect(cond, what):
        if not cond:
            raise _Violation(what)

    def producer(r):
        in_flight.append(("Q", r, 0, 0))
        for j in range(n_kv):
            st = j % ns
            if j >= ns:
                yield (r, ("KEMPTY", st)), ((j // ns) - 1) & 1
            in_flight.append(("K", r, st, j))
            if j >= ns:
                yield (r, ("VEMPTY", st)), ((j // ns) - 1) & 1
            in_flight.append(("V", r, st, j))

    def copies():
        while True:
            if in_flight:
                t, r, st, j = in_flight.pop(rng.randrange(len(in_flight)))
                if t == "Q":
                    q_in[r] = True
                    bar(r, "QFULL").arrive()
                elif t == "K":
                    k_half[(r, st)] = j
                    bar(r, ("KFULL", st)).arrive()
                else:
                    v_half[(r, st)] = j
                    bar(r, ("VFULL", st)).arrive()
            yield None

    def relay(r):
        yield (r, "QFULL"), 0
        if relays == 2 or r == 0:
            bar(0, "QREADY").arrive()
        for j in range(n_kv):
            st = j % ns
            yield (r, ("KFULL", st)), (j // ns) & 1
            if relays == 2 or r == 0:
                bar(0, ("KREADY", st)).arrive()
            yield (r, ("VFULL", st)), (j // ns) & 1
            if relays == 2 or r == 0:
                bar(0, ("VREADY", st)).arrive()

    def tensor_pipe():
        while True:
            if pipe:
                op = pipe.pop(0)
                if op[0] == "S":
                    x, j = op[1], op[2]
                    for r in (0, 1):
                        expect(q_in[r], "S before Q landed")
                        expect(k_half[(r, j % ns)] == j,
                               f"S_{x}({j}) read CTA {r}'s K half of {k_half[(r, j % ns)]}")
                        s_buf[(r, x)] = ("S", j)
                elif op[0] == "PV":
                    x, j = op[1], op[2]
                    for r in (0, 1):
                        expect(s_buf[(r, x)] == ("P", j), f"PV_{x}({j}) read {s_buf[(r, x)]}")
                        expect(v_half[(r, j % ns)] == j,
                               f"PV_{x}({j}) read CTA {r}'s V half of {v_half[(r, j % ns)]}")
                    o_done[x] += 1
                else:  # commit to both CTAs
                    for r in (0, 1):
                        bar(r, op[1]).arrive()
            yield None

    def issuer():
        def issue_s(x, j):
            pipe.append(("S", x, j))
            pipe.append(("commit", ("SFULL", x)))

        yield (0, "QREADY"), 0
        if n_kv:
            yield (0, ("KREADY", 0)), 0
            for x in (0, 1):
                if nx[x] > 0:
                    issue_s(x, 0)
            pipe.append(("commit", ("KEMPTY", 0)))
        for j in range(n_kv):
            st = j % ns
            yield (0, ("VREADY", st)), (j // ns) & 1
            kn = False
            for x in (0, 1):
                if j >= nx[x]:
                    continue
                nxt = j + 1 < n_kv and j + 1 < nx[x]
                if nxt and not s_after_pv:
                    if not kn:
                        yield (0, ("KREADY", (j + 1) % ns)), ((j + 1) // ns) & 1
                        kn = True
                    issue_s(x, j + 1)  # mutation: before O += P_x(j) V, over P_x(j)
                yield (0, ("PFULL", x)), j & 1
                pipe.append(("PV", x, j))
                pipe.append(("commit", ("ODONE", x)))
                if nxt and s_after_pv:
                    if not kn:
                        yield (0, ("KREADY", (j + 1) % ns)), ((j + 1) // ns) & 1
                        kn = True
                    issue_s(x, j + 1)
            pipe.append(("commit", ("VEMPTY", st)))
            if kn:
                pipe.append(("commit", ("KEMPTY", (j + 1) % ns)))

    def softmax(r, x):
        nt = nx[x]
        for j in range(nt):
            yield (r, ("SFULL", x)), j & 1
            expect(s_buf[(r, x)] == ("S", j), f"softmax {r}/{x} read {s_buf[(r, x)]} as S({j})")
            s_buf[(r, x)] = ("P", j)
            if j > 0 and rng.random() < 0.5:
                yield (r, ("ODONE", x)), (j - 1) & 1
                expect(o_done[x] >= j, f"rescale {r}/{x} at {j} saw {o_done[x]} products")
            bar(0, ("PFULL", x)).arrive()
        if nt:
            yield (r, ("ODONE", x)), (nt - 1) & 1
            expect(o_done[x] == nt, f"epilogue {r}/{x} saw {o_done[x]} of {nt} products")

    finite = {("producer", r): producer(r) for r in (0, 1)}
    finite.update({("relay", r): relay(r) for r in (0, 1)})
    finite.update({("softmax", r, x): softmax(r, x) for r in (0, 1) for x in (0, 1)})
    finite["issuer"] = issuer()
    endless = {"copies": copies(), "pipe": tensor_pipe()}
    order = sorted(finite, key=str)
    waiting = dict.fromkeys(finite)
    alive = set(finite)
    while alive:
        ready = [k for k in order if k in alive and (
            waiting[k] is None or bar(*waiting[k][0]).passed(waiting[k][1]))]
        helpers = [k for k in ("copies", "pipe") if (k == "copies" and in_flight) or (k == "pipe" and pipe)]
        if not ready and not helpers:
            return "deadlock"
        k = rng.choice(ready + helpers)
        if k in endless:
            next(endless[k])
            continue
        try:
            waiting[k] = next(finite[k])
        except StopIteration:
            alive.discard(k)
    return "ok"


def _outcomes(seed, ns=4, tries=12, **kw):
    rng = random.Random(seed)
    seen = {}
    for nA in range(0, 6):
        for nB in range(0, 6):
            for _ in range(tries):
                try:
                    r = _run(nA, nB, ns, rng, **kw)
                except _Violation as e:
                    r = str(e).split(" ")[0] + " violation"
                seen[r] = seen.get(r, 0) + 1
    return seen


@pytest.mark.parametrize("seed", [1, 2])
def test_protocol_is_safe_under_any_interleaving(seed):
    assert _outcomes(seed) == {"ok": 6 * 6 * 12}


def test_one_relay_for_both_halves_fails_in_the_model():
    """The issuer must wait for both CTAs' halves (two relay arrivals)."""
    seen = _outcomes(3, relays=1)
    assert any(k != "ok" for k in seen), seen


def test_next_s_before_the_product_fails_in_the_model():
    seen = _outcomes(4, s_after_pv=False)
    assert any(k != "ok" for k in seen), seen
