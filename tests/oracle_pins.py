"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each pin takes a loaded oracle (`oracle.load()` or a deliberately mutated
build) and raises AssertionError when the oracle disagrees.  They are chosen
so that a plausible slip anywhere in the oracle (a dropped scale, a wrong
sign, an off-by-one mask, a transposed operand, a wrong head mapping, a
missing normalisation) fails at least one of them; `test_oracle_mutations.py`
plants such slips in copies of the oracle and checks exactly that.

None of these re-types the oracle's own loops: the references are values the
pages print, closed forms, invariances, an exact-summation evaluation from the
definition, finite differences, and PyTorch's own double-precision attention
routine treated as an independent library implementation.
"""

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "worked_examples.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _row_problem(scores, values):
    """Q/K/V for one query whose scaled scores are exactly `scores` (scale 1).

    The head dimension is the width w of the values; q = e_0 and k_j = s_j e_0,
    so q.k_j = s_j exactly."""
    n = len(scores)
    v = np.asarray(values, dtype=np.float64).reshape(1, 1, n, -1)
    w = v.shape[-1]
    q = np.zeros((1, 1, 1, w))
    q[..., 0] = 1.0
    k = np.zeros((1, 1, n, w))
    k[0, 0, :, 0] = np.asarray(scores, dtype=np.float64)
    return q, k, v


# ---------------------------------------------------------------- pages' examples

def pin_two_block_note(orc):
    """paweldubiel.com note: [0,0,ln3,ln3] with values [0,0,1,1] gives 0.75."""
    g = golden()["two_block_note"]
    # Scores through Q K^T * scale: q = 1, k = (0, 0, 1, 1), scale = ln 3.
    q = np.ones((1, 1, 1, 1))
    k = np.array([0.0, 0.0, 1.0, 1.0]).reshape(1, 1, 4, 1)
    v = np.array(g["values"], dtype=np.float64).reshape(1, 1, 4, 1)
    o, lse = orc.forward(q, k, v, scale=math.log(3.0), causal=False)
    assert abs(o[0, 0, 0, 0] - g["exact_result"]) < 1e-14, o
    # unnormalised weights 1, 1, 3, 3 sum to 8: L = ln 8
    assert abs(lse[0, 0, 0] - math.log(sum(g["unnormalised_weight_ratio"]))) < 1e-14, lse


def pin_four_scores_weights(orc):
    """Page 1's s = (1, 3, 2, 4): one-shot weights (0.032, 0.237, 0.087, 0.644)."""
    g = golden()["four_scores"]
    # values = identity, so O's row is P's row.
    q, k, v = _row_problem(g["scores"], np.eye(4))
    o, lse = orc.forward(q, k, v, scale=1.0, causal=False)
    tol = 0.5 * 10 ** (-g["digits"]) + 1e-12
    for got, want in zip(o[0, 0, 0], g["softmax_weights"]):
        assert abs(got - want) <= tol, (got, want)
    # page 1: the blockwise total l_2 ~ 1.553 equals the one-shot sum taken
    # against the final record m = 4, so L = 4 + ln(1.553...)
    assert abs((lse[0, 0, 0] - 4.0) - math.log(g["block2"]["l"])) < 1e-3


def pin_figure_7_9(orc):
    """Fig. 7.9: eight scores, eight values, o / l = 5.257."""
    g = golden()["figure_7_9"]
    q, k, v = _row_problem(g["scores"], g["values"])
    o, _ = orc.forward(q, k, v, scale=1.0, causal=False)
    assert abs(o[0, 0, 0, 0] - g["result"]) <= 0.5 * 10 ** (-g["digits"]), o


# ---------------------------------------------------------------- invariants / closed forms

def _random_problem(seed, B=1, Hq=2, Hkv=1, N=9, d=5, Nk=None):
    r = _rng(seed)
    Nk = N if Nk is None else Nk
    return (r.standard_normal((B, Hq, N, d)), r.standard_normal((B, Hkv, Nk, d)),
            r.standard_normal((B, Hkv, Nk, d)))


def pin_rows_of_p_sum_to_one(orc):
    """With V = identity the output row is P's row: non-negative, sums to 1."""
    r = _rng(1)
    N = 11
    for causal in (False, True):
        q = np.zeros((1, 1, N, N))
        k = np.zeros((1, 1, N, N))
        q[..., :4] = r.standard_normal((1, 1, N, 4))
        k[..., :4] = r.standard_normal((1, 1, N, 4))
        v = np.eye(N).reshape(1, 1, N, N)
        o, _ = orc.forward(q, k, v, scale=0.7, causal=causal)
        P = o[0, 0]
        assert np.all(P >= 0.0)
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) <= 1e-12
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)


def pin_causal_first_query(orc):
    """Causal query 0 sees only key 0: O[0] = v_0 exactly, L_0 = scale q_0.k_0."""
    q, k, v = _random_problem(2, Hq=1, Hkv=1, N=7, d=6)
    scale = 0.37
    o, lse = orc.forward(q, k, v, scale=scale, causal=True)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - scale * float(q[0, 0, 0] @ k[0, 0, 0])) <= 1e-13


def pin_uniform_scores(orc):
    """Q = 0 makes every score equal: O is a plain mean, L = ln(count)."""
    r = _rng(3)
    N, d = 10, 3
    q = np.zeros((1, 1, N, d))
    k = r.standard_normal((1, 1, N, d))
    v = r.standard_normal((1, 1, N, d))
    o, lse = orc.forward(q, k, v, scale=0.5, causal=False)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(axis=0))) <= 1e-13
    assert np.max(np.abs(lse[0, 0] - math.log(N))) <= 1e-13
    o, lse = orc.forward(q, k, v, scale=0.5, causal=True)
    for i in range(N):
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, :i + 1].mean(axis=0))) <= 1e-13
        assert abs(lse[0, 0, i] - math.log(i + 1)) <= 1e-13


def pin_constant_values(orc):
    """V = c everywhere gives O = c whatever the scores."""
    q, k, _ = _random_problem(4, N=8, d=4)
    v = np.full((1, 1, 8, 4), -2.25)
    for causal in (False, True):
        o, _ = orc.forward(q, k, v, scale=1.3, causal=causal)
        assert np.max(np.abs(o + 2.25)) <= 1e-13


def pin_key_shift(orc):
    """k_j -> k_j + u for all j adds scale q_i.u to row i: O unchanged, L shifted."""
    q, k, v = _random_problem(5, Hq=2, Hkv=2, N=9, d=5)
    u = _rng(6).standard_normal(5)
    scale = 0.45
    for causal in (False, True):
        o1, l1 = orc.forward(q, k, v, scale, causal)
        o2, l2 = orc.forward(q, k + u, v, scale, causal)
        assert np.max(np.abs(o1 - o2)) <= 1e-12
        assert np.max(np.abs((l2 - l1) - scale * (q @ u))) <= 1e-12


def pin_key_permutation(orc):
    """Non-causal: permuting keys and values together leaves O and L unchanged."""
    q, k, v = _random_problem(7, Hq=1, Hkv=1, N=12, d=3)
    perm = _rng(8).permutation(12)
    o1, l1 = orc.forward(q, k, v, 0.8, False)
    o2, l2 = orc.forward(q, k[:, :, perm], v[:, :, perm], 0.8, False)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs(l1 - l2)) <= 1e-12


def pin_blockwise_equals_one_shot(orc):
    """The pages' blockwise rules give the one-shot result for any block size."""
    from oracle.online_softmax import online_softmax_row
    r = _rng(9)
    N = 13
    s = r.standard_normal(N) * 3.0
    vals = r.standard_normal((N, 2))
    q, k, v = _row_problem(s, vals)
    o, lse = orc.forward(q, k, v, scale=1.0, causal=False)
    for block in (1, 2, 3, 7, N):
        out, l, _ = online_softmax_row(list(s), [list(x) for x in vals], block)
        assert np.max(np.abs(np.array(out) - o[0, 0, 0])) <= 1e-12
        assert abs(l - lse[0, 0, 0]) <= 1e-12


# ---------------------------------------------------------------- exact summation

def _fsum_attention(q, k, v, scale, causal):
    """Row by row from the definition with math.fsum / math.exp (tiny inputs)."""
    B, Hq, N, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    o = np.zeros((B, Hq, N, d))
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            kk, vv = k[b, h // G], v[b, h // G]
            for i in range(N):
                s = [scale * math.fsum(q[b, h, i, c] * kk[j, c] for c in range(d))
                     if not (causal and j > i) else -math.inf for j in range(Nk)]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                z = math.fsum(w)
                lse[b, h, i] = m + math.log(z)
                for c in range(v.shape[3]):
                    o[b, h, i, c] = math.fsum(w[j] * vv[j, c] for j in range(Nk)) / z
    return o, lse


def pin_exact_summation(orc):
    """Agreement with an exact-summation evaluation on tiny shapes, d in {1,3,5,8}."""
    for seed, (N, d, G, causal) in enumerate([(1, 1, 1, False), (5, 3, 1, True),
                                              (7, 5, 2, False), (8, 8, 2, True),
                                              (6, 3, 3, True)]):
        r = _rng(100 + seed)
        q = r.standard_normal((2, 2 * G, N, d))
        k = r.standard_normal((2, 2, N, d))
        v = r.standard_normal((2, 2, N, d))
        o, lse = orc.forward(q, k, v, 0.6, causal)
        o2, l2 = _fsum_attention(q, k, v, 0.6, causal)
        assert np.max(np.abs(o - o2)) <= 1e-12
        assert np.max(np.abs(lse - l2)) <= 1e-12


# ---------------------------------------------------------------- library routine

def _torch_sdpa(q, k, v, scale, causal, dout=None):
    """PyTorch's float64 CPU attention (K/V heads repeated per group)."""
    G = q.shape[1] // k.shape[1]
    tq = torch.tensor(q, requires_grad=dout is not None)
    tk = torch.tensor(k, requires_grad=dout is not None)
    tv = torch.tensor(v, requires_grad=dout is not None)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1),
        is_causal=causal, scale=scale)
    if dout is None:
        return o.detach().numpy()
    o.backward(torch.tensor(dout))
    return (o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


def pin_library_forward(orc):
    """PyTorch's double-precision scaled_dot_product_attention, incl. GQA groups."""
    for seed, (Hq, Hkv, N, d, causal) in enumerate([(1, 1, 33, 16, False), (4, 2, 40, 8, True),
                                                    (6, 2, 17, 12, True)]):
        r = _rng(200 + seed)
        q = r.standard_normal((2, Hq, N, d))
        k = r.standard_normal((2, Hkv, N, d))
        v = r.standard_normal((2, Hkv, N, d))
        o, lse = orc.forward(q, k, v, 0.3, causal)
        assert np.max(np.abs(o - _torch_sdpa(q, k, v, 0.3, causal))) <= 1e-12
        # L against a log-sum-exp taken by torch over the masked scores
        s = 0.3 * torch.tensor(q) @ torch.tensor(k).repeat_interleave(Hq // Hkv, 1).transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
        assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-12


def pin_library_backward(orc):
    """Gradients equal PyTorch autograd through its double-precision attention."""
    for seed, (Hq, Hkv, N, d, causal) in enumerate([(2, 2, 19, 8, True), (4, 1, 16, 5, False),
                                                    (4, 2, 23, 6, True)]):
        r = _rng(300 + seed)
        q = r.standard_normal((1, Hq, N, d))
        k = r.standard_normal((1, Hkv, N, d))
        v = r.standard_normal((1, Hkv, N, d))
        do = r.standard_normal((1, Hq, N, d))
        dq, dk, dv = orc.backward(q, k, v, do, 0.4, causal)
        _, tq, tk, tv = _torch_sdpa(q, k, v, 0.4, causal, dout=do)
        for got, want in ((dq, tq), (dk, tk), (dv, tv)):
            assert np.max(np.abs(got - want)) <= 1e-11 * max(1.0, np.max(np.abs(want)))


# ---------------------------------------------------------------- gradients from first principles

def pin_finite_differences(orc):
    """Central differences of f = sum(dO o O) match the backward (double)."""
    r = _rng(400)
    B, Hq, Hkv, N, d = 1, 2, 1, 5, 3
    q = r.standard_normal((B, Hq, N, d))
    k = r.standard_normal((B, Hkv, N, d))
    v = r.standard_normal((B, Hkv, N, d))
    do = r.standard_normal((B, Hq, N, d))
    scale = 0.9
    for causal in (False, True):
        dq, dk, dv = orc.backward(q, k, v, do, scale, causal)

        def f(args):
            o = orc.forward(args["q"], args["k"], args["v"], scale, causal)[0]
            return float(np.sum(do * o))

        h = 1e-5
        for name, g in (("q", dq), ("k", dk), ("v", dv)):
            x = {"q": q, "k": k, "v": v}[name]
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                plus = {"q": q, "k": k, "v": v, name: xp}
                minus = {"q": q, "k": k, "v": v, name: xm}
                num[idx] = (f(plus) - f(minus)) / (2 * h)
            err = np.max(np.abs(num - g)) / max(1e-3, np.max(np.abs(g)))
            assert err <= 1e-6, (name, causal, err)


def pin_delta_identity(orc):
    """sum_j P_ij dP_ij equals sum_c dO_ic O_ic (the fused method's shortcut)."""
    r = _rng(500)
    q = r.standard_normal((2, 4, 14, 6))
    k = r.standard_normal((2, 2, 14, 6))
    v = r.standard_normal((2, 2, 14, 6))
    do = r.standard_normal((2, 4, 14, 6))
    for causal in (False, True):
        o, _ = orc.forward(q, k, v, 0.5, causal)
        *_, rowdot = orc.backward(q, k, v, do, 0.5, causal, want_rowdot=True)
        assert np.max(np.abs(rowdot - orc.row_dot(do, o))) <= 1e-12
        assert np.max(np.abs(orc.row_dot(do, o) - np.einsum("bhnc,bhnc->bhn", do, o))) <= 1e-12


def pin_gqa_gradient_is_group_sum(orc):
    """A shared K/V head's gradient is the sum over its query heads' gradients."""
    r = _rng(600)
    G = 3
    q = r.standard_normal((1, 2 * G, 10, 4))
    k = r.standard_normal((1, 2, 10, 4))
    v = r.standard_normal((1, 2, 10, 4))
    do = r.standard_normal((1, 2 * G, 10, 4))
    dq, dk, dv = orc.backward(q, k, v, do, 0.7, True)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    dq2, dk2, dv2 = orc.backward(q, kr, vr, do, 0.7, True)
    assert np.max(np.abs(dq - dq2)) <= 1e-12
    assert np.max(np.abs(dk - dk2.reshape(1, 2, G, 10, 4).sum(axis=2))) <= 1e-12
    assert np.max(np.abs(dv - dv2.reshape(1, 2, G, 10, 4).sum(axis=2))) <= 1e-12


def pin_sampled_rows_match_full(orc):
    """Evaluating selected query rows gives those rows of the full evaluation."""
    q, k, v = _random_problem(700, B=2, Hq=4, Hkv=2, N=21, d=4)
    rows = [0, 5, 20, 13]
    for causal in (False, True):
        o, l = orc.forward(q, k, v, 0.5, causal)
        o2, l2 = orc.forward(q, k, v, 0.5, causal, rows=rows)
        assert np.array_equal(o[:, :, rows], o2)
        assert np.array_equal(l[:, :, rows], l2)


def pin_query_offset_is_a_row_block(orc):
    """Queries at absolute positions o..o+n-1 (N_q = n, offset o, all N_k keys)
    get exactly rows o..o+n-1 of the full causal result, and a single query at
    the last position sees every key (the non-causal result for that row)."""
    q, k, v = _random_problem(800, B=2, Hq=4, Hkv=2, N=29, d=5)
    o_full, l_full = orc.forward(q, k, v, 0.6, True)
    for off, n in ((0, 7), (5, 11), (20, 9), (28, 1)):
        o, l = orc.forward(q[:, :, off:off + n], k, v, 0.6, True, q_offset=off)
        assert np.array_equal(o, o_full[:, :, off:off + n])
        assert np.array_equal(l, l_full[:, :, off:off + n])
    o_nc, l_nc = orc.forward(q[:, :, -1:], k, v, 0.6, False)
    o_last, l_last = orc.forward(q[:, :, -1:], k, v, 0.6, True, q_offset=28)
    assert np.max(np.abs(o_last - o_nc)) <= 1e-13 and np.max(np.abs(l_last - l_nc)) <= 1e-13


ALL_PINS = [
    pin_two_block_note, pin_four_scores_weights, pin_figure_7_9, pin_rows_of_p_sum_to_one,
    pin_causal_first_query, pin_uniform_scores, pin_constant_values, pin_key_shift,
    pin_key_permutation, pin_blockwise_equals_one_shot, pin_exact_summation,
    pin_library_forward, pin_library_backward, pin_finite_differences, pin_delta_identity,
    pin_gqa_gradient_is_group_sum, pin_sampled_rows_match_full, pin_query_offset_is_a_row_block,
]
