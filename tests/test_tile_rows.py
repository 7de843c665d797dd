"""Host logic of the forward's per-shape tile choice (fa_forward_tile_rows_for
of include/fa.h; no GPU needed).

The choice is the B_r of the tiling in "FlashAttention: l'attenzione che non
spreca memoria", section "L'idea: lavorare a tessere", picked per problem size
as the autotuning row of "Flash Attention ... NVIDIA CUDA Tile", section
"Resumen: La pila de optimización", does.  The library estimates each grid's
finish time by list scheduling; these tests restate that model in Python
(heapq) and in closed form, and check the special cases.
"""

import heapq
import itertools
import math

import pytest

import exact_attention_27_gb300 as fa
from exact_attention_27_gb300 import _build

# Cost model stated in include/fa.h and fa_fwd.cu: per-CTA overhead and cost
# per key-tile step, in units of one step of the two-tile CTA.
COSTS = {64: dict(o2=0.0, o1=1.0, r1=1.35), 96: dict(o2=1.0, o1=2.5, r1=1.05),
         128: dict(o2=1.0, o1=3.0, r1=1.0)}


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def rows_for(B, Hq, Hkv, Nq, Nk, d, causal, q_offset=0, sms=152):
    return fa.fa_forward_tile_rows_for(B, Hq, Hkv, Nq, Nk, d, causal, q_offset, sms)


def model(B, Hq, Hkv, Nq, Nk, d, causal, q_offset, sms):
    nq, nk = -(-Nq // 128), -(-Nk // 128)
    npair, nheads = (nq + 1) // 2, B * Hq
    if nheads * npair > 16 * sms:
        return 256
    hpg = min(max(1, int(48 * 1024 * 1024 / (2.0 * Nk * d * 2))) * (Hq // Hkv), nheads)

    def tiles(qt):
        if qt >= nq:
            return 0
        return min((q_offset + qt * 128 + 127) // 128 + 1, nk) if causal else nk

    def finish(units, cost):
        free = [0.0] * sms
        end = 0.0
        for g0 in range(0, nheads, hpg):
            for i in range(units):
                c = cost(units - 1 - i if causal else i)
                for _ in range(min(hpg, nheads - g0)):
                    t = heapq.heappop(free) + c
                    heapq.heappush(free, t)
                    end = max(end, t)
        return end

    k = COSTS[d]
    two = finish(npair, lambda u: k["o2"] + tiles(2 * u) + tiles(2 * u + 1))
    one = finish(nq, lambda u: k["o1"] + k["r1"] * tiles(u))
    return 128 if one < two else 256


def test_fixed_head_dimensions():
    assert rows_for(1, 2, 2, 1024, 1024, 256, 1) == 128
    assert rows_for(8, 64, 64, 8192, 8192, 256, 0) == 128


def test_invalid_arguments_give_zero():
    assert rows_for(1, 2, 3, 1024, 1024, 64, 1) == 0      # H_q not a multiple of H_kv
    assert rows_for(0, 2, 2, 1024, 1024, 64, 1) == 0
    assert rows_for(1, 2, 2, 1024, 0, 64, 1) == 0
    assert rows_for(1, 2, 2, 1024, 1024, 80, 1) == 0
    assert fa.library().fa_forward_tile_rows_for(1, 2, 2, 1024, 1024, 64, 2, 0, 152) == 0
    assert rows_for(1, 2, 2, 1024, 1024, 64, 1, q_offset=-1) == 0
    assert rows_for(1, 2, 2, 1024, 1024, 64, 1, sms=0) == 0


@pytest.mark.parametrize("d", [64, 96, 128])
def test_few_ctas_take_one_tile_and_many_take_two(d):
    # One head: the two-tile grid leaves almost every SM idle.
    assert rows_for(1, 1, 1, 4096, 4096, d, 1) == 128
    assert rows_for(1, 1, 1, 4096, 4096, d, 0) == 128
    # Past 16 two-tile waves the cheaper two-tile step decides.
    assert rows_for(16, 64, 64, 8192, 8192, d, 1) == 256
    assert rows_for(16, 64, 8, 8192, 8192, d, 0) == 256


@pytest.mark.parametrize("d", [64, 96, 128])
def test_non_causal_matches_the_closed_form(d):
    # Without the mask every CTA of a grid costs the same, so list scheduling
    # finishes after ceil(CTAs / SMs) CTA durations whatever the order.
    k = COSTS[d]
    for bh, n, sms in itertools.product((1, 2, 3, 5, 8, 16, 32, 48), (256, 1000, 2048, 4096, 8192),
                                        (148, 152)):
        nq = -(-n // 128)
        npair = (nq + 1) // 2
        if bh * npair > 16 * sms:
            continue
        two = math.ceil(bh * npair / sms) * (k["o2"] + 2 * nq)
        one = math.ceil(bh * nq / sms) * (k["o1"] + k["r1"] * nq)
        if nq % 2:  # the last pair has one tile
            continue
        want = 128 if one < two else 256
        assert rows_for(1, bh, bh, n, n, d, 0, sms=sms) == want, (bh, n, sms)


@pytest.mark.parametrize("d", [64, 96, 128])
def test_causal_and_grouped_match_list_scheduling(d):
    cases = [
        (1, 8, 8, 1024, 1024, 1, 0), (2, 8, 8, 4096, 4096, 1, 0), (1, 16, 16, 8192, 8192, 1, 0),
        (1, 32, 32, 4096, 4096, 1, 0), (4, 16, 4, 2048, 2048, 1, 0), (1, 24, 24, 8192, 8192, 1, 0),
        (1, 64, 8, 8192, 8192, 0, 0), (2, 16, 2, 3000, 3000, 1, 0), (1, 8, 8, 1000, 5000, 1, 4000),
        (1, 12, 4, 640, 4096, 1, 3456), (3, 20, 5, 8192, 8192, 0, 0), (1, 40, 40, 8192, 8192, 1, 0),
    ]
    for B, Hq, Hkv, Nq, Nk, causal, off in cases:
        for sms in (148, 152):
            want = model(B, Hq, Hkv, Nq, Nk, d, causal, off, sms)
            assert rows_for(B, Hq, Hkv, Nq, Nk, d, causal, q_offset=off, sms=sms) == want, \
                (B, Hq, Hkv, Nq, Nk, causal, off, sms)


def test_wave_quantisation_decides_at_d128():
    # 32 heads x 16 tile pairs = 512 two-tile CTAs, 3.37 waves (4 rounds) on
    # 152 SMs, against 1024 one-tile CTAs in 6.7 waves (7 rounds) of half the
    # length: one tile per CTA finishes first.  At 16 heads (1.7 and 3.4
    # waves: 2 and 4 rounds) the two-tile grid does.
    assert rows_for(1, 32, 32, 4096, 4096, 128, 0) == 128
    assert rows_for(1, 16, 16, 4096, 4096, 128, 0) == 256
