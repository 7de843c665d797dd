"""Two shard launches on one GPU give what one full launch gives: the forward
bit for bit, dK/dV bit for bit, dQ within the gradient tolerance (its fp32
sums are added in a run-dependent order)."""

import math

import pytest
import torch

from exact_attention_27_gb300 import shard
from parity import check_grads, nan_backward, nan_forward
from workloads import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from exact_attention_27_gb300 import _build
    _build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(2, 8, 2, 515, 64), (3, 4, 4, 300, 128)])
def test_shard_launches_match_full_launch(B, Hq, Hkv, N, d):
    import exact_attention_27_gb300 as fa
    scale = 1.0 / math.sqrt(d)
    inp = {n: t.cuda() for n, t in make_inputs(B, Hq, Hkv, N, d, seed=3, with_grad=True).items()}
    o, lse = nan_forward(inp["q"], inp["k"], inp["v"], causal=True, scale=scale)
    dq, dk, dv = nan_backward(inp["q"], inp["k"], inp["v"], o, lse, inp["do"],
                              causal=True, scale=scale)
    outs = {n: torch.full_like(t, float("nan"))
            for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    world = 2
    for rank in range(world):
        views, (Bs, Hqs, Hkvs) = shard.shard(dict(inp, **outs), Hq, Hkv, rank, world)
        fa.fa_forward(views["q"], views["k"], views["v"], views["o"], views["lse"], scale, True)
        fa.fa_backward(views["q"], views["k"], views["v"], views["o"], views["lse"], views["do"],
                       views["dq"], views["dk"], views["dv"], scale, True)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == 0
    assert torch.equal(outs["o"], o) and torch.equal(outs["lse"], lse)
    assert torch.equal(outs["dk"], dk) and torch.equal(outs["dv"], dv)
    check_grads([outs["dq"]], [dq.double().cpu().numpy()], "shard dq")
