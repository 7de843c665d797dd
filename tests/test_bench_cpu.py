"""Host logic of bench.py: the oracle sample's row rotation and the error
report it attaches to the CPU baseline (no GPU needed)."""

import types

import numpy as np

import bench
import oracle


def tiny():
    return types.SimpleNamespace(B=1, Hq=2, Hkv=1, N=512, d=64, scale=0.125, name="tiny-512")


def full_outputs(w):
    """The oracle's own full outputs, standing in for the GPU's."""
    inp = bench._oracle_inputs(w)
    o, lse = oracle.attention_forward(inp["q"], inp["k"], inp["v"], w.scale, True)
    dq, dk, dv = oracle.attention_backward(inp["q"], inp["k"], inp["v"], inp["do"], w.scale, True)
    return {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}


def test_first_sample_is_the_last_block_and_rows_rotate():
    w = tiny()
    keep = []
    for i in range(3):
        bench.oracle_sample(w, 128, i, keep)
    starts = [r0 for r0, _, _ in keep]
    assert starts[0] == w.N - 128
    assert all(r0 % 128 == 0 and 0 <= r0 < w.N for r0 in starts)
    assert len(set(starts)) == 3


def test_errors_vanish_against_the_oracle_itself_and_catch_a_wrong_dk():
    w = tiny()
    gpu = full_outputs(w)
    keep = []
    for i in range(2):
        bench.oracle_sample(w, 128, i, keep)
    rep = bench.sampled_errors(w, keep, gpu, 128)
    assert rep["within_tolerance"]
    for key in ("o_max_abs", "o_mean_abs", "lse_max_abs", "dq_rel", "dk_rel", "dv_rel"):
        assert rep[key] is not None and rep[key] <= 1e-9, key
    # the last block's keys are complete in the sample: a dK error there shows
    bad = dict(gpu)
    bad["dk"] = gpu["dk"].copy()
    bad["dk"][:, :, -1, 0] += 0.1 * np.abs(gpu["dk"][:, :, -128:]).max()
    rep = bench.sampled_errors(w, keep, bad, 128)
    assert not rep["within_tolerance"]
    assert abs(rep["dk_rel"] - 0.1) < 1e-6


def test_median_and_min():
    assert bench._med_min([3.0, 1.0, 2.0]) == {"median": 2.0, "min": 1.0}


def test_reference_arm_line_carries_the_contract_keys_and_the_same_config():
    """The reference arm (the oracle on the host cores) prints the keys the
    benchmark line needs, and its `config` is the dict the device arm prints
    for the same workload, so the two lines compare as the same config."""
    import json
    args = types.SimpleNamespace(steps=1, warmup=3)
    line = bench.run_reference(args, rank=0, world=1)
    json.dumps(line)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
    w = bench.WORKLOADS[bench.STEP_WORKLOAD]
    assert line["config"] == bench.bench_config(w, 1)
    assert line["config"]["workload"] == w.describe()
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert bench.bench_config(w, 2)["parallelism"] == "replicas x2"
