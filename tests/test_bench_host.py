"""bench.py's algorithmic byte and exponential counts (the roofline's
numerators) against values worked out by hand from the workload shapes."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_scan_algorithmic_counts():
    # B8 L2048 D4096 N16 bf16 (M = 16384 rows, 2-byte activations):
    # forward  4 M D s (u, delta_raw, z in; out) + 2 M N s (B, C) + A_log, D
    #        = 536870912 + 1048576 + 278528
    # backward 7 M D s + 4 M N s + 2 (A_log, D and their gradients)
    #        = 939524096 + 2097152 + 557056
    fwd, bwd, exps = bench.algorithmic(dict(batch=8, seqlen=2048, dinner=4096, dstate=16, dtype="bf16"))
    assert fwd == 538_198_016
    assert bwd == 942_178_304
    assert exps == 1_073_741_824     # one exp(delta A) per (row, channel, state)


def test_decode_bytes():
    scan, conv = bench.decode_bytes(dict(batch=64, dinner=4096, dstate=16, dconv=4))
    # state read + written, u / delta_raw / z read and out written, B and C, A_log and D
    assert scan == 2 * 64 * 16 * 4096 * 4 + 4 * 64 * 4096 * 4 + 2 * 64 * 16 * 4 + 4096 * 16 * 4 + 4096 * 4
    assert scan == 38_035_456
    # x, the 3 state slots in and out, out; taps and bias
    assert conv == 64 * 4096 * 4 * (1 + 2 * 3 + 1) + 4096 * 4 * 4 + 4096 * 4


def test_alu_roofline_counts_the_recurrences_minimal_fp32_work():
    import bench
    cfg = dict(batch=8, seqlen=2048, dinner=4096, dstate=16)
    el = 8 * 2048 * 4096 * 16
    r = bench.alu_roofline(cfg, 1.0, 3.0, 128.0, 2000.0, "test")
    peak = 128.0 * 152 * 2000e6
    assert abs(r["peak"] - peak / 1e12) < 1e-3
    assert abs(r["fwd_frac"] - 4 * el / peak / 1e-3) < 1e-4
    assert abs(r["bwd_frac"] - 12 * el / peak / 3e-3) < 1e-4
    assert abs(r["step_frac"] - 16 * el / peak / 4e-3) < 1e-4


def test_cpu_sample_counts_only_rows_it_has():
    """The CPU oracle sample never counts batch rows its inputs do not hold:
    with one batch row of data it runs and counts one row, whatever the
    workload's batch."""
    from selective_state_space_ssm_gb300 import workloads
    cfg = dict(batch=8, seqlen=16, dinner=64, dstate=4)
    inp = workloads.scan_inputs(1, 16, 64, 4, seed=1)
    v, sample, secs = bench.cpu_oracle_sample(cfg, inp, target_s=0.5, threads=1)
    assert sample.startswith("batch rows [0, 1)")
    assert v > 0 and secs > 0


def test_reference_arm_line(monkeypatch, capsys):
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the metric, unit and config of the GPU arm, a cpu_baseline and an
    e2e object with zero host-device bytes; every step times the same slice,
    sized once."""
    import json
    import types
    monkeypatch.setattr(bench, "WORKLOAD", "tiny_scan_fp32")
    calls = []
    real = bench.oracle_slice_seconds

    def counted(inp, L, nb, dsub, threads):
        calls.append((nb, dsub))
        return real(inp, L, nb, dsub, threads)

    monkeypatch.setattr(bench, "oracle_slice_seconds", counted)
    args = types.SimpleNamespace(steps=3, warmup=2)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "Mtokens/s" and line["steps"] == 3 and line["warmup"] == 2
    assert line["config"]["workload"].startswith("tiny_scan_fp32")
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # the 5 steps all ran the slice that the sizing ended on
    assert len(set(calls[-5:])) == 1


def test_conv_bytes():
    """The conv's algorithmic bytes: 8 per element forward (x in, out out), 12
    backward (x, dout in; dx out), plus the taps and bias (and, backward,
    their gradients)."""
    fwd, bwd = bench.conv_bytes(16384, 1536, 4)
    assert fwd == 16384 * 1536 * 8 + 1536 * 5 * 4
    assert bwd == 16384 * 1536 * 12 + 2 * 1536 * 5 * 4
