"""bench.py's CPU legs, no GPU: the reference arm prints the contract's JSON
line (the fp64 oracle timed on the host), the oracle leg runs the ring
hybrid's steps for a hybrid workload, the permutation byte counts, and the
JSON line the GPU arm assembles from its measurements (fed fixed numbers)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "C2",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] >= 3
    assert d["config"]["workload"] == "C2"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_leg_runs_the_ring_hybrid():
    sys.path.insert(0, ROOT)
    import bench
    from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS
    w = WORKLOADS["C2"].with_(name="C2-ring", P=8, ring=2, n_head=16, n_kv_head=16)
    ob = bench.OracleBench(w, nthreads=2)
    t_full, n_rows, pairs, wall = ob.step(8)
    assert t_full > 0 and 0 < n_rows <= 8 and pairs > 0 and wall > 0
    assert "2 ring positions" in ob.describe(n_rows)


def test_pack_bytes_count_replicas_within_an_all_to_all_group():
    """K and V are written once per replica only when there are fewer
    kv-heads than ranks in one All-to-All group (P / ring ranks): the ring
    hybrid at P = 256 with 32 kv-heads replicates nothing, C4 with 4 kv-heads
    writes each kv-head to 2 ranks."""
    sys.path.insert(0, ROOT)
    import bench
    from ulysses_sequence_attention_seq_gb300.synthetic import EXTRA_WORKLOADS, WORKLOADS
    c4 = WORKLOADS["C4"]
    per_head = c4.B * c4.S * c4.head_dim * 2            # one bf16 head over the sequence
    assert bench.permute_bytes(c4, 2) == 6 * 32 * per_head
    assert bench.permute_bytes(EXTRA_WORKLOADS["C4-ring8"], 2) == 6 * 32 * per_head
    kv4 = EXTRA_WORKLOADS["C4-kv4"]
    assert bench.permute_bytes(kv4, 2) == per_head * (2 * 32 + 2 * 4 + 2 * 8)


def _fake_measurements(backward, steps):
    """What run_ulysses returns, with plausible timings (no GPU involved): the
    dS-store backward on the headline, the other two modes beside it."""
    per = {"pack_qkv": [0.29] * steps, "attn_fwd": [5.4] * steps, "unpack_out": [0.08] * steps}
    alt_per = {}
    if backward:
        per.update(bwd_prepare=[0.17] * steps, bwd_dkdv_ds=[13.0] * steps, bwd_dq_ds=[5.0] * steps)
        alt_per = {"two_kernel": {"bwd_prepare": [0.17] * steps, "bwd_dkdv": [10.9] * steps, "bwd_dq": [8.4] * steps},
                   "fused": {"bwd_prepare": [0.17] * steps, "bwd_dkdvq": [20.0] * steps,
                             "bwd_dq_finish": [1.0] * steps}}
    total = sum(v[0] for v in per.values()) * steps
    return dict(total_ms=total, per=per, alt_per=alt_per, bwd_mode="ds_store" if backward else None,
                clocks={"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": []},
                e2e_ms=total * 1.03, h2d=1 << 30, d2h=1 << 30, launches=6 * steps, status=0, backward=backward,
                folded={"fwd": {"unfolded_ms": 5.8, "ms": 5.6}, "bwd": {"unfolded_ms": 19.8, "ms": 19.9}},
                ex2_rate=32.0, sms=152)


def test_bench_line_carries_the_contract_keys(monkeypatch, capsys):
    """The JSON line bench.py assembles from its measurements (run_ulysses
    replaced by fixed numbers): every key the contract asks for, with the
    roofline of the dominant kernel and its traffic."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "run_ulysses", lambda args, w, rank, world: _fake_measurements(True, args.steps))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "4", "--no-cpu-baseline"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["steps"] == 4 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "C4"
    r = line["roofline"]
    assert r["kernel"] == "dkdv_kernel<128>" and r["bound"] == "tensor" and r["bwd_mode"] == "ds_store"
    assert r["traffic"] == bench.TRAFFIC.get(("bwd_dkdv_ds", "C4"))
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    # dK/dV (storing dS): dV, dP, dK = 1.5 forwards of algorithmic FLOPs over 13.0 ms
    c4 = bench.WORKLOADS["C4"]
    assert abs(r["achieved"] - 1.5 * bench.attn_fwd_flops(c4) / 13.0e-3 / 1e12) < 1e-6
    # dQ from the stored tiles: HBM-bound, every causal tile pair's 32 KB once, K and dQ once
    h = line["secondary_rooflines"]["bwd_dq_ds"]
    tiles = c4.B * c4.n_head * (256 * 257 // 2)
    assert h["bound"] == "hbm" and h["bytes_per_launch"] == tiles * 32768 + c4.B * c4.S * (32 + 32) * 128 * 2
    assert abs(h["achieved"] - h["bytes_per_launch"] / 5.0e-3 / 1e9) < 1e-6
    assert abs(line["attn_bwd_tflops_2p5x"] - 1.25 * line["attn_bwd_tflops"]) < 1e-9
    assert line["value"] == pytest.approx(32768 / (line["ms_per_step"] * 1e-3))
    assert set(line["e2e"]) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert line["folded_mode"]["bwd"] == {"unfolded_ms": 19.8, "ms": 19.9}
    assert line["folded_mode"]["on_headline_path"] is False
    m = line["bwd_modes"]
    assert m["headline_uses"] == "ds_store"
    assert m["ds_store"]["ms"] == pytest.approx(0.17 + 13.0 + 5.0) == line["attn_bwd_ms"]
    assert m["two_kernel"]["ms"] == pytest.approx(0.17 + 10.9 + 8.4) and m["two_kernel"]["kernel"] == "dkdv_kernel<128>"
    assert m["fused"]["ms"] == pytest.approx(0.17 + 20.0 + 1.0) and m["fused"]["kernel"] == "dkdvq_kernel<128>"


def test_fp32_workload_reports_the_cuda_core_kernel_against_its_fma_peak(monkeypatch, capsys):
    """The fp32 workload (C1) runs its forward on the CUDA cores: the roofline
    names that kernel, bound "alu", against SMs x 128 fp32 lanes x 2 FLOP x
    the maximum SM clock, and carries no tensor-core figures."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "run_ulysses", lambda args, w, rank, world: _fake_measurements(False, args.steps))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "C1", "--steps", "4", "--no-cpu-baseline"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    r = line["roofline"]
    assert line["dtype"] == "f32" and line["config"]["workload"] == "C1"
    assert r["kernel"] == "attn_fwd_simt_kernel<32>" and r["bound"] == "alu"
    assert r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12)
    assert r["achieved"] == pytest.approx(bench.attn_fwd_flops(bench.WORKLOADS["C1"]) / 5.4e-3 / 1e12)
    assert r["peak_burst"] is None and r["frac_burst"] is None
    assert "attn_fwd_mufu" not in line["secondary_rooflines"]


def test_reference_arm_times_both_passes_with_the_gpu_arms_config(monkeypatch, capsys):
    """For a workload with a backward the reference arm times the oracle's
    forward and backward (passes fwd+bwd, like the GPU arm's headline), labels
    its per-step time as extrapolated from a sample, and its config has the
    GPU arm's keys."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "C3",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    ref = json.loads([ln for ln in out.stdout.splitlines() if ln.startswith("{")][0])
    assert ref["config"]["passes"] == "fwd+bwd"
    assert ref["ms_per_step_kind"] == "extrapolated_from_sample" and ref["sample_wall_ms_per_step"] > 0
    assert "backward" in ref["cpu_baseline"]["sample"]
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "run_ulysses", lambda args, w, rank, world: _fake_measurements(True, args.steps))
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "2", "--workload", "C3", "--no-cpu-baseline"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    bench.main()
    gpu = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert set(gpu["config"]) == set(ref["config"])
    assert all(gpu["config"][k] == ref["config"][k] for k in gpu["config"] if k not in ("l2", "parallelism"))
    r = gpu["roofline"]
    assert abs(r["frac_burst"] - r["achieved"] / r["peak_burst"]) < 1e-12 and r["sm_mhz"] == 2040.0


def test_ds_store_byte_counts():
    """The dS store holds one tile per causal (key tile, query tile) pair of
    every (batch, q-head), or every pair without the mask; the dQ step's
    algorithmic bytes are those tiles, K and dQ once each."""
    sys.path.insert(0, ROOT)
    import bench
    from ulysses_sequence_attention_seq_gb300.synthetic import WORKLOADS
    c3 = WORKLOADS["C3"]                                   # S = 8192: 64 tiles
    assert bench.ds_tiles(c3) == 64 * 65 // 2
    assert bench.ds_tiles(c3.with_(causal=False)) == 64 * 64
    assert bench.ds_tiles(c3.with_(S=8193)) == 65 * 66 // 2
    nb = bench.dq_ds_bytes(c3, 2)
    assert nb == c3.B * c3.n_head * (64 * 65 // 2) * 32768 + c3.B * c3.S * (c3.n_kv_head + c3.n_head) * 128 * 2
