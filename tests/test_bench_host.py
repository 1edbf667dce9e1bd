"""Host logic of bench.py that needs no GPU: the multi-rank reduction (two gloo ranks on the
CPU), the whole-job throughput, the reference arm's rank rule and the traffic record."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 3.0 + 4.0 * rank          # rank 1 is the slow replica
        got = bench.max_over_ranks(local)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 7.0, 1: 7.0}


def test_max_over_ranks_without_a_group_is_identity():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(2.5) == 2.5


def test_job_throughput_is_weak_scaling():
    one = bench.job_gbps(1, 9.45e6, 0.005)
    assert one == pytest.approx(1890.0)
    assert bench.job_gbps(4, 9.45e6, 0.005) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_traffic_record_is_used_only_for_the_source_it_was_measured_on(monkeypatch, tmp_path):
    # the committed record carries the kernel source's sha256 it was captured on; bench.py
    # reports its figures only while the source is unchanged, and null otherwise
    rec = json.load(open(bench.TRAFFIC_PATH))
    assert len(rec["kernel_source_sha256"]) == 64 and rec["dram_bytes_per_launch"]
    fake = dict(rec, kernel_source_sha256=bench.kernel_source_sha256())
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(fake))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    name = next(iter(rec["dram_bytes_per_launch"]))
    assert bench.kernel_traffic(name) == rec["dram_bytes_per_launch"][name]
    monkeypatch.setattr(bench, "kernel_source_sha256", lambda: "0" * 64)
    assert bench.kernel_traffic(name) is None


def test_workload_byte_accounting():
    # the fused call reads both weights and writes [M, N]; gate_up writes [M, 2N]
    calls = {k: bench.Call(spec, "cpu", 1, "cpu") for k, spec in
             (("sw", ("gate_up_swiglu", 64, 256, 2, 5, "bf16")), ("gu", ("gate_up", 64, 256, 2, 5, "f32")))}
    per_row = 256 * 0.5 + 256 / 16
    assert calls["sw"].weight_bytes() == calls["gu"].weight_bytes() == 2 * 64 * per_row
    assert calls["sw"].alg_bytes() == 2 * 64 * per_row + 2 * 256 * 2 + 2 * 64 * 2
    assert calls["gu"].alg_bytes() == 2 * 64 * per_row + 2 * 256 * 2 + 2 * 128 * 4


def test_cpu_baseline_reports_the_oracle_on_a_bounded_sample():
    calls = [bench.Call(("dense", 64, 256, 1, 0, "f32"), "cpu", 1, "cpu"),
             bench.Call(("gate_up_swiglu", 32, 256, 2, 1, "bf16"), "cpu", 1, "cpu")]
    base = bench.cpu_baseline(calls, target_s=0.3)
    assert base["kind"] == "oracle" and base["cores"] >= 1 and base["value"] > 0
    assert base["unit"].startswith("GB/s")
    assert "every GEMV of one step" in base["sample"] or "% of the output rows" in base["sample"]


def test_in_run_output_check_accepts_oracle_outputs_and_flags_a_wrong_one():
    # bench.py checks a sample of every timed output against the oracle; here the "timed"
    # outputs are the oracle's own values (accepted), then one column is spoiled (flagged)
    import oracle
    from nvfp4_weight_only_gemv_gb300 import synth
    calls = [bench.Call(("dense", 40, 256, 2, 3, "bf16"), "cpu", 1, "cpu"),
             bench.Call(("gate_up_swiglu", 24, 256, 1, 4, "f32"), "cpu", 1, "cpu")]
    h = calls[0].host
    yr, _ = oracle.gemv(h["w"].numpy(), h["s"].numpy(), h["g"], synth.bf16_bits(h["x"]))
    calls[0].sets[0]["y"].copy_(torch.from_numpy(yr).to(torch.bfloat16))
    h = calls[1].host
    yr, _ = oracle.gate_up_swiglu(h["wg"].numpy(), h["sg"].numpy(), h["gg"], h["wu"].numpy(), h["su"].numpy(),
                                  h["gu"], synth.bf16_bits(h["x"]), bench.SWIGLU_CLAMP)
    calls[1].sets[0]["y"].copy_(torch.from_numpy(yr).float())
    res = bench.check_outputs(calls, n_cols=64)
    assert res["ok"] and res["checked"] == 2 * 40 + 24 and res["outside_tolerance"] == 0
    calls[0].sets[0]["y"][1, 7] += 0.5
    res = bench.check_outputs(calls, n_cols=64)
    assert not res["ok"] and res["outside_tolerance"] == 1
