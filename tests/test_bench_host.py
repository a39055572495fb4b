"""Host-side logic of bench.py, on the CPU: byte accounting, the max-over-ranks
reduction across two gloo ranks, the reference arm under torchrun, and the
traffic record that ties an ncu capture to the kernel sources it measured."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_step_bytes_by_hand():
    inp = workloads.make_case(B=3, Hq=4, Hkv=2, D=64, P=16, seq_lens=[17, 1, 40], active=[1, 0, 1], seed=1)
    by = bench.step_bytes(inp)
    kv = (17 + 40) * 2 * 64 * 2 * 2
    assert by["kv"] == kv and by["active"] == 2
    pt = (2 + 3) * 4
    per_row = 4 * 64 * 2 + 2 * 2 * 64 * 2 + 2 * 2 * 64 * 2 + 4 * 64 * 2
    assert by["step"] == kv + 2 * per_row + pt + 8 * 3
    assert by["attn"] == kv + 2 * (4 * 64 * 4 + 4 * 64 * 2) + pt + 8 * 3
    assert by["flops"] == 4 * 4 * 64 * (17 + 40)     # q.K and p.V: 2 flops per element each, active rows only


def test_oracle_accuracy_check_flags_a_wrong_output():
    import oracle
    inp = workloads.make_case(B=3, Hq=4, Hkv=2, D=64, P=16, seq_lens=[17, 1, 40], active=[1, 0, 1], seed=3)
    ref = oracle.reference_step(inp)["out"]
    ok = bench.oracle_accuracy(inp, ref.clone(), {})
    assert ok["within_tolerance"] and ok["max_abs_err"] == 0.0 and ok["worst_margin"] < 0
    bad = ref.clone()
    bad[2, 3, 5] += 0.05                              # an active row, far outside 2e-3 + 1e-2 |ref|
    got = bench.oracle_accuracy(inp, bad, {})
    assert not got["within_tolerance"] and abs(got["max_abs_err"] - 0.05) < 1e-2
    junk = ref.clone()
    junk[1] = float("nan")                            # the padding row is not compared
    assert bench.oracle_accuracy(inp, junk, {})["within_tolerance"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w = bench.dist_setup()
    bench.barrier(w)
    q.put((r, bench.max_over_ranks(1.5 + r, w)))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2.5), (1, 2.5)]


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "6", "--warmup", "2", "--workload", "tiny"]
    env = {**os.environ, "CUDA_VISIBLE_DEVICES": ""}
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_must_match_kernel_sources(tmp_path):
    sha = bench.kernel_source_sha()
    f = tmp_path / "rec.md"
    f.write_text(f"kernel source sha256[:16]: {sha}\ndram bytes per launch (read + write): 123456\n")
    assert bench.recorded_traffic("c64", str(f)) == 123456
    f.write_text("kernel source sha256[:16]: 0000000000000000\ndram bytes per launch (read + write): 1\n")
    assert bench.recorded_traffic("c64", str(f)) is None
    assert bench.recorded_traffic("c64", str(tmp_path / "missing.md")) is None


def test_clock_summary_uses_samples_under_load_and_collects_throttle_reasons():
    # nvidia-smi csv rows: index, sm, max sm, power, active reasons, hw_slowdown,
    # hw_thermal, sw_thermal, sw_power_cap, utilisation
    rows = ["0, 1000, 2070, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active, 0",
            "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active, 100",
            "0, 2055, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active, 98",
            "0, 2070, 2070, 910.0, 0x0, Not Active, Not Active, Not Active, Not Active, 99",
            "garbage line"]
    c = bench.Clocks.summarise(rows)
    assert c["samples"] == 4 and c["samples_under_load"] == 3
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0       # the idle 1000 MHz sample is left out
    assert c["reasons"] == ["sw_power_cap"]
    assert c["power_w_median"] == 910.0
    idle = bench.Clocks.summarise(rows[:1])                           # no sample under load: all samples
    assert idle["samples_under_load"] == 0 and idle["sm_mhz"] == 1000.0


def test_rates_fractions_of_measured_peak_and_specification():
    by = {"step": 6_000_000, "active": 64}
    r = bench.rates(by, ms_step=0.001, world=2, peak=6000.0, L=4)     # 1 us per step
    assert r["hbm_gbs"] == 6000.0 and r["frac_of_peak"] == 1.0
    assert r["frac_of_spec"] == round(6000.0 / bench.SPEC_HBM_GBS, 4)
    assert r["tokens_per_s"] == 64 * 2 / 1e-6                        # whole job: both ranks
    assert r["ms_per_launch"] == 0.00025
    assert "tflops" not in r
    r = bench.rates({**by, "flops": 2_000_000}, ms_step=0.001, world=1, peak=6000.0, L=1)
    assert r["tflops"] == 2.0                                         # 2 MFLOP in 1 us
