"""Host logic of the multi-rank benchmark on CPU with two gloo ranks: every rank runs its own
copy of the workload (no collective on the data path); the step time reported is the max over
ranks, and the reference arm runs on rank 0 only."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.reduce_max(float(rank + 1) * 1.5, world)
        w, r, local = bench._dist()
        q.put((rank, got, w, r, local))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_rank_env():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got, w, r, local in res:
        assert got == pytest.approx(3.0)      # max of 1.5 and 3.0 on every rank
        assert (w, r, local) == (world, rank, rank)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes_match_the_stated_formula():
    import bench
    from selective_state_space_145_b300 import inputs

    w = inputs.WORKLOADS["block_bf16_b8_d2048_l2048_n16_k4"]
    assert bench.algorithmic_bytes(w) == 270_721_024
    w = inputs.WORKLOADS["longscan_bf16_b1_d1536_l131072_n16"]
    assert bench.algorithmic_bytes(w) == 1_619_210_240
    w = inputs.WORKLOADS["decode_bf16_b256_d5120_n16_k4_x64"]
    assert bench.algorithmic_bytes(w) == 194_473_984 * 64


def test_issue_floor_and_backward_bytes():
    """The special-function-pipe floor and the backward's algorithmic bytes, spelled out for one
    shape."""
    import bench
    from selective_state_space_145_b300 import inputs

    w = inputs.WORKLOADS["block_f32_b2_d1024_l1024_n16_k4"]
    per_t = 2 * 1024 * 16
    # 8 chunks of 128: main 1024 steps, carry 7 * 128 steps; one exp2 per update at 32 per clock
    # per SM, 148 SMs at the maximum SM clock
    r = bench.alu_roofline(w, 1e-3, 128, 148)
    floor = (per_t * 1024 + per_t * 7 * 128) / (148 * 32 * bench._sm_max_mhz() * 1e6)
    assert r["frac"] == pytest.approx(floor / 1e-3)
    assert r["carry_updates"] == per_t * 7 * 128
    assert bench.alu_roofline(inputs.WORKLOADS["decode_bf16_b256_d5120_n16_k4_x64"], 1e-3, 0, 148) is None
    tok, bnl = 2 * 1024 * 1024, 2 * 16 * 1024
    assert bench.bwd_algorithmic_bytes(w) == (tok * 4 * 7 + bnl * (2 * 4 + 8) + 2 * 1024 * 16 * 4 * 3
                                              + 1024 * 16 * 4 * 2 + 1024 * 4 * 4)


def test_ssd_work_and_bytes():
    """The state-space-duality workload's FLOP and byte accounting, spelled out."""
    import bench
    from selective_state_space_145_b300 import inputs

    w = inputs.SSD_WORKLOADS["ssd_bf16_b8_l2048_h32_p64_n128"]
    Q, N, P = 128, 128, 64
    units = 8 * 32 * (2048 // Q)
    alg, exe = bench.ssd_flops(w)
    assert alg == units * (2 * Q * Q * N + 2 * Q * Q * P + 2 * Q * N * P + 2 * N * Q * P)
    # the three computed operands (G', H_in and the decay-scaled B) enter as hi + lo pairs: their
    # three GEMMs run twice
    assert exe == alg + units * (2 * Q * Q * P + 2 * Q * N * P + 2 * N * Q * P)
    tok = 8 * 2048
    assert bench.ssd_algorithmic_bytes(w) == (tok * 32 * 64 * 2 * 2 + tok * 32 * 2 + 2 * tok * 128 * 2
                                              + 8 * 32 * 64 * 128 * 4 + 32 * 4 * 3)
    assert w.updates == 8 * 2048 * 32 * 64 * 128


def test_traffic_records_follow_code_not_comments():
    """A recorded DRAM-traffic figure belongs to the code it was measured on: the source hash
    ignores comments and layout, and changes with any code token or string literal."""
    import bench

    base = 'int f(int a) {\n  // old note\n  return a * 2; /* x */\n}\nconst char* s = "a // b";\n'
    same = 'int f(int a)\n{\n  /* a new, longer\n     note */\n  return a * 2;   // y\n}\nconst char* s = "a // b";\n'
    code = 'int f(int a) {\n  return a * 3;\n}\nconst char* s = "a // b";\n'
    lit = 'int f(int a) {\n  return a * 2;\n}\nconst char* s = "a // c";\n'
    cb = bench.source_code_only(base)
    assert cb == bench.source_code_only(same)
    assert cb != bench.source_code_only(code)
    assert cb != bench.source_code_only(lit)
    assert "old note" not in cb and '"a // b"' in cb


@pytest.mark.parametrize("workload", ["block_f32_b2_d1024_l1024_n16_k4", "ssd_bf16_b8_l2048_h32_p64_n128"])
def test_reference_arm_line_on_rank_zero(monkeypatch, capsys, workload):
    """Rank 0 prints one JSON line carrying the contract's keys; the oracle's sampling is replaced
    by a fixed rate so that only the line's assembly is under test."""
    import json

    import bench
    from selective_state_space_145_b300 import inputs

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    rate = 2.5e9
    monkeypatch.setattr(bench, "oracle_sample_rate", lambda *a, **k: (rate, 4, "stub sample"))
    monkeypatch.setattr(bench, "ssd_oracle_rate", lambda *a, **k: (rate, 4, "stub sample"))
    assert bench.main(["--impl", "reference", "--workload", workload, "--steps", "2", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    w = inputs.WORKLOADS.get(workload) or inputs.SSD_WORKLOADS[workload]
    assert line["impl"] == "reference" and line["value"] == rate and line["config"]["workload"] == workload
    assert line["steps"] == 2 and line["warmup"] == 3 and line["higher_is_better"] is True
    assert abs(line["ms_per_step"] - w.updates / rate * 1e3) < 1e-9 * line["ms_per_step"]
    assert line["cpu_baseline"] == {"value": rate, "unit": line["unit"], "cores": 4, "kind": "oracle",
                                    "sample": "stub sample"}
    assert line["e2e"] == {"value": rate, "unit": line["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
