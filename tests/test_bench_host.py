"""Host-side logic of bench.py on CPU: the replica (weak-scaling) reduction
over two gloo ranks, the algorithmic byte counts, and the clock summary."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    ws, r = bench.dist_init("gloo")
    bench.barrier()
    # each replica timed a different number of ms and did 10 steps
    t = bench.max_over_ranks(100.0 + 50.0 * rank)
    n = bench.sum_over_ranks(10)
    q.put((r, ws, t, n))
    dist.destroy_process_group()


def test_replica_reduction_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    for _, ws, t, n in res:
        assert ws == 2 and t == 150.0 and n == 20.0  # max time, summed units


def test_single_process_reduction_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.sum_over_ranks(7) == 7.0


def test_algorithmic_bytes_qwen_shape():
    from workload import CONFIGS
    cfg = CONFIGS["qwen3_4b_bf16"]
    fused = bench.algorithmic(cfg, 1, 512, 4.5, True)
    sep = bench.algorithmic(cfg, 1, 512, 4.5, False)
    # weights: draft (Hq*dh + 2*Hkv*dh + N) * D + D * (Hq*dh + Hm*P), commit
    # (2*Hkv*dh + Hm*P + N + Hm) * D, bf16
    w = ((4096 + 2048 + 128) * 2560 + 2560 * (4096 + 5120) + (2048 + 5120 + 128 + 80) * 2560) * 2
    assert w < fused["step_bytes"] < w * 1.1
    # the separate path moves the same bytes plus one more read of the state
    state = 80 * 64 * 128 * 4
    tot = lambda a: sum(b for b, _ in a["families"].values())
    assert tot(fused) == fused["step_bytes"]
    assert tot(sep) - tot(fused) == pytest.approx(state)
    # one layer: every family of the fused path launches once, except the
    # later-layer slot projections (none)
    assert fused["families"]["draft_proj"] == (0, 0)
    assert all(n == 1 for k, (_, n) in fused["families"].items() if k != "draft_proj")


def test_algorithmic_bytes_memory_horizon():
    from workload import CONFIGS
    cfg = CONFIGS["qwen3_4b_bf16"]
    base = bench.algorithmic(cfg, 1, 512, 4.5, True)["families"]["commit_state"][0]
    last = bench.algorithmic(cfg.replace(mem_horizon=1), 1, 512, 4.5, True)["families"]
    ring = bench.algorithmic(cfg.replace(mem_horizon=512), 1, 512, 4.5, True)["families"]
    state = 80 * 64 * 128 * 4
    # last feature: the state is written, never read
    assert base - last["commit_state"][0] == pytest.approx(state)
    # horizon 512: leaving and new rows of x, B, dt, and 512 dt per head
    extra = 4.5 * 2 * (5120 + 128 + 80) * 4 + 80 * 512 * 4
    assert ring["commit_state"][0] - base == pytest.approx(extra)
    assert bench.ablation_config(cfg) == {}
    assert bench.ablation_config(cfg.replace(cross_slot=False, mem_horizon=1))["ablation"][
        "mem_horizon"] == 1


def test_round_projection_launch_count():
    """The serving batch's commit product (512 rows x 3 layers' columns) has
    more 128 x 256 tiles than SMs: the round projection is two launches (the
    commit projection, then the slot projection); one request's is one
    grouped launch, and without an SM count the model keeps one."""
    from workload import CONFIGS
    serving = CONFIGS["serving_qwen3_4b_b64"]
    Nc = 2 * 8 * 128 + 80 * 64 + 128 + 80
    tiles = (64 * 8 // 128) * -(-(3 * Nc) // 256)
    assert tiles >= 152
    fam = bench.algorithmic(serving, 64, 512, 4.5, True, 152)["families"]
    assert fam["round_proj"][1] == 2
    assert bench.algorithmic(serving, 64, 512, 4.5, True)["families"]["round_proj"][1] == 1
    c1 = CONFIGS["qwen3_4b_bf16"]
    assert bench.algorithmic(c1, 1, 512, 4.5, True, 152)["families"]["round_proj"][1] == 1
    # the bytes do not depend on how the projection is launched
    assert fam["round_proj"][0] == bench.algorithmic(serving, 64, 512, 4.5, True)["families"][
        "round_proj"][0]


def test_clock_summary_parses_samples(tmp_path):
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "clk.csv")
    with open(c.path, "w") as f:
        f.write("0, 1900, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    c.proc = object()
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1985.0) and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_only_for_unchanged_kernels(tmp_path, monkeypatch):
    import json
    (tmp_path / "profiles").mkdir()
    real = bench.kernel_sources_digest()
    for digest, want in ((real, 123), ("0" * 64, None)):
        (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
            {"workloads": {"w": {"kernel_sources_sha256": digest,
                                 "per_launch_bytes": {"round_proj": 123}}}}))
        monkeypatch.setattr(bench, "ROOT", str(tmp_path))
        monkeypatch.setattr(bench, "kernel_sources_digest", lambda: real)
        assert bench.measured_traffic("w", "round_proj") == want
        assert bench.measured_traffic("w", "out_proj") is None


def test_reference_arm_line(capsys):
    """The reference arm (the float64 oracle on the host cores) prints one
    JSON line with the GPU arm's metric, unit and workload keys, its sample
    described as the oracle's, and an e2e entry that moves no bytes."""
    import json
    assert bench.main(["--impl", "reference", "--config", "tiny_fp32",
                       "--steps", "3", "--warmup", "3"]) in (0, None)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True
    c = d["config"]
    assert c["workload"] == "tiny_fp32"
    for k in ("batch_per_gpu", "prefix", "prefix_cap", "layers", "window", "block"):
        assert k in c
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
