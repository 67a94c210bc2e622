"""Benchmark of the HyFlash drafter hot path on one GB300 (or N replicas).

A step is one speculative round on device-resident inputs: hf_draft (all
layers: slot projections, window+block attention, memory read, output
projections) followed by hf_commit (count check, projections, ring append,
sequential memory update) for every request of the batch. The two calls are
captured once into a CUDA graph that reads fixed staging buffers; each step
stages its round's inputs and replays the graph (how a serving loop would
run it, without per-kernel host launch cost). The prefix is folded once
beforehand with hf_prefill, which is timed on its own under "prefill".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl hyflash|reference]

Multi-GPU (torchrun, one rank per GPU): each rank runs an independent replica
with its own requests (weak scaling, no collective on the data path); the
barrier/max-over-ranks timing is the only communication.

--impl reference times the float64 CPU oracle (plain NumPy, as it stands) on
the host cores for the same metric: there is no other implementation of this
method to run.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "drafter draft-steps/s and committed tokens/s at 1 GB300; % of HBM/tensor roofline"
UNIT = "draft-steps/s"
DEFAULT_CONFIG = "serving_qwen3_4b_b64"


# ------------------------------------------------------------------ distributed helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ algorithmic sizes

def algorithmic(cfg, batch: int, window_fill: float, mean_accept: float, fused: bool,
                num_sms: int = 0):
    """Bytes each step must move at minimum (weights, window, state and the
    slot / feature I/O read or written once), per kernel family of the path
    that runs: {family: (bytes per step, launches per step)}.

    fused (hf_round): the commit projection and the first layer's slot
    projection share one launch, and the first layer's memory read is made
    on the updated state inside the state update, so that state is read once
    per step; later layers read their state again at draft time (their C
    depends on the layer below, which needs the updated state first).
    step_bytes is the fused figure: the least traffic any schedule of a
    step needs. With num_sms given, a wide batch whose commit product alone
    has a 128 x 256 tile per SM counts two round-projection launches (the
    commit projection on the persistent GEMM, then the slot projection).

    Memory horizon M (ablation): M = 1 writes the state without reading it;
    M > 1 also reads the leaving rows' and writes the new rows' x, B, dt
    and reads M dt values per head for the horizon's decay sum."""
    e = cfg.elem_bytes
    D, hq, hkv, dh, W = cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.window
    din, N, Hm, P, S, L = cfg.d_inner, cfg.d_state, cfg.ssm_heads, cfg.ssm_headdim, cfg.block, cfg.n_layers
    QD = hq * dh
    Nd = QD + 2 * hkv * dh + N
    Nz = QD + din
    gdn = getattr(cfg, "memory", "mamba2") == "gdn"
    Nc = 2 * hkv * dh + din + N + Hm * (2 if gdn else 1)   # gated delta: + beta columns
    R = batch * S
    rows = batch * mean_accept
    we = e if getattr(cfg, "weight_bits", 16) != 4 else 0.5 + 4.0 / 128  # 4-bit codes + group params
    w_draft, w_out, w_commit = we * Nd * D, we * D * Nz, we * L * Nc * D
    io_draft = e * R * D + 4 * R * Nd                 # slot rows in, projections out
    io_out = e * R * Nz + 2 * e * R * D                # mix in, residual in, output out
    window = batch * window_fill * 2 * hkv * dh * e    # one layer's valid K and V
    state = batch * Hm * P * N * 4                     # one layer's states, read once
    io_attn = 4 * R * Nd + e * R * QD                  # projections in, attention out
    io_mem = 4 * R * N + e * R * din                   # C in, memory read out
    ns = din + N + Hm * (2 if gdn else 1)              # memory-input columns per row
    commit_io = e * rows * D + L * rows * (2 * hkv * dh * e + ns * 4)
    state_io = L * rows * ns * 4
    M = int(getattr(cfg, "mem_horizon", 0) or 0)
    state_rw = 1 if M == 1 else 2                      # M = 1: the old state is not read
    if M > 1:
        state_io += L * (rows * 2 * (din + N + Hm) * 4 + batch * Hm * min(M, window_fill) * 4)

    n0 = batch * (S + 1)
    two = bool(num_sms) and n0 > 32 and (-(-n0 // 128)) * (-(-(L * Nc) // 256)) >= num_sms

    def fused_fams():
        return {
            "round_proj": (w_commit + commit_io + w_draft + io_draft, 2 if two else 1),
            "draft_proj": ((L - 1) * (w_draft + io_draft), L - 1),
            "commit_state": (L * state_rw * state + state_io + io_mem, 1),
            "attn_mem": (L * (window + io_attn) + (L - 1) * (state + io_mem), L),
            "out_proj": (L * (w_out + io_out), L),
        }

    fam = fused_fams() if fused else {
        "draft_proj": (L * (w_draft + io_draft), L),
        "attn_mem": (L * (window + state + io_attn + io_mem), L),
        "out_proj": (L * (w_out + io_out), L),
        "commit_proj": (w_commit + commit_io, 1),
        "commit_state": (L * state_rw * state + state_io, 1),
    }
    flops = L * 2 * R * D * (Nd + Nz) + 2 * rows * D * L * Nc
    if getattr(cfg, "full_block", False):
        # the full block runs hf_commit then hf_draft_tokens: the layer's
        # products plus x_s | z_s in the slot projection, the norms, the
        # commit's conv / RoPE pass, the SwiGLU MLP and the LM head
        F, V = cfg.mlp_dim, cfg.vocab
        xz = 2 * din
        fam = {
            "draft_proj": (L * (we * (Nd + xz) * D + io_draft + 4 * R * xz), L),
            "attn_mem": (L * (window + state + io_attn + io_mem), L),
            "out_proj": (L * (w_out + io_out), L),
            "commit_proj": (w_commit + commit_io, 1),
            "commit_state": (L * 2 * state + state_io + L * (batch * 6 * (din + N) * 4
                                                             + rows * 2 * (din + N) * 4), 2),
            "mlp": (L * (3 * we * D * F + e * R * D + 4 * R * 2 * F * 2 + e * R * F * 2
                         + 2 * e * R * D), 3 * L),
            "head": (we * V * D + e * R * D + 4 * R * V * 2 + 4 * R, 2),
            "other": (L * (2 * 2 * e * R * D + 4 * R * (QD + 2 * hkv * dh) * 2
                           + 2 * e * R * din + 4 * R * 2 * din) + 2 * e * R * D, 4 * L + 1),
        }
        flops += L * 2 * R * D * (xz + 3 * F) + 2 * R * D * V
        return {"families": fam, "step_bytes": sum(b for b, _ in fam.values()), "step_flops": flops}
    step = sum(b for b, _ in fused_fams().values())
    return {"families": fam, "step_bytes": step, "step_flops": flops}


def layer_weights(cfg, layer: int):
    """The workload's weights of one layer (4-bit codes when weight_bits = 4)."""
    from workload import make_layer_weights, make_layer_weights_q4
    return (make_layer_weights_q4 if getattr(cfg, "weight_bits", 16) == 4 else make_layer_weights)(
        cfg, layer)


def set_layer_weights(drafter, cfg, layer: int):
    if getattr(cfg, "full_block", False):
        from workload import make_block_weights
        drafter.set_block_weights(layer, make_block_weights(cfg, layer))
        return
    w = layer_weights(cfg, layer)
    (drafter.set_weights_q4 if getattr(cfg, "weight_bits", 16) == 4 else drafter.set_weights)(layer, w)


def ablation_config(cfg) -> dict:
    """The ablation modes in force, if any (config keys of the JSON line)."""
    out = {}
    if not getattr(cfg, "cross_slot", True):
        out["cross_slot"] = "off (each slot sees the window and its own key)"
    if getattr(cfg, "mem_horizon", 0):
        out["mem_horizon"] = int(cfg.mem_horizon)
    res = {"ablation": out} if out else {}
    if getattr(cfg, "memory", "mamba2") == "gdn":
        res["memory"] = "gated delta rule (GDN)"
    if getattr(cfg, "weight_bits", 16) == 4:
        res["weights"] = "4-bit codes, bf16 scale + zero point per 128 inputs (skinny products dequantise on chip)"
    if getattr(cfg, "full_block", False):
        res["block"] = {"kind": "full drafter block (pre-norms, RoPE, conv1d, skip/gate, SwiGLU, LM head + argmax)",
                        "mlp_dim": cfg.mlp_dim, "vocab": cfg.vocab,
                        "step": "hf_commit then hf_draft_tokens"}
    return res


def kernel_sources_digest() -> str:
    """sha256 over the CUDA sources (names and bytes, sorted by name)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_drafter_hf_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload: str, family: str):
    """DRAM bytes per launch of a kernel family from the committed ncu
    captures (profiles/traffic.json), or None when none was taken for this
    workload or the kernels changed since."""
    import json as _json
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            t = _json.load(fh)
    except (OSError, ValueError):
        return None
    # one capture per workload, keyed by the sources it was taken with
    w = t.get("workloads", {}).get(workload, {})
    if w.get("kernel_sources_sha256") != kernel_sources_digest():
        return None
    return w.get("per_launch_bytes", {}).get(family)


def prefill_flops(cfg, total_tokens: int, ring_rows: int) -> float:
    D, din, N, Hm, P = cfg.d_model, cfg.d_inner, cfg.d_state, cfg.ssm_heads, cfg.ssm_headdim
    kvd = cfg.n_kv_heads * cfg.head_dim
    per_tok = 2 * D * (din + N + Hm) + 2 * Hm * P * N
    return cfg.n_layers * (total_tokens * per_tok + ring_rows * 2 * D * 2 * kvd)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle timing

def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


ORACLE_PREFIX_CAP = 8192    # oracle prefill length cap (a round's cost does not depend on it)
ORACLE_BATCH_CAP = 2        # requests the oracle drafts for in its timed sample


def oracle_rounds(cfg, batch: int, steps: int, warmup: int, budget_s: float, seed: int = 0):
    """Time the float64 oracle on host cores: prefill untimed, then rounds of
    draft + commit; stops early after budget_s seconds of timed work. Large
    workloads run on a bounded sample: at most ORACLE_BATCH_CAP requests whose
    prefixes are capped at ORACLE_PREFIX_CAP tokens (the window and memory
    are full either way, so a round costs the same)."""
    from oracle import hyflash_oracle as O
    from workload import (make_accepted, make_layer_weights, make_prefix_feats,
                          make_prefix_lens, make_round_inputs)
    if getattr(cfg, "full_block", False):  # the block oracle with its LM head
        from oracle import full_block as FB
        from workload import make_block_weights, make_head_weights
        orc = FB.OracleBlockDrafter(cfg, [make_block_weights(cfg, l) for l in range(cfg.n_layers)],
                                    make_head_weights(cfg), batch)
    else:
        weights = [layer_weights(cfg, l) for l in range(cfg.n_layers)]
        orc = O.OracleDrafter(cfg, weights, batch)
    lens = [min(L, ORACLE_PREFIX_CAP) for L in make_prefix_lens(cfg)[:batch]]
    orc.prefill(lens, make_prefix_feats(cfg, lens, seed=seed))
    for r in range(warmup):
        slot, feats = make_round_inputs(cfg, r, batch, seed=seed)
        orc.draft(slot)
        orc.commit(feats, make_accepted(cfg, r, batch, seed=seed).numpy())
    done, accepted, t_total = 0, 0, 0.0
    for r in range(warmup, warmup + steps):
        slot, feats = make_round_inputs(cfg, r, batch, seed=seed)
        n = make_accepted(cfg, r, batch, seed=seed).numpy()
        t0 = time.perf_counter()
        orc.draft(slot)
        orc.commit(feats, n)
        t_total += time.perf_counter() - t0
        done += 1
        accepted += int(n.sum())
        if t_total > budget_s:
            break
    return done, accepted, t_total


def cpu_sample(cfg, steps: int, warmup: int, budget: float):
    """Oracle draft-steps/s for the whole batch, from a bounded sample."""
    sb = min(cfg.batch, ORACLE_BATCH_CAP)
    done, acc, t = oracle_rounds(cfg, sb, steps, warmup, budget)
    scale = sb / cfg.batch  # a step drafts and commits for every request of the batch
    v = done / t * scale if t > 0 else 0.0
    sample = (f"{done} rounds (draft+commit) of {cfg.name} for {sb} of {cfg.batch} requests "
              f"(rate scaled by {sb}/{cfg.batch}), prefixes capped at {ORACLE_PREFIX_CAP} tokens, "
              f"the float64 NumPy oracle as it stands (no fp32 instantiation), after an untimed "
              f"oracle prefill and {warmup} warm-up rounds")
    return v, acc / t * (1 / scale) if t > 0 else 0.0, done, t, sample


def run_reference(args, cfg):
    ws, rank = dist_init("gloo")
    if rank != 0:
        return 0
    if cfg.rounds == 0:
        print(json.dumps({"impl": "reference", "unavailable":
                          "prefill sweep: the float64 oracle folds 4K-128K-token prefixes at "
                          "batch 8 far beyond a bounded run"}), flush=True)
        return 0
    budget = float(os.environ.get("HF_REF_BUDGET_S", "120"))
    v, tok_rate, done, t, sample = cpu_sample(cfg, args.steps, args.warmup, budget)
    batch = cfg.batch
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 * t / max(done, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "committed_tokens_per_s": tok_rate,
        "config": {"workload": cfg.name, "batch_per_gpu": batch,
                   "prefix": (f"log-uniform [{cfg.prefix_lo}, {cfg.prefix_hi}]"
                              if cfg.prefix_lo else cfg.prefix),
                   "prefix_cap": ORACLE_PREFIX_CAP,
                   "api": "the oracle's draft, then its commit of the round",
                   "layers": cfg.n_layers, "window": cfg.window, "block": cfg.block,
                   "l2": "n/a (CPU)", **ablation_config(cfg)},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def prefix_features(cfg, lens, seed, dev):
    """Seeded prefix features ~N(0,1) on the device. Up to 2^26 values they
    come from the shared CPU generator (the bytes the oracle sees); larger
    prefixes are drawn directly on the GPU (a seeded CUDA generator)."""
    import torch
    from workload import make_prefix_feats
    total = sum(lens)
    if total * cfg.d_model <= (1 << 26):
        return make_prefix_feats(cfg, lens, seed=seed).to(dev)
    g = torch.Generator(device=dev).manual_seed(7919 + seed)
    return torch.randn((total, cfg.d_model), generator=g, device=dev).to(cfg.torch_dtype)


def run_prefill_sweep(args, cfg):
    """Prefill throughput: each step folds a batch of prefixes (all layers)."""
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    from speculative_decoding_drafter_hf_gb300 import build as _b
    _b.build()
    import speculative_decoding_drafter_hf_gb300 as hf
    from workload import make_layer_weights
    cfg = cfg.replace(chunk=args.chunk, n_layers=args.layers,
                      prefix=args.prefix if args.prefix else cfg.prefix)
    batch = cfg.batch
    lens = [cfg.prefix] * batch
    tseg = max(4096, min(cfg.prefix, 16384))
    drafter = hf.Drafter(cfg, batch, device=local, prefill_tokens_max=tseg)
    for l in range(cfg.n_layers):
        drafter.set_weights(l, make_layer_weights(cfg, l))
    feats = prefix_features(cfg, lens, rank, dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        drafter.prefill(feats, lens)
    drafter.sync()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    n0 = drafter.launch_count()
    ev = []
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            drafter.prefill(feats, lens)
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
    barrier()
    drafter.sync()
    launches = drafter.launch_count() - n0
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dev)
    tokens = sum(lens)
    all_tok = sum_over_ranks(tokens * args.steps, dev)
    value = all_tok / (total_ms / 1e3)
    ring_rows = sum(min(L, cfg.window) for L in lens)
    flops = prefill_flops(cfg, tokens, ring_rows)
    peaks = {}
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        peaks = json.load(open(pp))
    tc_peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
    achieved = flops * args.steps / (total_ms / 1e3) / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "prefill tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
            "data": "synthetic",
            "config": {"workload": cfg.name, "batch_per_gpu": batch, "prefix": cfg.prefix,
                       "layers": cfg.n_layers, "chunk": cfg.chunk,
                       "l2": f"flushed between steps ({2 * l2 >> 20} MiB write, untimed)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "tensor", "kernel": "whole prefill", "achieved": achieved,
                         "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                         "traffic": None,
                         "peak_source": "measured (sustained)" if peaks else "fallback",
                         "algorithmic_flops_per_step": flops},
            "gpu_launches": int(launches), "cpu_baseline": None,
            "e2e": None, "clocks": clk.summary()}), flush=True)
    drafter.close()
    return 0


def run_hyflash(args, cfg):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)

    from speculative_decoding_drafter_hf_gb300 import build as _b
    _b.build()
    import speculative_decoding_drafter_hf_gb300 as hf
    from workload import (make_accepted, make_layer_weights, make_prefix_feats, make_prefix_lens,
                          make_round_inputs)

    batch = cfg.batch
    seed = rank  # each replica drafts for its own requests
    drafter = hf.Drafter(cfg, batch, device=local)
    for l in range(cfg.n_layers):
        set_layer_weights(drafter, cfg, l)
    block = getattr(cfg, "full_block", False)
    if block:
        from workload import make_head_weights
        drafter.set_head_weights(make_head_weights(cfg))
    lens = make_prefix_lens(cfg, seed=0)[:batch]
    if args.prefix_max:  # smaller prefill (e.g. for profiling); rounds unchanged once windows fill
        lens = [min(L, args.prefix_max) for L in lens]
    total = sum(lens)
    feats = prefix_features(cfg, lens, seed, dev)
    stream = torch.cuda.current_stream()

    # ---- prefill (one warm-up, then timed)
    drafter.prefill(feats, lens)
    drafter.sync()
    pf_times = []
    for _ in range(2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        drafter.prefill(feats, lens)
        b.record(stream)
        b.synchronize()
        pf_times.append(a.elapsed_time(b))
    drafter.sync()
    pf_ms = min(pf_times)
    ring_rows = sum(min(L, cfg.window) for L in lens)
    pf_flops = prefill_flops(cfg, total, ring_rows)
    del feats

    # ---- per-round inputs, resident on the device
    nsteps = args.warmup + args.steps
    slots, commits, counts = [], [], []
    for r in range(nsteps):
        s, f = make_round_inputs(cfg, r, batch, seed=seed)
        slots.append(s)
        commits.append(f)
        counts.append(make_accepted(cfg, r, batch, seed=seed))
    d_slot = torch.stack(slots).to(dev)
    d_feat = torch.stack(commits).to(dev)
    d_cnt = torch.stack(counts).to(dev)
    out = torch.empty((batch, cfg.block, cfg.d_model), dtype=drafter.torch_dtype, device=dev)
    tokens = torch.empty((batch, cfg.block), dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    # Fixed staging buffers: one round (draft + commit) is captured into a
    # CUDA graph reading from them; each step stages its round's inputs
    # (device to device, outside the timed events) and replays the graph. The
    # three inputs sit in one byte buffer (16-byte aligned parts), so that the
    # end-to-end run moves a step's inputs with one host-to-device copy.
    parts = [(d_slot[0].numel() * d_slot.element_size(), d_slot.dtype, d_slot.shape[1:]),
             (d_feat[0].numel() * d_feat.element_size(), d_feat.dtype, d_feat.shape[1:]),
             (d_cnt[0].numel() * d_cnt.element_size(), d_cnt.dtype, d_cnt.shape[1:])]
    offs, o = [], 0
    for nb, _, _ in parts:
        offs.append(o)
        o += (nb + 15) // 16 * 16
    st_blob = torch.zeros(o, dtype=torch.uint8, device=dev)
    st_slot, st_feat, st_cnt = [st_blob[of:of + nb].view(dt).view(sh)
                                for of, (nb, dt, sh) in zip(offs, parts)]

    def stage(r):
        st_slot.copy_(d_slot[r])
        st_feat.copy_(d_feat[r])
        st_cnt.copy_(d_cnt[r])

    fused = args.api == "round" and not block

    def round_calls():
        if block:  # the full block: commit the verified round, draft the next with tokens
            drafter.commit(st_feat, st_cnt)
            drafter.draft_tokens(st_slot, out, tokens)
        elif fused:  # one serving iteration: commit the verified round, draft the next
            drafter.round(st_feat, st_cnt, st_slot, out)
        else:
            drafter.draft(st_slot, out)
            drafter.commit(st_feat, st_cnt)

    # eager warm-up rounds, marked with NVTX ranges ("round", or "draft" and
    # "commit") so a profiler can select one round's launches by range
    nvtx = torch.cuda.nvtx
    for r in range(args.warmup):
        stage(r)
        if block:
            round_calls()
        elif fused:
            nvtx.range_push("round")
            drafter.round(st_feat, st_cnt, st_slot, out)
            nvtx.range_pop()
        else:
            nvtx.range_push("draft")
            drafter.draft(st_slot, out)
            nvtx.range_pop()
            nvtx.range_push("commit")
            drafter.commit(st_feat, st_cnt)
            nvtx.range_pop()
    drafter.sync()

    def capture():
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        n0 = drafter.launch_count()
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            round_calls()
        torch.cuda.current_stream().wait_stream(side)
        return g, drafter.launch_count() - n0

    # Two captures of the same round: a clean one (timed for `value`, kernels
    # chained by programmatic dependent launch) and one with the library's
    # event nodes around each kernel family (they serialise the kernels; it
    # gives the per-family device times used for the roofline).
    drafter.profile(0)
    graph, launches_per_step = capture()
    drafter.profile(2)
    graph_prof, _ = capture()
    for r in range(args.warmup):
        stage(r)
        graph.replay()
        graph_prof.replay()
    torch.cuda.synchronize()
    drafter.profile_collect()
    for fam in hf.Family:
        drafter.profile_read(fam, reset=True)

    # ---- timed region: per-step events around the graph replay, L2 flushed
    # between steps (untimed)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            stage(args.warmup + i)
            flush.zero_()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    barrier()
    drafter.sync()
    launches = launches_per_step * args.steps
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)

    # ---- the same K steps four more times (L2 flushed), for the median of
    # five runs, and once with the L2 left warm between steps (steady state)
    def timed_run(flush_l2: bool) -> float:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            stage(args.warmup + i)
            if flush_l2:
                flush.zero_()
            evs[i][0].record(stream)
            graph.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    run_ms = [total_ms] + [timed_run(True) for _ in range(4)]
    warm_ms = timed_run(False)

    # ---- per-family device times: the same rounds through the profiled graph
    for i in range(args.steps):
        stage(args.warmup + i)
        flush.zero_()
        graph_prof.replay()
        drafter.profile_collect()
    torch.cuda.synchronize()
    fam_ms = {}
    for fam in hf.Family:
        ms, n = drafter.profile_read(fam, reset=True)
        fam_ms[fam.name.lower()] = (ms, n)
    accepted = int(d_cnt[args.warmup:].sum().item())
    total_ms_max = max_over_ranks(total_ms, dev)
    all_steps = sum_over_ranks(args.steps, dev)
    all_acc = sum_over_ranks(accepted, dev)
    value = all_steps / (total_ms_max / 1e3)

    # ---- e2e: the same rounds from pinned host buffers, the copies inside the
    # timed region: host -> staging buffers, the captured round, output -> host
    h_blob = torch.zeros((d_slot.shape[0], st_blob.numel()), dtype=torch.uint8).pin_memory()
    for r in range(d_slot.shape[0]):  # each step's inputs, laid out as the staging buffer
        for of, (nb, _, _), src in zip(offs, parts, (d_slot[r], d_feat[r], d_cnt[r])):
            h_blob[r, of:of + nb].copy_(src.cpu().contiguous().view(-1).view(torch.uint8))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_tok = torch.empty(tokens.shape, dtype=tokens.dtype).pin_memory()
    e2e_ev = []
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        r = args.warmup + i
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st_blob.copy_(h_blob[r], non_blocking=True)  # the step's inputs, one copy
        graph.replay()
        h_out.copy_(out, non_blocking=True)
        if block:
            h_tok.copy_(tokens, non_blocking=True)
        b.record(stream)
        e2e_ev.append((a, b))
    torch.cuda.synchronize()
    barrier()
    drafter.sync()
    del graph, graph_prof
    drafter.profile(0)
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), dev)
    e2e_value = all_steps / (e2e_ms / 1e3)
    es = drafter.np_elem
    h2d = sum(nb for nb, _, _ in parts)
    d2h = h_out.numel() * es + (h_tok.numel() * 4 if block else 0)

    # ---- roofline of the dominant kernel family
    import json as _json
    peaks = {}
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        peaks = _json.load(open(pp))
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_src = "measured" if peaks else "fallback"
    fill = sum(min(L, cfg.window) for L in lens) / max(len(lens), 1)  # valid window rows
    alg = algorithmic(cfg, batch, fill, (cfg.block + 2) / 2.0, fused,
                      torch.cuda.get_device_properties(dev).multi_processor_count)
    fams = {k: v for k, v in alg["families"].items() if v[1] > 0}
    top = max(fams, key=lambda k: fam_ms.get(k, (0, 0))[0])
    ms_top, _ = fam_ms[top]
    step_bytes_top, launches_top = fams[top]
    avg_ms = ms_top / max(args.steps * launches_top, 1)  # one profiled scope per launch
    per_launch = step_bytes_top / launches_top
    achieved = per_launch / (avg_ms / 1e3) / 1e9 if avg_ms > 0 else 0.0
    roofline = {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": measured_traffic(cfg.name, top) if fused else None,
                "peak_source": peak_src,
                "algorithmic_bytes_per_launch": per_launch, "avg_launch_ms": avg_ms}

    # ---- CPU oracle beside it (rank 0, N=1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        budget = float(os.environ.get("HF_CPU_BUDGET_S", "20"))
        v_cpu, _, _, _, sample = cpu_sample(cfg, args.steps, 1, budget)
        cpu = {"value": v_cpu, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": sample}

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic",
            "config": {"workload": cfg.name, "batch_per_gpu": batch,
                       "prefix": (f"log-uniform [{cfg.prefix_lo}, {cfg.prefix_hi}]"
                                  if cfg.prefix_lo else cfg.prefix),
                       "prefix_cap": args.prefix_max or None,
                       "api": "hf_round (commit, then draft the next block)" if fused
                              else "hf_draft then hf_commit",
                       "layers": cfg.n_layers, "window": cfg.window, "block": cfg.block,
                       "l2": f"flushed between steps ({2 * l2 >> 20} MiB write, untimed)",
                       "timing": "CUDA graph of one round replayed per step; CUDA events; "
                                 "kernel-family times from a second pass with event nodes",
                       "parallelism": f"replicas x{ws}",
                       **ablation_config(cfg)},
            "committed_tokens_per_s": all_acc / (total_ms_max / 1e3),
            "step_ms_median": statistics.median(step_ms),
            "runs_l2_flushed": {"runs": len(run_ms),
                                "median_value": args.steps / (statistics.median(run_ms) / 1e3),
                                "min_value": args.steps / (max(run_ms) / 1e3),
                                "max_value": args.steps / (min(run_ms) / 1e3),
                                "unit": UNIT, "note": "this rank; run 1 is the value's"},
            "steady_state": {"value": args.steps / (warm_ms / 1e3), "unit": UNIT,
                             "ms_per_step": warm_ms / args.steps,
                             "note": "same graph, L2 not flushed between steps (this rank)"},
            "algorithmic": {"step_bytes": alg["step_bytes"],
                            "families": {k: {"bytes_per_step": b, "launches_per_step": n}
                                         for k, (b, n) in fams.items()},
                            "step_hbm_frac": alg["step_bytes"] / (total_ms / args.steps / 1e3) / 1e9 / hbm_peak},
            "kernels_ms_per_step": {k: v[0] / args.steps for k, v in fam_ms.items() if v[1]},
            "roofline": roofline,
            "prefill": {"tokens": total, "ms": pf_ms, "tokens_per_s": total / (pf_ms / 1e3),
                        "tflops": pf_flops / (pf_ms / 1e3) / 1e12,
                        "tensor_frac": pf_flops / (pf_ms / 1e3) / 1e12 / tc_peak},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h)},
            "gpu_launches": int(launches),
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    drafter.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="hyflash", choices=["hyflash", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--prefix", type=int, default=0, help="prefill sweep: prefix length")
    ap.add_argument("--api", default="round", choices=["round", "separate"],
                    help="round: hf_round per step (commit, then draft the next block); "
                         "separate: hf_draft then hf_commit")
    ap.add_argument("--prefix-max", type=int, default=0,
                    help="round configs: cap every request's prefix (0: the workload's own)")
    ap.add_argument("--chunk", type=int, default=128, help="prefill sweep: scan chunk")
    ap.add_argument("--layers", type=int, default=1, help="prefill sweep: drafter depth")
    ap.add_argument("--cross-slot-off", action="store_true",
                    help="ablation: mask attention among the draft slots")
    ap.add_argument("--mem-horizon", type=int, default=0,
                    help="ablation: memory of the last M committed features (0: all)")
    ap.add_argument("--memory", default="mamba2", choices=["mamba2", "gdn"],
                    help="memory kind: Mamba-2 (default) or the gated delta rule")
    ap.add_argument("--weight-bits", type=int, default=16, choices=[16, 4],
                    help="weights in the model dtype (16) or 4-bit codes (4)")
    ap.add_argument("--block", default="layer", choices=["layer", "full"],
                    help="layer: the HyFlash layer alone; full: the drafter block around it "
                         "(norms, RoPE, conv1d, skip/gate, SwiGLU MLP, LM head + argmax)")
    ap.add_argument("--mlp-dim", type=int, default=0,
                    help="full block: MLP width (0: the target family's, 9728 Qwen3-4B, 17920 Phi-4)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="full block: LM-head rows (0: the target family's, 151936 / 100352)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from workload import CONFIGS
    cfg = CONFIGS[args.config].replace(cross_slot=not args.cross_slot_off,
                                       mem_horizon=args.mem_horizon, memory=args.memory,
                                       weight_bits=args.weight_bits)
    if args.block == "full":
        # the target families' MLP widths and vocabularies (Qwen3-4B, Phi-4)
        fam_mlp, fam_vocab = (17920, 100352) if cfg.d_model == 5120 else (9728, 151936)
        cfg = cfg.replace(full_block=True, mlp_dim=args.mlp_dim or fam_mlp,
                          vocab=args.vocab or fam_vocab)
    if args.impl == "reference":
        return run_reference(args, cfg)
    if cfg.rounds == 0:
        return run_prefill_sweep(args, cfg)
    return run_hyflash(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
