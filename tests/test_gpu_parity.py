"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Bars: ring tags, positions and commit offsets bit-exact; floating point
within max-normalised 1e-4 (fp32 mode) or 2e-2 (bf16 mode) per tensor.
"""
import dataclasses

import numpy as np
import pytest
import torch

from _harness import Pair, maxnorm_err
from speculative_decoding_drafter_hf_gb300 import Tensor
from workload import (CONFIGS, make_accepted, make_prefix_feats, make_prefix_lens,
                      make_round_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_drafter_hf_gb300 import build
    build.build()


def check_mix(p: Pair, slot, what: str = ""):
    """The last layer's two branches on their own, read back from the handle
    after a draft: the attention output O and the memory read y (DRAFT_MIX)
    against the oracle's parts of the same layer, each within the tolerance
    of its own max-norm (the residual X dominates the final output, so a
    branch-level error could hide there). The oracle's context must be the
    one the draft ran against."""
    from oracle import hyflash_oracle as O
    cfg = p.cfg
    S, QD = cfg.block, cfg.n_q_heads * cfg.head_dim
    mix = p.gpu.read(Tensor.DRAFT_MIX)
    X = O.to64(slot)
    got_o, got_y, ref_o, ref_y = [], [], [], []
    for b in range(X.shape[0]):
        cur = X[b]
        for lw, c in zip(p.orc.layers[:-1], p.orc.ctx[b][:-1]):
            cur = O.draft_layer(lw, cfg, c, cur)
        _, parts = O.draft_layer(p.orc.layers[-1], cfg, p.orc.ctx[b][-1], cur, return_parts=True)
        rows = slice(b * S, (b + 1) * S)
        got_o.append(mix[rows, :QD])
        got_y.append(mix[rows, QD:])
        ref_o.append(parts["O"].reshape(S, -1))
        ref_y.append(parts["y"].reshape(S, -1))
    for name, g, r in (("attention", got_o, ref_o), ("memory read", got_y, ref_y)):
        e = maxnorm_err(np.concatenate(g), np.concatenate(r))
        assert e <= p.tol, f"{what}: {name} branch err {e:.3e}"


def run_rounds(p: Pair, rounds: int, check_every: int = 1, n_override=None):
    cfg = p.cfg
    worst = 0.0
    for r in range(rounds):
        slot, feats = make_round_inputs(cfg, r, p.B)
        got, ref = p.draft(slot)
        e = maxnorm_err(got, ref)
        assert e <= p.tol, f"round {r}: draft err {e:.3e}"
        check_mix(p, slot, f"round {r}")
        worst = max(worst, e)
        n = make_accepted(cfg, r, p.B) if n_override is None else n_override(r)
        offs, _ = p.commit(feats, n)
        got_offs = p.gpu.read(Tensor.OFFSETS)
        assert np.array_equal(got_offs[:p.B + 1], offs.astype(np.int32)), f"round {r}: offsets"
        if (r + 1) % check_every == 0 or r == rounds - 1:
            worst = max(worst, p.check_context(what=f"round {r}"))
    return worst


def test_tiny_fp32_all_rounds():
    cfg = CONFIGS["tiny_fp32"]
    p = Pair(cfg)
    lens = make_prefix_lens(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    run_rounds(p, cfg.rounds)
    p.close()


def test_tiny_fp32_batch_ragged_multilayer_segments():
    # several requests, prefixes empty / shorter than W / longer than W and not
    # a multiple of the prefill pass, three layers, tiny prefill passes
    cfg = CONFIGS["tiny_fp32"].replace(n_layers=3, batch=5)
    p = Pair(cfg, prefill_tokens_max=50)
    lens = [0, 13, 64, 65, 301]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    run_rounds(p, 6)
    p.close()


def test_prefill_subset_of_requests_leaves_others():
    cfg = CONFIGS["tiny_fp32"].replace(batch=4)
    p = Pair(cfg)
    lens = [100, 7, 70, 0]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    run_rounds(p, 2)
    lens2 = [33, 129]
    p.prefill(lens2, make_prefix_feats(cfg, lens2, seed=5), requests=[2, 0])
    p.check_context(what="re-prefill")
    run_rounds(p, 2)
    p.close()


def test_draft_is_read_only_bytewise():
    cfg = CONFIGS["tiny_fp32"].replace(batch=2)
    p = Pair(cfg, oracle=False)
    lens = [80, 20]
    p.gpu.prefill(make_prefix_feats(cfg, lens).cuda(), lens)
    before = p.gpu.export_context()
    slot, _ = make_round_inputs(cfg, 0, 2)
    p.gpu.draft(slot.cuda())
    torch.cuda.synchronize()
    assert p.gpu.export_context() == before
    p.close()


def test_rejected_rows_and_zero_counts_never_change_anything():
    cfg = CONFIGS["tiny_fp32"].replace(batch=3)
    p = Pair(cfg, oracle=False)
    lens = [70, 5, 0]
    p.gpu.prefill(make_prefix_feats(cfg, lens).cuda(), lens)
    start = p.gpu.export_context()
    _, feats = make_round_inputs(cfg, 1, 3)
    n = torch.tensor([3, 0, 8], dtype=torch.int32)
    p.gpu.commit(feats.cuda(), n.cuda())
    after_a = p.gpu.export_context()
    p.gpu.import_context(start)
    feats2 = feats.clone()
    feats2[0, 3:] = torch.randn(5, cfg.d_model) * 50
    feats2[1, :] = torch.randn(8, cfg.d_model) * 50
    p.gpu.commit(feats2.cuda(), n.cuda())
    assert p.gpu.export_context() == after_a
    p.gpu.import_context(start)
    p.gpu.commit(feats2.cuda(), torch.zeros(3, dtype=torch.int32).cuda())
    assert p.gpu.export_context() == start
    p.gpu.sync()
    p.close()


def test_invalid_accepted_count_is_flagged_and_skipped():
    cfg = CONFIGS["tiny_fp32"].replace(batch=3)
    p = Pair(cfg)
    lens = [40, 40, 40]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    _, feats = make_round_inputs(cfg, 2, 3)
    n = torch.tensor([2, 9, 5], dtype=torch.int32)
    offs, err = p.commit(feats, n)
    assert err
    import speculative_decoding_drafter_hf_gb300 as hf
    st, msg = p.gpu.sync_status()
    assert st == hf.Status.EDEVICE and "accepted" in msg
    assert p.gpu.sync_status()[0] == hf.Status.OK  # the word is cleared
    assert np.array_equal(p.gpu.read(hf.Tensor.OFFSETS)[:4], offs.astype(np.int32))
    p.check_context(what="after invalid count")
    n = torch.tensor([-1, 1, 1], dtype=torch.int32)
    p.commit(feats, n)
    assert p.gpu.sync_status()[0] == hf.Status.EDEVICE
    p.check_context(what="after negative count")
    p.close()


def test_qwen3_4b_shape_bf16():
    cfg = CONFIGS["qwen3_4b_bf16"]
    p = Pair(cfg)
    lens = make_prefix_lens(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    run_rounds(p, 8, check_every=4)
    p.close()


def test_serving_shape_bf16_subset():
    # serving-batch shape (3 layers, Qwen3-4B widths) with 6 requests of
    # log-uniform prefixes; requests are independent, so a subset is exact.
    cfg = CONFIGS["serving_qwen3_4b_b64"].replace(batch=6, prefix_lo=600, prefix_hi=3000)
    p = Pair(cfg)
    lens = make_prefix_lens(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    run_rounds(p, 4, check_every=2)
    p.close()


@pytest.mark.parametrize("name,lens", [("tiny_fp32", [300, 20]), ("qwen3_4b_bf16", [1500, 300])])
def test_draft_steps_individually(name, lens):
    """Rows a4 (slot projections), a5 (attention) and a6 (memory read) on
    their own, read back from the handle after one draft."""
    cfg = CONFIGS[name].replace(batch=len(lens))
    p = Pair(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    check_draft_parts(p, 3)
    p.close()


def check_draft_parts(p: Pair, round_: int):
    from oracle import hyflash_oracle as O
    cfg = p.cfg
    slot, _ = make_round_inputs(cfg, round_, p.B)
    got, ref = p.draft(slot)
    S, QD, KVD = cfg.block, cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    proj = p.gpu.read(Tensor.DRAFT_PROJ)
    mix = p.gpu.read(Tensor.DRAFT_MIX)
    lw = p.orc.layers[0]
    X = O.to64(slot)
    for b in range(p.B):
        _, parts = O.draft_layer(lw, cfg, p.orc.ctx[b][0], X[b], return_parts=True)
        rows = slice(b * S, (b + 1) * S)
        checks = [
            ("Q", proj[rows, :QD], parts["Q"].reshape(S, -1)),
            ("K_s", proj[rows, QD:QD + KVD], parts["Ks"].reshape(S, -1)),
            ("V_s", proj[rows, QD + KVD:QD + 2 * KVD], parts["Vs"].reshape(S, -1)),
            ("C_s", proj[rows, QD + 2 * KVD:], parts["Cs"]),
            ("attention", mix[rows, :QD], parts["O"].reshape(S, -1)),
            ("memory read", mix[rows, QD:], parts["y"].reshape(S, -1)),
        ]
        for what, g, r in checks:
            e = maxnorm_err(g, r)
            assert e <= p.tol, f"request {b}: {what} err {e:.3e}"
    assert maxnorm_err(got, ref) <= p.tol


# bf16 attention shapes away from the headline ones: windows that are not a
# multiple of the 64-key tile, 1..8 query heads per KV head, head_dim 64 /
# 128 / 256, empty / partial / wrapped windows, and batches that give one CTA
# per (request, KV head) walking several tiles as well as multi-CTA clusters.
ATTN_SHAPES = {
    "w100_dh64_g4": (dict(d_model=512, n_q_heads=8, n_kv_heads=2, head_dim=64, window=100,
                          ssm_heads=8, ssm_headdim=64, d_state=64), [0, 37, 100, 250]),
    "w200_dh128_g8": (dict(d_model=1024, n_q_heads=16, n_kv_heads=2, head_dim=128, window=200,
                           ssm_heads=8, ssm_headdim=64, d_state=64), [150, 1000]),
    "w70_dh256_g2": (dict(d_model=512, n_q_heads=4, n_kv_heads=2, head_dim=256, window=70,
                          ssm_heads=4, ssm_headdim=32, d_state=64), [69, 71, 500]),
    "w300_b80_one_cta": (dict(d_model=256, n_q_heads=8, n_kv_heads=4, head_dim=64, window=300,
                              ssm_heads=4, ssm_headdim=32, d_state=32),
                         [(37 * i) % 420 for i in range(80)]),
    # one CTA per (request, KV head) at the serving shape's head dim (128) and
    # query rows (28): partial and wrapped windows, and with cross-slot
    # attention off
    "w300_dh128_b80_one_cta": (dict(d_model=512, n_q_heads=16, n_kv_heads=4, head_dim=128,
                                    window=300, ssm_heads=4, ssm_headdim=32, d_state=32),
                               [(37 * i) % 420 for i in range(80)]),
    "w300_dh128_b80_one_cta_xoff": (dict(d_model=512, n_q_heads=16, n_kv_heads=4, head_dim=128,
                                         window=300, ssm_heads=4, ssm_headdim=32, d_state=32,
                                         cross_slot=False),
                                    [(53 * i) % 400 for i in range(80)]),
}


@pytest.mark.parametrize("name", sorted(ATTN_SHAPES))
def test_attention_shapes_bf16(name):
    dims, lens = ATTN_SHAPES[name]
    cfg = CONFIGS["qwen3_4b_bf16"].replace(batch=len(lens), **dims)
    p = Pair(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    check_draft_parts(p, 1)
    n = make_accepted(cfg, 1, p.B)
    _, feats = make_round_inputs(cfg, 1, p.B)
    p.commit(feats, n)
    check_draft_parts(p, 2)
    p.close()


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_4b_bf16"])
def test_rounds_captured_in_cuda_graph(name):
    """draft + commit captured once into a CUDA graph and replayed per round
    (with the profiler recording inside the graph) match the oracle."""
    cfg = CONFIGS[name].replace(batch=2)
    p = Pair(cfg)
    lens = [700, 90]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    st_slot = torch.empty((2, cfg.block, cfg.d_model), dtype=p.gpu.torch_dtype, device="cuda")
    st_feat = torch.empty((2, cfg.block + 1, cfg.d_model), dtype=p.gpu.torch_dtype, device="cuda")
    st_cnt = torch.empty((2,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(st_slot)
    p.gpu.profile(2)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        p.gpu.draft(st_slot, out)
        p.gpu.commit(st_feat, st_cnt)
    torch.cuda.current_stream().wait_stream(side)
    for r in range(3):
        slot, feats = make_round_inputs(cfg, r, 2)
        n = make_accepted(cfg, r, 2)
        st_slot.copy_(slot.cuda())
        st_feat.copy_(feats.cuda())
        st_cnt.copy_(n.cuda())
        g.replay()
        torch.cuda.synchronize()
        p.gpu.profile_collect()
        ref = p.orc.draft(slot)
        p.orc.commit(feats, n.numpy())
        e = maxnorm_err(out.float().cpu().numpy(), ref)
        assert e <= p.tol, f"round {r}: draft err {e:.3e}"
        p.check_context(what=f"graph round {r}")
    ms, launches = p.gpu.profile_read(0)
    assert ms > 0 and launches >= 3
    del g
    p.gpu.profile(0)
    p.close()


@pytest.mark.parametrize("chunk,tokens_max", [(64, 1000), (128, 4096), (256, 700)])
def test_prefill_chunked_scan_segments_bf16(chunk, tokens_max):
    """The prefill fold (dt projection, chunked decay scan, w-scaled x/B
    projection, contraction over tokens) with several chunk sizes and with
    prefixes split into segments at non-multiples of the chunk; three
    requests of different lengths (one empty)."""
    cfg = CONFIGS["qwen3_4b_bf16"].replace(batch=3, chunk=chunk)
    p = Pair(cfg, prefill_tokens_max=tokens_max)
    lens = [2500, 0, 333]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what=f"prefill chunk {chunk}")
    run_rounds(p, 2)
    p.close()


def run_round_api(p: Pair, rounds: int, check_every: int = 1):
    cfg = p.cfg
    for r in range(rounds):
        slot, feats = make_round_inputs(cfg, r, p.B)
        n = make_accepted(cfg, r, p.B)
        got, ref, offs = p.round(feats, n, slot)
        e = maxnorm_err(got, ref)
        assert e <= p.tol, f"round {r}: draft err {e:.3e}"
        check_mix(p, slot, f"round {r}")
        got_offs = p.gpu.read(Tensor.OFFSETS)
        assert np.array_equal(got_offs[:p.B + 1], offs.astype(np.int32)), f"round {r}: offsets"
        if (r + 1) % check_every == 0 or r == rounds - 1:
            p.check_context(what=f"round {r}")


@pytest.mark.parametrize("name,batch,rounds", [
    ("tiny_fp32", 3, 6),              # two entry points in turn
    ("qwen3_4b_bf16", 2, 5),          # grouped projection, memory read beside the attention
    ("qwen3_4b_bf16", 8, 3),          # 8 x 2.6 MB of state: memory read in the state update
    ("serving_qwen3_4b_b64", 5, 3),   # three layers: later layers draft as in hf_draft
])
def test_round_api(name, batch, rounds):
    """hf_round = hf_commit then hf_draft, against the oracle's commit then draft."""
    cfg = CONFIGS[name].replace(batch=batch, prefix_lo=300, prefix_hi=900) \
        if name.startswith("serving") else CONFIGS[name].replace(batch=batch)
    p = Pair(cfg)
    lens = make_prefix_lens(cfg)
    lens = [min(L, 1200) for L in lens]
    lens[0] = 0  # one empty window: attention over the slots only
    p.prefill(lens, make_prefix_feats(cfg, lens))
    run_round_api(p, rounds, check_every=2)
    p.close()


@pytest.mark.parametrize("variant", [
    {}, {"memory": "gdn"}, {"mem_horizon": 3}, {"mem_horizon": 512}, {"cross_slot": False},
    {"weight_bits": 4}])
def test_round_api_rejected_and_invalid_counts(variant):
    """Zero, full and invalid accepted counts through hf_round: invalid ones
    leave the request untouched, raise EDEVICE, and the draft still reads the
    (unchanged) state -- for the default layer and every optional mode."""
    import speculative_decoding_drafter_hf_gb300 as hf
    cfg = CONFIGS["qwen3_4b_bf16"].replace(batch=3, **variant)
    p = Pair(cfg, tweak=slow_decay(-6.0) if variant.get("mem_horizon") else None)
    lens = [700, 40, 1500]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    slot, feats = make_round_inputs(cfg, 0, p.B)
    n = torch.tensor([0, cfg.block + 1, 3], dtype=torch.int32)
    got, ref, _ = p.round(feats, n, slot)
    assert maxnorm_err(got, ref) <= p.tol
    p.check_context(what="zero / full counts")
    slot, feats = make_round_inputs(cfg, 1, p.B)
    bad = torch.tensor([2, -1, cfg.block + 2], dtype=torch.int32)
    out = p.gpu.round(feats.cuda(), bad.cuda(), slot.cuda())
    assert p.gpu.sync_status()[0] == hf.Status.EDEVICE
    p.orc.commit(feats, np.array([2, 0, 0]))  # invalid counts: requests 1, 2 untouched
    ref = p.orc.draft(slot)
    got = out.float().cpu().numpy().astype(np.float64)
    assert maxnorm_err(got, ref) <= p.tol
    p.check_context(what="after invalid counts")
    p.close()


def test_round_api_in_cuda_graph():
    """hf_round captured once and replayed per round (the benchmark's form)."""
    cfg = CONFIGS["qwen3_4b_bf16"].replace(batch=2)
    p = Pair(cfg)
    lens = [900, 130]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    dt = p.gpu.torch_dtype
    st_slot = torch.empty((2, cfg.block, cfg.d_model), dtype=dt, device="cuda")
    st_feat = torch.empty((2, cfg.block + 1, cfg.d_model), dtype=dt, device="cuda")
    st_cnt = torch.empty((2,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(st_slot)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        p.gpu.round(st_feat, st_cnt, st_slot, out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for r in range(4):
        slot, feats = make_round_inputs(cfg, r, 2)
        n = make_accepted(cfg, r, 2)
        st_slot.copy_(slot)
        st_feat.copy_(feats)
        st_cnt.copy_(n.to(torch.int32))
        g.replay()
        torch.cuda.synchronize()
        p.orc.commit(feats, n.numpy())
        ref = p.orc.draft(slot)
        got = out.float().cpu().numpy().astype(np.float64)
        assert maxnorm_err(got, ref) <= p.tol, f"round {r}"
    p.check_context(what="graph rounds")
    p.close()


@pytest.mark.parametrize("name,batch,api", [
    ("serving_qwen3_4b_b64", 4, "separate"),  # commit projection alone, 32 rows, 174 tiles
    ("serving_qwen3_4b_b64", 2, "round"),     # grouped with the slot projection, 16 rows
    ("phi4_bf16", 1, "round"),                # Phi-4 widths: 164 tiles
    ("serving_qwen3_4b_b64", 5, "round"),     # token-major stream-K: 40 and 35 token rows
    ("serving_qwen3_4b_b64", 33, "round"),    # token-major: three token tiles, ragged last
    ("serving_qwen3_4b_b64", 5, "separate"),  # token-major cluster split-K, 35 and 40 rows
])
def test_stream_k_products(name, batch, api):
    """Skinny products with more weight tiles than SMs run stream-K (equal
    shares of (tile, k-block) units per SM, split tiles summed in k order)."""
    cfg = CONFIGS[name].replace(batch=batch, prefix=700, prefix_lo=300, prefix_hi=900) \
        if name.startswith("serving") else CONFIGS[name].replace(batch=batch, prefix=700)
    p = Pair(cfg)
    lens = make_prefix_lens(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    if api == "round":
        run_round_api(p, 2, check_every=1)
    else:
        run_rounds(p, 2, check_every=1)
    p.close()


# ---------------------------------------------------------------- ablation modes

def slow_decay(a_log):
    """Weights whose memory decays slowly (A = -exp(a_log)), so that features
    far back still weigh in and a memory horizon visibly changes the state."""
    return lambda w: dataclasses.replace(w, A_log=torch.full_like(w.A_log, a_log))


@pytest.mark.parametrize("name,batch", [("tiny_fp32", 3), ("qwen3_4b_bf16", 2)])
def test_cross_slot_off(name, batch):
    """Cross-slot off: each slot attends to the window and its own key only
    (both attention paths: fp32 CUDA cores, bf16 tensor cores)."""
    cfg = CONFIGS[name].replace(batch=batch, prefix=100, cross_slot=False)
    p = Pair(cfg)
    lens = [0, 37, 700][:batch] if name == "tiny_fp32" else [5, 700]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    run_rounds(p, 3)
    # the attention branch differs from the default mode's (the slots
    # interact there): compared on the branch itself, where the mask shows
    slot, _ = make_round_inputs(cfg, 7, p.B)
    got, ref = p.draft(slot)
    assert maxnorm_err(got, ref) <= p.tol
    check_mix(p, slot, "cross-slot off")
    QD = cfg.n_q_heads * cfg.head_dim
    mine = p.gpu.read(Tensor.DRAFT_MIX)[:p.B * cfg.block, :QD]
    q = Pair(cfg.replace(cross_slot=True), oracle=False)
    q.prefill(lens, make_prefix_feats(cfg, lens))
    q.gpu.draft(slot.cuda())
    torch.cuda.synchronize()
    other = q.gpu.read(Tensor.DRAFT_MIX)[:p.B * cfg.block, :QD]
    q.close()
    p.close()
    assert maxnorm_err(mine, other) > 10 * p.tol


@pytest.mark.parametrize("name,batch,horizon,lens", [
    ("tiny_fp32", 4, 1, [0, 1, 9, 300]),        # last feature
    ("tiny_fp32", 4, 3, [0, 2, 9, 300]),        # leaving rows inside one commit
    ("tiny_fp32", 4, 20, [0, 7, 25, 300]),      # leaving rows from the ring
    ("tiny_fp32", 2, 64, [10, 500]),            # horizon = window
    ("qwen3_4b_bf16", 2, 1, [3, 700]),
    ("qwen3_4b_bf16", 2, 512, [300, 1200]),     # the paper's "last 512"
    ("qwen3_4b_bf16", 2, 20, [5, 20]),          # 25 window rows: the skinny prefill GEMM
])
def test_memory_horizon(name, batch, horizon, lens):
    """Memory restricted to the last M committed features (prefill folds the
    last M only; each commit adds its rows and removes the ones leaving)."""
    cfg = CONFIGS[name].replace(batch=batch, prefix=100, mem_horizon=horizon)
    p = Pair(cfg, tweak=slow_decay(-4.0 if horizon <= 64 else -7.0), prefill_tokens_max=256)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    rounds = 12 if horizon < 512 else 4
    run_rounds(p, rounds, check_every=1)
    if horizon > 1:
        x = p.gpu.read(Tensor.MEM_X)
        assert x.shape == (cfg.n_layers, batch, horizon + cfg.block + 1, cfg.d_inner)
    p.close()


@pytest.mark.parametrize("name,horizon,rounds,check_every", [
    ("tiny_fp32", 20, 300, 50),        # leaving rows from the ring, ~1,300 removals per request
    ("tiny_fp32", 3, 300, 50),         # leaving rows inside the commit, every round
    ("qwen3_4b_bf16", 20, 120, 40),
])
def test_memory_horizon_no_drift_over_many_rounds(name, horizon, rounds, check_every):
    """The GPU removes each feature leaving the horizon by subtracting its
    decayed term from the state, while the oracle refolds the last M features
    from zero at every commit (the plain definition): the rounding of the
    subtractions must not build up over hundreds of rounds. Drafts, both
    branches of the draft and the whole context are compared every
    `check_every` rounds, with the tolerance of a single round."""
    cfg = CONFIGS[name].replace(batch=2, prefix=100, mem_horizon=horizon)
    p = Pair(cfg, tweak=slow_decay(-4.0), prefill_tokens_max=256)
    lens = [5, 700]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    for r in range(rounds):
        slot, feats = make_round_inputs(cfg, r, p.B)
        if (r + 1) % check_every == 0:
            got, ref = p.draft(slot)
            e = maxnorm_err(got, ref)
            assert e <= p.tol, f"round {r}: draft err {e:.3e}"
            check_mix(p, slot, f"round {r}")
        p.commit(feats, make_accepted(cfg, r, p.B))
        if (r + 1) % check_every == 0:
            p.check_context(what=f"round {r}")
    assert all(p.orc.ctx[b][0].pos >= lens[b] + rounds for b in range(p.B))
    p.close()


def test_memory_horizon_round_api_and_graph():
    cfg = CONFIGS["tiny_fp32"].replace(batch=3, prefix=40, mem_horizon=6, n_layers=2)
    p = Pair(cfg, tweak=slow_decay(-4.0))
    lens = [0, 5, 40]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    run_round_api(p, 6, check_every=1)
    p.close()


# ---------------------------------------------------------------- gated-delta memory

@pytest.mark.parametrize("name,batch,lens,api", [
    ("tiny_fp32", 3, [0, 9, 300], "separate"),   # several prefill passes (128 tokens)
    ("qwen3_4b_bf16", 2, [5, 60], "separate"),
    ("qwen3_4b_bf16", 2, [5, 60], "round"),
    ("qwen3_4b_bf16", 8, [3, 7, 12, 20, 25, 30, 33, 40], "round"),  # fused memory read
])
def test_gated_delta_memory(name, batch, lens, api):
    """The gated delta rule as the memory: prefill (token-by-token scan),
    commits (the state kernel's gated-delta update) and the normalised read."""
    cfg = CONFIGS[name].replace(batch=batch, prefix=100, memory="gdn")
    p = Pair(cfg, prefill_tokens_max=128)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    if api == "round":
        run_round_api(p, 3, check_every=1)
    else:
        run_rounds(p, 4 if name == "tiny_fp32" else 3, check_every=1)
    p.close()


# ---------------------------------------------------------------- 4-bit weights

@pytest.mark.parametrize("batch,api,lens", [
    (1, "round", [700]),              # the skinny products read the 4-bit tiles
    (2, "separate", [5, 700]),
    (6, "round", [3, 9, 30, 60, 100, 700]),   # wide products: the bf16 dequantisation
])
def test_q4_weights(batch, api, lens):
    """4-bit weights (codes, bf16 group scales, zero points): the on-chip
    dequantisation of the skinny GEMMs and the host one of the wide paths
    against the oracle's exact dequantised weights."""
    cfg = CONFIGS["qwen3_4b_bf16"].replace(batch=batch, prefix=100, weight_bits=4)
    p = Pair(cfg)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="prefill")
    if api == "round":
        run_round_api(p, 3, check_every=1)
    else:
        run_rounds(p, 3, check_every=1)
    p.close()


def test_q4_weights_phi4_grouped_and_layers():
    """Phi-4 widths (164 commit tiles: the grouped 4-bit launch in two waves)
    and two layers (the later layer's slot projection)."""
    cfg = CONFIGS["phi4_bf16"].replace(batch=1, prefix=300, weight_bits=4, n_layers=2)
    p = Pair(cfg)
    p.prefill([300], make_prefix_feats(cfg, [300]))
    run_round_api(p, 2, check_every=1)
    p.close()


# ---------------------------------------------------------------- pipelined state update

@pytest.mark.parametrize("name,batch,layers,api", [
    ("serving_qwen3_4b_b64", 16, 1, "round"),     # 1280 heads: fused memory read in the walk
    ("serving_qwen3_4b_b64", 16, 1, "separate"),  # the walk without the read
    ("serving_qwen3_4b_b64", 9, 2, "round"),      # layer 1 items never read
    ("tiny_fp32", 320, 1, "separate"),            # small heads (P*N = 1024), fp32
])
def test_pipelined_state_walk(name, batch, layers, api):
    """Large batches run the persistent state-update walk (bulk copies of
    each head's state and rows, several heads in flight per SM): state, ring,
    offsets and both draft branches against the oracle, with zero, full and
    invalid accepted counts among the requests."""
    import speculative_decoding_drafter_hf_gb300 as hf
    cfg = CONFIGS[name].replace(batch=batch, n_layers=layers, prefix=60, prefix_lo=0, prefix_hi=0)
    p = Pair(cfg)
    lens = [(37 * i) % 700 for i in range(batch)] if name != "tiny_fp32" else \
        [(13 * i) % 90 for i in range(batch)]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    for r in range(3):
        slot, feats = make_round_inputs(cfg, r, batch)
        n = make_accepted(cfg, r, batch)
        n[0], n[1] = 0, cfg.block + 1
        if r == 1:
            n[2] = -3  # invalid: request 2 untouched, EDEVICE at sync
        if api == "round":
            out = p.gpu.round(feats.cuda(), n.cuda(), slot.cuda())
            torch.cuda.synchronize()
            offs, _ = p.orc.commit(feats, n.numpy())
            ref = p.orc.draft(slot)
            assert maxnorm_err(out.float().cpu().numpy(), ref) <= p.tol, f"round {r}"
            check_mix(p, slot, f"round {r}")
        else:
            offs, _ = p.commit(feats, n)
            got, ref = p.draft(slot)
            assert maxnorm_err(got, ref) <= p.tol, f"round {r}"
            check_mix(p, slot, f"round {r}")
        assert np.array_equal(p.gpu.read(Tensor.OFFSETS)[:batch + 1], offs.astype(np.int32))
        st = p.gpu.sync_status()[0]
        assert st == (hf.Status.EDEVICE if r == 1 else hf.Status.OK)
        p.check_context(what=f"round {r}")
    p.close()


@pytest.mark.parametrize("name,lens,tokens_max", [
    ("tiny_fp32", [700, 130, 1], 512),     # two passes, a one-token prefix
    ("qwen3_4b_bf16", [260, 64], 100),      # 100-token passes
])
def test_gated_delta_long_prefill_passes(name, lens, tokens_max):
    """The gated-delta prefill over long prefixes cut into several passes:
    the state after prefill and after rounds against the oracle's rule."""
    cfg = CONFIGS[name].replace(batch=len(lens), prefix=100, memory="gdn")
    p = Pair(cfg, prefill_tokens_max=tokens_max)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(what="gated-delta prefill in passes")
    run_rounds(p, 2, check_every=1)
    p.close()
