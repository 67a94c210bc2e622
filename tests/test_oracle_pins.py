"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

None of these re-types the oracle's own formula: each compares it with a
library routine (scipy lfilter, torch SDPA / softplus), an unrolled closed
form, a special case with a known answer, an invariant the pages state
(rejected drafts never enter the memory; drafting does not change it), or a
figure the pages print (tests/golden/sizing.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import hyflash_oracle as O
from workload import CONFIGS, make_layer_weights, make_ssm_core_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = CONFIGS["tiny_fp32"]


def small_cfg(**kw):
    base = dict(d_model=32, n_q_heads=4, n_kv_heads=2, head_dim=8, window=6,
                ssm_heads=2, ssm_headdim=4, d_state=3, n_layers=1, batch=2,
                prefix=10, rounds=3, chunk=4)
    base.update(kw)
    return TINY.replace(name="pin_small", **base)


def ssm_case(T=37, Hm=3, P=4, N=5, seed=0):
    x, B, dt_raw, A_log = make_ssm_core_inputs(T, Hm, P, N, seed)
    x, B = x.numpy(), B.numpy()
    dt = O.softplus(dt_raw.numpy())
    A = -np.exp(A_log.numpy())
    return x, B, dt, A


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- softplus

def test_softplus_closed_values():
    assert O.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert O.softplus(50.0) == pytest.approx(50.0, rel=1e-15)
    assert O.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    xs = np.linspace(-30, 30, 1001)
    ref = torch.nn.functional.softplus(torch.tensor(xs, dtype=torch.float64),
                                       threshold=1e6).numpy()
    assert np.max(np.abs(O.softplus(xs) - ref)) < 1e-14


# ---------------------------------------------------------------- the fold

@pytest.mark.parametrize("chunk", [1, 3, 8, 16, 37, 64, 100])
def test_chunked_fold_equals_recurrence(chunk):
    x, B, dt, A = ssm_case(T=37)
    h0 = np.random.default_rng(1).standard_normal((3, 4, 5))
    r = O.ssm_fold_recurrent(h0, x, B, dt, A)
    c = O.ssm_fold_chunked(h0, x, B, dt, A, chunk)
    assert rel(c, r) < 1e-12


def test_fold_unrolled_product_closed_form():
    # h_T = prod_t a_t h_0 + sum_t dt_t (prod_{s>t} exp(dt_s A)) x_t (x) B_t,
    # written with explicit scalar loops on a tiny case.
    x, B, dt, A = ssm_case(T=6, Hm=2, P=3, N=2, seed=3)
    h0 = np.random.default_rng(2).standard_normal((2, 3, 2))
    want = np.zeros((2, 3, 2))
    for hd in range(2):
        for p in range(3):
            for n in range(2):
                total = h0[hd, p, n]
                for s in range(6):
                    total *= math.exp(dt[s, hd] * A[hd])
                for t in range(6):
                    w = dt[t, hd]
                    for s in range(t + 1, 6):
                        w *= math.exp(dt[s, hd] * A[hd])
                    total += w * x[t, hd, p] * B[t, n]
                want[hd, p, n] = total
    got = O.ssm_fold_recurrent(h0, x, B, dt, A)
    assert rel(got, want) < 1e-13


def test_fold_constant_decay_matches_lfilter():
    signal = pytest.importorskip("scipy.signal")
    x, B, _, A = ssm_case(T=50, Hm=2, P=3, N=4, seed=5)
    dt = np.full((50, 2), 0.37)
    got = O.ssm_fold_recurrent(np.zeros((2, 3, 4)), x, B, dt, A)
    for hd in range(2):
        a = math.exp(0.37 * A[hd])
        for p in range(3):
            for n in range(4):
                u = dt[:, hd] * x[:, hd, p] * B[:, n]
                y = signal.lfilter([1.0], [1.0, -a], u)
                assert abs(got[hd, p, n] - y[-1]) < 1e-12 * max(1.0, abs(y[-1]))


def test_fold_zero_decay_is_plain_sum():
    x, B, dt, _ = ssm_case(T=20, seed=7)
    A = np.zeros(3)
    got = O.ssm_fold_recurrent(np.zeros((3, 4, 5)), x, B, dt, A)
    want = np.zeros((3, 4, 5))
    for t in range(20):
        want += dt[t][:, None, None] * np.multiply.outer(x[t], B[t]).reshape(3, 4, 5)
    assert rel(got, want) < 1e-13


def test_fold_huge_decay_keeps_last_token_only():
    x, B, dt, _ = ssm_case(T=9, seed=8)
    A = np.full(3, -1e9)
    got = O.ssm_fold_recurrent(np.ones((3, 4, 5)), x, B, dt, A)
    want = dt[-1][:, None, None] * x[-1][:, :, None] * B[-1][None, None, :]
    assert rel(got, want) < 1e-15


def test_fold_dt_zero_leaves_state_bit_identical():
    x, B, _, A = ssm_case(T=11, seed=9)
    h0 = np.random.default_rng(4).standard_normal((3, 4, 5))
    got = O.ssm_fold_recurrent(h0, x, B, np.zeros((11, 3)), A)
    assert np.array_equal(got, h0)


def test_outer_product_orientation_and_read():
    # one token, h0 = 0, x = e_p0, B = e_n0 -> only h[:, p0, n0] = dt
    x = np.zeros((1, 2, 4)); x[0, :, 1] = 1.0
    B = np.zeros((1, 5)); B[0, 3] = 1.0
    dt = np.array([[0.5, 0.25]])
    h = O.ssm_fold_recurrent(np.zeros((2, 4, 5)), x, B, dt, np.array([-1.0, -2.0]))
    want = np.zeros((2, 4, 5)); want[0, 1, 3] = 0.5; want[1, 1, 3] = 0.25
    assert np.array_equal(h, want)
    # read: one-hot C selects column n0 of every head's state
    hr = np.random.default_rng(0).standard_normal((2, 4, 5))
    C = np.zeros((2, 5)); C[0, 3] = 1.0; C[1, 0] = 2.0
    y = O.ssm_read(hr, C)
    assert np.array_equal(y[0], hr[:, :, 3]) and np.array_equal(y[1], 2.0 * hr[:, :, 0])


def test_ssm_inputs_use_softplus_and_bias():
    cfg = small_cfg()
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    f = np.random.default_rng(3).standard_normal((5, cfg.d_model))
    x, B, dt = O.ssm_inputs(lw, cfg, f)
    tf = torch.tensor(f)
    ref_dt = torch.nn.functional.softplus(tf @ torch.tensor(lw.w_dt) + torch.tensor(lw.dt_bias),
                                          threshold=1e6).numpy()
    assert rel(dt, ref_dt) < 1e-14
    assert x.shape == (5, cfg.ssm_heads, cfg.ssm_headdim) and B.shape == (5, cfg.d_state)
    assert np.all(lw.A < 0)


# ---------------------------------------------------------------- ring

def test_ring_matches_bruteforce_last_window():
    cfg = small_cfg(window=5)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(11)
    history = []  # every committed feature row, in order
    feats0 = rng.standard_normal((3, cfg.d_model))
    ctx = O.prefill_layer(lw, cfg, feats0)
    history += list(feats0)
    for _ in range(12):
        rows = rng.standard_normal((8, cfg.d_model))
        n = int(rng.integers(0, 9))
        ctx = O.commit_layer(lw, cfg, ctx, rows, n)
        history += list(rows[:n])
        T = len(history)
        assert ctx.pos == T
        last = list(range(max(0, T - cfg.window), T))
        for s in range(cfg.window):
            holders = [p for p in last if p % cfg.window == s]
            if holders:
                p = holders[0]
                assert ctx.tag[s] == p
                k, _ = O.kv_of(lw, cfg, np.asarray(history[p])[None])
                assert np.allclose(ctx.ring_k[:, s, :], k[0], rtol=0, atol=1e-13)
            else:
                assert ctx.tag[s] == -1


# ---------------------------------------------------------------- commit invariants

def test_commit_zero_and_rejected_rows():
    cfg = small_cfg()
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(12)
    ctx = O.prefill_layer(lw, cfg, rng.standard_normal((9, cfg.d_model)))
    rows = rng.standard_normal((8, cfg.d_model))
    z = O.commit_layer(lw, cfg, ctx, rows, 0)
    assert np.array_equal(z.h, ctx.h) and np.array_equal(z.ring_k, ctx.ring_k) and z.pos == ctx.pos
    for n in range(1, 9):
        a = O.commit_layer(lw, cfg, ctx, rows, n)
        rows2 = rows.copy()
        rows2[n:] = rng.standard_normal((8 - n, cfg.d_model)) * 100.0
        b = O.commit_layer(lw, cfg, ctx, rows2, n)
        assert np.array_equal(a.h, b.h) and np.array_equal(a.ring_k, b.ring_k)
        assert np.array_equal(a.ring_v, b.ring_v) and a.pos == b.pos


def test_split_commit_equals_single_and_prefill():
    cfg = small_cfg(window=4)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(13)
    pre = rng.standard_normal((7, cfg.d_model))
    rows = rng.standard_normal((8, cfg.d_model))
    base = O.prefill_layer(lw, cfg, pre, method="recurrent")
    one = O.commit_layer(lw, cfg, base, rows, 7)
    two = O.commit_layer(lw, cfg, O.commit_layer(lw, cfg, base, rows[:3], 3), rows[3:], 4)
    assert rel(two.h, one.h) < 1e-13 and np.array_equal(two.tag, one.tag)
    assert np.array_equal(two.ring_k, one.ring_k)
    full = O.prefill_layer(lw, cfg, np.concatenate([pre, rows[:7]]), method="chunked", chunk=3)
    assert rel(full.h, one.h) < 1e-12 and np.array_equal(full.tag, one.tag)
    assert np.allclose(full.ring_v, one.ring_v, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- attention

def test_window_covering_prefix_equals_full_attention_sdpa():
    cfg = small_cfg(window=64)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(14)
    pre = rng.standard_normal((23, cfg.d_model))
    ctx = O.prefill_layer(lw, cfg, pre)
    X = rng.standard_normal((7, cfg.d_model))
    _, parts = O.draft_layer(lw, cfg, ctx, X, return_parts=True)
    kp, vp = O.kv_of(lw, cfg, pre)
    keys = np.concatenate([kp, parts["Ks"]], 0)       # [L+7, Hkv, dh]
    vals = np.concatenate([vp, parts["Vs"]], 0)
    q = torch.tensor(parts["Q"]).permute(1, 0, 2)[None]   # [1, Hq, 7, dh]
    k = torch.tensor(keys).permute(1, 0, 2)[None]
    v = torch.tensor(vals).permute(1, 0, 2)[None]
    G = cfg.n_q_heads // cfg.n_kv_heads
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1))
    ref = ref[0].permute(1, 0, 2).numpy()
    assert rel(parts["O"], ref) < 1e-13


def test_equal_keys_give_mean_of_values():
    cfg = small_cfg(window=8)
    ctx = O.Context.empty(cfg)
    rng = np.random.default_rng(15)
    k = np.tile(rng.standard_normal((1, cfg.n_kv_heads, cfg.head_dim)), (5, 1, 1))
    v = rng.standard_normal((5, cfg.n_kv_heads, cfg.head_dim))
    O.ring_append(ctx, cfg, k, v, 0)
    ctx.pos = 5
    Q = rng.standard_normal((7, cfg.n_q_heads, cfg.head_dim))
    Ks = np.tile(k[:1], (7, 1, 1))
    Vs = rng.standard_normal((7, cfg.n_kv_heads, cfg.head_dim))
    out = O.window_block_attention(cfg, ctx, Q, Ks, Vs)
    G = cfg.n_q_heads // cfg.n_kv_heads
    for hq in range(cfg.n_q_heads):
        mean = np.concatenate([v[:, hq // G], Vs[:, hq // G]]).mean(0)
        assert np.allclose(out[:, hq], mean[None], rtol=0, atol=1e-14)


def test_empty_window_attends_slots_only():
    cfg = small_cfg()
    ctx = O.Context.empty(cfg)
    ctx.ring_k[:] = 1e3  # garbage in unused slots must not be read
    rng = np.random.default_rng(16)
    Q = rng.standard_normal((7, cfg.n_q_heads, cfg.head_dim))
    Ks = rng.standard_normal((7, cfg.n_kv_heads, cfg.head_dim))
    Vs = rng.standard_normal((7, cfg.n_kv_heads, cfg.head_dim))
    out = O.window_block_attention(cfg, ctx, Q, Ks, Vs)
    q = torch.tensor(Q).permute(1, 0, 2)[None]
    G = cfg.n_q_heads // cfg.n_kv_heads
    k = torch.tensor(Ks).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    v = torch.tensor(Vs).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v)[0].permute(1, 0, 2).numpy()
    assert rel(out, ref) < 1e-13


# ---------------------------------------------------------------- layer output

def test_layer_output_composition():
    cfg = small_cfg()
    w = make_layer_weights(cfg, 0)
    lw = O.Weights64.from_any(w)
    rng = np.random.default_rng(17)
    ctx = O.prefill_layer(lw, cfg, rng.standard_normal((9, cfg.d_model)))
    X = rng.standard_normal((7, cfg.d_model))
    # zero output projections: the layer is the identity on the residual
    lz = O.Weights64(**{**lw.__dict__, "w_o": np.zeros_like(lw.w_o), "w_mo": np.zeros_like(lw.w_mo)})
    assert np.array_equal(O.draft_layer(lz, cfg, ctx, X), X)
    # only the memory branch: out - X = y W_mo with y the one-hot-checked read
    lm = O.Weights64(**{**lw.__dict__, "w_o": np.zeros_like(lw.w_o)})
    out = O.draft_layer(lm, cfg, ctx, X)
    y = torch.einsum("hpn,sn->shp", torch.tensor(ctx.h), torch.tensor(X) @ torch.tensor(lw.w_C))
    ref = (y.reshape(7, -1) @ torch.tensor(lw.w_mo)).numpy()
    assert rel(out - X, ref) < 1e-10  # out - X cancels against |X| ~ 1


def test_draft_leaves_context_unchanged():
    cfg = small_cfg()
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(18)
    ctx = O.prefill_layer(lw, cfg, rng.standard_normal((9, cfg.d_model)))
    before = ctx.clone()
    O.draft_layer(lw, cfg, ctx, rng.standard_normal((7, cfg.d_model)))
    assert np.array_equal(before.h, ctx.h) and np.array_equal(before.ring_k, ctx.ring_k)
    assert np.array_equal(before.tag, ctx.tag) and before.pos == ctx.pos


def test_batched_drafter_invalid_count_is_noop_and_flagged():
    cfg = small_cfg()
    w = [make_layer_weights(cfg, 0)]
    d = O.OracleDrafter(cfg, w, 3)
    rng = np.random.default_rng(19)
    d.prefill([5, 0, 12], rng.standard_normal((17, cfg.d_model)))
    snap = [c[0].clone() for c in d.ctx]
    offs, err = d.commit(rng.standard_normal((3, 8, cfg.d_model)), [3, 9, 8])
    assert err and list(offs) == [0, 3, 3, 11]
    assert np.array_equal(d.ctx[1][0].h, snap[1].h) and d.ctx[1][0].pos == 0
    assert d.ctx[0][0].pos == 8 and d.ctx[2][0].pos == 20


# ---------------------------------------------------------------- sizing (pages' figures)

def test_sizing_matches_printed_figures():
    g = json.load(open(os.path.join(GOLDEN, "sizing.json")))
    t = g["target_kv_32k"]
    assert O.target_kv_bytes(t["n_layers"], t["n_kv_heads"], t["head_dim"], t["seq"],
                             t["elem_bytes"]) == t["bytes"] == int(6.25 * 2**30)
    k = g["drafter_window_kv"]
    kv = O.window_kv_bytes(k["n_layers"], k["n_kv_heads"], k["head_dim"], k["window"], k["elem_bytes"])
    assert kv == k["bytes"] == int(2.5 * 2**20)
    s = g["drafter_state"]
    st = O.state_bytes(s["n_layers"], s["d_inner"], s["d_state"], s["elem_bytes"])
    assert st == s["bytes"] == int(2.5 * 2**20)
    assert kv + st == g["drafter_context_total"]["bytes"]


# ---------------------------------------------------------------- ablation modes
# (paper, intervention table: "Cross-slot off", "SSM: Last 512", "SSM: Last
# feature"; explainer, paragraph on the ablations)

def test_cross_slot_off_empty_window_returns_own_value():
    # with no window entries each slot attends to its own key alone: O = V_s
    cfg = small_cfg(cross_slot=False)
    ctx = O.Context.empty(cfg)
    ctx.ring_k[:] = 1e3  # unused slots are never read
    rng = np.random.default_rng(30)
    Q = rng.standard_normal((7, cfg.n_q_heads, cfg.head_dim))
    Ks = rng.standard_normal((7, cfg.n_kv_heads, cfg.head_dim))
    Vs = rng.standard_normal((7, cfg.n_kv_heads, cfg.head_dim))
    out = O.window_block_attention(cfg, ctx, Q, Ks, Vs)
    G = cfg.n_q_heads // cfg.n_kv_heads
    for hq in range(cfg.n_q_heads):
        assert np.array_equal(out[:, hq], Vs[:, hq // G])


def test_cross_slot_off_matches_sdpa_with_mask():
    cfg = small_cfg(window=64, cross_slot=False)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(31)
    pre = rng.standard_normal((23, cfg.d_model))
    ctx = O.prefill_layer(lw, cfg, pre)
    X = rng.standard_normal((7, cfg.d_model))
    _, parts = O.draft_layer(lw, cfg, ctx, X, return_parts=True)
    kp, vp = O.kv_of(lw, cfg, pre)
    keys = np.concatenate([kp, parts["Ks"]], 0)
    vals = np.concatenate([vp, parts["Vs"]], 0)
    allowed = torch.ones((7, 23 + 7), dtype=torch.bool)
    allowed[:, 23:] = torch.eye(7, dtype=torch.bool)   # window + own key
    q = torch.tensor(parts["Q"]).permute(1, 0, 2)[None]
    G = cfg.n_q_heads // cfg.n_kv_heads
    k = torch.tensor(keys).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    v = torch.tensor(vals).permute(1, 0, 2)[None].repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed)
    assert rel(parts["O"], ref[0].permute(1, 0, 2).numpy()) < 1e-13
    # and it differs from the default (slots interact)
    full = O.window_block_attention(small_cfg(window=64), ctx, parts["Q"], parts["Ks"], parts["Vs"])
    assert rel(full, parts["O"]) > 1e-3


def _last_term(lw, cfg, f):
    """dt x (outer) B of one feature row via torch (softplus and matmuls)."""
    ft = torch.tensor(f[None])
    dt = torch.nn.functional.softplus(ft @ torch.tensor(lw.w_dt) + torch.tensor(lw.dt_bias),
                                      threshold=1e6)[0]
    x = (ft @ torch.tensor(lw.w_x))[0].reshape(cfg.ssm_heads, cfg.ssm_headdim)
    B = (ft @ torch.tensor(lw.w_B))[0]
    return (dt[:, None, None] * x[:, :, None] * B[None, None, :]).numpy()


def test_memory_horizon_one_is_last_feature():
    cfg = small_cfg(mem_horizon=1)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(32)
    pre = rng.standard_normal((9, cfg.d_model))
    ctx = O.prefill_layer(lw, cfg, pre)
    assert rel(ctx.h, _last_term(lw, cfg, pre[-1])) < 1e-14
    rows = rng.standard_normal((8, cfg.d_model))
    c = O.commit_layer(lw, cfg, ctx, rows, 3)
    assert rel(c.h, _last_term(lw, cfg, rows[2])) < 1e-14
    z = O.commit_layer(lw, cfg, c, rows, 0)    # n = 0: unchanged
    assert np.array_equal(z.h, c.h)


def test_memory_horizon_without_decay_is_window_sum():
    # A = 0: the memory is the plain sum of dt x (outer) B over the last M features
    cfg = small_cfg(mem_horizon=5)
    w = make_layer_weights(cfg, 0)
    lw = O.Weights64.from_any(w)
    lw.A_log[:] = -1e9                          # A = -exp(-1e9) = 0
    rng = np.random.default_rng(33)
    feats = rng.standard_normal((9 + 3 + 4, cfg.d_model))
    ctx = O.prefill_layer(lw, cfg, feats[:9])
    ctx = O.commit_layer(lw, cfg, ctx, feats[9:17], 3)
    ctx = O.commit_layer(lw, cfg, ctx, np.concatenate([feats[12:], feats[:4]]), 4)
    want = sum(_last_term(lw, cfg, feats[t]) for t in range(16 - 5, 16))
    assert rel(ctx.h, want) < 1e-13
    # the window moved past the early features: those no longer count at all
    assert rel(ctx.h, sum(_last_term(lw, cfg, feats[t]) for t in range(16 - 6, 16))) > 1e-3


def test_memory_horizon_long_enough_equals_whole_history():
    cfg_all = small_cfg()
    cfg_m = small_cfg(mem_horizon=40)
    lw = O.Weights64.from_any(make_layer_weights(cfg_all, 0))
    rng = np.random.default_rng(34)
    pre = rng.standard_normal((11, cfg_all.d_model))
    rows = rng.standard_normal((8, cfg_all.d_model))
    a = O.commit_layer(lw, cfg_all, O.prefill_layer(lw, cfg_all, pre), rows, 6)
    b = O.commit_layer(lw, cfg_m, O.prefill_layer(lw, cfg_m, pre), rows, 6)
    assert rel(b.h, a.h) < 1e-12


def test_memory_horizon_commits_equal_prefill_of_last_m():
    # whatever the commit pattern, the memory is the fold of the last M features
    cfg = small_cfg(mem_horizon=6)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(35)
    feats = rng.standard_normal((30, cfg.d_model))
    ctx = O.prefill_layer(lw, cfg, feats[:4])
    used = 4
    for n in (3, 0, 8, 1, 5):
        rows = np.concatenate([feats[used:used + n], rng.standard_normal((8 - n, cfg.d_model))])
        ctx = O.commit_layer(lw, cfg, ctx, rows, n)
        used += n
        ref = O.prefill_layer(lw, small_cfg(), feats[max(0, used - 6):used], method="recurrent")
        assert rel(ctx.h, ref.h) < 1e-12


# ---------------------------------------------------------------- gated-delta memory
# (gated delta rule of "Gated Delta Networks: Improving Mamba2 with Delta Rule";
# the paper's memory-swap table)

def test_gdn_delta_rule_retrieves_last_write_per_key():
    # alpha = 1, beta = 1 and orthonormal keys: S e_i is the last value
    # written at key i, and unwritten keys read zero
    Hm, P, N, T = 2, 3, 5, 9
    rng = np.random.default_rng(40)
    keys = rng.integers(0, 4, size=T)            # key 4 never written
    k = np.eye(N)[keys]
    v = rng.standard_normal((T, Hm, P))
    S = O.gdn_fold_recurrent(np.zeros((Hm, P, N)), v, k, np.ones((T, Hm)), np.ones((T, Hm)))
    for i in range(N):
        last = [t for t in range(T) if keys[t] == i]
        want = v[last[-1]] if last else np.zeros((Hm, P))
        assert np.allclose(S[:, :, i], want, rtol=0, atol=1e-14)


def test_gdn_zero_gate_keeps_only_the_last_token():
    Hm, P, N, T = 2, 3, 4, 6
    rng = np.random.default_rng(41)
    k = rng.standard_normal((T, N))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, Hm, P))
    beta = rng.uniform(0.1, 0.9, (T, Hm))
    S = O.gdn_fold_recurrent(rng.standard_normal((Hm, P, N)), v, k, np.zeros((T, Hm)), beta)
    want = beta[-1][:, None, None] * v[-1][:, :, None] * k[-1][None, None, :]
    assert rel(S, want) < 1e-15


def test_gdn_zero_beta_is_pure_decay():
    Hm, P, N, T = 2, 3, 4, 5
    rng = np.random.default_rng(42)
    k = rng.standard_normal((T, N))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    alpha = rng.uniform(0.5, 1.0, (T, Hm))
    S0 = rng.standard_normal((Hm, P, N))
    S = O.gdn_fold_recurrent(S0, rng.standard_normal((T, Hm, P)), k, alpha, np.zeros((T, Hm)))
    assert rel(S, np.prod(alpha, axis=0)[:, None, None] * S0) < 1e-14


def test_gdn_rank_one_scalar_loops():
    # the update written element by element: S[p,n] <- a (S[p,n] - b (S k)[p] k[n]) + b v[p] k[n]
    Hm, P, N, T = 1, 2, 3, 4
    rng = np.random.default_rng(43)
    k = rng.standard_normal((T, N))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, Hm, P))
    a = rng.uniform(0.3, 1.0, (T, Hm))
    b = rng.uniform(0.0, 1.0, (T, Hm))
    S0 = rng.standard_normal((Hm, P, N))
    want = S0[0].tolist()
    for t in range(T):
        sk = [sum(want[p][m] * k[t, m] for m in range(N)) for p in range(P)]
        want = [[a[t, 0] * (want[p][n] - b[t, 0] * sk[p] * k[t, n]) + b[t, 0] * v[t, 0, p] * k[t, n]
                 for n in range(N)] for p in range(P)]
    got = O.gdn_fold_recurrent(S0, v, k, a, b)
    assert rel(got[0], np.array(want)) < 1e-13


def test_gdn_inputs_and_read():
    cfg = small_cfg(memory="gdn")
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(44)
    f = rng.standard_normal((5, cfg.d_model))
    v, k, alpha, beta = O.gdn_inputs(lw, cfg, f)
    assert np.allclose(np.linalg.norm(k, axis=1), 1.0, rtol=0, atol=1e-14)
    ref_beta = torch.sigmoid(torch.tensor(f) @ torch.tensor(lw.w_beta)).numpy()
    assert rel(beta, ref_beta) < 1e-14
    assert np.all(alpha > 0) and np.all(alpha < 1)
    S = rng.standard_normal((cfg.ssm_heads, cfg.ssm_headdim, cfg.d_state))
    C = rng.standard_normal((7, cfg.d_state))
    y = O.gdn_read(S, C)
    assert rel(O.gdn_read(S, 3.5 * C), y) < 1e-15          # scale of the query drops out
    qt = torch.nn.functional.normalize(torch.tensor(C), dim=1)
    assert rel(y, torch.einsum("hpn,sn->shp", torch.tensor(S), qt).numpy()) < 1e-14


def test_gdn_prefill_equals_commits():
    cfg = small_cfg(memory="gdn")
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    rng = np.random.default_rng(45)
    pre = rng.standard_normal((9, cfg.d_model))
    rows = rng.standard_normal((8, cfg.d_model))
    a = O.commit_layer(lw, cfg, O.commit_layer(lw, cfg, O.prefill_layer(lw, cfg, pre), rows, 3),
                       rows[3:], 5)
    b = O.prefill_layer(lw, cfg, np.concatenate([pre, rows]))
    assert rel(a.h, b.h) < 1e-12 and np.array_equal(a.tag, b.tag)
    z = O.commit_layer(lw, cfg, a, rows, 0)
    assert np.array_equal(z.h, a.h)


# ---------------------------------------------------------------- 4-bit weights

def test_q4_dequantization_matches_torch_and_bounds():
    from workload import make_layer_weights_q4
    cfg = small_cfg(d_model=256, weight_bits=4)
    wq = make_layer_weights_q4(cfg, 0)
    m = wq.w_x
    got = O.dequantize_q4(m)
    # torch: expand the group parameters over their 128 rows
    s = m.scales.double().repeat_interleave(128, dim=0)
    z = m.zeros.double().repeat_interleave(128, dim=0)
    ref = (s * (m.codes.double() - z)).numpy()
    assert np.array_equal(got, ref)
    # values lie on the group's grid and inside [s (0 - z), s (15 - z)]
    assert np.all(np.abs(got) <= 15 * s.numpy() + 1e-30)


def test_q4_round_trip_error_bound():
    # quantising a matrix to the nearest grid point and dequantising it moves
    # each entry by at most half a step s/2 (round to nearest)
    rng = np.random.default_rng(50)
    w = rng.standard_normal((256, 7)) * 0.02
    g = np.arange(256) // 128
    lo = np.stack([w[g == k].min(0) for k in range(2)])
    hi = np.stack([w[g == k].max(0) for k in range(2)])
    s = (hi - lo) / 15.0
    z = np.round(-lo / s)
    q = np.clip(np.round(w / s[g] + z[g]), 0, 15)

    class M:  # the oracle's input form
        pass
    m = M()
    m.codes, m.scales, m.zeros = q, s, z
    back = O.dequantize_q4(m)
    assert np.max(np.abs(back - w) / s[g]) <= 0.5 + 1e-9


# ---------------------------------------------------------------- brute force

def _bf_project(f, W, ncol):
    """Row f times the [len(f), ncol] matrix W, one scalar product per column."""
    return [sum(f[i] * W[i][c] for i in range(len(f))) for c in range(ncol)]


def test_bruteforce_sequence_on_tiny_shapes():
    """A prefill, two commits with rejected rows and a draft on tiny shapes
    (4 query heads over 2 KV heads, a window of 4 that the sequence wraps),
    recomputed from the definitions with scalar Python loops — the memory
    folded token by token (h <- exp(dt A) h + dt x B^T, dt = softplus(f W_dt
    + bias), A = -exp(A_log)), each slot attending with scale 1/sqrt(dh)
    over the last W committed keys and the 7 slot keys of its query head's
    KV head, y = C h, out = X + O W_o + y W_mo — against the oracle."""
    D, Hq, Hkv, dh, Wn, Hm, P, N, S = 8, 4, 2, 2, 4, 2, 2, 2, 7
    cfg = small_cfg(d_model=D, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=dh, window=Wn,
                    ssm_heads=Hm, ssm_headdim=P, d_state=N, chunk=2)
    lw = O.Weights64.from_any(make_layer_weights(cfg, 0))
    Wt = {k: getattr(lw, k).tolist() for k in
          ("w_q", "w_k", "w_v", "w_o", "w_x", "w_B", "w_C", "w_dt", "w_mo")}
    bias = lw.dt_bias.tolist()
    A = [-math.exp(v) for v in lw.A_log.tolist()]
    rng = np.random.default_rng(23)
    prefix = rng.standard_normal((6, D))
    commits = [(rng.standard_normal((8, D)), 3), (rng.standard_normal((8, D)), 1)]
    X = rng.standard_normal((S, D))

    ctx = O.prefill_layer(lw, cfg, prefix)
    for f, n in commits:
        ctx = O.commit_layer(lw, cfg, ctx, f, n)
    out = O.draft_layer(lw, cfg, ctx, X)

    committed = [list(r) for r in prefix] + [list(r) for f, n in commits for r in f[:n]]
    h = [[[0.0] * N for _ in range(P)] for _ in range(Hm)]
    for f in committed:
        x, B = _bf_project(f, Wt["w_x"], Hm * P), _bf_project(f, Wt["w_B"], N)
        dtr = _bf_project(f, Wt["w_dt"], Hm)
        for m in range(Hm):
            v = dtr[m] + bias[m]
            dt = max(v, 0.0) + math.log1p(math.exp(-abs(v)))
            decay = math.exp(dt * A[m])
            for p in range(P):
                for n in range(N):
                    h[m][p][n] = decay * h[m][p][n] + dt * x[m * P + p] * B[n]
    keys_from = committed[-Wn:] + [list(r) for r in X]
    K = [_bf_project(f, Wt["w_k"], Hkv * dh) for f in keys_from]
    V = [_bf_project(f, Wt["w_v"], Hkv * dh) for f in keys_from]
    want = []
    for s in range(S):
        xs = list(X[s])
        q = _bf_project(xs, Wt["w_q"], Hq * dh)
        C = _bf_project(xs, Wt["w_C"], N)
        o = [0.0] * (Hq * dh)
        for hq in range(Hq):
            g = hq // (Hq // Hkv)
            sc = [sum(q[hq * dh + c] * K[j][g * dh + c] for c in range(dh)) / math.sqrt(dh)
                  for j in range(len(K))]
            mx = max(sc)
            e = [math.exp(v - mx) for v in sc]
            for c in range(dh):
                o[hq * dh + c] = sum(e[j] * V[j][g * dh + c] for j in range(len(K))) / sum(e)
        y = [sum(h[m][p][n] * C[n] for n in range(N)) for m in range(Hm) for p in range(P)]
        want.append([xs[d] + sum(o[i] * Wt["w_o"][i][d] for i in range(Hq * dh))
                     + sum(y[i] * Wt["w_mo"][i][d] for i in range(Hm * P)) for d in range(D)])
    assert ctx.pos == len(committed) == 10
    assert rel(ctx.h, np.array(h)) < 1e-12
    assert rel(out, np.array(want)) < 1e-12
