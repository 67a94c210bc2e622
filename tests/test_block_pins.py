"""Pins for the full drafter block around the layer (oracle/full_block.py):
library routines (torch rms_norm, conv1d, SDPA), closed forms (impulse
response of the convolution, relative-position invariance of RoPE, identity
blocks) and invariants (prefill == commits, drafting is read-only, argmax
ties go to the lowest id)."""
import numpy as np
import pytest
import torch

from oracle import full_block as FB
from oracle import hyflash_oracle as O
from workload import CONFIGS, make_block_weights, make_head_weights, make_prefix_feats

TINY = CONFIGS["tiny_fp32"].replace(mlp_dim=192, vocab=53)


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(60)
    x = rng.standard_normal((5, 64))
    g = rng.standard_normal(64)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (64,), torch.tensor(g), eps=FB.EPS)
    assert rel(FB.rms_norm(x, g), ref.numpy()) < 1e-14


def test_rope_rotation_properties():
    rng = np.random.default_rng(61)
    q = rng.standard_normal((1, 2, 16))
    k = rng.standard_normal((1, 2, 16))
    # a rotation: norms kept; position 0 is the identity
    r = FB.rope(q, np.array([37]))
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-13)
    assert np.array_equal(FB.rope(q, np.array([0])), q)
    # scores depend on the distance only
    def score(pq, pk):
        return np.sum(FB.rope(q, np.array([pq])) * FB.rope(k, np.array([pk])), axis=-1)
    assert np.allclose(score(5, 2), score(105, 102), rtol=1e-10, atol=1e-12)
    assert not np.allclose(score(5, 2), score(5, 3))
    # as complex numbers: pair (i, i + dh/2) times exp(i p theta^(-2i/dh))
    p = 11
    z = q[..., :8] + 1j * q[..., 8:]
    w = z * np.exp(1j * p * FB.ROPE_THETA ** (-np.arange(8) * 2.0 / 16))
    assert rel(FB.rope(q, np.array([p])), np.concatenate([w.real, w.imag], axis=-1)) < 1e-14


def test_causal_conv_matches_torch_and_carries_state():
    rng = np.random.default_rng(62)
    T, C, K = 13, 6, 4
    u = rng.standard_normal((T, C))
    w = rng.standard_normal((C, K))
    b = rng.standard_normal(C)
    got, last = FB.causal_conv(np.zeros((K - 1, C)), u, w, b)
    ut = torch.tensor(u.T)[None]                                   # [1, C, T]
    ref = torch.nn.functional.conv1d(torch.nn.functional.pad(ut, (K - 1, 0)),
                                     torch.tensor(w)[:, None, :], torch.tensor(b), groups=C)
    ref = torch.nn.functional.silu(ref)[0].T.numpy()
    assert rel(got, ref) < 1e-14
    assert np.array_equal(last, u[-(K - 1):])
    # in pieces, the carried rows make the same sequence
    a, st = FB.causal_conv(np.zeros((K - 1, C)), u[:5], w, b)
    c, _ = FB.causal_conv(st, u[5:], w, b)
    assert rel(np.concatenate([a, c]), got) < 1e-15


def test_causal_conv_impulse_response():
    # a one-hot row at t = 0 gives the taps newest-first at t = 0, 1, 2, 3
    K, C = 4, 1
    u = np.zeros((6, C))
    u[0, 0] = 1.0
    w = np.array([[0.5, -1.0, 2.0, 3.0]])
    got, _ = FB.causal_conv(np.zeros((K - 1, C)), u, w, np.zeros(1))
    want = FB.silu(np.array([3.0, 2.0, -1.0, 0.5, 0.0, 0.0]))
    assert np.allclose(got[:, 0], want, rtol=0, atol=1e-15)


def _block(cfg=TINY, layer=0):
    return FB.BlockWeights64.from_any(make_block_weights(cfg, layer))


def test_block_prefill_equals_commits_and_draft_is_read_only():
    bw = _block()
    rng = np.random.default_rng(63)
    feats = rng.standard_normal((90, TINY.d_model))
    ctx = FB.block_prefill(bw, TINY, feats[:70])
    ctx = FB.block_commit(bw, TINY, ctx, feats[70:78], 5)         # rows 75..77 rejected
    ctx = FB.block_commit(bw, TINY, ctx, feats[80:88], 0)
    ctx = FB.block_commit(bw, TINY, ctx, feats[75:83], 8)
    ref = FB.block_prefill(bw, TINY, feats[:83])
    assert ctx.pos == ref.pos == 83
    assert rel(ctx.h, ref.h) < 1e-12 and rel(ctx.conv, ref.conv) < 1e-15
    assert np.array_equal(ctx.tag, ref.tag)
    assert rel(ctx.ring_k, ref.ring_k) < 1e-13 and rel(ctx.ring_v, ref.ring_v) < 1e-13
    before = ctx.clone()
    FB.block_draft(bw, TINY, ctx, rng.standard_normal((7, TINY.d_model)))
    for name in ("ring_k", "ring_v", "tag", "h", "conv"):
        assert np.array_equal(getattr(ctx, name), getattr(before, name))
    assert ctx.pos == before.pos


def test_block_without_outputs_is_identity():
    bw = _block()
    for name in ("w_o", "w_mo"):
        setattr(bw.layer, name, np.zeros_like(getattr(bw.layer, name)))
    bw.w_down = np.zeros_like(bw.w_down)
    rng = np.random.default_rng(64)
    ctx = FB.block_prefill(bw, TINY, rng.standard_normal((30, TINY.d_model)))
    X = rng.standard_normal((7, TINY.d_model))
    assert np.array_equal(FB.block_draft(bw, TINY, ctx, X), X)


def test_block_attention_with_rope_matches_sdpa():
    # window covering the prefix: the block's attention over rotated prefix
    # keys and rotated slot keys equals torch SDPA on the same rotations
    cfg = TINY.replace(window=64)
    bw = _block(cfg)
    lw = bw.layer
    rng = np.random.default_rng(65)
    pre = rng.standard_normal((20, cfg.d_model))
    ctx = FB.block_prefill(bw, cfg, pre)
    X = rng.standard_normal((7, cfg.d_model))
    a = FB.rms_norm(X, bw.g_mix)
    pos = 20 + np.arange(7)
    Q = FB.rope((a @ lw.w_q).reshape(7, cfg.n_q_heads, cfg.head_dim), pos)
    Ks = FB.rope((a @ lw.w_k).reshape(7, cfg.n_kv_heads, cfg.head_dim), pos)
    Vs = (a @ lw.w_v).reshape(7, cfg.n_kv_heads, cfg.head_dim)
    kp, vp = O.kv_of(lw, cfg, pre)
    keys = np.concatenate([FB.rope(kp, np.arange(20)), Ks])
    vals = np.concatenate([vp, Vs])
    G = cfg.n_q_heads // cfg.n_kv_heads
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(Q).permute(1, 0, 2)[None],
        torch.tensor(keys).permute(1, 0, 2)[None].repeat_interleave(G, dim=1),
        torch.tensor(vals).permute(1, 0, 2)[None].repeat_interleave(G, dim=1))[0].permute(1, 0, 2)
    got = O.window_block_attention(cfg, ctx, Q, Ks, Vs)
    assert rel(got, ref.numpy()) < 1e-13


def test_head_argmax_ties_to_lowest_id():
    hw = FB.HeadWeights64(g_final=np.ones(4), w_lm=np.zeros((4, 6)))
    hw.w_lm[:, 2] = hw.w_lm[:, 4] = 1.0   # columns 2 and 4 tie for every input
    X = np.abs(np.random.default_rng(66).standard_normal((3, 4))) + 0.1
    logits, tok = FB.head(hw, X)
    assert np.array_equal(tok, [2, 2, 2])
    assert np.array_equal(logits[:, 2], logits[:, 4])


def test_block_drafter_runs_rounds():
    cfg = TINY.replace(batch=2, n_layers=2)
    from workload import make_round_inputs, make_accepted
    d = FB.OracleBlockDrafter(cfg, [make_block_weights(cfg, l) for l in range(2)],
                              make_head_weights(cfg), 2)
    d.prefill([0, 40], make_prefix_feats(cfg, [0, 40]))
    for r in range(2):
        slot, feats = make_round_inputs(cfg, r, 2)
        h, tok = d.draft(slot)
        assert h.shape == (2, 7, cfg.d_model) and tok.shape == (2, 7)
        assert np.all((tok >= 0) & (tok < cfg.vocab))
        d.commit(feats, make_accepted(cfg, r, 2))
    assert [c.pos for c in d.ctx[1]] == [d.ctx[1][0].pos] * 2


def _torch_rms(x, g):
    t = torch.tensor(x)
    return torch.nn.functional.rms_norm(t, (t.shape[-1],), torch.tensor(g), eps=FB.EPS)


def test_skip_and_gate_with_empty_memory():
    """B4 with h = 0 (nothing committed): the memory branch is
    (D[head] * x_s) * silu(z_s) per channel, taken through W_mo. Checked
    against torch (rms_norm, silu, matmuls) with distinct D per head and a
    random W_mo, so that a gate on the other side of W_mo, D per channel, or
    silu on x instead of z all fail."""
    cfg = TINY
    bw = _block(cfg)
    rng = np.random.default_rng(67)
    lw = bw.layer
    lw.w_o = np.zeros_like(lw.w_o)        # attention branch off
    bw.w_down = np.zeros_like(bw.w_down)  # MLP off
    bw.d_skip = np.array([0.3, -1.2, 2.0, 0.7])
    assert bw.d_skip.shape == (cfg.ssm_heads,)
    ctx = FB.BlockContext.empty(cfg)      # h = 0: C h vanishes
    X = rng.standard_normal((7, cfg.d_model))
    got = FB.block_draft(bw, cfg, ctx, X) - X
    a = _torch_rms(X, bw.g_mix)
    xs = a @ torch.tensor(lw.w_x)
    z = a @ torch.tensor(bw.w_z)
    D = torch.tensor(bw.d_skip).repeat_interleave(cfg.ssm_headdim)
    want = ((D * xs) * torch.nn.functional.silu(z)) @ torch.tensor(lw.w_mo)
    assert rel(got, want.numpy()) < 1e-12
    # a gate applied after W_mo, or D per channel index mod heads, differs
    wrong = (D * xs) @ torch.tensor(lw.w_mo) * torch.nn.functional.silu(z[:, :cfg.d_model])
    assert rel(got, wrong.numpy()) > 1e-2
    Dw = torch.tensor(bw.d_skip)[torch.arange(cfg.d_inner) % cfg.ssm_heads]
    wrong2 = ((Dw * xs) * torch.nn.functional.silu(z)) @ torch.tensor(lw.w_mo)
    assert rel(got, wrong2.numpy()) > 1e-2


def test_gated_read_with_state_and_no_skip():
    """B4 with a folded memory and D = 0: the branch is (C_s h) * silu(z_s)
    per channel, with C_s h written out as torch einsum over the state the
    fold left (the fold itself is pinned against the recurrence)."""
    cfg = TINY
    bw = _block(cfg)
    lw = bw.layer
    lw.w_o = np.zeros_like(lw.w_o)
    bw.w_down = np.zeros_like(bw.w_down)
    bw.d_skip = np.zeros_like(bw.d_skip)
    rng = np.random.default_rng(68)
    ctx = FB.block_prefill(bw, cfg, rng.standard_normal((40, cfg.d_model)))
    assert np.max(np.abs(ctx.h)) > 0
    X = rng.standard_normal((7, cfg.d_model))
    got = FB.block_draft(bw, cfg, ctx, X) - X
    a = _torch_rms(X, bw.g_mix)
    C = a @ torch.tensor(lw.w_C)                                   # [S, N]
    y = torch.einsum("hpn,sn->shp", torch.tensor(ctx.h), C).reshape(7, -1)
    want = (y * torch.nn.functional.silu(a @ torch.tensor(bw.w_z))) @ torch.tensor(lw.w_mo)
    assert rel(got, want.numpy()) < 1e-12


def test_swiglu_mlp_matches_torch():
    """B5: with both mixer branches off, out = X + W_down(silu(n W_gate) *
    (n W_up)) with n = rms_norm(X, g_mlp); torch silu / rms_norm / matmuls.
    Swapping gate and up, or leaving out the norm, fails."""
    cfg = TINY
    bw = _block(cfg)
    lw = bw.layer
    lw.w_o = np.zeros_like(lw.w_o)
    lw.w_mo = np.zeros_like(lw.w_mo)
    rng = np.random.default_rng(69)
    ctx = FB.block_prefill(bw, cfg, rng.standard_normal((10, cfg.d_model)))
    X = 3.0 * rng.standard_normal((7, cfg.d_model))
    got = FB.block_draft(bw, cfg, ctx, X)
    n = _torch_rms(X, bw.g_mlp)
    silu = torch.nn.functional.silu
    G, U, Dn = (torch.tensor(bw.w_gate), torch.tensor(bw.w_up), torch.tensor(bw.w_down))
    want = torch.tensor(X) + (silu(n @ G) * (n @ U)) @ Dn
    assert rel(got, want.numpy()) < 1e-12
    swapped = torch.tensor(X) + (silu(n @ U) * (n @ G)) @ Dn
    assert rel(got - X, (swapped - torch.tensor(X)).numpy()) > 1e-2
    no_norm = torch.tensor(X) + (silu(torch.tensor(X) @ G) * (torch.tensor(X) @ U)) @ Dn
    assert rel(got - X, (no_norm - torch.tensor(X)).numpy()) > 1e-2


def test_swiglu_closed_form_identity_weights():
    """B5 closed form: D = F, W_gate = W_up = W_down = I and unit gains give
    out = X + silu(n) * n elementwise."""
    cfg = TINY.replace(mlp_dim=TINY.d_model)
    bw = _block(cfg)
    lw = bw.layer
    lw.w_o = np.zeros_like(lw.w_o)
    lw.w_mo = np.zeros_like(lw.w_mo)
    I = np.eye(cfg.d_model)
    bw.w_gate, bw.w_up, bw.w_down = I.copy(), I.copy(), I.copy()
    bw.g_mlp = np.ones(cfg.d_model)
    X = np.random.default_rng(70).standard_normal((7, cfg.d_model))
    n = X / np.sqrt(np.mean(X * X, axis=-1, keepdims=True) + FB.EPS)
    got = FB.block_draft(bw, cfg, FB.BlockContext.empty(cfg), X)
    assert rel(got, X + n * n / (1.0 + np.exp(-n))) < 1e-13


def test_block_fold_with_newest_tap_is_fold_of_silu_inputs():
    """B3 inside the fold: with conv taps (0, 0, 0, 1) and zero bias the
    convolution is silu of the newest row, so the memory equals the layer's
    recurrence over silu(x), silu(B) (torch silu); with a memory that
    forgets at once (A -> -inf) it is dt_last * silu(x_last) (x) silu(B_last)."""
    cfg = TINY
    bw = _block(cfg)
    lw = bw.layer
    bw.conv_w = np.zeros_like(bw.conv_w)
    bw.conv_w[:, 3] = 1.0
    bw.conv_b = np.zeros_like(bw.conv_b)
    rng = np.random.default_rng(71)
    f = rng.standard_normal((25, cfg.d_model))
    ctx = FB.block_prefill(bw, cfg, f)
    silu = lambda a: torch.nn.functional.silu(torch.tensor(a)).numpy()
    x = silu(f @ lw.w_x).reshape(25, cfg.ssm_heads, cfg.ssm_headdim)
    B = silu(f @ lw.w_B)
    dt = torch.nn.functional.softplus(torch.tensor(f @ lw.w_dt + lw.dt_bias)).numpy()
    h = np.zeros_like(ctx.h)
    for t in range(25):   # h <- exp(dt A) h + dt x (x) B, written out per token
        h = np.exp(dt[t] * lw.A)[:, None, None] * h + dt[t][:, None, None] * x[t][:, :, None] * B[t][None, None, :]
    assert rel(ctx.h, h) < 1e-12
    lw.A_log = np.full_like(lw.A_log, 50.0)     # exp(dt A) underflows to 0
    ctx = FB.block_prefill(bw, cfg, f)
    want = dt[-1][:, None, None] * x[-1][:, :, None] * B[-1][None, None, :]
    assert rel(ctx.h, want) < 1e-12
