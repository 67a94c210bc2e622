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
