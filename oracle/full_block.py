"""The full drafter block around the HyFlash layer, in float64 NumPy -- TEST
INFRASTRUCTURE.

Only tests (and, later, the benchmark's CPU arms) use this module; it shares
nothing with the CUDA library. It extends the layer of hyflash_oracle (window
+ block attention, Mamba-2 memory written only by commits) into one complete
draft step of a drafter network: norms, rotary positions, the memory's
convolution and gating, an MLP, and an LM head with a per-slot argmax.

The pages ("HyFlash: A Prefix-Memory Prior for On-Device Speculative
Decoding"; the learnaivisually explainer, "That is HyFlash") describe a
two-layer drafter whose layers have a local-attention branch and a Mamba-2
branch, and name none of these surrounding parts. Each follows the plainest
reading of the model families the pages use (Qwen3 targets, Mamba-2 memory):

  B1 pre-norm: RMSNorm (eps 1e-6, learned gain) before the two mixer branches
     (one norm shared by attention and memory), one before the MLP, and a
     final one before the LM head;
  B2 rotary positions: rotate-half RoPE over the whole head dim, base 1e6;
     a committed feature's key is rotated at its position when it enters the
     window (the ring stores rotated keys); slot s's query and key sit at
     position pos + s, right after the committed prefix;
  B3 convolution: Mamba-2's depthwise causal conv1d of width 4 with bias,
     then SiLU, over the committed rows' x and B channels; its state is the
     last 3 committed pre-conv rows, carried across commits (zeros before the
     first feature). dt is not convolved; the draft-time C is not either
     (drafting is read-only and the slots are not committed);
  B4 D-skip and gate: y_s = C_s h + D * x_s with x_s = a_s W_x (the slot's
     own input), then y_s * silu(z_s) with z_s = a_s W_z; no gated norm;
  B5 MLP: SwiGLU, W_down(silu(n W_gate) * (n W_up)), width F;
  B6 LM head: logits = RMSNorm(X_L) W_lm; the token of a slot is the argmax,
     ties to the lowest token id;
  B7 committed features enter the K/V and x/B/dt projections without a norm,
     as in the layer (they are the target's features).
"""
from __future__ import annotations

import copy
import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

from . import hyflash_oracle as O

EPS = 1e-6
ROPE_THETA = 1e6
CONV_WIDTH = 4


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float = EPS) -> np.ndarray:
    """B1: x / sqrt(mean(x^2) + eps) * g over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x: np.ndarray, positions: np.ndarray, theta: float = ROPE_THETA) -> np.ndarray:
    """B2: x [T, H, dh] rotated at positions [T]; pairs (i, i + dh/2)."""
    T, H, dh = x.shape
    half = dh // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / dh)      # [half]
    ang = positions.astype(np.float64)[:, None] * inv[None, :]         # [T, half]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def causal_conv(hist: np.ndarray, u: np.ndarray, w: np.ndarray, b: np.ndarray):
    """B3: depthwise causal convolution of rows u [T, C] that follow the
    rows hist [K-1, C]; w [C, K] (tap K-1 on the newest row), b [C].
    Returns (SiLU of the convolution [T, C], the new last K-1 rows)."""
    K = w.shape[1]
    seq = np.concatenate([hist, u], axis=0)                             # [K-1+T, C]
    out = np.zeros_like(u)
    for t in range(u.shape[0]):
        window = seq[t:t + K]                                           # rows t-K+1 .. t
        out[t] = np.sum(window.T * w, axis=1) + b
    return silu(out), seq[-(K - 1):].copy()


@dataclasses.dataclass
class BlockWeights64:
    layer: O.Weights64
    g_mix: np.ndarray      # [D]
    g_mlp: np.ndarray      # [D]
    w_z: np.ndarray        # [D, Hm*P]
    d_skip: np.ndarray     # [Hm]
    conv_w: np.ndarray     # [Hm*P + N, K]
    conv_b: np.ndarray     # [Hm*P + N]
    w_gate: np.ndarray     # [D, F]
    w_up: np.ndarray       # [D, F]
    w_down: np.ndarray     # [F, D]

    @staticmethod
    def from_any(w) -> "BlockWeights64":
        names = [f.name for f in dataclasses.fields(BlockWeights64) if f.name != "layer"]
        return BlockWeights64(layer=O.Weights64.from_any(w.layer),
                              **{n: O.to64(getattr(w, n)) for n in names})


@dataclasses.dataclass
class HeadWeights64:
    g_final: np.ndarray    # [D]
    w_lm: np.ndarray       # [D, V]

    @staticmethod
    def from_any(w) -> "HeadWeights64":
        return HeadWeights64(g_final=O.to64(w.g_final), w_lm=O.to64(w.w_lm))


@dataclasses.dataclass
class BlockContext:
    ring_k: np.ndarray     # [Hkv, W, dh], rotated at the committed positions
    ring_v: np.ndarray
    tag: np.ndarray        # [W]
    pos: int
    h: np.ndarray          # [Hm, P, N]
    conv: np.ndarray       # [K-1, Hm*P + N] last committed pre-conv x | B rows

    @staticmethod
    def empty(cfg) -> "BlockContext":
        base = O.Context.empty(cfg)
        return BlockContext(ring_k=base.ring_k, ring_v=base.ring_v, tag=base.tag, pos=0,
                            h=base.h, conv=np.zeros((CONV_WIDTH - 1, cfg.d_inner + cfg.d_state)))

    def clone(self) -> "BlockContext":
        return copy.deepcopy(self)


def _fold(bw: BlockWeights64, cfg, ctx: BlockContext, feats: np.ndarray):
    """Append committed features [T, D] at positions ctx.pos.. (B2, B3, B7)."""
    lw = bw.layer
    T = feats.shape[0]
    positions = ctx.pos + np.arange(T)
    k, v = O.kv_of(lw, cfg, feats)
    first = max(0, T - cfg.window)  # only the last W can remain in the window
    O.ring_append(ctx, cfg, rope(k[first:], positions[first:]), v[first:], ctx.pos + first)
    x = feats @ lw.w_x
    B = feats @ lw.w_B
    dt = O.softplus(feats @ lw.w_dt + lw.dt_bias[None, :])
    u, ctx.conv = causal_conv(ctx.conv, np.concatenate([x, B], axis=1), bw.conv_w, bw.conv_b)
    xc = u[:, :cfg.d_inner].reshape(T, cfg.ssm_heads, cfg.ssm_headdim)
    ctx.h = O.ssm_fold_recurrent(ctx.h, xc, u[:, cfg.d_inner:], dt, lw.A)
    ctx.pos += T


def block_prefill(bw: BlockWeights64, cfg, feats: np.ndarray) -> BlockContext:
    """The committed prefix [L, D] folded into a fresh context."""
    ctx = BlockContext.empty(cfg)
    if feats.shape[0]:
        _fold(bw, cfg, ctx, feats)
    return ctx


def block_commit(bw: BlockWeights64, cfg, ctx: BlockContext, rows: np.ndarray,
                 n: int) -> BlockContext:
    """The first n accepted rows appended in order; rows >= n never read."""
    out = ctx.clone()
    if n > 0:
        _fold(bw, cfg, out, rows[:n])
    return out


def block_draft(bw: BlockWeights64, cfg, ctx: BlockContext, X: np.ndarray) -> np.ndarray:
    """One drafter block on the slot rows X [S, D] (read-only on ctx)."""
    lw = bw.layer
    S = X.shape[0]
    a = rms_norm(X, bw.g_mix)
    slot_pos = ctx.pos + np.arange(S)
    Q = rope((a @ lw.w_q).reshape(S, cfg.n_q_heads, cfg.head_dim), slot_pos)
    Ks = rope((a @ lw.w_k).reshape(S, cfg.n_kv_heads, cfg.head_dim), slot_pos)
    Vs = (a @ lw.w_v).reshape(S, cfg.n_kv_heads, cfg.head_dim)
    O_att = O.window_block_attention(cfg, ctx, Q, Ks, Vs)
    xs = (a @ lw.w_x).reshape(S, cfg.ssm_heads, cfg.ssm_headdim)
    y = O.ssm_read(ctx.h, a @ lw.w_C) + bw.d_skip[None, :, None] * xs       # B4
    y = y.reshape(S, -1) * silu(a @ bw.w_z)
    X1 = X + O_att.reshape(S, -1) @ lw.w_o + y @ lw.w_mo
    n = rms_norm(X1, bw.g_mlp)
    return X1 + (silu(n @ bw.w_gate) * (n @ bw.w_up)) @ bw.w_down          # B5


def head(hw: HeadWeights64, X: np.ndarray):
    """B6: logits [S, V] and the argmax token of every slot (lowest id on ties)."""
    logits = rms_norm(X, hw.g_final) @ hw.w_lm
    return logits, np.argmax(logits, axis=-1)


class OracleBlockDrafter:
    """Requests x blocks of contexts plus the LM head, driven like a handle."""

    def __init__(self, cfg, block_weights: Sequence, head_weights, max_batch: int):
        self.cfg = cfg
        self.blocks: List[BlockWeights64] = [BlockWeights64.from_any(w) for w in block_weights]
        self.head = HeadWeights64.from_any(head_weights)
        self.ctx = [[BlockContext.empty(cfg) for _ in self.blocks] for _ in range(max_batch)]

    def prefill(self, lens: Sequence[int], feats_packed, requests: Optional[Sequence[int]] = None):
        f = O.to64(feats_packed)
        reqs = list(range(len(lens))) if requests is None else list(requests)
        off = 0
        for b, L in zip(reqs, lens):
            self.ctx[b] = [block_prefill(bw, self.cfg, f[off:off + L]) for bw in self.blocks]
            off += L

    def commit(self, feats, n_accepted):
        f = O.to64(feats)
        limit = self.cfg.block + 1
        for b, nb in enumerate(int(v) for v in np.asarray(n_accepted).reshape(-1)):
            nb = nb if 0 <= nb <= limit else 0
            self.ctx[b] = [block_commit(bw, self.cfg, c, f[b], nb)
                           for bw, c in zip(self.blocks, self.ctx[b])]

    def draft(self, slot_emb):
        """Hidden states of the last block [B, S, D] and the slots' tokens [B, S]."""
        X = O.to64(slot_emb)
        out = np.zeros_like(X)
        tokens = np.zeros(X.shape[:2], dtype=np.int64)
        for b in range(X.shape[0]):
            cur = X[b]
            for bw, c in zip(self.blocks, self.ctx[b]):
                cur = block_draft(bw, self.cfg, c, cur)
            out[b] = cur
            tokens[b] = head(self.head, cur)[1]
        return out, tokens
