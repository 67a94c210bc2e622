"""HyFlash drafter layer, stated plainly in float64 NumPy -- TEST INFRASTRUCTURE.

Only tests, the smoke check and the benchmark's CPU arms use this module. It
is deliberately slow and literal; it shares nothing with the CUDA library.

What one drafter layer computes (sources):
  * "HyFlash: A Prefix-Memory Prior for On-Device Speculative Decoding",
    abstract: local attention captures recent context and draft-position
    interactions, recurrent memory compresses historical target features into
    fixed-size states; parallel block drafting predicts several positions in
    one pass.
  * learnaivisually explainer "HyFlash lifts on-device speculative decoding
    16.2%", paragraph "That is HyFlash": every layer has two branches; local
    attention sees the last committed target features and all seven draft
    positions in both directions; a Mamba-2 branch holds the compressed
    committed history and is only queried during drafting; after verification
    only newly committed features update the state.
  * same page, Jargon "Recurrent memory (Mamba-2)" and "Sliding-window
    attention"; FAQ "Why does the memory update only from committed features?".
  * Mamba-2 recurrence as stated with the workloads:
        h_t = exp(dt_t * A) * h_{t-1} + dt_t * x_t (outer) B_t,   y = C . h,
    dt = softplus(.), A = -exp(A_log) (learned negative decay).

Readings where the pages are silent (each is also listed in the design notes):
  R1 the layer output is out = X + O W_o + y W_mo: the two branches are summed
     into the residual; no norm, RoPE, MLP, conv1d, z-gate or D-skip;
  R2 the memory query at draft time is C_s = X_s W_C;
  R3 window K/V and memory inputs (x, B, dt) are projections of the committed
     target features by the layer's own weights; slot K/V use the same W_k/W_v;
  R4 one SSM group (B, C shared by all heads); softmax scale 1/sqrt(head_dim);
     each slot also attends to its own key; GQA maps query head h to KV head
     h // (Hq/Hkv);
  R5 ring slot of committed position t is t mod W; pos counts committed tokens;
     when pos < W the valid slots are 0..pos-1; pos = 0 means slots only;
  R6 commit applies accepted rows t = 0..n-1 in order, ignores rows >= n;
     n = 0 is a no-op; n outside 0..block+1 is an error and the request is
     left unchanged;
  R7 softplus(x) = max(x,0) + log1p(exp(-|x|)) (no threshold cut-off);
  R8 bf16 mode: float64 arithmetic on the bf16-rounded inputs and weights, no
     emulation of intermediate rounding.

Ablation modes (the paper's intervention table "Recurrent history" /
"Intra-block interactions", and the explainer's paragraph on the ablations),
off by default, selected by two fields of the shape:
  R9  cross_slot = False ("Cross-slot off"): attention among the draft slots
      is switched off -- slot s attends to the window entries and to its own
      key only; the other slots' keys are masked;
  R10 mem_horizon = M > 0 ("SSM: Last 512" with M = 512, "SSM: Last feature"
      with M = 1): the recurrent history is restricted to the last M
      committed features -- the memory is the fold from h = 0 over the last
      min(pos, M) committed features, whatever came before them. M = 0 keeps
      the whole history.

Gated-delta memory (the paper's memory-swap table "Mamba-2 / GDN-2", and the
explainer's last paragraph: swapping Mamba-2 for Gated DeltaNet-2 gives
comparable results). The pages do not define the variant; the gated delta
rule is taken from its published paper (Yang, Kautz, Hatamizadeh, "Gated
Delta Networks: Improving Mamba2 with Delta Rule"):
      S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T,
      o = S q,
with S [P x N] per head (value x key). Readings:
  R11 memory = "gdn": k_t = B_t / |B_t| (one group: shared by the heads),
      v_t = x_t (the head's P values), alpha_t = exp(dt_t A) with dt and A
      exactly as in the Mamba-2 memory (the paper's gate has this form),
      beta_t = sigmoid(f_t W_beta) per head (a new projection), and the read
      uses q = C_s / |C_s|; no memory horizon with this kind. Prefill is the
      same rule applied token by token (committing the whole prefix).

4-bit weights (the paper's INT4 / GPTQ table: the 4-bit drafter keeps
99.2% of the bf16 acceptance; explainer, "Where it earns its keep"):
  R12 a 4-bit matrix of shape [in, out] holds codes q in 0..15 and, per
      group of 128 consecutive inputs and per output, a scale s and a zero
      point z (GPTQ's asymmetric group format); its value is
      w[i, o] = s[i // 128, o] * (q[i, o] - z[i // 128, o]). How the codes
      were chosen (GPTQ's error-compensating rounding) is outside the hot
      path: the layer computes with these values.

Parity pins (tests/test_oracle_pins.py): the chunked fold equals the
token-by-token recurrence and the unrolled product closed form; constant decay
matches scipy.signal.lfilter; A = 0 gives the plain sum, huge decay keeps only
the last term, dt = 0 and n = 0 leave the state unchanged; attention matches
torch's scaled_dot_product_attention when the window covers the prefix; all
keys equal gives the mean of V; rejected rows never matter; splitting a commit
equals one commit; ring slots match a brute-force list of the last W tokens;
softplus matches closed values and torch; context sizing matches the pages'
printed byte figures (tests/golden/sizing.json); a prefill, two commits and a
draft on tiny shapes equal a recomputation from the definitions in scalar
loops. No function here is "parity unpinned"; the layer's full output values
have no printed worked example, so they are pinned by that brute force and
through the pieces above.
"""
from __future__ import annotations

import copy
import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

# --------------------------------------------------------------------------
# helpers


def to64(a) -> np.ndarray:
    """float64 copy of a NumPy array or a torch tensor (bf16 included)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if hasattr(a, "double"):
            a = a.double()
        return a.numpy().astype(np.float64, copy=True)
    return np.asarray(a, dtype=np.float64).copy()


def softplus(x):
    """Stable softplus, R7: max(x,0) + log1p(exp(-|x|))."""
    x = np.asarray(x, dtype=np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


@dataclasses.dataclass
class Weights64:
    w_q: np.ndarray
    w_k: np.ndarray
    w_v: np.ndarray
    w_o: np.ndarray
    w_x: np.ndarray
    w_B: np.ndarray
    w_C: np.ndarray
    w_dt: np.ndarray
    w_mo: np.ndarray
    dt_bias: np.ndarray
    A_log: np.ndarray
    w_beta: Optional[np.ndarray] = None   # gated-delta memory only

    @staticmethod
    def from_any(w) -> "Weights64":
        names = [f.name for f in dataclasses.fields(Weights64)]
        vals = {n: getattr(w, n, None) for n in names}
        return Weights64(**{n: (None if v is None else
                                (dequantize_q4(v) if hasattr(v, "codes") else to64(v)))
                            for n, v in vals.items()})

    @property
    def A(self) -> np.ndarray:
        """Learned negative decay A = -exp(A_log), one scalar per SSM head."""
        return -np.exp(self.A_log)


def dequantize_q4(m) -> np.ndarray:
    """R12: w[i, o] = s[i // 128, o] * (q[i, o] - z[i // 128, o]), float64."""
    q = to64(m.codes)
    s = to64(m.scales)
    z = to64(m.zeros)
    g = np.arange(q.shape[0]) // 128
    return s[g, :] * (q - z[g, :])


# --------------------------------------------------------------------------
# Mamba-2 memory (commit-only writer, draft-time reader)


def ssm_inputs(lw: Weights64, cfg, feats: np.ndarray):
    """x [T,Hm,P], B [T,N], dt [T,Hm] from committed features [T,D] (R3)."""
    T = feats.shape[0]
    x = (feats @ lw.w_x).reshape(T, cfg.ssm_heads, cfg.ssm_headdim)
    B = feats @ lw.w_B
    dt = softplus(feats @ lw.w_dt + lw.dt_bias[None, :])
    return x, B, dt


def ssm_fold_recurrent(h: np.ndarray, x, B, dt, A) -> np.ndarray:
    """Token by token: h <- exp(dt_t A) h + dt_t x_t (outer) B_t, t in order."""
    h = np.array(h, dtype=np.float64, copy=True)
    for t in range(x.shape[0]):
        decay = np.exp(dt[t] * A)                          # [Hm]
        inc = (dt[t][:, None] * x[t])[:, :, None] * B[t][None, None, :]
        h = decay[:, None, None] * h + inc
    return h


def ssm_fold_chunked(h: np.ndarray, x, B, dt, A, chunk: int) -> np.ndarray:
    """The same fold in chunks of ``chunk`` tokens (state passing between chunks).

    Inside a chunk the contribution of token t to the chunk-end state is
    dt_t * exp(sum_{s>t, s in chunk} dt_s A) * x_t (outer) B_t; the state that
    enters the chunk decays by exp(sum_{s in chunk} dt_s A). The suffix sums are
    taken directly (never as a difference of prefix sums).
    """
    h = np.array(h, dtype=np.float64, copy=True)
    T = x.shape[0]
    Hm, P = x.shape[1], x.shape[2]
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        a = dt[c0:c1] * A[None, :]                         # [Q,Hm]
        incl = np.cumsum(a[::-1], axis=0)[::-1]            # sum_{s>=t}
        after = np.concatenate([incl[1:], np.zeros((1, Hm))], axis=0)
        w = dt[c0:c1] * np.exp(after)                      # [Q,Hm]
        wx = (w[:, :, None] * x[c0:c1]).reshape(c1 - c0, Hm * P)
        S = (wx.T @ B[c0:c1]).reshape(Hm, P, -1)
        h = np.exp(incl[0])[:, None, None] * h + S
    return h


def ssm_read(h: np.ndarray, C: np.ndarray) -> np.ndarray:
    """y[s, hd, p] = sum_n h[hd, p, n] C[s, n] (draft-time read, state untouched)."""
    return np.einsum("hpn,sn->shp", h, C)


# --------------------------------------------------------------------------
# gated-delta memory (R11)


def memory_kind(cfg) -> str:
    return str(getattr(cfg, "memory", "mamba2") or "mamba2")


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def gdn_inputs(lw: Weights64, cfg, feats: np.ndarray):
    """v = x [T,Hm,P], unit keys k [T,N], alpha [T,Hm], beta [T,Hm] (R11)."""
    x, B, dt = ssm_inputs(lw, cfg, feats)
    k = B / np.linalg.norm(B, axis=1, keepdims=True)
    alpha = np.exp(dt * lw.A[None, :])
    beta = sigmoid(feats @ lw.w_beta)
    return x, k, alpha, beta


def gdn_fold_recurrent(S: np.ndarray, v, k, alpha, beta) -> np.ndarray:
    """Token by token, per head: S <- S (alpha (I - beta k k^T)) + beta v k^T."""
    S = np.array(S, dtype=np.float64, copy=True)
    N = S.shape[2]
    eye = np.eye(N)
    for t in range(v.shape[0]):
        kk = np.outer(k[t], k[t])                                   # k k^T
        trans = alpha[t][:, None, None] * (eye[None] - beta[t][:, None, None] * kk[None])
        S = S @ trans + beta[t][:, None, None] * (v[t][:, :, None] * k[t][None, None, :])
    return S


def gdn_read(S: np.ndarray, C: np.ndarray) -> np.ndarray:
    """y[s, hd, p] = (S_hd q_s)[p] with q_s = C_s / |C_s| (R11)."""
    q = C / np.linalg.norm(C, axis=1, keepdims=True)
    return np.einsum("hpn,sn->shp", S, q)


# --------------------------------------------------------------------------
# per-request, per-layer context: window ring + recurrent state


@dataclasses.dataclass
class Context:
    ring_k: np.ndarray   # [Hkv, W, dh]
    ring_v: np.ndarray   # [Hkv, W, dh]
    tag: np.ndarray      # [W] committed position held by each slot, -1 if empty
    pos: int             # committed tokens so far
    h: np.ndarray        # [Hm, P, N]
    hist: Optional[tuple] = None  # R10: (x, B, dt) of the last M committed features

    @staticmethod
    def empty(cfg) -> "Context":
        return Context(
            ring_k=np.zeros((cfg.n_kv_heads, cfg.window, cfg.head_dim)),
            ring_v=np.zeros((cfg.n_kv_heads, cfg.window, cfg.head_dim)),
            tag=np.full((cfg.window,), -1, dtype=np.int64),
            pos=0,
            h=np.zeros((cfg.ssm_heads, cfg.ssm_headdim, cfg.d_state)))

    def clone(self) -> "Context":
        return copy.deepcopy(self)


def mem_horizon(cfg) -> int:
    """R10: 0 = whole history, M > 0 = the last M committed features."""
    return int(getattr(cfg, "mem_horizon", 0) or 0)


def cross_slot(cfg) -> bool:
    """R9: False masks slot-to-slot attention (each slot keeps its own key)."""
    return bool(getattr(cfg, "cross_slot", True))


def ring_slot(position: int, window: int) -> int:
    """R5: committed position t lives in slot t mod W."""
    return position % window


def ring_append(ctx: Context, cfg, k: np.ndarray, v: np.ndarray, first_pos: int):
    """Write K/V rows [n, Hkv, dh] for committed positions first_pos.. ."""
    for t in range(k.shape[0]):
        s = ring_slot(first_pos + t, cfg.window)
        ctx.ring_k[:, s, :] = k[t]
        ctx.ring_v[:, s, :] = v[t]
        ctx.tag[s] = first_pos + t


def kv_of(lw: Weights64, cfg, feats: np.ndarray):
    T = feats.shape[0]
    k = (feats @ lw.w_k).reshape(T, cfg.n_kv_heads, cfg.head_dim)
    v = (feats @ lw.w_v).reshape(T, cfg.n_kv_heads, cfg.head_dim)
    return k, v


def prefill_layer(lw: Weights64, cfg, feats: np.ndarray,
                  method: str = "chunked", chunk: Optional[int] = None) -> Context:
    """Fold a whole committed prefix [L, D] into a fresh context.

    Equivalent to committing all L features at once: the state is the fold
    from h = 0 and the ring holds the last min(L, W) features' K/V.
    """
    ctx = Context.empty(cfg)
    L = feats.shape[0]
    if L == 0:
        return ctx
    if memory_kind(cfg) == "gdn":  # R11: the delta rule over the whole prefix
        ctx.h = gdn_fold_recurrent(ctx.h, *gdn_inputs(lw, cfg, feats))
        first = max(0, L - cfg.window)
        k, v = kv_of(lw, cfg, feats[first:])
        ring_append(ctx, cfg, k, v, first)
        ctx.pos = L
        return ctx
    x, B, dt = ssm_inputs(lw, cfg, feats)
    M = mem_horizon(cfg)
    if M > 0:  # R10: only the last M features are remembered
        x, B, dt = x[-M:], B[-M:], dt[-M:]
        ctx.hist = (x, B, dt)
    if method == "recurrent":
        ctx.h = ssm_fold_recurrent(ctx.h, x, B, dt, lw.A)
    else:
        ctx.h = ssm_fold_chunked(ctx.h, x, B, dt, lw.A, chunk or cfg.chunk)
    first = max(0, L - cfg.window)
    k, v = kv_of(lw, cfg, feats[first:])
    ring_append(ctx, cfg, k, v, first)
    ctx.pos = L
    return ctx


def commit_layer(lw: Weights64, cfg, ctx: Context, feats_rows: np.ndarray,
                 n: int) -> Context:
    """Append the first n accepted rows (R6); rows >= n are never read."""
    out = ctx.clone()
    if n <= 0:
        return out
    f = feats_rows[:n]
    k, v = kv_of(lw, cfg, f)
    ring_append(out, cfg, k, v, out.pos)
    if memory_kind(cfg) == "gdn":  # R11
        out.h = gdn_fold_recurrent(out.h, *gdn_inputs(lw, cfg, f))
        out.pos += n
        return out
    x, B, dt = ssm_inputs(lw, cfg, f)
    M = mem_horizon(cfg)
    if M > 0:
        # R10: keep the last M committed features and fold them afresh
        if out.hist is not None:
            x = np.concatenate([out.hist[0], x])
            B = np.concatenate([out.hist[1], B])
            dt = np.concatenate([out.hist[2], dt])
        out.hist = (x[-M:], B[-M:], dt[-M:])
        out.h = ssm_fold_recurrent(np.zeros_like(out.h), *out.hist, lw.A)
    else:
        out.h = ssm_fold_recurrent(out.h, x, B, dt, lw.A)
    out.pos += n
    return out


# --------------------------------------------------------------------------
# drafting (read-only on the context)


def softmax_rows(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def window_block_attention(cfg, ctx: Context, Q, Ks, Vs) -> np.ndarray:
    """Bidirectional attention of the slot queries over the valid window
    entries plus all slot keys (R4, R5); with cross_slot off (R9) slot s sees
    the window and its own key only. Q [S,Hq,dh], Ks/Vs [S,Hkv,dh]."""
    S = Q.shape[0]
    G = cfg.n_q_heads // cfg.n_kv_heads
    valid = np.nonzero(ctx.tag >= 0)[0]
    O = np.zeros((S, cfg.n_q_heads, cfg.head_dim))
    scale = 1.0 / math.sqrt(cfg.head_dim)
    for hq in range(cfg.n_q_heads):
        g = hq // G
        keys = np.concatenate([ctx.ring_k[g, valid, :], Ks[:, g, :]], axis=0)
        vals = np.concatenate([ctx.ring_v[g, valid, :], Vs[:, g, :]], axis=0)
        scores = (Q[:, hq, :] @ keys.T) * scale
        if not cross_slot(cfg):
            slot_part = scores[:, len(valid):]
            slot_part[~np.eye(S, dtype=bool)] = -np.inf
        p = softmax_rows(scores)
        O[:, hq, :] = p @ vals
    return O


def draft_layer(lw: Weights64, cfg, ctx: Context, X: np.ndarray,
                return_parts: bool = False):
    """One drafter layer for one request; X [S, D] -> out [S, D] (R1, R2)."""
    S = X.shape[0]
    Q = (X @ lw.w_q).reshape(S, cfg.n_q_heads, cfg.head_dim)
    Ks = (X @ lw.w_k).reshape(S, cfg.n_kv_heads, cfg.head_dim)
    Vs = (X @ lw.w_v).reshape(S, cfg.n_kv_heads, cfg.head_dim)
    Cs = X @ lw.w_C
    O = window_block_attention(cfg, ctx, Q, Ks, Vs)
    y = gdn_read(ctx.h, Cs) if memory_kind(cfg) == "gdn" else ssm_read(ctx.h, Cs)
    out = X + O.reshape(S, -1) @ lw.w_o + y.reshape(S, -1) @ lw.w_mo
    if return_parts:
        return out, dict(Q=Q, Ks=Ks, Vs=Vs, Cs=Cs, O=O, y=y)
    return out


# --------------------------------------------------------------------------
# batched drafter over requests and layers


class OracleDrafter:
    """Requests x layers of contexts, driven like the library's handle."""

    def __init__(self, cfg, layer_weights: Sequence, max_batch: int):
        self.cfg = cfg
        self.layers: List[Weights64] = [Weights64.from_any(w) for w in layer_weights]
        self.ctx = [[Context.empty(cfg) for _ in self.layers] for _ in range(max_batch)]
        self.last_offsets = np.zeros((max_batch + 1,), dtype=np.int64)

    def prefill(self, lens: Sequence[int], feats_packed, method: str = "chunked",
                requests: Optional[Sequence[int]] = None):
        f = to64(feats_packed)
        reqs = list(range(len(lens))) if requests is None else list(requests)
        off = 0
        for b, L in zip(reqs, lens):
            seg = f[off:off + L]
            off += L
            self.ctx[b] = [prefill_layer(lw, self.cfg, seg, method) for lw in self.layers]

    def commit(self, feats, n_accepted):
        """feats [B, block+1, D], n [B]; returns (offsets [B+1], error flag)."""
        f = to64(feats)
        n = [int(v) for v in np.asarray(n_accepted).reshape(-1)]
        B = len(n)
        limit = self.cfg.block + 1
        offs = np.zeros((B + 1,), dtype=np.int64)
        err = False
        for b in range(B):
            nb = n[b]
            if nb < 0 or nb > limit:
                err = True
                nb = 0
            offs[b + 1] = offs[b] + nb
            self.ctx[b] = [commit_layer(lw, self.cfg, c, f[b], nb)
                           for lw, c in zip(self.layers, self.ctx[b])]
        self.last_offsets = offs
        return offs, err

    def draft(self, slot_emb) -> np.ndarray:
        X = to64(slot_emb)
        out = np.zeros_like(X)
        for b in range(X.shape[0]):
            cur = X[b]
            for lw, c in zip(self.layers, self.ctx[b]):
                cur = draft_layer(lw, self.cfg, c, cur)
            out[b] = cur
        return out


# --------------------------------------------------------------------------
# sizing (pinned against the pages' printed byte figures)


def window_kv_bytes(n_layers, n_kv_heads, head_dim, window, elem_bytes) -> int:
    """Local K and V of the window: layers x 2 x Hkv x dh x W x bytes."""
    return n_layers * 2 * n_kv_heads * head_dim * window * elem_bytes


def state_bytes(n_layers, d_inner, d_state, elem_bytes=4) -> int:
    """Recurrent state: layers x d_inner x d_state x bytes (fp32 state)."""
    return n_layers * d_inner * d_state * elem_bytes


def target_kv_bytes(n_layers, n_kv_heads, head_dim, seq, elem_bytes) -> int:
    """A full-attention KV cache of ``seq`` tokens (same formula, W = seq)."""
    return window_kv_bytes(n_layers, n_kv_heads, head_dim, seq, elem_bytes)
