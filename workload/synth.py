"""Synthetic workloads shaped like the HyFlash drafter configurations.

Sources for the shapes and laws (HyFlash: A Prefix-Memory Prior for On-Device
Speculative Decoding, and the learnaivisually explainer of it, "That is
HyFlash" and "Where it earns its keep" sections):
  * one drafter layer = local attention over the most recent committed target
    features plus the 7 draft slots, and a Mamba-2 recurrent memory;
  * block of 7 draft positions; accepted counts per round 1..8 (7 drafts plus
    the target's bonus token).

Distributions (stated with the workloads): features and slot embeddings
~N(0,1); projection weights ~N(0, 0.02); dt = softplus(N(0,1) - 2) obtained
through W_dt with std 1/sqrt(D) and dt_bias = -2; A = -exp(U(0,1)) through
A_log ~ U(0,1); B, C ~ N(0, 1/16) (1/16 read as a standard deviation) through
W_B, W_C with std (1/16)/sqrt(D).

Everything is drawn with torch's CPU generator so that the exact same bytes can
be handed to the GPU path and to the oracle. bf16 configurations round once
to bfloat16 here; both sides then consume those rounded values.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class DrafterShape:
    name: str
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    window: int
    block: int
    ssm_heads: int
    ssm_headdim: int
    d_state: int
    n_layers: int
    batch: int
    prefix: int            # prefix length for batch configs with a single length
    rounds: int
    dtype: str             # "f32" or "bf16"
    chunk: int = 128
    n_groups: int = 1
    prefix_lo: int = 0     # log-uniform prefix range (serving batch)
    prefix_hi: int = 0
    # ablation modes (off by default): slot-to-slot attention masked; memory
    # restricted to the last mem_horizon committed features (0: all of them)
    cross_slot: bool = True
    mem_horizon: int = 0
    # memory kind: "mamba2" (the pages' memory) or "gdn" (gated delta rule,
    # the paper's Gated DeltaNet-2 swap)
    memory: str = "mamba2"
    # weight precision: 16 (model dtype) or 4 (4-bit codes, group 128)
    weight_bits: int = 16
    # full drafter block around the layer (on/off, MLP width, LM-head vocabulary)
    mlp_dim: int = 0
    vocab: int = 0
    full_block: bool = False

    @property
    def d_inner(self) -> int:
        return self.ssm_heads * self.ssm_headdim

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "DrafterShape":
        return dataclasses.replace(self, **kw)


# The five workloads, in the order they are listed with the baseline metric.
CONFIGS = {
    "tiny_fp32": DrafterShape(
        name="tiny_fp32", d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
        window=64, block=7, ssm_heads=4, ssm_headdim=64, d_state=16,
        n_layers=1, batch=1, prefix=512, rounds=20, dtype="f32"),
    "qwen3_4b_bf16": DrafterShape(
        name="qwen3_4b_bf16", d_model=2560, n_q_heads=32, n_kv_heads=8,
        head_dim=128, window=512, block=7, ssm_heads=80, ssm_headdim=64,
        d_state=128, n_layers=1, batch=1, prefix=8192, rounds=200,
        dtype="bf16"),
    "phi4_bf16": DrafterShape(
        name="phi4_bf16", d_model=5120, n_q_heads=40, n_kv_heads=10,
        head_dim=128, window=512, block=7, ssm_heads=160, ssm_headdim=64,
        d_state=128, n_layers=1, batch=1, prefix=32768, rounds=200,
        dtype="bf16"),
    "serving_qwen3_4b_b64": DrafterShape(
        name="serving_qwen3_4b_b64", d_model=2560, n_q_heads=32, n_kv_heads=8,
        head_dim=128, window=512, block=7, ssm_heads=80, ssm_headdim=64,
        d_state=128, n_layers=3, batch=64, prefix=0, rounds=500,
        dtype="bf16", prefix_lo=2048, prefix_hi=32768),
    "prefill_phi4_sweep": DrafterShape(
        name="prefill_phi4_sweep", d_model=5120, n_q_heads=40, n_kv_heads=10,
        head_dim=128, window=512, block=7, ssm_heads=160, ssm_headdim=64,
        d_state=128, n_layers=1, batch=8, prefix=4096, rounds=0,
        dtype="bf16", chunk=128),
}
CONFIG_ORDER = list(CONFIGS)


def rng(*key) -> torch.Generator:
    """A CPU generator seeded from a stable hash of ``key``."""
    h = hashlib.sha256(repr(key).encode()).digest()
    return torch.Generator().manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))


def _round(t: torch.Tensor, cfg: DrafterShape) -> torch.Tensor:
    return t.to(cfg.torch_dtype).contiguous()


@dataclasses.dataclass
class LayerWeightsT:
    """Per-layer weights, row-major [in, out]; dt_bias and A_log stay fp32."""
    w_q: torch.Tensor
    w_k: torch.Tensor
    w_v: torch.Tensor
    w_o: torch.Tensor
    w_x: torch.Tensor
    w_B: torch.Tensor
    w_C: torch.Tensor
    w_dt: torch.Tensor
    w_mo: torch.Tensor
    dt_bias: torch.Tensor
    A_log: torch.Tensor
    w_beta: torch.Tensor = None   # gated-delta memory only: writing strength projection [D, Hm]

    FIELDS = ("w_q", "w_k", "w_v", "w_o", "w_x", "w_B", "w_C", "w_dt", "w_mo",
              "dt_bias", "A_log", "w_beta")


def make_layer_weights(cfg: DrafterShape, layer: int, seed: int = 0) -> LayerWeightsT:
    g = rng("weights", cfg.name, seed, layer)
    D, hq, hkv, dh = cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    din, N, Hm = cfg.d_inner, cfg.d_state, cfg.ssm_heads

    def n(shape, std):
        return _round(torch.randn(shape, generator=g) * std, cfg)

    return LayerWeightsT(
        w_q=n((D, hq * dh), 0.02),
        w_k=n((D, hkv * dh), 0.02),
        w_v=n((D, hkv * dh), 0.02),
        w_o=n((hq * dh, D), 0.02),
        w_x=n((D, din), 0.02),
        w_B=n((D, N), (1.0 / 16.0) / math.sqrt(D)),
        w_C=n((D, N), (1.0 / 16.0) / math.sqrt(D)),
        w_dt=n((D, Hm), 1.0 / math.sqrt(D)),
        w_mo=n((din, D), 0.02),
        dt_bias=torch.full((Hm,), -2.0, dtype=torch.float32),
        A_log=torch.rand((Hm,), generator=g, dtype=torch.float32),
        w_beta=n((D, Hm), 1.0 / math.sqrt(D)),   # drawn last: earlier draws unchanged
    )


@dataclasses.dataclass
class Q4Matrix:
    """A 4-bit weight of shape [in, out]: codes uint8 [in, out] in 0..15,
    scales bf16 [in/128, out], zeros uint8 [in/128, out] in 0..15."""
    codes: torch.Tensor
    scales: torch.Tensor
    zeros: torch.Tensor


@dataclasses.dataclass
class LayerWeightsQ4:
    """Per-layer 4-bit weights (the matrices of LayerWeightsT as Q4Matrix);
    dt_bias and A_log fp32."""
    w_q: Q4Matrix
    w_k: Q4Matrix
    w_v: Q4Matrix
    w_o: Q4Matrix
    w_x: Q4Matrix
    w_B: Q4Matrix
    w_C: Q4Matrix
    w_dt: Q4Matrix
    w_mo: Q4Matrix
    dt_bias: torch.Tensor
    A_log: torch.Tensor
    w_beta: Q4Matrix = None

    MATRICES = ("w_q", "w_k", "w_v", "w_o", "w_x", "w_B", "w_C", "w_dt", "w_mo", "w_beta")


def make_layer_weights_q4(cfg: DrafterShape, layer: int, seed: int = 0) -> LayerWeightsQ4:
    """Random 4-bit weights with the same spread as the bf16 ones: codes
    uniform in 0..15, zero points 7 or 8, and per (group of 128 inputs,
    output) a scale drawn around std / 4.6 (the std of code - zero), rounded
    to bf16."""
    g = rng("weights_q4", cfg.name, seed, layer)
    D, hq, hkv, dh = cfg.d_model, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    din, N, Hm = cfg.d_inner, cfg.d_state, cfg.ssm_heads

    def m(shape, std):
        i, o = shape
        codes = torch.randint(0, 16, (i, o), generator=g, dtype=torch.uint8)
        zeros = torch.randint(7, 9, (i // 128, o), generator=g, dtype=torch.uint8)
        scales = (torch.rand((i // 128, o), generator=g) * 0.4 + 0.8) * (std / 4.6)
        return Q4Matrix(codes, scales.to(torch.bfloat16).contiguous(), zeros)

    return LayerWeightsQ4(
        w_q=m((D, hq * dh), 0.02),
        w_k=m((D, hkv * dh), 0.02),
        w_v=m((D, hkv * dh), 0.02),
        w_o=m((hq * dh, D), 0.02),
        w_x=m((D, din), 0.02),
        w_B=m((D, N), (1.0 / 16.0) / math.sqrt(D)),
        w_C=m((D, N), (1.0 / 16.0) / math.sqrt(D)),
        w_dt=m((D, Hm), 1.0 / math.sqrt(D)),
        w_mo=m((din, D), 0.02),
        dt_bias=torch.full((Hm,), -2.0, dtype=torch.float32),
        A_log=torch.rand((Hm,), generator=g, dtype=torch.float32),
        w_beta=m((D, Hm), 1.0 / math.sqrt(D)),
    )


@dataclasses.dataclass
class BlockWeightsT:
    """One full drafter block: the layer's weights plus the norms' gains, the
    memory's gate / skip / convolution and the MLP ([in, out] row-major)."""
    layer: LayerWeightsT
    g_mix: torch.Tensor
    g_mlp: torch.Tensor
    w_z: torch.Tensor
    d_skip: torch.Tensor
    conv_w: torch.Tensor
    conv_b: torch.Tensor
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor


@dataclasses.dataclass
class HeadWeightsT:
    g_final: torch.Tensor
    w_lm: torch.Tensor


def make_block_weights(cfg: DrafterShape, layer: int, seed: int = 0) -> BlockWeightsT:
    """The layer's weights (the same draws as make_layer_weights) and the
    block's extra parts: gains ~1 + N(0, 0.1), W_z and the MLP ~N(0, 0.02),
    D ~U(0, 1), conv taps ~N(0, 1/2) and bias ~N(0, 0.1) (conv width 4)."""
    g = rng("block", cfg.name, seed, layer)
    D, din, N, Hm, F = cfg.d_model, cfg.d_inner, cfg.d_state, cfg.ssm_heads, cfg.mlp_dim

    def n(shape, std):
        return _round(torch.randn(shape, generator=g) * std, cfg)

    def f32(t):
        return t.to(torch.float32).contiguous()

    return BlockWeightsT(
        layer=make_layer_weights(cfg, layer, seed),
        g_mix=f32(1.0 + 0.1 * torch.randn((D,), generator=g)),
        g_mlp=f32(1.0 + 0.1 * torch.randn((D,), generator=g)),
        w_z=n((D, din), 0.02),
        d_skip=f32(torch.rand((Hm,), generator=g)),
        conv_w=f32(torch.randn((din + N, 4), generator=g) * 0.5),
        conv_b=f32(torch.randn((din + N,), generator=g) * 0.1),
        w_gate=n((D, F), 0.02),
        w_up=n((D, F), 0.02),
        w_down=n((F, D), 0.02),
    )


def make_head_weights(cfg: DrafterShape, seed: int = 0) -> HeadWeightsT:
    g = rng("head", cfg.name, seed)
    return HeadWeightsT(
        g_final=(1.0 + 0.1 * torch.randn((cfg.d_model,), generator=g)).to(torch.float32),
        w_lm=_round(torch.randn((cfg.d_model, cfg.vocab), generator=g) * 0.02, cfg),
    )


def make_prefix_lens(cfg: DrafterShape, seed: int = 0) -> list:
    """Per-request prefix lengths: fixed, or log-uniform in [lo, hi]."""
    if cfg.prefix_lo:
        g = rng("lens", cfg.name, seed)
        u = torch.rand((cfg.batch,), generator=g, dtype=torch.float64)
        lo, hi = math.log(cfg.prefix_lo), math.log(cfg.prefix_hi)
        return [int(math.floor(math.exp(lo + (hi - lo) * float(x)))) for x in u]
    return [cfg.prefix] * cfg.batch


def make_prefix_feats(cfg: DrafterShape, lens: Sequence[int], seed: int = 0,
                      request_offset: int = 0) -> torch.Tensor:
    """Packed committed target features [sum(lens), D] ~ N(0,1).

    Each request draws from its own stream, so a subset of requests can be
    regenerated on its own (``request_offset`` names the first request).
    """
    parts = []
    for i, L in enumerate(lens):
        g = rng("prefix", cfg.name, seed, request_offset + i)
        parts.append(torch.randn((L, cfg.d_model), generator=g))
    if not parts:
        return torch.zeros((0, cfg.d_model), dtype=cfg.torch_dtype)
    return _round(torch.cat(parts, 0), cfg)


def make_round_inputs(cfg: DrafterShape, rnd: int, batch: Optional[int] = None,
                      seed: int = 0):
    """Slot embeddings [B, 7, D] and commit features [B, 8, D] for one round.

    All 8 commit rows are filled; rows at or beyond the accepted count stand for
    rejected drafts and must never influence anything.
    """
    B = cfg.batch if batch is None else batch
    g = rng("round", cfg.name, seed, rnd)
    slot = torch.randn((B, cfg.block, cfg.d_model), generator=g)
    feats = torch.randn((B, cfg.block + 1, cfg.d_model), generator=g)
    return _round(slot, cfg), _round(feats, cfg)


def make_attention_inputs(cfg: DrafterShape, batch: int, seed: int = 0):
    """Inputs of the window+block attention on its own: slot projections
    [batch*block, Hq*dh + 2*Hkv*dh] fp32 (queries | slot keys | slot values,
    ~N(0,1), the spread of the workloads' projections), window rings
    [batch, Hkv, W, dh] ~N(0,1) rounded once to the model dtype."""
    g = rng("attention", cfg.name, seed, batch, cfg.window, cfg.head_dim)
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    proj = torch.randn((batch * cfg.block, qd + 2 * kvd), generator=g)
    shape = (batch, cfg.n_kv_heads, cfg.window, cfg.head_dim)
    ring_k = _round(torch.randn(shape, generator=g), cfg)
    ring_v = _round(torch.randn(shape, generator=g), cfg)
    return proj, ring_k, ring_v


def make_accepted(cfg: DrafterShape, rnd: int, batch: Optional[int] = None,
                  seed: int = 0) -> torch.Tensor:
    """Accepted counts per request, uniform integers in 1..block+1 (int32)."""
    B = cfg.batch if batch is None else batch
    g = rng("accepted", cfg.name, seed, rnd)
    return torch.randint(1, cfg.block + 2, (B,), generator=g, dtype=torch.int32)


def make_ssm_core_inputs(T: int, Hm: int, P: int, N: int, seed: int = 0):
    """Direct SSM inputs with the workload laws: x ~ N(0,1), B ~ N(0,1/16),
    dt = softplus(N(0,1) - 2) drawn as its pre-activation, A_log ~ U(0,1).

    Returns (x [T,Hm,P], B [T,N], dt_raw [T,Hm], A_log [Hm]) as float64 tensors;
    the caller applies softplus (the method's arithmetic) itself.
    """
    g = rng("ssm_core", T, Hm, P, N, seed)
    x = torch.randn((T, Hm, P), generator=g, dtype=torch.float64)
    B = torch.randn((T, N), generator=g, dtype=torch.float64) / 16.0
    dt_raw = torch.randn((T, Hm), generator=g, dtype=torch.float64) - 2.0
    A_log = torch.rand((Hm,), generator=g, dtype=torch.float64)
    return x, B, dt_raw, A_log
