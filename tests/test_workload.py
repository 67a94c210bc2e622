"""The seeded synthetic inputs both sides consume: their laws (the input
recipe the parity tests and the benchmark rely on), their determinism, and
the per-request streams that let a test regenerate a subset of requests."""
import math

import numpy as np
import torch

from workload import (CONFIGS, make_accepted, make_layer_weights, make_prefix_feats,
                      make_prefix_lens, make_round_inputs)

SERVING = CONFIGS["serving_qwen3_4b_b64"]


def test_serving_prefixes_log_uniform_2k_32k():
    lens = make_prefix_lens(SERVING)
    assert len(lens) == SERVING.batch == 64
    assert lens == make_prefix_lens(SERVING)  # seeded
    assert lens != make_prefix_lens(SERVING, seed=1)
    assert all(2048 <= L <= 32768 for L in lens)
    # log-uniform: log L uniform on [log 2K, log 32K]; the median sits at the
    # geometric mean (8K) and each quarter of the log range holds ~1/4
    many = make_prefix_lens(SERVING.replace(batch=8000))
    logs = np.log(np.array(many, dtype=np.float64))
    lo, hi = math.log(2048), math.log(32768)
    assert abs(float(np.median(many)) / 8192 - 1) < 0.05
    counts, _ = np.histogram(logs, bins=4, range=(lo, hi))
    assert np.all(np.abs(counts / len(many) - 0.25) < 0.03)


def test_fixed_prefix_configs():
    c1 = CONFIGS["qwen3_4b_bf16"]
    assert make_prefix_lens(c1) == [c1.prefix] * c1.batch


def test_accepted_counts_uniform_1_to_8():
    n = torch.cat([make_accepted(SERVING, r) for r in range(50)])
    assert n.dtype == torch.int32
    assert int(n.min()) == 1 and int(n.max()) == SERVING.block + 1 == 8
    counts = torch.bincount(n.long(), minlength=9)[1:].double() / n.numel()
    assert torch.all((counts - 1 / 8).abs() < 0.02)
    assert torch.equal(make_accepted(SERVING, 3), make_accepted(SERVING, 3))


def test_round_inputs_shapes_and_model_dtype():
    slot, feats = make_round_inputs(SERVING, 0)
    assert slot.shape == (64, 7, 2560) and feats.shape == (64, 8, 2560)
    assert slot.dtype == torch.bfloat16 and feats.dtype == torch.bfloat16
    tiny = CONFIGS["tiny_fp32"]
    s32, f32 = make_round_inputs(tiny, 0, 3)
    assert s32.dtype == torch.float32 and f32.shape == (3, 8, tiny.d_model)
    # different rounds draw different inputs, the same round the same ones
    assert not torch.equal(slot, make_round_inputs(SERVING, 1)[0])
    assert torch.equal(slot, make_round_inputs(SERVING, 0)[0])
    # ~N(0,1) before the rounding
    x = slot.double()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1) < 0.01


def test_prefix_features_regenerate_per_request():
    cfg = CONFIGS["tiny_fp32"]
    lens = [5, 0, 9, 4]
    full = make_prefix_feats(cfg, lens)
    assert full.shape == (sum(lens), cfg.d_model)
    # requests 2..3 drawn on their own equal their rows of the whole batch
    part = make_prefix_feats(cfg, lens[2:], request_offset=2)
    assert torch.equal(part, full[5:])
    assert make_prefix_feats(cfg, []).shape == (0, cfg.d_model)


def test_layer_weight_laws():
    cfg = CONFIGS["qwen3_4b_bf16"]
    w = make_layer_weights(cfg, 0)
    D = cfg.d_model
    for name in ("w_q", "w_k", "w_v", "w_o", "w_x", "w_mo"):
        assert abs(float(getattr(w, name).double().std()) / 0.02 - 1) < 0.02, name
    for name in ("w_B", "w_C"):
        assert abs(float(getattr(w, name).double().std()) * 16 * math.sqrt(D) - 1) < 0.05, name
    assert abs(float(w.w_dt.double().std()) * math.sqrt(D) - 1) < 0.05
    assert torch.all(w.dt_bias == -2.0)
    assert float(w.A_log.min()) >= 0.0 and float(w.A_log.max()) < 1.0
    assert w.w_q.dtype == torch.bfloat16 and w.A_log.dtype == torch.float32
    # layers and seeds draw different weights; the same key the same ones
    assert not torch.equal(w.w_q, make_layer_weights(cfg, 1).w_q)
    assert torch.equal(w.w_q, make_layer_weights(cfg, 0).w_q)
