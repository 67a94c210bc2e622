"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package holds only shapes, seeds and random draws (plus the one rounding
to the model dtype that both sides consume). It contains none of the drafter's
arithmetic, so it can serve both sides without coupling them.
"""
from .synth import (  # noqa: F401
    CONFIGS,
    DrafterShape,
    LayerWeightsT,
    make_layer_weights,
    make_layer_weights_q4,
    make_block_weights,
    make_head_weights,
    BlockWeightsT,
    HeadWeightsT,
    LayerWeightsQ4,
    Q4Matrix,
    make_prefix_feats,
    make_round_inputs,
    make_accepted,
    make_attention_inputs,
    make_prefix_lens,
    make_ssm_core_inputs,
    rng,
)
