"""GPU parity of the full drafter block (block_kind = 1) against the float64
oracle of oracle/full_block.py, through the C ABI.

Compared: the last block's hidden output, the LM-head logits (max-normalised,
1e-4 fp32 / 2e-2 bf16), the slot tokens (bit-exact wherever the oracle's
top-2 logit margin exceeds the tolerance; elsewhere the GPU's token must be
a valid argmax -- its oracle logit within the tolerance of the maximum -- and
always exactly the argmax of the GPU's own logits, ties to the lowest id),
and after prefill and every commit the context: rotated ring keys, values,
tags, positions, the recurrent state and the convolution's carried rows.
"""
import numpy as np
import pytest
import torch

from _harness import TOL, maxnorm_err
from oracle import full_block as FB
from workload import (CONFIGS, make_accepted, make_block_weights, make_head_weights,
                      make_prefix_feats, make_round_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_drafter_hf_gb300 import build
    build.build()


class BlockPair:
    def __init__(self, cfg, batch, prefill_tokens_max=0, oracle=True, head=None):
        import speculative_decoding_drafter_hf_gb300 as hf
        self.cfg, self.B = cfg, batch
        self.blocks = [make_block_weights(cfg, l) for l in range(cfg.n_layers)]
        self.head = make_head_weights(cfg) if head is None else head
        self.gpu = hf.Drafter(cfg, batch, prefill_tokens_max=prefill_tokens_max)
        for l, bw in enumerate(self.blocks):
            self.gpu.set_block_weights(l, bw)
        self.gpu.set_head_weights(self.head)
        self.orc = FB.OracleBlockDrafter(cfg, self.blocks, self.head, batch) if oracle else None
        self.tol = TOL[cfg.dtype]

    def close(self):
        self.gpu.check_guards()
        self.gpu.close()

    def prefill(self, lens, feats):
        self.gpu.prefill(feats.cuda(), lens)
        if self.orc:
            self.orc.prefill(lens, feats)

    def commit(self, feats, n):
        self.gpu.commit(feats.cuda(), n.to(torch.int32).cuda())
        if self.orc:
            self.orc.commit(feats, n.numpy())

    def draft_check(self, slot, what=""):
        import speculative_decoding_drafter_hf_gb300 as hf
        out, tok = self.gpu.draft_tokens(slot.cuda())
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        tok = tok.cpu().numpy().reshape(-1)
        logits = self.gpu.read(hf.Tensor.LOGITS)[:self.B * self.cfg.block].astype(np.float64)
        ref, ref_tok = self.orc.draft(slot)
        e = maxnorm_err(got, ref)
        assert e <= self.tol, f"{what}: block output err {e:.3e}"
        X = ref.reshape(-1, self.cfg.d_model)
        ref_logits, _ = FB.head(FB.HeadWeights64.from_any(self.head), X)
        e = maxnorm_err(logits, ref_logits)
        assert e <= self.tol, f"{what}: logits err {e:.3e}"
        check_tokens(tok, logits, ref_logits, ref_tok.reshape(-1), self.tol, what)

    def check_context(self, what=""):
        import speculative_decoding_drafter_hf_gb300 as hf
        g = self.gpu
        state, rk, rv = g.read(hf.Tensor.STATE), g.read(hf.Tensor.RING_K), g.read(hf.Tensor.RING_V)
        tags, pos, conv = g.read(hf.Tensor.RING_TAG), g.read(hf.Tensor.POS), g.read(hf.Tensor.CONV)
        for b in range(self.B):
            for l in range(self.cfg.n_layers):
                c = self.orc.ctx[b][l]
                assert pos[b] == c.pos, f"{what}: pos of request {b}"
                assert np.array_equal(tags[b], c.tag.astype(np.int32)), f"{what}: tags of {b}"
                for name, gg, rr in (("state", state[l, b], c.h), ("conv rows", conv[l, b], c.conv)):
                    e = maxnorm_err(gg, rr)
                    assert e <= self.tol, f"{what}: {name} err {e:.3e} (layer {l}, request {b})"
                valid = c.tag >= 0
                if valid.any():
                    for name, gr, orr in (("K", rk, c.ring_k), ("V", rv, c.ring_v)):
                        e = maxnorm_err(gr[l, b][:, valid, :], orr[:, valid, :])
                        assert e <= self.tol, f"{what}: ring {name} err {e:.3e} (layer {l}, request {b})"


def check_tokens(tok, logits, ref_logits, ref_tok, tol, what):
    """Tokens: the GPU's own argmax exactly (lowest id on ties); the oracle's
    wherever its margin exceeds the tolerance; a valid argmax elsewhere."""
    for r in range(len(tok)):
        row = logits[r]
        own = int(np.flatnonzero(row == row.max())[0])
        assert tok[r] == own, f"{what}: row {r}: token {tok[r]} is not the argmax {own} of its logits"
        scale = np.max(np.abs(ref_logits))
        top2 = np.sort(ref_logits[r])[-2:]
        if top2[1] - top2[0] > 2 * tol * scale:
            assert tok[r] == ref_tok[r], f"{what}: row {r}: token {tok[r]} != oracle {ref_tok[r]}"
        else:
            assert ref_logits[r, tok[r]] >= top2[1] - 2 * tol * scale, f"{what}: row {r}"


def run_block_rounds(p: BlockPair, rounds: int):
    cfg = p.cfg
    for r in range(rounds):
        slot, feats = make_round_inputs(cfg, r, p.B)
        p.draft_check(slot, f"round {r}")
        p.commit(feats, make_accepted(cfg, r, p.B))
        p.check_context(f"after commit {r}")


TINY = CONFIGS["tiny_fp32"].replace(full_block=True, mlp_dim=192, vocab=96)
QWEN = CONFIGS["qwen3_4b_bf16"].replace(full_block=True, mlp_dim=9728, vocab=4096)


def test_block_tiny_fp32_layers_segments():
    """fp32, two blocks, requests with an empty, a short and a long prefix
    folded in several prefill passes (the convolution's rows carried across
    passes), then draft / commit rounds."""
    cfg = TINY.replace(n_layers=2, batch=3)
    p = BlockPair(cfg, 3, prefill_tokens_max=128)
    lens = [0, 37, 300]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context("prefill")
    run_block_rounds(p, 4)
    p.close()


@pytest.mark.parametrize("batch,lens,layers", [(2, [700, 90], 1), (2, [5, 1300], 2)])
def test_block_qwen3_widths_bf16(batch, lens, layers):
    """bf16 at Qwen3-4B widths with its SwiGLU width (9728): the tensor-core
    GEMMs for the slot, output, MLP and head products."""
    cfg = QWEN.replace(batch=batch, n_layers=layers)
    p = BlockPair(cfg, batch)
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context("prefill")
    run_block_rounds(p, 3)
    p.close()


@pytest.mark.parametrize("chunk,tokens_max", [(64, 1000), (256, 700)])
def test_block_bf16_prefill_passes_and_chunks(chunk, tokens_max):
    cfg = QWEN.replace(batch=3, chunk=chunk)
    p = BlockPair(cfg, 3, prefill_tokens_max=tokens_max)
    lens = [2500, 0, 333]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    p.check_context(f"prefill chunk {chunk}")
    run_block_rounds(p, 2)
    p.close()


def test_block_wide_batch_bf16():
    """Five requests: 35 slot rows and 40 commit rows, so the block's products
    run token-major (more than 32 activation rows)."""
    cfg = QWEN.replace(batch=5, n_layers=2, vocab=1000)
    p = BlockPair(cfg, 5)
    lens = [3, 40, 520, 800, 0]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    run_block_rounds(p, 2)
    p.close()


def test_block_draft_read_only_and_rejected_rows():
    cfg = TINY.replace(batch=2)
    p = BlockPair(cfg, 2, oracle=False)
    lens = [90, 6]
    p.gpu.prefill(make_prefix_feats(cfg, lens).cuda(), lens)
    start = p.gpu.export_context()
    slot, feats = make_round_inputs(cfg, 0, 2)
    p.gpu.draft_tokens(slot.cuda())
    torch.cuda.synchronize()
    assert p.gpu.export_context() == start
    n = torch.tensor([3, 0], dtype=torch.int32)
    p.gpu.commit(feats.cuda(), n.cuda())
    after = p.gpu.export_context()
    p.gpu.import_context(start)
    feats2 = feats.clone()
    feats2[0, 3:] = torch.randn(5, cfg.d_model) * 50
    feats2[1] = torch.randn(8, cfg.d_model) * 50
    p.gpu.commit(feats2.cuda(), n.cuda())
    assert p.gpu.export_context() == after
    p.close()


def test_block_head_ties_go_to_lowest_id():
    """Two identical LM-head columns (4 and 11) and zeros elsewhere: logits 4
    and 11 are equal, so the token is 4 where they are positive, else 0 (all
    other logits tie at zero)."""
    cfg = TINY.replace(batch=2)
    hw = make_head_weights(cfg)
    w = torch.zeros_like(hw.w_lm)
    w[:, 4] = w[:, 11] = hw.w_lm[:, 7]
    hw.w_lm = w
    import speculative_decoding_drafter_hf_gb300 as hf
    p = BlockPair(cfg, 2, head=hw)
    lens = [50, 9]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    slot, _ = make_round_inputs(cfg, 2, 2)
    _, tok = p.gpu.draft_tokens(slot.cuda())
    torch.cuda.synchronize()
    logits = p.gpu.read(hf.Tensor.LOGITS)[:2 * cfg.block]
    assert np.array_equal(logits[:, 4], logits[:, 11])
    want = np.where(logits[:, 4] > 0, 4, 0)
    assert np.array_equal(tok.cpu().numpy().reshape(-1), want)
    p.draft_check(slot, "ties")
    p.close()
