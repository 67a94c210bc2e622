"""Shared driver for parity tests: one library handle and one oracle fed the
same seeded inputs (from the workload module), compared element by element."""
from __future__ import annotations

import numpy as np
import torch

from oracle import hyflash_oracle as O
from workload import make_layer_weights, make_layer_weights_q4

# Tolerances: max-normalised error |g - r|_inf / |r|_inf per compared tensor.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def maxnorm_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


class Pair:
    """A GPU handle and an oracle over the same weights and inputs."""

    def __init__(self, cfg, batch=None, prefill_tokens_max=0, seed=0, oracle=True, tweak=None):
        import speculative_decoding_drafter_hf_gb300 as hf
        self.cfg = cfg
        self.B = cfg.batch if batch is None else batch
        q4 = getattr(cfg, "weight_bits", 16) == 4
        make = make_layer_weights_q4 if q4 else make_layer_weights
        self.weights = [make(cfg, l, seed) for l in range(cfg.n_layers)]
        if tweak is not None:  # e.g. a slower decay, so that old features still count
            self.weights = [tweak(w) for w in self.weights]
        self.gpu = hf.Drafter(cfg, self.B, prefill_tokens_max=prefill_tokens_max)
        for l, w in enumerate(self.weights):
            (self.gpu.set_weights_q4 if q4 else self.gpu.set_weights)(l, w)
        self.orc = O.OracleDrafter(cfg, self.weights, self.B) if oracle else None
        self.tol = TOL[cfg.dtype]

    def close(self):
        self.gpu.check_guards()  # no kernel wrote outside its buffers
        self.gpu.close()

    def prefill(self, lens, feats, requests=None):
        self.gpu.prefill(feats.cuda(), lens, requests)
        if self.orc is not None:
            self.orc.prefill(lens, feats, requests=requests)

    def commit(self, feats, n):
        self.gpu.commit(feats.cuda(), n.to(torch.int32).cuda())
        if self.orc is not None:
            return self.orc.commit(feats, n.numpy())
        return None

    def draft(self, slot):
        out = self.gpu.draft(slot.cuda())
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        ref = self.orc.draft(slot) if self.orc is not None else None
        return got, ref

    def round(self, feats, n, slot):
        """hf_round on the GPU; the oracle commits, then drafts."""
        out = self.gpu.round(feats.cuda(), n.to(torch.int32).cuda(), slot.cuda())
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        offs = ref = None
        if self.orc is not None:
            offs, _ = self.orc.commit(feats, n.numpy())
            ref = self.orc.draft(slot)
        return got, ref, offs

    def check_context(self, requests=None, what=""):
        """State, ring (valid slots), tags and positions against the oracle."""
        cfg, g = self.cfg, self.gpu
        import speculative_decoding_drafter_hf_gb300 as hf
        state = g.read(hf.Tensor.STATE)
        rk = g.read(hf.Tensor.RING_K)
        rv = g.read(hf.Tensor.RING_V)
        tags = g.read(hf.Tensor.RING_TAG)
        pos = g.read(hf.Tensor.POS)
        reqs = range(self.B) if requests is None else requests
        worst = 0.0
        for b in reqs:
            for l in range(cfg.n_layers):
                c = self.orc.ctx[b][l]
                assert pos[b] == c.pos, f"{what}: pos of request {b}: {pos[b]} != {c.pos}"
                assert np.array_equal(tags[b], c.tag.astype(np.int32)), f"{what}: ring tags of request {b}"
                e = maxnorm_err(state[l, b], c.h)
                assert e <= self.tol, f"{what}: state err {e:.3e} (layer {l}, request {b})"
                worst = max(worst, e)
                M = int(getattr(cfg, "mem_horizon", 0) or 0)
                if M > 1 and c.hist is not None and len(c.hist[0]):
                    # memory-input ring: rows of the last M committed positions
                    hx, hB, hdt = c.hist
                    mx, mb, mdt = (g.read(hf.Tensor.MEM_X), g.read(hf.Tensor.MEM_B),
                                   g.read(hf.Tensor.MEM_DT))
                    Mr = M + cfg.block + 1
                    first = c.pos - len(hx)
                    rows = [(q - first, q % Mr) for q in range(first, c.pos)]
                    for name, gg, rr in (
                            ("x", np.stack([mx[l, b, r] for _, r in rows]),
                             np.stack([hx[i].reshape(-1) for i, _ in rows])),
                            ("B", np.stack([mb[l, b, r] for _, r in rows]),
                             np.stack([hB[i] for i, _ in rows])),
                            ("dt", np.stack([mdt[l, b, :, r] for _, r in rows]),
                             np.stack([hdt[i] for i, _ in rows]))):
                        e = maxnorm_err(gg, rr)
                        assert e <= self.tol, f"{what}: memory-input {name} err {e:.3e} (layer {l}, request {b})"
                valid = c.tag >= 0
                if valid.any():
                    for name, gr, orr in (("K", rk, c.ring_k), ("V", rv, c.ring_v)):
                        e = maxnorm_err(gr[l, b][:, valid, :], orr[:, valid, :])
                        assert e <= self.tol, f"{what}: ring {name} err {e:.3e} (layer {l}, request {b})"
                        worst = max(worst, e)
        return worst
