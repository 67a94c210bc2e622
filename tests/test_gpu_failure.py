"""Failure detection on the GPU without faulting it.

  * a bounded device wait that gives up: the CUDA-core attention's ring-tile
    wait is given a limit of 0 cycles (it gives up before its first poll),
    the kernel takes its expiry path and returns, hf_sync reports
    HF_ETIMEOUT once, the context is untouched and the next draft matches
    the oracle again;
  * an allocation that fails inside hf_create (a host-side hook fails the
    k-th cudaMalloc): HF_ENOMEM for every k, and no device memory leaks;
  * guard regions around every buffer of a handle stay intact after rounds
    of every call (the parity harness checks them at every close as well).
"""
import numpy as np
import pytest
import torch

from _harness import Pair, maxnorm_err
from oracle import hyflash_oracle as O
from workload import CONFIGS, make_accepted, make_prefix_feats, make_round_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_drafter_hf_gb300 import build
    build.build()


def test_wait_expiry_reports_timeout_and_context_survives():
    import speculative_decoding_drafter_hf_gb300 as hf
    cfg = CONFIGS["tiny_fp32"].replace(batch=2)
    p = Pair(cfg)
    lens = [100, 30]
    p.prefill(lens, make_prefix_feats(cfg, lens))
    before = p.gpu.export_context()
    slot, feats = make_round_inputs(cfg, 0, 2)
    p.gpu.set_wait_limit(0)
    out = p.gpu.draft(slot.cuda())
    st, msg = p.gpu.sync_status()
    p.gpu.set_wait_limit(-1)
    assert st == hf.Status.ETIMEOUT and "wait" in msg
    assert p.gpu.sync_status()[0] == hf.Status.OK  # the word was cleared
    assert p.gpu.export_context() == before         # drafting stayed read-only
    # the expiry path left the window out of that draft: slots and memory only
    X = O.to64(slot)
    ref = []
    for b in range(2):
        c = p.orc.ctx[b][0].clone()
        c.tag[:] = -1
        ref.append(O.draft_layer(p.orc.layers[0], cfg, c, X[b]))
    assert maxnorm_err(out.cpu().numpy(), np.stack(ref)) <= p.tol
    # and everything works again with the default limit
    got, ref = p.draft(slot)
    assert maxnorm_err(got, ref) <= p.tol
    p.commit(feats, make_accepted(cfg, 0, 2))
    p.check_context(what="after the expiry")
    assert p.gpu.sync_status()[0] == hf.Status.OK
    p.close()


def test_allocation_failure_in_create_leaks_nothing():
    import speculative_decoding_drafter_hf_gb300 as hf
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    cfg = CONFIGS["qwen3_4b_bf16"].replace(batch=2, n_layers=2)
    hf.Drafter(cfg, 2).close()          # module load, context set-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    try:
        for k in range(1, 200):
            assert B.hf_debug_fail_alloc(k) == 0
            try:
                d = hf.Drafter(cfg, 2)
            except hf.HyflashError as e:
                assert e.status == hf.Status.ENOMEM, str(e)
                failures += 1
                free = torch.cuda.mem_get_info()[0]
                assert abs(free - free0) <= (4 << 20), f"k={k}: {(free0 - free) >> 20} MiB leaked"
                continue
            d.close()   # k is past the last allocation: created normally
            break
    finally:
        B.hf_debug_fail_alloc(0)
    assert failures >= 20   # every allocation of hf_create was made to fail once
    assert abs(torch.cuda.mem_get_info()[0] - free0) <= (4 << 20)


@pytest.mark.parametrize("name,batch", [("tiny_fp32", 3), ("qwen3_4b_bf16", 2)])
def test_guard_regions_intact_after_every_call(name, batch):
    cfg = CONFIGS[name].replace(batch=batch, n_layers=2)
    p = Pair(cfg, oracle=False, prefill_tokens_max=256)
    lens = [600, 3, 0][:batch]
    p.gpu.prefill(make_prefix_feats(cfg, lens).cuda(), lens)
    for r in range(3):
        slot, feats = make_round_inputs(cfg, r, batch)
        n = make_accepted(cfg, r, batch).cuda()
        p.gpu.draft(slot.cuda())
        p.gpu.commit(feats.cuda(), n)
        p.gpu.round(feats.cuda(), n, slot.cuda())
    p.gpu.sync()
    p.gpu.check_guards()
    for w in range(5):
        p.gpu.read(w)   # inspection copies stay inside their buffers too
    p.close()
