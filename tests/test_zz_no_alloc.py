"""The allocation-free attention entry point against the draft path.

hf_attention_noalloc is for callers that cannot allocate device memory when
they run the op (an arena that owns the GPU's memory, memory sized once at
start-up, or no tolerance for the device-wide sync of cudaMalloc/cudaFree).
It keeps its split partials in a fixed array inside the library. This test
feeds it the exact inputs hf_draft used (the slot projections, window rings
and positions read back from a handle) and checks its output against the
attention half of hf_draft's output, on two calls in a row. It lives in a
file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from workload import CONFIGS, make_layer_weights, make_prefix_feats, make_round_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from speculative_decoding_drafter_hf_gb300 import build
    build.build()


def _raw(drafter, which):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    n = drafter.tensor_bytes(which)
    buf = np.empty(n, dtype=np.uint8)
    assert B.hf_read_tensor(drafter._h, int(which), buf.ctypes.data, n) == 0
    return torch.from_numpy(buf)


def _err(got, ref):
    return float((got - ref).abs().max() / ref.abs().max().clamp_min(1e-30))


@pytest.mark.parametrize("name,batch,lens", [
    ("tiny_fp32", 3, [100, 0, 30]),
    ("qwen3_4b_bf16", 2, [1000, 200]),
])
def test_noalloc_attention_matches_draft(name, batch, lens):
    import speculative_decoding_drafter_hf_gb300 as hf
    from speculative_decoding_drafter_hf_gb300 import _binding as B

    cfg = CONFIGS[name].replace(batch=batch)
    d = hf.Drafter(cfg, batch)
    for l in range(cfg.n_layers):
        d.set_weights(l, make_layer_weights(cfg, l))
    d.prefill(make_prefix_feats(cfg, lens).cuda(), lens)
    slot, _ = make_round_inputs(cfg, 0, batch)
    d.draft(slot.cuda())
    d.sync()

    S, QD = cfg.block, cfg.n_q_heads * cfg.head_dim
    Nd = QD + 2 * cfg.n_kv_heads * cfg.head_dim + cfg.d_state
    Nz = QD + cfg.d_inner
    tdt = d.torch_dtype
    proj = _raw(d, hf.Tensor.DRAFT_PROJ).view(torch.float32).reshape(batch * S, Nd).cuda()
    shp = (cfg.n_layers, batch, cfg.n_kv_heads, cfg.window, cfg.head_dim)
    rk = _raw(d, hf.Tensor.RING_K).view(tdt).reshape(shp)[-1].contiguous().cuda()
    rv = _raw(d, hf.Tensor.RING_V).view(tdt).reshape(shp)[-1].contiguous().cuda()
    pos = _raw(d, hf.Tensor.POS).view(torch.int64).cuda()
    ref = _raw(d, hf.Tensor.DRAFT_MIX).view(tdt).reshape(batch * S, Nz)[:, :QD].float()

    out = torch.empty((batch * S, QD), dtype=tdt, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out.fill_(float("nan"))
        s = B.hf_attention_noalloc(0 if cfg.dtype == "f32" else 1, batch, cfg.n_q_heads,
                                   cfg.n_kv_heads, cfg.head_dim, cfg.window, S,
                                   proj.data_ptr(), Nd, rk.data_ptr(), rv.data_ptr(),
                                   pos.data_ptr(), out.data_ptr(), QD, st)
        assert s == 0, B.hf_last_error(None).decode()
        torch.cuda.synchronize()
        got = out.float().cpu()
        assert torch.isfinite(got).all(), f"call {call}: output not fully written"
        e = _err(got, ref)
        assert e <= TOL[cfg.dtype], f"call {call}: error {e:.3e}"
    d.close()


def test_noalloc_rejects_sizes_beyond_its_array():
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    # 4096 requests x 8 KV heads x 16 splits x 28 rows x 130 floats >> 4 Mi floats
    s = B.hf_attention_noalloc(1, 4096, 32, 8, 128, 512, 7, 16, 6272, 16, 16, 16, 16, 4096, None)
    assert s == 1
    assert "scratch" in B.hf_last_error(None).decode()
