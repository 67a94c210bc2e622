"""The allocation-free attention entry point (hf_attention_noalloc).

It is for callers that cannot allocate device memory when they run the op:
an arena that owns the GPU's memory, memory sized once at start-up, or no
tolerance for the device-wide synchronisation of cudaMalloc/cudaFree. It
keeps its split partials in a fixed array inside the library.

Checked here, through the C ABI, on two calls in a row each:
  * against the oracle's window+block attention on seeded inputs (windows
    empty, partial, full and wrapped, a window that is not a multiple of
    the 32-key split, (Hq/Hkv)*block of 56 and 64, fp32 and bf16);
  * against the attention half of hf_draft's output on the inputs hf_draft
    used (the existing entry point);
  * a ring-tile wait made to give up: the status word reports it and the
    call leaves the window out (slot keys only);
  * sizes beyond the fixed array or the device's shared memory are refused.
This file sorts last, so a run that stops at the first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

from oracle import hyflash_oracle as O
from workload import (CONFIGS, make_attention_inputs, make_layer_weights, make_prefix_feats,
                      make_round_inputs)

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
TIMEOUT_BIT = 2


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
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def _call(cfg, batch, proj, rk, rv, pos, out, status=None):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    S = cfg.block
    qd = cfg.n_q_heads * cfg.head_dim
    return B.hf_attention_noalloc(
        0 if cfg.dtype == "f32" else 1, batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
        cfg.window, S, proj.data_ptr(), proj.shape[1], rk.data_ptr(), rv.data_ptr(),
        pos.data_ptr(), out.data_ptr(), qd, None if status is None else status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def _oracle_attention(cfg, proj, rk, rv, pos, window_on=True):
    """O.window_block_attention per request on the same inputs: ring slot j
    is valid for j < min(pos, W) (a ring after pos commits)."""
    S, H, G, dh = cfg.block, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    qd, kvd = H * dh, G * dh
    P = proj.double().numpy()
    out = []
    for b in range(rk.shape[0]):
        ctx = O.Context.empty(cfg)
        ctx.ring_k = rk[b].double().numpy()
        ctx.ring_v = rv[b].double().numpy()
        nv = min(int(pos[b]), cfg.window) if window_on else 0
        ctx.tag = np.where(np.arange(cfg.window) < nv, np.arange(cfg.window), -1)
        rows = P[b * S:(b + 1) * S]
        Q = rows[:, :qd].reshape(S, H, dh)
        Ks = rows[:, qd:qd + kvd].reshape(S, G, dh)
        Vs = rows[:, qd + kvd:qd + 2 * kvd].reshape(S, G, dh)
        out.append(O.window_block_attention(cfg, ctx, Q, Ks, Vs).reshape(S, -1))
    return np.concatenate(out)


# name -> (config overrides, positions per request)
SHAPES = {
    "tiny_fp32_full_and_empty": ("tiny_fp32", {}, [100, 0, 30, 64]),
    "qwen3_bf16_wrapped": ("qwen3_4b_bf16", {}, [1000, 200, 512]),
    "w50_fp32_ragged_split": ("tiny_fp32", dict(window=50), [10, 49, 50, 51, 333]),
    "w50_bf16_ragged_split": ("qwen3_4b_bf16", dict(window=50, n_q_heads=16, n_kv_heads=4,
                                                    head_dim=64), [3, 33, 50, 90]),
    "g8_rows56_bf16": ("qwen3_4b_bf16", dict(window=200, n_q_heads=16, n_kv_heads=2), [150, 700]),
    "g4_block16_rows64_fp32": ("tiny_fp32", dict(window=96, block=16, n_q_heads=8, n_kv_heads=2),
                               [40, 96, 500]),
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_noalloc_attention_matches_oracle(name):
    base, over, pos_list = SHAPES[name]
    cfg = CONFIGS[base].replace(**over)
    batch = len(pos_list)
    proj, rk, rv = make_attention_inputs(cfg, batch, seed=3)
    pos = torch.tensor(pos_list, dtype=torch.int64)
    ref = _oracle_attention(cfg, proj, rk, rv, pos)
    d_proj, d_rk, d_rv, d_pos = proj.cuda(), rk.cuda(), rv.cuda(), pos.cuda()
    qd = cfg.n_q_heads * cfg.head_dim
    out = torch.empty((batch * cfg.block, qd), dtype=cfg.torch_dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        s = _call(cfg, batch, d_proj, d_rk, d_rv, d_pos, out, status)
        from speculative_decoding_drafter_hf_gb300 import _binding as B
        assert s == 0, B.hf_last_error(None).decode()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: output not fully written"
        e = _err(got, ref)
        assert e <= TOL[cfg.dtype], f"call {call}: error {e:.3e} vs the oracle"
        assert int(status.item()) == 0


@pytest.mark.parametrize("name,batch,lens", [
    ("tiny_fp32", 3, [100, 0, 30]),
    ("qwen3_4b_bf16", 2, [1000, 200]),
])
def test_noalloc_attention_matches_draft(name, batch, lens):
    """The same op as hf_draft's attention (the existing entry point), on the
    projections and rings hf_draft used."""
    import speculative_decoding_drafter_hf_gb300 as hf
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
    ref = _raw(d, hf.Tensor.DRAFT_MIX).view(tdt).reshape(batch * S, Nz)[:, :QD].float().numpy()
    out = torch.empty((batch * S, QD), dtype=tdt, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        assert _call(cfg, batch, proj, rk, rv, pos, out) == 0
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: output not fully written"
        e = _err(got, ref)
        assert e <= TOL[cfg.dtype], f"call {call}: error {e:.3e} vs hf_draft"
    d.close()


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_4b_bf16"])
def test_noalloc_wait_expiry_is_reported(name):
    """A ring-tile wait that gives up (limit 0: before its first poll) sets
    the timeout bit in the caller's status word, and the call leaves the
    window out: the result is the attention over the slot keys alone. The
    default limit then gives the full result again with a clear status."""
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    cfg = CONFIGS[name]
    pos_list = [70, 300, 5]
    batch = len(pos_list)
    proj, rk, rv = make_attention_inputs(cfg, batch, seed=4)
    pos = torch.tensor(pos_list, dtype=torch.int64)
    d_proj, d_rk, d_rv, d_pos = proj.cuda(), rk.cuda(), rv.cuda(), pos.cuda()
    qd = cfg.n_q_heads * cfg.head_dim
    out = torch.empty((batch * cfg.block, qd), dtype=cfg.torch_dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        assert B.hf_debug_set_wait_limit(None, 0) == 0
        assert _call(cfg, batch, d_proj, d_rk, d_rv, d_pos, out, status) == 0
        torch.cuda.synchronize()
    finally:
        B.hf_debug_set_wait_limit(None, -1)
    assert int(status.item()) & TIMEOUT_BIT
    slots_only = _oracle_attention(cfg, proj, rk, rv, pos, window_on=False)
    assert _err(out.float().cpu().numpy(), slots_only) <= TOL[cfg.dtype]
    status.zero_()
    assert _call(cfg, batch, d_proj, d_rk, d_rv, d_pos, out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    full = _oracle_attention(cfg, proj, rk, rv, pos)
    assert _err(out.float().cpu().numpy(), full) <= TOL[cfg.dtype]


def test_noalloc_rejects_sizes_beyond_its_array():
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    # 4096 requests x 8 KV heads x 16 splits x 28 rows x 130 floats >> 4 Mi floats
    s = B.hf_attention_noalloc(1, 4096, 32, 8, 128, 512, 7, 16, 6272, 16, 16, 16, 16, 4096, None,
                               None)
    assert s == 1
    assert "scratch" in B.hf_last_error(None).decode()


def test_noalloc_rejects_shapes_beyond_shared_memory():
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    # fp32, head_dim 256, 64 query rows per CTA, 128 splits: ~274 KB per CTA
    s = B.hf_attention_noalloc(0, 1, 4, 1, 256, 4096, 16, 16, 1536, 16, 16, 16, 16, 1024, None,
                               None)
    assert s == 1
    assert "shared memory" in B.hf_last_error(None).decode()
