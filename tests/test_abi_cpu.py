"""The C-ABI library loads here (no GPU) and exports every declared symbol;
host-side argument checks answer without touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hyflash.h")


def _ensure_built():
    from speculative_decoding_drafter_hf_gb300 import build
    return build.build()


@pytest.fixture(scope="module")
def hf():
    _ensure_built()
    import speculative_decoding_drafter_hf_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hf_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(hf):
    lib = ctypes.CDLL(hf.LIB_PATH)
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in hyflash.h but not exported"
    assert set(names) == set(hf.EXPORTED)


def test_config_struct_layout(hf):
    # 14 int32, the int64 pass size, two int32 ablation fields, the memory
    # kind, the weight bits, the three block fields, padding to the int64
    # alignment
    assert ctypes.sizeof(hf.HfConfig) == 96
    assert hf.HfConfig.mem_horizon.offset == 68 and hf.HfConfig.memory_kind.offset == 72
    assert hf.HfConfig.weight_bits.offset == 76
    assert hf.HfConfig.block_kind.offset == 80 and hf.HfConfig.vocab.offset == 88
    assert ctypes.sizeof(hf.HfBlockWeights) == 9 * ctypes.sizeof(ctypes.c_void_p)
    assert ctypes.sizeof(hf.HfLayerWeights) == 12 * ctypes.sizeof(ctypes.c_void_p)


def _cfg(hf, **kw):
    from workload import CONFIGS
    c = hf.make_config(CONFIGS["tiny_fp32"], 2)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value", [
    ("n_groups", 2), ("n_kv_heads", 3), ("head_dim", 66), ("window", 7), ("chunk", 100),
    ("dtype", 5), ("d_model", 250), ("block", 17), ("d_state", 18), ("max_batch", 0),
    ("prefill_tokens_max", -1), ("ssm_headdim", 130), ("cross_slot_off", 2),
    ("mem_horizon", -1), ("mem_horizon", 65), ("memory_kind", 2), ("weight_bits", 8),
    ("weight_bits", 4)])  # (4 bits need a bf16 handle; this one is fp32)
def test_invalid_config_is_einval_without_cuda(hf, field, value):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    h = ctypes.c_void_p()
    s = B.hf_create(ctypes.byref(_cfg(hf, **{field: value})), 0, ctypes.byref(h))
    assert s == hf.Status.EINVAL and not h.value
    assert B.hf_last_error(None).decode()


def test_null_handle_calls_are_einval(hf):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    assert B.hf_draft(None, None, None, 1, None) == hf.Status.EINVAL
    assert B.hf_commit(None, None, None, 1, None) == hf.Status.EINVAL
    assert B.hf_sync(None, None) == hf.Status.EINVAL
    assert B.hf_context_bytes(None) == 0
    assert B.hf_launch_count(None) == 0
    B.hf_destroy(None)
    assert B.hf_status_string(5) == b"HF_EDEVICE"


def test_valid_config_without_gpu_is_ecuda(hf):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    h = ctypes.c_void_p()
    s = B.hf_create(ctypes.byref(_cfg(hf)), 0, ctypes.byref(h))
    assert s == hf.Status.ECUDA and not h.value


def test_gated_delta_with_horizon_is_einval(hf):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    h = ctypes.c_void_p()
    s = B.hf_create(ctypes.byref(_cfg(hf, memory_kind=1, mem_horizon=4)), 0, ctypes.byref(h))
    assert s == hf.Status.EINVAL and not h.value


@pytest.mark.parametrize("kw", [
    dict(block_kind=2),
    dict(block_kind=1, mlp_dim=0, vocab=10),          # no MLP width
    dict(block_kind=1, mlp_dim=100, vocab=10),        # not a multiple of 8
    dict(block_kind=1, mlp_dim=64, vocab=1),          # one-token vocabulary
    dict(block_kind=1, mlp_dim=64, vocab=10, memory_kind=1),
    dict(block_kind=1, mlp_dim=64, vocab=10, mem_horizon=3),
])
def test_invalid_block_config_is_einval_without_cuda(hf, kw):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    h = ctypes.c_void_p()
    s = B.hf_create(ctypes.byref(_cfg(hf, **kw)), 0, ctypes.byref(h))
    assert s == hf.Status.EINVAL and not h.value


def test_block_calls_on_null_handle_are_einval(hf):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    assert B.hf_set_block_weights(None, 0, None, None) == hf.Status.EINVAL
    assert B.hf_set_head_weights(None, None, None) == hf.Status.EINVAL
    assert B.hf_draft_tokens(None, None, None, None, 1, None) == hf.Status.EINVAL
    assert B.hf_debug_check_guards(None) == hf.Status.EINVAL
    assert B.hf_debug_fail_alloc(-1) == hf.Status.EINVAL


# hf_attention_noalloc: a valid call (bf16, 2 requests, 4 query heads over 2
# KV heads, head dim 64, window 64, 7 slots) and one argument changed at a
# time; every refusal comes from the host-side checks, before any CUDA call
# (the pointers are never dereferenced).
_NOALLOC_OK = dict(dtype=1, batch=2, hq=4, hkv=2, dh=64, window=64, block=7, proj=16,
                   proj_ld=512, ring_k=16, ring_v=16, pos=16, out=16, out_ld=256, status=None)


@pytest.mark.parametrize("change,msg", [
    (dict(dtype=5), "dtype"),
    (dict(batch=-1), "positive"),
    (dict(window=0), "positive"),
    (dict(hkv=3), "divide"),
    (dict(dh=12), "multiple of 8"),
    (dict(dh=264, proj_ld=2112, out_ld=1056), "<= 256"),
    (dict(block=17), "block"),
    (dict(hq=32, hkv=1, proj_ld=4352, out_ld=2048), "block"),   # 32 heads x 7 slots > 64 rows
    (dict(proj_ld=510), "proj_ld"),
    (dict(proj_ld=508), "proj_ld"),
    (dict(out_ld=255), "out_ld"),
    (dict(proj=None), "NULL"),
    (dict(out=None), "NULL"),
    (dict(ring_k=8), "16-byte"),
    (dict(proj=20), "16-byte"),
    (dict(status=2), "4-byte"),
    (dict(batch=4096, hq=32, hkv=8, dh=128, window=512, proj_ld=6272, out_ld=4096), "scratch"),
])
def test_noalloc_argument_checks_without_cuda(hf, change, msg):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    a = {**_NOALLOC_OK, **change}
    s = B.hf_attention_noalloc(a["dtype"], a["batch"], a["hq"], a["hkv"], a["dh"], a["window"],
                               a["block"], a["proj"], a["proj_ld"], a["ring_k"], a["ring_v"],
                               a["pos"], a["out"], a["out_ld"], a["status"], None)
    assert s == hf.Status.EINVAL
    assert msg in B.hf_last_error(None).decode()


def test_noalloc_empty_batch_is_ok_without_buffers(hf):
    from speculative_decoding_drafter_hf_gb300 import _binding as B
    a = {**_NOALLOC_OK, "batch": 0, "proj": None, "ring_k": None, "ring_v": None, "pos": None,
         "out": None}
    s = B.hf_attention_noalloc(a["dtype"], a["batch"], a["hq"], a["hkv"], a["dh"], a["window"],
                               a["block"], a["proj"], a["proj_ld"], a["ring_k"], a["ring_v"],
                               a["pos"], a["out"], a["out_ld"], a["status"], None)
    assert s == hf.Status.OK
