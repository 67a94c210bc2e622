"""ctypes binding of libhyflash.so (include/hyflash.h): argument marshalling only.

Every computation happens in the library's CUDA kernels. PyTorch is used here
only to hand over device pointers and streams. If the shared library has not
been built, importing this module raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import enum
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhyflash.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -m speculative_decoding_drafter_hf_gb300.build` (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)


class Status(enum.IntEnum):
    OK = 0
    EINVAL = 1
    ENOMEM = 2
    ECUDA = 3
    ETIMEOUT = 4
    EDEVICE = 5


class Tensor(enum.IntEnum):
    STATE = 0
    RING_K = 1
    RING_V = 2
    RING_TAG = 3
    POS = 4
    OFFSETS = 5
    DRAFT_PROJ = 6
    DRAFT_MIX = 7
    MEM_X = 8
    MEM_B = 9
    MEM_DT = 10
    CONV = 11
    LOGITS = 12


class Family(enum.IntEnum):
    DRAFT_PROJ = 0
    ATTN_MEM = 1
    OUT_PROJ = 2
    ROUND_PROJ = 3
    COMMIT_PROJ = 4
    COMMIT_STATE = 5
    PREFILL = 6
    OTHER = 7
    MLP = 8
    HEAD = 9


HF_F32, HF_BF16 = 0, 1


class HfConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "d_model", "n_q_heads", "n_kv_heads", "head_dim", "window", "block",
        "ssm_heads", "ssm_headdim", "d_state", "n_groups", "n_layers",
        "max_batch", "chunk", "dtype")] + [("prefill_tokens_max", ctypes.c_int64),
                                           ("cross_slot_off", ctypes.c_int32),
                                           ("mem_horizon", ctypes.c_int32),
                                           ("memory_kind", ctypes.c_int32),
                                           ("weight_bits", ctypes.c_int32),
                                           ("block_kind", ctypes.c_int32),
                                           ("mlp_dim", ctypes.c_int32),
                                           ("vocab", ctypes.c_int32)]


WEIGHT_FIELDS = ("w_q", "w_k", "w_v", "w_o", "w_x", "w_B", "w_C", "w_dt", "w_mo",
                 "dt_bias", "A_log", "w_beta")
MEMORY_KINDS = {"mamba2": 0, "gdn": 1}


class HfLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


BLOCK_FIELDS = ("g_mix", "g_mlp", "w_z", "d_skip", "conv_w", "conv_b", "w_gate", "w_up", "w_down")
BLOCK_F32 = ("g_mix", "g_mlp", "d_skip", "conv_w", "conv_b")


class HfBlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in BLOCK_FIELDS]


class HfQ4Matrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p)]


Q4_MATRICES = ("w_q", "w_k", "w_v", "w_o", "w_x", "w_B", "w_C", "w_dt", "w_mo", "w_beta")


class HfLayerWeightsQ4(ctypes.Structure):
    _fields_ = [(n, HfQ4Matrix) for n in Q4_MATRICES] + [
        ("dt_bias", ctypes.c_void_p), ("A_log", ctypes.c_void_p)]


_h = ctypes.c_void_p
_st = ctypes.c_int
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


def _sig(name, res, *args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


hf_create = _sig("hf_create", _st, ctypes.POINTER(HfConfig), _i32, ctypes.POINTER(_h))
hf_destroy = _sig("hf_destroy", None, _h)
hf_set_weights = _sig("hf_set_weights", _st, _h, _i32, ctypes.POINTER(HfLayerWeights))
hf_set_weights_q4 = _sig("hf_set_weights_q4", _st, _h, _i32, ctypes.POINTER(HfLayerWeightsQ4))
hf_prefill = _sig("hf_prefill", _st, _h, _vp, ctypes.POINTER(_i32), ctypes.POINTER(_i32), _i32, _vp)
hf_commit = _sig("hf_commit", _st, _h, _vp, _vp, _i32, _vp)
hf_draft = _sig("hf_draft", _st, _h, _vp, _vp, _i32, _vp)
hf_round = _sig("hf_round", _st, _h, _vp, _vp, _vp, _vp, _i32, _vp)
hf_sync = _sig("hf_sync", _st, _h, _vp)
hf_last_error = _sig("hf_last_error", ctypes.c_char_p, _h)
hf_status_string = _sig("hf_status_string", ctypes.c_char_p, _st)
hf_tensor_bytes = _sig("hf_tensor_bytes", _st, _h, _i32, ctypes.POINTER(ctypes.c_size_t))
hf_read_tensor = _sig("hf_read_tensor", _st, _h, _i32, _vp, ctypes.c_size_t)
hf_context_bytes = _sig("hf_context_bytes", ctypes.c_size_t, _h)
hf_export_context = _sig("hf_export_context", _st, _h, _vp, ctypes.c_size_t)
hf_import_context = _sig("hf_import_context", _st, _h, _vp, ctypes.c_size_t)
hf_profile_enable = _sig("hf_profile_enable", _st, _h, _i32)
hf_profile_collect = _sig("hf_profile_collect", _st, _h)
hf_profile_read = _sig("hf_profile_read", _st, _h, _i32, ctypes.POINTER(ctypes.c_double),
                       ctypes.POINTER(ctypes.c_int64), _i32)
hf_launch_count = _sig("hf_launch_count", ctypes.c_int64, _h)
hf_attention_noalloc = _sig("hf_attention_noalloc", _st, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                            _vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp)
hf_set_block_weights = _sig("hf_set_block_weights", _st, _h, _i32, ctypes.POINTER(HfLayerWeights),
                            ctypes.POINTER(HfBlockWeights))
hf_set_head_weights = _sig("hf_set_head_weights", _st, _h, _vp, _vp)
hf_draft_tokens = _sig("hf_draft_tokens", _st, _h, _vp, _vp, _vp, _i32, _vp)
hf_debug_set_wait_limit = _sig("hf_debug_set_wait_limit", _st, _h, ctypes.c_int64)
hf_debug_fail_alloc = _sig("hf_debug_fail_alloc", _st, ctypes.c_int64)
hf_debug_check_guards = _sig("hf_debug_check_guards", _st, _h)

EXPORTED = ("hf_create", "hf_destroy", "hf_set_weights", "hf_set_weights_q4", "hf_prefill", "hf_commit", "hf_draft",
            "hf_round", "hf_sync", "hf_last_error", "hf_status_string", "hf_tensor_bytes", "hf_read_tensor",
            "hf_context_bytes", "hf_export_context", "hf_import_context", "hf_profile_enable",
            "hf_profile_collect", "hf_profile_read", "hf_launch_count", "hf_attention_noalloc",
            "hf_debug_set_wait_limit", "hf_debug_fail_alloc", "hf_debug_check_guards",
            "hf_set_block_weights", "hf_set_head_weights", "hf_draft_tokens")


class HyflashError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = Status(status)
        super().__init__(f"{self.status.name}: {message}")


def make_config(shape, max_batch: int, prefill_tokens_max: int = 0) -> HfConfig:
    """HfConfig from any object with the drafter shape attributes."""
    return HfConfig(
        d_model=shape.d_model, n_q_heads=shape.n_q_heads, n_kv_heads=shape.n_kv_heads,
        head_dim=shape.head_dim, window=shape.window, block=shape.block,
        ssm_heads=shape.ssm_heads, ssm_headdim=shape.ssm_headdim, d_state=shape.d_state,
        n_groups=getattr(shape, "n_groups", 1), n_layers=shape.n_layers, max_batch=max_batch,
        chunk=getattr(shape, "chunk", 128),
        dtype=HF_F32 if shape.dtype in ("f32", "fp32", "float32") else HF_BF16,
        prefill_tokens_max=prefill_tokens_max,
        cross_slot_off=0 if getattr(shape, "cross_slot", True) else 1,
        mem_horizon=int(getattr(shape, "mem_horizon", 0) or 0),
        memory_kind=MEMORY_KINDS[getattr(shape, "memory", "mamba2") or "mamba2"],
        weight_bits=int(getattr(shape, "weight_bits", 16) or 16),
        block_kind=1 if getattr(shape, "full_block", False) else 0,
        mlp_dim=int(getattr(shape, "mlp_dim", 0) or 0) if getattr(shape, "full_block", False) else 0,
        vocab=int(getattr(shape, "vocab", 0) or 0) if getattr(shape, "full_block", False) else 0)


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_ptr(t, dtype=None, shape=None, name="tensor"):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


class Drafter:
    """One library handle: windows, memories and weights of ``max_batch``
    requests on one GPU. Methods map one-to-one onto the C calls."""

    def __init__(self, shape, max_batch: int, device: int = 0, prefill_tokens_max: int = 0):
        import torch
        self.shape = shape
        self.max_batch = max_batch
        self.device = device
        self.cfg = make_config(shape, max_batch, prefill_tokens_max)
        self.torch_dtype = torch.float32 if self.cfg.dtype == HF_F32 else torch.bfloat16
        self.np_elem = 4 if self.cfg.dtype == HF_F32 else 2
        h = _h()
        s = hf_create(ctypes.byref(self.cfg), device, ctypes.byref(h))
        if s != 0:
            raise HyflashError(s, hf_last_error(None).decode())
        self._h = h

    # -- lifecycle
    def close(self):
        if getattr(self, "_h", None):
            hf_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, s):
        if s != 0:
            raise HyflashError(s, hf_last_error(self._h).decode())

    # -- weights
    def set_weights(self, layer: int, w):
        import torch
        keep = []
        lw = HfLayerWeights()
        for name in WEIGHT_FIELDS:
            t = getattr(w, name, None)
            if t is None:  # optional (w_beta outside the gated-delta memory)
                continue
            want = torch.float32 if name in ("dt_bias", "A_log") else self.torch_dtype
            t = t.detach().to("cpu", want).contiguous()
            keep.append(t)
            setattr(lw, name, t.data_ptr())
        self._check(hf_set_weights(self._h, layer, ctypes.byref(lw)))

    def _layer_struct(self, w, keep):
        import torch
        lw = HfLayerWeights()
        for name in WEIGHT_FIELDS:
            t = getattr(w, name, None)
            if t is None:  # optional (w_beta outside the gated-delta memory)
                continue
            want = torch.float32 if name in ("dt_bias", "A_log") else self.torch_dtype
            t = t.detach().to("cpu", want).contiguous()
            keep.append(t)
            setattr(lw, name, t.data_ptr())
        return lw

    def set_block_weights(self, layer: int, bw):
        """Full block: the layer's weights (bw.layer) and the parts around it."""
        import torch
        keep = []
        lw = self._layer_struct(bw.layer, keep)
        b = HfBlockWeights()
        for name in BLOCK_FIELDS:
            want = torch.float32 if name in BLOCK_F32 else self.torch_dtype
            t = getattr(bw, name).detach().to("cpu", want).contiguous()
            keep.append(t)
            setattr(b, name, t.data_ptr())
        self._check(hf_set_block_weights(self._h, layer, ctypes.byref(lw), ctypes.byref(b)))

    def set_head_weights(self, hw):
        import torch
        g = hw.g_final.detach().to("cpu", torch.float32).contiguous()
        w = hw.w_lm.detach().to("cpu", self.torch_dtype).contiguous()
        self._check(hf_set_head_weights(self._h, g.data_ptr(), w.data_ptr()))

    def draft_tokens(self, slot_emb, out=None, tokens=None, stream=None):
        """hf_draft_tokens: (hidden out [B, S, D], tokens int32 [B, S])."""
        import torch
        B = int(slot_emb.shape[0])
        shp = (B, self.shape.block, self.shape.d_model)
        sp = _dev_ptr(slot_emb, self.torch_dtype, shp, "slot_emb")
        if out is None:
            out = torch.empty(shp, dtype=self.torch_dtype, device=slot_emb.device)
        if tokens is None:
            tokens = torch.empty((B, self.shape.block), dtype=torch.int32, device=slot_emb.device)
        op = _dev_ptr(out, self.torch_dtype, shp, "out")
        tp = _dev_ptr(tokens, torch.int32, (B, self.shape.block), "tokens")
        self._check(hf_draft_tokens(self._h, sp, op, tp, B, _stream_ptr(stream)))
        return out, tokens

    def set_weights_q4(self, layer: int, w):
        """4-bit weights (weight_bits = 4): each matrix as codes uint8 [in, out],
        scales bf16 [in/128, out], zeros uint8 [in/128, out]."""
        import torch
        keep = []
        lw = HfLayerWeightsQ4()

        def host(t, dtype):
            t = t.detach().to("cpu", dtype).contiguous()
            keep.append(t)
            return t.data_ptr()

        for name in Q4_MATRICES:
            m = getattr(w, name, None)
            if m is None:
                continue
            q = getattr(lw, name)
            q.codes = host(m.codes, torch.uint8)
            q.scales = host(m.scales, torch.bfloat16)
            q.zeros = host(m.zeros, torch.uint8)
        lw.dt_bias = host(w.dt_bias, torch.float32)
        lw.A_log = host(w.A_log, torch.float32)
        self._check(hf_set_weights_q4(self._h, layer, ctypes.byref(lw)))

    # -- the three operations of the method
    def prefill(self, feats, lens: Sequence[int], requests: Optional[Sequence[int]] = None,
                stream=None):
        n = len(lens)
        la = (_i32 * max(n, 1))(*[int(x) for x in lens])
        ra = None
        if requests is not None:
            ra = (_i32 * max(n, 1))(*[int(x) for x in requests])
        total = int(sum(int(x) for x in lens))
        fp = _dev_ptr(feats, self.torch_dtype, (total, self.shape.d_model), "feats") if total else None
        self._check(hf_prefill(self._h, fp, la, ra, n, _stream_ptr(stream)))

    def commit(self, feats, n_accepted, stream=None):
        import torch
        B = int(n_accepted.shape[0])
        fp = _dev_ptr(feats, self.torch_dtype, (B, self.shape.block + 1, self.shape.d_model), "feats")
        npp = _dev_ptr(n_accepted, torch.int32, (B,), "n_accepted")
        self._check(hf_commit(self._h, fp, npp, B, _stream_ptr(stream)))

    def draft(self, slot_emb, out=None, stream=None):
        import torch
        B = int(slot_emb.shape[0])
        shp = (B, self.shape.block, self.shape.d_model)
        sp = _dev_ptr(slot_emb, self.torch_dtype, shp, "slot_emb")
        if out is None:
            out = torch.empty(shp, dtype=self.torch_dtype, device=slot_emb.device)
        op = _dev_ptr(out, self.torch_dtype, shp, "out")
        self._check(hf_draft(self._h, sp, op, B, _stream_ptr(stream)))
        return out

    def round(self, feats, n_accepted, slot_emb, out=None, stream=None):
        """hf_round: commit (feats, n_accepted), then draft slot_emb -> out."""
        import torch
        B = int(n_accepted.shape[0])
        if int(slot_emb.shape[0]) != B:
            raise ValueError("feats, n_accepted and slot_emb must have the same batch")
        fp = _dev_ptr(feats, self.torch_dtype, (B, self.shape.block + 1, self.shape.d_model), "feats")
        npp = _dev_ptr(n_accepted, torch.int32, (B,), "n_accepted")
        shp = (B, self.shape.block, self.shape.d_model)
        sp = _dev_ptr(slot_emb, self.torch_dtype, shp, "slot_emb")
        if out is None:
            out = torch.empty(shp, dtype=self.torch_dtype, device=slot_emb.device)
        op = _dev_ptr(out, self.torch_dtype, shp, "out")
        self._check(hf_round(self._h, fp, npp, sp, op, B, _stream_ptr(stream)))
        return out

    def sync(self, stream=None):
        self._check(hf_sync(self._h, _stream_ptr(stream)))

    def sync_status(self, stream=None):
        """hf_sync's status without raising: (status, message)."""
        s = hf_sync(self._h, _stream_ptr(stream))
        return Status(s), hf_last_error(self._h).decode()

    # -- inspection
    def tensor_bytes(self, which: int) -> int:
        n = ctypes.c_size_t()
        self._check(hf_tensor_bytes(self._h, int(which), ctypes.byref(n)))
        return n.value

    def read(self, which: int) -> np.ndarray:
        """Whole inspectable tensor as a NumPy array (bf16 returned as float32)."""
        nb = self.tensor_bytes(which)
        if nb == 0:  # memory-horizon rows of a handle without them
            return np.zeros((0,), dtype=np.float32)
        buf = np.empty(nb, dtype=np.uint8)
        self._check(hf_read_tensor(self._h, int(which), buf.ctypes.data, nb))
        sh, L, Bm = self.shape, self.shape.n_layers, self.max_batch
        which = Tensor(which)
        if which == Tensor.STATE:
            return buf.view(np.float32).reshape(L, Bm, sh.ssm_heads, sh.ssm_headdim, sh.d_state)
        if which in (Tensor.RING_K, Tensor.RING_V):
            a = self._model_to_f32(buf)
            return a.reshape(L, Bm, sh.n_kv_heads, sh.window, sh.head_dim)
        if which == Tensor.RING_TAG:
            return buf.view(np.int32).reshape(Bm, sh.window)
        if which == Tensor.POS:
            return buf.view(np.int64).copy()
        if which == Tensor.OFFSETS:
            return buf.view(np.int32).copy()
        if which == Tensor.DRAFT_PROJ:
            return buf.view(np.float32).reshape(Bm * sh.block, -1)
        if which == Tensor.CONV:
            return buf.view(np.float32).reshape(L, Bm, 3, -1)
        if which == Tensor.LOGITS:
            return buf.view(np.float32).reshape(Bm * sh.block, -1)
        if which in (Tensor.MEM_X, Tensor.MEM_B, Tensor.MEM_DT):
            R = int(getattr(sh, "mem_horizon", 0)) + sh.block + 1
            a = buf.view(np.float32)
            if which == Tensor.MEM_DT:
                return a.reshape(L, Bm, sh.ssm_heads, R)
            return a.reshape(L, Bm, R, -1)
        return self._model_to_f32(buf).reshape(Bm * sh.block, -1)

    def _model_to_f32(self, buf: np.ndarray) -> np.ndarray:
        if self.np_elem == 4:
            return buf.view(np.float32).copy()
        u = buf.view(np.uint16).astype(np.uint32) << 16
        return u.view(np.float32)

    def context_bytes(self) -> int:
        return int(hf_context_bytes(self._h))

    def export_context(self) -> bytes:
        n = self.context_bytes()
        buf = np.empty(n, dtype=np.uint8)
        self._check(hf_export_context(self._h, buf.ctypes.data, n))
        return buf.tobytes()

    def import_context(self, blob: bytes):
        buf = np.frombuffer(blob, dtype=np.uint8).copy()
        self._check(hf_import_context(self._h, buf.ctypes.data, buf.size))

    # -- measurement
    def profile(self, mode):
        """0 off, 1 (or True) per-call records, 2 records kept for graph replays."""
        self._check(hf_profile_enable(self._h, int(mode)))

    def profile_collect(self):
        self._check(hf_profile_collect(self._h))

    def profile_read(self, family: int, reset: bool = False):
        ms = ctypes.c_double()
        n = ctypes.c_int64()
        self._check(hf_profile_read(self._h, int(family), ctypes.byref(ms), ctypes.byref(n),
                                    1 if reset else 0))
        return ms.value, n.value

    def launch_count(self) -> int:
        return int(hf_launch_count(self._h))

    # -- failure detection (tests)
    def set_wait_limit(self, cycles: int):
        """Limit of the CUDA-core attention's ring-tile wait (-1: default)."""
        self._check(hf_debug_set_wait_limit(self._h, int(cycles)))

    def check_guards(self):
        """Raise if a guard region around one of the handle's buffers changed."""
        self._check(hf_debug_check_guards(self._h))
