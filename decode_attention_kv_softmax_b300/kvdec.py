"""Python binding of libkvdec (the C ABI in include/kvdec.h).

Argument marshalling only: every operation runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
fallback: if libkvdec.so is missing or a call fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvdec.so")

ABI_VERSION = 3
F32, BF16 = 0, 1
KV_BF16, KV_FP8_E4M3 = 0, 1
APPEND_MLA, APPEND_GQA = 0, 1
DEVERR_BAD_PAGE, DEVERR_SEQLEN, DEVERR_TIMEOUT = 0x1, 0x2, 0x4
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
          4: "workspace too small"}


class GqaParams(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p),
                ("block_table", c_void_p), ("seqlens", c_void_p),
                ("batch", c_int32), ("num_heads", c_int32), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("capacity", c_int32), ("num_pages", c_int32),
                ("max_blocks", c_int32), ("scale", c_float), ("out", c_void_p),
                ("out_dtype", c_int32), ("lse", c_void_p), ("workspace", c_void_p),
                ("workspace_bytes", c_size_t), ("error_flag", c_void_p),
                ("max_ctas", c_int32), ("kv_format", c_int32), ("k_scale", c_void_p),
                ("v_scale", c_void_p), ("window", c_int32), ("reserved", c_int32)]


class MlaParams(ctypes.Structure):
    _fields_ = [("q_absorbed", c_void_p), ("q_rope", c_void_p), ("cache", c_void_p),
                ("block_table", c_void_p), ("seqlens", c_void_p), ("batch", c_int32),
                ("num_heads", c_int32), ("num_pages", c_int32), ("max_blocks", c_int32),
                ("scale", c_float), ("out", c_void_p), ("out_dtype", c_int32),
                ("lse", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t),
                ("error_flag", c_void_p), ("max_ctas", c_int32), ("kv_format", c_int32),
                ("kv_scale", c_void_p)]


class AppendParams(ctypes.Structure):
    _fields_ = [("mode", c_int32), ("batch", c_int32), ("seqlens", c_void_p),
                ("block_table", c_void_p), ("num_pages", c_int32), ("max_blocks", c_int32),
                ("rope_theta", c_float), ("c_kv", c_void_p), ("k_rope", c_void_p),
                ("cache", c_void_p), ("k_new", c_void_p), ("v_new", c_void_p),
                ("k", c_void_p), ("v", c_void_p), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("capacity", c_int32), ("reserved", c_int32),
                ("error_flag", c_void_p), ("kv_format", c_int32), ("window", c_int32),
                ("k_scale", c_void_p), ("v_scale", c_void_p)]


class CombineParams(ctypes.Structure):
    _fields_ = [("partial_o", c_void_p), ("partial_lse", c_void_p),
                ("split_counts", c_void_p), ("num_splits", c_int32), ("rows", c_int32),
                ("head_dim", c_int32), ("out_dtype", c_int32), ("out", c_void_p),
                ("lse", c_void_p)]


class MlaProjParams(ctypes.Structure):
    _fields_ = [("x", c_void_p), ("w", c_void_p), ("y", c_void_p), ("batch", c_int32),
                ("num_heads", c_int32), ("out_dtype", c_int32), ("reserved", c_int32)]


class MlaExpandParams(ctypes.Structure):
    _fields_ = [("c_kv", c_void_p), ("w_uk", c_void_p), ("w_uv", c_void_p), ("k_nope", c_void_p),
                ("v", c_void_p), ("s", c_int32), ("num_heads", c_int32)]


class MlaPrefillParams(ctypes.Structure):
    _fields_ = [("q_nope", c_void_p), ("q_rope", c_void_p), ("k_nope", c_void_p),
                ("k_rope", c_void_p), ("v", c_void_p), ("s_q", c_int32), ("s_kv", c_int32),
                ("num_heads", c_int32), ("kv_offset", c_int32), ("scale", c_float),
                ("out_dtype", c_int32), ("out", c_void_p), ("lse", c_void_p)]


EXPORTS = ["kvdec_abi_version", "kvdec_params_size", "kvdec_status_string",
           "kvdec_last_error", "kvdec_gqa_workspace_bytes", "kvdec_gqa_decode",
           "kvdec_mla_workspace_bytes", "kvdec_mla_decode_absorbed", "kvdec_append_rope",
           "kvdec_combine_splits", "kvdec_selftest_wait_timeout",
           "kvdec_gqa_decode_noalloc", "kvdec_mla_absorb_q", "kvdec_mla_project_out",
           "kvdec_mla_prefill_expand", "kvdec_mla_prefill", "kvdec_mla_max_batch"]

_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libkvdec.so (once) and check the struct layouts against it."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -m decode_attention_kv_softmax_b300.build` (no CPU fallback)")
        lib = ctypes.CDLL(path)
        lib.kvdec_abi_version.restype = ctypes.c_int
        lib.kvdec_mla_max_batch.restype = ctypes.c_int32
        lib.kvdec_params_size.restype = c_int64
        lib.kvdec_params_size.argtypes = [ctypes.c_int]
        lib.kvdec_status_string.restype = ctypes.c_char_p
        lib.kvdec_status_string.argtypes = [ctypes.c_int]
        lib.kvdec_last_error.restype = ctypes.c_char_p
        for name, st in [("gqa", GqaParams), ("mla", MlaParams)]:
            f = getattr(lib, f"kvdec_{name}_workspace_bytes")
            f.restype = c_size_t
            f.argtypes = [ctypes.POINTER(st)]
        for name, st in [("kvdec_gqa_decode", GqaParams), ("kvdec_gqa_decode_noalloc", GqaParams),
                         ("kvdec_mla_decode_absorbed", MlaParams),
                         ("kvdec_append_rope", AppendParams),
                         ("kvdec_combine_splits", CombineParams),
                         ("kvdec_mla_absorb_q", MlaProjParams),
                         ("kvdec_mla_project_out", MlaProjParams),
                         ("kvdec_mla_prefill_expand", MlaExpandParams),
                         ("kvdec_mla_prefill", MlaPrefillParams)]:
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.POINTER(st), c_void_p]
        lib.kvdec_selftest_wait_timeout.restype = ctypes.c_int
        lib.kvdec_selftest_wait_timeout.argtypes = [c_uint64, c_void_p, c_void_p]
        if lib.kvdec_abi_version() != ABI_VERSION:
            raise RuntimeError("libkvdec ABI version mismatch")
        for kind, st in enumerate([GqaParams, MlaParams, AppendParams, CombineParams, MlaProjParams,
                                   MlaExpandParams, MlaPrefillParams]):
            if lib.kvdec_params_size(kind) != ctypes.sizeof(st):
                raise RuntimeError(f"params struct {st.__name__} layout mismatch")
        _lib = lib
        return lib


class KvdecError(RuntimeError):
    pass


def _check(status: int, what: str):
    if status != 0:
        msg = _lib.kvdec_last_error().decode(errors="replace")
        raise KvdecError(f"{what}: {STATUS.get(status, status)}: {msg}")


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise ValueError(f"output dtype {dt} (float32 or bfloat16)")


def _need(t, name, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


# ---------------------------------------------------------------- workspace

class Workspace:
    """A device buffer reused across calls (grown on demand).  The library
    needs no initialisation of it: split counters carry a per-call epoch."""

    def __init__(self):
        self._bufs = {}

    def get(self, device, nbytes: int) -> torch.Tensor:
        key = (device.index if device.index is not None else torch.cuda.current_device())
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf

    def reset(self):
        for b in self._bufs.values():
            b.zero_()


_default_ws = Workspace()


def default_workspace() -> Workspace:
    return _default_ws


def new_error_flag(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


# ---------------------------------------------------------------- GQA

_FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _kv_format(k, v, k_scale, v_scale, dev) -> int:
    """KV_BF16 for a bf16 cache; KV_FP8_E4M3 for E4M3 bytes (uint8 or
    float8_e4m3fn) with fp32 per-KV-head scales on the same device."""
    if k.dtype == torch.bfloat16:
        _need(v, "v", torch.bfloat16, dev)
        return KV_BF16
    if k.dtype not in _FP8_DTYPES or v.dtype not in _FP8_DTYPES:
        raise TypeError(f"k, v must be bf16 or E4M3 bytes, got {k.dtype}, {v.dtype}")
    if k_scale is None or v_scale is None:
        raise ValueError("an FP8 cache needs k_scale and v_scale")
    n_kv = k.shape[1]
    for t, n in [(k_scale, "k_scale"), (v_scale, "v_scale")]:
        _need(t, n, torch.float32, dev)
        if t.numel() != n_kv:
            raise ValueError(f"{n} must hold num_kv_heads={n_kv} values")
    return KV_FP8_E4M3


def gqa_params(q, k, v, seqlens, block_table=None, scale=None, out=None, lse=None,
               error_flag=None, max_ctas=0, workspace=None, k_scale=None, v_scale=None,
               window=0):
    p = GqaParams()
    if k.dtype in _FP8_DTYPES:
        p.kv_format = KV_FP8_E4M3
        p.k_scale, p.v_scale = _ptr(k_scale), _ptr(v_scale)
    p.window = int(window)
    B, H, D = q.shape
    p.q, p.k, p.v = _ptr(q), _ptr(k), _ptr(v)
    p.block_table = _ptr(block_table)
    p.seqlens = _ptr(seqlens)
    p.batch, p.num_heads, p.head_dim = B, H, D
    p.num_kv_heads = k.shape[1]
    if block_table is None:
        p.capacity = k.shape[2]
    else:
        p.num_pages = k.shape[0]
        p.max_blocks = block_table.shape[1]
    p.scale = float(scale) if scale else 0.0
    p.out = _ptr(out)
    p.out_dtype = _dtype_code(out.dtype) if out is not None else F32
    p.lse = _ptr(lse)
    p.error_flag = _ptr(error_flag)
    p.max_ctas = int(max_ctas)
    if workspace is not None:
        p.workspace = _ptr(workspace)
        p.workspace_bytes = workspace.numel() * workspace.element_size()
    return p


def gqa_workspace_bytes(q, k, v, seqlens, block_table=None, max_ctas=0, window=0) -> int:
    lib = load()
    p = gqa_params(q, k, v, seqlens, block_table, max_ctas=max_ctas, window=window)
    n = lib.kvdec_gqa_workspace_bytes(ctypes.byref(p))
    if n == 0:
        raise KvdecError("kvdec_gqa_workspace_bytes: " + lib.kvdec_last_error().decode())
    return n


def gqa_decode(q, k, v, seqlens, block_table=None, scale=None, out_dtype=torch.float32,
               out=None, return_lse=True, error_flag=None, max_ctas=0, workspace=None,
               stream=None, k_scale=None, v_scale=None, window=0):
    """MHA/GQA/MQA decode.  q [B,h,d] bf16; k, v contiguous [B,n_kv,cap,d] or
    paged [pages,n_kv,64,d] (with block_table [B,max_blocks] int32), bf16 or
    E4M3 bytes with fp32 k_scale, v_scale [n_kv]; seqlens [B] int32;
    window > 0 reads a ring cache of the last ``window`` tokens.  Returns
    (out [B,h,d], lse [B,h] or None)."""
    lib = load()
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", k.dtype, dev)
    _kv_format(k, v, k_scale, v_scale, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, dev)
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=dev)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev) if return_lse else None
    p = gqa_params(q, k, v, seqlens, block_table, scale, out, lse, error_flag, max_ctas,
                   k_scale=k_scale, v_scale=v_scale, window=window)
    need = lib.kvdec_gqa_workspace_bytes(ctypes.byref(p))
    if need == 0:
        raise KvdecError("kvdec_gqa_decode: " + lib.kvdec_last_error().decode())
    if workspace is None:
        workspace = _default_ws.get(dev, need)
    p.workspace = _ptr(workspace)
    p.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.kvdec_gqa_decode(ctypes.byref(p), _stream(stream)), "kvdec_gqa_decode")
    return out, lse


def gqa_decode_noalloc(q, k, v, seqlens, block_table=None, scale=None,
                       out_dtype=torch.float32, out=None, return_lse=True, error_flag=None,
                       max_ctas=0, stream=None, k_scale=None, v_scale=None, window=0):
    """kvdec_gqa_decode_noalloc: the same decode for callers that cannot
    allocate device memory; the library keeps the split scratch in its own
    fixed 16 MiB array per GPU, so only inputs and outputs are passed (the
    tensors returned here are allocated by this Python helper, not by the
    library).  Calls sharing a device must not overlap on the GPU."""
    lib = load()
    dev = q.device
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", k.dtype, dev)
    _kv_format(k, v, k_scale, v_scale, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, dev)
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=dev)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev) if return_lse else None
    p = gqa_params(q, k, v, seqlens, block_table, scale, out, lse, error_flag, max_ctas,
                   k_scale=k_scale, v_scale=v_scale, window=window)
    _check(lib.kvdec_gqa_decode_noalloc(ctypes.byref(p), _stream(stream)),
           "kvdec_gqa_decode_noalloc")
    return out, lse


# ---------------------------------------------------------------- MLA

def _mla_kv_format(cache, kv_scale, dev) -> int:
    """KV_BF16 for a bf16 latent cache; KV_FP8_E4M3 for E4M3 bytes (uint8 or
    float8_e4m3fn) with fp32 [c_kv scale, k_R scale] on the same device."""
    if cache.dtype == torch.bfloat16:
        return KV_BF16
    if cache.dtype not in _FP8_DTYPES:
        raise TypeError(f"cache must be bf16 or E4M3 bytes, got {cache.dtype}")
    if kv_scale is None:
        raise ValueError("an FP8 latent cache needs kv_scale")
    _need(kv_scale, "kv_scale", torch.float32, dev)
    if kv_scale.numel() != 2:
        raise ValueError("kv_scale must hold [c_kv scale, k_R scale]")
    return KV_FP8_E4M3


def mla_params(q_abs, q_rope, cache, block_table, seqlens, scale=None, out=None, lse=None,
               error_flag=None, max_ctas=0, kv_scale=None):
    p = MlaParams()
    if cache.dtype in _FP8_DTYPES:
        p.kv_format = KV_FP8_E4M3
        p.kv_scale = _ptr(kv_scale)
    B, H, _ = q_abs.shape
    p.q_absorbed, p.q_rope, p.cache = _ptr(q_abs), _ptr(q_rope), _ptr(cache)
    p.block_table, p.seqlens = _ptr(block_table), _ptr(seqlens)
    p.batch, p.num_heads = B, H
    p.num_pages, p.max_blocks = cache.shape[0], block_table.shape[1]
    p.scale = float(scale) if scale else 0.0
    p.out = _ptr(out)
    p.out_dtype = _dtype_code(out.dtype) if out is not None else F32
    p.lse = _ptr(lse)
    p.error_flag = _ptr(error_flag)
    p.max_ctas = int(max_ctas)
    return p


def mla_decode_absorbed(q_abs, q_rope, cache, block_table, seqlens, scale=None,
                        out_dtype=torch.float32, out=None, return_lse=True, error_flag=None,
                        max_ctas=0, workspace=None, stream=None, kv_scale=None):
    """MLA absorbed decode.  q_abs [B,128,512], q_rope [B,128,64] bf16; cache
    [pages,64,576] bf16, or E4M3 bytes (uint8 / float8_e4m3fn) with kv_scale
    = fp32 [c_kv scale, k_R scale]; block_table [B,max_blocks] and seqlens
    [B] int32.  Returns (out [B,128,512] latent, lse [B,128] or None)."""
    lib = load()
    dev = q_abs.device
    for t, n in [(q_abs, "q_abs"), (q_rope, "q_rope")]:
        _need(t, n, torch.bfloat16, dev)
    _need(cache, "cache", cache.dtype, dev)
    _mla_kv_format(cache, kv_scale, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    if out is None:
        out = torch.empty(q_abs.shape, dtype=out_dtype, device=dev)
    lse = torch.empty(q_abs.shape[:2], dtype=torch.float32, device=dev) if return_lse else None
    p = mla_params(q_abs, q_rope, cache, block_table, seqlens, scale, out, lse, error_flag, max_ctas,
                   kv_scale)
    need = lib.kvdec_mla_workspace_bytes(ctypes.byref(p))
    if need == 0:
        raise KvdecError("kvdec_mla_decode_absorbed: " + lib.kvdec_last_error().decode())
    if workspace is None:
        workspace = _default_ws.get(dev, need)
    p.workspace = _ptr(workspace)
    p.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.kvdec_mla_decode_absorbed(ctypes.byref(p), _stream(stream)),
           "kvdec_mla_decode_absorbed")
    return out, lse


# ---------------------------------------------------------------- append

def append_rope_mla(cache, block_table, seqlens, c_kv, k_rope, rope_theta=10000.0,
                    error_flag=None, stream=None, kv_scale=None):
    """Write [c_kv ; RoPE_pos(k_rope)] at slot seqlens[b] of the paged latent
    cache (in place).  The caller increments seqlens afterwards.  An E4M3
    cache (uint8 / float8_e4m3fn) stores the codes of c_kv / kv_scale[0] and
    RoPE(k_rope) / kv_scale[1]."""
    lib = load()
    dev = cache.device
    for t, n in [(c_kv, "c_kv"), (k_rope, "k_rope")]:
        _need(t, n, torch.bfloat16, dev)
    _need(cache, "cache", cache.dtype, dev)
    fmt = _mla_kv_format(cache, kv_scale, dev)
    _need(block_table, "block_table", torch.int32, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    p = AppendParams()
    p.mode = APPEND_MLA
    p.kv_format = fmt
    if fmt == KV_FP8_E4M3:
        p.k_scale = _ptr(kv_scale)
    p.batch = c_kv.shape[0]
    p.seqlens, p.block_table = _ptr(seqlens), _ptr(block_table)
    p.num_pages, p.max_blocks = cache.shape[0], block_table.shape[1]
    p.rope_theta = rope_theta
    p.c_kv, p.k_rope, p.cache = _ptr(c_kv), _ptr(k_rope), _ptr(cache)
    p.error_flag = _ptr(error_flag)
    _check(lib.kvdec_append_rope(ctypes.byref(p), _stream(stream)), "kvdec_append_rope")


def append_rope_gqa(k, v, seqlens, k_new, v_new, block_table=None, rope_theta=10000.0,
                    error_flag=None, stream=None, k_scale=None, v_scale=None, window=0):
    """K[.., slot, :] = RoPE_pos(k_new), V[.., slot, :] = v_new at pos =
    seqlens[b] (in place), contiguous or paged caches; slot = pos, or pos mod
    window for a ring cache.  E4M3 caches (uint8 / float8_e4m3fn k, v) store
    the codes of the values divided by k_scale / v_scale [n_kv]."""
    lib = load()
    dev = k.device
    for t, n in [(k_new, "k_new"), (v_new, "v_new")]:
        _need(t, n, torch.bfloat16, dev)
    _need(k, "k", k.dtype, dev)
    fmt = _kv_format(k, v, k_scale, v_scale, dev)
    _need(seqlens, "seqlens", torch.int32, dev)
    p = AppendParams()
    p.mode = APPEND_GQA
    p.kv_format = fmt
    p.window = int(window)
    if fmt == KV_FP8_E4M3:
        p.k_scale, p.v_scale = _ptr(k_scale), _ptr(v_scale)
    p.batch = k_new.shape[0]
    p.seqlens = _ptr(seqlens)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, dev)
        p.block_table = _ptr(block_table)
        p.num_pages, p.max_blocks = k.shape[0], block_table.shape[1]
    else:
        p.capacity = k.shape[2]
    p.rope_theta = rope_theta
    p.k_new, p.v_new, p.k, p.v = _ptr(k_new), _ptr(v_new), _ptr(k), _ptr(v)
    p.num_kv_heads, p.head_dim = k_new.shape[1], k_new.shape[2]
    p.error_flag = _ptr(error_flag)
    _check(lib.kvdec_append_rope(ctypes.byref(p), _stream(stream)), "kvdec_append_rope")


# ---------------------------------------------------------------- combine

def combine_splits(partial_o, partial_lse, split_counts=None, out_dtype=torch.float32,
                   out=None, return_lse=True, stream=None):
    """partial_o [S, R, D] fp32 (normalised), partial_lse [S, R] fp32,
    split_counts [R] int32 or None.  Returns (out [R, D], lse [R])."""
    lib = load()
    dev = partial_o.device
    _need(partial_o, "partial_o", torch.float32, dev)
    _need(partial_lse, "partial_lse", torch.float32, dev)
    S, R, D = partial_o.shape
    if split_counts is not None:
        _need(split_counts, "split_counts", torch.int32, dev)
    if out is None:
        out = torch.empty((R, D), dtype=out_dtype, device=dev)
    lse = torch.empty(R, dtype=torch.float32, device=dev) if return_lse else None
    p = CombineParams()
    p.partial_o, p.partial_lse = _ptr(partial_o), _ptr(partial_lse)
    p.split_counts = _ptr(split_counts)
    p.num_splits, p.rows, p.head_dim = S, R, D
    p.out_dtype = _dtype_code(out.dtype)
    p.out, p.lse = _ptr(out), _ptr(lse)
    _check(lib.kvdec_combine_splits(ctypes.byref(p), _stream(stream)), "kvdec_combine_splits")
    return out, lse


def _mla_proj(fn, name, x, w, width, out_dtype, out, stream):
    lib = load()
    dev = x.device
    _need(x, "x", torch.bfloat16, dev)
    _need(w, "w", torch.bfloat16, dev)
    B, H, _ = x.shape
    if tuple(w.shape) != (H, 128, 512):
        raise ValueError(f"{name}: w must be [{H}, 128, 512], got {tuple(w.shape)}")
    if out is None:
        out = torch.empty((B, H, width), dtype=out_dtype, device=dev)
    p = MlaProjParams()
    p.x, p.w, p.y = _ptr(x), _ptr(w), _ptr(out)
    p.batch, p.num_heads = B, H
    p.out_dtype = _dtype_code(out.dtype)
    _check(getattr(lib, fn)(ctypes.byref(p), _stream(stream)), fn)
    return out


def mla_absorb_q(q_nope, W_UK, out_dtype=torch.bfloat16, out=None, stream=None):
    """q_absorbed[b,h] = W_UK[h]^T q_nope[b,h]: q_nope [B,H,128] bf16, W_UK
    [H,128,512] bf16 -> [B,H,512] (bf16 by default: the decode's input)."""
    if q_nope.shape[-1] != 128:
        raise ValueError("mla_absorb_q: q_nope must be [B, H, 128]")
    return _mla_proj("kvdec_mla_absorb_q", "mla_absorb_q", q_nope, W_UK, 512, out_dtype, out, stream)


def mla_project_out(latent, W_UV, out_dtype=torch.float32, out=None, stream=None):
    """out[b,h] = W_UV[h] latent[b,h]: latent [B,H,512] bf16, W_UV [H,128,512]
    bf16 -> [B,H,128]."""
    if latent.shape[-1] != 512:
        raise ValueError("mla_project_out: latent must be [B, H, 512]")
    return _mla_proj("kvdec_mla_project_out", "mla_project_out", latent, W_UV, 128, out_dtype, out, stream)


def selftest_wait_timeout(timeout_ns: int, error_flag, stream=None):
    lib = load()
    _check(lib.kvdec_selftest_wait_timeout(timeout_ns, _ptr(error_flag), _stream(stream)),
           "kvdec_selftest_wait_timeout")


# ---------------------------------------------------------------- MLA prefill (non-absorbed)

def mla_prefill_expand(c_kv, W_UK, W_UV, stream=None):
    """kvdec_mla_prefill_expand: k_nope[t,h] = W_UK[h] c_kv[t], v[t,h] =
    W_UV[h] c_kv[t].  c_kv [s, 512] bf16; W_UK, W_UV [n_h, 128, 512] bf16.
    Returns (k_nope, v), bf16 [s, n_h, 128]."""
    lib = load()
    dev = c_kv.device
    for t, n in [(c_kv, "c_kv"), (W_UK, "W_UK"), (W_UV, "W_UV")]:
        _need(t, n, torch.bfloat16, dev)
    s_len, n_h = c_kv.shape[0], W_UK.shape[0]
    k_nope = torch.empty((s_len, n_h, 128), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k_nope)
    p = MlaExpandParams()
    p.c_kv, p.w_uk, p.w_uv, p.k_nope, p.v = _ptr(c_kv), _ptr(W_UK), _ptr(W_UV), _ptr(k_nope), _ptr(v)
    p.s, p.num_heads = s_len, n_h
    _check(lib.kvdec_mla_prefill_expand(ctypes.byref(p), _stream(stream)), "kvdec_mla_prefill_expand")
    return k_nope, v


def mla_prefill(q_nope, q_rope, k_nope, k_rope, v, kv_offset=-1, scale=None,
                out_dtype=torch.float32, return_lse=True, stream=None):
    """kvdec_mla_prefill: causal attention of a prefill chunk on the
    non-absorbed path.  q_nope [s_q, n_h, 128], q_rope [s_q, n_h, 64],
    k_nope, v [s_kv, n_h, 128], k_rope [s_kv, 64], all bf16; query i sits at
    position kv_offset + i (kv_offset < 0: s_kv - s_q).  Returns (out
    [s_q, n_h, 128], lse [s_q, n_h] or None)."""
    lib = load()
    dev = q_nope.device
    for t, n in [(q_nope, "q_nope"), (q_rope, "q_rope"), (k_nope, "k_nope"), (k_rope, "k_rope"), (v, "v")]:
        _need(t, n, torch.bfloat16, dev)
    s_q, n_h, _ = q_nope.shape
    out = torch.empty((s_q, n_h, 128), dtype=out_dtype, device=dev)
    lse = torch.empty((s_q, n_h), dtype=torch.float32, device=dev) if return_lse else None
    p = MlaPrefillParams()
    p.q_nope, p.q_rope, p.k_nope, p.k_rope, p.v = (_ptr(q_nope), _ptr(q_rope), _ptr(k_nope),
                                                    _ptr(k_rope), _ptr(v))
    p.s_q, p.s_kv, p.num_heads, p.kv_offset = s_q, k_nope.shape[0], n_h, int(kv_offset)
    p.scale = float(scale) if scale else 0.0
    p.out_dtype = _dtype_code(out.dtype)
    p.out, p.lse = _ptr(out), _ptr(lse)
    _check(lib.kvdec_mla_prefill(ctypes.byref(p), _stream(stream)), "kvdec_mla_prefill")
    return out, lse
