"""Python binding of the GB300 attention-forward C ABI (``include/attn.h``).

The functions here carry the same names as the C entry points and only marshal
arguments: they check tensor dtypes, devices and shapes, allocate outputs the caller
did not pass, and hand raw device pointers and the current CUDA stream to
``libattn_gb300.so``.  Every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if the library is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "AttnError", "ATTN_BF16", "ATTN_F32", "library_path", "load_library",
    "attn_fwd_prefill", "attn_fwd_decode", "attn_decode_workspace_bytes",
    "attn_prefill_workspace_bytes",
    "attn_gen_mask_decode", "attn_get_device_error", "attn_status_string",
    "attn_fwd_decode_static_ws",
]

ATTN_BF16, ATTN_F32 = 0, 1
_STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
           4: "ATTN_ERR_PAGE_OOB", 5: "ATTN_ERR_DEVICE_TIMEOUT", 6: "ATTN_ERR_WORKSPACE",
           7: "ATTN_ERR_CACHE_LEN"}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}")


def library_path() -> str:
    from . import _build

    return _build.LIB


ATTN_KV_BF16, ATTN_KV_E4M3 = 0, 1


class AttnOpts(ctypes.Structure):
    """attn_opts of attn.h: optional features of the _ex calls."""
    _fields_ = [("sink", ctypes.c_void_p), ("kv_dtype", ctypes.c_int),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("window", ctypes.c_int), ("circular", ctypes.c_int),
                ("rope_inv_freq", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
                ("cu_seqlens_k", ctypes.c_void_p), ("nseq", ctypes.c_int),
                ("prefill_workspace", ctypes.c_void_p),
                ("prefill_workspace_bytes", ctypes.c_size_t)]


def load_library(build_if_missing: bool = False):
    """Load libattn_gb300.so (building it first only if asked).  Raises if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing:
            from . import _build

            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(the attention path has no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        O = ctypes.POINTER(AttnOpts)
        lib.attn_fwd_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P]
        lib.attn_fwd_prefill.restype = I
        lib.attn_fwd_prefill_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, O, P]
        lib.attn_fwd_prefill_ex.restype = I
        lib.attn_prefill_workspace_bytes.argtypes = [I]
        lib.attn_prefill_workspace_bytes.restype = S
        lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.attn_decode_workspace_bytes.restype = S
        lib.attn_fwd_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P, I, I, P,
                                        S, P]
        lib.attn_fwd_decode.restype = I
        lib.attn_fwd_decode_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, P, P, I, I,
                                           O, P, S, P]
        lib.attn_fwd_decode_ex.restype = I
        lib.attn_append_kv.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, O, P]
        lib.attn_append_kv.restype = I
        lib.attn_fwd_decode_static_ws.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, F,
                                                  P, P, I, I, P]
        lib.attn_fwd_decode_static_ws.restype = I
        lib.attn_gen_mask_decode.argtypes = [P, I, I, I, I, P, P]
        lib.attn_gen_mask_decode.restype = I
        lib.attn_check_wait_timeout.argtypes = [ctypes.c_longlong, P]
        lib.attn_check_wait_timeout.restype = I
        lib.attn_get_device_error.argtypes = [P]
        lib.attn_get_device_error.restype = I
        lib.attn_status_string.argtypes = [I]
        lib.attn_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise AttnError(status, where)


def _stream_ptr(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _req(t, name, dtype, device=None):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dtype_code(dtype):
    import torch

    if dtype == torch.bfloat16:
        return ATTN_BF16
    if dtype == torch.float32:
        return ATTN_F32
    raise TypeError("output dtype must be torch.bfloat16 or torch.float32")


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_check_wait_timeout(wait_cycles: int, stream=None) -> None:
    """Launch the failure-path check: a bounded wait on a phase nothing completes, which
    sets the device timeout word (read it with attn_get_device_error)."""
    _check(load_library().attn_check_wait_timeout(int(wait_cycles), _stream_ptr(stream)),
           "attn_check_wait_timeout")


def attn_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device error status."""
    return load_library().attn_get_device_error(_stream_ptr(stream))


def _prefill_marshal(q, k, v, o, lse, o_dtype):
    import torch

    _req(q, "q", torch.bfloat16)
    _req(k, "k", torch.bfloat16, q.device)
    _req(v, "v", torch.bfloat16, q.device)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [b,hq,sq,d]; k and v [b,hkv,skv,d] with equal shapes")
    b, hq, sq, d = q.shape
    _, hkv, skv, dk = k.shape
    if k.shape[0] != b or dk != d:
        raise ValueError("q and k disagree on batch or head_dim")
    if o is None:
        o = torch.empty((b, hq, sq, d), dtype=o_dtype or torch.bfloat16, device=q.device)
    _req(o, "o", o.dtype, q.device)
    if tuple(o.shape) != (b, hq, sq, d):
        raise ValueError("o has the wrong shape")
    if lse is not None:
        _req(lse, "lse", torch.float32, q.device)
        if tuple(lse.shape) != (b, hq, sq):
            raise ValueError("lse must be [b,hq,sq]")
    return o, (b, hq, hkv, sq, skv, d)


def _opts(sink, hq, device, kv_dtype=ATTN_KV_BF16, k_scale=1.0, v_scale=1.0, window=0,
          circular=False, rope_inv_freq=None, d=None):
    """attn_opts for the _ex calls: sink is an fp32 tensor [hq] on the device, or None;
    rope_inv_freq an fp32 tensor [d/2] on the device, or None."""
    import torch

    if sink is not None:
        _req(sink, "sink", torch.float32, device)
        if tuple(sink.shape) != (hq,):
            raise ValueError("sink must hold one fp32 logit per query head: shape [hq]")
    if rope_inv_freq is not None:
        _req(rope_inv_freq, "rope_inv_freq", torch.float32, device)
        if tuple(rope_inv_freq.shape) != (d // 2,):
            raise ValueError("rope_inv_freq must be fp32 [d/2]")
    return AttnOpts(sink=None if sink is None else sink.data_ptr(), kv_dtype=kv_dtype,
                    k_scale=float(k_scale), v_scale=float(v_scale), window=int(window),
                    circular=int(bool(circular)),
                    rope_inv_freq=None if rope_inv_freq is None else rope_inv_freq.data_ptr())


def attn_fwd_prefill(q, k, v, *, causal: bool, window: int = 0, scale: float | None = None,
                     o=None, lse=None, o_dtype=None, stream=None):
    """O, LSE of softmax(scale Q K^T + mask) V.  q [b,hq,sq,d], k/v [b,hkv,skv,d] bf16."""
    lib = load_library()
    o, (b, hq, hkv, sq, skv, d) = _prefill_marshal(q, k, v, o, lse, o_dtype)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(lib.attn_fwd_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), b, hq, hkv, sq,
                                skv, d, sc, int(bool(causal)), int(window), _dtype_code(o.dtype),
                                _stream_ptr(stream)), "attn_fwd_prefill")
    return o, lse


def attn_fwd_prefill_ex(q, k, v, *, causal: bool, window: int = 0, scale: float | None = None,
                        o=None, lse=None, o_dtype=None, sink=None, cu_seqlens_q=None,
                        cu_seqlens_k=None, balance: bool = True, workspace=None, stream=None):
    """attn_fwd_prefill with the attn_opts options: sink, an fp32 [hq] tensor of
    per-query-head sink logits (scaled-score units) on q's device, or None; and packed
    sequences: cu_seqlens_q / cu_seqlens_k int32 [nseq + 1] offsets along sq and skv of a
    b = 1 problem (each sequence its own problem, queries at the tail of its keys).  With
    packed sequences and balance, the library's work order (query units by sequence, then
    by KV-tile count) goes to `workspace` (a uint8 tensor of attn_prefill_workspace_bytes(sq)
    bytes on q's device; allocated here when None); results do not depend on it."""
    import torch

    lib = load_library()
    o, (b, hq, hkv, sq, skv, d) = _prefill_marshal(q, k, v, o, lse, o_dtype)
    opts = _opts(sink, hq, q.device)
    if cu_seqlens_q is not None or cu_seqlens_k is not None:
        if cu_seqlens_q is None or cu_seqlens_k is None:
            raise ValueError("packed sequences need both cu_seqlens_q and cu_seqlens_k")
        _req(cu_seqlens_q, "cu_seqlens_q", torch.int32, q.device)
        _req(cu_seqlens_k, "cu_seqlens_k", torch.int32, q.device)
        if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape != cu_seqlens_k.shape:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must be int32 [nseq + 1]")
        opts.cu_seqlens_q = cu_seqlens_q.data_ptr()
        opts.cu_seqlens_k = cu_seqlens_k.data_ptr()
        opts.nseq = cu_seqlens_q.shape[0] - 1
        if balance and sq > 0:
            nbytes = lib.attn_prefill_workspace_bytes(sq)
            if workspace is None:
                ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
                if stream is not None:
                    ws.record_stream(stream)  # freed only once the call on `stream` is done
            else:
                _req(workspace, "workspace", torch.uint8, q.device)
                ws = workspace
                if ws.numel() < nbytes:
                    raise ValueError(f"workspace holds {ws.numel()} bytes, {nbytes} needed")
            opts.prefill_workspace = ws.data_ptr()
            opts.prefill_workspace_bytes = nbytes
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(lib.attn_fwd_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), b, hq, hkv, sq,
                                   skv, d, sc, int(bool(causal)), int(window),
                                   _dtype_code(o.dtype), ctypes.byref(opts), _stream_ptr(stream)),
           "attn_fwd_prefill_ex")
    return o, lse


def _decode_marshal(q, k_cache, v_cache, block_table, cache_len, max_cache_len, o, lse,
                    o_dtype, cache_dtype=None, want_o=True):
    import torch

    _req(q, "q", torch.bfloat16)
    dev = q.device
    cache_dtype = cache_dtype or torch.bfloat16
    _req(k_cache, "k_cache", cache_dtype, dev)
    _req(v_cache, "v_cache", cache_dtype, dev)
    _req(cache_len, "cache_len", torch.int32, dev)
    if v_cache.shape != k_cache.shape or q.dim() != 4 or k_cache.dim() != 4:
        raise ValueError("bad q / cache shapes")
    b, hq, s_active, d = q.shape
    if block_table is not None:
        _req(block_table, "block_table", block_table.dtype, dev)
        if block_table.dtype not in (torch.int32, torch.uint32):
            raise TypeError("block_table must hold 32-bit entries (uint32 bit patterns)")
        if block_table.dim() != 2 or block_table.shape[0] != b:
            raise ValueError("block_table must be [b, max_pages_per_seq]")
        num_pages, hkv, page, dk = k_cache.shape
        max_pages = block_table.shape[1]
    else:
        bb, hkv, ml, dk = k_cache.shape
        if bb != b or ml != max_cache_len:
            raise ValueError("a flat cache must be [b, hkv, max_cache_len, d]")
        num_pages, page, max_pages = 0, 0, 0
    if dk != d or cache_len.shape != (b,):
        raise ValueError("head_dim or cache_len shape mismatch")
    if want_o:
        if o is None:
            o = torch.empty((b, hq, s_active, d), dtype=o_dtype or torch.bfloat16, device=dev)
        _req(o, "o", o.dtype, dev)
    if lse is not None:
        _req(lse, "lse", torch.float32, dev)
    dims = (b, hq, hkv, d, s_active, page, max_pages, num_pages, max_cache_len)
    return o, dims


def attn_fwd_decode_static_ws(q, k_cache, v_cache, block_table, cache_len, *,
                              max_cache_len: int, scale: float | None = None, o=None, lse=None,
                              o_dtype=None, kv_chunk: int = 0, stream=None):
    """attn_fwd_decode without a workspace argument, for callers that cannot allocate
    device memory: the split-KV scratch is the library's fixed 64 MiB device array.
    Calls sharing it must not overlap on the GPU.  Same layouts as attn_fwd_decode."""
    lib = load_library()
    o, (b, hq, hkv, d, s_active, page, max_pages, num_pages, mcl) = _decode_marshal(
        q, k_cache, v_cache, block_table, cache_len, max_cache_len, o, lse, o_dtype)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(lib.attn_fwd_decode_static_ws(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                         _ptr(cache_len), b, hq, hkv, d, s_active, page, max_pages,
                                         num_pages, mcl, sc, _ptr(o), _ptr(lse),
                                         _dtype_code(o.dtype), kv_chunk, _stream_ptr(stream)),
           "attn_fwd_decode_static_ws")
    return o, lse


def attn_prefill_workspace_bytes(sq: int) -> int:
    return int(load_library().attn_prefill_workspace_bytes(sq))


def attn_decode_workspace_bytes(b: int, hq: int, s_active: int, d: int, max_cache_len: int,
                                kv_chunk: int = 0) -> int:
    return int(load_library().attn_decode_workspace_bytes(b, hq, s_active, d, max_cache_len,
                                                           kv_chunk))


def attn_fwd_decode(q, k_cache, v_cache, block_table, cache_len, *, max_cache_len: int,
                    scale: float | None = None, o=None, lse=None, o_dtype=None, kv_chunk: int = 0,
                    workspace=None, stream=None):
    """Decode attention.  q [b,hq,s_active,d] bf16; paged caches [num_pages,hkv,page,d] with
    block_table int32/uint32-bits [b,max_pages], or flat caches [b,hkv,max_cache_len,d] with
    block_table None; cache_len int32 [b]."""
    lib = load_library()
    o, (b, hq, hkv, d, s_active, page, max_pages, num_pages, mcl) = _decode_marshal(
        q, k_cache, v_cache, block_table, cache_len, max_cache_len, o, lse, o_dtype)
    workspace = _decode_workspace(workspace, b, hq, s_active, d, mcl, kv_chunk, q.device)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(lib.attn_fwd_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                               _ptr(cache_len), b, hq, hkv, d, s_active, page, max_pages,
                               num_pages, mcl, sc, _ptr(o), _ptr(lse), _dtype_code(o.dtype),
                               kv_chunk, _ptr(workspace), workspace.numel(), _stream_ptr(stream)),
           "attn_fwd_decode")
    return o, lse


def _decode_workspace(workspace, b, hq, s_active, d, max_cache_len, kv_chunk, dev):
    import torch

    need = attn_decode_workspace_bytes(b, hq, s_active, d, max_cache_len, kv_chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _req(workspace, "workspace", torch.uint8, dev)
    return workspace


def attn_fwd_decode_ex(q, k_cache, v_cache, block_table, cache_len, *, max_cache_len: int,
                       scale: float | None = None, o=None, lse=None, o_dtype=None,
                       kv_chunk: int = 0, sink=None, k_scale: float = 1.0, v_scale: float = 1.0,
                       window: int = 0, circular: bool = False, rope_inv_freq=None,
                       workspace=None, stream=None):
    """attn_fwd_decode with the attn_opts options: sink, an fp32 [hq] tensor of
    per-query-head sink logits (scaled-score units) on q's device, or None; and an e4m3
    cache: k_cache and v_cache of dtype torch.float8_e4m3fn (or their bytes as uint8),
    where element x stands for e4m3(x) * k_scale (K) or e4m3(x) * v_scale (V); a window;
    a circular flat cache (max_cache_len rows, cache_len may exceed it); and RoPE of the
    queries (rope_inv_freq fp32 [d/2])."""
    import torch

    lib = load_library()
    fp8 = k_cache.dtype in (torch.float8_e4m3fn, torch.uint8)
    o, (b, hq, hkv, d, s_active, page, max_pages, num_pages, mcl) = _decode_marshal(
        q, k_cache, v_cache, block_table, cache_len, max_cache_len, o, lse, o_dtype,
        cache_dtype=k_cache.dtype if fp8 else None)
    workspace = _decode_workspace(workspace, b, hq, s_active, d, mcl, kv_chunk, q.device)
    opts = _opts(sink, hq, q.device, ATTN_KV_E4M3 if fp8 else ATTN_KV_BF16, k_scale, v_scale,
                 window, circular, rope_inv_freq, d)
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    _check(lib.attn_fwd_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                  _ptr(cache_len), b, hq, hkv, d, s_active, page, max_pages,
                                  num_pages, mcl, sc, _ptr(o), _ptr(lse), _dtype_code(o.dtype),
                                  kv_chunk, ctypes.byref(opts), _ptr(workspace),
                                  workspace.numel(), _stream_ptr(stream)), "attn_fwd_decode_ex")
    return o, lse


def attn_append_kv(k_new, v_new, k_cache, v_cache, block_table, cache_len, *,
                   max_cache_len: int, circular: bool = False, rope_inv_freq=None, stream=None):
    """Write the new tokens' K (RoPE'd with rope_inv_freq, if given) and V into a bf16 cache:
    k_new, v_new bf16 [b, hkv, s_active, d]; token t at logical position
    cache_len[b] - s_active + t.  Caches and block_table as for attn_fwd_decode."""
    import torch

    lib = load_library()
    _req(k_new, "k_new", torch.bfloat16)
    dev = k_new.device
    _req(v_new, "v_new", torch.bfloat16, dev)
    if k_new.dim() != 4 or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [b, hkv, s_active, d] with equal shapes")
    b, hkv, s_active, d = k_new.shape
    # the new tokens' shape stands in for q: one row per (sequence, kv head, new token)
    _, (_, _, hkv2, _, _, page, max_pages, num_pages, mcl) = _decode_marshal(
        k_new, k_cache, v_cache, block_table, cache_len, max_cache_len, None, None, None,
        want_o=False)
    if hkv2 != hkv:
        raise ValueError("k_new and the cache disagree on kv heads")
    opts = _opts(None, hkv, dev, circular=circular, rope_inv_freq=rope_inv_freq, d=d)
    _check(lib.attn_append_kv(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                              _ptr(block_table), _ptr(cache_len), b, hkv, d, s_active, page,
                              max_pages, num_pages, mcl, ctypes.byref(opts), _stream_ptr(stream)),
           "attn_append_kv")


def attn_gen_mask_decode(cache_len, hq: int, s_active: int, max_len: int, mask=None,
                         stream=None):
    """uint8 [b, hq, s_active, max_len] 0/1 decode mask."""
    import torch

    lib = load_library()
    _req(cache_len, "cache_len", torch.int32)
    b = cache_len.shape[0]
    if mask is None:
        mask = torch.empty((b, hq, s_active, max_len), dtype=torch.uint8, device=cache_len.device)
    _req(mask, "mask", torch.uint8, cache_len.device)
    _check(lib.attn_gen_mask_decode(_ptr(cache_len), b, hq, s_active, max_len, _ptr(mask),
                                    _stream_ptr(stream)), "attn_gen_mask_decode")
    return mask
