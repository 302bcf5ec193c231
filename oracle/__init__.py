"""fp64 CPU oracle for the attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and
its ``--impl reference`` arm) may import this package.  The attention library never
does: it shares no code, header, table or helper with this directory.

The arithmetic lives in ``attn_oracle.c`` (plain loops in double, the full score row
materialised, then softmax, then P.V).  This module only compiles it with gcc,
marshals numpy arrays into it, and spreads independent heads or rows over a thread
pool (ctypes releases the GIL during each call).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORACLE_ERRORS = {1: "invalid argument", 2: "page index out of range", 3: "out of memory"}


_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]
_STAMP = _LIB_PATH + ".stamp"


def _fingerprint() -> str:
    """The source, the flags, gcc's version and the machine: a library built from anything
    else (a copied tree, another architecture) is rebuilt."""
    h = hashlib.sha256()
    with open(_SRC, "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(_CFLAGS).encode())
    h.update(platform.machine().encode())
    h.update(subprocess.run(["gcc", "--version"], capture_output=True, text=True).stdout.encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (gcc, -O2, strict IEEE: no fast-math)."""
    fp = _fingerprint()
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(_STAMP):
        with open(_STAMP) as fh:
            if fh.read().strip() == fp:
                return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    with open(_STAMP + f".tmp{os.getpid()}", "w") as fh:
        fh.write(fp + "\n")
    os.replace(_STAMP + f".tmp{os.getpid()}", _STAMP)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point this at a deliberately broken build to check the pins.
            lib = ctypes.CDLL(os.environ.get("ATTN_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            L = ctypes.c_long
            I = ctypes.c_int
            D = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = D
            lib.oracle_kv_head.argtypes = [I, I, I]
            lib.oracle_kv_head.restype = I
            lib.oracle_q_pos.argtypes = [L, L, L]
            lib.oracle_q_pos.restype = L
            lib.oracle_allowed.argtypes = [L, L, L, I, L]
            lib.oracle_allowed.restype = I
            lib.oracle_attention_rows.argtypes = [P, L, P, P, L, I, D, P, I, L, P, P, P]
            lib.oracle_attention_rows.restype = I
            lib.oracle_attention_rows_sink.argtypes = [P, L, P, P, L, I, D, P, I, L, D, P, P, P]
            lib.oracle_attention_rows_sink.restype = I
            lib.oracle_prefill.argtypes = [P, P, P, I, I, I, L, L, I, D, I, L, L, L, P, P]
            lib.oracle_prefill.restype = I
            lib.oracle_prefill_sink.argtypes = [P, P, P, I, I, I, L, L, I, D, I, L, P, L, L, P, P]
            lib.oracle_prefill_sink.restype = I
            lib.oracle_prefill_varlen.argtypes = [P, P, P, I, I, I, P, P, I, D, I, L, P, L, L, P, P]
            lib.oracle_prefill_varlen.restype = I
            lib.oracle_gather_paged.argtypes = [P, P, L, I, I, I, I, L, P]
            lib.oracle_gather_paged.restype = I
            lib.oracle_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, I, L, L, L, D, L, L, P, P]
            lib.oracle_decode.restype = I
            lib.oracle_decode_sink.argtypes = [P, P, P, P, P, I, I, I, I, I, I, L, L, L, D, P, L, L,
                                               P, P]
            lib.oracle_decode_sink.restype = I
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f64.restype = D
            lib.oracle_decode_e4m3.argtypes = [P, P, P, P, P, I, I, I, I, I, I, L, L, L, D, D, D,
                                               P, L, L, P, P]
            lib.oracle_decode_e4m3.restype = I
            lib.oracle_rope_row.argtypes = [P, I, D, P]
            lib.oracle_rope_row.restype = None
            lib.oracle_decode_ext.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, L, L, L, D, L,
                                              I, P, P, L, L, P, P]
            lib.oracle_decode_ext.restype = I
            lib.oracle_decode_mask.argtypes = [P, I, I, I, L, P]
            lib.oracle_decode_mask.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle error {rc}: {ORACLE_ERRORS.get(rc, '?')}")


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "oracle inputs are bf16 bit patterns (uint16)"
    return a


def default_threads() -> int:
    return os.cpu_count() or 1


def kv_head(h: int, hq: int, hkv: int) -> int:
    return _load().oracle_kv_head(h, hq, hkv)


def q_pos(i: int, sq: int, skv: int) -> int:
    return _load().oracle_q_pos(i, sq, skv)


def allowed(j: int, skv: int, qpos: int, causal: bool, window: int) -> bool:
    return bool(_load().oracle_allowed(j, skv, qpos, int(causal), window))


def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).reshape(-1)
    return np.array([lib.oracle_bf16_to_f64(int(x)) for x in flat]).reshape(np.shape(bits))


def _sinks(sink, hq):
    """Per-query-head sink logits as a float64 array [hq], or None for no sink."""
    if sink is None:
        return None
    a = np.ascontiguousarray(sink, dtype=np.float64).reshape(-1)
    assert a.shape == (hq,), "sink holds one logit per query head"
    return a


def attention_rows(q_rows, k, v, qpos, scale, causal, window, want_p=False, sink=None):
    """Rows of one head.  q_rows [n, d], k/v [skv, d] (bf16 bits), qpos [n]; sink: the
    head's sink logit (None = no sink).

    Returns (o [n, d] float64, lse [n] float64[, p [n, skv] float64])."""
    q_rows, k, v = _u16(q_rows), _u16(k), _u16(v)
    n, d = q_rows.shape
    skv = k.shape[0]
    assert k.shape == (skv, d) and v.shape == (skv, d)
    qp = np.ascontiguousarray(qpos, dtype=np.int64).reshape(n)
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    p = np.empty((n, skv), dtype=np.float64) if want_p else None
    sk = -np.inf if sink is None else float(sink)
    _check(_load().oracle_attention_rows_sink(_ptr(q_rows), n, _ptr(k), _ptr(v), skv, d,
                                              float(scale), _ptr(qp), int(causal), int(window),
                                              sk, _ptr(o), _ptr(lse), _ptr(p)))
    return (o, lse, p) if want_p else (o, lse)


def prefill(q, k, v, scale, causal, window, threads=None, sink=None):
    """Full prefill.  q [B,HQ,SQ,D], k/v [B,HKV,SKV,D] bf16 bits -> (o f64, lse f64).
    sink: [HQ] per-query-head sink logits, or None."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, HQ, SQ, D = q.shape
    _, HKV, SKV, _ = k.shape
    sk = _sinks(sink, HQ)
    o = np.empty((B, HQ, SQ, D), dtype=np.float64)
    lse = np.empty((B, HQ, SQ), dtype=np.float64)
    lib = _load()
    nbh = B * HQ

    def run(bh):
        return lib.oracle_prefill_sink(_ptr(q), _ptr(k), _ptr(v), B, HQ, HKV, SQ, SKV, D,
                                       float(scale), int(causal), int(window), _ptr(sk), bh,
                                       bh + 1, _ptr(o), _ptr(lse))

    with ThreadPoolExecutor(max_workers=min(threads or default_threads(), nbh)) as ex:
        for rc in ex.map(run, range(nbh)):
            _check(rc)
    return o, lse


def prefill_varlen(q, k, v, cu_q, cu_k, scale, causal, window, sink=None, threads=None):
    """Packed prefill.  q [HQ,SQ,D], k/v [HKV,SKV,D] bf16 bits; cu_q, cu_k int32 [nseq+1]
    sequence offsets along SQ and SKV -> (o [HQ,SQ,D] f64, lse [HQ,SQ] f64)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    HQ, SQ, D = q.shape
    HKV, SKV, _ = k.shape
    cq = np.ascontiguousarray(cu_q, dtype=np.int32)
    ck = np.ascontiguousarray(cu_k, dtype=np.int32)
    assert cq.shape == ck.shape and cq[-1] == SQ and ck[-1] == SKV
    sk = _sinks(sink, HQ)
    o = np.zeros((HQ, SQ, D), dtype=np.float64)
    lse = np.full((HQ, SQ), -np.inf, dtype=np.float64)
    lib = _load()

    def run(h):
        return lib.oracle_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), HQ, HKV, D, _ptr(cq), _ptr(ck),
                                         cq.shape[0] - 1, float(scale), int(causal), int(window),
                                         _ptr(sk), h, h + 1, _ptr(o), _ptr(lse))

    with ThreadPoolExecutor(max_workers=min(threads or default_threads(), HQ)) as ex:
        for rc in ex.map(run, range(HQ)):
            _check(rc)
    return o, lse


def gather_paged(cache, table_row, num_pages, g, length):
    """Logical rows [0, length) of kv head g, gathered through one page-table row."""
    cache = _u16(cache)
    npg, hkv, page, d = cache.shape
    tr = np.ascontiguousarray(table_row, dtype=np.uint32)
    out = np.empty((length, d), dtype=np.uint16)
    _check(_load().oracle_gather_paged(_ptr(cache), _ptr(tr), num_pages, hkv, g, page, d, length,
                                       _ptr(out)))
    return out


def decode(q, k_cache, v_cache, table, cache_len, scale, threads=None, sink=None):
    """Decode.  q [B,HQ,s_active,D]; paged caches [num_pages,HKV,page,D] with table
    [B,max_pages] uint32, or flat caches [B,HKV,max_len,D] with table None.
    sink: [HQ] per-query-head sink logits, or None."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    B, HQ, SA, D = q.shape
    sk = _sinks(sink, HQ)
    cl = np.ascontiguousarray(cache_len, dtype=np.int32)
    if table is not None:
        table = np.ascontiguousarray(table, dtype=np.uint32)
        num_pages, HKV, page, _ = k_cache.shape
        max_pages, max_len = table.shape[1], 0
    else:
        _, HKV, max_len, _ = k_cache.shape
        num_pages, page, max_pages = 0, 1, 0
    o = np.empty((B, HQ, SA, D), dtype=np.float64)
    lse = np.empty((B, HQ, SA), dtype=np.float64)
    lib = _load()

    def run(bh):
        return lib.oracle_decode_sink(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(table),
                                      _ptr(cl), B, HQ, HKV, D, SA, page, max_pages, num_pages,
                                      max_len, float(scale), _ptr(sk), bh, bh + 1, _ptr(o),
                                      _ptr(lse))

    with ThreadPoolExecutor(max_workers=min(threads or default_threads(), B * HQ)) as ex:
        for rc in ex.map(run, range(B * HQ)):
            _check(rc)
    return o, lse


def e4m3_to_f64(codes) -> np.ndarray:
    """e4m3 byte codes -> float64 values (NaN for the NaN codes)."""
    lib = _load()
    flat = np.asarray(codes, dtype=np.uint8).reshape(-1)
    return np.array([lib.oracle_e4m3_to_f64(int(x)) for x in flat]).reshape(np.shape(codes))


def decode_e4m3(q, k_cache, v_cache, table, cache_len, scale, k_scale, v_scale, threads=None,
                sink=None):
    """Decode over an e4m3 cache.  q [B,HQ,s_active,D] bf16 bits; caches of e4m3 bytes
    (uint8), paged [num_pages,HKV,page,D] with table [B,max_pages], or flat
    [B,HKV,max_len,D] with table None; a cache byte stands for e4m3(byte) * k_scale (K) or
    * v_scale (V).  sink: [HQ] per-query-head sink logits, or None."""
    q = _u16(q)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
    B, HQ, SA, D = q.shape
    sk = _sinks(sink, HQ)
    cl = np.ascontiguousarray(cache_len, dtype=np.int32)
    if table is not None:
        table = np.ascontiguousarray(table, dtype=np.uint32)
        num_pages, HKV, page, _ = k_cache.shape
        max_pages, max_len = table.shape[1], 0
    else:
        _, HKV, max_len, _ = k_cache.shape
        num_pages, page, max_pages = 0, 1, 0
    o = np.empty((B, HQ, SA, D), dtype=np.float64)
    lse = np.empty((B, HQ, SA), dtype=np.float64)
    lib = _load()

    def run(bh):
        return lib.oracle_decode_e4m3(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(table),
                                      _ptr(cl), B, HQ, HKV, D, SA, page, max_pages, num_pages,
                                      max_len, float(scale), float(k_scale), float(v_scale),
                                      _ptr(sk), bh, bh + 1, _ptr(o), _ptr(lse))

    with ThreadPoolExecutor(max_workers=min(threads or default_threads(), B * HQ)) as ex:
        for rc in ex.map(run, range(B * HQ)):
            _check(rc)
    return o, lse


def rope_row(x, pos, inv_freq):
    """Half-split RoPE of one row (float64 [d]) at position pos; returns a new array."""
    x = np.array(x, dtype=np.float64)
    f = np.ascontiguousarray(inv_freq, dtype=np.float64)
    assert f.shape == (x.shape[0] // 2,)
    _load().oracle_rope_row(_ptr(x), x.shape[0], float(pos), _ptr(f))
    return x


def decode_ext(q, k_cache, v_cache, table, cache_len, scale, window=0, circular=False,
               k_new=None, v_new=None, inv_freq=None, sink=None, threads=None):
    """Decode with a window (and a circular flat cache), new tokens' K/V given apart from
    the cache, RoPE and a sink (see oracle_decode_ext).  q [B,HQ,s_active,D] and the caches
    are bf16 bits; k_new / v_new [B,HKV,s_active,D] bf16 bits or None; inv_freq [D/2]."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    B, HQ, SA, D = q.shape
    sk = _sinks(sink, HQ)
    kn = None if k_new is None else _u16(k_new)
    vn = None if v_new is None else _u16(v_new)
    f = None if inv_freq is None else np.ascontiguousarray(inv_freq, dtype=np.float64)
    cl = np.ascontiguousarray(cache_len, dtype=np.int32)
    if table is not None:
        table = np.ascontiguousarray(table, dtype=np.uint32)
        num_pages, HKV, page, _ = k_cache.shape
        max_pages, max_len = table.shape[1], 0
    else:
        _, HKV, max_len, _ = k_cache.shape
        num_pages, page, max_pages = 0, 1, 0
    o = np.empty((B, HQ, SA, D), dtype=np.float64)
    lse = np.empty((B, HQ, SA), dtype=np.float64)
    lib = _load()

    def run(bh):
        return lib.oracle_decode_ext(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kn), _ptr(vn),
                                     _ptr(table), _ptr(cl), B, HQ, HKV, D, SA, page, max_pages,
                                     num_pages, max_len, float(scale), int(window), int(circular),
                                     _ptr(f), _ptr(sk), bh, bh + 1, _ptr(o), _ptr(lse))

    with ThreadPoolExecutor(max_workers=min(threads or default_threads(), B * HQ)) as ex:
        for rc in ex.map(run, range(B * HQ)):
            _check(rc)
    return o, lse


def decode_mask(cache_len, hq, s_active, max_len):
    """0/1 decode mask [B, HQ, s_active, max_len] (uint8)."""
    cl = np.ascontiguousarray(cache_len, dtype=np.int32)
    B = cl.shape[0]
    m = np.empty((B, hq, s_active, max_len), dtype=np.uint8)
    _check(_load().oracle_decode_mask(_ptr(cl), B, hq, s_active, max_len, _ptr(m)))
    return m
