"""The C-ABI library loads without a GPU, exports every entry point attn.h declares, and
its host-side checks reject invalid calls before anything reaches CUDA."""
import ctypes
import os
import re

import pytest

import flash_attention_forward_attn_gb300 as A
from flash_attention_forward_attn_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return A.load_library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_symbols() == sorted([
        "attn_fwd_prefill", "attn_decode_workspace_bytes", "attn_fwd_decode",
        "attn_gen_mask_decode", "attn_get_device_error", "attn_status_string",
        "attn_fwd_decode_static_ws", "attn_fwd_prefill_ex", "attn_fwd_decode_ex",
        "attn_append_kv", "attn_check_wait_timeout", "attn_prefill_workspace_bytes"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (2, "ATTN_ERR_UNSUPPORTED"),
                       (3, "ATTN_ERR_CUDA"), (4, "ATTN_ERR_PAGE_OOB"), (5, "ATTN_ERR_DEVICE_TIMEOUT"),
                       (6, "ATTN_ERR_WORKSPACE"), (7, "ATTN_ERR_CACHE_LEN")]:
        assert A.attn_status_string(code) == name


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails validation first


def prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, b=1, hq=4, hkv=2, sq=16, skv=16, d=128,
             scale=0.1, causal=1, window=0, o_dtype=0)
    a.update(kw)
    return lib.attn_fwd_prefill(a["q"], a["k"], a["v"], a["o"], a["lse"], a["b"], a["hq"], a["hkv"],
                                a["sq"], a["skv"], a["d"], a["scale"], a["causal"], a["window"],
                                a["o_dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(hq=3, hkv=2), 1), (dict(b=0), 1), (dict(sq=-1), 1), (dict(window=-2), 1),
    (dict(d=96), 2), (dict(d=512), 2), (dict(causal=0, window=8), 2), (dict(q=None), 1),
    (dict(o=ctypes.c_void_p((1 << 20) + 8)), 1), (dict(scale=float("nan")), 1),
    (dict(o_dtype=7), 1),
])
def test_prefill_rejects_before_launch(lib, kw, status):
    assert prefill(lib, **kw) == status


def test_prefill_zero_queries_is_a_no_op(lib):
    assert prefill(lib, sq=0) == 0


def decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, table=FAKE, cl=FAKE, b=2, hq=8, hkv=2, d=128, sa=4, page=32,
             maxp=4, npages=8, maxlen=128, scale=0.1, o=FAKE, lse=None, odt=0, chunk=0, ws=FAKE,
             wsb=1 << 30)
    a.update(kw)
    return lib.attn_fwd_decode(a["q"], a["k"], a["v"], a["table"], a["cl"], a["b"], a["hq"], a["hkv"],
                               a["d"], a["sa"], a["page"], a["maxp"], a["npages"], a["maxlen"],
                               a["scale"], a["o"], a["lse"], a["odt"], a["chunk"], a["ws"], a["wsb"],
                               None)


@pytest.mark.parametrize("kw,status", [
    (dict(hq=6, hkv=4), 1), (dict(sa=0), 1), (dict(page=24), 1), (dict(page=8), 1),
    (dict(maxp=3), 1), (dict(chunk=48), 1), (dict(d=80), 2), (dict(sa=5), 2),
    (dict(ws=None), 6), (dict(wsb=100), 6), (dict(ws=ctypes.c_void_p((1 << 20) + 4)), 6),
    (dict(cl=None), 1), (dict(npages=0), 1),
])
def test_decode_rejects_before_launch(lib, kw, status):
    assert decode(lib, **kw) == status


def test_ex_calls_check_their_options_before_launch(lib):
    bad = A.AttnOpts(sink=(1 << 20) + 2)  # a sink pointer that is not 4-byte aligned
    none = A.AttnOpts()
    args = (FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 0, 16, 128, 0.1, 1, 0, 0)
    assert lib.attn_fwd_prefill_ex(*args, ctypes.byref(bad), None) == 1
    assert lib.attn_fwd_prefill_ex(*args, ctypes.byref(none), None) == 0  # sq = 0: no-op
    assert lib.attn_fwd_prefill_ex(*args, None, None) == 0
    dargs = (FAKE, FAKE, FAKE, FAKE, FAKE, 2, 8, 2, 128, 4, 32, 4, 8, 128, 0.1, FAKE, None, 0, 0)
    assert lib.attn_fwd_decode_ex(*dargs, ctypes.byref(bad), FAKE, 1 << 30, None) == 1
    e4 = lambda **kw: A.AttnOpts(**dict(dict(kv_dtype=1, k_scale=1.0, v_scale=1.0), **kw))
    assert lib.attn_fwd_decode_ex(*dargs, ctypes.byref(A.AttnOpts(kv_dtype=5)), FAKE, 1 << 30,
                                  None) == 1  # unknown cache type
    assert lib.attn_fwd_decode_ex(*dargs, ctypes.byref(e4(k_scale=float("nan"))), FAKE, 1 << 30,
                                  None) == 1
    assert lib.attn_fwd_decode_ex(*dargs, ctypes.byref(e4(v_scale=float("inf"))), FAKE, 1 << 30,
                                  None) == 1
    d64 = dargs[:8] + (64,) + dargs[9:]
    assert lib.attn_fwd_decode_ex(*d64, ctypes.byref(e4()), FAKE, 1 << 30, None) == 2
    assert lib.attn_fwd_prefill_ex(*args, ctypes.byref(e4()), None) == 2  # prefill reads bf16
    op = lambda **kw: ctypes.byref(A.AttnOpts(**kw))
    call = lambda a, o: lib.attn_fwd_decode_ex(*a, o, FAKE, 1 << 30, None)
    flat = dargs[:3] + (None,) + dargs[4:]  # no block table
    assert call(dargs, op(window=-1)) == 1
    assert call(dargs, op(window=8, circular=1)) == 1  # a paged cache cannot be circular
    assert call(flat, op(circular=1)) == 1  # circular needs a window
    assert call(flat, op(window=126, circular=1)) == 1  # 126 + 4 - 1 > 128 rows
    assert call(flat, op(window=8, circular=2)) == 1
    assert call(dargs, op(rope_inv_freq=(1 << 20) + 2)) == 1  # misaligned
    for kw in (dict(window=4), dict(circular=1), dict(rope_inv_freq=1 << 20)):
        assert lib.attn_fwd_prefill_ex(*args, op(**kw), None) == 2  # decode options
    cu = 1 << 20
    assert lib.attn_fwd_prefill_ex(*args, op(cu_seqlens_q=cu, nseq=2), None) == 1  # no k offsets
    assert lib.attn_fwd_prefill_ex(*args, op(cu_seqlens_q=cu, cu_seqlens_k=cu, nseq=0), None) == 1
    assert lib.attn_fwd_prefill_ex(*args, op(cu_seqlens_q=cu + 2, cu_seqlens_k=cu, nseq=1),
                                   None) == 1
    b2 = args[:5] + (2,) + args[6:]  # packing needs b = 1
    assert lib.attn_fwd_prefill_ex(*b2, op(cu_seqlens_q=cu, cu_seqlens_k=cu, nseq=1), None) == 1
    assert call(dargs, op(cu_seqlens_q=cu, cu_seqlens_k=cu, nseq=1)) == 2  # a prefill option
    # the packed-prefill work-order scratch: only with packing, 4-byte aligned, large enough
    packed = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, nseq=1)
    a16 = args[:8] + (16,) + args[9:]  # sq = 16: every call below must fail validation
    assert lib.attn_fwd_prefill_ex(*a16, op(prefill_workspace=cu, prefill_workspace_bytes=64),
                                   None) == 1
    assert lib.attn_fwd_prefill_ex(*a16, op(prefill_workspace=cu + 2, prefill_workspace_bytes=64,
                                             **packed), None) == 1
    assert lib.attn_fwd_prefill_ex(*a16, op(prefill_workspace=cu, prefill_workspace_bytes=3,
                                             **packed), None) == 1  # sq = 16 needs 4 bytes
    assert call(dargs, op(prefill_workspace=cu, prefill_workspace_bytes=64)) == 2
    # an invalid size is still reported first, with or without options
    dbad = dargs[:8] + (80,) + dargs[9:]  # d = 80
    assert lib.attn_fwd_decode_ex(*dbad, ctypes.byref(none), FAKE, 1 << 30, None) == 2


def _ws(b, hq, s_active, d, max_len, chunk):
    # rows = b*hq*s_active; slots = ceil(max_len / chunk) + 1; O partials (256-byte padded),
    # (m, l) pairs (16-byte padded), one int per (sequence, head)
    rows, slots = b * hq * s_active, -(-max_len // chunk) + 1
    return (((rows * slots * d * 4 + 255) // 256) * 256 + ((rows * slots * 8 + 15) // 16) * 16
            + b * hq * 4)


@pytest.mark.parametrize("b,max_len,chunk", [
    (64, 32768, 4096),   # long batch: the largest default split
    (16, 32768, 4096),   # b * max_len / 128 = 4096
    (8, 16384, 1024),    # 1024
    (1, 32768, 256),     # 256: one long sequence still gets 128 splits
    (4, 4096, 256),      # 128 -> clamped to the smallest default split
])
def test_workspace_default_chunk(lib, b, max_len, chunk):
    """kv_chunk = 0: the largest power of two in [256, 4096] not above b * max_len / 128."""
    assert A.attn_decode_workspace_bytes(b, 32, 4, 128, max_len) == _ws(b, 32, 4, 128, max_len, chunk)
    assert A.attn_decode_workspace_bytes(b, 32, 4, 128, max_len, chunk) == _ws(b, 32, 4, 128, max_len, chunk)


def test_workspace_bytes_formula(lib):
    assert A.attn_decode_workspace_bytes(64, 32, 4, 128, 32768, 1024) == _ws(64, 32, 4, 128, 32768, 1024)
    assert A.attn_decode_workspace_bytes(1, 1, 1, 64, 100, 64) == ((3 * 64 * 4 + 255) // 256) * 256 + 32 + 4
    assert A.attn_decode_workspace_bytes(1, 1, 1, 96, 100) == 0
    assert A.attn_decode_workspace_bytes(1, 1, 1, 64, 100, 33) == 0


def test_mask_rejects_before_launch(lib):
    assert lib.attn_gen_mask_decode(FAKE, 0, 1, 1, 10, FAKE, None) == 1
    assert lib.attn_gen_mask_decode(None, 1, 1, 1, 10, FAKE, None) == 1
    assert lib.attn_gen_mask_decode(FAKE, 1, 1, 1, 0, FAKE, None) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib

    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(A, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        A.load_library()
    monkeypatch.setattr(A, "_lib", None)
    importlib.reload(_build)


def test_append_rejects_before_launch(lib):
    def app(**kw):
        a = dict(kn=FAKE, vn=FAKE, k=FAKE, v=FAKE, table=FAKE, cl=FAKE, b=2, hkv=2, d=128, sa=4,
                 page=32, maxp=4, npages=8, maxlen=128, opts=None)
        a.update(kw)
        return lib.attn_append_kv(a["kn"], a["vn"], a["k"], a["v"], a["table"], a["cl"], a["b"],
                                  a["hkv"], a["d"], a["sa"], a["page"], a["maxp"], a["npages"],
                                  a["maxlen"], a["opts"], None)
    assert app(b=0) == 1
    assert app(kn=None) == 1
    assert app(cl=None) == 1
    assert app(d=96) == 2
    assert app(page=24) == 1
    assert app(maxp=3) == 1
    assert app(opts=ctypes.byref(A.AttnOpts(circular=1))) == 1  # a paged cache cannot be circular
    assert app(opts=ctypes.byref(A.AttnOpts(kv_dtype=1, k_scale=1.0, v_scale=1.0))) == 2
    assert app(v=ctypes.c_void_p((1 << 20) + 8)) == 1


def test_wait_timeout_check_rejects_bad_limits(lib):
    assert lib.attn_check_wait_timeout(0, None) == 1
    assert lib.attn_check_wait_timeout(-5, None) == 1
    assert lib.attn_check_wait_timeout((1 << 33) + 1, None) == 1


def test_prefill_workspace_bytes(lib):
    """One int per 128-row query tile."""
    for sq, n in [(-5, 0), (0, 0), (1, 4), (128, 4), (129, 8), (34910, 4 * 273)]:
        assert A.attn_prefill_workspace_bytes(sq) == n


def test_a_library_without_a_matching_stamp_is_rebuilt(lib, tmp_path, monkeypatch):
    """The rebuild decision rests on the fingerprint of the sources, flags, compiler and
    machine, not on file times: a library whose stamp does not match (one copied in with a
    tree, or built elsewhere) is never taken for a current build."""
    assert _build.up_to_date()
    stale = tmp_path / "stale.stamp"
    stale.write_text("0" * 64 + "\n")
    monkeypatch.setattr(_build, "STAMP", str(stale))
    assert not _build.up_to_date()
    monkeypatch.setattr(_build, "STAMP", str(tmp_path / "missing.stamp"))
    assert not _build.up_to_date()
