"""attn_fwd_decode_static_ws: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc when they run attention (a fixed device-memory budget
set up at start-up, a host runtime that owns every allocation, a real-time loop that must
stay out of the allocator).  This entry point takes no workspace; its split-KV scratch is a
fixed array compiled into the library, shared by every call and never cleared.

The tests call it through the C ABI, several times in a row with changing shapes: long
caches with many splits first, then short and mixed caches whose sequences have fewer
splits than the earlier call wrote, with the default and an explicit split length.  Each
result must be bit-identical to the regular attn_fwd_decode run with the same split length
on a NaN-filled caller workspace (a read of any partial the call did not write would show
as NaN there, or as a difference), and must match the fp64 oracle.  The file name makes
pytest collect it last.
"""
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, bits_of
from workloads import configs as C

pytestmark = pytest.mark.gpu

MIXED_LENS = (40, 3000, 300, 33, 1000, 64, 2999, 700)

# workload, kv_chunk: run in this order against the same static array
CALLS = [
    (C.DecodeWorkload("noalloc_long", 8, 32, 8, 128, 4, len_lo=2000, len_hi=3000, seed=0x5A7), 256),
    (C.DecodeWorkload("noalloc_long", 8, 32, 8, 128, 4, len_lo=2000, len_hi=3000, seed=0x5A7), 256),
    (C.DecodeWorkload("noalloc_mixed", 8, 32, 8, 128, 4, len_hi=3000, fixed_lens=MIXED_LENS,
                      seed=0x5A8), 0),
    (C.DecodeWorkload("noalloc_mixed_sa1", 8, 32, 8, 128, 1, len_hi=3000, fixed_lens=MIXED_LENS,
                      seed=0x5A9), 96),
]


def _nan_workspace(A, w, max_cache_len, kv_chunk, dev):
    need = A.attn_decode_workspace_bytes(w.b, w.hq, w.s_active, w.d, max_cache_len, kv_chunk)
    return torch.full((need // 4 + 4,), float("nan"), dtype=torch.float32, device=dev).view(torch.uint8)


def test_static_scratch_decode_matches_workspace_decode(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    for w, kv_chunk in CALLS:
        t = C.decode_inputs_torch(w, cuda_device)
        args = (t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["cache_len"])
        mcl = t["max_cache_len"]
        lse_ref = torch.empty((w.b, w.hq, w.s_active), dtype=torch.float32, device=cuda_device)
        o_ref, _ = A.attn_fwd_decode(*args, max_cache_len=mcl, scale=w.scale, lse=lse_ref,
                                     o_dtype=torch.float32, kv_chunk=kv_chunk,
                                     workspace=_nan_workspace(A, w, mcl, kv_chunk, cuda_device))
        lse = torch.empty_like(lse_ref)
        o, _ = A.attn_fwd_decode_static_ws(*args, max_cache_len=mcl, scale=w.scale, lse=lse,
                                           o_dtype=torch.float32, kv_chunk=kv_chunk)
        torch.cuda.synchronize()
        assert A.attn_get_device_error() == 0
        assert torch.isfinite(o_ref).all(), f"{w.name}: a partial the call did not write was read"
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), w.name
        o_or, lse_or = oracle.decode(bits_of(t["q"]), bits_of(t["k_cache"]), bits_of(t["v_cache"]),
                                     t["table"], t["lens"], w.scale)
        assert_o_close(o.cpu().numpy(), o_or, w.name)
        assert_lse_close(lse.cpu().numpy(), lse_or, w.name)


def test_static_scratch_rejects_calls_larger_than_the_array(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    # 64 sequences x 32 heads x 4 tokens x 32 splits (1024-token chunks) x 128 dims of fp32
    # partials > 64 MiB
    w = C.PAGED_DECODE_SPEC4
    need = A.attn_decode_workspace_bytes(w.b, w.hq, w.s_active, w.d, 32768, 1024)
    assert need > 64 << 20
    q = torch.zeros((w.b, w.hq, w.s_active, w.d), dtype=torch.bfloat16, device=cuda_device)
    kc = torch.zeros((4, w.hkv, 32, w.d), dtype=torch.bfloat16, device=cuda_device)
    bt = torch.zeros((w.b, 1024), dtype=torch.int32, device=cuda_device)
    cl = torch.full((w.b,), 32, dtype=torch.int32, device=cuda_device)
    with pytest.raises(A.AttnError, match="ATTN_ERR_WORKSPACE"):
        A.attn_fwd_decode_static_ws(q, kc, kc, bt, cl, max_cache_len=32768, kv_chunk=1024)
