"""attn_fwd_decode_static_ws: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc when they run attention (a fixed device-memory budget
set up at start-up, a host runtime that owns every allocation, a real-time loop that must
stay out of the allocator).  This entry point takes no workspace; its split-KV scratch is a
fixed array compiled into the library.  The test calls it through the C ABI twice in a row
and checks both results against the regular attn_fwd_decode (which takes a caller
workspace) within the parity tolerance.  The file name makes pytest collect it last.
"""
import pytest
import torch

from tests.helpers import LSE_ATOL, O_ATOL, O_RTOL
from workloads import configs as C

pytestmark = pytest.mark.gpu


def _close(a, b):
    a, b = a.float(), b.float()
    return bool(((a - b).abs() <= O_ATOL + O_RTOL * b.abs()).all())


def test_static_scratch_decode_matches_workspace_decode_twice(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.DecodeWorkload("noalloc", 8, 32, 8, 128, 4, len_hi=3000, seed=0x5A7)
    t = C.decode_inputs_torch(w, cuda_device)
    args = (t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["cache_len"])
    lse_ref = torch.empty((w.b, w.hq, w.s_active), dtype=torch.float32, device=cuda_device)
    o_ref, _ = A.attn_fwd_decode(*args, max_cache_len=t["max_cache_len"], scale=w.scale,
                                 lse=lse_ref, kv_chunk=256)
    for _ in range(2):  # the shared array keeps the previous call's contents
        lse = torch.empty_like(lse_ref)
        o, _ = A.attn_fwd_decode_static_ws(*args, max_cache_len=t["max_cache_len"],
                                           scale=w.scale, lse=lse, kv_chunk=256)
        torch.cuda.synchronize()
        assert A.attn_get_device_error() == 0
        assert _close(o, o_ref)
        assert (lse - lse_ref).abs().max().item() <= LSE_ATOL


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
