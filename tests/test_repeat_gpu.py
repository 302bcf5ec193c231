"""Repeated launches of each persistent prefill kernel and of the decode passes: every launch
must finish without a device-side error and give bit-identical outputs.  The kernels'
pipelines hand tiles between warps through mbarriers whose phases are read by parity, so
an ordering mistake shows up as a wait that passes a phase early (different outputs) or
never ends (a bounded wait that gives up and sets the device error word), and then often
only under some interleavings: many back-to-back launches, with an L2 flush between some
of them to vary the timing, give such a mistake many chances to show."""
import pytest
import torch

from workloads import configs as C

pytestmark = pytest.mark.gpu

REPEATS = 40


def _repeat(call, outs, dev):
    import flash_attention_forward_attn_gb300 as A

    flush = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
    call()
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    ref = [x.clone() for x in outs]
    for i in range(REPEATS):
        if i % 3 == 0:
            flush.fill_(i & 0xFF)
        call()
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    call()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(outs, ref))


@pytest.mark.parametrize("b,hq,hkv,s,d,window", [
    (1, 16, 8, 4096, 256, 1024),  # the head_dim-256 kernel, window band
    (1, 8, 4, 2048, 256, 0),      # the head_dim-256 kernel, causal only
    (1, 32, 8, 4096, 128, 0),     # the two-tile kernel
    (1, 16, 16, 2048, 64, 512),   # the two-tile kernel, head_dim 64 with a window
])
def test_prefill_repeats_are_identical_and_error_free(b, hq, hkv, s, d, window, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.PrefillWorkload("repeat", b, hq, hkv, s, s, d, True, window, seed=0x5EED + d)
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
    _repeat(lambda: A.attn_fwd_prefill(q, k, v, causal=True, window=window, scale=w.scale, o=o,
                                       lse=lse), (o, lse), cuda_device)


def test_packed_prefill_repeats_are_identical_and_error_free(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    pw = C.PackedPrefillWorkload("repeat_packed", 16, 4, 256, 8, 128, 1500, 300, seed=0x5EED)
    w = pw.as_prefill()
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
    cu_q, cu_k = (torch.from_numpy(x).to(cuda_device) for x in pw.offsets())
    _repeat(lambda: A.attn_fwd_prefill_ex(q, k, v, causal=True, window=128, scale=pw.scale, o=o,
                                          lse=lse, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k),
            (o, lse), cuda_device)


@pytest.mark.parametrize("e4m3", [False, True], ids=["bf16_cache", "e4m3_cache"])
@pytest.mark.parametrize("s_active", [1, 4])
def test_decode_repeats_are_identical_and_error_free(e4m3, s_active, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    base = C.PAGED_DECODE if s_active == 1 else C.PAGED_DECODE_SPEC4
    w = base.with_(b=16, len_hi=8192)
    t = (C.decode_inputs_e4m3_torch if e4m3 else C.decode_inputs_torch)(w, cuda_device)
    o = torch.empty(t["q"].shape, dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty(t["q"].shape[:3], dtype=torch.float32, device=cuda_device)
    _repeat(lambda: A.attn_fwd_decode_ex(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                         t["cache_len"], max_cache_len=t["max_cache_len"],
                                         scale=w.scale, o=o, lse=lse), (o, lse), cuda_device)
