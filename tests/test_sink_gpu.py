"""Parity of the attention sink (attn_fwd_prefill_ex / attn_fwd_decode_ex, through the C
ABI) against the fp64 oracle: one logit per query head that joins every row's maximum and
sum with no value row ("Flash-Attention: Context (CTE)", "Algorithm - the per-section max
update" and "Algorithm - fused exp and the running sum")."""
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, bits_of, tensor_of_bits
from workloads import configs as C

pytestmark = pytest.mark.gpu

sinks_for = C.sink_logits  # neutral, moderate, dominant, negligible and absent sinks


PREFILL = [
    # name, b, hq, hkv, sq, skv, d, causal, window, out
    ("sink_causal_gqa_d128", 1, 8, 2, 300, 300, 128, True, 0, torch.bfloat16),
    ("sink_noncausal_rect_d64_f32", 2, 8, 4, 200, 333, 64, False, 0, torch.float32),
    ("sink_window_d256", 1, 8, 4, 400, 400, 256, True, 100, torch.bfloat16),
    ("sink_more_q_than_k_d128_f32", 1, 8, 8, 300, 100, 128, True, 0, torch.float32),
    ("sink_more_q_than_k_d256_f32", 1, 8, 2, 300, 100, 256, True, 0, torch.float32),
    ("sink_multi_unit_d128", 1, 48, 8, 640, 640, 128, True, 0, torch.bfloat16),
    ("sink_multi_unit_window_d256", 1, 40, 8, 640, 640, 256, True, 200, torch.bfloat16),
]


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: c[0])
def test_prefill_sink_all_rows(case, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    name, b, hq, hkv, sq, skv, d, causal, window, out = case
    w = C.PrefillWorkload(name, b, hq, hkv, sq, skv, d, causal, window, seed=0x5111C + len(name))
    qb, kb, vb = C.prefill_inputs_np(w)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    sk = sinks_for(hq)
    lse = torch.empty((b, hq, sq), dtype=torch.float32, device=cuda_device)
    o, _ = A.attn_fwd_prefill_ex(q, k, v, causal=causal, window=window, scale=w.scale, lse=lse,
                                 o_dtype=out, sink=torch.from_numpy(sk).to(cuda_device))
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    o_ref, lse_ref = oracle.prefill(qb, kb, vb, w.scale, causal, window, sink=sk)
    assert_o_close(o.float().cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_prefill_sink_of_minus_inf_is_bit_identical_to_the_plain_call(d, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.PrefillWorkload("sink_none", 1, 4, 2, 260, 260, d, True, 0, seed=77 + d)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in C.prefill_inputs_np(w))
    l1 = torch.empty((1, 4, 260), dtype=torch.float32, device=cuda_device)
    l2 = torch.empty_like(l1)
    o1, _ = A.attn_fwd_prefill(q, k, v, causal=True, scale=w.scale, lse=l1)
    o2, _ = A.attn_fwd_prefill_ex(q, k, v, causal=True, scale=w.scale, lse=l2,
                                  sink=torch.full((4,), float("-inf"), device=cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


DECODE = [
    # name, b, hq, hkv, d, s_active, page, lens, paged, kv_chunk
    ("sink_paged_sa1_g4", 3, 8, 2, 128, 1, 32, (40, 1030, 77), True, 64),
    ("sink_paged_sa4_g4", 3, 8, 2, 128, 4, 32, (40, 1030, 77), True, 0),
    ("sink_flat_sa2_g8", 2, 8, 1, 128, 2, 32, (5, 513), False, 96),
    ("sink_paged16_d64", 2, 8, 4, 64, 3, 16, (17, 100), True, 64),
    ("sink_paged64_d256", 2, 8, 2, 256, 2, 64, (70, 129), True, 128),
]


@pytest.mark.parametrize("case", DECODE, ids=lambda c: c[0])
def test_decode_sink(case, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    name, b, hq, hkv, d, sa, page, lens, paged, chunk = case
    w = C.DecodeWorkload(name, b, hq, hkv, d, sa, page_size=page, len_hi=max(lens) + 7,
                         paged=paged, fixed_lens=lens, seed=0x5EC0 + len(name))
    t = C.decode_inputs_torch(w, cuda_device)
    sk = sinks_for(hq)
    lse = torch.empty((b, hq, sa), dtype=torch.float32, device=cuda_device)
    o, _ = A.attn_fwd_decode_ex(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                t["cache_len"], max_cache_len=t["max_cache_len"], scale=w.scale,
                                lse=lse, o_dtype=torch.float32, kv_chunk=chunk,
                                sink=torch.from_numpy(sk).to(cuda_device))
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    o_ref, lse_ref = oracle.decode(bits_of(t["q"]), bits_of(t["k_cache"]), bits_of(t["v_cache"]),
                                   t["table"], t["lens"], w.scale, sink=sk)
    assert_o_close(o.cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)


def test_decode_sink_of_minus_inf_is_bit_identical_to_the_plain_call(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.DecodeWorkload("sink_none_dec", 2, 8, 2, 128, 4, len_hi=600, fixed_lens=(300, 517),
                         seed=78)
    t = C.decode_inputs_torch(w, cuda_device)
    args = (t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["cache_len"])
    kw = dict(max_cache_len=t["max_cache_len"], scale=w.scale, kv_chunk=64)
    l1 = torch.empty((2, 8, 4), dtype=torch.float32, device=cuda_device)
    l2 = torch.empty_like(l1)
    o1, _ = A.attn_fwd_decode(*args, lse=l1, **kw)
    o2, _ = A.attn_fwd_decode_ex(*args, lse=l2, sink=torch.full((8,), float("-inf"),
                                                                device=cuda_device), **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sink_prefill_full_size_sampled(cuda_device):
    """The benchmark's 2K causal prefill with per-head sink logits, in the launch the
    benchmark times; sampled rows of heads with a neutral, a dominant (e^9, e^60) and an
    absent sink are checked against the oracle's rows with the same sink."""
    import numpy as np

    import flash_attention_forward_attn_gb300 as A
    from workloads import rng

    w = C.CAUSAL_PREFILL_2K
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    sk = C.sink_logits(w.hq)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=cuda_device)
    o, _ = A.attn_fwd_prefill_ex(q, k, v, causal=True, scale=w.scale, lse=lse,
                                 sink=torch.from_numpy(sk).to(cuda_device))
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    u = rng.uniform_np(rng.stream_seed(3, "rows"), 0, 12)
    rows = sorted({0, 1, 127, 128, 1023, w.sq - 1} | {int(x) for x in (u * w.sq).astype(np.int64)})
    for h in (0, 3, 5, 7):  # sinks 0, 9, -inf, 60
        g = oracle.kv_head(h, w.hq, w.hkv)
        kh = C.prefill_kv_head_np(w, "k", 0, g)
        vh = C.prefill_kv_head_np(w, "v", 0, g)
        qr = np.stack([C.prefill_q_rows_np(w, 0, h, r, 1)[0] for r in rows])
        qp = [oracle.q_pos(r, w.sq, w.skv) for r in rows]
        o_ref, lse_ref = oracle.attention_rows(qr, kh, vh, qp, w.scale, True, 0,
                                               sink=float(sk[h]))
        assert_o_close(o[0, h, rows].float().cpu().numpy(), o_ref, f"2K sink h{h}")
        assert_lse_close(lse[0, h, rows].cpu().numpy(), lse_ref, f"2K sink h{h}")
