"""Parity of decode over an FP8-e4m3 KV cache (attn_fwd_decode_ex with kv_dtype e4m3,
through the C ABI) against the fp64 oracle ("Flash-Attention: Decode (TKG)", "Decode (TKG)
vs context (CTE) - the diff": the FP8-e4m3 KV cache).  A cache byte x stands for
e4m3(x) * k_scale (K) or e4m3(x) * v_scale (V)."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, bits_of
from workloads import configs as C

pytestmark = pytest.mark.gpu


def run_e4m3(t, w, kv_chunk, k_scale, v_scale, sink=None, o_dtype=torch.float32):
    import flash_attention_forward_attn_gb300 as A

    lse = torch.empty((w.b, w.hq, w.s_active), dtype=torch.float32, device=t["q"].device)
    o, _ = A.attn_fwd_decode_ex(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                t["cache_len"], max_cache_len=t["max_cache_len"], scale=w.scale,
                                lse=lse, o_dtype=o_dtype, kv_chunk=kv_chunk, sink=sink,
                                k_scale=k_scale, v_scale=v_scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


def cache_bytes(c):
    return c.view(torch.uint8).cpu().numpy()


SMALL = [
    # name, b, hq, hkv, d, s_active, page, lens, paged, kv_chunk, k_scale, v_scale, sink
    ("e4m3_paged_sa1_g4", 3, 8, 2, 128, 1, 32, (40, 1030, 77), True, 64, 1.0, 1.0, False),
    ("e4m3_paged_sa4_scales", 3, 8, 2, 128, 4, 32, (40, 1030, 77), True, 0, 0.5, 2.0, False),
    ("e4m3_flat_sa2_g8", 2, 8, 1, 128, 2, 32, (5, 513), False, 96, 0.03125, 3.0, False),
    ("e4m3_paged16_sa3_sink", 2, 8, 4, 128, 3, 16, (17, 100), True, 64, 1.5, 0.75, True),
    ("e4m3_paged64_d256", 2, 4, 2, 256, 2, 64, (70, 129), True, 128, 1.0, 1.0, False),
    ("e4m3_flat_d256_sink", 2, 8, 2, 256, 1, 32, (33, 260), False, 64, 0.25, 1.25, True),
    ("e4m3_paged_mha_sa16", 1, 2, 2, 128, 16, 32, (50,), True, 32, 1.0, 1.0, False),
    ("e4m3_len_equals_sa", 2, 4, 1, 128, 4, 32, (4, 33), True, 32, 2.0, 0.5, False),
    # head_dim 128 reads 64-token tiles: pages larger than a tile, a split length that is not
    # a multiple of the tile (empty trailing splits), a flat cache of 64 k + 32 rows
    ("e4m3_paged128_sa2", 2, 8, 2, 128, 2, 128, (300, 1000), True, 0, 1.0, 1.0, False),
    ("e4m3_paged256_chunk96", 2, 8, 2, 128, 3, 256, (700, 95), True, 96, 1.0, 1.0, True),
    ("e4m3_flat_rows_64k_plus_32", 2, 8, 2, 128, 1, 32, (100, 281), False, 32, 1.0, 1.0, False),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0])
def test_decode_e4m3_small(case, cuda_device):
    name, b, hq, hkv, d, sa, page, lens, paged, chunk, ks, vs, with_sink = case
    w = C.DecodeWorkload(name, b, hq, hkv, d, sa, page_size=page, len_hi=max(lens) + 7,
                         paged=paged, fixed_lens=lens, seed=0xE4 + len(name))
    t = C.decode_inputs_e4m3_torch(w, cuda_device)
    sk = C.sink_logits(hq) if with_sink else None
    o, lse = run_e4m3(t, w, chunk, ks, vs,
                      sink=None if sk is None else torch.from_numpy(sk).to(cuda_device))
    o_ref, lse_ref = oracle.decode_e4m3(bits_of(t["q"]), cache_bytes(t["k_cache"]),
                                        cache_bytes(t["v_cache"]), t["table"], t["lens"],
                                        w.scale, ks, vs, sink=sk)
    assert_o_close(o.cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)


def test_decode_e4m3_paged_equals_flat_bit_exact(cuda_device):
    base = C.DecodeWorkload("e4pf", 3, 8, 2, 128, 4, len_hi=1100, fixed_lens=(40, 1030, 77),
                            seed=19)
    outs = []
    for paged, permute in ((True, True), (True, False), (False, False)):
        w = base.with_(paged=paged)
        t = C.decode_inputs_e4m3_torch(w, cuda_device, permute=permute)
        outs.append(run_e4m3(t, w, 64, 0.75, 1.5))
    for o, l in outs[1:]:
        assert torch.equal(outs[0][0], o) and torch.equal(outs[0][1], l)


@pytest.mark.parametrize("w", [C.PAGED_DECODE, C.PAGED_DECODE_SPEC4], ids=lambda w: w.name)
def test_decode_e4m3_full_size_sampled(w, cuda_device):
    """The full workloads with e4m3 caches, in the launch the benchmark times; sequences
    are checked one by one: their pages are gathered into a one-sequence flat cache for
    the oracle."""
    t = C.decode_inputs_e4m3_torch(w, cuda_device)
    o, lse = run_e4m3(t, w, 0, 1.0, 1.0, o_dtype=torch.bfloat16)
    lens = t["lens"]
    q = bits_of(t["q"])
    for b in sorted({int(np.argmax(lens)), int(np.argmin(lens)), 7, 33}):
        n = int(lens[b])
        npg = -(-n // w.page_size)
        idx = torch.from_numpy(t["table"][b, :npg].astype(np.int64)).to(cuda_device)
        flat = [t[c].view(torch.uint8)[idx].permute(1, 0, 2, 3)
                .reshape(1, w.hkv, npg * w.page_size, w.d)[:, :, :n] for c in ("k_cache", "v_cache")]
        o_ref, lse_ref = oracle.decode_e4m3(q[b:b + 1], cache_bytes(flat[0].contiguous()),
                                            cache_bytes(flat[1].contiguous()), None,
                                            np.array([n], np.int32), w.scale, 1.0, 1.0)
        assert_o_close(o[b:b + 1].float().cpu().numpy(), o_ref, f"{w.name} e4m3 b{b}")
        assert_lse_close(lse[b:b + 1].cpu().numpy(), lse_ref, f"{w.name} e4m3 b{b}")


def test_decode_e4m3_rejects_d64_and_bad_scales(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.DecodeWorkload("e4bad", 1, 4, 1, 64, 1, len_hi=100, fixed_lens=(50,), seed=20)
    t = C.decode_inputs_e4m3_torch(w, cuda_device)
    with pytest.raises(A.AttnError):
        run_e4m3(t, w, 0, 1.0, 1.0)
    w2 = w.with_(d=128)
    t2 = C.decode_inputs_e4m3_torch(w2, cuda_device)
    with pytest.raises(A.AttnError):
        run_e4m3(t2, w2, 0, float("nan"), 1.0)
