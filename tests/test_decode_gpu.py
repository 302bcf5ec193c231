"""Parity of the CUDA decode path (split-KV + log-sum-exp combine, flat and paged caches)
and of the decode mask materialiser, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, bits_of
from workloads import configs as C

pytestmark = pytest.mark.gpu


def run_decode(t, w, kv_chunk=0, o_dtype=torch.float32):
    import flash_attention_forward_attn_gb300 as A

    lse = torch.empty((w.b, w.hq, w.s_active), dtype=torch.float32, device=t["q"].device)
    o, _ = A.attn_fwd_decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["cache_len"],
                             max_cache_len=t["max_cache_len"], scale=w.scale, lse=lse,
                             o_dtype=o_dtype, kv_chunk=kv_chunk)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


def oracle_of(t, w):
    q = bits_of(t["q"])
    kc, vc = bits_of(t["k_cache"]), bits_of(t["v_cache"])
    return oracle.decode(q, kc, vc, t["table"], t["lens"], w.scale)


SMALL = [
    # name, b, hq, hkv, d, s_active, page, lens, paged, kv_chunk
    ("paged_sa1_g4", 3, 8, 2, 128, 1, 32, (40, 1030, 77), True, 64),
    ("paged_sa4_g4", 3, 8, 2, 128, 4, 32, (40, 1030, 77), True, 0),
    ("paged_sa4_chunk32", 2, 8, 2, 128, 4, 32, (35, 300), True, 32),
    ("flat_sa1_g4", 3, 8, 2, 128, 1, 32, (40, 1030, 77), False, 64),
    ("flat_sa2_g8", 2, 8, 1, 128, 2, 32, (5, 513), False, 96),
    ("paged16_d64", 2, 4, 4, 64, 3, 16, (17, 100), True, 64),
    ("paged64_d256", 2, 4, 2, 256, 2, 64, (70, 129), True, 128),
    ("paged_mha_sa16", 1, 2, 2, 128, 16, 32, (50,), True, 32),
    ("paged_len_equals_sa", 2, 4, 1, 128, 4, 32, (4, 33), True, 32),
    # one long sequence: every CTA of the wave reads a piece of the same pair (79 pieces
    # per pair against a bound of 80 partial slots)
    ("one_long_seq_79_pieces", 1, 8, 2, 128, 1, 32, (20000,), True, 0),
    # short sequences: each CTA's run crosses several pairs, so the two Q slots are reused
    # and many pieces are shorter than the four consumer warps
    ("short_seqs_many_pieces_per_cta", 24, 8, 2, 128, 4, 32,
     (300, 31, 32, 64, 4, 40, 300, 17, 4, 9, 5, 32, 300, 40, 17, 33, 64, 5, 300, 17, 4, 17, 33, 31),
     True, 256),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0])
def test_decode_small(case, cuda_device):
    name, b, hq, hkv, d, sa, page, lens, paged, chunk = case
    w = C.DecodeWorkload(name, b, hq, hkv, d, sa, page_size=page, len_hi=max(lens) + 7,
                         paged=paged, fixed_lens=lens, seed=0xDEC0 + len(name))
    t = C.decode_inputs_torch(w, cuda_device)
    o, lse = run_decode(t, w, kv_chunk=chunk)
    o_ref, lse_ref = oracle_of(t, w)
    assert_o_close(o.cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)


def test_decode_paged_equals_flat_and_identity_bit_exact(cuda_device):
    base = C.DecodeWorkload("pf", 3, 8, 2, 128, 4, len_hi=1100, fixed_lens=(40, 1030, 77), seed=9)
    outs = []
    for paged, permute in ((True, True), (True, False), (False, False)):
        w = base.with_(paged=paged)
        t = C.decode_inputs_torch(w, cuda_device, permute=permute)
        outs.append(run_decode(t, w, kv_chunk=64))
    for o, l in outs[1:]:
        assert torch.equal(outs[0][0], o) and torch.equal(outs[0][1], l)


def test_decode_split_count_does_not_change_result(cuda_device):
    w = C.DecodeWorkload("sp", 2, 8, 2, 128, 4, len_hi=2100, fixed_lens=(2050, 700), seed=10)
    t = C.decode_inputs_torch(w, cuda_device)
    o1, l1 = run_decode(t, w, kv_chunk=32)
    o2, l2 = run_decode(t, w, kv_chunk=4096)
    assert (o1 - o2).abs().max().item() < 2e-3
    assert (l1 - l2).abs().max().item() < 1e-4


def test_decode_repeat_runs_bit_identical(cuda_device):
    w = C.PAGED_DECODE_SPEC4.with_(b=8, len_hi=4096)
    t = C.decode_inputs_torch(w, cuda_device)
    o0, l0 = run_decode(t, w, o_dtype=torch.bfloat16)
    for _ in range(20):
        o1, l1 = run_decode(t, w, o_dtype=torch.bfloat16)
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.parametrize("w", [C.PAGED_DECODE, C.PAGED_DECODE_SPEC4], ids=lambda w: w.name)
def test_decode_full_size_sampled(w, cuda_device):
    t = C.decode_inputs_torch(w, cuda_device)
    o, lse = run_decode(t, w, o_dtype=torch.bfloat16)
    lens = t["lens"]
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 7, 33})
    for b in seqs:
        n = int(lens[b])
        for h in (0, 13, 31):
            g = oracle.kv_head(h, w.hq, w.hkv)
            kh = C.decode_kv_logical_np(w, "k", b, g, n)
            vh = C.decode_kv_logical_np(w, "v", b, g, n)
            qh = C.decode_q_np(w, b, h)
            qp = [n - w.s_active + t_ for t_ in range(w.s_active)]
            o_ref, lse_ref = oracle.attention_rows(qh, kh, vh, qp, w.scale, True, 0)
            assert_o_close(o[b, h].float().cpu().numpy(), o_ref, f"{w.name} b{b} h{h}")
            assert_lse_close(lse[b, h].cpu().numpy(), lse_ref, f"{w.name} b{b} h{h}")


def test_decode_page_table_out_of_range_is_reported(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.DecodeWorkload("oob", 2, 4, 1, 128, 1, len_hi=200, fixed_lens=(100, 64), seed=11)
    t = C.decode_inputs_torch(w, cuda_device)
    bt = t["block_table"].clone()
    bt[1, 1] = t["num_pages"] + 5  # a page past the pool: the kernel must not read it
    t2 = dict(t, block_table=bt)
    A.attn_fwd_decode(t2["q"], t2["k_cache"], t2["v_cache"], bt, t2["cache_len"],
                      max_cache_len=t2["max_cache_len"])
    assert A.attn_get_device_error() == 4  # ATTN_ERR_PAGE_OOB
    assert A.attn_get_device_error() == 0  # reading clears it
    o, _ = run_decode(t, w)  # the library keeps working afterwards
    assert torch.isfinite(o).all()


def test_decode_bad_cache_len_is_reported(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.DecodeWorkload("badlen", 2, 4, 1, 128, 4, len_hi=200, fixed_lens=(100, 64), seed=12)
    t = C.decode_inputs_torch(w, cuda_device)
    cl = t["cache_len"].clone()
    cl[0] = 2  # fewer than s_active
    A.attn_fwd_decode(t["q"], t["k_cache"], t["v_cache"], t["block_table"], cl,
                      max_cache_len=t["max_cache_len"])
    assert A.attn_get_device_error() == 7  # ATTN_ERR_CACHE_LEN


@pytest.mark.parametrize("sa", [1, 4])
def test_gen_mask_bit_exact(sa, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    lens = np.array([5, 37, 4, 1000], dtype=np.int32)
    max_len = 1003
    m = A.attn_gen_mask_decode(torch.from_numpy(lens).to(cuda_device), 3, sa, max_len)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(m.cpu().numpy(), oracle.decode_mask(lens, 3, sa, max_len))


def test_gen_mask_full_size(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    w = C.PAGED_DECODE_SPEC4
    lens = C.decode_cache_lens(w)
    m = A.attn_gen_mask_decode(torch.from_numpy(lens).to(cuda_device), 4, w.s_active, w.len_hi)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(m.cpu().numpy(), oracle.decode_mask(lens, 4, w.s_active, w.len_hi))


def test_bounded_wait_times_out_and_the_context_stays_usable(cuda_device):
    """The failure path without a fault: a bounded wait on a phase nothing completes gives
    up, sets the timeout word (ATTN_ERR_DEVICE_TIMEOUT), and the library keeps working."""
    import time

    import flash_attention_forward_attn_gb300 as A

    t0 = time.perf_counter()
    A.attn_check_wait_timeout(20_000_000)  # about 10 ms of SM clock
    assert A.attn_get_device_error() == 5  # ATTN_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert A.attn_get_device_error() == 0  # reading clears it
    w = C.DecodeWorkload("after_timeout", 2, 8, 2, 128, 1, len_hi=300, fixed_lens=(100, 257),
                         seed=13)
    t = C.decode_inputs_torch(w, cuda_device)
    o, lse = run_decode(t, w)
    o_ref, lse_ref = oracle_of(t, w)
    assert_o_close(o.cpu().numpy(), o_ref, "after timeout")


@pytest.mark.parametrize("d,sa,paged", [(128, 1, True), (128, 4, True), (64, 3, False),
                                        (256, 2, True)])
def test_decode_cache_length_residue_sweep(d, sa, paged, cuda_device):
    """Cache lengths around the 32-token tile and the split length (kv_chunk 64): every
    sequence of the batch sits at another residue."""
    lens = tuple(max(sa, n) for n in (1, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 128, 129, 200))
    w = C.DecodeWorkload(f"residues_{d}_{sa}_{paged}", len(lens), 8, 2, d, sa, len_hi=max(lens) + 3,
                         paged=paged, fixed_lens=lens, seed=0x5EE1 + d + sa)
    t = C.decode_inputs_torch(w, cuda_device)
    o, lse = run_decode(t, w, kv_chunk=64)
    o_ref, lse_ref = oracle_of(t, w)
    assert_o_close(o.cpu().numpy(), o_ref, w.name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, w.name)
