"""Parity of the decode options of the pages' decode kernel ("Flash-Attention: Decode
(TKG)"), through the C ABI, against the fp64 oracle: a window ("gen_mask_tkg" type B), a
circular flat cache (its wrapped case), RoPE of the queries ("Algorithm", step 0) and the
append of the new tokens' RoPE'd K and V ("New-token K/V append")."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, bits_of, tensor_of_bits
from workloads import configs as C
from workloads import rng

pytestmark = pytest.mark.gpu


def decode_ex(t, w, **kw):
    import flash_attention_forward_attn_gb300 as A

    lse = torch.empty((w.b, w.hq, w.s_active), dtype=torch.float32, device=t["q"].device)
    o, _ = A.attn_fwd_decode_ex(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                t["cache_len"], max_cache_len=t["max_cache_len"], scale=w.scale,
                                lse=lse, o_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


def as_bf16_bits(cache):
    """bf16 bit patterns of a cache (an e4m3 cache's values are exact in bf16)."""
    return bits_of(cache.to(torch.bfloat16) if cache.dtype != torch.bfloat16 else cache)


def inv_freq(d, base=10000.0):
    return (base ** (-np.arange(d // 2, dtype=np.float64) / (d // 2))).astype(np.float32)


WINDOW = [
    # name, b, hq, hkv, d, s_active, page, lens, paged, kv_chunk, window, e4m3
    ("win1_paged_sa1", 3, 8, 2, 128, 1, 32, (40, 1030, 77), True, 64, 1, False),
    ("win40_paged_sa4", 3, 8, 2, 128, 4, 32, (40, 1030, 77), True, 0, 40, False),
    ("win300_flat_sa2", 2, 8, 1, 128, 2, 32, (5, 513), False, 96, 300, False),
    ("win1000_paged16_sa3_d64", 2, 4, 4, 64, 3, 16, (17, 2100), True, 256, 1000, False),
    ("win129_paged64_d256", 2, 4, 2, 256, 2, 64, (70, 700), True, 128, 129, False),
    ("win300_paged_e4m3", 3, 8, 2, 128, 4, 32, (40, 1030, 777), True, 128, 300, True),
    ("win333_paged128_e4m3_chunk96", 2, 8, 2, 128, 2, 128, (700, 1500), True, 96, 333, True),
    # lengths whose window start is rounded down by a whole tile less one slot, so the span
    # read is window + s_active - 1 + 31: the largest one, which fixes how many splits launch
    ("win66_flat_sa1_span_bound", 4, 8, 2, 128, 1, 32, (129, 128, 160, 97), False, 96, 66, False),
    ("win93_paged_sa4_span_bound", 3, 8, 2, 128, 4, 32, (159, 127, 1000), True, 64, 93, False),
]


@pytest.mark.parametrize("case", WINDOW, ids=lambda c: c[0])
def test_decode_window(case, cuda_device):
    name, b, hq, hkv, d, sa, page, lens, paged, chunk, win, e4m3 = case
    w = C.DecodeWorkload(name, b, hq, hkv, d, sa, page_size=page, len_hi=max(lens) + 7,
                         paged=paged, fixed_lens=lens, seed=0x3100 + len(name))
    t = (C.decode_inputs_e4m3_torch if e4m3 else C.decode_inputs_torch)(w, cuda_device)
    o, lse = decode_ex(t, w, kv_chunk=chunk, window=win)
    o_ref, lse_ref = oracle.decode_ext(bits_of(t["q"]), as_bf16_bits(t["k_cache"]),
                                       as_bf16_bits(t["v_cache"]), t["table"], t["lens"], w.scale,
                                       window=win)
    assert_o_close(o.cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)


def ring_of(t, w, cap):
    """A circular flat cache of cap rows holding each sequence's last cap positions of the
    flat cache t (position j at row j mod cap; rows never written hold NaN)."""
    nan = torch.tensor(rng.BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    rings = []
    for c in ("k_cache", "v_cache"):
        full = t[c] if t[c].dtype == torch.bfloat16 else t[c].to(torch.bfloat16)
        r = torch.full((w.b, w.hkv, cap, w.d), nan, dtype=torch.bfloat16, device=full.device)
        for i, n in enumerate(t["lens"]):
            js = torch.arange(max(0, int(n) - cap), int(n), device=full.device)
            r[i, :, js % cap] = full[i, :, js]
        rings.append(r if t[c].dtype == torch.bfloat16 else r.to(t[c].dtype))
    return rings


CIRCULAR = [
    # name, b, hq, hkv, d, s_active, lens, cap, window, kv_chunk, e4m3
    ("ring256_sa1", 3, 8, 2, 128, 1, (40, 1030, 700), 256, 256, 64, False),
    ("ring512_sa4_wrapped", 2, 8, 2, 128, 4, (1500, 513), 512, 400, 128, False),
    ("ring96_sa2_d64", 2, 4, 1, 64, 2, (95, 1000), 96, 95, 32, False),
    ("ring256_d256_e4m3", 2, 4, 2, 256, 3, (900, 41), 256, 200, 64, True),
    ("ring288_e4m3_d128", 2, 8, 2, 128, 2, (1000, 150), 288, 250, 96, True),
]


@pytest.mark.parametrize("case", CIRCULAR, ids=lambda c: c[0])
def test_decode_circular_cache(case, cuda_device):
    name, b, hq, hkv, d, sa, lens, cap, win, chunk, e4m3 = case
    w = C.DecodeWorkload(name, b, hq, hkv, d, sa, len_hi=max(lens) + 3, paged=False,
                         fixed_lens=lens, seed=0x3200 + len(name))
    full = (C.decode_inputs_e4m3_torch if e4m3 else C.decode_inputs_torch)(w, cuda_device)
    kr, vr = ring_of(full, w, cap)
    t = dict(full, k_cache=kr, v_cache=vr, max_cache_len=cap)
    o, lse = decode_ex(t, w, kv_chunk=chunk, window=win, circular=True)
    o_ref, lse_ref = oracle.decode_ext(bits_of(t["q"]), as_bf16_bits(kr), as_bf16_bits(vr), None,
                                       t["lens"], w.scale, window=win, circular=True)
    assert_o_close(o.cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)


@pytest.mark.parametrize("paged,d,sa", [(True, 128, 1), (True, 128, 4), (False, 64, 3),
                                        (True, 256, 2)])
def test_decode_rope_of_the_queries(paged, d, sa, cuda_device):
    hq, hkv = 8, 2
    w = C.DecodeWorkload(f"rope_{paged}_{d}_{sa}", 3, hq, hkv, d, sa, len_hi=3000, paged=paged,
                         fixed_lens=(40, 2990, 777), seed=0x3300 + d + sa)
    t = C.decode_inputs_torch(w, cuda_device)
    f = inv_freq(d)
    o, lse = decode_ex(t, w, kv_chunk=256, rope_inv_freq=torch.from_numpy(f).to(cuda_device))
    o_ref, lse_ref = oracle.decode_ext(bits_of(t["q"]), bits_of(t["k_cache"]),
                                       bits_of(t["v_cache"]), t["table"], t["lens"], w.scale,
                                       inv_freq=f.astype(np.float64))
    assert_o_close(o.cpu().numpy(), o_ref, w.name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, w.name)


def _append_case(cuda_device, paged, circular, d, sa, lens, cap=None, seed=0x3400):
    """A decode step as a serving loop runs it: the new tokens' K/V are appended (RoPE'd
    K) into a cache whose new slots hold NaN, then decode attends with RoPE'd queries."""
    import flash_attention_forward_attn_gb300 as A

    hq, hkv = 8, 2
    w = C.DecodeWorkload(f"append_{paged}_{circular}_{d}", len(lens), hq, hkv, d, sa,
                         len_hi=max(lens) + 5, paged=paged, fixed_lens=lens, seed=seed + d + sa)
    t = C.decode_inputs_torch(w, cuda_device)
    if circular:
        kr, vr = ring_of(t, w, cap)
        t = dict(t, k_cache=kr, v_cache=vr, max_cache_len=cap)
    kn = rng.normal_bf16_np(rng.stream_seed(w.seed, "k_new"), 0, w.b * hkv * sa * d).reshape(
        w.b, hkv, sa, d)
    vn = rng.normal_bf16_np(rng.stream_seed(w.seed, "v_new"), 0, w.b * hkv * sa * d).reshape(
        w.b, hkv, sa, d)
    # the new tokens' slots start as NaN: only the append fills them
    nan = rng.BF16_NAN_BITS
    kc, vc = bits_of(t["k_cache"]).copy(), bits_of(t["v_cache"]).copy()
    slots = []
    for i, n in enumerate(t["lens"]):
        for j in range(int(n) - sa, int(n)):
            if paged:
                slots.append((int(t["table"][i, j // w.page_size]), slice(None), j % w.page_size))
            else:
                slots.append((i, slice(None), j % cap if circular else j))
    for s_ in slots:
        kc[s_] = nan
        vc[s_] = nan
    k_cache, v_cache = tensor_of_bits(kc, cuda_device), tensor_of_bits(vc, cuda_device)
    f = inv_freq(d)
    ft = torch.from_numpy(f).to(cuda_device)
    A.attn_append_kv(tensor_of_bits(kn, cuda_device), tensor_of_bits(vn, cuda_device), k_cache,
                     v_cache, t["block_table"], t["cache_len"], max_cache_len=t["max_cache_len"],
                     circular=circular, rope_inv_freq=ft)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    # the append wrote exactly the new slots: V bit for bit, K the rotated rows in bf16
    kg, vg = bits_of(k_cache), bits_of(v_cache)
    mask = np.zeros(kc.shape, bool)
    for s_ in slots:
        mask[s_] = True
    np.testing.assert_array_equal(kg[~mask], kc[~mask])
    np.testing.assert_array_equal(vg[~mask], vc[~mask])
    kf = rng.bf16_bits_to_f32_np(kg).astype(np.float64)
    for i, n in enumerate(t["lens"]):
        for tt, j in enumerate(range(int(n) - sa, int(n))):
            s_ = slots[i * sa + tt]
            vrow = vg[s_[0], :, s_[2]]
            np.testing.assert_array_equal(vrow, vn[i, :, tt])
            for g in range(hkv):
                ref = oracle.rope_row(rng.bf16_bits_to_f32_np(kn[i, g, tt]).astype(np.float64),
                                      j, f.astype(np.float64))
                got = kf[s_[0], g, s_[2]]
                assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6), (i, j, g)
    t2 = dict(t, k_cache=k_cache, v_cache=v_cache)
    o, lse = decode_ex(t2, w, kv_chunk=64, rope_inv_freq=ft,
                       **(dict(window=cap - sa + 1, circular=True) if circular else {}))
    o_ref, lse_ref = oracle.decode_ext(bits_of(t["q"]), kc, vc, t["table"], t["lens"], w.scale,
                                       window=(cap - sa + 1) if circular else 0, circular=circular,
                                       k_new=kn, v_new=vn, inv_freq=f.astype(np.float64))
    assert_o_close(o.cpu().numpy(), o_ref, w.name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, w.name)


@pytest.mark.parametrize("d,sa", [(128, 1), (128, 4), (64, 2)])
def test_append_then_decode_paged(d, sa, cuda_device):
    _append_case(cuda_device, True, False, d, sa, (40, 1030, 77))


def test_append_then_decode_flat(cuda_device):
    _append_case(cuda_device, False, False, 256, 2, (9, 300))


def test_append_then_decode_circular(cuda_device):
    _append_case(cuda_device, False, True, 128, 3, (1000, 150, 511), cap=256)


def test_decode_window_repeat_runs_bit_identical(cuda_device):
    w = C.PAGED_DECODE_SPEC4.with_(b=8, len_hi=4096)
    t = C.decode_inputs_torch(w, cuda_device)
    f = torch.from_numpy(inv_freq(w.d)).to(cuda_device)
    o0, l0 = decode_ex(t, w, window=1000, rope_inv_freq=f)
    for _ in range(10):
        o1, l1 = decode_ex(t, w, window=1000, rope_inv_freq=f)
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


def _one_sequence(t, w, b):
    """Sequence b of a paged cache gathered into a one-sequence flat cache (bf16 bits) for
    the oracle, with its query rows and cache length."""
    n = int(t["lens"][b])
    npg = -(-n // w.page_size)
    idx = torch.from_numpy(t["table"][b, :npg].astype(np.int64)).to(t["q"].device)
    flat = [bits_of(t[c][idx].permute(1, 0, 2, 3).reshape(1, w.hkv, npg * w.page_size, w.d)
                    [:, :, :n].contiguous()) for c in ("k_cache", "v_cache")]
    return bits_of(t["q"][b:b + 1]), flat[0], flat[1], np.array([n], np.int32)


def test_window_rope_decode_full_size_sampled(cuda_device):
    """The benchmark's windowed decode with RoPE of the queries (64 sequences, 4 new tokens,
    window 4096, inverse frequencies 10000^(-2i/d)), in the launch the benchmark times;
    sequences are checked one by one against the oracle over their gathered pages."""
    w = C.PAGED_DECODE_SPEC4
    t = C.decode_inputs_torch(w, cuda_device)
    f = inv_freq(w.d)
    o, lse = decode_ex(t, w, window=4096, rope_inv_freq=torch.from_numpy(f).to(cuda_device))
    lens = t["lens"]
    for b in sorted({int(np.argmax(lens)), int(np.argmin(lens)), 5, 41}):
        q, fk, fv, cl = _one_sequence(t, w, b)
        o_ref, lse_ref = oracle.decode_ext(q, fk, fv, None, cl, w.scale, window=4096,
                                           inv_freq=f.astype(np.float64))
        assert_o_close(o[b:b + 1].cpu().numpy(), o_ref, f"window+rope b{b}")
        assert_lse_close(lse[b:b + 1].cpu().numpy(), lse_ref, f"window+rope b{b}")


def test_sink_decode_full_size_sampled(cuda_device):
    """The benchmark's decode with per-head sink logits (64 sequences, 1 new token), checked
    on sampled sequences against the oracle with the same sinks."""
    w = C.PAGED_DECODE
    t = C.decode_inputs_torch(w, cuda_device)
    sk = C.sink_logits(w.hq)
    o, lse = decode_ex(t, w, sink=torch.from_numpy(sk).to(cuda_device))
    lens = t["lens"]
    for b in sorted({int(np.argmax(lens)), int(np.argmin(lens)), 9, 50}):
        q, fk, fv, cl = _one_sequence(t, w, b)
        o_ref, lse_ref = oracle.decode(q, fk, fv, None, cl, w.scale, sink=sk)
        assert_o_close(o[b:b + 1].cpu().numpy(), o_ref, f"sink b{b}")
        assert_lse_close(lse[b:b + 1].cpu().numpy(), lse_ref, f"sink b{b}")
