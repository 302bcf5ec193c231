"""The seeded input generator: numpy and torch sides agree bit for bit, slices of a
stream regenerate independently, bf16 rounding is nearest-even, and the decode
workload's lengths, page table and padding follow the recipe."""
import numpy as np
import pytest
import torch

from workloads import configs as C
from workloads import rng


def test_splitmix64_reference_values():
    # First outputs of SplitMix64 seeded with 0 (published test vector of splitmix64.c).
    got = rng.u64_np(0, 0, 3)
    assert [int(x) for x in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_numpy_and_torch_agree_bit_for_bit():
    s = rng.stream_seed(7, "q")
    a = rng.normal_bf16_np(s, 12345, 200_000)
    b = rng.normal_bf16_torch(s, 12345, 200_000, "cpu").view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(a, b)
    ua = rng.uniform_np(s, 5, 1000)
    ub = rng.uniform_torch(s, 5, 1000, "cpu").numpy()
    np.testing.assert_array_equal(ua, ub)


def test_counter_slices_regenerate():
    s = rng.stream_seed(3, "k")
    whole = rng.normal_bf16_np(s, 0, 5000)
    np.testing.assert_array_equal(whole[1234:2345], rng.normal_bf16_np(s, 1234, 1111))


def test_streams_differ_and_moments():
    a = rng.bf16_bits_to_f32_np(rng.normal_bf16_np(rng.stream_seed(1, "q"), 0, 400_000))
    b = rng.bf16_bits_to_f32_np(rng.normal_bf16_np(rng.stream_seed(1, "k"), 0, 400_000))
    assert not np.array_equal(a, b)
    for x in (a, b):
        assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_bf16_round_to_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 1.0 + 2 ** -8 + 2 ** -20],
                 dtype=np.float32)
    got = rng.bf16_bits_to_f32_np(rng.f32_to_bf16_bits_np(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0 + 2 ** -6, -1.0, 1.0 + 2 ** -7], np.float32))
    t = rng.f32_to_bf16_torch(torch.from_numpy(x)).float().numpy()
    np.testing.assert_array_equal(t, got)


def test_prefill_rows_match_full_generation():
    w = C.GQA_PREFILL_32K.with_(sq=64, skv=64, hq=4, hkv=2)
    q, k, v = C.prefill_inputs_np(w)
    tq, tk, tv = C.prefill_inputs_torch(w, "cpu")
    for a, t in ((q, tq), (k, tk), (v, tv)):
        np.testing.assert_array_equal(a, t.contiguous().view(torch.int16).numpy().view(np.uint16))
    x = rng.bf16_bits_to_f32_np(q)
    frac = np.mean(np.abs(x) > 4.5)  # almost only outliers exceed 4.5 sigma
    assert 0.004 < frac < 0.02


def test_decode_workload_recipe():
    w = C.PAGED_DECODE
    lens = C.decode_cache_lens(w)
    assert lens.min() >= 1024 and lens.max() <= 32768 and len(lens) == 64
    table, total = C.decode_block_table(w, lens)
    used = np.concatenate([table[b, : -(-lens[b] // 32)] for b in range(64)])
    np.testing.assert_array_equal(np.sort(used), np.arange(total, dtype=np.uint32))
    assert not np.array_equal(used, np.arange(total))
    assert (table[0, -(-lens[0] // 32):] == 0xFFFFFFFF).all()


def test_decode_inputs_place_logical_rows_and_nan_padding():
    w = C.PAGED_DECODE_SPEC4.with_(b=3, hq=4, hkv=2, d=16, fixed_lens=(37, 64, 5), len_hi=96)
    t = C.decode_inputs_torch(w, "cpu")
    kc = t["k_cache"].view(torch.int16).numpy().view(np.uint16)
    for b, n in enumerate(t["lens"]):
        for g in range(2):
            logical = C.decode_kv_logical_np(w, "k", b, g, int(n))
            for j in (0, n - 5, n - 1):
                np.testing.assert_array_equal(kc[t["table"][b, j // 32], g, j % 32], logical[j])
        last = t["table"][b, (n - 1) // 32]
        if n % 32:
            assert np.isnan(rng.bf16_bits_to_f32_np(kc[last, :, n % 32:])).all()
    q = t["q"].view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(q[2, 3], C.decode_q_np(w, 2, 3))
