"""Pins of the fp64 oracle to facts outside itself.

Each test ties the oracle to something the pages or the mathematics fix: hand-worked
golden cases, closed forms, invariants of the softmax, an independent library routine
(PyTorch's scaled_dot_product_attention in float64, scipy's logsumexp), and brute-force
cross-mode identities.  Together they are chosen so that a dropped term, a wrong sign,
a wrong index, a wrong head map or a transposed operand fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import rng

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiny_cases.json")


def bits(x):
    """float values that are exact in bf16 -> bf16 bit patterns."""
    b = rng.f32_to_bf16_bits_np(np.asarray(x, dtype=np.float32))
    assert np.array_equal(rng.bf16_bits_to_f32_np(b), np.asarray(x, dtype=np.float32))
    return b


def rand_bits(seed, shape, name="x"):
    n = int(np.prod(shape))
    return rng.normal_bf16_np(rng.stream_seed(seed, name), 0, n).reshape(shape)


def f64(b):
    return rng.bf16_bits_to_f32_np(b).astype(np.float64)


def frac_arr(a):
    return np.vectorize(lambda nd: float(Fraction(nd[0], nd[1])), signature="(n)->()")(np.asarray(a))


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- golden
@pytest.mark.parametrize("case", load_golden()["prefill"], ids=lambda c: c["name"])
def test_golden_prefill(case):
    q = bits(case["q"])[None]
    k = bits(case["k"])[None]
    v = bits(case["v"])[None]
    o, lse = oracle.prefill(q, k, v, math.log(case["scale_exp"]), case["causal"], case["window"])
    np.testing.assert_allclose(o[0], frac_arr(case["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], np.log(np.asarray(case["lse_exp"], dtype=np.float64)),
                               rtol=0, atol=1e-13)


@pytest.mark.parametrize("case", load_golden()["decode"], ids=lambda c: c["name"])
def test_golden_decode_paged(case):
    page, n = case["page"], case["cache_len"]
    lk, lv = bits(case["logical_k"]), bits(case["logical_v"])
    table = np.asarray([case["block_table"]], dtype=np.uint32)
    npages = len(case["block_table"])
    kc = np.full((npages, 1, page, case["d"]), rng.BF16_NAN_BITS, dtype=np.uint16)
    vc = kc.copy()
    for j in range(n):
        kc[table[0, j // page], 0, j % page] = lk[j]
        vc[table[0, j // page], 0, j % page] = lv[j]
    q = bits(case["q"])[None]
    o, lse = oracle.decode(q, kc, vc, table, np.array([n], dtype=np.int32),
                           math.log(case["scale_exp"]))
    np.testing.assert_allclose(o[0, 0], frac_arr(case["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.log(np.asarray(case["lse_exp"], float)), atol=1e-13)
    m = oracle.decode_mask(np.array([n], np.int32), 1, case["s_active"], case["mask_max_len"])
    np.testing.assert_array_equal(m[0, 0], np.asarray(case["mask"], dtype=np.uint8))


# ----------------------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal,window,sq,skv", [(0, 0, 40, 56), (1, 0, 48, 48), (1, 7, 40, 56),
                                                  (1, 0, 60, 20)])
def test_rows_of_p_sum_to_one_and_masked_p_is_zero(causal, window, sq, skv):
    d = 16
    q, k, v = rand_bits(1, (sq, d), "q"), rand_bits(1, (skv, d), "k"), rand_bits(1, (skv, d), "v")
    qp = np.array([oracle.q_pos(i, sq, skv) for i in range(sq)])
    o, lse, p = oracle.attention_rows(q, k, v, qp, 0.3, causal, window, want_p=True)
    for r in range(sq):
        allowed = np.array([oracle.allowed(j, skv, qp[r], causal, window) for j in range(skv)])
        if allowed.any():
            assert abs(p[r].sum() - 1.0) < 1e-12
            assert (p[r][allowed] > 0).all()
            np.testing.assert_allclose(o[r], p[r] @ f64(v), atol=1e-12)
        else:  # fully masked row (queries before the first key): O = 0, LSE = -inf
            assert lse[r] == -np.inf and (o[r] == 0).all()
        assert (p[r][~allowed] == 0.0).all()


def test_allowed_predicate_counts_by_hand():
    # sq = skv = 6, causal, window 3: row i sees keys max(0, i-2) .. i -> 1, 2, 3, 3, 3, 3
    counts = [sum(oracle.allowed(j, 6, i, 1, 3) for j in range(6)) for i in range(6)]
    assert counts == [1, 2, 3, 3, 3, 3]
    # causal only: row i sees i + 1 keys
    assert [sum(oracle.allowed(j, 6, i, 1, 0) for j in range(6)) for i in range(6)] == [1, 2, 3, 4, 5, 6]
    # queries at the tail: 2 queries after 5 keys sit at positions 3 and 4
    assert [oracle.q_pos(i, 2, 5) for i in range(2)] == [3, 4]
    # keys at or past skv are never allowed
    assert not oracle.allowed(5, 5, 9, 0, 0) and not oracle.allowed(-1, 5, 3, 0, 0)


def test_gqa_head_map_by_hand():
    assert [oracle.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head(h, 6, 3) for h in range(6)] == [0, 0, 1, 1, 2, 2]
    assert [oracle.kv_head(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]


def test_constant_v_gives_that_constant():
    sq, skv, d = 24, 40, 8
    q, k = rand_bits(2, (1, 1, sq, d), "q"), rand_bits(2, (1, 1, skv, d), "k")
    c = np.array([0.75, -2.0, 3.5, 0.0, 1.0, -0.125, 8.0, 0.5], dtype=np.float32)
    v = np.broadcast_to(bits(c), (1, 1, skv, d)).copy()
    for causal, window in [(0, 0), (1, 0), (1, 5)]:
        o, _ = oracle.prefill(q, k, v, 0.7, causal, window)
        np.testing.assert_allclose(o[0, 0], np.broadcast_to(c, (sq, d)), rtol=0, atol=1e-12)


def test_single_allowed_key_gives_its_v_row_and_score():
    # window 1 with causal: each row sees only its own position
    sq = skv = 20
    d = 8
    q, k, v = (rand_bits(3, (1, 1, sq, d), n) for n in "qkv")
    scale = 0.37
    o, lse = oracle.prefill(q, k, v, scale, 1, 1)
    np.testing.assert_array_equal(o[0, 0], f64(v[0, 0]))
    s_diag = scale * np.einsum("ix,ix->i", f64(q[0, 0]), f64(k[0, 0]))
    np.testing.assert_allclose(lse[0, 0], s_diag, atol=1e-12)


def test_first_causal_row_is_v0():
    q, k, v = (rand_bits(4, (1, 2, 16, 8), n) for n in "qkv")
    o, _ = oracle.prefill(q, k, v, 0.5, 1, 0)
    np.testing.assert_array_equal(o[0, :, 0], f64(v[0, :, 0]))


@pytest.mark.parametrize("causal,window,sq,skv,counts", [
    (1, 3, 6, 6, [1, 2, 3, 3, 3, 3]),
    (1, 3, 4, 6, [3, 3, 3, 3]),
    (1, 0, 3, 5, [3, 4, 5]),
    (0, 0, 3, 5, [5, 5, 5]),
])
def test_zero_q_gives_mean_of_allowed_v_and_log_count(causal, window, sq, skv, counts):
    d = 4
    q = np.zeros((1, 1, sq, d), dtype=np.uint16)
    k, v = rand_bits(5, (1, 1, skv, d), "k"), rand_bits(5, (1, 1, skv, d), "v")
    o, lse = oracle.prefill(q, k, v, 1.0, causal, window)
    vf = f64(v[0, 0])
    for i, c in enumerate(counts):
        last = i + skv - sq  # the row's own position: the newest allowed key when causal
        hi = last if causal else skv - 1
        np.testing.assert_allclose(o[0, 0, i], vf[hi - c + 1: hi + 1].mean(0), atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(c)) < 1e-12


def test_changing_masked_kv_changes_nothing():
    sq = skv = 32
    d = 8
    q, k, v = (rand_bits(6, (1, 1, sq, d), n) for n in "qkv")
    o1, l1 = oracle.prefill(q, k, v, 0.4, 1, 9)
    # rows 20..31 never see keys < 11 (window 9) nor keys after themselves
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, :11] = rand_bits(7, (11, d), "k")
    v2[0, 0, :11] = rng.BF16_NAN_BITS
    o2, l2 = oracle.prefill(q, k2, v2, 0.4, 1, 9)
    np.testing.assert_array_equal(o1[0, 0, 20:], o2[0, 0, 20:])
    np.testing.assert_array_equal(l1[0, 0, 20:], l2[0, 0, 20:])
    assert not np.array_equal(o1[0, 0, :20], o2[0, 0, :20])


def test_noncausal_key_permutation_invariance():
    sq, skv, d = 12, 50, 8
    q, k, v = (rand_bits(8, (1, 1, n_, d), n) for n_, n in ((sq, "q"), (skv, "k"), (skv, "v")))
    perm = np.argsort(rng.u64_np(99, 0, skv), kind="stable")
    o1, l1 = oracle.prefill(q, k, v, 0.6, 0, 0)
    o2, l2 = oracle.prefill(q, k[:, :, perm], v[:, :, perm], 0.6, 0, 0)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    # a causal mask is not permutation invariant: the same permutation must change it
    o3, _ = oracle.prefill(q, k, v, 0.6, 1, 0)
    o4, _ = oracle.prefill(q, k[:, :, perm], v[:, :, perm], 0.6, 1, 0)
    assert not np.allclose(o3, o4)


def test_gqa_equals_mha_with_repeated_kv():
    b, hq, hkv, s, d = 2, 6, 2, 20, 8
    q = rand_bits(9, (b, hq, s, d), "q")
    k, v = rand_bits(9, (b, hkv, s, d), "k"), rand_bits(9, (b, hkv, s, d), "v")
    o1, l1 = oracle.prefill(q, k, v, 0.3, 1, 0)
    rep = hq // hkv
    o2, l2 = oracle.prefill(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1), 0.3, 1, 0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ----------------------------------------------------------------------------- library routines
def test_matches_torch_sdpa_float64():
    """PyTorch's scaled_dot_product_attention (float64, CPU) is an independent implementation
    of the same definition: its own causal triangle and its own GQA expansion."""
    import torch
    import torch.nn.functional as F

    b, hq, hkv, s, d = 2, 8, 2, 70, 32
    q = rand_bits(10, (b, hq, s, d), "q")
    k, v = rand_bits(10, (b, hkv, s, d), "k"), rand_bits(10, (b, hkv, s, d), "v")
    t = lambda a: torch.from_numpy(f64(a))
    scale = 1 / math.sqrt(d)
    for causal in (0, 1):
        o, _ = oracle.prefill(q, k, v, scale, causal, 0)
        ref = F.scaled_dot_product_attention(t(q), t(k).repeat_interleave(hq // hkv, 1),
                                             t(v).repeat_interleave(hq // hkv, 1),
                                             is_causal=bool(causal), scale=scale)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_lse_matches_scipy_logsumexp():
    from scipy.special import logsumexp

    sq, skv, d = 10, 33, 16
    q, k, v = (rand_bits(11, (1, 1, n_, d), n) for n_, n in ((sq, "q"), (skv, "k"), (skv, "v")))
    _, lse = oracle.prefill(q, k, v, 0.25, 0, 0)
    s = 0.25 * f64(q[0, 0]) @ f64(k[0, 0]).T
    np.testing.assert_allclose(lse[0, 0], logsumexp(s, axis=1), atol=1e-12)


# ----------------------------------------------------------------------------- decode
def _flat_and_paged(seed, b, hkv, d, lens, page, permute):
    max_len = int(max(lens))
    flat_k = np.full((b, hkv, max_len, d), rng.BF16_NAN_BITS, dtype=np.uint16)
    flat_v = flat_k.copy()
    for i, n in enumerate(lens):
        flat_k[i, :, :n] = rand_bits(seed + i, (hkv, n, d), "k")
        flat_v[i, :, :n] = rand_bits(seed + i, (hkv, n, d), "v")
    npg = [-(-n // page) for n in lens]
    total = sum(npg)
    phys = (np.argsort(rng.u64_np(seed, 0, total), kind="stable") if permute
            else np.arange(total)).astype(np.uint32)
    maxp = -(-max_len // page)
    table = np.full((b, maxp), 0xFFFFFFFF, dtype=np.uint32)
    kc = np.full((total, hkv, page, d), rng.BF16_NAN_BITS, dtype=np.uint16)
    vc = kc.copy()
    off = 0
    for i, n in enumerate(lens):
        table[i, : npg[i]] = phys[off: off + npg[i]]
        off += npg[i]
        for j in range(n):
            kc[table[i, j // page], :, j % page] = flat_k[i, :, j]
            vc[table[i, j // page], :, j % page] = flat_v[i, :, j]
    return flat_k, flat_v, kc, vc, table


def test_decode_equals_last_rows_of_causal_prefill():
    hq, hkv, d, n, sa = 4, 2, 16, 45, 3
    fk, fv, _, _, _ = _flat_and_paged(20, 1, hkv, d, [n], 8, False)
    q = rand_bits(21, (1, hq, sa, d), "q")
    o_dec, l_dec = oracle.decode(q, fk, fv, None, np.array([n], np.int32), 0.2)
    # prefill with sq = s_active queries at the tail of n keys
    o_pre, l_pre = oracle.prefill(q, fk[:, :, :n], fv[:, :, :n], 0.2, 1, 0)
    np.testing.assert_array_equal(o_dec, o_pre)
    np.testing.assert_array_equal(l_dec, l_pre)


def test_decode_paged_permuted_equals_identity_equals_flat():
    b, hq, hkv, d, page, sa = 3, 4, 2, 8, 4, 2
    lens = [9, 16, 5]
    q = rand_bits(30, (b, hq, sa, d), "q")
    cl = np.array(lens, np.int32)
    fk, fv, kc, vc, table = _flat_and_paged(31, b, hkv, d, lens, page, True)
    _, _, kc2, vc2, table2 = _flat_and_paged(31, b, hkv, d, lens, page, False)
    assert not np.array_equal(table, table2)
    o1, l1 = oracle.decode(q, kc, vc, table, cl, 0.3)
    o2, l2 = oracle.decode(q, kc2, vc2, table2, cl, 0.3)
    o3, l3 = oracle.decode(q, fk, fv, None, cl, 0.3)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(l1, l3)
    assert np.isfinite(o1).all()  # NaN padding slots never leak


def test_decode_single_cached_key():
    d = 8
    fk, fv, _, _, _ = _flat_and_paged(40, 1, 1, d, [1], 4, False)
    q = rand_bits(41, (1, 2, 1, d), "q")
    o, lse = oracle.decode(q, fk, fv, None, np.array([1], np.int32), 0.5)
    np.testing.assert_array_equal(o[0, :, 0], np.broadcast_to(f64(fv[0, 0, 0]), (2, d)))
    np.testing.assert_allclose(lse[0, :, 0], 0.5 * f64(q[0, :, 0]) @ f64(fk[0, 0, 0]), atol=1e-12)


def test_gather_rejects_out_of_range_page():
    cache = np.zeros((2, 1, 4, 2), np.uint16)
    with pytest.raises(RuntimeError, match="page index"):
        oracle.gather_paged(cache, np.array([0, 2], np.uint32), 2, 0, 6)


def test_decode_mask_structure():
    lens = np.array([5, 9, 4], np.int32)
    sa, max_len = 4, 12
    m = oracle.decode_mask(lens, 2, sa, max_len)
    for b, n in enumerate(lens):
        for t in range(sa):
            # each query row sees exactly the prefix up to its own position
            assert m[b, 0, t].sum() == n - sa + t + 1
            assert (m[b, 0, t, n:] == 0).all()
        # the new tokens' block is tril(ones) and the prior block is all ones
        np.testing.assert_array_equal(m[b, 1, :, n - sa: n], np.tril(np.ones((sa, sa), np.uint8)))
        assert (m[b, 1, :, : n - sa] == 1).all()
    # one new token: the mask is exactly the length cut (type A)
    m1 = oracle.decode_mask(lens, 1, 1, max_len)
    np.testing.assert_array_equal(m1[:, 0, 0], (np.arange(max_len)[None] < lens[:, None]))


# ----------------------------------------------------------------------------- attention sink
# The sink is one logit per query head that joins the row's maximum and sum and has no
# value row (Flash-Attention: Context (CTE), "Algorithm - the per-section max update" and
# "Algorithm - fused exp and the running sum"; TKG keeps it per query head).

def test_sink_of_minus_inf_is_no_sink():
    b, hq, hkv, sq, skv, d = 1, 4, 2, 12, 20, 8
    q = rand_bits(50, (b, hq, sq, d), "q")
    k, v = rand_bits(50, (b, hkv, skv, d), "k"), rand_bits(50, (b, hkv, skv, d), "v")
    for causal, window in [(0, 0), (1, 0), (1, 5)]:
        o1, l1 = oracle.prefill(q, k, v, 0.3, causal, window)
        o2, l2 = oracle.prefill(q, k, v, 0.3, causal, window, sink=np.full(hq, -np.inf))
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)
    fk, fv, _, _, _ = _flat_and_paged(51, 1, hkv, d, [17], 8, False)
    qd = rand_bits(52, (1, hq, 2, d), "q")
    cl = np.array([17], np.int32)
    o1, l1 = oracle.decode(qd, fk, fv, None, cl, 0.3)
    o2, l2 = oracle.decode(qd, fk, fv, None, cl, 0.3, sink=np.full(hq, -np.inf))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("causal,window,sq,skv,counts", [
    (1, 3, 6, 6, [1, 2, 3, 3, 3, 3]),
    (1, 0, 3, 5, [3, 4, 5]),
    (0, 0, 3, 5, [5, 5, 5]),
])
def test_zero_q_with_sink_closed_form(causal, window, sq, skv, counts):
    """All allowed scores are 0, so with n allowed keys and sink s the row's weights are
    1 / (n + e^s) per key: O = mean(allowed V) * n / (n + e^s), LSE = ln(n + e^s)."""
    d = 4
    sinks = np.array([0.5, -1.25, 30.0, 1000.0])
    hq = len(sinks)
    q = np.zeros((1, hq, sq, d), dtype=np.uint16)
    k, v = rand_bits(53, (1, 1, skv, d), "k"), rand_bits(53, (1, 1, skv, d), "v")
    o, lse = oracle.prefill(q, k, v, 1.0, causal, window, sink=sinks)
    vf = f64(v[0, 0])
    for h, s in enumerate(sinks):
        for i, c in enumerate(counts):
            last = i + skv - sq
            hi = last if causal else skv - 1
            mean = vf[hi - c + 1: hi + 1].mean(0)
            if s < 700:
                np.testing.assert_allclose(o[0, h, i], mean * c / (c + math.exp(s)), rtol=1e-12,
                                           atol=1e-300)
                assert abs(lse[0, h, i] - math.log(c + math.exp(s))) < 1e-12
            else:  # e^s overflows a double: the row's mass is all on the sink
                np.testing.assert_allclose(o[0, h, i], mean * c * math.exp(-s), rtol=1e-12,
                                           atol=1e-300)
                assert abs(lse[0, h, i] - (s + math.log1p(c * math.exp(-s)))) < 1e-9


def test_row_with_only_the_sink():
    """Queries before the first key (sq > skv, causal) allow no key: O = 0, LSE = sink."""
    hq, sq, skv, d = 2, 6, 3, 4
    q = rand_bits(54, (1, hq, sq, d), "q")
    k, v = rand_bits(54, (1, 1, skv, d), "k"), rand_bits(54, (1, 1, skv, d), "v")
    sinks = np.array([0.75, -2.5])
    o, lse = oracle.prefill(q, k, v, 0.5, 1, 0, sink=sinks)
    for i in range(sq - skv):  # q_pos = i + skv - sq < 0
        np.testing.assert_array_equal(o[0, :, i], 0.0)
        np.testing.assert_array_equal(lse[0, :, i], sinks)
    o0, _ = oracle.prefill(q, k, v, 0.5, 1, 0)
    np.testing.assert_array_equal(o0[0, :, : sq - skv], 0.0)


def _sink_as_key(q, k, v, scale, sink_val):
    """The sink written as an ordinary key at position 0 of an extended problem: one more
    head dimension holding 1 in every query and sink/scale in the extra key (0 in the
    real keys), a zero value row, and a zero extra value column.  Requires sink/scale
    exact in bf16."""
    b, hq, sq, d = q.shape
    _, hkv, skv, _ = k.shape
    one = bits(np.array([1.0], np.float32))[0]
    ks = bits(np.array([sink_val / scale], np.float32))[0]
    q2 = np.concatenate([q, np.full((b, hq, sq, 1), one, np.uint16)], axis=3)
    k2 = np.zeros((b, hkv, skv + 1, d + 1), np.uint16)
    k2[:, :, 1:, :d] = k
    k2[:, :, 0, d] = ks
    v2 = np.zeros((b, hkv, skv + 1, d + 1), np.uint16)
    v2[:, :, 1:, :d] = v
    return q2, k2, v2


@pytest.mark.parametrize("causal", [0, 1])
def test_sink_equals_an_extra_zero_value_key(causal):
    """The pages append the sink as one more column of the max and of the sum; the same
    row, built as an ordinary key (score = sink, value 0) through the no-sink oracle,
    must give the same O and LSE.  The extra key sits at position 0, which every causal
    row with q_pos >= -1 sees."""
    b, hq, hkv, sq, skv, d, scale, s = 1, 2, 1, 9, 14, 8, 0.5, 1.5
    q = rand_bits(55, (b, hq, sq, d), "q")
    k, v = rand_bits(55, (b, hkv, skv, d), "k"), rand_bits(55, (b, hkv, skv, d), "v")
    o1, l1 = oracle.prefill(q, k, v, scale, causal, 0, sink=np.full(hq, s))
    q2, k2, v2 = _sink_as_key(q, k, v, scale, s)
    o2, l2 = oracle.prefill(q2, k2, v2, scale, causal, 0)
    np.testing.assert_array_equal(o2[..., d], 0.0)
    np.testing.assert_allclose(o1, o2[..., :d], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_decode_sink_equals_an_extra_zero_value_key():
    hq, hkv, d, n, sa, scale, s = 4, 2, 8, 21, 2, 0.25, -0.75
    fk, fv, _, _, _ = _flat_and_paged(56, 1, hkv, d, [n], 8, False)
    q = rand_bits(57, (1, hq, sa, d), "q")
    sinks = np.full(hq, s)
    o1, l1 = oracle.decode(q, fk, fv, None, np.array([n], np.int32), scale, sink=sinks)
    q2, k2, v2 = _sink_as_key(q, fk[:, :, :n], fv[:, :, :n], scale, s)
    o2, l2 = oracle.decode(q2, k2, v2, None, np.array([n + 1], np.int32), scale)
    np.testing.assert_allclose(o1, o2[..., :d], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- e4m3 KV cache
# An FP8-e4m3 KV cache (Flash-Attention: Decode (TKG), "Decode (TKG) vs context (CTE) - the
# diff"): a cache byte stands for e4m3(byte) * k_scale (K) or * v_scale (V).

def test_e4m3_decoding_matches_torch_float8():
    """All 256 codes against PyTorch's own float8_e4m3fn -> float conversion."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(ours, ref, equal_nan=True)
    assert np.isnan(ours[[0x7F, 0xFF]]).all() and np.isfinite(np.delete(ours, [0x7F, 0xFF])).all()
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _e4m3_codes(seed, n):
    """Seeded e4m3 codes without the NaN codes."""
    c = (rng.u64_np(seed, 0, n) & 0xFF).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0
    return c


def _e4m3_caches(seed, b, hkv, d, lens, page):
    """Paged e4m3 caches through a permuted table (padding slots hold the NaN code), and
    the same values as bf16 bit patterns (e4m3 values are exact in bf16)."""
    npg = [-(-n // page) for n in lens]
    total = sum(npg)
    phys = np.argsort(rng.u64_np(seed + 1, 0, total), kind="stable").astype(np.uint32)
    table = np.full((b, -(-max(lens) // page)), 0xFFFFFFFF, dtype=np.uint32)
    kc = np.full((total, hkv, page, d), 0x7F, dtype=np.uint8)
    vc = kc.copy()
    off = 0
    for i, n in enumerate(lens):
        table[i, : npg[i]] = phys[off: off + npg[i]]
        off += npg[i]
        kk = _e4m3_codes(seed + 10 + i, hkv * n * d).reshape(hkv, n, d)
        vv = _e4m3_codes(seed + 20 + i, hkv * n * d).reshape(hkv, n, d)
        for j in range(n):
            kc[table[i, j // page], :, j % page] = kk[:, j]
            vc[table[i, j // page], :, j % page] = vv[:, j]
    as_bf16 = lambda c: bits(oracle.e4m3_to_f64(np.where((c & 0x7F) == 0x7F, 0, c)).astype(np.float32))
    kb, vb = as_bf16(kc), as_bf16(vc)
    kb[(kc & 0x7F) == 0x7F] = rng.BF16_NAN_BITS
    vb[(vc & 0x7F) == 0x7F] = rng.BF16_NAN_BITS
    return kc, vc, kb, vb, table


def test_e4m3_decode_equals_bf16_decode_on_the_same_values():
    b, hq, hkv, d, page, sa = 2, 4, 2, 16, 8, 2
    lens = [13, 30]
    kc, vc, kb, vb, table = _e4m3_caches(60, b, hkv, d, lens, page)
    q = rand_bits(61, (b, hq, sa, d), "q")
    cl = np.array(lens, np.int32)
    o1, l1 = oracle.decode_e4m3(q, kc, vc, table, cl, 0.05, 1.0, 1.0)
    o2, l2 = oracle.decode(q, kb, vb, table, cl, 0.05)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    assert np.isfinite(o1).all()  # the NaN codes of the padding slots never leak


def test_e4m3_scales_are_exact_factors():
    """k_scale = 2 at scale s equals k_scale = 1 at scale 2s; v_scale = 1/2 halves O and
    leaves LSE alone (powers of two scale exactly)."""
    b, hq, hkv, d, page, sa = 2, 4, 1, 16, 8, 3
    lens = [9, 27]
    kc, vc, _, _, table = _e4m3_caches(62, b, hkv, d, lens, page)
    q = rand_bits(63, (b, hq, sa, d), "q")
    cl = np.array(lens, np.int32)
    o1, l1 = oracle.decode_e4m3(q, kc, vc, table, cl, 0.03, 2.0, 1.0)
    o2, l2 = oracle.decode_e4m3(q, kc, vc, table, cl, 0.06, 1.0, 1.0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    o3, l3 = oracle.decode_e4m3(q, kc, vc, table, cl, 0.06, 1.0, 0.5)
    np.testing.assert_array_equal(o3, o2 * 0.5)
    np.testing.assert_array_equal(l3, l2)


# ----------------------------------------------------------------------------- decode extras
# Window and circular flat cache (TKG "gen_mask_tkg" type B), new tokens' K/V given apart
# from the cache (TKG "New-token K/V append"), fused RoPE (TKG "Algorithm", step 0).

def test_decode_ext_without_options_is_decode():
    b, hq, hkv, d, page, sa = 3, 4, 2, 8, 4, 2
    lens = [9, 16, 5]
    q = rand_bits(70, (b, hq, sa, d), "q")
    cl = np.array(lens, np.int32)
    fk, fv, kc, vc, table = _flat_and_paged(71, b, hkv, d, lens, page, True)
    for kk, vv, tt in ((kc, vc, table), (fk, fv, None)):
        o1, l1 = oracle.decode(q, kk, vv, tt, cl, 0.3)
        o2, l2 = oracle.decode_ext(q, kk, vv, tt, cl, 0.3)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("window", [1, 3, 10, 100])
def test_decode_window_equals_last_rows_of_windowed_prefill(window):
    hq, hkv, d, n, sa = 4, 2, 16, 45, 3
    fk, fv, _, _, _ = _flat_and_paged(72, 1, hkv, d, [n], 8, False)
    q = rand_bits(73, (1, hq, sa, d), "q")
    o_dec, l_dec = oracle.decode_ext(q, fk, fv, None, np.array([n], np.int32), 0.2, window=window)
    o_pre, l_pre = oracle.prefill(q, fk[:, :, :n], fv[:, :, :n], 0.2, 1, window)
    np.testing.assert_array_equal(o_dec, o_pre)
    np.testing.assert_array_equal(l_dec, l_pre)


@pytest.mark.parametrize("n", [40, 64, 101, 300])
def test_circular_cache_equals_the_full_cache(n):
    """Logical position j at row j mod cap of a cap-row cache gives the same result as the
    full cache, whenever the window (plus the new tokens) fits in cap."""
    hq, hkv, d, sa, cap, window = 4, 2, 8, 3, 32, 28
    fk, fv, _, _, _ = _flat_and_paged(74, 1, hkv, d, [n], 8, False)
    ck = np.full((1, hkv, cap, d), rng.BF16_NAN_BITS, dtype=np.uint16)
    cv = ck.copy()
    for j in range(max(0, n - cap), n):
        ck[:, :, j % cap] = fk[:, :, j]
        cv[:, :, j % cap] = fv[:, :, j]
    q = rand_bits(75, (1, hq, sa, d), "q")
    cl = np.array([n], np.int32)
    o1, l1 = oracle.decode_ext(q, ck, cv, None, cl, 0.25, window=window, circular=True)
    o2, l2 = oracle.decode_ext(q, fk, fv, None, cl, 0.25, window=window)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    assert np.isfinite(o1).all()


@pytest.mark.parametrize("n", [40, 101, 300])
def test_circular_cache_with_rope_and_new_tokens_equals_the_full_cache(n):
    """The same equivalence with every decode option at once: RoPE of the queries and of
    the new keys (given apart from the cache) must use logical positions, never ring rows,
    so a wrapped ring gives exactly the full cache's result."""
    hq, hkv, d, sa, cap, window = 4, 2, 8, 3, 32, 28
    fk, fv, _, _, _ = _flat_and_paged(79, 1, hkv, d, [n], 8, False)
    kn, vn = fk[:, :, n - sa:n].copy(), fv[:, :, n - sa:n].copy()
    ck = np.full((1, hkv, cap, d), rng.BF16_NAN_BITS, dtype=np.uint16)
    cv = ck.copy()
    for j in range(max(0, n - cap), n - sa):  # the new tokens' rows come from k_new / v_new
        ck[:, :, j % cap] = fk[:, :, j]
        cv[:, :, j % cap] = fv[:, :, j]
    fk2, fv2 = fk.copy(), fv.copy()
    fk2[:, :, n - sa:n] = rng.BF16_NAN_BITS  # likewise in the full cache
    fv2[:, :, n - sa:n] = rng.BF16_NAN_BITS
    q = rand_bits(80, (1, hq, sa, d), "q")
    cl = np.array([n], np.int32)
    f = 10000.0 ** (-np.arange(d // 2) / (d // 2))
    o1, l1 = oracle.decode_ext(q, ck, cv, None, cl, 0.25, window=window, circular=True,
                               k_new=kn, v_new=vn, inv_freq=f)
    o2, l2 = oracle.decode_ext(q, fk2, fv2, None, cl, 0.25, window=window, k_new=kn, v_new=vn,
                               inv_freq=f)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    assert np.isfinite(o1).all()
    # and the rotation matters: without it the result differs
    o3, _ = oracle.decode_ext(q, fk2, fv2, None, cl, 0.25, window=window, k_new=kn, v_new=vn)
    assert not np.array_equal(o1, o3)


def test_new_tokens_given_apart_equal_tokens_in_the_cache():
    b, hq, hkv, d, page, sa = 2, 4, 2, 8, 4, 3
    lens = [7, 18]
    q = rand_bits(76, (b, hq, sa, d), "q")
    cl = np.array(lens, np.int32)
    fk, fv, kc, vc, table = _flat_and_paged(77, b, hkv, d, lens, page, True)
    kn = np.stack([fk[i, :, n - sa:n] for i, n in enumerate(lens)])
    vn = np.stack([fv[i, :, n - sa:n] for i, n in enumerate(lens)])
    kc2, vc2 = kc.copy(), vc.copy()
    for i, n in enumerate(lens):  # the tail slots hold garbage: the new rows come from k_new
        for j in range(n - sa, n):
            kc2[table[i, j // page], :, j % page] = rng.BF16_NAN_BITS
            vc2[table[i, j // page], :, j % page] = rng.BF16_NAN_BITS
    o1, l1 = oracle.decode(q, kc, vc, table, cl, 0.3)
    o2, l2 = oracle.decode_ext(q, kc2, vc2, table, cl, 0.3, k_new=kn, v_new=vn)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_rope_quarter_turn_and_identity_by_hand():
    # d = 2, theta = pi/2: (a, b) -> (-b, a)
    np.testing.assert_allclose(oracle.rope_row([1.0, 0.0], 1.0, [math.pi / 2]), [0.0, 1.0], atol=1e-15)
    np.testing.assert_allclose(oracle.rope_row([3.0, 5.0], 1.0, [math.pi / 2]), [-5.0, 3.0], atol=1e-14)
    # half-split pairing: element i rotates with element i + d/2
    np.testing.assert_allclose(oracle.rope_row([1.0, 2.0, 3.0, 4.0], 2.0, [math.pi / 2, 0.0]),
                               [-1.0, 2.0, -3.0, 4.0], atol=1e-14)
    x = np.arange(1.0, 9.0)
    np.testing.assert_array_equal(oracle.rope_row(x, 0.0, np.linspace(0.1, 1, 4)), x)
    np.testing.assert_array_equal(oracle.rope_row(x, 37.0, np.zeros(4)), x)


def test_rope_matches_complex_rotation_and_keeps_relative_positions():
    d = 16
    f = 10000.0 ** (-np.arange(d // 2) / (d // 2))
    x = f64(rand_bits(78, (d,), "x"))
    y = f64(rand_bits(78, (d,), "y"))
    for pos in (0.0, 1.0, 17.0, 4093.0):
        z = (x[: d // 2] + 1j * x[d // 2:]) * np.exp(1j * pos * f)  # numpy's own complex product
        np.testing.assert_allclose(oracle.rope_row(x, pos, f), np.concatenate([z.real, z.imag]),
                                   rtol=0, atol=1e-12)
    # q(m).k(n) depends on m - n only
    a = oracle.rope_row(x, 30.0, f) @ oracle.rope_row(y, 11.0, f)
    b = oracle.rope_row(x, 519.0, f) @ oracle.rope_row(y, 500.0, f)
    assert abs(a - b) < 1e-10


def _quarter(bits_arr, pos):
    """Exact RoPE with theta = pos * pi/2 on bf16 bits [..., d]: quarter turns of each
    (i, i + d/2) pair, i.e. swaps and sign flips."""
    x = bits_arr.copy()
    h = x.shape[-1] // 2
    a, b = x[..., :h].copy(), x[..., h:].copy()
    for _ in range(int(pos) % 4):
        a, b = b ^ np.uint16(0x8000), a  # (a, b) -> (-b, a)
    x[..., :h], x[..., h:] = a, b
    return x


def test_decode_rope_equals_pre_rotated_inputs():
    """With every inverse frequency pi/2 the rotations are exact quarter turns; decode with
    RoPE (queries at q_pos, new keys at their positions) then equals plain decode on Q and
    new K rotated by hand."""
    b, hq, hkv, d, sa = 2, 4, 2, 8, 3
    lens = [9, 14]
    q = rand_bits(79, (b, hq, sa, d), "q")
    cl = np.array(lens, np.int32)
    fk, fv, _, _, _ = _flat_and_paged(80, b, hkv, d, lens, 8, False)
    kn = np.stack([fk[i, :, n - sa:n] for i, n in enumerate(lens)])
    vn = np.stack([fv[i, :, n - sa:n] for i, n in enumerate(lens)])
    inv = np.full(d // 2, math.pi / 2)
    o1, l1 = oracle.decode_ext(q, fk, fv, None, cl, 0.3, k_new=kn, v_new=vn, inv_freq=inv)
    q2, fk2 = q.copy(), fk.copy()
    for i, n in enumerate(lens):
        for t in range(sa):
            q2[i, :, t] = _quarter(q[i, :, t], n - sa + t)
            fk2[i, :, n - sa + t] = _quarter(kn[i, :, t], n - sa + t)
    o2, l2 = oracle.decode(q2, fk2, fv, None, cl, 0.3)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_decode_rope_rounds_the_rotated_rows_to_bf16():
    """With a general frequency the rotated query and new-key rows are bf16 operands:
    decode with RoPE equals plain decode on rows rotated (numpy's complex product) and
    rounded to bf16 by the input module's own RNE rounding."""
    b, hq, hkv, d, sa = 1, 2, 1, 16, 2
    n = 11
    q = rand_bits(81, (b, hq, sa, d), "q")
    fk, fv, _, _, _ = _flat_and_paged(82, b, hkv, d, [n], 8, False)
    kn, vn = fk[:, :, n - sa:n].copy(), fv[:, :, n - sa:n].copy()
    f = 10000.0 ** (-np.arange(d // 2) / (d // 2))

    def rot(bits_row, pos):
        x = f64(bits_row)
        z = (x[: d // 2] + 1j * x[d // 2:]) * np.exp(1j * pos * f)
        return rng.f32_to_bf16_bits_np(np.concatenate([z.real, z.imag]).astype(np.float32))

    o1, l1 = oracle.decode_ext(q, fk, fv, None, np.array([n], np.int32), 0.25, k_new=kn,
                               v_new=vn, inv_freq=f)
    q2, fk2 = q.copy(), fk.copy()
    for t in range(sa):
        for h in range(hq):
            q2[0, h, t] = rot(q[0, h, t], n - sa + t)
        fk2[0, 0, n - sa + t] = rot(kn[0, 0, t], n - sa + t)
    o2, l2 = oracle.decode(q2, fk2, fv, None, np.array([n], np.int32), 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- packed prefill
# Sequences packed along the sequence axis, each its own problem (CTE "Algorithm - the
# dynamic range_select family": per-row key bounds for sequence packing / prefix length).
VARLEN = [
    # cu_q, cu_k, causal, window
    ([0, 5, 12, 12, 30], [0, 5, 20, 23, 41], 1, 0),    # prefixes, an empty query range
    ([0, 9, 10, 25], [0, 9, 10, 25], 1, 4),            # equal lengths, window 4
    ([0, 7, 16], [0, 3, 30], 1, 0),                    # more queries than keys in sequence 0
    ([0, 6, 14], [0, 11, 19], 0, 0),                   # non-causal
]


def _varlen_inputs(seed, hq, hkv, cu_q, cu_k, d):
    q = rand_bits(seed, (hq, cu_q[-1], d), "q")
    k, v = rand_bits(seed, (hkv, cu_k[-1], d), "k"), rand_bits(seed, (hkv, cu_k[-1], d), "v")
    return q, k, v


def test_varlen_one_sequence_is_plain_prefill():
    q, k, v = _varlen_inputs(90, 4, 2, [0, 21], [0, 33], 8)
    for causal, window in ((0, 0), (1, 0), (1, 6)):
        o1, l1 = oracle.prefill_varlen(q, k, v, [0, 21], [0, 33], 0.3, causal, window)
        o2, l2 = oracle.prefill(q[None], k[None], v[None], 0.3, causal, window)
        np.testing.assert_array_equal(o1, o2[0])
        np.testing.assert_array_equal(l1, l2[0])


@pytest.mark.parametrize("cu_q,cu_k,causal,window", VARLEN)
def test_varlen_zero_q_gives_mean_of_own_sequence(cu_q, cu_k, causal, window):
    """Q = 0: each row averages the allowed V rows of its own sequence, LSE = ln(count);
    the allowed keys of row i of sequence s are counted here from the sequence's own
    bottom-right alignment."""
    d = 4
    q = np.zeros((1, cu_q[-1], d), np.uint16)
    _, k, v = _varlen_inputs(91, 1, 1, cu_q, cu_k, d)
    o, lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, 1.0, causal, window)
    vf = f64(v[0])
    for s in range(len(cu_q) - 1):
        nq, nk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        for i in range(nq):
            qp = i + nk - nq
            hi = min(qp, nk - 1) if causal else nk - 1
            lo = max(0, qp - window + 1) if window else 0
            row = cu_q[s] + i
            if hi < lo:
                assert (o[0, row] == 0).all() and lse[0, row] == -np.inf
                continue
            np.testing.assert_allclose(o[0, row], vf[cu_k[s] + lo: cu_k[s] + hi + 1].mean(0),
                                       atol=1e-12)
            assert abs(lse[0, row] - math.log(hi - lo + 1)) < 1e-12


def test_varlen_other_sequences_do_not_matter():
    cu_q, cu_k = [0, 8, 20, 27], [0, 12, 20, 40]
    q, k, v = _varlen_inputs(92, 2, 1, cu_q, cu_k, 8)
    o1, l1 = oracle.prefill_varlen(q, k, v, cu_q, cu_k, 0.4, 1, 0)
    k2, v2 = k.copy(), v.copy()
    k2[:, cu_k[1]:cu_k[2]] = rand_bits(93, (1, cu_k[2] - cu_k[1], 8), "k")
    v2[:, cu_k[1]:cu_k[2]] = rand_bits(93, (1, cu_k[2] - cu_k[1], 8), "v")
    o2, l2 = oracle.prefill_varlen(q, k2, v2, cu_q, cu_k, 0.4, 1, 0)
    for s in (0, 2):  # sequences 0 and 2 are untouched
        r = slice(cu_q[s], cu_q[s + 1])
        np.testing.assert_array_equal(o1[:, r], o2[:, r])
        np.testing.assert_array_equal(l1[:, r], l2[:, r])


@pytest.mark.parametrize("cu_q,cu_k,causal,window", VARLEN)
def test_varlen_matches_torch_sdpa_with_a_block_mask(cu_q, cu_k, causal, window):
    """PyTorch's scaled_dot_product_attention (float64) with a boolean mask built here from
    the sequence offsets: an independent implementation of the packed problem."""
    import torch
    import torch.nn.functional as F

    hq, hkv, d = 4, 2, 8
    q, k, v = _varlen_inputs(94, hq, hkv, cu_q, cu_k, d)
    o, lse = oracle.prefill_varlen(q, k, v, cu_q, cu_k, 0.35, causal, window)
    SQ, SKV = cu_q[-1], cu_k[-1]
    mask = np.zeros((SQ, SKV), bool)
    for s in range(len(cu_q) - 1):
        nq, nk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        for i in range(nq):
            qp = i + nk - nq
            for j in range(nk):
                ok = (not causal or j <= qp) and (not window or j >= qp - window + 1)
                mask[cu_q[s] + i, cu_k[s] + j] = ok
    t = lambda a: torch.from_numpy(f64(a))
    ref = F.scaled_dot_product_attention(t(q), t(k).repeat_interleave(hq // hkv, 0),
                                         t(v).repeat_interleave(hq // hkv, 0),
                                         attn_mask=torch.from_numpy(mask), scale=0.35).numpy()
    live = mask.any(1)
    np.testing.assert_allclose(o[:, live], ref[:, live], rtol=0, atol=1e-12)
    assert (o[:, ~live] == 0).all()
