"""Parity of packed (variable-length) prefill (attn_fwd_prefill_ex with cu_seqlens, through
the C ABI) against the fp64 oracle ("Flash-Attention: Context (CTE)", "Algorithm - the
dynamic range_select family": per-row key bounds for sequence packing and a dynamic
prefix length).  Each packed sequence is its own problem, its queries at the tail of its
keys."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, tensor_of_bits
from workloads import configs as C
from workloads import rng

pytestmark = pytest.mark.gpu


def packed_lengths(seed, nseq, q_hi, prefix_hi):
    """Seeded query lengths in [0, q_hi] and cached-prefix lengths in [0, prefix_hi]."""
    u = rng.u64_np(seed, 0, 2 * nseq)
    nq = (u[:nseq] % np.uint64(q_hi + 1)).astype(np.int64)
    pre = (u[nseq:] % np.uint64(prefix_hi + 1)).astype(np.int64) if prefix_hi else np.zeros(nseq, np.int64)
    cu_q = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(nq + pre)]).astype(np.int32)
    return cu_q, cu_k


def run_varlen(cu_q, cu_k, hq, hkv, d, causal, window, out, seed, dev, sink=None,
               balance=True):
    import flash_attention_forward_attn_gb300 as A

    w = C.PrefillWorkload("varlen", 1, hq, hkv, int(cu_q[-1]), int(cu_k[-1]), d, causal, window,
                          seed=seed)
    qb, kb, vb = C.prefill_inputs_np(w)
    q, k, v = (tensor_of_bits(x, dev) for x in (qb, kb, vb))
    lse = torch.empty((1, hq, w.sq), dtype=torch.float32, device=dev)
    o, _ = A.attn_fwd_prefill_ex(q, k, v, causal=causal, window=window, scale=w.scale, lse=lse,
                                 o_dtype=out, sink=sink,
                                 cu_seqlens_q=torch.from_numpy(cu_q).to(dev),
                                 cu_seqlens_k=torch.from_numpy(cu_k).to(dev), balance=balance)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return (qb, kb, vb, w), o, lse


CASES = [
    # name, cu_q, cu_k (or a seeded packing: nseq, q_hi, prefix_hi), hq, hkv, d, causal, window, out
    ("two_seqs_mid_tile_d128", [0, 100, 300], [0, 100, 300], 4, 2, 128, True, 0, torch.bfloat16),
    ("prefix_cached_d128", [0, 70, 200, 200, 333], [0, 300, 530, 600, 733], 4, 1, 128, True, 0,
     torch.float32),
    ("more_q_than_k_d64", [0, 150, 260], [0, 40, 300], 4, 4, 64, True, 0, torch.float32),
    ("noncausal_d64", [0, 33, 160, 161], [0, 80, 200, 330], 2, 1, 64, False, 0, torch.bfloat16),
    ("window_d256", [0, 200, 450], [0, 260, 700], 4, 2, 256, True, 64, torch.bfloat16),
    ("many_seqs_d128", (40, 180, 0), None, 8, 2, 128, True, 0, torch.bfloat16),
    ("many_prefixed_d128_w", (30, 150, 400), None, 4, 2, 128, True, 100, torch.float32),
    ("many_seqs_d256", (24, 200, 100), None, 4, 2, 256, True, 0, torch.float32),
    ("many_seqs_d64_multi_unit", (60, 300, 64), None, 40, 8, 64, True, 0, torch.bfloat16),
    # 27 query tiles (the last pair has tile A only) and 560 units, so CTAs run three or four
    # units each: the packed kernel's three-slot Q ring wraps, and the tile-A-only units
    # shift its slot order
    ("d128_ring_wraps_tile_a_only", (50, 128, 60), None, 40, 8, 128, True, 0, torch.bfloat16),
    # a sequence of 600 queries and no keys: the first two units of every head have no KV
    # tile at all (no Q load in the ring, no MMA turns), 128 of them among 256 units, so
    # CTAs run them back to back before units with work
    ("d128_keyless_units", [0, 600, 1024], [0, 0, 424], 64, 16, 128, True, 0, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_varlen_prefill_all_rows(case, cuda_device):
    name, a, b_, hq, hkv, d, causal, window, out = case
    if b_ is None:
        cu_q, cu_k = packed_lengths(0xA11 + len(name), *a)
    else:
        cu_q, cu_k = np.array(a, np.int32), np.array(b_, np.int32)
    (qb, kb, vb, w), o, lse = run_varlen(cu_q, cu_k, hq, hkv, d, causal, window, out,
                                         0x7A0 + len(name), cuda_device)
    o_ref, lse_ref = oracle.prefill_varlen(qb[0], kb[0], vb[0], cu_q, cu_k, w.scale, causal,
                                           window)
    assert_o_close(o[0].float().cpu().numpy(), o_ref, name)
    assert_lse_close(lse[0].cpu().numpy(), lse_ref, name)
    masked = np.isneginf(lse_ref)
    if masked.any():  # rows with no allowed key are exactly zero
        assert (o[0].float().cpu().numpy()[masked] == 0).all()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_varlen_one_sequence_is_bit_identical_to_plain_prefill(d, cuda_device):
    import flash_attention_forward_attn_gb300 as A

    cu = np.array([0, 700], np.int32)
    (qb, kb, vb, w), o1, l1 = run_varlen(cu, cu, 4, 2, d, True, 0, torch.bfloat16, 0x7B0 + d,
                                         cuda_device)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    l2 = torch.empty_like(l1)
    o2, _ = A.attn_fwd_prefill(q, k, v, causal=True, scale=w.scale, lse=l2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d,hq,hkv,packing,causal,window", [
    (128, 8, 2, (40, 300, 200), True, 0),
    (64, 16, 4, (60, 400, 64), True, 0),
    (128, 4, 4, (20, 500, 300), False, 0),  # every tile of a sequence ties
    (256, 4, 2, (24, 260, 100), True, 64),
])
def test_work_order_leaves_results_bit_identical(d, hq, hkv, packing, causal, window,
                                                 cuda_device):
    """The work-order pass only decides which CTA runs a query tile and when; every tile is
    computed the same way, so results are bit-identical with and without it."""
    cu_q, cu_k = packed_lengths(0xB0 + d, *packing)
    _, o1, l1 = run_varlen(cu_q, cu_k, hq, hkv, d, causal, window, torch.bfloat16, 0x7D0 + d,
                           cuda_device, balance=True)
    _, o2, l2 = run_varlen(cu_q, cu_k, hq, hkv, d, causal, window, torch.bfloat16, 0x7D0 + d,
                           cuda_device, balance=False)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_varlen_with_sink(cuda_device):
    cu_q, cu_k = packed_lengths(0xA99, 12, 200, 150)
    sk = C.sink_logits(8)
    (qb, kb, vb, w), o, lse = run_varlen(cu_q, cu_k, 8, 2, 128, True, 0, torch.float32, 0x7C0,
                                         cuda_device, sink=torch.from_numpy(sk).to(cuda_device))
    o_ref, lse_ref = oracle.prefill_varlen(qb[0], kb[0], vb[0], cu_q, cu_k, w.scale, True, 0,
                                           sink=sk)
    assert_o_close(o[0].cpu().numpy(), o_ref, "varlen sink")
    assert_lse_close(lse[0].cpu().numpy(), lse_ref, "varlen sink")


def test_packed_benchmark_workload_sampled(cuda_device):
    """The packed workload the benchmark times, in the same launch; sampled sequences and
    heads are checked row by row against the oracle over that sequence's own keys."""
    import flash_attention_forward_attn_gb300 as A

    pw = C.PACKED_PREFILL
    w = pw.as_prefill()
    cu_q, cu_k = pw.offsets()
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    lse = torch.empty((1, w.hq, w.sq), dtype=torch.float32, device=cuda_device)
    o, _ = A.attn_fwd_prefill_ex(q, k, v, causal=True, scale=pw.scale, lse=lse,
                                 cu_seqlens_q=torch.from_numpy(cu_q).to(cuda_device),
                                 cu_seqlens_k=torch.from_numpy(cu_k).to(cuda_device))
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    for s in (0, 7, pw.nseq - 1):
        q0, nq, k0, nk = int(cu_q[s]), int(cu_q[s + 1] - cu_q[s]), int(cu_k[s]), int(cu_k[s + 1] - cu_k[s])
        rows = sorted({0, 1, nq // 2, nq - 1, min(nq - 1, 127), min(nq - 1, 128)})
        for h in (0, 21):
            g = oracle.kv_head(h, pw.hq, pw.hkv)
            kh = C.prefill_kv_head_np(w, "k", 0, g)[k0:k0 + nk]
            vh = C.prefill_kv_head_np(w, "v", 0, g)[k0:k0 + nk]
            qh = np.stack([C.prefill_q_rows_np(w, 0, h, q0 + r, 1)[0] for r in rows])
            qp = [oracle.q_pos(r, nq, nk) for r in rows]
            o_ref, lse_ref = oracle.attention_rows(qh, kh, vh, qp, pw.scale, True, 0)
            got = o[0, h, [q0 + r for r in rows]].float().cpu().numpy()
            assert_o_close(got, o_ref, f"packed s{s} h{h}")
            assert_lse_close(lse[0, h, [q0 + r for r in rows]].cpu().numpy(), lse_ref,
                             f"packed s{s} h{h}")


def _tile_cost(cu_q, cu_k, sq, skv, causal, window, bm, bn, qt):
    """KV tiles of packed query tile qt (rows [qt*bm, qt*bm + bm)), from the definition of
    the allowed keys: each row's own sequence, its queries at the tail of its keys."""
    q0 = qt * bm
    rows = min(bm, sq - q0)
    if rows <= 0:
        return 0

    def bounds(i):
        s = int(np.searchsorted(cu_q, i, side="right") - 1)
        nq, k0, nk = int(cu_q[s + 1] - cu_q[s]), int(cu_k[s]), int(cu_k[s + 1] - cu_k[s])
        qpos = (i - int(cu_q[s])) + nk - nq
        hi = k0 + (min(qpos, nk - 1) if causal else nk - 1)
        lo = k0 + (max(0, qpos - window + 1) if window > 0 else 0)
        return s, lo, hi

    s0, lo0, _ = bounds(q0)
    s1, _, hi1 = bounds(q0 + rows - 1)
    k_end, k_begin = min(skv, hi1 + 1), max(0, lo0)
    if s0 != s1:
        k_end = max(k_end, min(skv, int(cu_k[s1])))
    return 0 if k_end <= k_begin else -(-k_end // bn) - k_begin // bn


@pytest.mark.parametrize("d,packing,causal,window", [
    (128, (40, 300, 200), True, 0),
    (128, (25, 500, 0), False, 0),   # ties: every tile of a sequence has the same count
    (256, (24, 260, 100), True, 64),
])
def test_work_order_is_the_units_sorted_by_kv_tiles(d, packing, causal, window, cuda_device):
    """The work-order pass writes a permutation of the query units.  Head_dim 256 (single
    128-row tiles, a static schedule): KV-tile counts non-increasing, ties in index order.
    Head_dim <= 128 (pairs of tiles, handed out at run time): grouped by the sequence of the
    unit's first row, counts non-increasing within a sequence; the counter after the order
    was reset by the pass and drawn past the last unit by the kernel."""
    import ctypes

    import flash_attention_forward_attn_gb300 as A

    cu_q, cu_k = packed_lengths(0xC0 + d, *packing)
    w = C.PrefillWorkload("order", 1, 4, 2, int(cu_q[-1]), int(cu_k[-1]), d, causal, window,
                          seed=0x7E0)
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=cuda_device)
    nbytes = A.attn_prefill_workspace_bytes(w.sq)
    ws = torch.full((nbytes // 4,), -1, dtype=torch.int32, device=cuda_device)
    dq, dk = (torch.from_numpy(x).to(cuda_device) for x in (cu_q, cu_k))
    opts = A.AttnOpts(cu_seqlens_q=dq.data_ptr(), cu_seqlens_k=dk.data_ptr(), nseq=len(cu_q) - 1,
                      prefill_workspace=ws.data_ptr(), prefill_workspace_bytes=nbytes)
    lib = A.load_library()
    st = lib.attn_fwd_prefill_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, 1,
                                 4, 2, w.sq, w.skv, d, w.scale, int(causal), window, 0,
                                 ctypes.byref(opts), None)
    torch.cuda.synchronize()
    assert st == 0 and A.attn_get_device_error() == 0
    nqt = -(-w.sq // 128)
    per, bn = (2, 128) if d <= 128 else (1, 64)
    nu = -(-nqt // per)
    cost = [sum(_tile_cost(cu_q, cu_k, w.sq, w.skv, causal, window, 128, bn, per * u + x)
                for x in range(per)) for u in range(nu)]
    order = ws[:nu].cpu().numpy().tolist()
    assert sorted(order) == list(range(nu))
    if per == 2:
        seq = [int(np.searchsorted(cu_q, min(u * per * 128, w.sq - 1), side="right") - 1)
               for u in range(nu)]
        keys = [(seq[u], -cost[u], u) for u in order]
        units = nu * 4  # query-tile pairs x heads
        assert int(ws[nu].item()) >= units  # every unit was drawn, then one failed draw per CTA
    else:
        keys = [(-cost[u], u) for u in order]
    assert keys == sorted(keys)
