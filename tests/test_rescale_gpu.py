"""The lazy alpha correction of both prefill kernels, forced and checked against the oracle.

The online softmax rescales O and l by alpha = exp(m_old - m_new) when a row's max grows
("Flash-Attention: Context (CTE)", "Algorithm - the per-section max update" and
"running-sum update, reciprocal, output accumulate"; minfer "03 - 8n", section 2.1).  The
kernels do it lazily, only when the max has grown by more than 2^8 over the max O was last
scaled to.  The inputs of ``tests/rescale_inputs.py`` make row maxima jump by just under
and just over that threshold, by about 40 and by about 316 log2 units (past fp32's range),
at KV tiles after each row's first.  The CPU tests below check that the inputs really do
that, tile by tile, for the tile width each kernel uses; the GPU tests compare every row of
the kernels' output with the oracle and require bit-identical repeats.

A rescale the kernel skipped would stay correct while the growth is small (any reference
max gives the same O / l); past 2^128 the exponents overflow, so the ~316-unit jumps fail
loudly unless the branch runs.  The branch's other failure modes -- a wrong factor, a
rescale racing the P.V product that is still writing O (the head_dim-256 kernel waits for
it), lanes that need it mixed with lanes that do not, a rescale right after a unit change
-- all show as differences from the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import rescale_inputs as R
from tests.helpers import assert_lse_close, assert_o_close, tensor_of_bits
from workloads import configs as C

SMS = 152  # GB300 streaming multiprocessors

# name, b, hq, hkv, sq, skv, d, causal, window, o dtype, multi-unit
PLAIN = [
    ("d64_causal_multi_unit", 1, 64, 16, 1280, 1280, 64, True, 0, torch.bfloat16, True),
    ("d64_window300_ragged", 1, 8, 2, 1100, 1100, 64, True, 300, torch.float32, False),
    ("d128_causal_multi_unit", 1, 64, 8, 1280, 1280, 128, True, 0, torch.bfloat16, True),
    ("d128_window200_bottom_right", 2, 8, 4, 700, 1000, 128, True, 200, torch.float32, False),
    ("d128_noncausal", 1, 4, 1, 300, 900, 128, False, 0, torch.float32, False),
    ("d256_causal_multi_unit", 1, 40, 8, 1024, 1024, 256, True, 0, torch.bfloat16, True),
    ("d256_window260", 1, 4, 2, 1000, 1000, 256, True, 260, torch.float32, False),
    ("d256_window130_multi_unit", 1, 40, 8, 1024, 1024, 256, True, 130, torch.float32, True),
]

# packed sequences: name, cu_q, cu_k, hq, hkv, d, window, o dtype
PACKED = [
    ("packed_d128_prefixes", [0, 300, 700, 760, 1300], [0, 900, 1500, 2100, 2900], 8, 2, 128, 0,
     torch.float32),
    ("packed_d64_window", [0, 257, 900, 1201], [0, 800, 1443, 2000], 4, 4, 64, 333, torch.bfloat16),
    ("packed_d256_window", [0, 200, 777, 1000], [0, 950, 1527, 2200], 4, 2, 256, 190,
     torch.float32),
]


def _bn(d):
    return 128 if d <= 128 else 64


def _units(b, hq, sq, d):
    nqt = (sq + 127) // 128
    return (nqt + 1) // 2 * b * hq if d <= 128 else nqt * b * hq


def _plain_bounds(sq, skv, causal, window):
    i = np.arange(sq)
    qp = i + skv - sq
    hi = np.minimum(qp, skv - 1) if causal else np.full(sq, skv - 1)
    lo = np.maximum(0, qp - window + 1) if window > 0 else np.zeros(sq, np.int64)
    return lo, hi


def _packed_bounds(cu_q, cu_k, window):
    lo = np.zeros(cu_q[-1], np.int64)
    hi = np.zeros(cu_q[-1], np.int64)
    for s in range(len(cu_q) - 1):
        nq, nk = cu_q[s + 1] - cu_q[s], cu_k[s + 1] - cu_k[s]
        qp = np.arange(nq) + nk - nq
        hi[cu_q[s]:cu_q[s + 1]] = cu_k[s] + np.minimum(qp, nk - 1)
        lo[cu_q[s]:cu_q[s + 1]] = cu_k[s] + (np.maximum(0, qp - window + 1) if window else 0)
    return lo, hi


def _check_growth(q_rows, k, scale, lo, hi, bn, windowed, reaches_700, tile_starts=None):
    g, first = R.tile_max_growth(q_rows, k, scale, lo, hi, bn)
    just_over = (g > R.THRESHOLD_LOG2) & (g < 8.5)
    just_under = (g > 7.5) & (g < R.THRESHOLD_LOG2)
    assert just_over.any(), "no row max grows by just over 2^8 in one tile"
    assert just_under.any(), "no row max grows by just under 2^8 in one tile"
    assert (g >= 30).any(), "no row max grows by 30 log2 units in one tile"
    if reaches_700:
        assert (g > 128).any(), "no row max grows past fp32's exponent range in one tile"
    big = np.nan_to_num(g, nan=-1.0) > R.THRESHOLD_LOG2
    if windowed:
        assert (big & (first == 1)[:, None]).any(), \
            "no row with a single allowed key in its first tile then needs a rescale"
    # a softmax warp (32 consecutive rows of a 128-row query tile) in which, at one KV
    # tile, some lanes need the rescale and others have keys but do not
    starts = tile_starts if tile_starts is not None else np.arange(0, len(lo), 128)
    mixed = False
    for t0 in starts:
        for w0 in range(t0, min(t0 + 128, len(lo)), 32):
            gw = g[w0:w0 + 32]
            need = np.nan_to_num(gw, nan=-1.0) > R.THRESHOLD_LOG2
            calm = np.nan_to_num(gw, nan=99.0) <= R.THRESHOLD_LOG2
            if (need.any(axis=0) & calm.any(axis=0)).any():
                mixed = True
                break
        if mixed:
            break
    assert mixed, "no warp mixes lanes that need the rescale with lanes that do not"


@pytest.mark.parametrize("case", PLAIN, ids=lambda c: c[0])
def test_inputs_force_the_lazy_rescale(case):
    """The inputs grow row maxima past the threshold after the first tile (CPU, fp64)."""
    name, b, hq, hkv, sq, skv, d, causal, window, _, multi = case
    w = C.PrefillWorkload(name, b, hq, hkv, sq, skv, d, causal, window, seed=0x2E5C + d)
    q, k, _ = R.prefill_inputs(w)
    lo, hi = _plain_bounds(sq, skv, causal, window)
    for (bb, h) in ((0, 0), (b - 1, hq - 1)):
        g = oracle.kv_head(h, hq, hkv)
        _check_growth(q[bb, h], k[bb, g], w.scale, lo, hi, _bn(d), window > 0,
                      reaches_700=skv > 700)
    if multi:  # every persistent CTA runs at least two units
        assert _units(b, hq, sq, d) >= 2 * SMS


@pytest.mark.parametrize("case", PACKED, ids=lambda c: c[0])
def test_packed_inputs_force_the_lazy_rescale(case):
    name, cu_q, cu_k, hq, hkv, d, window, _ = case
    cu_q, cu_k = np.array(cu_q, np.int32), np.array(cu_k, np.int32)
    w = C.PrefillWorkload(name, 1, hq, hkv, int(cu_q[-1]), int(cu_k[-1]), d, True, window,
                          seed=0x9A5C + d)
    q, k, _ = R.packed_inputs(w, cu_k)
    lo, hi = _packed_bounds(cu_q, cu_k, window)
    _check_growth(q[0, 0], k[0, 0], w.scale, lo, hi, _bn(d), window > 0,
                  reaches_700=bool((np.diff(cu_k) > 700).any()))


def _run_gpu(q, k, v, causal, window, scale, out, dev, cu=None):
    import flash_attention_forward_attn_gb300 as A

    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    if cu is None:
        o, _ = A.attn_fwd_prefill(q, k, v, causal=causal, window=window, scale=scale, lse=lse,
                                  o_dtype=out)
    else:
        o, _ = A.attn_fwd_prefill_ex(q, k, v, causal=causal, window=window, scale=scale, lse=lse,
                                     o_dtype=out, cu_seqlens_q=cu[0], cu_seqlens_k=cu[1])
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


@pytest.mark.gpu
@pytest.mark.parametrize("case", PLAIN, ids=lambda c: c[0])
def test_forced_rescale_matches_oracle(case, cuda_device):
    name, b, hq, hkv, sq, skv, d, causal, window, out, multi = case
    w = C.PrefillWorkload(name, b, hq, hkv, sq, skv, d, causal, window, seed=0x2E5C + d)
    qb, kb, vb = R.prefill_inputs(w)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    o, lse = _run_gpu(q, k, v, causal, window, w.scale, out, cuda_device)
    o_ref, lse_ref = oracle.prefill(qb, kb, vb, w.scale, causal, window)
    assert_o_close(o.float().cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)
    if multi:  # scheduling-dependent races around the rescale show as run-to-run differences
        for _ in range(20):
            o1, l1 = _run_gpu(q, k, v, causal, window, w.scale, out, cuda_device)
            assert torch.equal(o, o1) and torch.equal(lse, l1)


@pytest.mark.gpu
@pytest.mark.parametrize("case", PACKED, ids=lambda c: c[0])
def test_forced_rescale_packed_matches_oracle(case, cuda_device):
    name, cu_q, cu_k, hq, hkv, d, window, out = case
    cu_q, cu_k = np.array(cu_q, np.int32), np.array(cu_k, np.int32)
    w = C.PrefillWorkload(name, 1, hq, hkv, int(cu_q[-1]), int(cu_k[-1]), d, True, window,
                          seed=0x9A5C + d)
    qb, kb, vb = R.packed_inputs(w, cu_k)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    cu = (torch.from_numpy(cu_q).to(cuda_device), torch.from_numpy(cu_k).to(cuda_device))
    o, lse = _run_gpu(q, k, v, True, window, w.scale, out, cuda_device, cu)
    o_ref, lse_ref = oracle.prefill_varlen(qb[0], kb[0], vb[0], cu_q, cu_k, w.scale, True, window)
    assert_o_close(o[0].float().cpu().numpy(), o_ref, name)
    assert_lse_close(lse[0].cpu().numpy(), lse_ref, name)
    for _ in range(5):
        o1, l1 = _run_gpu(q, k, v, True, window, w.scale, out, cuda_device, cu)
        assert torch.equal(o, o1) and torch.equal(lse, l1)
