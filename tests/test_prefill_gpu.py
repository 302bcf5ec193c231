"""Parity of the CUDA prefill path (through the C ABI) against the fp64 oracle.

Small cases are compared element by element over every row; the full-size workloads
run in the same launch configuration the benchmark times and are compared on sampled
rows that the oracle computes one by one (tile-boundary rows, first/last rows, rows
after Q outliers, seeded random rows).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_lse_close, assert_o_close, bits_of, tensor_of_bits
from workloads import configs as C
from workloads import rng

pytestmark = pytest.mark.gpu


def run_gpu(q, k, v, causal, window, scale, o_dtype=torch.bfloat16):
    import flash_attention_forward_attn_gb300 as A

    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    o, _ = A.attn_fwd_prefill(q, k, v, causal=causal, window=window, scale=scale, lse=lse,
                              o_dtype=o_dtype)
    torch.cuda.synchronize()
    assert A.attn_get_device_error() == 0
    return o, lse


SMALL = [
    # name, b, hq, hkv, sq, skv, d, causal, window, out
    ("tiny_noncausal_d64_f32", 1, 1, 1, 128, 128, 64, False, 0, torch.float32),
    ("causal_ragged_gqa_d128", 1, 4, 2, 300, 300, 128, True, 0, torch.bfloat16),
    ("noncausal_rect_d128", 2, 2, 1, 200, 333, 128, False, 0, torch.bfloat16),
    ("causal_window_d256", 1, 2, 1, 400, 400, 256, True, 100, torch.bfloat16),
    ("causal_window_d128_w1", 1, 2, 2, 260, 260, 128, True, 1, torch.float32),
    ("causal_bottom_right_d64", 1, 3, 1, 100, 260, 64, True, 0, torch.float32),
    ("causal_more_q_than_k_d128", 1, 2, 2, 300, 100, 128, True, 0, torch.float32),
    ("one_query_d128", 2, 4, 4, 1, 77, 128, True, 0, torch.bfloat16),
    ("causal_window_d64_gqa8", 1, 8, 1, 257, 257, 64, True, 64, torch.bfloat16),
    ("noncausal_d256_tail", 1, 1, 1, 129, 65, 256, False, 0, torch.float32),
    ("causal_more_q_than_k_d256", 1, 2, 1, 300, 100, 256, True, 0, torch.float32),
]

# More work units than SMs, so each persistent CTA runs several units: Q reloads between
# units, the epilogue hand-over, odd query-tile counts (a last unit without tile B) and units
# whose query rows precede every key (no KV tile at all).
MULTI_UNIT = [
    # name, b, hq, hkv, sq, skv, d, causal, window, out
    ("multi_unit_causal_d128", 1, 40, 8, 1024, 1024, 128, True, 0, torch.bfloat16),
    ("multi_unit_odd_tiles_d128", 1, 60, 10, 640, 640, 128, True, 0, torch.float32),
    ("multi_unit_empty_units_d64", 1, 64, 16, 700, 300, 64, True, 0, torch.bfloat16),
    ("multi_unit_window_d256", 1, 40, 8, 640, 640, 256, True, 200, torch.bfloat16),
    ("multi_unit_empty_units_d256", 1, 48, 8, 520, 200, 256, True, 0, torch.float32),
]


@pytest.mark.parametrize("case", SMALL + MULTI_UNIT, ids=lambda c: c[0])
def test_prefill_small_all_rows(case, cuda_device):
    name, b, hq, hkv, sq, skv, d, causal, window, out = case
    w = C.PrefillWorkload(name, b, hq, hkv, sq, skv, d, causal, window, seed=0xC0FFEE + len(name))
    qb, kb, vb = C.prefill_inputs_np(w)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    o, lse = run_gpu(q, k, v, causal, window, w.scale, out)
    o_ref, lse_ref = oracle.prefill(qb, kb, vb, w.scale, causal, window)
    assert_o_close(o.float().cpu().numpy(), o_ref, name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, name)
    masked = np.isneginf(lse_ref)
    if masked.any():  # fully masked rows are exactly zero
        assert (o.float().cpu().numpy()[masked] == 0).all()


@pytest.mark.parametrize("scale", [0.0, -0.07])
@pytest.mark.parametrize("d,window", [(128, 0), (64, 40), (256, 90)])
def test_prefill_nonpositive_scale(scale, d, window, cuda_device):
    """scale <= 0 is a valid finite scale: masked keys still get zero weight (scale 0 gives a
    uniform average over the allowed keys, a negative scale favours the least similar)."""
    w = C.PrefillWorkload("nonpos", 1, 2, 1, 200, 260, d, True, window, seed=0x5CA1E + d)
    qb, kb, vb = C.prefill_inputs_np(w)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    o, lse = run_gpu(q, k, v, True, window, scale, torch.float32)
    o_ref, lse_ref = oracle.prefill(qb, kb, vb, scale, True, window)
    assert_o_close(o.cpu().numpy(), o_ref, f"scale={scale}")
    assert_lse_close(lse.cpu().numpy(), lse_ref, f"scale={scale}")


def test_prefill_empty_keys(cuda_device):
    q = torch.randn(1, 2, 50, 128, device=cuda_device).bfloat16()
    k = torch.empty(1, 2, 0, 128, device=cuda_device, dtype=torch.bfloat16)
    o, lse = run_gpu(q, k, k.clone(), True, 0, 0.1, torch.float32)
    assert (o == 0).all() and torch.isneginf(lse).all()


def test_prefill_empty_queries(cuda_device):
    import flash_attention_forward_attn_gb300 as A

    q = torch.empty(1, 2, 0, 64, device=cuda_device, dtype=torch.bfloat16)
    k = torch.randn(1, 2, 10, 64, device=cuda_device).bfloat16()
    o, _ = A.attn_fwd_prefill(q, k, k, causal=True)
    assert o.shape == (1, 2, 0, 64)


def test_prefill_7b_shape_reduced_heads_all_rows(cuda_device):
    w = C.CAUSAL_PREFILL_2K.with_(hq=4, hkv=4)
    qb, kb, vb = C.prefill_inputs_np(w)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    o, lse = run_gpu(q, k, v, True, 0, w.scale)
    o_ref, lse_ref = oracle.prefill(qb, kb, vb, w.scale, True, 0)
    assert_o_close(o.float().cpu().numpy(), o_ref, w.name)
    assert_lse_close(lse.cpu().numpy(), lse_ref, w.name)


def test_masked_keys_do_not_matter_bit_exact(cuda_device):
    """Changing K/V only where the mask forbids (or whole skipped tiles) leaves O bit-identical."""
    w = C.PrefillWorkload("swa_mask", 1, 2, 2, 512, 512, 128, True, 150, seed=77)
    qb, kb, vb = C.prefill_inputs_np(w)
    q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
    o1, l1 = run_gpu(q, k, v, True, 150, w.scale)
    # rows >= 400 attend keys >= 251 only: replace every key and value before 251
    k2, v2 = k.clone(), v.clone()
    k2[:, :, :251] = (3 * torch.randn_like(k2[:, :, :251].float())).bfloat16()
    v2[:, :, :251] = (5 * torch.randn_like(v2[:, :, :251].float())).bfloat16()
    o2, l2 = run_gpu(q, k2, v2, True, 150, w.scale)
    assert torch.equal(o1[:, :, 400:], o2[:, :, 400:])
    assert torch.equal(l1[:, :, 400:], l2[:, :, 400:])


def test_repeat_runs_bit_identical(cuda_device):
    """Scheduling-dependent races show up as run-to-run differences."""
    w = C.PrefillWorkload("rep", 1, 8, 2, 1000, 1000, 128, True, 0, seed=5)
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    o0, l0 = run_gpu(q, k, v, True, 0, w.scale)
    for _ in range(20):
        o1, l1 = run_gpu(q, k, v, True, 0, w.scale)
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


def _sample_rows(w, n_random=24, seed=1):
    rows = {0, w.sq - 1, 127, 128, 129, 255, 256, w.sq // 2, w.sq - 128, w.sq - 129}
    u = rng.uniform_np(rng.stream_seed(seed, "rows"), 0, n_random)
    rows.update(int(x) for x in (u * w.sq).astype(np.int64))
    return sorted(r for r in rows if 0 <= r < w.sq)


def _check_full(w, cuda_device, heads):
    q, k, v = C.prefill_inputs_torch(w, cuda_device)
    o, lse = run_gpu(q, k, v, w.causal, w.window, w.scale)
    rows = _sample_rows(w)
    for (b, h) in heads:
        g = oracle.kv_head(h, w.hq, w.hkv)
        kh = C.prefill_kv_head_np(w, "k", b, g)
        vh = C.prefill_kv_head_np(w, "v", b, g)
        # the generator's rows must be the very values the GPU read
        assert np.array_equal(kh[:4], bits_of(k[b, g, :4]))
        qr = np.stack([C.prefill_q_rows_np(w, b, h, r, 1)[0] for r in rows])
        qp = [oracle.q_pos(r, w.sq, w.skv) for r in rows]
        o_ref, lse_ref = oracle.attention_rows(qr, kh, vh, qp, w.scale, w.causal, w.window)
        assert_o_close(o[b, h, rows].float().cpu().numpy(), o_ref, f"{w.name} b{b} h{h}")
        assert_lse_close(lse[b, h, rows].cpu().numpy(), lse_ref, f"{w.name} b{b} h{h}")
    return o


def test_full_causal_prefill_2k_sampled(cuda_device):
    _check_full(C.CAUSAL_PREFILL_2K, cuda_device, [(0, 0), (0, 31)])


def test_full_gqa_prefill_32k_outliers_sampled(cuda_device):
    w = C.GQA_PREFILL_32K
    _check_full(w, cuda_device, [(0, 0), (0, 5), (0, 31)])


def test_full_swa_prefill_8k_d256_sampled(cuda_device):
    _check_full(C.SWA_PREFILL_8K, cuda_device, [(0, 0), (1, 17), (1, 31)])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_prefill_tile_boundary_residue_sweep(d, causal, cuda_device):
    """Every combination of query and key lengths around the 128-row query tile and the
    64/128-key KV tile (1, one below, at and above each boundary), compared on every row."""
    sqs = (1, 2, 127, 128, 129, 255, 257)
    skvs = (1, 63, 64, 65, 128, 129, 256, 385)
    for sq in sqs:
        for skv in skvs:
            name = f"sweep_d{d}_c{int(causal)}_q{sq}_k{skv}"
            w = C.PrefillWorkload(name, 1, 2, 1, sq, skv, d, causal, 0, seed=0x5EE0 + sq * 1000 + skv)
            qb, kb, vb = C.prefill_inputs_np(w)
            q, k, v = (tensor_of_bits(x, cuda_device) for x in (qb, kb, vb))
            o, lse = run_gpu(q, k, v, causal, 0, w.scale, torch.float32)
            o_ref, lse_ref = oracle.prefill(qb, kb, vb, w.scale, causal, 0)
            assert_o_close(o.cpu().numpy(), o_ref, name)
            assert_lse_close(lse.cpu().numpy(), lse_ref, name)
