"""Prefill inputs whose row maxima jump by chosen amounts at chosen key positions.

The prefill kernels correct O and l lazily: a row's accumulators are rescaled only when
its running max grows by more than 2^8 (in log2 units of the scaled scores) over the max
they were last scaled to ("Flash-Attention: Context (CTE)", "Algorithm - the per-section
max update" and "running-sum update, reciprocal, output accumulate"; minfer "03 - 8n",
section 2.1, "Online softmax").  Seeded N(0,1) inputs almost never grow a row max that
much after its first KV tile, so these inputs build the growth in:

* Head dim 0 of every key holds a staircase B(p) of the key's position p (within its
  sequence when sequences are packed): B steps up at the positions of ``STEPS``.
* Head dim 0 of every value holds 1 + the number of steps passed, so O[:, 0] weighs the
  staircase's treads against each other and any error in a rescale factor shows there.
* Query rows by index mod 4:
    0  ordinary seeded row: its jumps are q[0] * dB, random in size and sign;
    1  A_lo * e_0: every 16-unit step raises its score by just under 8 log2 units;
    2  A_hi * e_0: just over 8 log2 units;
    3  head dim 0 set to 2, the rest seeded: large jumps with noise on top.
  Rows 1 and 2 alternate inside every warp of the softmax, so each rescale meets lanes
  that need it and lanes that do not.

The steps at 512 and 700 (80 and 640 units) lift the max by about 40 and 316 log2 units
for rows of kind 1: beyond fp32's range, so a rescale that is skipped shows as inf/NaN.

Everything is built from bf16 bit patterns with numpy; nothing here computes attention.
"""
from __future__ import annotations

import math

import numpy as np

from workloads import configs as C
from workloads import rng

# (position within the sequence, increase of B there)
STEPS = ((64, 16.0), (128, 16.0), (320, 16.0), (512, 80.0), (700, 640.0))
THRESHOLD_LOG2 = 8.0  # the kernels' lazy-rescale threshold
LOG2E = 1.4426950408889634


def _bf16(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float32)
    return rng.f32_to_bf16_bits_np(a.reshape(-1)).reshape(a.shape)


def _f32(bits) -> np.ndarray:
    return rng.bf16_bits_to_f32_np(bits)


def staircase(p: np.ndarray) -> np.ndarray:
    """B(p) and the number of steps passed at positions p (int array)."""
    b = np.zeros(p.shape, dtype=np.float64)
    n = np.zeros(p.shape, dtype=np.int64)
    for pos, inc in STEPS:
        b += np.where(p >= pos, inc, 0.0)
        n += (p >= pos).astype(np.int64)
    return b, n


def row_amplitudes(d: int) -> tuple[float, float]:
    """bf16 values A_lo, A_hi whose 16-unit steps are just below / above 2^8 in log2 units."""
    c16 = 16.0 / math.sqrt(d) * LOG2E
    a_lo, a_hi = (float(x) for x in _f32(_bf16([7.9 / c16, 8.1 / c16])))
    assert 7.8 < a_lo * c16 < THRESHOLD_LOG2 < a_hi * c16 < 8.2, (a_lo * c16, a_hi * c16)
    return a_lo, a_hi


def shape_q(qb: np.ndarray, d: int) -> np.ndarray:
    """Rows of kind 1, 2, 3 (index mod 4 along the second-to-last axis) as described above."""
    q = qb.copy()
    a_lo, a_hi = row_amplitudes(d)
    kind = np.arange(q.shape[-2]) % 4
    q[..., kind == 1, :] = 0
    q[..., kind == 1, 0] = _bf16(a_lo)
    q[..., kind == 2, :] = 0
    q[..., kind == 2, 0] = _bf16(a_hi)
    q[..., kind == 3, 0] = _bf16(2.0)
    return q


def shape_kv(kb: np.ndarray, vb: np.ndarray, pos: np.ndarray):
    """Head dim 0 of K and V from the staircase at key positions pos (last-but-one axis)."""
    k, v = kb.copy(), vb.copy()
    b, n = staircase(pos)
    k[..., 0] = _bf16(b)
    v[..., 0] = _bf16(1.0 + n)
    return k, v


def prefill_inputs(w: C.PrefillWorkload):
    """(q, k, v) bf16 bits [b, h, s, d] of a plain (one sequence per batch) prefill."""
    qb, kb, vb = C.prefill_inputs_np(w)
    k, v = shape_kv(kb, vb, np.arange(w.skv))
    return shape_q(qb, w.d), k, v


def packed_inputs(w: C.PrefillWorkload, cu_k: np.ndarray):
    """(q, k, v) of a packed b = 1 prefill: the staircase restarts with every sequence."""
    qb, kb, vb = C.prefill_inputs_np(w)
    j = np.arange(w.skv)
    seq = np.searchsorted(cu_k, j, side="right") - 1
    k, v = shape_kv(kb, vb, j - cu_k[seq])
    return shape_q(qb, w.d), k, v


def tile_max_growth(q_rows, k, scale, key_lo, key_hi, bn):
    """For rows with allowed keys [key_lo[r], key_hi[r]], the growth of the running row max
    (log2 units of the scaled scores, fp64 from the bf16 values) at each BN-key tile after
    the row's first non-empty one, and the number of allowed keys in that first tile.

    Returns (growth [rows, tiles] with NaN where undefined, first_count [rows])."""
    s = (_f32(q_rows).astype(np.float64) @ _f32(k).astype(np.float64).T) * scale * LOG2E
    n, skv = s.shape
    j = np.arange(skv)
    ok = (j[None, :] >= key_lo[:, None]) & (j[None, :] <= key_hi[:, None])
    s = np.where(ok, s, -np.inf)
    nt = (skv + bn - 1) // bn
    pad = np.full((n, nt * bn), -np.inf)
    pad[:, :skv] = s
    tmax = pad.reshape(n, nt, bn).max(axis=2)
    counts = np.pad(ok, ((0, 0), (0, nt * bn - skv))).reshape(n, nt, bn).sum(axis=2)
    run = np.maximum.accumulate(tmax, axis=1)
    growth = np.full((n, nt), np.nan)
    first = np.full(n, 0, dtype=np.int64)
    for r in range(n):
        nz = np.nonzero(counts[r])[0]
        if nz.size == 0:
            continue
        t0 = nz[0]
        first[r] = counts[r, t0]
        growth[r, t0 + 1:] = run[r, t0 + 1:] - run[r, t0:-1]
        growth[r, counts[r] == 0] = np.nan
    return growth, first
