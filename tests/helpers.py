"""Shared test helpers: bit views between torch and numpy, the parity tolerance."""
import numpy as np

# Parity bar for bf16 inputs with fp32 accumulation: |dO| <= 1e-2 + 1e-2 |O_ref|, |dLSE| <= 1e-3.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 1e-3


def bits_of(t):
    """bf16 torch tensor (any device) -> numpy uint16 bit patterns."""
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def tensor_of_bits(bits, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def assert_o_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = O_ATOL + O_RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs out of tolerance; "
                           f"max |dO| = {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    neg = np.isneginf(ref)
    assert (np.isneginf(got) == neg).all(), f"{what}: fully masked rows differ"
    if (~neg).any():
        err = np.abs(got[~neg] - ref[~neg])
        assert err.max() <= LSE_ATOL, f"{what}: max |dLSE| = {err.max():.3e}"
