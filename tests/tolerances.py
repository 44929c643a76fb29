"""Parity bars shared by the GPU tests.

bf16 outputs: |gpu - oracle| <= ATOL + RTOL * |oracle| element-wise; lse: absolute
LSE_ATOL.  The bar comes from the arithmetic: inputs are exact in both, the GPU
rounds the probabilities to bf16 (relative 2^-9) before the P.V product,
accumulates in fp32, and rounds the output to bf16 (relative 2^-9 ~ 2e-3), so a
1 % relative plus 2e-3 absolute bound holds with margin; lse is accumulated in
fp32 over at most ~1e5 terms, far inside 1e-3.
"""
import numpy as np
import torch

ATOL, RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-3


def check_out(gpu_out: torch.Tensor, ref: np.ndarray, mask=None, what="out", v_mag=1.0):
    """v_mag: how much larger than the N(0,1) data the values V are (a number, or an array
    that broadcasts against out).  The output is linear in V, so V multiplied by c
    multiplies the output and every rounding error in it by c: the absolute part of the
    bar scales with it, the relative part stays."""
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    vm = np.broadcast_to(np.asarray(v_mag, dtype=np.float64), ref.shape)
    if mask is not None:
        g, ref, vm = g[mask], ref[mask], vm[mask]
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - ref)
    bound = ATOL * vm + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                           f"max err {err.max():.3e}, worst excess {(err - bound).max():.3e}")


def check_lse(gpu_lse: torch.Tensor, ref: np.ndarray, mask=None, what="lse"):
    g = gpu_lse.detach().double().cpu().numpy()
    if mask is not None:
        g, ref = g[mask], ref[mask]
    both_inf = np.isneginf(g) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(g - ref))
    assert np.all(np.isfinite(err)), f"{what}: inf/nan mismatch"
    assert err.max(initial=0.0) <= LSE_ATOL, f"{what}: max err {err.max():.3e}"
