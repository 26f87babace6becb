"""Shared helpers for the GPU parity tests (test infrastructure)."""
import numpy as np
import torch

# Tolerances stated for the method: fp32 GEMV |y - y_ref| <= 1e-5 * mag,
# bf16 tensor-core prefill 8e-3 * mag, router weights 1e-6 relative, router
# indices exact.  mag = |rs[o]| * sum_i |q[o,i] * xs[i]| (Q2: the dequantised
# weight in place of rs*q).
TOL_GEMV = 1e-5
TOL_GEMM = 8e-3
TOL_ROUTER_W = 1e-6


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()


def assert_within(y, y_ref, mag, tol, what, floor=0.0):
    """Element-wise |y - y_ref| <= tol * mag (+ floor); reports the worst ratio."""
    y = np.asarray(y, np.float64)
    err = np.abs(y - y_ref)
    bound = tol * mag + floor
    bad = err > bound
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outside tolerance; "
                           f"worst err/bound = {ratio:.3g} at {np.unravel_index(np.argmax(err / np.maximum(bound, 1e-300)), err.shape)}")
    return ratio


def d16(d_bits: np.ndarray) -> torch.Tensor:
    """f16 bit patterns (uint16 numpy) as a CUDA int16 tensor for the binding."""
    return torch.from_numpy(np.ascontiguousarray(d_bits).view(np.int16)).cuda()


def moe_bound(m, sel, w, parts):
    """Composite bound: the GEMV bound on each stage, propagated through
    silu(g)*u and the weighted down projection, times 4."""
    g, u, act = parts["g"], parts["u"], parts["act"]
    x = np.abs(m.x.astype(np.float64))
    tol = TOL_GEMV * parts["mag"]
    for s, e in enumerate(sel):
        mag_g = np.abs(m.grs[e].astype(np.float64)) * (np.abs(m.gq[e].astype(np.float64)) @ x)
        mag_u = np.abs(m.urs[e].astype(np.float64)) * (np.abs(m.uq[e].astype(np.float64)) @ x)
        sig = 1.0 / (1.0 + np.exp(-g[s]))
        dsilu = np.abs(sig * (1.0 + g[s] * (1.0 - sig)))
        dact = (dsilu * np.abs(u[s]) * TOL_GEMV * mag_g + np.abs(g[s] * sig) * TOL_GEMV * mag_u
                + 1e-6 * np.abs(act[s]))
        tol = tol + abs(w[s]) * np.abs(m.drs[e].astype(np.float64)) * (np.abs(m.dq[e].astype(np.float64)) @ dact)
    return 4.0 * tol
