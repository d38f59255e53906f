"""Tolerances used by the GPU-vs-oracle parity tests.

fp32 outputs (the path's stated tolerance): |gpu - ref| <= atol + rtol |ref| with
rtol = 1e-5, atol = 1e-6.  Every fp32 output of the path is a sum, and a sum
whose terms cancel has no relative accuracy in any summation order, so the
bound adds the standard a-priori forward-error term of recursive summation,
gamma_k * sum|terms| with gamma_k = k u / (1 - k u), u = 2^-24 and k the
longest chain of dependent fp32 additions the kernel performs for that output
(its reduction depth).  The oracle reports sum|terms| (the "magnitude") next
to every value.  For outputs whose terms do not cancel the extra term is below
the stated one, and the exact-arithmetic tests (dyadic inputs, where every
sum is exact) compare bit for bit, so a dropped or doubled term cannot hide in
the tolerance.

bf16 outputs: |gpu - ref| <= rtol |ref| + atol + gamma_k sum|terms| with
rtol = 1e-2 (the stated bf16 tolerance), the fp32 accumulation term as above, and atol = 1e-5
for pooled bf16 values (atol 0 for interaction outputs).

`mrel` adds mrel * sum|terms| to the bound.  It is used where a sum's inputs
are themselves rounded results that may differ by the pooled tolerance: a
bf16 pair dot computed from pooled vectors that each carry up to one bf16
rounding differs by at most about 2 * 2^-8 * sum_c |x_ic x_jc|, so those
checks take the magnitude-aware bound 1e-2 * <|x_i|, |x_j|> next to the
relative one.
"""
import numpy as np

U = 2.0 ** -24


def gamma(k: float) -> float:
    ku = k * U
    return ku / (1.0 - ku)


def f32_close(got, ref, mag=None, depth=0, rtol=1e-5, atol=1e-6, what="", mrel=0.0):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = atol + rtol * np.abs(ref)
    if mag is not None and (depth or mrel):
        tol = tol + (gamma(depth) + mrel) * np.asarray(mag, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argmax(np.where(bad, err - tol, -np.inf))
        idx = np.unravel_index(i, got.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.size} values outside tolerance; worst at {idx}: "
            f"gpu={got[idx]!r} ref={ref[idx]!r} err={err[idx]:.3e} tol={tol[idx]:.3e}")


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        b = b.view(np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_close(got_bits, ref_bits, mag=None, depth=0, rtol=1e-2, atol=0.0, what="", mrel=0.0):
    got = bf16_to_f64(got_bits)
    ref = bf16_to_f64(ref_bits)
    tol = atol + rtol * np.abs(ref)
    if mag is not None and (depth or mrel):
        tol = tol + (gamma(depth) + mrel) * np.asarray(mag, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argmax(np.where(bad, err - tol, -np.inf))
        idx = np.unravel_index(i, got.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.size} values outside tolerance; worst at {idx}: "
            f"gpu={got[idx]!r} ref={ref[idx]!r} err={err[idx]:.3e} tol={tol[idx]:.3e}")
