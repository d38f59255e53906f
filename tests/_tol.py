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

`depth` may be a scalar or an array broadcast against the values (each output's
own reduction depth, e.g. its bag's length).  Every check also counts the
values that pass only through the a-priori term (outside atol + rtol |ref|
but inside the full bound) and fails if their share exceeds `max_gamma_share`
(default 1%): the summation term is there for the few outputs whose terms
cancel, not to widen the stated tolerance for all of them.  The last check's
counts are kept in `last` for tests that report them.

`mrel` adds mrel * sum|terms| to the bound.  It is used where a sum's inputs
are themselves rounded results that may differ by the pooled tolerance: a
bf16 pair dot computed from pooled vectors that each carry up to one bf16
rounding differs by at most about 2 * 2^-8 * sum_c |x_ic x_jc|, so those
checks take the magnitude-aware bound 1e-2 * <|x_i|, |x_j|> next to the
relative one.
"""
import numpy as np

U = 2.0 ** -24


def gamma(k):
    ku = np.asarray(k, dtype=np.float64) * U
    return ku / (1.0 - ku)


last = {}


def _check(got, ref, mag, depth, rtol, atol, what, mrel, max_gamma_share):
    base = atol + rtol * np.abs(ref)
    tol = base
    if mag is not None and (np.any(np.asarray(depth) != 0) or mrel):
        tol = tol + (gamma(depth) + mrel) * np.asarray(mag, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argmax(np.where(bad, err - tol, -np.inf))
        idx = np.unravel_index(i, got.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.size} values outside tolerance; worst at {idx}: "
            f"gpu={got[idx]!r} ref={ref[idx]!r} err={err[idx]:.3e} tol={tol[idx]:.3e}")
    via_gamma = int(np.count_nonzero(err > base))
    last.clear()
    last.update(what=what, n=int(got.size), via_gamma=via_gamma)
    if got.size and via_gamma > max_gamma_share * got.size:
        raise AssertionError(
            f"{what}: {via_gamma} of {got.size} values pass only through the summation-error term "
            f"(more than {max_gamma_share:.2%})")


def f32_close(got, ref, mag=None, depth=0, rtol=1e-5, atol=1e-6, what="", mrel=0.0, max_gamma_share=0.01):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    _check(got, ref, mag, depth, rtol, atol, what, mrel, max_gamma_share)


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        b = b.view(np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_close(got_bits, ref_bits, mag=None, depth=0, rtol=1e-2, atol=0.0, what="", mrel=0.0,
               max_gamma_share=0.01):
    got = bf16_to_f64(got_bits)
    ref = bf16_to_f64(ref_bits)
    _check(got, ref, mag, depth, rtol, atol, what, mrel, max_gamma_share)


# Reduction depth of the row-update kernels for a run of L occurrences: runs
# of at most 128 are summed by one warp (L terms, any order: depth L); longer
# runs are cut into pieces of 128 summed in order; a run of at most 32 pieces
# is finished by one warp summing its partials in order (depth 128 + pieces);
# a longer one by 8 warps each summing ceil(pieces / 8) consecutive partials
# in order, joined by a pairwise tree (3 levels).
SHORT_RUN, PIECE, COMBINE_WARPS, WARP_PIECES = 128, 128, 8, 32


def bwd_depth(run_len):
    L = np.asarray(run_len, dtype=np.int64)
    pieces = -(-L // PIECE)
    cta_depth = PIECE + (-(-pieces // COMBINE_WARPS)) + int(np.log2(COMBINE_WARPS))
    return np.where(L <= SHORT_RUN, L, np.where(pieces <= WARP_PIECES, PIECE + pieces, cta_depth))


def pool_depth(offsets, num_fields, batch):
    """Per-output reduction depth of pooled rows laid out [B, F, d]: a bag of L
    rows is a sum of L terms (depth L in any order; a mean's division is one
    more rounding, still within L + 1 >= 1)."""
    lens = np.diff(np.asarray(offsets, dtype=np.int64)).reshape(num_fields, batch).T
    return (lens + 1)[:, :, None]


def fm_depth(lens, d):
    """Depth of the FM term 1/2 (|sum v|^2 - sum |v|^2) evaluated in fp32, in
    units of u times (2 sum_{i<j} |v_i . v_j| + sum |v|^2): the row sum (depth L)
    enters |sum v|^2 twice, the square norm is a d-term dot product, sum |v|^2
    is a chain of at most 4L + 5 fused terms in any of the gathers (halved by
    the 1/2), and the final subtraction is one rounding:
    L + d/2 + 2L + 3 + 1."""
    L = np.asarray(lens, dtype=np.int64)
    return 3 * L + d // 2 + 4
