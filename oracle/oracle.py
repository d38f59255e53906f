"""numpy front end of the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg are the only callers.  Nothing here is imported
by the product package, and nothing here imports it.

Each function states the definition it evaluates; oracle.c cites the page
passage behind each one.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional, Sequence

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
SUM, MEAN = 0, 1
GEN_UNIFORM, GEN_NORMAL4 = 0, 1
_DT = {"f32": F32, "bf16": BF16}
_POOL = {"sum": SUM, "mean": MEAN}

_lib = None
_p = C.c_void_p


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.oracle_splitmix64.restype = C.c_uint64
        L.oracle_splitmix64.argtypes = [C.c_uint64]
        L.oracle_set_threads.argtypes = [C.c_int]
        L.oracle_max_threads.restype = C.c_int
        L.oracle_table_rows.argtypes = [C.c_int, C.c_uint64, C.c_float, C.c_int32, _p, C.c_int64, _p]
        L.oracle_dedup.restype = C.c_int
        L.oracle_dedup.argtypes = [_p, _p, C.c_int32, C.c_int32, _p, _p, C.c_int32, _p, _p, _p, _p, _p, _p, _p]
        L.oracle_embedding_bag_fwd.restype = C.c_int
        L.oracle_embedding_bag_fwd.argtypes = [_p, C.c_int, C.c_int, C.c_uint64, C.c_float, C.c_int32, _p, _p,
                                               C.c_int32, C.c_int32, _p, _p, C.c_int32, C.c_int, _p, C.c_int64,
                                               _p, C.c_int, C.c_int64, C.c_int64, _p]
        L.oracle_dot_interaction.restype = C.c_int
        L.oracle_dot_interaction.argtypes = [_p, C.c_int, C.c_int32, C.c_int32, C.c_int32, _p, C.c_int64, _p, _p]
        L.oracle_dot_interaction_bwd.restype = C.c_int
        L.oracle_dot_interaction_bwd.argtypes = [_p, _p, C.c_int32, C.c_int32, C.c_int32, _p, C.c_int64, _p, _p]
        L.oracle_bf16_stochastic_round.restype = C.c_int
        L.oracle_bf16_stochastic_round.argtypes = [_p, _p, C.c_int64, C.c_int32, C.c_uint64, _p]
        L.oracle_optimizer_step.restype = C.c_int
        L.oracle_optimizer_step.argtypes = [C.c_int, C.c_double, C.c_double, C.c_double, C.c_double, C.c_int64,
                                            C.c_int32, C.c_int64, _p, _p, _p, _p, _p, C.c_int, _p, _p, _p]
        L.oracle_bag_fm.restype = C.c_int
        L.oracle_bag_fm.argtypes = [_p, C.c_int, C.c_int, C.c_uint64, C.c_float, C.c_int32, _p, _p, C.c_int32,
                                    C.c_int32, _p, _p, C.c_int32, _p, C.c_int64, _p, _p]
        L.oracle_dot_interaction_mode.restype = C.c_int
        L.oracle_dot_interaction_mode.argtypes = [_p, C.c_int, C.c_int32, C.c_int32, C.c_int32, C.c_int, _p, C.c_int64,
                                                  _p, _p]
        L.oracle_dot_interaction_bwd_mode.restype = C.c_int
        L.oracle_dot_interaction_bwd_mode.argtypes = [_p, _p, C.c_int32, C.c_int32, C.c_int32, C.c_int, _p, C.c_int64,
                                                      _p, _p]
        L.oracle_embedding_bag_bwd_update.restype = C.c_int
        L.oracle_embedding_bag_bwd_update.argtypes = [_p, C.c_int64, C.c_int64, _p, _p, C.c_int32, C.c_int32, _p,
                                                      _p, C.c_int32, C.c_int, C.c_float, C.c_int32, _p, C.c_int64,
                                                      _p, C.c_int, C.c_int, C.c_uint64, C.c_float, _p, _p, _p]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def splitmix64(x: int) -> int:
    return int(lib().oracle_splitmix64(C.c_uint64(x & ((1 << 64) - 1))))


class OracleError(RuntimeError):
    pass


def _check(st: int, what: str) -> None:
    if st != 0:
        raise OracleError(f"{what} failed with status {st}")


def table_rows(kind: int, seed: int, scale: float, d: int, rows: Sequence[int]) -> np.ndarray:
    """Generated values of the listed global rows: fp32 (uniform) or bf16 bits (normal4)."""
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, d), dtype=np.float32 if kind == GEN_UNIFORM else np.uint16)
    lib().oracle_table_rows(int(kind), C.c_uint64(seed), C.c_float(scale), int(d), _ptr(rows), rows.size, _ptr(out))
    return out


def dedup(ids, offsets, num_fields, batch, bag_to_table, row_base) -> Dict[str, np.ndarray]:
    """Sorted unique global rows, inverse map, sort permutation and run bounds."""
    ids = _c(ids, np.int64)
    offsets = _c(offsets, np.int64)
    b2t = _c(bag_to_table, np.int32)
    rb = _c(row_base, np.int64)
    n = int(offsets[-1])
    T = rb.size - 1
    uniq = np.empty(max(n, 1), dtype=np.int64)
    nu = np.zeros(1, dtype=np.int64)
    inv = np.empty(max(n, 1), dtype=np.int32)
    spos = np.empty(max(n, 1), dtype=np.int32)
    sbag = np.empty(max(n, 1), dtype=np.int32)
    runs = np.empty(n + 1, dtype=np.int32)
    uoff = np.empty(T + 1, dtype=np.int64)
    st = lib().oracle_dedup(_ptr(ids), _ptr(offsets), int(num_fields), int(batch), _ptr(b2t), _ptr(rb), T,
                            _ptr(uniq), _ptr(nu), _ptr(inv), _ptr(spos), _ptr(sbag), _ptr(runs), _ptr(uoff))
    _check(st, "oracle_dedup")
    k = int(nu[0])
    return {"unique_rows": uniq[:k].copy(), "n_unique": k, "inverse": inv[:n], "sorted_pos": spos[:n],
            "sorted_bag": sbag[:n], "run_offsets": runs[:k + 1].copy(), "unique_offsets": uoff}


def embedding_bag_fwd(ids, offsets, num_fields, batch, bag_to_table, row_base, d, pool="sum",
                      table=None, dtype="f32", gen=None, bag_list=None, out_dtype=None, with_mag=False):
    """Pooled bags.  Returns out[B, F, d] (or [len(bag_list), d]) and optionally the magnitude sums.

    table: host array [total_rows, d] (fp32, or bf16 bits as uint16), or None with
    gen = (kind, seed, scale) to regenerate rows.  bf16 outputs are uint16 bits.
    """
    ids = _c(ids, np.int64)
    offsets = _c(offsets, np.int64)
    b2t = _c(bag_to_table, np.int32)
    rb = _c(row_base, np.int64)
    dt = _DT[dtype]
    odt = _DT[out_dtype or dtype]
    if table is not None:
        table = np.ascontiguousarray(table)
        gk, gs, gsc = 0, 0, 0.0
    else:
        gk, gs, gsc = gen
    F, B = int(num_fields), int(batch)
    npdt = np.float32 if odt == F32 else np.uint16
    if bag_list is None:
        out = np.zeros((B, F, d), dtype=npdt)
        bl, nl = None, 0
        sb, sf = F * d, d
    else:
        bl = _c(bag_list, np.int64)
        nl = bl.size
        out = np.zeros((nl, d), dtype=npdt)
        sb, sf = 0, 0
    mag = np.zeros(out.shape, dtype=np.float64) if with_mag else None
    st = lib().oracle_embedding_bag_fwd(_ptr(table), dt, int(gk), C.c_uint64(gs), C.c_float(gsc), int(d),
                                        _ptr(ids), _ptr(offsets), F, B, _ptr(b2t), _ptr(rb), rb.size - 1,
                                        _POOL[pool], _ptr(bl), nl, _ptr(out), odt, sb, sf, _ptr(mag))
    _check(st, "oracle_embedding_bag_fwd")
    return (out, mag) if with_mag else out


def bag_fm(ids, offsets, num_fields, batch, bag_to_table, row_base, d, table=None, dtype="f32", gen=None,
           bag_list=None, with_mag=False):
    """FM second-order term of each bag: sum over pairs of positions i < j of <v_i, v_j>.

    Returns fm[F * B] (bag-major: bag f * B + b) or fm[len(bag_list)], fp32, and
    optionally the magnitude sums (double)."""
    ids = _c(ids, np.int64)
    offsets = _c(offsets, np.int64)
    b2t = _c(bag_to_table, np.int32)
    rb = _c(row_base, np.int64)
    if table is not None:
        table = np.ascontiguousarray(table)
        gk, gs, gsc = 0, 0, 0.0
    else:
        gk, gs, gsc = gen
    F, B = int(num_fields), int(batch)
    bl = None if bag_list is None else _c(bag_list, np.int64)
    nb = F * B if bl is None else bl.size
    out = np.zeros(nb, dtype=np.float32)
    mag = np.zeros(nb, dtype=np.float64) if with_mag else None
    st = lib().oracle_bag_fm(_ptr(table), _DT[dtype], int(gk), C.c_uint64(gs), C.c_float(gsc), int(d), _ptr(ids),
                             _ptr(offsets), F, B, _ptr(b2t), _ptr(rb), rb.size - 1, _ptr(bl),
                             0 if bl is None else bl.size, _ptr(out), _ptr(mag))
    _check(st, "oracle_bag_fm")
    return (out, mag) if with_mag else out


def dot_interaction(X, n, d, dtype="f32", sample_list=None, with_mag=False):
    """[dense | strict-lower-triangle dots] per sample.  X: [B, n, d] fp32 or bf16 bits."""
    X = np.ascontiguousarray(X)
    B = X.shape[0]
    width = d + n * (n - 1) // 2
    sl = None if sample_list is None else _c(sample_list, np.int64)
    ns = B if sl is None else sl.size
    out = np.zeros((ns, width), dtype=np.float32 if dtype == "f32" else np.uint16)
    mag = np.zeros((ns, width), dtype=np.float64) if with_mag else None
    st = lib().oracle_dot_interaction(_ptr(X), _DT[dtype], B, int(n), int(d), _ptr(sl), 0 if sl is None else sl.size,
                                      _ptr(out), _ptr(mag))
    _check(st, "oracle_dot_interaction")
    return (out, mag) if with_mag else out


def dot_interaction_bwd(dout, X, n, d, sample_list=None, with_mag=False):
    """dX[B, n, d] of the interaction for upstream gradient dout[B, d + n(n-1)/2] (fp32)."""
    dout = _c(dout, np.float32)
    X = _c(X, np.float32)
    B = X.shape[0]
    sl = None if sample_list is None else _c(sample_list, np.int64)
    ns = B if sl is None else sl.size
    dX = np.zeros((ns, n, d), dtype=np.float32)
    mag = np.zeros((ns, n, d), dtype=np.float64) if with_mag else None
    st = lib().oracle_dot_interaction_bwd(_ptr(dout), _ptr(X), B, int(n), int(d), _ptr(sl),
                                          0 if sl is None else sl.size, _ptr(dX), _ptr(mag))
    _check(st, "oracle_dot_interaction_bwd")
    return (dX, mag) if with_mag else dX


INTERACTION_MODES = {"cross": 0, "with_self": 1, "full": 2}


def interaction_width(n, d, mode="cross"):
    m = INTERACTION_MODES[mode]
    return d + n * (n - 1) // 2 if m == 0 else (d + n * (n + 1) // 2 if m == 1 else n * n)


def dot_interaction_mode(X, n, d, mode="cross", dtype="f32", sample_list=None, with_mag=False):
    """The interaction variants: "cross" (i > j, after the dense vector), "with_self"
    (i >= j, after the dense vector) or "full" (the n x n Gram matrix, row-major)."""
    X = np.ascontiguousarray(X)
    B = X.shape[0]
    width = interaction_width(n, d, mode)
    sl = None if sample_list is None else _c(sample_list, np.int64)
    ns = B if sl is None else sl.size
    out = np.zeros((ns, width), dtype=np.float32 if dtype == "f32" else np.uint16)
    mag = np.zeros((ns, width), dtype=np.float64) if with_mag else None
    st = lib().oracle_dot_interaction_mode(_ptr(X), _DT[dtype], B, int(n), int(d), INTERACTION_MODES[mode], _ptr(sl),
                                           0 if sl is None else sl.size, _ptr(out), _ptr(mag))
    _check(st, "oracle_dot_interaction_mode")
    return (out, mag) if with_mag else out


def dot_interaction_bwd_mode(dout, X, n, d, mode="cross", sample_list=None, with_mag=False):
    """dX[B, n, d] of an interaction variant for upstream gradient dout[B, width] (fp32)."""
    dout = _c(dout, np.float32)
    X = _c(X, np.float32)
    B = X.shape[0]
    sl = None if sample_list is None else _c(sample_list, np.int64)
    ns = B if sl is None else sl.size
    dX = np.zeros((ns, n, d), dtype=np.float32)
    mag = np.zeros((ns, n, d), dtype=np.float64) if with_mag else None
    st = lib().oracle_dot_interaction_bwd_mode(_ptr(dout), _ptr(X), B, int(n), int(d), INTERACTION_MODES[mode],
                                               _ptr(sl), 0 if sl is None else sl.size, _ptr(dX), _ptr(mag))
    _check(st, "oracle_dot_interaction_bwd_mode")
    return (dX, mag) if with_mag else dX


OPTIMIZERS = {"sgd": 0, "adagrad": 1, "rowwise_adagrad": 2, "adam": 3}


def optimizer_step(opt, w_old, g, lr, state0=None, state1=None, eps=1e-8, beta1=0.9, beta2=0.999, step=1,
                   dtype="f32", sr_seed=None, rows=None):
    """One optimizer step on rows w_old [n, d] (fp64 values) with exact gradients g [n, d] (fp64).

    Returns (w_new in the table dtype, state0_new, state1_new) with fp32 states:
    Adagrad's sum of squares [n, d] (row-wise: [n]) or Adam's m [n, d]; Adam's v [n, d].
    With sr_seed (bf16 tables) the new rows are stochastically rounded at table rows `rows`."""
    o = OPTIMIZERS[opt]
    w_old = _c(w_old, np.float64)
    g = _c(g, np.float64)
    n, d = w_old.shape
    s0 = None if state0 is None else _c(state0, np.float32)
    s1 = None if state1 is None else _c(state1, np.float32)
    w_new = np.zeros((n, d), dtype=np.float32 if dtype == "f32" else np.uint16)
    s0o = None if s0 is None else np.zeros_like(s0)
    s1o = None if s1 is None else np.zeros_like(s1)
    x = np.zeros((n, d), dtype=np.float64)
    st = lib().oracle_optimizer_step(o, float(lr), float(eps), float(beta1), float(beta2), int(step), int(d), int(n),
                                     _ptr(w_old), _ptr(g), _ptr(s0), _ptr(s1), _ptr(w_new), _DT[dtype], _ptr(s0o),
                                     _ptr(s1o), _ptr(x))
    _check(st, "oracle_optimizer_step")
    if sr_seed is not None:
        assert dtype == "bf16" and rows is not None
        w_new = bf16_stochastic_round(x, rows, sr_seed)
    return w_new, s0o, s1o


def bf16_stochastic_round(x, rows, seed):
    """Stochastically rounded bf16 bits of values x [n, d] (fp64) at table rows `rows` [n]."""
    x = _c(x, np.float64)
    rows = _c(rows, np.int64)
    n, d = x.shape
    out = np.zeros((n, d), dtype=np.uint16)
    _check(lib().oracle_bf16_stochastic_round(_ptr(x), _ptr(rows), n, d, C.c_uint64(seed & (2 ** 64 - 1)), _ptr(out)),
           "oracle_bf16_stochastic_round")
    return out


def embedding_bag_bwd_update(G, ids, offsets, num_fields, batch, bag_to_table, row_base, d, lr, target_rows,
                             pool="sum", table=None, dtype="f32", gen=None):
    """SGD-updated values, fp64 gradient and magnitude sums of the listed global rows.

    G: fp32 gradient of the pooled outputs, shape [B, F, d] (any memory layout).
    """
    G = _c(G, np.float32)
    assert G.shape == (int(batch), int(num_fields), int(d)), G.shape
    ids = _c(ids, np.int64)
    offsets = _c(offsets, np.int64)
    b2t = _c(bag_to_table, np.int32)
    rb = _c(row_base, np.int64)
    tr = _c(target_rows, np.int64)
    F, B = int(num_fields), int(batch)
    sb, sf = F * d, d
    if table is not None:
        table = np.ascontiguousarray(table)
        gk, gs, gsc = 0, 0, 0.0
    else:
        gk, gs, gsc = gen
    new = np.zeros((tr.size, d), dtype=np.float32 if dtype == "f32" else np.uint16)
    grad = np.zeros((tr.size, d), dtype=np.float64)
    mag = np.zeros((tr.size, d), dtype=np.float64)
    st = lib().oracle_embedding_bag_bwd_update(_ptr(G), sb, sf, _ptr(ids), _ptr(offsets), F, B, _ptr(b2t), _ptr(rb),
                                               rb.size - 1, _POOL[pool], C.c_float(lr), int(d), _ptr(tr), tr.size,
                                               _ptr(table), _DT[dtype], int(gk), C.c_uint64(gs), C.c_float(gsc),
                                               _ptr(new), _ptr(grad), _ptr(mag))
    _check(st, "oracle_embedding_bag_bwd_update")
    return new, grad, mag
