"""Thin Python binding of libctr (the C-ABI declared in include/ctr.h).

Every function here has the name of the C call it wraps and only marshals
arguments: torch tensors become device pointers, the current CUDA stream is
passed along, and a negative ctr_status becomes a CtrError.  All computation
happens in libctr's CUDA kernels; there is no CPU fallback.  If the library
cannot be built or loaded the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

F32, BF16 = 0, 1
POOL_SUM, POOL_MEAN = 0, 1
DTYPES = {torch.float32: F32, torch.bfloat16: BF16}
# status codes (ctr_status in include/ctr.h)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE = 0, -1, -2, -3
ERR_INDEX_OUT_OF_RANGE, ERR_CUDA, ERR_TIMEOUT, ERR_NOT_IMPLEMENTED, ERR_BAD_OFFSETS = -4, -5, -6, -7, -8

_lock = threading.Lock()
_lib = None
_p = C.c_void_p
_i32, _i64, _u64, _f32, _sz = C.c_int32, C.c_int64, C.c_uint64, C.c_float, C.c_size_t

# name -> (restype, argtypes), mirroring include/ctr.h
_SIGS = {
    "ctr_status_string": (C.c_char_p, [C.c_int]),
    "ctr_version": (C.c_int, []),
    "ctr_set_timing_events": (C.c_int, [C.c_int, _p, _p]),
    "ctr_launch_count": (C.c_uint64, []),
    "ctr_set_tma_gather": (C.c_int, [C.c_int]),
    "ctr_set_tile_slices": (C.c_int, [C.c_int]),
    "ctr_set_wait_limit_ns": (C.c_uint64, [C.c_uint64]),
    "ctr_status_reset": (C.c_int, [_p, _p]),
    "ctr_check_status": (C.c_int, [_p, _p]),
    "ctr_fill_table": (C.c_int, [_p, C.c_int, _i64, _i32, _i64, C.c_int, _u64, _f32, _p]),
    "ctr_dedup_workspace_size": (_sz, [_i64, _i32, _i32, _i64]),
    "ctr_dedup": (C.c_int, [_p, _p, _i32, _i32, _p, _p, _i32, _i64, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "ctr_dedup_phases": (C.c_int, [_p, _p, _i32, _i32, _p, _p, _i32, _i64, _p, _p, _p, _p, _p, _p, _p, _i32, _p, _sz,
                                   _p]),
    "ctr_gather_rows": (C.c_int, [_p, C.c_int, _i32, _i64, _p, _p, _i64, _p, _p, _sz, _p]),
    "ctr_embedding_bag_workspace_size": (_sz, []),
    "ctr_embedding_bag_fwd": (C.c_int, [_p, C.c_int, _i32, _i64, _p, C.c_int, _i64, _p, _i32, _i32, _p, _p, _i32, C.c_int,
                                        _p, C.c_int, _i64, _i64, _p, _sz, _p]),
    "ctr_embedding_bag_fwd_fm": (C.c_int, [_p, C.c_int, _i32, _i64, _p, C.c_int, _i64, _p, _i32, _i32, _p, _p, _i32,
                                           C.c_int, _p, C.c_int, _i64, _i64, _p, _p, _sz, _p]),
    "ctr_interaction_workspace_size": (_sz, []),
    "ctr_dot_interaction": (C.c_int, [_p, C.c_int, _i32, _i32, _i32, _p, _p, _sz, _p]),
    "ctr_dot_interaction_bwd": (C.c_int, [_p, _p, _i32, _i32, _i32, _p, _p, _sz, _p]),
    "ctr_bwd_update_workspace_size": (_sz, [_i64, _i32]),
    "ctr_embedding_bag_bwd_update": (C.c_int, [_p, _i64, _i64, _p, _i32, _i32, C.c_int, _p, _p, _p, _p, _i64, _f32,
                                               _p, C.c_int, _i32, _i64, _p, _p, _sz, _p]),
    "ctr_interaction_width": (C.c_int64, [_i32, _i32, C.c_int]),
    "ctr_embedding_bag_bwd_update_opt": (C.c_int, [_p, _i64, _i64, _p, _i32, _i32, C.c_int, _p, _p, _p, _p, _i64,
                                                   _f32, _p, C.c_int, _i32, _i64, _p, C.c_int, _p, _p, _sz, _p]),
    "ctr_dot_interaction_mode": (C.c_int, [_p, C.c_int, _i32, _i32, _i32, C.c_int, _p, _p, _sz, _p]),
    "ctr_dot_interaction_bwd_mode": (C.c_int, [_p, _p, _i32, _i32, _i32, C.c_int, _p, _p, _sz, _p]),
    "ctr_embedding_bag_bwd_update_phases": (C.c_int, [_p, _i64, _i64, _p, _i32, _i32, C.c_int, _p, _p, _p, _p, _i64,
                                                      _f32, _p, C.c_int, _i32, _i64, _p, C.c_int, _p, _sz, _p]),
}


class CtrError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {status} ({status_string(status)})")
        self.status = status


def lib() -> C.CDLL:
    """Load libctr.so, building it first if the sources changed.  Raises if that fails."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libctr not found at {path}")
            L = C.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def status_string(status: int) -> str:
    return lib().ctr_status_string(int(status)).decode()


def _ok(name: str, st: int) -> None:
    if st != 0:
        raise CtrError(name, st)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _host_i32(a) -> C.Array:
    a = np.ascontiguousarray(a, dtype=np.int32)
    return (C.c_int32 * a.size)(*a.tolist())


def _host_i64(a) -> C.Array:
    a = np.ascontiguousarray(a, dtype=np.int64)
    return (C.c_int64 * a.size)(*a.tolist())


def _dev(t: torch.Tensor, what: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    return t


KERNEL_GATHER, KERNEL_BWD_TILES, KERNEL_BWD_PIECES, KERNEL_SORT, KERNEL_INTERACTION, KERNEL_INTERACTION_BWD, \
    KERNEL_GATHER_ROWS = 1, 2, 3, 4, 5, 6, 7


def ctr_set_timing_events(kernel: int, before=None, after=None) -> None:
    """Record torch.cuda.Events around every later launch of `kernel` (None, None: off).

    The events must already have been recorded once, so that torch has created them.
    """
    b = None if before is None else C.c_void_p(before.cuda_event)
    e = None if after is None else C.c_void_p(after.cuda_event)
    _ok("ctr_set_timing_events", lib().ctr_set_timing_events(int(kernel), b, e))


def ctr_launch_count() -> int:
    """Kernel launches the library has issued in this process so far."""
    return int(lib().ctr_launch_count())


def ctr_set_tma_gather(on: bool) -> bool:
    """Select the TMA row-gather variant of the fp32 d=128 pooled gather; returns the previous setting."""
    return bool(lib().ctr_set_tma_gather(1 if on else 0))


def ctr_set_wait_limit_ns(ns: int) -> int:
    """Wall-clock limit of each radix-pass look-back wait of ctr_dedup (diagnostics); returns the previous."""
    return int(lib().ctr_set_wait_limit_ns(int(ns)))


def ctr_set_tile_slices(mode: int) -> int:
    """Short-run pass of the fp32 d=128 SGD row update: 0 automatic, 1 never sliced, 2 always in
    64-column slices; returns the previous mode."""
    return int(lib().ctr_set_tile_slices(int(mode)))


# ---------------------------------------------------------------------------
# status / workspace
# ---------------------------------------------------------------------------
def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed device buffer usable as a libctr workspace (torch allocations are 512-byte aligned)."""
    return torch.zeros(int(nbytes), dtype=torch.uint8, device=device or "cuda")


def ctr_status_reset(ws: torch.Tensor, stream=None) -> None:
    _ok("ctr_status_reset", lib().ctr_status_reset(_ptr(ws), _stream(stream)))


def ctr_check_status(ws: torch.Tensor, stream=None) -> int:
    return int(lib().ctr_check_status(_ptr(ws), _stream(stream)))


def ctr_dedup_workspace_size(n_ids: int, num_fields: int, batch: int, total_rows: int) -> int:
    return int(lib().ctr_dedup_workspace_size(n_ids, num_fields, batch, total_rows))


def ctr_embedding_bag_workspace_size() -> int:
    return int(lib().ctr_embedding_bag_workspace_size())


def ctr_interaction_workspace_size() -> int:
    return int(lib().ctr_interaction_workspace_size())


def ctr_bwd_update_workspace_size(n_ids: int, d: int) -> int:
    return int(lib().ctr_bwd_update_workspace_size(n_ids, d))


# ---------------------------------------------------------------------------
# calls
# ---------------------------------------------------------------------------
def ctr_fill_table(table: torch.Tensor, d: int, row0: int, gen_kind: int, seed: int, scale: float,
                   stream=None) -> None:
    _dev(table, "table")
    rows = table.numel() // d
    _ok("ctr_fill_table", lib().ctr_fill_table(_ptr(table), DTYPES[table.dtype], rows, d, row0, gen_kind,
                                               C.c_uint64(seed & ((1 << 64) - 1)), scale, _stream(stream)))


def ctr_dedup(ids: torch.Tensor, offsets: torch.Tensor, num_fields: int, batch: int, bag_to_table: Sequence[int],
              row_base: Sequence[int], unique_rows: torch.Tensor, n_unique: torch.Tensor,
              inverse: Optional[torch.Tensor], sorted_pos: Optional[torch.Tensor], sorted_bag: Optional[torch.Tensor],
              run_offsets: Optional[torch.Tensor], unique_offsets: Optional[torch.Tensor], ws: torch.Tensor,
              n_ids: Optional[int] = None, stream=None) -> None:
    n = int(ids.numel()) if n_ids is None else int(n_ids)
    rb = np.asarray(row_base, dtype=np.int64)
    st = lib().ctr_dedup(_ptr(ids), _ptr(offsets), num_fields, batch, _host_i32(bag_to_table), _host_i64(rb),
                         rb.size - 1, n, _ptr(unique_rows), _ptr(n_unique), _ptr(inverse), _ptr(sorted_pos),
                         _ptr(sorted_bag), _ptr(run_offsets), _ptr(unique_offsets), _ptr(ws), ws.numel(),
                         _stream(stream))
    _ok("ctr_dedup", st)


DEDUP_PREPARE, DEDUP_SORT, DEDUP_ALL = 1, 2, 3


def ctr_dedup_phases(ids: torch.Tensor, offsets: torch.Tensor, num_fields: int, batch: int,
                     bag_to_table: Sequence[int], row_base: Sequence[int], unique_rows: torch.Tensor,
                     n_unique: torch.Tensor, inverse: Optional[torch.Tensor], sorted_pos: Optional[torch.Tensor],
                     sorted_bag: Optional[torch.Tensor], run_offsets: Optional[torch.Tensor],
                     unique_offsets: Optional[torch.Tensor], phases: int, ws: torch.Tensor,
                     n_ids: Optional[int] = None, stream=None) -> None:
    n = int(ids.numel()) if n_ids is None else int(n_ids)
    rb = np.asarray(row_base, dtype=np.int64)
    st = lib().ctr_dedup_phases(_ptr(ids), _ptr(offsets), num_fields, batch, _host_i32(bag_to_table),
                                _host_i64(rb), rb.size - 1, n, _ptr(unique_rows), _ptr(n_unique), _ptr(inverse),
                                _ptr(sorted_pos), _ptr(sorted_bag), _ptr(run_offsets), _ptr(unique_offsets),
                                int(phases), _ptr(ws), ws.numel(), _stream(stream))
    _ok("ctr_dedup_phases", st)


def ctr_gather_rows(table: torch.Tensor, d: int, unique_rows: torch.Tensor, n_unique: torch.Tensor, U: torch.Tensor,
                    ws: torch.Tensor, stream=None) -> None:
    total_rows = table.numel() // d
    capacity = U.numel() // d
    st = lib().ctr_gather_rows(_ptr(table), DTYPES[table.dtype], d, total_rows, _ptr(unique_rows), _ptr(n_unique),
                               capacity, _ptr(U), _ptr(ws), ws.numel(), _stream(stream))
    _ok("ctr_gather_rows", st)


def ctr_embedding_bag_fwd(table: torch.Tensor, d: int, indices: torch.Tensor, offsets: torch.Tensor,
                          num_fields: int, batch: int, bag_to_table: Optional[Sequence[int]],
                          row_base: Optional[Sequence[int]], pool: int, out: torch.Tensor, out_stride_b: int,
                          out_stride_f: int, ws: torch.Tensor, total_rows: Optional[int] = None,
                          n_indices: Optional[int] = None, stream=None, fm_out: Optional[torch.Tensor] = None) -> None:
    """Pooled gather; with fm_out (fp32 [F*B]) the ctr_embedding_bag_fwd_fm call, which also
    writes each bag's FM second-order term."""
    total = int(table.numel() // d) if total_rows is None else int(total_rows)
    if bag_to_table is not None:
        rb = np.asarray(row_base, dtype=np.int64)
        b2t, rbp, T = _host_i32(bag_to_table), _host_i64(rb), rb.size - 1
    else:
        b2t, rbp, T = None, None, 0
    n_idx = int(indices.numel()) if n_indices is None else int(n_indices)
    args = (_ptr(table), DTYPES[table.dtype], d, total, _ptr(indices), 1 if indices.dtype == torch.int32 else 0, n_idx,
            _ptr(offsets), num_fields, batch, b2t, rbp, T, pool, _ptr(out), DTYPES[out.dtype], out_stride_b,
            out_stride_f)
    if fm_out is None:
        st = lib().ctr_embedding_bag_fwd(*args, _ptr(ws), ws.numel(), _stream(stream))
        _ok("ctr_embedding_bag_fwd", st)
    else:
        st = lib().ctr_embedding_bag_fwd_fm(*args, _ptr(fm_out), _ptr(ws), ws.numel(), _stream(stream))
        _ok("ctr_embedding_bag_fwd_fm", st)


def ctr_dot_interaction(X: torch.Tensor, n: int, d: int, out: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    batch = X.numel() // (n * d)
    st = lib().ctr_dot_interaction(_ptr(X), DTYPES[X.dtype], batch, n, d, _ptr(out), _ptr(ws), ws.numel(),
                                   _stream(stream))
    _ok("ctr_dot_interaction", st)


def ctr_dot_interaction_bwd(dout: torch.Tensor, X: torch.Tensor, n: int, d: int, dX: torch.Tensor,
                            ws: torch.Tensor, stream=None) -> None:
    batch = X.numel() // (n * d)
    st = lib().ctr_dot_interaction_bwd(_ptr(dout), _ptr(X), batch, n, d, _ptr(dX), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _ok("ctr_dot_interaction_bwd", st)


INTERACT_CROSS, INTERACT_WITH_SELF, INTERACT_FULL_GRAM = 0, 1, 2


def ctr_interaction_width(n: int, d: int, mode: int) -> int:
    return int(lib().ctr_interaction_width(n, d, mode))


def ctr_dot_interaction_mode(X: torch.Tensor, n: int, d: int, mode: int, out: torch.Tensor, ws: torch.Tensor,
                             stream=None) -> None:
    batch = X.numel() // (n * d)
    st = lib().ctr_dot_interaction_mode(_ptr(X), DTYPES[X.dtype], batch, n, d, int(mode), _ptr(out), _ptr(ws),
                                        ws.numel(), _stream(stream))
    _ok("ctr_dot_interaction_mode", st)


def ctr_dot_interaction_bwd_mode(dout: torch.Tensor, X: torch.Tensor, n: int, d: int, mode: int, dX: torch.Tensor,
                                 ws: torch.Tensor, stream=None) -> None:
    batch = X.numel() // (n * d)
    st = lib().ctr_dot_interaction_bwd_mode(_ptr(dout), _ptr(X), batch, n, d, int(mode), _ptr(dX), _ptr(ws),
                                            ws.numel(), _stream(stream))
    _ok("ctr_dot_interaction_bwd_mode", st)


def ctr_embedding_bag_bwd_update(grad_pooled: torch.Tensor, g_stride_b: int, g_stride_f: int, offsets: torch.Tensor,
                                 num_fields: int, batch: int, pool: int, unique_rows: torch.Tensor,
                                 n_unique: torch.Tensor, run_offsets: torch.Tensor, sorted_bag: torch.Tensor,
                                 n_ids: int, lr: float, table: torch.Tensor, d: int,
                                 grad_unique_out: Optional[torch.Tensor], ws: torch.Tensor, stream=None) -> None:
    total_rows = table.numel() // d
    st = lib().ctr_embedding_bag_bwd_update(_ptr(grad_pooled), g_stride_b, g_stride_f, _ptr(offsets), num_fields,
                                            batch, pool, _ptr(unique_rows), _ptr(n_unique), _ptr(run_offsets),
                                            _ptr(sorted_bag), n_ids, lr, _ptr(table), DTYPES[table.dtype], d,
                                            total_rows, _ptr(grad_unique_out), _ptr(ws), ws.numel(), _stream(stream))
    _ok("ctr_embedding_bag_bwd_update", st)


BWD_LONG_RUNS, BWD_SHORT_RUNS, BWD_FINISH = 1, 2, 4
BWD_ALL = BWD_SHORT_RUNS | BWD_LONG_RUNS | BWD_FINISH
OPT_SGD, OPT_ADAGRAD, OPT_ROWWISE_ADAGRAD, OPT_ADAM = 0, 1, 2, 3


class CtrOptimizer(C.Structure):
    """ctr_optimizer of ctr.h."""
    _fields_ = [("kind", C.c_int), ("eps", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("step", C.c_int64), ("state0", C.c_void_p), ("state1", C.c_void_p),
                ("stochastic_rounding", C.c_int32), ("sr_seed", C.c_uint64)]


def optimizer(kind: int, eps: float = 1e-8, beta1: float = 0.9, beta2: float = 0.999, step: int = 1,
              state0: Optional[torch.Tensor] = None, state1: Optional[torch.Tensor] = None,
              stochastic_rounding: bool = False, sr_seed: int = 0) -> CtrOptimizer:
    return CtrOptimizer(int(kind), float(eps), float(beta1), float(beta2), int(step),
                        None if state0 is None else _ptr(state0), None if state1 is None else _ptr(state1),
                        1 if stochastic_rounding else 0, int(sr_seed) & ((1 << 64) - 1))


def ctr_embedding_bag_bwd_update_opt(grad_pooled: torch.Tensor, g_stride_b: int, g_stride_f: int,
                                     offsets: torch.Tensor, num_fields: int, batch: int, pool: int,
                                     unique_rows: torch.Tensor, n_unique: torch.Tensor, run_offsets: torch.Tensor,
                                     sorted_bag: torch.Tensor, n_ids: int, lr: float, table: torch.Tensor, d: int,
                                     grad_unique_out: Optional[torch.Tensor], phases: int, opt: CtrOptimizer,
                                     ws: torch.Tensor, stream=None) -> None:
    total_rows = table.numel() // d
    st = lib().ctr_embedding_bag_bwd_update_opt(_ptr(grad_pooled), g_stride_b, g_stride_f, _ptr(offsets), num_fields,
                                                batch, pool, _ptr(unique_rows), _ptr(n_unique), _ptr(run_offsets),
                                                _ptr(sorted_bag), n_ids, lr, _ptr(table), DTYPES[table.dtype], d,
                                                total_rows, _ptr(grad_unique_out), int(phases), C.addressof(opt),
                                                _ptr(ws), ws.numel(), _stream(stream))
    _ok("ctr_embedding_bag_bwd_update_opt", st)


def ctr_embedding_bag_bwd_update_phases(grad_pooled: torch.Tensor, g_stride_b: int, g_stride_f: int,
                                        offsets: torch.Tensor, num_fields: int, batch: int, pool: int,
                                        unique_rows: torch.Tensor, n_unique: torch.Tensor, run_offsets: torch.Tensor,
                                        sorted_bag: torch.Tensor, n_ids: int, lr: float, table: torch.Tensor, d: int,
                                        grad_unique_out: Optional[torch.Tensor], phases: int, ws: torch.Tensor,
                                        stream=None) -> None:
    total_rows = table.numel() // d
    st = lib().ctr_embedding_bag_bwd_update_phases(_ptr(grad_pooled), g_stride_b, g_stride_f, _ptr(offsets),
                                                   num_fields, batch, pool, _ptr(unique_rows), _ptr(n_unique),
                                                   _ptr(run_offsets), _ptr(sorted_bag), n_ids, lr, _ptr(table),
                                                   DTYPES[table.dtype], d, total_rows, _ptr(grad_unique_out),
                                                   int(phases), _ptr(ws), ws.numel(), _stream(stream))
    _ok("ctr_embedding_bag_bwd_update_phases", st)
