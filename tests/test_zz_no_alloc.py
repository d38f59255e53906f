"""The allocation-free dedup (ctr_dedup_static) against the regular ctr_dedup.

Callers that may not allocate device memory (a plugin inside a runtime that
owns all device allocation, a server with a fixed memory budget, a
latency-critical loop) use ctr_dedup_static, whose scratch lives in a fixed
array inside the library.  This file runs last (pytest collects it last by
name) and must also pass on its own in a fresh process.  Calls in a row on
different inputs check that the shared array, which keeps the previous call's
contents, gives the same results as the workspace-based entry point and as
the oracle: the dedup's outputs are unique under the stable ascending order,
so all three must agree bit for bit.  The two internal paths of the dedup (a
presence bitmap when the tables are at most 64 rows per ID, sorted keys
otherwise) leave different scratch behind, so they run in both orders.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import ctr
from sparse_embeddings_feature_gb300 import workload as W

pytestmark = pytest.mark.gpu

_p = C.c_void_p


def _static_fn():
    fn = ctr.lib().ctr_dedup_static
    fn.restype = C.c_int
    fn.argtypes = [_p, _p, C.c_int32, C.c_int32, _p, _p, C.c_int32, C.c_int64, _p, _p, _p, _p, _p, _p, _p, _p, _p]
    return fn


def _outputs(n, T):
    cap = max(n, 1)
    return {
        "unique_rows": torch.full((cap,), -9, dtype=torch.int64, device="cuda"),
        "n_unique": torch.full((1,), -9, dtype=torch.int64, device="cuda"),
        "inverse": torch.full((cap,), -9, dtype=torch.int32, device="cuda"),
        "sorted_pos": torch.full((cap,), -9, dtype=torch.int32, device="cuda"),
        "sorted_bag": torch.full((cap,), -9, dtype=torch.int32, device="cuda"),
        "run_offsets": torch.full((cap + 1,), -9, dtype=torch.int32, device="cuda"),
        "unique_offsets": torch.full((T + 1,), -9, dtype=torch.int64, device="cuda"),
    }


def _host(o, n):
    torch.cuda.synchronize()
    k = int(o["n_unique"].item())
    return {"n_unique": k, "unique_rows": o["unique_rows"][:k].cpu().numpy(), "inverse": o["inverse"][:n].cpu().numpy(),
            "sorted_pos": o["sorted_pos"][:n].cpu().numpy(), "sorted_bag": o["sorted_bag"][:n].cpu().numpy(),
            "run_offsets": o["run_offsets"][:k + 1].cpu().numpy(),
            "unique_offsets": o["unique_offsets"].cpu().numpy()}


def _run_both(cfg=None, w=None, F=None, B=None):
    """The static and the workspace dedup on one input (a workload config, or
    arrays w with F fields of B bags), and the oracle's dedup of it."""
    if w is None:
        w = W.make_workload(cfg, with_grads=False)
        F, B = cfg.num_fields, cfg.batch
    n = int(w["ids"].size)
    T = int(np.asarray(w["row_base"]).size - 1)
    total_rows = int(np.asarray(w["row_base"])[-1])
    ids = torch.from_numpy(w["ids"]).cuda()
    offs = torch.from_numpy(w["offsets"]).cuda()
    # regular entry point with a workspace
    ref = _outputs(n, T)
    ws = ctr.workspace(ctr.ctr_dedup_workspace_size(n, F, B, total_rows))
    ctr.ctr_dedup(ids, offs, F, B, w["bag_to_table"], w["row_base"], ref["unique_rows"], ref["n_unique"],
                  ref["inverse"], ref["sorted_pos"], ref["sorted_bag"], ref["run_offsets"], ref["unique_offsets"],
                  ws, n_ids=n)
    assert ctr.ctr_check_status(ws) == 0
    # allocation-free entry point
    got = _outputs(n, T)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    b2t = np.ascontiguousarray(w["bag_to_table"], dtype=np.int32)
    rb = np.ascontiguousarray(w["row_base"], dtype=np.int64)
    st = _static_fn()(ids.data_ptr(), offs.data_ptr(), F, B, b2t.ctypes.data, rb.ctypes.data, T, n,
                      got["unique_rows"].data_ptr(), got["n_unique"].data_ptr(), got["inverse"].data_ptr(),
                      got["sorted_pos"].data_ptr(), got["sorted_bag"].data_ptr(), got["run_offsets"].data_ptr(),
                      got["unique_offsets"].data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, ctr.status_string(st)
    assert int(status.item()) == 0
    orc = O.dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    return _host(got, n), _host(ref, n), orc


def _assert_same(got, ref, orc):
    assert got["n_unique"] == ref["n_unique"] == orc["n_unique"]
    for k in ("unique_rows", "inverse", "sorted_pos", "sorted_bag", "run_offsets", "unique_offsets"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k + " (static vs workspace)")
        np.testing.assert_array_equal(got[k], orc[k], err_msg=k + " (static vs oracle)")


def _uses_bitmap(cfg):
    return cfg.total_rows <= 64 * int(W.make_workload(cfg, with_grads=False)["ids"].size)


SORTED_A = W.CONFIGS["full_step"].shrink(batch=384)        # 208M rows for ~250k IDs: sorted keys
SORTED_B = W.CONFIGS["tensornet"].shrink(batch=300)        # 2^26 rows for ~165k IDs: sorted keys
BITMAP = W.CONFIGS["tiny"]                                 # 4000 rows for 256 IDs: presence bitmap


def test_static_dedup_matches_workspace_dedup_and_oracle_twice():
    # two calls in a row on different inputs: the shared array is reused
    assert not _uses_bitmap(SORTED_A) and not _uses_bitmap(SORTED_B)
    for cfg in (SORTED_A, SORTED_B):
        _assert_same(*_run_both(cfg))


def test_static_dedup_bitmap_and_sorted_paths_in_both_orders():
    assert _uses_bitmap(BITMAP)
    for cfg in (BITMAP, SORTED_A, BITMAP, SORTED_B, BITMAP):
        _assert_same(*_run_both(cfg))


def test_static_dedup_at_its_limit_on_the_largest_scratch():
    # 2^20 IDs over 64 x 2^20 rows: the presence bitmap's largest scratch (46 MB), the
    # peak of the dedup's workspace at this many IDs
    n = 1 << 20
    rows = 64 * n
    rng = np.random.default_rng(123)
    ranks = rng.zipf(1.1, size=3 * n)
    ranks = ranks[ranks <= rows][:n] - 1
    assert ranks.size == n
    ids = (ranks * 2654435761 + 12345) % rows
    F, B = 4, n // 4
    w = {"ids": ids.astype(np.int64), "offsets": np.arange(0, n + 1, dtype=np.int64),
         "bag_to_table": np.zeros(F, dtype=np.int32), "row_base": np.array([0, rows], dtype=np.int64)}
    assert ctr.ctr_dedup_workspace_size(n, F, B, rows) > (40 << 20)
    got, ref, orc = _run_both(w=w, F=F, B=B)
    _assert_same(got, ref, orc)


def test_static_dedup_rejects_batches_beyond_its_array():
    fn = _static_fn()
    b2t = np.zeros(1, dtype=np.int32)
    rb = np.array([0, 10], dtype=np.int64)
    dummy = 256
    st = fn(dummy, dummy, 1, 1, b2t.ctypes.data, rb.ctypes.data, 1, (1 << 20) + 1, dummy, dummy, None, None, None,
            None, None, None, None)
    assert st == -2  # CTR_ERR_UNSUPPORTED, nothing launched
