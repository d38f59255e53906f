"""The bounded waits of the dedup's radix passes, made to run out on purpose.

Each radix pass waits (bounded by wall-clock time) for earlier tiles to publish
their digit counts.  ctr_set_wait_limit_ns shortens that limit so that ordinary
waits run out: nothing faults or hangs, the waiting tile records
CTR_ERR_TIMEOUT in the workspace and keeps every write inside its buffers, and
the context stays usable.  Guard zones around every output and after the
workspace must keep their sentinel bytes; afterwards, with the default limit,
the same dedup must again equal the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import ctr
from sparse_embeddings_feature_gb300 import workload as W

pytestmark = pytest.mark.gpu

GUARD = 256  # guard elements on each side of every output (16-byte aligned views)


def _guarded(n, dtype, fill):
    full = torch.full((n + 2 * GUARD,), fill, dtype=dtype, device="cuda")
    return full, full[GUARD:GUARD + n]


def _run(w, F, B, limit_ns=None):
    n = int(w["ids"].size)
    T = int(np.asarray(w["row_base"]).size - 1)
    total_rows = int(np.asarray(w["row_base"])[-1])
    ids = torch.from_numpy(w["ids"]).cuda()
    offs = torch.from_numpy(w["offsets"]).cuda()
    bufs = {"unique_rows": _guarded(n, torch.int64, -7), "n_unique": _guarded(1, torch.int64, -7),
            "inverse": _guarded(n, torch.int32, -7), "sorted_pos": _guarded(n, torch.int32, -7),
            "sorted_bag": _guarded(n, torch.int32, -7), "run_offsets": _guarded(n + 1, torch.int32, -7),
            "unique_offsets": _guarded(T + 1, torch.int64, -7)}
    need = ctr.ctr_dedup_workspace_size(n, F, B, total_rows)
    ws_full = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    ws_full[:256].zero_()                              # a cleared error word and counters, as ctr.workspace gives
    ws = ws_full[:need]
    prev = ctr.ctr_set_wait_limit_ns(limit_ns) if limit_ns is not None else None
    try:
        ctr.ctr_dedup(ids, offs, F, B, w["bag_to_table"], w["row_base"], *(bufs[k][1] for k in bufs), ws, n_ids=n)
        status = ctr.ctr_check_status(ws)
    finally:
        if prev is not None:
            ctr.ctr_set_wait_limit_ns(prev)
    torch.cuda.synchronize()
    for k, (full, _) in bufs.items():
        g = full.cpu().numpy()
        assert np.all(g[:GUARD] == -7) and np.all(g[-GUARD:] == -7), f"a write left {k}"
    assert np.all(ws_full[need:].cpu().numpy() == 0xA5), "a write left the workspace"
    return status, {k: v[1].cpu().numpy() for k, v in bufs.items()}


def test_radix_lookback_timeout_is_reported_and_writes_stay_in_bounds():
    cfg = W.CONFIGS["full_step"].shrink(batch=8192, rows_per_table=tuple([100_000] * 26))
    w = W.make_workload(cfg, with_grads=False)
    F, B = cfg.num_fields, cfg.batch
    assert w["ids"].size > 5_000_000                   # over a thousand 4096-key tiles per pass
    # a zero limit: a tile that finds an earlier tile's counts unpublished gives up at once;
    # with over a thousand tiles per pass in flight that happens in practice on every call,
    # but scheduling decides, so a few calls are allowed to find one
    seen = []
    for _ in range(5):
        st, _ = _run(w, F, B, limit_ns=0)
        seen.append(st)
        if st == ctr.ERR_TIMEOUT:
            break
    assert ctr.ERR_TIMEOUT in seen, seen
    assert all(s in (0, ctr.ERR_TIMEOUT) for s in seen), seen
    # the context is still usable and the default limit gives the oracle's result again
    st, got = _run(w, F, B)
    assert st == 0
    ref = O.dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    nu = int(got["n_unique"][0])
    assert nu == ref["n_unique"]
    np.testing.assert_array_equal(got["unique_rows"][:nu], ref["unique_rows"])
    for k in ("inverse", "sorted_pos", "sorted_bag"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    np.testing.assert_array_equal(got["run_offsets"][:nu + 1], ref["run_offsets"])
    np.testing.assert_array_equal(got["unique_offsets"], ref["unique_offsets"])
