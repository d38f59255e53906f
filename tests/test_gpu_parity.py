"""GPU parity: every libctr call against the CPU oracle on the same seeded inputs.

Indexing outputs (dedup) must match bit for bit; floating-point outputs within
the tolerances of tests/_tol.py.  Sizes span several tiles of every kernel and
end in ragged tails; edge cases cover empty bags and batches, repeated IDs,
IDs at the ends of their tables, long runs and the degenerate shapes.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import ctr
from sparse_embeddings_feature_gb300 import workload as W
from sparse_embeddings_feature_gb300.pipeline import CtrPath, HostPipeline

from _tol import bf16_close, bwd_depth, f32_close, fm_depth, gamma, pool_depth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _t(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV)


def _np(t):
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _gen(cfg):
    return (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)


def _csr(lens, rng, rows_of_field, B):
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ids = np.empty(int(offsets[-1]), dtype=np.int64)
    for bag in range(lens.size):
        f = bag // B
        ids[offsets[bag]:offsets[bag + 1]] = rng.integers(0, rows_of_field[f], size=lens[bag])
    return ids, offsets


def gpu_dedup(ids, offsets, F, B, b2t, row_base, with_pos=True):
    n = int(offsets[-1])
    cap = max(n, 1)
    T = len(row_base) - 1
    dev = {k: torch.full((cap,), -7, dtype=torch.int32, device=DEV)
           for k in ("inverse", "sorted_pos", "sorted_bag")}
    if not with_pos:
        dev["sorted_pos"] = None
    uq = torch.full((cap,), -7, dtype=torch.int64, device=DEV)
    nu = torch.full((1,), -7, dtype=torch.int64, device=DEV)
    ro = torch.full((cap + 1,), -7, dtype=torch.int32, device=DEV)
    uo = torch.full((T + 1,), -7, dtype=torch.int64, device=DEV)
    ws = ctr.workspace(ctr.ctr_dedup_workspace_size(cap, F, B, int(row_base[-1])))
    ids_d = _t(ids if n else np.zeros(1, np.int64))
    ctr.ctr_dedup(ids_d, _t(offsets), F, B, b2t, row_base, uq, nu, dev["inverse"], dev["sorted_pos"],
                  dev["sorted_bag"], ro, uo, ws, n_ids=n)
    st = ctr.ctr_check_status(ws)
    k = int(_np(nu)[0])
    return st, {"unique_rows": _np(uq)[:k], "n_unique": k, "inverse": _np(dev["inverse"])[:n],
                "sorted_pos": _np(dev["sorted_pos"])[:n] if with_pos else None,
                "sorted_bag": _np(dev["sorted_bag"])[:n],
                "run_offsets": _np(ro)[:k + 1], "unique_offsets": _np(uo)}


def assert_dedup_equal(got, ref):
    assert got["n_unique"] == ref["n_unique"]
    for k in ("unique_rows", "inverse", "sorted_pos", "sorted_bag", "run_offsets", "unique_offsets"):
        if got[k] is not None:
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


# ---------------------------------------------------------------------------
# input generator: device fill == oracle fill, bit for bit
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["dlrm_fp32", "bf16_large"])
def test_fill_table_bit_exact(name):
    cfg = W.CONFIGS[name]
    d = cfg.d
    rows = 5000
    row0 = 3_999_000
    tdt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    t = torch.empty((rows, d), dtype=tdt, device=DEV)
    ctr.ctr_fill_table(t, d, row0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    ref = O.table_rows(cfg.fill_kind, cfg.fill_seed, cfg.fill_scale, d, np.arange(row0, row0 + rows))
    np.testing.assert_array_equal(_np(t), ref)


# ---------------------------------------------------------------------------
# a1 dedup
# ---------------------------------------------------------------------------
DEDUP_CASES = {
    "tiny": W.CONFIGS["tiny"],
    "dlrm_fp32": W.CONFIGS["dlrm_fp32"],
    "tensornet_b512": W.CONFIGS["tensornet"].shrink(batch=512),
    "full_step_b256": W.CONFIGS["full_step"].shrink(batch=256),
    "bf16_b128": W.CONFIGS["bf16_large"].shrink(batch=128),
}


@pytest.mark.parametrize("name", list(DEDUP_CASES))
def test_dedup_configs(name):
    cfg = DEDUP_CASES[name]
    w = W.make_workload(cfg, with_grads=False)
    args = (w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"], w["row_base"])
    ref = O.dedup(*args)
    for with_pos in (True, False):
        st, got = gpu_dedup(*args, with_pos=with_pos)
        assert st == 0, ctr.status_string(st)
        assert_dedup_equal(got, ref)


# Tables at most 64x the batch's ID count take the presence-bitmap path (ranks
# from a bitmap, a sort of the ranks); larger ones sort the keys themselves.
# These cases put both paths, and rank keys of 24 and 25 bits (3 and 4 radix
# passes), against the oracle.
BITMAP_CASES = {
    "tensornet_b4096": W.CONFIGS["tensornet"].shrink(batch=4096),
    "uniform_b32768_25bit_ranks": W.CONFIGS["full_step"].shrink(batch=32768, ids=("uniform",)),
    "full_step_b16384": W.CONFIGS["full_step"].shrink(batch=16384),
}


@pytest.mark.parametrize("name", list(BITMAP_CASES))
def test_dedup_bitmap_path(name):
    cfg = BITMAP_CASES[name]
    w = W.make_workload(cfg, with_grads=False)
    assert cfg.total_rows <= 64 * w["ids"].size           # the bitmap path
    args = (w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"], w["row_base"])
    ref = O.dedup(*args)
    if name.endswith("25bit_ranks"):
        assert ref["n_unique"] > 1 << 24
    for with_pos in (True, False):
        st, got = gpu_dedup(*args, with_pos=with_pos)
        assert st == 0, ctr.status_string(st)
        assert_dedup_equal(got, ref)


@pytest.mark.parametrize("name", ["full_step_b256", "bitmap"])
def test_dedup_in_two_parts_equals_one_call(name):
    """ctr_dedup_phases: the prepare part, then (on another stream, behind an
    event) the sort part, give the one-call dedup's outputs, on both paths."""
    cfg = DEDUP_CASES["full_step_b256"] if name != "bitmap" else BITMAP_CASES["tensornet_b4096"]
    w = W.make_workload(cfg, with_grads=False)
    args = (w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"], w["row_base"])
    ref = O.dedup(*args)
    n = int(w["offsets"][-1])
    F, B, T = cfg.num_fields, cfg.batch, len(w["row_base"]) - 1
    for with_pos in (True, False):
        out = {k: torch.full((n,), -7, dtype=torch.int32, device=DEV) for k in ("inverse", "sorted_pos", "sorted_bag")}
        if not with_pos:
            out["sorted_pos"] = None
        uq = torch.full((n,), -7, dtype=torch.int64, device=DEV)
        nu = torch.full((1,), -7, dtype=torch.int64, device=DEV)
        ro = torch.full((n + 1,), -7, dtype=torch.int32, device=DEV)
        uo = torch.full((T + 1,), -7, dtype=torch.int64, device=DEV)
        ws = ctr.workspace(ctr.ctr_dedup_workspace_size(n, F, B, int(w["row_base"][-1])))
        ids, offs = _t(w["ids"]), _t(w["offsets"])
        call = (ids, offs, F, B, w["bag_to_table"], w["row_base"], uq, nu, out["inverse"], out["sorted_pos"],
                out["sorted_bag"], ro, uo)
        side = torch.cuda.Stream()
        ev = torch.cuda.Event()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            ctr.ctr_dedup_phases(*call, ctr.DEDUP_PREPARE, ws)
            ev.record(side)
        torch.cuda.current_stream().wait_event(ev)
        ctr.ctr_dedup_phases(*call, ctr.DEDUP_SORT, ws)
        assert ctr.ctr_check_status(ws) == 0
        k = int(_np(nu)[0])
        got = {"unique_rows": _np(uq)[:k], "n_unique": k, "inverse": _np(out["inverse"]),
               "sorted_pos": _np(out["sorted_pos"]) if with_pos else None, "sorted_bag": _np(out["sorted_bag"]),
               "run_offsets": _np(ro)[:k + 1], "unique_offsets": _np(uo)}
        assert_dedup_equal(got, ref)


def test_dedup_permuted_tables_and_empty_fields():
    # fields read tables in another order (the outputs follow table order), one field
    # has only empty bags, and one field's IDs span many sort tiles with a ragged tail
    rng = np.random.default_rng(21)
    F, B = 5, 3000
    rows = [4000, 90, 1, 70_000, 600]
    b2t = np.array([3, 0, 4, 1, 2], dtype=np.int32)
    rb = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    lens = rng.integers(0, 9, size=F * B)
    lens[2 * B:3 * B] = 0                              # field 2 (table 4) has no IDs
    ids, offsets = _csr(lens, rng, [rows[t] for t in b2t], B)
    assert sum(rows) <= 64 * ids.size
    ref = O.dedup(ids, offsets, F, B, b2t, rb)
    for with_pos in (True, False):
        st, got = gpu_dedup(ids, offsets, F, B, b2t, rb, with_pos=with_pos)
        assert st == 0, ctr.status_string(st)
        assert_dedup_equal(got, ref)


def test_dedup_table_with_more_than_2_20_distinct_rows():
    # one table with about 2.1M distinct rows in the batch (22-bit ranks within the table)
    rng = np.random.default_rng(22)
    F, B, rows = 2, 1_500_000, [1 << 22, 1000]
    lens = np.concatenate([np.full(B, 2), rng.integers(0, 3, size=B)]).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ids = np.concatenate([rng.integers(0, rows[0], size=2 * B), rng.integers(0, rows[1], size=int(lens[B:].sum()))])
    b2t = np.array([0, 1], dtype=np.int32)
    rb = np.array([0, rows[0], rows[0] + rows[1]], dtype=np.int64)
    assert sum(rows) <= 64 * ids.size
    ref = O.dedup(ids, offsets, F, B, b2t, rb)
    assert ref["unique_offsets"][1] - ref["unique_offsets"][0] > (1 << 20)
    st, got = gpu_dedup(ids, offsets, F, B, b2t, rb, with_pos=False)
    assert st == 0, ctr.status_string(st)
    assert_dedup_equal(got, ref)


def test_dedup_edge_cases():
    rng = np.random.default_rng(0)
    # (F, B, rows per table, bag lengths builder)
    cases = []
    F, B = 3, 50
    rows = [7, 1, 100_000]
    lens = rng.integers(0, 4, size=F * B)
    lens[:20] = 0                                     # empty bags interleaved
    cases.append((F, B, rows, lens, None))
    cases.append((2, 10, [5, 5], np.zeros(20, np.int64), None))   # every bag empty: n_ids = 0
    lens = np.full(4, 3000)                           # one ID repeated: long runs, ragged tail
    cases.append((1, 4, [9], lens, "same"))
    lens = rng.integers(4090, 4100, size=6)           # n_ids just around tile multiples
    cases.append((2, 3, [2 ** 20, 2 ** 20], lens, "ends"))
    for F, B, rows, lens, mode in cases:
        b2t = np.arange(F, dtype=np.int32)
        rb = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
        ids, offsets = _csr(np.asarray(lens), rng, rows, B)
        if mode == "same":
            ids[:] = 4
        if mode == "ends":
            ids[::2] = np.array(rows)[np.repeat(np.arange(F), [offsets[(f + 1) * B] - offsets[f * B]
                                                                for f in range(F)])][::2] - 1
            ids[1::3] = 0
        ref = O.dedup(ids, offsets, F, B, b2t, rb)
        for with_pos in (True, False):
            st, got = gpu_dedup(ids, offsets, F, B, b2t, rb, with_pos=with_pos)
            assert st == 0
            assert_dedup_equal(got, ref)


def test_dedup_tables_sharing_and_empty_tables():
    rng = np.random.default_rng(5)
    F, B = 4, 64
    rows = [300, 0, 50]                               # table 1 is empty; fields 0 and 3 share table 0
    b2t = np.array([0, 2, 2, 0], dtype=np.int32)
    rb = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    lens = rng.integers(0, 9, size=F * B)
    ids, offsets = _csr(lens, rng, [rows[t] for t in b2t], B)
    st, got = gpu_dedup(ids, offsets, F, B, b2t, rb)
    assert st == 0
    assert_dedup_equal(got, O.dedup(ids, offsets, F, B, b2t, rb))


def test_dedup_flags_out_of_range_id():
    ids = np.array([0, 3, 5, 1], dtype=np.int64)      # 5 is outside a 5-row table
    offsets = np.array([0, 2, 4], dtype=np.int64)
    st, _ = gpu_dedup(ids, offsets, 1, 2, np.array([0], np.int32), np.array([0, 5], np.int64))
    assert st == -4, ctr.status_string(st)


def test_dedup_flags_id_of_empty_table():
    # field 0 reads table 0, which has no rows: every such ID is out of range
    ids = np.array([0, 1, 7, 3], dtype=np.int64)
    offsets = np.array([0, 2, 4], dtype=np.int64)
    st, _ = gpu_dedup(ids, offsets, 2, 1, np.array([0, 1], np.int32), np.array([0, 0, 10], np.int64))
    assert st == -4, ctr.status_string(st)


def test_dedup_flags_bad_offsets():
    ids = np.zeros(4, dtype=np.int64)
    offsets = np.array([0, 3, 2, 4], dtype=np.int64)  # not monotone
    st, _ = gpu_dedup(ids, offsets, 1, 3, np.array([0], np.int32), np.array([0, 5], np.int64))
    assert st == -8


def test_dedup_is_deterministic():
    cfg = DEDUP_CASES["full_step_b256"]
    w = W.make_workload(cfg, with_grads=False)
    args = (w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"], w["row_base"])
    _, a = gpu_dedup(*args)
    _, b = gpu_dedup(*args)
    assert_dedup_equal(a, b)


# ---------------------------------------------------------------------------
# a2 pooled embedding bag
# ---------------------------------------------------------------------------
def _fwd_case(cfg, w, table=None, out_dtype=None):
    """GPU pooled output [B, F, d] (fp32 array or bf16 bits) for cfg's tables."""
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    tdt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    odt = tdt if out_dtype is None else out_dtype
    if table is None:
        tab = torch.empty((cfg.total_rows, d), dtype=tdt, device=DEV)
        ctr.ctr_fill_table(tab, d, 0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    else:
        tab = _t(table)
    out = torch.full((B, F, d), float("nan"), dtype=odt, device=DEV)
    ws = ctr.workspace(ctr.ctr_embedding_bag_workspace_size())
    pool = ctr.POOL_MEAN if cfg.pool == "mean" else ctr.POOL_SUM
    ctr.ctr_embedding_bag_fwd(tab, d, _t(w["ids"]), _t(w["offsets"]), F, B, w["bag_to_table"], w["row_base"], pool,
                              out, F * d, d, ws)
    assert ctr.ctr_check_status(ws) == 0
    return _np(out)


FWD_CASES = {
    "tiny": W.CONFIGS["tiny"],
    "dlrm_fp32": W.CONFIGS["dlrm_fp32"],
    "bf16_mean_b256": W.CONFIGS["bf16_large"].shrink(batch=256, rows_per_table=tuple([200_000] * 26)),
    "full_step_b128": W.CONFIGS["full_step"].shrink(batch=128, rows_per_table=tuple([100_000] * 26)),
}


@pytest.mark.parametrize("name", list(FWD_CASES))
def test_embedding_bag_fwd_configs(name):
    cfg = FWD_CASES[name]
    w = W.make_workload(cfg, with_grads=False)
    got = _fwd_case(cfg, w)
    ref, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"],
                                   w["row_base"], cfg.d, pool=cfg.pool, dtype=cfg.dtype, gen=_gen(cfg),
                                   with_mag=True)
    depth = pool_depth(w["offsets"], cfg.num_fields, cfg.batch)
    if cfg.dtype == "f32":
        f32_close(got, ref, mag, depth, what=name)
    else:
        bf16_close(got, ref, mag, depth, atol=1e-5, what=name)


@pytest.mark.parametrize("d,dtype,pool", [(12, "f32", "sum"), (20, "f32", "mean"), (32, "f32", "sum"),
                                          (64, "f32", "mean"), (256, "f32", "sum"), (512, "f32", "sum"),
                                          (8, "bf16", "sum"), (16, "bf16", "mean"), (128, "bf16", "sum"),
                                          (36, "bf16", "mean"), (16, "f32", "mean"), (32, "bf16", "mean"),
                                          (64, "bf16", "sum")])
def test_embedding_bag_fwd_shapes(d, dtype, pool):
    cfg = W.CONFIGS["dlrm_fp32"].shrink(batch=97, num_fields=5, field_to_table=(0, 1, 2, 3, 4),
                                        rows_per_table=(1000, 1, 50, 70_000, 9), d=d, dtype=dtype, pool=pool,
                                        table_init=("uniform", 0.5) if dtype == "f32" else ("normal4", 0.1),
                                        bag_len=("uniform", 0, 40))
    w = W.make_workload(cfg, with_grads=False)
    got = _fwd_case(cfg, w)
    ref, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"],
                                   w["row_base"], d, pool=pool, dtype=dtype, gen=_gen(cfg), with_mag=True)
    depth = pool_depth(w["offsets"], cfg.num_fields, cfg.batch)
    if dtype == "f32":
        f32_close(got, ref, mag, depth, what=f"d={d}")
    else:
        bf16_close(got, ref, mag, depth, atol=1e-5, what=f"d={d}")


@pytest.mark.parametrize("d,dtype,pool", [(16, "f32", "mean"), (32, "f32", "mean"), (64, "f32", "sum"),
                                          (32, "bf16", "mean"), (64, "bf16", "sum"), (128, "bf16", "mean")])
def test_embedding_bag_fwd_narrow_rows_unaligned_output(d, dtype, pool):
    """Rows of 4, 8 and 16 chunks of 16 bytes (several rows per warp step) written
    through an output whose row stride is odd, so no 16-byte vector store applies:
    the same bits as the aligned output, and the oracle's values."""
    cfg = W.CONFIGS["dlrm_fp32"].shrink(batch=131, num_fields=6, field_to_table=(0, 1, 2, 3, 4, 2),
                                        rows_per_table=(3000, 1, 70_000, 17, 500), d=d, dtype=dtype, pool=pool,
                                        table_init=("uniform", 0.5) if dtype == "f32" else ("normal4", 0.1),
                                        bag_len=("uniform", 0, 70))
    w = W.make_workload(cfg, with_grads=False)
    F, B = cfg.num_fields, cfg.batch
    aligned = _fwd_case(cfg, w)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    tab = torch.empty((cfg.total_rows, d), dtype=tdt, device=DEV)
    ctr.ctr_fill_table(tab, d, 0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    sb = F * d + 1
    out = torch.full((B * sb,), float("nan"), dtype=tdt, device=DEV)
    ws = ctr.workspace(ctr.ctr_embedding_bag_workspace_size())
    cpool = ctr.POOL_MEAN if pool == "mean" else ctr.POOL_SUM
    ctr.ctr_embedding_bag_fwd(tab, d, _t(w["ids"]), _t(w["offsets"]), F, B, w["bag_to_table"], w["row_base"], cpool,
                              out, sb, d, ws)
    assert ctr.ctr_check_status(ws) == 0
    got = _np(out).reshape(B, sb)
    untouched = _np(torch.full((B,), float("nan"), dtype=tdt))
    np.testing.assert_array_equal(got[:, -1].view(np.uint32 if dtype == "f32" else np.uint16),
                                  untouched.view(np.uint32 if dtype == "f32" else np.uint16))  # the gap column
    got = got[:, :F * d].reshape(B, F, d)
    np.testing.assert_array_equal(got, aligned)
    ref, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, pool=pool,
                                   dtype=dtype, gen=_gen(cfg), with_mag=True)
    depth = pool_depth(w["offsets"], F, B)
    if dtype == "f32":
        f32_close(got, ref, mag, depth, what=f"d={d}")
    else:
        bf16_close(got, ref, mag, depth, atol=1e-5, what=f"d={d}")


def test_embedding_bag_fwd_exact_and_int32_unique_path():
    # dyadic table: sums are exact, so GPU == oracle bit for bit; pooling from the
    # unique-row matrix through the int32 inverse map gives the same bits
    cfg = W.CONFIGS["tensornet"].shrink(batch=300, rows_per_table=(5000,),
                                        ids=("zipf_hashed", 1.1, 10 ** 6, 12))
    w = W.make_workload(cfg, with_grads=False)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    rng = np.random.default_rng(3)
    table = (rng.integers(-512, 512, size=(cfg.total_rows, d)) / 1024).astype(np.float32)
    direct = _fwd_case(cfg, w, table=table)
    ref = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, table=table)
    np.testing.assert_array_equal(direct, ref)
    st, dd = gpu_dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    assert st == 0
    tab = _t(table)
    nu = torch.tensor([dd["n_unique"]], dtype=torch.int64, device=DEV)
    U = torch.full((w["ids"].size, d), float("nan"), device=DEV)
    ws = ctr.workspace(256)
    ctr.ctr_gather_rows(tab, d, _t(dd["unique_rows"]), nu, U, ws)
    np.testing.assert_array_equal(_np(U)[:dd["n_unique"]], table[dd["unique_rows"]])
    out = torch.empty((B, F, d), device=DEV)
    ctr.ctr_embedding_bag_fwd(U, d, _t(dd["inverse"], torch.int32), _t(w["offsets"]), F, B, None, None,
                              ctr.POOL_SUM, out, F * d, d, ws)
    assert ctr.ctr_check_status(ws) == 0
    np.testing.assert_array_equal(_np(out), ref)


@pytest.mark.parametrize("d,dtype", [(8, "bf16"), (16, "f32"), (32, "f32"), (64, "f32"), (128, "f32"),
                                     (256, "bf16"), (24, "bf16"), (3, "f32"), (160, "f32")])
def test_gather_rows_copies_the_unique_rows(d, dtype):
    """The batch-sized matrix of the unique rows: row k of U is table row
    unique_rows[k] for k < n_unique, bit for bit, and the rows past n_unique are
    not written (rows of 1 to 32 chunks of 16 bytes, and other widths)."""
    rng = np.random.default_rng(d)
    rows = 5000
    table = rng.standard_normal((rows, d)).astype(np.float32)
    tab = _t(table) if dtype == "f32" else _t(table).to(torch.bfloat16)
    cap = 1300
    nu = 1237                                                        # ragged against every warp step
    uq = np.sort(rng.choice(rows, size=cap, replace=False)).astype(np.int64)
    U = torch.full((cap, d), float("nan"), dtype=tab.dtype, device=DEV)
    ws = ctr.workspace(256)
    ctr.ctr_gather_rows(tab, d, _t(uq), torch.tensor([nu], dtype=torch.int64, device=DEV), U, ws)
    assert ctr.ctr_check_status(ws) == 0
    got, want = _np(U), _np(tab)
    np.testing.assert_array_equal(got[:nu], want[uq[:nu]])
    nan_bits = _np(torch.full((cap - nu, d), float("nan"), dtype=tab.dtype))
    np.testing.assert_array_equal(got[nu:].view(nan_bits.dtype), nan_bits)


def test_embedding_bag_fwd_strided_into_interaction_slots():
    cfg = FWD_CASES["full_step_b128"]
    w = W.make_workload(cfg, with_grads=False)
    path = CtrPath(cfg, w["ids"].size)
    path.upload(w)
    path.forward()
    X = _np(path.X)
    ref, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"],
                                   w["row_base"], cfg.d, gen=_gen(cfg), with_mag=True)
    f32_close(X[:, 1:, :], ref, mag, pool_depth(w["offsets"], cfg.num_fields, cfg.batch), what="X slots")
    np.testing.assert_array_equal(X[:, 0, :], w["dense"])


def test_embedding_bag_fwd_flags_out_of_range():
    cfg = W.CONFIGS["tiny"]
    w = W.make_workload(cfg, with_grads=False)
    w["ids"][17] = 1000                                # rows are 0..999
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    tab = torch.zeros((cfg.total_rows, d), device=DEV)
    out = torch.empty((B, F, d), device=DEV)
    ws = ctr.workspace(256)
    ctr.ctr_embedding_bag_fwd(tab, d, _t(w["ids"]), _t(w["offsets"]), F, B, w["bag_to_table"], w["row_base"],
                              ctr.POOL_SUM, out, F * d, d, ws)
    assert ctr.ctr_check_status(ws) == -4


# ---------------------------------------------------------------------------
# a3 dot interaction
# ---------------------------------------------------------------------------
def _rand_X(B, n, d, dtype, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, n, d)).astype(np.float32)
    X[:, 1:, :] *= 0.03
    if dtype == "bf16":
        return W.f32_to_bf16_bits(X)
    return X


@pytest.mark.parametrize("B,n,d,dtype", [(1001, 27, 128, "f32"), (64, 5, 16, "f32"), (33, 9, 40, "f32"),
                                         (1001, 27, 64, "bf16"), (257, 5, 64, "bf16"), (130, 32, 128, "bf16"),
                                         (77, 2, 256, "bf16"), (40, 16, 192, "bf16"), (50, 27, 48, "bf16"),
                                         (3, 27, 64, "bf16"), (515, 17, 256, "bf16"), (129, 20, 64, "bf16")])
def test_dot_interaction(B, n, d, dtype):
    X = _rand_X(B, n, d, dtype, seed=B + n + d)
    Xd = _t(X.view(np.int16) if dtype == "bf16" else X)
    if dtype == "bf16":
        Xd = Xd.view(torch.bfloat16)
    width = d + n * (n - 1) // 2
    out = torch.full((B, width), float("nan"), dtype=Xd.dtype, device=DEV)
    ws = ctr.workspace(ctr.ctr_interaction_workspace_size())
    ctr.ctr_dot_interaction(Xd, n, d, out, ws)
    assert ctr.ctr_check_status(ws) == 0
    got = _np(out)
    ref, mag = O.dot_interaction(X, n, d, dtype=dtype, with_mag=True)
    if dtype == "f32":
        f32_close(got, ref, mag, d, what="interaction")
    else:
        bf16_close(got, ref, mag, d, what="interaction")
        np.testing.assert_array_equal(got[:, :d], ref[:, :d])


def test_dot_interaction_fm_identity_on_gpu_output():
    # sum of the GPU's pair outputs = 1/2 (|sum x|^2 - sum |x|^2) computed independently
    B, n, d = 256, 27, 128
    X = _rand_X(B, n, d, "f32", seed=1)
    out = torch.empty((B, d + n * (n - 1) // 2), device=DEV)
    ctr.ctr_dot_interaction(_t(X), n, d, out, ctr.workspace(256))
    got = _np(out)[:, d:].astype(np.float64).sum(axis=1)
    X64 = X.astype(np.float64)
    s = X64.sum(axis=1)
    rhs = 0.5 * ((s * s).sum(axis=1) - (X64 * X64).sum(axis=(1, 2)))
    mag = 0.5 * ((np.abs(X64).sum(axis=1) ** 2).sum(axis=1))
    # each output is a d-term dot rounded once (depth d + 1); the host sums them exactly
    # enough, and sum_{i<j} sum_c |x_ic x_jc| <= mag
    assert np.all(np.abs(got - rhs) <= 1e-5 * np.abs(rhs) + gamma(d + 1) * mag)


# ---------------------------------------------------------------------------
# a4 interaction backward
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,n,d", [(1001, 27, 128), (64, 5, 16), (17, 27, 64)])
def test_dot_interaction_bwd(B, n, d):
    X = _rand_X(B, n, d, "f32", seed=7)
    rng = np.random.default_rng(8)
    dout = rng.standard_normal((B, d + n * (n - 1) // 2)).astype(np.float32)
    dX = torch.full((B, n, d), float("nan"), device=DEV)
    ws = ctr.workspace(256)
    ctr.ctr_dot_interaction_bwd(_t(dout), _t(X), n, d, dX, ws)
    ref, mag = O.dot_interaction_bwd(dout, X, n, d, with_mag=True)
    f32_close(_np(dX), ref, mag, n + 1, what="interaction bwd")


# ---------------------------------------------------------------------------
# a5 sparse backward + SGD row update
# ---------------------------------------------------------------------------
def gpu_bwd(cfg, w, table_np=None, G=None, with_grad=True):
    """Runs dedup + bwd_update on the GPU; returns (new table, grad per unique, dedup)."""
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    st, dd = gpu_dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    assert st == 0
    tdt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    if table_np is None:
        tab = torch.empty((cfg.total_rows, d), dtype=tdt, device=DEV)
        ctr.ctr_fill_table(tab, d, 0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    else:
        tab = _t(table_np.view(np.int16) if table_np.dtype == np.uint16 else table_np)
        if table_np.dtype == np.uint16:
            tab = tab.view(torch.bfloat16)
    n = w["ids"].size
    Gd = _t(w["grad_pooled"] if G is None else G)
    gu = torch.full((max(n, 1), d), float("nan"), device=DEV) if with_grad else None
    ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(max(n, 1), d))
    pool = ctr.POOL_MEAN if cfg.pool == "mean" else ctr.POOL_SUM
    nu = torch.tensor([dd["n_unique"]], dtype=torch.int64, device=DEV)
    ro = torch.from_numpy(np.concatenate([dd["run_offsets"], np.zeros(max(n, 1) - dd["n_unique"], np.int32)])).to(DEV)
    ctr.ctr_embedding_bag_bwd_update(Gd, F * d, d, _t(w["offsets"]), F, B, pool, _t(dd["unique_rows"]), nu, ro,
                                     _t(dd["sorted_bag"]) if n else torch.zeros(1, dtype=torch.int32, device=DEV),
                                     max(n, 1), cfg.lr, tab, d, gu, ws)
    assert ctr.ctr_check_status(ws) == 0
    gnp = _np(gu)[:dd["n_unique"]] if with_grad else None
    return _np(tab), gnp, dd


def test_bwd_update_exact_arithmetic_with_long_runs():
    # dyadic gradients and table, lr a power of two: every sum is exact, so
    # the GPU must equal the oracle bit for bit, whatever its summation order
    rng = np.random.default_rng(11)
    F, B, d = 3, 700, 32
    rows = [40, 3, 5000]
    lens = rng.integers(0, 12, size=F * B)
    lens[B:B + 40] = 400                               # long runs in field 1 (3 rows)
    ids, offsets = _csr(lens, rng, rows, B)
    cfg = W.CONFIGS["tiny"].shrink(batch=B, num_fields=F, field_to_table=(0, 1, 2), rows_per_table=tuple(rows),
                                   d=d, lr=2.0 ** -6)
    table = (rng.integers(-256, 256, size=(sum(rows), d)) / 256).astype(np.float32)
    G = (rng.integers(-16, 17, size=(B, F, d)) / 16).astype(np.float32)
    w = {"ids": ids, "offsets": offsets, "bag_to_table": np.arange(F, dtype=np.int32),
         "row_base": cfg.row_base, "grad_pooled": G}
    new_tab, g, dd = gpu_bwd(cfg, w, table_np=table)
    assert int(np.diff(dd["run_offsets"]).max()) > 128 * 8   # several pieces, several warps per combine
    rows_t = dd["unique_rows"]
    ref_new, ref_g, _ = O.embedding_bag_bwd_update(G, ids, offsets, F, B, w["bag_to_table"], cfg.row_base, d,
                                                   cfg.lr, rows_t, table=table)
    np.testing.assert_array_equal(g, ref_g.astype(np.float32))
    np.testing.assert_array_equal(new_tab[rows_t], ref_new)
    untouched = np.setdiff1d(np.arange(sum(rows)), rows_t)
    np.testing.assert_array_equal(new_tab[untouched], table[untouched])


@pytest.fixture
def tile_slices():
    """Sets the short-run pass's column-slice mode for one test, restoring it after."""
    prev = []

    def set_mode(mode):
        prev.append(ctr.ctr_set_tile_slices(mode))

    yield set_mode
    if prev:
        ctr.ctr_set_tile_slices(prev[0])


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("d", [128, 64, 32, 20, 4])
def test_bwd_update_exact_arithmetic_sliced_and_plain(mode, d, tile_slices):
    # fp32 rows under SGD: mode 2 forces the pair kernel (slices of at most 64 columns, two
    # occurrences per warp step), mode 1 the plain tile kernel; dyadic inputs make every
    # sum exact, so both must equal the oracle bit for bit, long runs and ragged tiles included
    tile_slices(mode)
    rng = np.random.default_rng(12 + mode + d)
    F, B = 3, 901
    rows = [37, 5, 4000]
    lens = rng.integers(0, 9, size=F * B)
    lens[B:B + 30] = 300                               # long runs in field 1
    ids, offsets = _csr(lens, rng, rows, B)
    cfg = W.CONFIGS["tiny"].shrink(batch=B, num_fields=F, field_to_table=(0, 1, 2), rows_per_table=tuple(rows),
                                   d=d, lr=2.0 ** -6)
    table = (rng.integers(-256, 256, size=(sum(rows), d)) / 256).astype(np.float32)
    G = (rng.integers(-16, 17, size=(B, F, d)) / 16).astype(np.float32)
    w = {"ids": ids, "offsets": offsets, "bag_to_table": np.arange(F, dtype=np.int32),
         "row_base": cfg.row_base, "grad_pooled": G}
    new_tab, g, dd = gpu_bwd(cfg, w, table_np=table)
    run_len = np.diff(dd["run_offsets"])
    assert (run_len <= 128).sum() > 1000 and (run_len > 128).any()
    rows_t = dd["unique_rows"]
    ref_new, ref_g, _ = O.embedding_bag_bwd_update(G, ids, offsets, F, B, w["bag_to_table"], cfg.row_base, d,
                                                   cfg.lr, rows_t, table=table)
    np.testing.assert_array_equal(g, ref_g.astype(np.float32))
    np.testing.assert_array_equal(new_tab[rows_t], ref_new)
    untouched = np.setdiff1d(np.arange(sum(rows)), rows_t)
    np.testing.assert_array_equal(new_tab[untouched], table[untouched])


@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_bwd_update_sliced_pass_against_oracle_and_deterministic(pool, tile_slices):
    # the pair kernel on the full step's row shape (d = 128, Zipf IDs, 26 tables), forced on
    # at a small batch: the oracle within each run's depth, and the same bits twice
    tile_slices(2)
    cfg = W.CONFIGS["full_step"].shrink(batch=700, rows_per_table=tuple([40_000] * 26), backward="pooled_grad",
                                        pool=pool)
    w = W.make_workload(cfg)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    new_tab, g, dd = gpu_bwd(cfg, w)
    new_tab2, g2, _ = gpu_bwd(cfg, w)
    np.testing.assert_array_equal(g, g2)
    np.testing.assert_array_equal(new_tab, new_tab2)
    rows_t = dd["unique_rows"]
    ref_new, ref_g, mag = O.embedding_bag_bwd_update(w["grad_pooled"], w["ids"], w["offsets"], F, B,
                                                     w["bag_to_table"], w["row_base"], d, cfg.lr, rows_t,
                                                     pool=pool, gen=_gen(cfg))
    depth = bwd_depth(np.diff(dd["run_offsets"]))[:, None]
    f32_close(g, ref_g, mag, depth, what=f"sliced grad ({pool})")
    old = O.table_rows(cfg.fill_kind, cfg.fill_seed, cfg.fill_scale, d, rows_t)
    f32_close(new_tab[rows_t], ref_new, cfg.lr * mag + np.abs(old), depth + 2, what=f"sliced rows ({pool})")


BWD_CASES = {
    "tiny": W.CONFIGS["tiny"],
    "tensornet_b512": W.CONFIGS["tensornet"].shrink(batch=512),
    "tensornet_mean_b256": W.CONFIGS["tensornet"].shrink(batch=256, pool="mean"),
    "bf16_b64": W.CONFIGS["bf16_large"].shrink(batch=64, rows_per_table=tuple([30_000] * 26),
                                               backward="pooled_grad"),
    "d128_b300": W.CONFIGS["full_step"].shrink(batch=300, rows_per_table=tuple([20_000] * 26),
                                              backward="pooled_grad"),
}


@pytest.mark.parametrize("name", list(BWD_CASES))
def test_bwd_update_configs(name):
    cfg = BWD_CASES[name]
    w = W.make_workload(cfg)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    new_tab, g, dd = gpu_bwd(cfg, w)
    rows_t = dd["unique_rows"]
    ref_new, ref_g, mag = O.embedding_bag_bwd_update(w["grad_pooled"], w["ids"], w["offsets"], F, B,
                                                     w["bag_to_table"], w["row_base"], d, cfg.lr, rows_t,
                                                     pool=cfg.pool, dtype=cfg.dtype, gen=_gen(cfg))
    depth = bwd_depth(np.diff(dd["run_offsets"]))[:, None]
    f32_close(g, ref_g, mag, depth, what=f"{name} grad")
    old = O.table_rows(cfg.fill_kind, cfg.fill_seed, cfg.fill_scale, d, rows_t)
    # the update adds two roundings: the product lr * g and the subtraction
    if cfg.dtype == "f32":
        f32_close(new_tab[rows_t], ref_new, cfg.lr * mag + np.abs(old), depth + 2, what=f"{name} rows")
    else:
        bf16_close(new_tab[rows_t], ref_new, cfg.lr * mag, depth + 2, atol=1e-5, what=f"{name} rows")
    # rows the batch does not touch keep their bits
    probe = np.setdiff1d(np.arange(0, cfg.total_rows, max(1, cfg.total_rows // 5000)), rows_t)
    np.testing.assert_array_equal(new_tab[probe], O.table_rows(cfg.fill_kind, cfg.fill_seed, cfg.fill_scale, d, probe))


def test_bwd_update_is_deterministic():
    cfg = BWD_CASES["tensornet_b512"]
    w = W.make_workload(cfg)
    a, ga, _ = gpu_bwd(cfg, w)
    b, gb, _ = gpu_bwd(cfg, w)
    np.testing.assert_array_equal(ga, gb)
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# the whole step, composed, against the oracle composed the same way
# ---------------------------------------------------------------------------
def test_full_step_composed_small():
    cfg = W.CONFIGS["full_step"].shrink(batch=192, rows_per_table=tuple([60_000] * 26))
    w = W.make_workload(cfg)
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    path = CtrPath(cfg, w["ids"].size, keep_sorted_pos=True)
    path.upload(w)
    path.reset_status()
    path.step()
    assert all(v == 0 for v in path.check_status().values())
    gen = _gen(cfg)
    # oracle chain
    dd = O.dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    pooled, pmag = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen,
                                       with_mag=True)
    rows_t = dd["unique_rows"]
    got_dd = {"unique_rows": _np(path.unique_rows)[:dd["n_unique"]], "n_unique": int(_np(path.n_unique)[0]),
              "inverse": _np(path.inverse), "sorted_pos": _np(path.sorted_pos), "sorted_bag": _np(path.sorted_bag),
              "run_offsets": _np(path.run_offsets)[:dd["n_unique"] + 1], "unique_offsets": _np(path.unique_offsets)}
    assert_dedup_equal(got_dd, dd)
    Xg, dXg = _np(path.X), _np(path.dX)
    np.testing.assert_array_equal(Xg[:, 0, :], w["dense"])
    f32_close(Xg[:, 1:, :], pooled, pmag, pool_depth(w["offsets"], F, B), what="pooled")
    # the oracle chain from here on takes the GPU's own input of each step (checked just before),
    # so every bound is that step's own reduction depth
    out_ref, out_mag = O.dot_interaction(Xg, n, d, with_mag=True)
    dX_ref, dX_mag = O.dot_interaction_bwd(w["dout"], Xg, n, d, with_mag=True)
    f32_close(_np(path.out), out_ref, out_mag, d, what="interaction")
    f32_close(dXg, dX_ref, dX_mag, n, what="interaction bwd")
    new_ref, _, mag = O.embedding_bag_bwd_update(dXg[:, 1:, :], w["ids"], w["offsets"], F, B,
                                                 w["bag_to_table"], w["row_base"], d, cfg.lr, rows_t, gen=gen)
    old = O.table_rows(gen[0], gen[1], gen[2], d, rows_t)
    depth = bwd_depth(np.diff(dd["run_offsets"]))[:, None] + 2
    f32_close(_np(path.table)[rows_t], new_ref, cfg.lr * mag + np.abs(old), depth, what="updated rows")


def test_launch_counter_counts_each_step_alike():
    cfg = W.CONFIGS["full_step"].shrink(batch=64, rows_per_table=tuple([5_000] * 26))
    w = W.make_workload(cfg)
    path = CtrPath(cfg, w["ids"].size)
    path.upload(w)
    path.reset_status()
    c0 = ctr.ctr_launch_count()
    path.step()
    c1 = ctr.ctr_launch_count()
    path.step()
    c2 = ctr.ctr_launch_count()
    torch.cuda.synchronize()
    assert all(v == 0 for v in path.check_status().values())
    # dedup (clear, keygen, radix passes, unique count, scan, unique write), gather,
    # interaction, interaction backward, and the backward's clear + tiles + pieces + combine
    assert c1 - c0 >= 14
    assert c2 - c1 == c1 - c0


def test_host_pipeline_matches_sequential_steps():
    # three different batches through the overlapped host pipeline give the same
    # outputs and the same updated table, bit for bit, as plain sequential steps
    from sparse_embeddings_feature_gb300.pipeline import HostPipeline
    base = W.CONFIGS["full_step"].shrink(batch=96, rows_per_table=tuple([4_000] * 26))
    ws_ = [W.make_workload(base.shrink(seed=s)) for s in (11, 12, 13)]
    cap = max(w["ids"].size for w in ws_)

    def pinned(w):
        return {k: torch.from_numpy(np.ascontiguousarray(w[k])).pin_memory() for k in ("ids", "offsets", "dense", "dout")}

    seq = CtrPath(base, cap)
    seq_out = []
    for w in ws_:
        n = w["ids"].size
        seq.n_ids = n
        seq.ids[:n].copy_(torch.from_numpy(w["ids"]))
        seq.offsets.copy_(torch.from_numpy(w["offsets"]))
        seq.X[:, 0, :].copy_(torch.from_numpy(w["dense"]))
        seq.dout.copy_(torch.from_numpy(w["dout"]))
        seq.reset_status()
        seq.step()
        seq_out.append(_np(seq.out).copy())
        assert all(v == 0 for v in seq.check_status().values())

    pip = CtrPath(base, cap)
    pipe = HostPipeline(pip)
    outs = [torch.empty(tuple(pip.out.shape), dtype=torch.float32).pin_memory() for _ in ws_]
    pip.reset_status()
    pipe.run([pinned(w) for w in ws_], outs)
    torch.cuda.synchronize()
    assert all(v == 0 for v in pip.check_status().values())
    for k in range(len(ws_)):
        np.testing.assert_array_equal(outs[k].numpy(), seq_out[k])
    np.testing.assert_array_equal(_np(pip.table), _np(seq.table))


@pytest.mark.parametrize("mode", ["sequential", "two_streams"])
def test_bwd_update_phases_match_single_call(mode):
    # the phased update (long runs, short runs, finish), in order on one stream or
    # with the long runs on a second stream, gives the single call's bits
    cfg = BWD_CASES["tensornet_b512"]
    w = W.make_workload(cfg)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    ref_tab, ref_g, dd = gpu_bwd(cfg, w)
    assert int(np.diff(dd["run_offsets"]).max()) > 128            # there are long runs
    n = w["ids"].size
    tab = torch.empty((cfg.total_rows, d), dtype=torch.float32, device=DEV)
    ctr.ctr_fill_table(tab, d, 0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    gu = torch.full((n, d), float("nan"), device=DEV)
    ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(n, d))
    nu = torch.tensor([dd["n_unique"]], dtype=torch.int64, device=DEV)
    ro = torch.from_numpy(np.concatenate([dd["run_offsets"], np.zeros(n - dd["n_unique"], np.int32)])).to(DEV)
    args = (_t(w["grad_pooled"]), F * d, d, _t(w["offsets"]), F, B, ctr.POOL_SUM, _t(dd["unique_rows"]), nu, ro,
            _t(dd["sorted_bag"]), n, cfg.lr, tab, d, gu)
    torch.cuda.synchronize()
    if mode == "sequential":
        for ph in (ctr.BWD_LONG_RUNS, ctr.BWD_SHORT_RUNS, ctr.BWD_FINISH):
            ctr.ctr_embedding_bag_bwd_update_phases(*args, ph, ws)
    else:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            ctr.ctr_embedding_bag_bwd_update_phases(*args, ctr.BWD_LONG_RUNS, ws)
        ctr.ctr_embedding_bag_bwd_update_phases(*args, ctr.BWD_SHORT_RUNS, ws)
        torch.cuda.current_stream().wait_stream(side)
        ctr.ctr_embedding_bag_bwd_update_phases(*args, ctr.BWD_FINISH, ws)
    assert ctr.ctr_check_status(ws) == 0
    np.testing.assert_array_equal(_np(tab), ref_tab)
    np.testing.assert_array_equal(_np(gu)[:dd["n_unique"]], ref_g)


def test_bwd_update_phases_rejects_empty_mask():
    n, d = 8, 16
    ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(n, d))
    z = torch.zeros(64, device=DEV)
    i64 = torch.zeros(8, dtype=torch.int64, device=DEV)
    i32 = torch.zeros(9, dtype=torch.int32, device=DEV)
    with pytest.raises(ctr.CtrError):
        ctr.ctr_embedding_bag_bwd_update_phases(z, d, d, i64, 1, 2, ctr.POOL_SUM, i64, i64, i32, i32, n, 0.1,
                                                z.view(4, 16), d, None, 0, ws)


# ---------------------------------------------------------------------------
# interaction variants: with the diagonal, full Gram matrix
# ---------------------------------------------------------------------------
MODES = {"cross": ctr.INTERACT_CROSS, "with_self": ctr.INTERACT_WITH_SELF, "full": ctr.INTERACT_FULL_GRAM}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("B,n,d,dtype", [(1001, 27, 128, "f32"), (33, 9, 40, "f32"), (1001, 27, 64, "bf16"),
                                         (130, 32, 128, "bf16"), (77, 2, 256, "bf16"), (50, 27, 48, "bf16"),
                                         (129, 20, 64, "bf16"), (6, 17, 192, "bf16")])
def test_dot_interaction_modes(mode, B, n, d, dtype):
    X = _rand_X(B, n, d, dtype, seed=B + n + d + 7)
    Xd = _t(X.view(np.int16) if dtype == "bf16" else X)
    if dtype == "bf16":
        Xd = Xd.view(torch.bfloat16)
    width = ctr.ctr_interaction_width(n, d, MODES[mode])
    assert width == O.interaction_width(n, d, mode)
    out = torch.full((B, width), float("nan"), dtype=Xd.dtype, device=DEV)
    ws = ctr.workspace(ctr.ctr_interaction_workspace_size())
    ctr.ctr_dot_interaction_mode(Xd, n, d, MODES[mode], out, ws)
    assert ctr.ctr_check_status(ws) == 0
    got = _np(out)
    ref, mag = O.dot_interaction_mode(X, n, d, mode, dtype=dtype, with_mag=True)
    if dtype == "f32":
        f32_close(got, ref, mag, d, what=f"interaction {mode}")
    else:
        bf16_close(got, ref, mag, d, what=f"interaction {mode}")
    if mode != "full":
        np.testing.assert_array_equal(got[:, :d], ref[:, :d])


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("B,n,d", [(1001, 27, 128), (64, 5, 16), (17, 27, 64)])
def test_dot_interaction_bwd_modes(mode, B, n, d):
    rng = np.random.default_rng(B * n + d)
    X = rng.standard_normal((B, n, d)).astype(np.float32)
    width = O.interaction_width(n, d, mode)
    dout = rng.standard_normal((B, width)).astype(np.float32)
    dX = torch.full((B, n, d), float("nan"), device=DEV)
    ws = ctr.workspace(ctr.ctr_interaction_workspace_size())
    ctr.ctr_dot_interaction_bwd_mode(_t(dout), _t(X), n, d, MODES[mode], dX, ws)
    assert ctr.ctr_check_status(ws) == 0
    ref, mag = O.dot_interaction_bwd_mode(dout, X, n, d, mode, with_mag=True)
    # dx_i sums at most 2n products (the full Gram matrix counts <x_i, x_j> and <x_j, x_i>
    # apart; the other modes n - 1 or n), plus the dense pass-through
    depth = 2 * n + 1 if mode == "full" else n + 1
    f32_close(_np(dX), ref, mag, depth, what=f"interaction bwd {mode}")


def test_dot_interaction_mode_rejects_bad_mode():
    X = torch.zeros((4, 5, 16), device=DEV)
    out = torch.zeros((4, 64), device=DEV)
    with pytest.raises(ctr.CtrError):
        ctr.ctr_dot_interaction_mode(X, 5, 16, 3, out, ctr.workspace(256))
    assert ctr.ctr_interaction_width(5, 16, 3) == -1


# ---------------------------------------------------------------------------
# FM second-order term of each bag, fused into the pooled gather
# ---------------------------------------------------------------------------
FM_CASES = {
    "tiny": W.CONFIGS["tiny"],
    "dlrm_fp32": W.CONFIGS["dlrm_fp32"],
    "bf16_mean_b256": W.CONFIGS["bf16_large"].shrink(batch=256, rows_per_table=tuple([200_000] * 26)),
    "tensornet_b300": W.CONFIGS["tensornet"].shrink(batch=300),
    "full_step_b128": W.CONFIGS["full_step"].shrink(batch=128, rows_per_table=tuple([100_000] * 26)),
}


@pytest.mark.parametrize("name", list(FM_CASES))
def test_embedding_bag_fwd_fm(name):
    cfg = FM_CASES[name]
    w = W.make_workload(cfg, with_grads=False)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    tdt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    tab = torch.empty((cfg.total_rows, d), dtype=tdt, device=DEV)
    ctr.ctr_fill_table(tab, d, 0, cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    out = torch.empty((B, F, d), dtype=tdt, device=DEV)
    fm = torch.full((F * B,), float("nan"), device=DEV)
    ws = ctr.workspace(ctr.ctr_embedding_bag_workspace_size())
    pool = ctr.POOL_MEAN if cfg.pool == "mean" else ctr.POOL_SUM
    ctr.ctr_embedding_bag_fwd(tab, d, _t(w["ids"]), _t(w["offsets"]), F, B, w["bag_to_table"], w["row_base"], pool,
                              out, F * d, d, ws, fm_out=fm)
    assert ctr.ctr_check_status(ws) == 0
    ref, mag = O.bag_fm(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, dtype=cfg.dtype,
                        gen=_gen(cfg), with_mag=True)
    # the GPU evaluates 1/2 (|sum v|^2 - sum |v|^2) in fp32: its error is bounded by the
    # accumulation depth times the two terms' magnitudes, 2 (sum |v_i v_j| + sum |v|^2 / 2)
    lens = np.diff(w["offsets"])
    rows = cfg.row_base[np.asarray(cfg.field_to_table)[np.repeat(np.arange(F * B) // B, lens)]] + w["ids"]
    vals = O.table_rows(cfg.fill_kind, cfg.fill_seed, cfg.fill_scale, d, rows)
    if cfg.dtype == "bf16":
        vals = W.bf16_bits_to_f32(vals)
    per_id = np.concatenate([(vals.astype(np.float64) ** 2).sum(axis=1), [0.0]])  # sentinel: empty last bag
    sq = np.add.reduceat(per_id, w["offsets"][:-1]) * (lens > 0)
    f32_close(_np(fm), ref, 2.0 * mag + sq, fm_depth(lens, d), what=f"FM term {name}")
    # the pooled output is the plain gather's
    out2 = torch.empty_like(out)
    ctr.ctr_embedding_bag_fwd(tab, d, _t(w["ids"]), _t(w["offsets"]), F, B, w["bag_to_table"], w["row_base"], pool,
                              out2, F * d, d, ws)
    assert torch.equal(out.view(torch.int16) if cfg.dtype == "bf16" else out,
                       out2.view(torch.int16) if cfg.dtype == "bf16" else out2)


# ---------------------------------------------------------------------------
# optimizer state in the row update (Adagrad, row-wise Adagrad, Adam)
# ---------------------------------------------------------------------------
U32 = 2.0 ** -24


def _opt_case(seed, d, dtype, opt):
    """Dyadic table, gradients and states: the reduced gradients are exact on both
    sides, so only the optimizer's own fp32 arithmetic differs from the oracle."""
    rng = np.random.default_rng(seed)
    F, B = 3, 700
    rows = [40, 3, 5000]
    lens = rng.integers(0, 12, size=F * B)
    lens[B:B + 40] = 400                               # long runs (pieces, combine)
    ids, offsets = _csr(lens, rng, rows, B)
    T = sum(rows)
    table = (rng.integers(-256, 256, size=(T, d)) / 256).astype(np.float32)
    if dtype == "bf16":
        table = W.bf16_bits_to_f32(W.f32_to_bf16_bits(table))  # bf16-exact values
    G = (rng.integers(-16, 17, size=(B, F, d)) / 16).astype(np.float32)
    rb = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    s0 = (rng.integers(0, 64, size=(T,) if opt == "rowwise_adagrad" else (T, d)) / 16).astype(np.float32)
    s1 = (rng.integers(0, 64, size=(T, d)) / 64).astype(np.float32) if opt == "adam" else None
    if opt == "adam":
        s0 = (rng.integers(-32, 33, size=(T, d)) / 64).astype(np.float32)
    return F, B, rows, ids, offsets, table, G, rb, s0, s1


@pytest.mark.parametrize("opt", ["adagrad", "rowwise_adagrad", "adam"])
@pytest.mark.parametrize("d,dtype", [(32, "f32"), (128, "f32"), (256, "f32"), (64, "bf16"),
                                     (44, "bf16"), (116, "bf16")])   # odd uniques per tile x odd d/4
def test_bwd_update_optimizers_exact_gradients(opt, d, dtype):
    F, B, rows, ids, offsets, table, G, rb, s0, s1 = _opt_case(d + len(opt), d, dtype, opt)
    b2t = np.arange(F, dtype=np.int32)
    st, dd = gpu_dedup(ids, offsets, F, B, b2t, rb)
    assert st == 0
    n = ids.size
    lr, eps, b1, b2, step = 2.0 ** -6, 1e-3, 0.875, 0.9375, 3
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    tab = _t(table).to(tdt)
    S0 = _t(s0)
    S1 = _t(s1) if s1 is not None else None
    gu = torch.full((n, d), float("nan"), device=DEV)
    ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(n, d))
    nu = torch.tensor([dd["n_unique"]], dtype=torch.int64, device=DEV)
    ro = torch.from_numpy(np.concatenate([dd["run_offsets"], np.zeros(n - dd["n_unique"], np.int32)])).to(DEV)
    kind = {"adagrad": ctr.OPT_ADAGRAD, "rowwise_adagrad": ctr.OPT_ROWWISE_ADAGRAD, "adam": ctr.OPT_ADAM}[opt]
    o = ctr.optimizer(kind, eps=eps, beta1=b1, beta2=b2, step=step, state0=S0, state1=S1)
    ctr.ctr_embedding_bag_bwd_update_opt(_t(G), F * d, d, _t(offsets), F, B, ctr.POOL_SUM, _t(dd["unique_rows"]), nu,
                                         ro, _t(dd["sorted_bag"]), n, lr, tab, d, gu, ctr.BWD_ALL, o, ws)
    assert ctr.ctr_check_status(ws) == 0
    rows_t = dd["unique_rows"]
    _, g_ref, _ = O.embedding_bag_bwd_update(G, ids, offsets, F, B, b2t, rb, d, lr, rows_t, table=table)
    np.testing.assert_array_equal(_np(gu)[:dd["n_unique"]], g_ref.astype(np.float32))   # exact gradients
    w_new, s0_new, s1_new = O.optimizer_step(opt, table[rows_t].astype(np.float64), g_ref, lr, state0=s0[rows_t],
                                             state1=None if s1 is None else s1[rows_t], eps=eps, beta1=b1, beta2=b2,
                                             step=step, dtype=dtype)
    got = _np(tab)[rows_t]
    if dtype == "f32":
        step_ref = np.abs(table[rows_t].astype(np.float64) - w_new.astype(np.float64))
        err = np.abs(got.astype(np.float64) - w_new.astype(np.float64))
        tol = 2 * U32 * np.abs(w_new.astype(np.float64)) + 12 * U32 * step_ref + 1e-30
        assert np.all(err <= tol), (opt, float((err - tol).max()))
    else:
        # bf16 rows: at most one bf16 rounding step apart (the rounding boundary may fall between fp32 and fp64)
        a = W.bf16_bits_to_f32(got).astype(np.float64)
        r = W.bf16_bits_to_f32(w_new).astype(np.float64)
        assert np.all(np.abs(a - r) <= np.abs(r) * 2.0 ** -7 + 1e-30)
    S0n = _np(S0)
    if opt == "rowwise_adagrad":
        np.testing.assert_allclose(S0n[rows_t], s0_new, rtol=4 * U32)
    else:
        np.testing.assert_allclose(S0n[rows_t], s0_new, rtol=4 * U32, atol=1e-30)
    if s1 is not None:
        np.testing.assert_allclose(_np(S1)[rows_t], s1_new, rtol=4 * U32, atol=1e-30)
    # rows and states the batch does not touch are unchanged
    untouched = np.setdiff1d(np.arange(sum(rows)), rows_t)
    np.testing.assert_array_equal(S0n[untouched], s0[untouched])
    if dtype == "f32":
        np.testing.assert_array_equal(_np(tab)[untouched], table[untouched])


def test_bwd_update_optimizer_validation():
    n, d = 8, 16
    ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(n, d))
    z = torch.zeros(64, device=DEV)
    i64 = torch.zeros(8, dtype=torch.int64, device=DEV)
    i32 = torch.zeros(9, dtype=torch.int32, device=DEV)
    tab = torch.zeros((4, 16), device=DEV)
    for o in (ctr.optimizer(ctr.OPT_ADAGRAD, state0=None),                          # state missing
              ctr.optimizer(ctr.OPT_ADAM, state0=tab, state1=tab, step=0),           # step must be >= 1
              ctr.optimizer(ctr.OPT_ADAGRAD, eps=0.0, state0=tab),                   # eps must be > 0
              ctr.optimizer(7)):
        with pytest.raises(ctr.CtrError):
            ctr.ctr_embedding_bag_bwd_update_opt(z, d, d, i64, 1, 2, ctr.POOL_SUM, i64, i64, i32, i32, n, 0.1, tab, d,
                                                 None, ctr.BWD_ALL, o, ws)


# ---------------------------------------------------------------------------
# stochastic rounding of the updated bf16 rows
# ---------------------------------------------------------------------------
def _bf16_ulp(v):
    """Spacing of bf16 values at |v| (8 significant bits; subnormal spacing 2^-133)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("opt", ["sgd", "adagrad", "rowwise_adagrad", "adam"])
@pytest.mark.parametrize("d", [32, 44, 64, 256])
def test_bwd_update_stochastic_rounding(opt, d):
    F, B, rows, ids, offsets, table, G, rb, s0, s1 = _opt_case(3 * d + len(opt), d, "bf16",
                                                               "adagrad" if opt == "sgd" else opt)
    b2t = np.arange(F, dtype=np.int32)
    st, dd = gpu_dedup(ids, offsets, F, B, b2t, rb)
    assert st == 0
    n = ids.size
    lr, eps, b1, b2, step = 2.0 ** -6, 1e-3, 0.875, 0.9375, 2
    seed = 0x5EED0000 + 977 * d + len(opt)
    tab = _t(table).to(torch.bfloat16)
    S0 = None if opt == "sgd" else _t(s0)
    S1 = _t(s1) if (opt == "adam") else None
    ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(n, d))
    nu = torch.tensor([dd["n_unique"]], dtype=torch.int64, device=DEV)
    ro = torch.from_numpy(np.concatenate([dd["run_offsets"], np.zeros(n - dd["n_unique"], np.int32)])).to(DEV)
    kind = {"sgd": ctr.OPT_SGD, "adagrad": ctr.OPT_ADAGRAD, "rowwise_adagrad": ctr.OPT_ROWWISE_ADAGRAD,
            "adam": ctr.OPT_ADAM}[opt]
    o = ctr.optimizer(kind, eps=eps, beta1=b1, beta2=b2, step=step, state0=S0, state1=S1,
                      stochastic_rounding=True, sr_seed=seed)
    ctr.ctr_embedding_bag_bwd_update_opt(_t(G), F * d, d, _t(offsets), F, B, ctr.POOL_SUM, _t(dd["unique_rows"]), nu,
                                         ro, _t(dd["sorted_bag"]), n, lr, tab, d, None, ctr.BWD_ALL, o, ws)
    assert ctr.ctr_check_status(ws) == 0
    rows_t = dd["unique_rows"]
    _, g_ref, _ = O.embedding_bag_bwd_update(G, ids, offsets, F, B, b2t, rb, d, lr, rows_t, table=table)
    w_old = table[rows_t].astype(np.float64)
    kw = dict(state0=None if opt == "sgd" else s0[rows_t], state1=s1[rows_t] if opt == "adam" else None,
              eps=eps, beta1=b1, beta2=b2, step=step, dtype="bf16")
    w_sr, _, _ = O.optimizer_step(opt, w_old, g_ref, lr, sr_seed=seed, rows=rows_t, **kw)
    w_rn, _, _ = O.optimizer_step(opt, w_old, g_ref, lr, **kw)
    got = _np(tab).view(np.uint16)[rows_t]
    if opt == "sgd":
        # dyadic inputs: w - lr g is exact in fp32 and fp64, so the same random bits give the same bits
        np.testing.assert_array_equal(got, w_sr)
    else:
        # the fp32 and fp64 values may straddle a rounding boundary: one bf16 step apart at most, rarely
        a = W.bf16_bits_to_f32(got).astype(np.float64)
        r = W.bf16_bits_to_f32(w_sr).astype(np.float64)
        assert np.all(np.abs(a - r) <= _bf16_ulp(np.maximum(np.abs(a), np.abs(r))) + 1e-300)
        assert np.mean(got != w_sr) < 0.01
    # stochastic, not nearest: a good share of the values that were not representable round the other way
    inexact = W.bf16_bits_to_f32(w_rn).astype(np.float64) != W.bf16_bits_to_f32(w_sr).astype(np.float64)
    assert inexact.mean() > 0.05 and np.mean(got != w_rn) > 0.05
    # rows the batch does not touch are unchanged
    untouched = np.setdiff1d(np.arange(sum(rows)), rows_t)
    np.testing.assert_array_equal(_np(tab).view(np.uint16)[untouched], W.f32_to_bf16_bits(table[untouched]))


def test_bwd_update_stochastic_rounding_ignored_for_f32():
    d = 64
    F, B, rows, ids, offsets, table, G, rb, s0, s1 = _opt_case(11, d, "f32", "adagrad")
    b2t = np.arange(F, dtype=np.int32)
    st, dd = gpu_dedup(ids, offsets, F, B, b2t, rb)
    n = ids.size
    nu = torch.tensor([dd["n_unique"]], dtype=torch.int64, device=DEV)
    ro = torch.from_numpy(np.concatenate([dd["run_offsets"], np.zeros(n - dd["n_unique"], np.int32)])).to(DEV)
    outs = []
    for sr in (False, True):
        tab = _t(table)
        ws = ctr.workspace(ctr.ctr_bwd_update_workspace_size(n, d))
        o = ctr.optimizer(ctr.OPT_SGD, stochastic_rounding=sr, sr_seed=12345)
        ctr.ctr_embedding_bag_bwd_update_opt(_t(G), F * d, d, _t(offsets), F, B, ctr.POOL_SUM,
                                             _t(dd["unique_rows"]), nu, ro, _t(dd["sorted_bag"]), n, 2.0 ** -6, tab,
                                             d, None, ctr.BWD_ALL, o, ws)
        assert ctr.ctr_check_status(ws) == 0
        outs.append(_np(tab))
    np.testing.assert_array_equal(outs[0], outs[1])


# ---------------------------------------------------------------------------
# captured steps (CUDA graphs)
# ---------------------------------------------------------------------------
def _small_path(name, **kw):
    cfg = W.CONFIGS[name]
    if name == "full_step":
        cfg = cfg.shrink(batch=512, rows_per_table=tuple([20000] * 26))
    elif name == "tensornet":
        cfg = cfg.shrink(batch=1024, rows_per_table=(1 << 20,), ids=cfg.ids[:3] + (20,))
    w = W.make_workload(cfg)
    path = CtrPath(cfg, w["ids"].size, **kw)
    path.upload(w)
    return cfg, w, path


@pytest.mark.parametrize("name,opt", [("full_step", "sgd"), ("tensornet", "sgd"), ("full_step", "rowwise_adagrad")])
def test_captured_step_equals_eager_steps(name, opt):
    # two identical paths: one steps eagerly, the other replays a captured step;
    # after three steps every output, the table and the optimizer state agree bit for bit
    _, _, pe = _small_path(name, optimizer=opt)
    _, _, pg = _small_path(name, optimizer=opt)
    g = pg.capture()
    assert g.launches > 0
    for _ in range(3):
        pe.step()
        g.replay()
    torch.cuda.synchronize()
    assert pe.check_status() == pg.check_status() == {k: 0 for k in pe.check_status()}
    nu = int(pe.n_unique.item())
    assert nu == int(pg.n_unique.item())
    n = pe.n_ids
    defined = {"unique_rows": nu, "run_offsets": nu + 1, "inverse": n, "sorted_bag": n}  # capacity-sized buffers
    for attr in ("unique_rows", "inverse", "sorted_bag", "run_offsets", "X", "out", "pooled", "dX", "table", "state0"):
        a, b = getattr(pe, attr, None), getattr(pg, attr, None)
        if a is None:
            continue
        if attr in defined:
            a, b = a[:defined[attr]], b[:defined[attr]]
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), attr


def test_capture_refuses_step_dependent_values():
    _, _, p = _small_path("tensornet", optimizer="adam")
    with pytest.raises(ValueError):
        p.capture()
    base = W.CONFIGS["tensornet"]
    cfg = base.shrink(batch=256, dtype="bf16", table_init=("normal4", 0.01), rows_per_table=(1 << 20,),
                      ids=base.ids[:3] + (20,))
    w = W.make_workload(cfg)
    p = CtrPath(cfg, w["ids"].size, stochastic_rounding=True)
    with pytest.raises(ValueError):
        p.capture()


def test_host_pipeline_with_captured_steps_equals_eager():
    cfg = W.CONFIGS["full_step"].shrink(batch=512, rows_per_table=tuple([20000] * 26))
    w = W.make_workload(cfg)
    host = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in w.items()
            if k in ("ids", "offsets", "dense", "dout")}
    outs = {}
    for graphs in (False, True):
        path = CtrPath(cfg, w["ids"].size)
        path.upload(w)
        pipe = HostPipeline(path, graphs=graphs)
        res = [torch.empty(path.out.shape, dtype=path.out.dtype).pin_memory() for _ in range(4)]
        pipe.run([host] * 4, res)
        torch.cuda.synchronize()
        outs[graphs] = ([r.clone() for r in res], path.table.cpu())
    for a, b in zip(outs[False][0], outs[True][0]):
        assert torch.equal(a, b)
    assert torch.equal(outs[False][1], outs[True][1])


@pytest.mark.parametrize("name", ["dlrm_fp32", "full_step_b128"])
def test_embedding_bag_fwd_tma_gather_variant(name):
    # the TMA row-gather variant (fp32, d = 128), off by default: same bags, same
    # summation order as the default gather, so the same bits; and the oracle's values
    cfg = FWD_CASES[name]
    w = W.make_workload(cfg, with_grads=False)
    plain = _fwd_case(cfg, w)
    prev = ctr.ctr_set_tma_gather(True)
    try:
        got = _fwd_case(cfg, w)
    finally:
        ctr.ctr_set_tma_gather(prev)
    ref, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"],
                                   w["row_base"], cfg.d, pool=cfg.pool, dtype=cfg.dtype, gen=_gen(cfg),
                                   with_mag=True)
    f32_close(got, ref, mag, pool_depth(w["offsets"], cfg.num_fields, cfg.batch), what=f"TMA gather {name}")
    np.testing.assert_array_equal(got, plain)


def test_full_path_with_every_bag_empty():
    # zero IDs: the dedup finds no rows, the pooled vectors are zero, the
    # interaction sees only the dense vector, and no table row changes
    cfg = W.CONFIGS["full_step"].shrink(batch=64, rows_per_table=tuple([1000] * 26), bag_len=("fixed", 0))
    w = W.make_workload(cfg)
    assert w["ids"].size == 0
    path = CtrPath(cfg, 0)
    before = path.table.clone()
    path.upload(w)
    path.reset_status()
    path.step()
    torch.cuda.synchronize()
    assert all(v == 0 for v in path.check_status().values())
    assert int(path.n_unique.item()) == 0
    n, d = cfg.n_vectors, cfg.d
    X = np.concatenate([w["dense"][:, None, :], np.zeros((cfg.batch, n - 1, d), np.float32)], axis=1)
    ref, mag = O.dot_interaction(X, n, d, with_mag=True)
    f32_close(_np(path.out), ref, mag, d, what="interaction of empty bags")
    assert torch.equal(path.table, before)
