"""Parity at the full-step size, in the launch configuration the benchmark times.

Workload: B = 131072, 26 tables x 8M rows x d = 128 fp32 (106.5 GB), bag
lengths uniform 1..50, Zipf(1.05) IDs; one CtrPath.step() (dedup -> pooled
gather -> interaction -> interaction backward -> SGD row update).

* dedup: checked through properties that fix its outputs uniquely (ascending
  distinct keys, unique_rows[inverse] = key, the bags in the order of a stable
  host sort of the keys, run bounds, per-table offsets), all vectorised over
  the 86.9M IDs;
* pooled rows: on sampled samples, recomputed by the oracle from the
  generator's table values;
* interaction outputs and gradients: the oracle applied to the GPU's own
  interaction input (checked just before), so each step is checked on its
  real input with the bound of its own reduction depth;
* row updates: on the 20 hottest rows (the Zipf head) and 2000 random unique
  rows, with the oracle summing the GPU's own pooled gradient over every
  occurrence of the batch; and on sampled rows the batch does not touch
  (unchanged bits).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import workload as W
from sparse_embeddings_feature_gb300.pipeline import CtrPath

from _tol import bwd_depth, f32_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def full_step():
    cfg = W.CONFIGS["full_step"]
    w = W.make_workload(cfg)
    path = CtrPath(cfg, w["ids"].size)
    path.upload(w)
    path.reset_status()
    path.step()
    torch.cuda.synchronize()
    status = path.check_status()
    assert all(v == 0 for v in status.values()), status
    yield cfg, w, path
    del path
    torch.cuda.empty_cache()


def _np(t):
    return t.cpu().numpy()


def test_full_size_dedup_properties(full_step):
    cfg, w, path = full_step
    F, B = cfg.num_fields, cfg.batch
    n = w["ids"].size
    lens = np.diff(w["offsets"])
    bag_of = np.repeat(np.arange(F * B, dtype=np.int64), lens)
    keys = cfg.row_base[np.asarray(cfg.field_to_table)[bag_of // B]] + w["ids"]
    nu = int(path.n_unique.item())
    uq = _np(path.unique_rows[:nu])
    inv = _np(path.inverse[:n]).astype(np.int64)
    sbag = _np(path.sorted_bag[:n]).astype(np.int64)
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    uo = _np(path.unique_offsets)
    assert path.sorted_pos is None                                   # the step skips the permutation
    assert np.all(np.diff(uq) > 0)                                   # distinct, ascending
    assert nu == np.unique(keys).size
    np.testing.assert_array_equal(uq[inv], keys)                     # unique_rows[inverse[i]] = key[i]
    sp = np.argsort(keys, kind="stable")                             # the stable sort, on the host
    np.testing.assert_array_equal(sbag, bag_of[sp])                  # bags grouped by key, in stable order
    ks = keys[sp]
    assert ro[0] == 0 and ro[-1] == n
    np.testing.assert_array_equal(ks[ro[:-1]], uq)                   # runs start at each distinct key
    np.testing.assert_array_equal(np.diff(ro), np.bincount(inv, minlength=nu))
    np.testing.assert_array_equal(uo, np.searchsorted(uq, cfg.row_base, side="left"))


def _oracle_pooled(cfg, w, samples):
    """Oracle pooled rows [len(samples), F, d], their magnitude sums and bag lengths."""
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    bags = (np.arange(F)[None, :] * B + np.asarray(samples)[:, None]).ravel()
    pooled, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen,
                                      bag_list=bags, with_mag=True)
    lens = np.diff(w["offsets"])[bags]
    shape = (len(samples), F, d)
    return pooled.reshape(shape), mag.reshape(shape), lens.reshape(len(samples), F, 1)


def test_full_size_forward_interaction_and_backward_on_samples(full_step):
    cfg, w, path = full_step
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    rng = np.random.default_rng(77)
    samples = np.sort(rng.choice(B, size=300, replace=False))
    samples[-1] = B - 1                                              # include the ragged end
    pooled, pmag, lens = _oracle_pooled(cfg, w, samples)
    sel = torch.from_numpy(samples).cuda()
    Xg = _np(path.X[sel])
    np.testing.assert_array_equal(Xg[:, 0, :], w["dense"][samples])  # slot 0: the dense vector, copied
    # a bag of L rows is a sum of L terms: depth L in any summation order
    f32_close(Xg[:, 1:, :], pooled, pmag, lens, what="pooled rows")
    # each later step is checked on its real input, the GPU's own X (checked just above)
    out_ref, out_mag = O.dot_interaction(Xg, n, d, with_mag=True)
    np.testing.assert_array_equal(_np(path.out[sel])[:, :d], w["dense"][samples])
    f32_close(_np(path.out[sel]), out_ref, out_mag, d, what="interaction")  # a d-term dot product
    dX_ref, dX_mag = O.dot_interaction_bwd(w["dout"][samples], Xg, n, d, with_mag=True)
    # dx_i: n - 1 products, plus the pass-through gradient added to the dense slot
    f32_close(_np(path.dX[sel]), dX_ref, dX_mag, n, what="interaction bwd")


def test_full_size_row_updates_on_hot_and_sampled_rows(full_step):
    """The row update at the real skew: the 20 longest runs (the Zipf head, about
    0.29 M occurrences each, summed by the long-run pieces and the combine) and
    2000 random unique rows, from the GPU's own pooled gradient dX[:, 1:, :]
    (the interaction backward is checked on its own above)."""
    cfg, w, path = full_step
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    nu = int(path.n_unique.item())
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    run_len = np.diff(ro)
    rng = np.random.default_rng(5)
    hot = np.argsort(run_len, kind="stable")[-20:]
    picks = np.unique(np.concatenate([hot, rng.choice(nu, size=2000, replace=False)]))
    assert run_len[hot].min() > 100_000                              # the long-run path, many pieces
    uq = _np(path.unique_rows[:nu])
    rows = uq[picks]
    G = _np(path.dX[:, 1:, :])                                       # [B, F, d], as the update reads it
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    new_ref, _, mag = O.embedding_bag_bwd_update(G, w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"],
                                                 d, cfg.lr, rows, gen=gen)
    del G
    got = _np(path.table[torch.from_numpy(rows).cuda()])
    old = O.table_rows(gen[0], gen[1], gen[2], d, rows)
    depth = bwd_depth(run_len[picks])[:, None] + 2                   # + the product lr * g and the subtraction
    f32_close(got, new_ref, cfg.lr * mag + np.abs(old), depth, what="updated rows (hot and sampled)")
    # rows no bag touches keep their bits
    probe = rng.integers(0, cfg.total_rows, size=4000)
    probe = np.setdiff1d(probe, uq)
    got = _np(path.table[torch.from_numpy(probe).cuda()])
    np.testing.assert_array_equal(got, O.table_rows(gen[0], gen[1], gen[2], d, probe))
