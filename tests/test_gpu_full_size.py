"""Parity at the full-step size, in the launch configuration the benchmark times.

Workload: B = 131072, 26 tables x 8M rows x d = 128 fp32 (106.5 GB), bag
lengths uniform 1..50, Zipf(1.05) IDs; one CtrPath.step() (dedup -> pooled
gather -> interaction -> interaction backward -> SGD row update).

* dedup: checked through properties that fix its outputs uniquely (ascending
  distinct keys, unique_rows[inverse] = key, the bags in the order of a stable
  host sort of the keys, run bounds, per-table offsets), all vectorised over
  the 86.9M IDs;
* pooled rows, interaction outputs and interaction gradients: on sampled bags
  and samples, recomputed by the oracle from the generator's table values;
* row updates: on sampled rows the batch touches only a few times, whose
  gradient the oracle can rebuild from the few samples that contain them; and
  on sampled rows the batch does not touch (unchanged bits).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import workload as W
from sparse_embeddings_feature_gb300.pipeline import CtrPath

from _tol import f32_close

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


def _oracle_X(cfg, w, samples):
    """Oracle interaction input [len(samples), 27, 128] for the listed samples."""
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    bags = (np.arange(F)[None, :] * B + np.asarray(samples)[:, None]).ravel()
    pooled = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen,
                                 bag_list=bags)
    return np.concatenate([w["dense"][samples][:, None, :], pooled.reshape(len(samples), F, d)], axis=1)


def test_full_size_forward_interaction_and_backward_on_samples(full_step):
    cfg, w, path = full_step
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    rng = np.random.default_rng(77)
    samples = np.sort(rng.choice(B, size=300, replace=False))
    samples[-1] = B - 1                                              # include the ragged end
    X = _oracle_X(cfg, w, samples)
    sel = torch.from_numpy(samples).cuda()
    f32_close(_np(path.X[sel]), X, None, 0, atol=2e-6, what="pooled rows")
    out_ref, out_mag = O.dot_interaction(X, n, d, with_mag=True)
    f32_close(_np(path.out[sel]), out_ref, out_mag, d + 64, what="interaction")
    dX_ref, dX_mag = O.dot_interaction_bwd(w["dout"][samples], X, n, d, with_mag=True)
    f32_close(_np(path.dX[sel]), dX_ref, dX_mag, n + 64, what="interaction bwd")


def test_full_size_row_updates_on_sampled_rows(full_step):
    cfg, w, path = full_step
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    nu = int(path.n_unique.item())
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    run_len = np.diff(ro)
    rng = np.random.default_rng(5)
    cold = np.nonzero(run_len <= 3)[0]
    picks = np.sort(rng.choice(cold, size=40, replace=False))
    uq = _np(path.unique_rows[:nu])
    rows = uq[picks]
    sbag = _np(path.sorted_bag)
    # the samples whose bags hold the picked rows (the dedup is checked above)
    occ_bags = np.concatenate([sbag[ro[u]:ro[u + 1]] for u in picks]).astype(np.int64)
    samples = np.unique(occ_bags % B)
    X = _oracle_X(cfg, w, samples)
    dX = O.dot_interaction_bwd(w["dout"][samples], X, n, d)
    # gradient of the pooled outputs, scattered back to a [B, F, d] view over the needed samples only
    G = np.zeros((B, F, d), dtype=np.float32)
    G[samples] = dX[:, 1:, :]
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    new_ref, _, mag = O.embedding_bag_bwd_update(G, w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"],
                                                 d, cfg.lr, rows, gen=gen)
    got = _np(path.table[torch.from_numpy(rows).cuda()])
    old = O.table_rows(gen[0], gen[1], gen[2], d, rows)
    f32_close(got, new_ref, cfg.lr * mag + np.abs(old), 200, what="updated cold rows")
    # rows no bag touches keep their bits
    probe = rng.integers(0, cfg.total_rows, size=4000)
    probe = np.setdiff1d(probe, uq)
    got = _np(path.table[torch.from_numpy(probe).cuda()])
    np.testing.assert_array_equal(got, O.table_rows(gen[0], gen[1], gen[2], d, probe))
