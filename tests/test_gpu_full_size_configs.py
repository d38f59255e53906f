"""Parity at full size for the bf16 large-batch workload and the TensorNet-style
workload, each run as one CtrPath.step() (the launch configuration
`bench.py --workload bf16_large` and `--workload tensornet` time).

bf16_large: B = 65536, 26 tables x 4M rows x d = 64 bf16, bag lengths
Poisson(30) clipped to 1..100, Zipf(1.2) IDs, mean pooling, tensor-core pair
dots.  Pooled rows and interaction outputs are checked on sampled samples
against the oracle (which regenerates the table rows it needs).

tensornet: B = 16384, 100 fields sharing one table of 2^26 rows x d = 32 fp32,
1..10 IDs per field, hashed Zipf(1.1) IDs.  The dedup is checked through the
properties that fix it uniquely, the unique-row matrix bit for bit on sampled
rows, pooled rows on sampled bags, and updated rows (hot and cold) on sampled
unique rows, whose gradient the oracle rebuilds from the full upstream gradient.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import workload as W
from sparse_embeddings_feature_gb300.pipeline import CtrPath

from _tol import bf16_close, bwd_depth, f32_close

pytestmark = pytest.mark.gpu


def _np(t):
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _run(name):
    cfg = W.CONFIGS[name]
    w = W.make_workload(cfg)
    path = CtrPath(cfg, w["ids"].size)
    path.upload(w)
    path.reset_status()
    path.step()
    torch.cuda.synchronize()
    status = path.check_status()
    assert all(v == 0 for v in status.values()), status
    return cfg, w, path


@pytest.fixture(scope="module")
def bf16_large():
    cfg, w, path = _run("bf16_large")
    yield cfg, w, path
    del path
    torch.cuda.empty_cache()


def test_bf16_large_pooled_and_interaction_on_samples(bf16_large):
    cfg, w, path = bf16_large
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    rng = np.random.default_rng(31)
    samples = np.sort(rng.choice(B, size=400, replace=False))
    samples[0], samples[-1] = 0, B - 1
    bags = (np.arange(F)[None, :] * B + samples[:, None]).ravel()
    pooled, pmag = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d,
                                       pool="mean", dtype="bf16", gen=gen, bag_list=bags, with_mag=True)
    sel = torch.from_numpy(samples).cuda()
    X_gpu = _np(path.X[sel])
    depth = (np.diff(w["offsets"])[bags] + 1)[:, None]                # L terms, then the mean's division
    bf16_close(X_gpu[:, 1:, :].reshape(-1, d), pooled, pmag, depth, atol=1e-5, what="pooled (mean, bf16)")
    np.testing.assert_array_equal(X_gpu[:, 0, :], w["dense"][samples].view(np.uint16))
    # the interaction is checked on its real input, the GPU's own (checked) X: each pair is a
    # d-term fp32 dot rounded once to bf16
    out_ref, out_mag = O.dot_interaction(X_gpu, n, d, dtype="bf16", with_mag=True)
    got = _np(path.out[sel])
    np.testing.assert_array_equal(got[:, :d], out_ref[:, :d])
    bf16_close(got[:, d:], out_ref[:, d:], out_mag[:, d:], d, what="interaction (bf16, tensor cores)")


@pytest.fixture(scope="module")
def tensornet():
    cfg, w, path = _run("tensornet")
    yield cfg, w, path
    del path
    torch.cuda.empty_cache()


def test_tensornet_dedup_properties(tensornet):
    cfg, w, path = tensornet
    F, B = cfg.num_fields, cfg.batch
    n = w["ids"].size
    lens = np.diff(w["offsets"])
    bag_of = np.repeat(np.arange(F * B, dtype=np.int64), lens)
    keys = w["ids"]                                                  # one table, row_base 0
    nu = int(path.n_unique.item())
    uq = _np(path.unique_rows[:nu])
    inv = _np(path.inverse[:n]).astype(np.int64)
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    np.testing.assert_array_equal(uq, np.unique(keys))
    np.testing.assert_array_equal(uq[inv], keys)
    sp = np.argsort(keys, kind="stable")
    np.testing.assert_array_equal(_np(path.sorted_bag[:n]).astype(np.int64), bag_of[sp])
    ks = keys[sp]
    np.testing.assert_array_equal(ks[ro[:-1]], uq)
    np.testing.assert_array_equal(np.diff(ro), np.bincount(inv, minlength=nu))
    np.testing.assert_array_equal(_np(path.unique_offsets), [0, nu])


def test_tensornet_unique_matrix_and_pooled_on_samples(tensornet):
    cfg, w, path = tensornet
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    rng = np.random.default_rng(41)
    nu = int(path.n_unique.item())
    pick = np.sort(rng.choice(nu, size=5000, replace=False))
    pick[-1] = nu - 1
    uq = _np(path.unique_rows[:nu])
    # the batch matrix holds the rows as they were before this step's update
    np.testing.assert_array_equal(_np(path.U[torch.from_numpy(pick).cuda()]),
                                  O.table_rows(gen[0], gen[1], gen[2], d, uq[pick]))
    bags = np.sort(rng.choice(F * B, size=3000, replace=False))
    bags[-1] = F * B - 1
    ref, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen,
                                   bag_list=bags, with_mag=True)
    got = _np(path.pooled).reshape(B * F, d)
    # pooled[b, f] holds bag f * B + b
    f_, b_ = bags // B, bags % B
    f32_close(got[b_ * F + f_], ref, mag, np.diff(w["offsets"])[bags][:, None], what="pooled from the unique-row matrix")


def test_tensornet_row_updates_on_sampled_rows(tensornet):
    cfg, w, path = tensornet
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    nu = int(path.n_unique.item())
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    run_len = np.diff(ro)
    rng = np.random.default_rng(43)
    hot = np.argsort(run_len)[-20:]                                  # the longest runs (split into pieces)
    pick = np.unique(np.concatenate([hot, rng.choice(nu, size=2000, replace=False)]))
    rows = _np(path.unique_rows[:nu])[pick]
    new_ref, _, mag = O.embedding_bag_bwd_update(w["grad_pooled"], w["ids"], w["offsets"], F, B, w["bag_to_table"],
                                                 w["row_base"], d, cfg.lr, rows, gen=gen)
    got = _np(path.table[torch.from_numpy(rows).cuda()])
    old = O.table_rows(gen[0], gen[1], gen[2], d, rows)
    depth = bwd_depth(run_len[pick])[:, None] + 2                     # + the product lr * g and the subtraction
    f32_close(got, new_ref, cfg.lr * mag + np.abs(old), depth, what="updated rows")
    probe = np.setdiff1d(rng.integers(0, cfg.total_rows, size=4000), _np(path.unique_rows[:nu]))
    np.testing.assert_array_equal(_np(path.table[torch.from_numpy(probe).cuda()]),
                                  O.table_rows(gen[0], gen[1], gen[2], d, probe))
