"""Parity at full size for the path's options, each run as one CtrPath.step()
with the options `bench.py` takes for them:

* the full step (B = 131072, 26 tables x 8M rows x d = 128 fp32) with the FM
  term, the full Gram-matrix interaction and row-wise Adagrad
  (`--fm --interaction-mode full --optimizer rowwise_adagrad`): FM terms on
  sampled bags, the interaction and its gradient on sampled samples, updated
  rows and their state on sampled rows that occur a few times;
* the TensorNet-style workload (B = 16384, 100 fields, one 2^26-row table,
  d = 32) with bf16 tables, Adam and stochastic rounding
  (`--dtype bf16 --optimizer adam --stochastic-rounding`): updated rows (the
  longest runs and random ones) and Adam's state on sampled unique rows.

The oracle rebuilds each sampled row's exact gradient; the GPU's fp32 gradient
differs from it by at most e = gamma_k * (sum of |terms|), and the tolerances
push e through each rule's arithmetic (derivatives below), plus the rule's own
fp32 rounding.
"""
import gc

import numpy as np
import pytest
import torch

from oracle import oracle as O
from sparse_embeddings_feature_gb300 import workload as W
from sparse_embeddings_feature_gb300.pipeline import CtrPath

from _tol import bwd_depth, f32_close, fm_depth, gamma

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def _np(t):
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _run(cfg, **kw):
    gc.collect()                    # another module's full-size path must be gone first
    torch.cuda.empty_cache()
    w = W.make_workload(cfg)
    path = CtrPath(cfg, w["ids"].size, **kw)
    path.upload(w)
    path.reset_status()
    path.step()
    torch.cuda.synchronize()
    status = path.check_status()
    assert all(v == 0 for v in status.values()), status
    return w, path


@pytest.fixture(scope="module")
def full_opts():
    cfg = W.CONFIGS["full_step"].shrink(interaction_mode="full")
    w, path = _run(cfg, fm=True, optimizer="rowwise_adagrad")
    yield cfg, w, path
    del path
    torch.cuda.empty_cache()


def _checked_X(cfg, w, path, samples):
    """The GPU's interaction input for the listed samples, after checking its pooled
    slots against the oracle (depth: each bag's length) and its dense slot bit for bit."""
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    bags = (np.arange(F)[None, :] * B + np.asarray(samples)[:, None]).ravel()
    pooled, mag = O.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen,
                                      bag_list=bags, with_mag=True)
    Xg = _np(path.X[torch.from_numpy(np.asarray(samples)).cuda()])
    np.testing.assert_array_equal(Xg[:, 0, :], w["dense"][samples])
    lens = np.diff(w["offsets"])[bags].reshape(len(samples), F, 1)
    shape = (len(samples), F, d)
    f32_close(Xg[:, 1:, :], pooled.reshape(shape), mag.reshape(shape), lens, what="pooled rows")
    return Xg


def test_full_step_fm_term_on_sampled_bags(full_opts):
    cfg, w, path = full_opts
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    rng = np.random.default_rng(91)
    bags = np.sort(rng.choice(F * B, size=3000, replace=False))
    bags[-1] = F * B - 1
    ref, mag = O.bag_fm(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen, bag_list=bags,
                        with_mag=True)
    # 1/2 (|sum v|^2 - sum |v|^2) in fp32: bounded by the depth times both terms' magnitudes
    lens = np.diff(w["offsets"])[bags]
    sq = np.array([(O.table_rows(gen[0], gen[1], gen[2], d, cfg.row_base[w["bag_to_table"][b // B]] +
                                 w["ids"][w["offsets"][b]:w["offsets"][b + 1]]).astype(np.float64) ** 2).sum()
                   for b in bags])
    f32_close(_np(path.fm)[bags], ref, 2.0 * mag + sq, fm_depth(lens, d), what="FM term")


def test_full_step_full_gram_interaction_on_samples(full_opts):
    cfg, w, path = full_opts
    B, d, n = cfg.batch, cfg.d, cfg.n_vectors
    rng = np.random.default_rng(92)
    samples = np.sort(rng.choice(B, size=200, replace=False))
    samples[-1] = B - 1
    X = _checked_X(cfg, w, path, samples)
    sel = torch.from_numpy(samples).cuda()
    # the oracle takes the GPU's own (checked) input: each product is a d-term dot
    out_ref, out_mag = O.dot_interaction_mode(X, n, d, "full", with_mag=True)
    got = _np(path.out[sel])
    assert got.shape == (len(samples), n * n)
    f32_close(got, out_ref, out_mag, d, what="full Gram interaction")
    g = got.reshape(len(samples), n, n)
    np.testing.assert_array_equal(g, np.transpose(g, (0, 2, 1)))        # one product, stored twice
    dX_ref, dX_mag = O.dot_interaction_bwd_mode(w["dout"][samples], X, n, d, "full", with_mag=True)
    # dx_i sums 2n products (<x_i, x_j> and <x_j, x_i> apart)
    f32_close(_np(path.dX[sel]), dX_ref, dX_mag, 2 * n + 1, what="full Gram interaction bwd")


def test_full_step_rowwise_adagrad_on_sampled_rows(full_opts):
    cfg, w, path = full_opts
    F, B, d, n = cfg.num_fields, cfg.batch, cfg.d, cfg.n_vectors
    nu = int(path.n_unique.item())
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    run_len = np.diff(ro)
    rng = np.random.default_rng(93)
    # the 20 hottest rows (long runs: pieces and combine) and 200 random ones
    picks = np.unique(np.concatenate([np.argsort(run_len, kind="stable")[-20:], rng.choice(nu, size=200,
                                                                                          replace=False)]))
    rows = _np(path.unique_rows[:nu])[picks]
    # the update's real input: the GPU's pooled gradient (the interaction backward is checked above)
    G = _np(path.dX[:, 1:, :])
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    _, g, mag = O.embedding_bag_bwd_update(G, w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d,
                                           cfg.lr, rows, gen=gen)
    del G
    # gradient error: the fp32 reduction of each run (its own depth)
    e = gamma(bwd_depth(run_len[picks]))[:, None] * mag + 1e-30
    w_old = O.table_rows(gen[0], gen[1], gen[2], d, rows).astype(np.float64)
    s0 = np.zeros(len(rows), dtype=np.float32)
    # the oracle takes the hyperparameters as the C-ABI receives them: fp32 values
    eps = float(np.float32(path.eps))
    w_ref, s_ref, _ = O.optimizer_step("rowwise_adagrad", w_old, g, float(np.float32(cfg.lr)), state0=s0, eps=eps)
    # s = mean_c g_c^2: ds <= (1/d) sum_c (2|g_c| e_c + e_c^2); the step lr g_c / (sqrt(s) + eps)
    # moves by lr (e_c / (sqrt(s) + eps) + |g_c| ds / (2 sqrt(s_lo) (sqrt(s_lo) + eps)^2))
    s = s_ref.astype(np.float64)
    ds = (2 * np.abs(g) * e + e * e).mean(axis=1) + 4 * U * s
    s_lo = np.maximum(s - ds, 0.0)
    r_lo = np.sqrt(s_lo)[:, None] + eps
    dstep = cfg.lr * (e / r_lo + np.abs(g) * ds[:, None] / (2 * np.maximum(np.sqrt(s_lo), 1e-30)[:, None] * r_lo ** 2))
    step = cfg.lr * np.abs(g) / r_lo
    tol = np.minimum(dstep, 2 * step) + 8 * U * step + 2 * U * np.abs(w_ref.astype(np.float64)) + 1e-30
    got = _np(path.table[torch.from_numpy(rows).cuda()]).astype(np.float64)
    err = np.abs(got - w_ref.astype(np.float64))
    assert np.all(err <= tol), float((err - tol).max())
    got_s = _np(path.state0[torch.from_numpy(rows).cuda()]).astype(np.float64)
    assert np.all(np.abs(got_s - s) <= ds + 1e-30)
    # rows the batch does not touch keep their values and a zero state
    probe = np.setdiff1d(rng.integers(0, cfg.total_rows, size=4000), _np(path.unique_rows[:nu]))
    pt = torch.from_numpy(probe).cuda()
    np.testing.assert_array_equal(_np(path.table[pt]), O.table_rows(gen[0], gen[1], gen[2], d, probe))
    assert not np.any(_np(path.state0[pt]))


@pytest.fixture(scope="module")
def tensornet_bf16_adam_sr():
    base = W.CONFIGS["tensornet"]
    cfg = base.shrink(dtype="bf16", table_init=("normal4", base.table_init[1]))
    w, path = _run(cfg, optimizer="adam", stochastic_rounding=True)
    yield cfg, w, path
    del path
    torch.cuda.empty_cache()


def _bf16_ulp(v):
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def test_tensornet_bf16_adam_stochastic_rounding_on_sampled_rows(tensornet_bf16_adam_sr):
    cfg, w, path = tensornet_bf16_adam_sr
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    gen = (cfg.fill_kind, cfg.fill_seed, cfg.fill_scale)
    nu = int(path.n_unique.item())
    ro = _np(path.run_offsets[:nu + 1]).astype(np.int64)
    run_len = np.diff(ro)
    rng = np.random.default_rng(94)
    pick = np.unique(np.concatenate([np.argsort(run_len)[-20:], rng.choice(nu, size=2000, replace=False)]))
    rows = _np(path.unique_rows[:nu])[pick]
    _, g, mag = O.embedding_bag_bwd_update(w["grad_pooled"], w["ids"], w["offsets"], F, B, w["bag_to_table"],
                                           w["row_base"], d, cfg.lr, rows, dtype="bf16", gen=gen)
    e = gamma(bwd_depth(run_len[pick]))[:, None] * mag + 1e-30
    w_old = W.bf16_bits_to_f32(O.table_rows(gen[0], gen[1], gen[2], d, rows)).astype(np.float64)
    z = np.zeros((len(rows), d), dtype=np.float32)
    # the oracle takes the hyperparameters as the C-ABI receives them: fp32 values (0.9 is not one)
    b1, b2 = (float(np.float32(b)) for b in path.betas)
    eps = float(np.float32(path.eps))
    w_ref, m_ref, v_ref = O.optimizer_step("adam", w_old, g, float(np.float32(cfg.lr)), state0=z, state1=z, eps=eps, beta1=b1,
                                           beta2=b2, step=1, dtype="bf16", sr_seed=path.last_sr_seed, rows=rows)
    # step 1 from zero state: the update is lr g / (|g| + eps), whose derivative in g is
    # lr eps / (|g| + eps)^2; fp32 rounding of m, v, the corrections and the quotient adds ~8u lr
    ag = np.abs(g)
    dx = cfg.lr * (e * eps / np.maximum(ag - e + eps, eps) ** 2 + 8 * U) + U * (np.abs(w_old) + cfg.lr)
    got = W.bf16_bits_to_f32(_np(path.table[torch.from_numpy(rows).cuda()])).astype(np.float64)
    ref = W.bf16_bits_to_f32(w_ref).astype(np.float64)
    # the same random bits: the results agree unless the fp32 and fp64 values straddle the
    # rounding threshold, and then they are neighbouring bf16 values
    assert np.all(np.abs(got - ref) <= _bf16_ulp(np.maximum(np.abs(got), np.abs(ref))) + 1e-300)
    straddle_room = np.mean(dx / _bf16_ulp(np.abs(ref)))  # expected share of flipped decisions
    assert np.mean(got != ref) <= 4 * straddle_room + 0.002
    # stochastic, not nearest: values off the bf16 grid round both ways
    x_rn, _, _ = O.optimizer_step("adam", w_old, g, float(np.float32(cfg.lr)), state0=z, state1=z, eps=eps, beta1=b1, beta2=b2,
                                  step=1, dtype="bf16")
    assert np.mean(W.bf16_bits_to_f32(x_rn) != got) > 0.05
    # Adam's state: m = (1 - b1) g, v = (1 - b2) g^2 (fp32)
    rt = torch.from_numpy(rows).cuda()
    got_m = _np(path.state0[rt]).astype(np.float64)
    got_v = _np(path.state1[rt]).astype(np.float64)
    assert np.all(np.abs(got_m - m_ref) <= (1 - b1) * e + 2 * U * np.abs(m_ref) + 1e-30)
    assert np.all(np.abs(got_v - v_ref) <= (1 - b2) * (2 * ag * e + e * e) + 4 * U * np.abs(v_ref) + 1e-30)
