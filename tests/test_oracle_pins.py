"""Pins of the CPU oracle to facts other than itself (CPU only, seconds).

Each test checks one oracle function against something the pages or the
mathematics fix: a closed form (the FM squared-norm identity), a library routine
that reaches the same definition (numpy.unique, a scipy CSR product, a numpy
Gram matrix, torch autograd), brute force in exact arithmetic on tiny inputs,
or an invariant.  The cases are chosen so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from sparse_embeddings_feature_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _csr(bags):
    lens = np.array([len(b) for b in bags], dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ids = np.array([i for b in bags for i in b], dtype=np.int64)
    return ids, offsets


def _small_case(seed=7, F=3, B=5, rows=(9, 4, 7), d=6, max_len=6, empty=True):
    rng = np.random.default_rng(seed)
    bags = []
    for f in range(F):
        for _ in range(B):
            L = int(rng.integers(0 if empty else 1, max_len + 1))
            bags.append(list(rng.integers(0, rows[f], size=L)))
    ids, offsets = _csr(bags)
    rb = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    return bags, ids, offsets, np.arange(F, dtype=np.int32), rb


# ---------------------------------------------------------------------------
# dedup
# ---------------------------------------------------------------------------
def test_dedup_golden_bruteforce(oracle):
    g = _golden("tensornet_dedup_small.json")
    F, B = g["num_fields"], g["batch"]
    bags = g["bags_field_major"]
    ids, offsets = _csr(bags)
    rb = np.concatenate([[0], np.cumsum(g["rows_per_table"])]).astype(np.int64)
    r = oracle.dedup(ids, offsets, F, B, g["bag_to_table"], rb)
    # brute force: global key per occurrence, then distinct keys in ascending order
    keys, bag_of = [], []
    for bag, content in enumerate(bags):
        t = g["bag_to_table"][bag // B]
        for i in content:
            keys.append(int(rb[t]) + i)
            bag_of.append(bag)
    distinct = sorted(set(keys))
    assert list(r["unique_rows"]) == distinct
    assert r["n_unique"] == len(distinct)
    assert list(r["inverse"]) == [distinct.index(k) for k in keys]
    order = sorted(range(len(keys)), key=lambda i: (keys[i], i))
    assert list(r["sorted_pos"]) == order
    assert list(r["sorted_bag"]) == [bag_of[i] for i in order]
    runs = [0] + [s for s in range(1, len(order)) if keys[order[s]] != keys[order[s - 1]]] + [len(order)]
    assert list(r["run_offsets"]) == runs
    assert list(r["unique_offsets"]) == [sum(1 for k in distinct if k < int(b)) for b in rb]
    # raw ID 3 occurs in table 0 and raw ID 5 in table 1: each keeps its own key
    assert 3 in distinct and int(rb[1]) + 5 in distinct


@pytest.mark.parametrize("name", ["tiny", "dlrm_fp32"])
def test_dedup_matches_numpy_unique(oracle, name):
    cfg = W.CONFIGS[name]
    w = W.make_workload(cfg, with_grads=False)
    F, B = cfg.num_fields, cfg.batch
    r = oracle.dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    lens = np.diff(w["offsets"])
    bag_of = np.repeat(np.arange(F * B), lens)
    keys = w["row_base"][w["bag_to_table"][bag_of // B]] + w["ids"]
    u, inv, cnt = np.unique(keys, return_inverse=True, return_counts=True)
    np.testing.assert_array_equal(r["unique_rows"], u)
    np.testing.assert_array_equal(r["inverse"], inv)
    order = np.argsort(keys, kind="stable")
    np.testing.assert_array_equal(r["sorted_pos"], order)
    np.testing.assert_array_equal(r["sorted_bag"], bag_of[order])
    np.testing.assert_array_equal(r["run_offsets"], np.concatenate([[0], np.cumsum(cnt)]))
    np.testing.assert_array_equal(r["unique_offsets"], np.searchsorted(u, w["row_base"], side="left"))


def test_dedup_hashed_single_table_invariants(oracle):
    cfg = W.CONFIGS["tensornet"].shrink(batch=256)
    w = W.make_workload(cfg, with_grads=False)
    r = oracle.dedup(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"], w["row_base"])
    uq, inv = r["unique_rows"], r["inverse"]
    assert np.all(np.diff(uq) > 0)
    np.testing.assert_array_equal(uq[inv], w["ids"])           # unique_rows[inverse[i]] == key[i]
    assert r["run_offsets"][-1] == w["ids"].size               # run lengths sum to n_ids
    # stability: inside a run, positions increase
    sp = r["sorted_pos"]
    ro = r["run_offsets"]
    run_id = np.repeat(np.arange(r["n_unique"]), np.diff(ro))
    same = run_id[1:] == run_id[:-1]
    assert np.all(sp[1:][same] > sp[:-1][same])


def test_dedup_rejects_out_of_range(oracle):
    ids, offsets = _csr([[0, 5], [1]])
    with pytest.raises(oracle.OracleError):
        oracle.dedup(ids, offsets, 1, 2, [0], np.array([0, 5]))


# ---------------------------------------------------------------------------
# pooled embedding bag
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_pooling_equals_count_matrix_times_table(oracle, pool):
    import scipy.sparse as sp
    bags, ids, offsets, b2t, rb = _small_case(seed=11, F=3, B=7, rows=(50, 20, 33), d=9, max_len=12)
    F, B, d = 3, 7, 9
    rng = np.random.default_rng(3)
    table = rng.uniform(-1, 1, size=(int(rb[-1]), d)).astype(np.float32)
    out = oracle.embedding_bag_fwd(ids, offsets, F, B, b2t, rb, d, pool=pool, table=table)
    lens = np.diff(offsets)
    bag_of = np.repeat(np.arange(F * B), lens)
    keys = rb[b2t[bag_of // B]] + ids
    A = sp.csr_matrix((np.ones(ids.size), (bag_of, keys)), shape=(F * B, int(rb[-1])))  # counts duplicates
    ref = A @ table.astype(np.float64)
    if pool == "mean":
        ref = ref / np.maximum(lens, 1)[:, None]
    ref = ref.reshape(F, B, d).transpose(1, 0, 2)
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)
    # empty bags give zero in both modes
    for bag in np.nonzero(lens == 0)[0]:
        assert np.all(out[bag % B, bag // B] == 0)


def test_pooling_bruteforce_exact(oracle):
    # integer-valued table: every sum is exact, so the comparison is bit for bit
    bags, ids, offsets, b2t, rb = _small_case(seed=5, F=2, B=4, rows=(8, 5), d=3, max_len=5)
    F, B, d = 2, 4, 3
    table = (np.arange(int(rb[-1]) * d, dtype=np.float32).reshape(-1, d) % 13) - 6
    out = oracle.embedding_bag_fwd(ids, offsets, F, B, b2t, rb, d, table=table)
    for f in range(F):
        for b in range(B):
            acc = [0] * d
            for i in bags[f * B + b]:
                for c in range(d):
                    acc[c] += int(table[int(rb[f]) + int(i), c])
            assert list(out[b, f]) == acc


def test_pooling_one_id_per_bag_is_row_copy(oracle):
    cfg = W.CONFIGS["tiny"]
    w = W.make_workload(cfg)
    gen = (oracle.GEN_UNIFORM, cfg.fill_seed, cfg.fill_scale)
    out = oracle.embedding_bag_fwd(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"],
                                   w["row_base"], cfg.d, gen=gen)
    keys = w["row_base"][np.repeat(w["bag_to_table"], cfg.batch)] + w["ids"]
    rows = oracle.table_rows(oracle.GEN_UNIFORM, cfg.fill_seed, cfg.fill_scale, cfg.d, keys)
    np.testing.assert_array_equal(out.transpose(1, 0, 2).reshape(-1, cfg.d), rows)


def test_dedup_then_gather_equals_direct_gather(oracle):
    # TensorNet: the batch-sized matrix of unique rows, indexed by the virtual
    # sparse feature, replaces the full table
    cfg = W.CONFIGS["tensornet"].shrink(batch=64)
    w = W.make_workload(cfg, with_grads=False)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    r = oracle.dedup(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"])
    gen = (oracle.GEN_UNIFORM, cfg.fill_seed, cfg.fill_scale)
    U = oracle.table_rows(gen[0], gen[1], gen[2], d, r["unique_rows"])
    via_u = oracle.embedding_bag_fwd(r["inverse"].astype(np.int64), w["offsets"], F, B, np.zeros(F, np.int32),
                                     np.array([0, r["n_unique"]]), d, table=U)
    direct = oracle.embedding_bag_fwd(w["ids"], w["offsets"], F, B, w["bag_to_table"], w["row_base"], d, gen=gen)
    np.testing.assert_array_equal(via_u, direct)


def test_mean_of_bf16_table_rounds_once(oracle):
    cfg = W.CONFIGS["bf16_large"].shrink(batch=8, rows_per_table=tuple([1000] * 26))
    w = W.make_workload(cfg, with_grads=False)
    gen = (oracle.GEN_NORMAL4, cfg.fill_seed, cfg.fill_scale)
    out = oracle.embedding_bag_fwd(w["ids"], w["offsets"], cfg.num_fields, cfg.batch, w["bag_to_table"],
                                   w["row_base"], cfg.d, pool="mean", dtype="bf16", gen=gen)
    # reference: exact mean in fractions of the bf16 table values, rounded to nearest-even bf16
    lens = np.diff(w["offsets"])
    f, b = 3, 5
    bag = f * cfg.batch + b
    keys = w["row_base"][f] + w["ids"][w["offsets"][bag]:w["offsets"][bag + 1]]
    rows = W.bf16_bits_to_f32(oracle.table_rows(gen[0], gen[1], gen[2], cfg.d, keys)).astype(np.float64)
    for c in range(0, cfg.d, 7):
        exact = sum(Fraction(float(v)) for v in rows[:, c]) / int(lens[bag])
        assert W.bf16_bits_to_f32(out[b, f, c:c + 1])[0] == _nearest_bf16(exact)


# ---------------------------------------------------------------------------
# dot interaction
# ---------------------------------------------------------------------------
def _nearest_bf16(q: Fraction) -> float:
    """Nearest bf16 to an exact rational, ties to even (brute force over neighbours)."""
    if q == 0:
        return 0.0
    x = float(q)
    e = int(np.frexp(abs(x))[1])  # |x| in [2^(e-1), 2^e)
    ulp = Fraction(2) ** (e - 8)
    lo = (abs(q) // ulp) * ulp
    cands = [lo, lo + ulp]
    best = min(cands, key=lambda c: (abs(abs(q) - c), int(c / ulp) % 2))
    return float(best if q > 0 else -best)


def test_fm_identity_golden(oracle):
    g = _golden("fm_identity_small.json")
    v = np.array(g["vectors"], dtype=np.float32)
    n, d = v.shape
    out = oracle.dot_interaction(v[None], n, d)
    pairs = out[0, d:]
    s = v.astype(np.int64).sum(axis=0)
    rhs = Fraction(int((s * s).sum()) - int((v.astype(np.int64) ** 2).sum()), 2)
    assert Fraction(int(pairs.astype(np.int64).sum())) == rhs
    np.testing.assert_array_equal(out[0, :d], v[0])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fm_identity_random(oracle, seed):
    rng = np.random.default_rng(seed)
    B, n, d = 16, 27, 128
    X = rng.standard_normal((B, n, d)).astype(np.float32) * rng.uniform(0.01, 2, size=(B, n, 1)).astype(np.float32)
    out, mag = oracle.dot_interaction(X, n, d, with_mag=True)
    X64 = X.astype(np.float64)
    s = X64.sum(axis=1)
    rhs = 0.5 * ((s * s).sum(axis=1) - (X64 * X64).sum(axis=(1, 2)))
    lhs = out[:, d:].astype(np.float64).sum(axis=1)
    # each stored dot carries at most half an fp32 ulp of rounding
    bound = np.abs(out[:, d:]).astype(np.float64).sum(axis=1) * 2.0 ** -24 + 1e-9 * mag[:, d:].sum(axis=1)
    assert np.all(np.abs(lhs - rhs) <= bound)


def test_interaction_golden_bruteforce(oracle):
    g = _golden("dlrm_interaction_small.json")
    vecs = [g["dense"]] + g["pooled"]
    X = np.array(vecs, dtype=np.float32)[None]
    n, d = X.shape[1], X.shape[2]
    out = oracle.dot_interaction(X, n, d)[0]
    expect = list(g["dense"])
    for i in range(1, n):
        for j in range(i):
            expect.append(sum(a * b for a, b in zip(vecs[i], vecs[j])))
    assert out.tolist() == expect
    assert out.size == d + n * (n - 1) // 2


def test_interaction_matches_numpy_gram(oracle):
    rng = np.random.default_rng(9)
    B, n, d = 33, 27, 128
    X = rng.standard_normal((B, n, d)).astype(np.float32)
    out = oracle.dot_interaction(X, n, d)
    Xd = X.astype(np.float64)
    gram = np.einsum("bic,bjc->bij", Xd, Xd)
    ii, jj = np.tril_indices(n, -1)
    ref = np.concatenate([Xd[:, 0, :], gram[:, ii, jj]], axis=1)
    np.testing.assert_array_equal(out, ref.astype(np.float32))
    # sampled mode returns the same rows
    sub = oracle.dot_interaction(X, n, d, sample_list=[32, 0, 7])
    np.testing.assert_array_equal(sub, out[[32, 0, 7]])


def test_interaction_bf16_rounding_golden(oracle):
    g = _golden("bf16_ties.json")
    for case in g["cases"]:
        x = np.array([case["x0"], case["x1"]], dtype=np.float32)
        X = W.f32_to_bf16_bits(x)[None]
        assert np.array_equal(W.bf16_bits_to_f32(X[0]), x), "fixture values must be bf16-exact"
        out = W.bf16_bits_to_f32(oracle.dot_interaction(X, 2, 2, dtype="bf16")[0])
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(case["x0"], case["x1"]))
        assert out[2] == _nearest_bf16(exact), case


def test_interaction_bf16_random_half_ulp(oracle):
    rng = np.random.default_rng(4)
    B, n, d = 8, 27, 64
    X = W.f32_to_bf16_bits(rng.standard_normal((B, n, d)).astype(np.float32))
    out = W.bf16_bits_to_f32(oracle.dot_interaction(X, n, d, dtype="bf16"))
    Xf = W.bf16_bits_to_f32(X).astype(np.float64)
    gram = np.einsum("bic,bjc->bij", Xf, Xf)
    ii, jj = np.tril_indices(n, -1)
    ref = gram[:, ii, jj]
    got = out[:, d:].astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8)    # within half a bf16 ulp (8 bits)
    np.testing.assert_array_equal(out[:, :d], Xf[:, 0, :])


def test_interaction_bwd_matches_autograd(oracle):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    B, n, d = 6, 27, 32
    X = rng.standard_normal((B, n, d)).astype(np.float32)
    dout = rng.standard_normal((B, d + n * (n - 1) // 2)).astype(np.float32)
    dX = oracle.dot_interaction_bwd(dout, X, n, d)
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    gram = torch.bmm(Xt, Xt.transpose(1, 2))
    ii, jj = np.tril_indices(n, -1)
    out = torch.cat([Xt[:, 0, :], gram[:, ii, jj]], dim=1)
    (out * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    np.testing.assert_allclose(dX, Xt.grad.numpy().astype(np.float32), rtol=1e-6, atol=1e-6)
    sub = oracle.dot_interaction_bwd(dout, X, n, d, sample_list=[5, 2])
    np.testing.assert_array_equal(sub, dX[[5, 2]])


# ---------------------------------------------------------------------------
# FM second-order term of a bag
# ---------------------------------------------------------------------------
def test_bag_fm_golden_identity(oracle):
    # the golden vectors as the rows of a one-bag table: the pairwise sum equals
    # 1/2 (|sum v|^2 - sum |v|^2), exactly (integers)
    g = _golden("fm_identity_small.json")
    v = np.array(g["vectors"], dtype=np.float32)
    m, d = v.shape
    ids = np.arange(m, dtype=np.int64)
    offsets = np.array([0, m], dtype=np.int64)
    fm = oracle.bag_fm(ids, offsets, 1, 1, [0], [0, m], d, table=v)
    s = v.astype(np.int64).sum(axis=0)
    rhs = Fraction(int((s * s).sum()) - int((v.astype(np.int64) ** 2).sum()), 2)
    assert Fraction(int(fm[0])) == rhs


def test_bag_fm_identity_random_bags(oracle):
    # integer rows, bags with repeated IDs, empty bags and single-ID bags
    rng = np.random.default_rng(31)
    F, B, d, rows = 2, 40, 8, 50
    table = rng.integers(-30, 31, size=(2 * rows, d)).astype(np.float32)
    lens = rng.integers(0, 9, size=F * B)
    lens[:3] = [0, 1, 6]
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ids = rng.integers(0, 6, size=offsets[-1]).astype(np.int64)   # many repeats
    rb = np.array([0, rows, 2 * rows], dtype=np.int64)
    fm = oracle.bag_fm(ids, offsets, F, B, [0, 1], rb, d, table=table)
    for bag in range(F * B):
        f = bag // B
        vs = table[rb[f] + ids[offsets[bag]:offsets[bag + 1]]].astype(np.int64)
        s = vs.sum(axis=0)
        expect = ((s * s).sum() - (vs * vs).sum()) // 2
        assert int(fm[bag]) == expect, bag
    assert fm[0] == 0 and fm[1] == 0                                 # empty and single-ID bags


def test_bag_fm_bruteforce_and_list(oracle):
    rng = np.random.default_rng(32)
    F, B, d, rows = 3, 7, 5, 9
    table = (rng.integers(-64, 64, size=(F * rows, d)) / 16).astype(np.float32)
    lens = rng.integers(0, 5, size=F * B)
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    ids = rng.integers(0, rows, size=offsets[-1]).astype(np.int64)
    rb = np.arange(F + 1, dtype=np.int64) * rows
    fm = oracle.bag_fm(ids, offsets, F, B, list(range(F)), rb, d, table=table)
    for bag in range(F * B):
        f = bag // B
        rws = [table[rb[f] + k] for k in ids[offsets[bag]:offsets[bag + 1]]]
        ref = sum(Fraction(float(a)) * Fraction(float(b)) for i in range(len(rws)) for j in range(i + 1, len(rws))
                  for a, b in zip(rws[i], rws[j]))
        assert Fraction(float(fm[bag])) == ref, bag
    sub = oracle.bag_fm(ids, offsets, F, B, list(range(F)), rb, d, table=table, bag_list=[20, 3])
    np.testing.assert_array_equal(sub, fm[[20, 3]])


# ---------------------------------------------------------------------------
# optimizer step on the batch's rows
# ---------------------------------------------------------------------------
def _rows_and_grads(seed, n=6, d=8):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n, d)) * 0.1
    g = rng.standard_normal((n, d))
    return w, g, rng


def test_optimizer_sgd_is_the_plain_update(oracle):
    w, g, _ = _rows_and_grads(40)
    new, _, _ = oracle.optimizer_step("sgd", w, g, 0.01)
    np.testing.assert_array_equal(new, (w - 0.01 * g).astype(np.float32))


def test_optimizer_adagrad_matches_torch(oracle):
    torch = pytest.importorskip("torch")
    w, g, rng = _rows_and_grads(41)
    s0 = rng.uniform(0, 2, size=w.shape).astype(np.float32)
    lr, eps = 0.05, 1e-6
    new, s_new, _ = oracle.optimizer_step("adagrad", w, g, lr, state0=s0, eps=eps)
    p = torch.nn.Parameter(torch.tensor(w, dtype=torch.float64))
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps)
    opt.state[p]["sum"] = torch.tensor(s0, dtype=torch.float64)
    opt.state[p]["step"] = torch.tensor(0.0)
    p.grad = torch.tensor(g, dtype=torch.float64)
    opt.step()
    np.testing.assert_allclose(new, p.detach().numpy().astype(np.float32), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(s_new, opt.state[p]["sum"].numpy().astype(np.float32), rtol=1e-6)


def test_optimizer_rowwise_adagrad(oracle):
    # a gradient constant along the row and a uniform state make row-wise and
    # elementwise Adagrad the same rule; in general the row's state grows by the
    # mean squared gradient
    w, _, rng = _rows_and_grads(42)
    g = np.repeat(rng.standard_normal((w.shape[0], 1)), w.shape[1], axis=1)
    srow = rng.uniform(0, 1, size=w.shape[0]).astype(np.float32)
    a, sa, _ = oracle.optimizer_step("rowwise_adagrad", w, g, 0.1, state0=srow, eps=1e-7)
    b, sb, _ = oracle.optimizer_step("adagrad", w, g, 0.1, state0=np.repeat(srow[:, None], w.shape[1], axis=1),
                                     eps=1e-7)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(sa, sb[:, 0])
    w, g, _ = _rows_and_grads(43)
    _, s2, _ = oracle.optimizer_step("rowwise_adagrad", w, g, 0.1, state0=srow)
    np.testing.assert_allclose(s2, srow + (g * g).mean(axis=1), rtol=1e-6)


@pytest.mark.parametrize("step", [1, 7])
def test_optimizer_adam_matches_torch(oracle, step):
    torch = pytest.importorskip("torch")
    w, g, rng = _rows_and_grads(44 + step)
    m0 = (rng.standard_normal(w.shape) * 0.1).astype(np.float32) if step > 1 else np.zeros(w.shape, np.float32)
    v0 = (rng.uniform(0, 0.5, size=w.shape)).astype(np.float32) if step > 1 else np.zeros(w.shape, np.float32)
    lr, b1, b2, eps = 0.01, 0.9, 0.99, 1e-6
    new, m, v = oracle.optimizer_step("adam", w, g, lr, state0=m0, state1=v0, eps=eps, beta1=b1, beta2=b2, step=step)
    p = torch.nn.Parameter(torch.tensor(w, dtype=torch.float64))
    opt = torch.optim.Adam([p], lr=lr, betas=(b1, b2), eps=eps)
    opt.state[p]["exp_avg"] = torch.tensor(m0, dtype=torch.float64)
    opt.state[p]["exp_avg_sq"] = torch.tensor(v0, dtype=torch.float64)
    opt.state[p]["step"] = torch.tensor(float(step - 1))
    p.grad = torch.tensor(g, dtype=torch.float64)
    opt.step()
    np.testing.assert_allclose(new, p.detach().numpy().astype(np.float32), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(m, opt.state[p]["exp_avg"].numpy().astype(np.float32), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(v, opt.state[p]["exp_avg_sq"].numpy().astype(np.float32), rtol=1e-6, atol=1e-9)


# ---------------------------------------------------------------------------
# stochastic rounding of updated bf16 rows
# ---------------------------------------------------------------------------
def _bf16_neighbours(x):
    """bf16 values just below and above |x| (toward zero first), as float64."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32) & np.uint32(0x7FFFFFFF)
    lo = ((bits >> np.uint32(16)) << np.uint32(16)).view(np.float32).astype(np.float64)
    hi = (((bits >> np.uint32(16)) + np.uint32(1)) << np.uint32(16)).view(np.float32).astype(np.float64)
    return lo, hi


def test_stochastic_round_keeps_bf16_values(oracle):
    rng = np.random.default_rng(50)
    x = W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal((5, 8)).astype(np.float32))).astype(np.float64)
    for seed in range(4):
        out = oracle.bf16_stochastic_round(x, np.arange(5), seed)
        np.testing.assert_array_equal(W.bf16_bits_to_f32(out).astype(np.float64), x)


def test_stochastic_round_picks_a_neighbour_unbiased(oracle):
    # one value per element, 4000 seeds: the result is always lo or hi, and the
    # fraction rounded up matches (|x| - lo) / (hi - lo) within a binomial bound
    rng = np.random.default_rng(51)
    x32 = (rng.standard_normal((1, 16)) * 3).astype(np.float32)
    x = x32.astype(np.float64)
    lo, hi = _bf16_neighbours(x32)
    frac = (np.abs(x) - lo) / (hi - lo)
    seeds = 4000
    ups = np.zeros(x.shape)
    for seed in range(seeds):
        got = np.abs(W.bf16_bits_to_f32(oracle.bf16_stochastic_round(x, [7], seed)).astype(np.float64))
        assert np.all((got == lo) | (got == hi))
        ups += got == hi
    p = ups / seeds
    assert np.all(np.abs(p - frac) <= 4.5 * np.sqrt(frac * (1 - frac) / seeds) + 1e-3)


def test_stochastic_round_matches_the_carry_formulation(oracle):
    # the same rounding written as fp32 bits: add the 16 random bits to the low
    # half and truncate (the carry reaches the bf16 bits exactly when f + u/2^16 >= 1)
    rng = np.random.default_rng(52)
    x32 = (rng.standard_normal((6, 12)) * 2.0 ** rng.integers(-20, 20, size=(6, 1))).astype(np.float32)
    rows = np.array([3, 0, 11, 5, 1 << 33, 17], dtype=np.int64)
    seed = 0x1234ABCD
    got = oracle.bf16_stochastic_round(x32.astype(np.float64), rows, seed)
    d = x32.shape[1]
    mask = (1 << 64) - 1

    def splitmix(z):
        z = (z + 0x9E3779B97F4A7C15) & mask
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        return z ^ (z >> 31)
    bits = x32.view(np.uint32)
    for r in range(x32.shape[0]):
        for c in range(d):
            u = (splitmix(seed ^ (int(rows[r]) * (d // 4) + c // 4)) >> (16 * (c % 4))) & 0xFFFF
            b = int(bits[r, c])
            expect = ((b & 0x80000000) | ((b & 0x7FFFFFFF) + u)) >> 16
            assert int(got[r, c]) == expect, (r, c)


# ---------------------------------------------------------------------------
# interaction variants: products with the diagonal, the full Gram matrix
# ---------------------------------------------------------------------------
def test_interaction_cross_mode_is_the_default_interaction(oracle):
    rng = np.random.default_rng(21)
    X = rng.standard_normal((9, 27, 64)).astype(np.float32)
    np.testing.assert_array_equal(oracle.dot_interaction_mode(X, 27, 64, "cross"), oracle.dot_interaction(X, 27, 64))
    dout = rng.standard_normal((9, 64 + 351)).astype(np.float32)
    np.testing.assert_allclose(oracle.dot_interaction_bwd_mode(dout, X, 27, 64, "cross"),
                               oracle.dot_interaction_bwd(dout, X, 27, 64), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("seed", [0, 1])
def test_interaction_with_self_identity(oracle, seed):
    # sum over i >= j of <x_i, x_j> = 1/2 (|sum x|^2 + sum |x|^2): the FM identity
    # with the diagonal terms added once (integer vectors: exact in fp32 and fp64)
    rng = np.random.default_rng(seed)
    B, n, d = 5, 27, 16
    X = rng.integers(-40, 41, size=(B, n, d)).astype(np.float32)
    out = oracle.dot_interaction_mode(X, n, d, "with_self")
    assert out.shape == (B, d + n * (n + 1) // 2)
    Xi = X.astype(np.int64)
    s = Xi.sum(axis=1)
    rhs = ((s * s).sum(axis=1) + (Xi * Xi).sum(axis=(1, 2))) // 2
    np.testing.assert_array_equal(out[:, d:].astype(np.int64).sum(axis=1), rhs)
    np.testing.assert_array_equal(out[:, :d], X[:, 0, :])
    # the diagonal entries are the squared norms, at i(i+1)/2 + i
    diag = np.array([d + i * (i + 1) // 2 + i for i in range(n)])
    np.testing.assert_array_equal(out[:, diag].astype(np.int64), (Xi * Xi).sum(axis=2))


def test_interaction_with_self_bruteforce(oracle):
    g = _golden("dlrm_interaction_small.json")
    vecs = [g["dense"]] + g["pooled"]
    X = np.array(vecs, dtype=np.float32)[None]
    n, d = X.shape[1], X.shape[2]
    out = oracle.dot_interaction_mode(X, n, d, "with_self")[0]
    expect = list(g["dense"])
    for i in range(n):
        for j in range(i + 1):
            expect.append(sum(a * b for a, b in zip(vecs[i], vecs[j])))
    assert out.tolist() == expect


def test_interaction_full_gram_matches_numpy(oracle):
    rng = np.random.default_rng(22)
    B, n, d = 7, 27, 128
    X = rng.standard_normal((B, n, d)).astype(np.float32)
    out = oracle.dot_interaction_mode(X, n, d, "full")
    Xd = X.astype(np.float64)
    gram = np.einsum("bic,bjc->bij", Xd, Xd)
    np.testing.assert_array_equal(out, gram.reshape(B, n * n).astype(np.float32))
    G = out.reshape(B, n, n)
    np.testing.assert_array_equal(G, G.transpose(0, 2, 1))           # symmetric
    sub = oracle.dot_interaction_mode(X, n, d, "full", sample_list=[6, 1])
    np.testing.assert_array_equal(sub, out[[6, 1]])


def test_interaction_full_gram_bf16_rounds_once(oracle):
    rng = np.random.default_rng(23)
    B, n, d = 3, 9, 64
    X = W.f32_to_bf16_bits(rng.standard_normal((B, n, d)).astype(np.float32))
    out = W.bf16_bits_to_f32(oracle.dot_interaction_mode(X, n, d, "full", dtype="bf16"))
    Xf = W.bf16_bits_to_f32(X).astype(np.float64)
    ref = np.einsum("bic,bjc->bij", Xf, Xf).reshape(B, n * n)
    assert np.all(np.abs(out - ref) <= np.abs(ref) * 2.0 ** -8)


@pytest.mark.parametrize("mode", ["cross", "with_self", "full"])
def test_interaction_mode_bwd_matches_autograd(oracle, mode):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(24)
    B, n, d = 4, 27, 32
    X = rng.standard_normal((B, n, d)).astype(np.float32)
    width = oracle.interaction_width(n, d, mode)
    dout = rng.standard_normal((B, width)).astype(np.float32)
    dX = oracle.dot_interaction_bwd_mode(dout, X, n, d, mode)
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    gram = torch.bmm(Xt, Xt.transpose(1, 2))
    if mode == "full":
        out = gram.reshape(B, n * n)
    else:
        ii, jj = np.tril_indices(n, -1 if mode == "cross" else 0)
        out = torch.cat([Xt[:, 0, :], gram[:, ii, jj]], dim=1)
    (out * torch.tensor(dout, dtype=torch.float64)).sum().backward()
    np.testing.assert_allclose(dX, Xt.grad.numpy().astype(np.float32), rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------------------
# sparse backward + SGD
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_bwd_update_matches_autograd(oracle, pool):
    torch = pytest.importorskip("torch")
    bags, ids, offsets, b2t, rb = _small_case(seed=21, F=3, B=9, rows=(40, 12, 25), d=8, max_len=9)
    F, B, d, lr = 3, 9, 8, 0.01
    rng = np.random.default_rng(8)
    table = rng.uniform(-0.1, 0.1, size=(int(rb[-1]), d)).astype(np.float32)
    G = rng.standard_normal((B, F, d)).astype(np.float32)
    lens = np.diff(offsets)
    bag_of = np.repeat(np.arange(F * B), lens)
    keys = rb[b2t[bag_of // B]] + ids
    targets = np.unique(keys)
    new, grad, mag = oracle.embedding_bag_bwd_update(G, ids, offsets, F, B, b2t, rb, d, lr, targets, pool=pool,
                                                     table=table)
    Wt = torch.tensor(table, dtype=torch.float64, requires_grad=True)
    pooled = torch.nn.functional.embedding_bag(torch.tensor(keys), Wt, torch.tensor(offsets[:-1]), mode=pool)
    Gt = torch.tensor(G, dtype=torch.float64).permute(1, 0, 2).reshape(F * B, d)   # field-major bags
    (pooled * Gt).sum().backward()
    tg = Wt.grad.numpy()
    np.testing.assert_allclose(grad, tg[targets], rtol=1e-12, atol=1e-12)
    untouched = np.setdiff1d(np.arange(int(rb[-1])), targets)
    assert np.all(tg[untouched] == 0)
    np.testing.assert_array_equal(new, (table[targets].astype(np.float64) - np.float32(lr) * grad).astype(np.float32))
    assert np.all(mag >= np.abs(grad) - 1e-12)


def test_bwd_column_sum_invariant(oracle):
    cfg = W.CONFIGS["tensornet"].shrink(batch=32)
    w = W.make_workload(cfg)
    F, B, d = cfg.num_fields, cfg.batch, cfg.d
    targets = np.unique(w["ids"])
    gen = (oracle.GEN_UNIFORM, cfg.fill_seed, cfg.fill_scale)
    _, grad, _ = oracle.embedding_bag_bwd_update(w["grad_pooled"], w["ids"], w["offsets"], F, B, w["bag_to_table"],
                                                 w["row_base"], d, cfg.lr, targets, gen=gen)
    lens = np.diff(w["offsets"]).reshape(F, B)
    expect = (w["grad_pooled"].astype(np.float64) * lens.T[:, :, None]).sum(axis=(0, 1))
    np.testing.assert_allclose(grad.sum(axis=0), expect, rtol=1e-10, atol=1e-9)


def test_bwd_exact_arithmetic(oracle):
    # dyadic gradients, table values and a power-of-two lr: every value is exact,
    # so the update equals a plain scatter-add bit for bit
    bags, ids, offsets, b2t, rb = _small_case(seed=2, F=2, B=11, rows=(6, 4), d=4, max_len=7)
    F, B, d = 2, 11, 4
    lr = 2.0 ** -4
    rng = np.random.default_rng(1)
    table = (rng.integers(-64, 64, size=(int(rb[-1]), d)) / 64).astype(np.float32)
    G = (rng.integers(-8, 9, size=(B, F, d)) / 8).astype(np.float32)
    lens = np.diff(offsets)
    bag_of = np.repeat(np.arange(F * B), lens)
    keys = rb[b2t[bag_of // B]] + ids
    targets = np.unique(keys)
    new, grad, _ = oracle.embedding_bag_bwd_update(G, ids, offsets, F, B, b2t, rb, d, lr, targets, table=table)
    acc = np.zeros((int(rb[-1]), d))
    np.add.at(acc, keys, G[bag_of % B, bag_of // B].astype(np.float64))
    np.testing.assert_array_equal(grad, acc[targets])
    np.testing.assert_array_equal(new, table[targets] - np.float32(lr) * acc[targets].astype(np.float32))


# ---------------------------------------------------------------------------
# counter-based table generator (input generation)
# ---------------------------------------------------------------------------
def test_table_generator_matches_numpy_definition(oracle):
    cfg = W.CONFIGS["dlrm_fp32"]
    rows = np.array([0, 1, 499_999, 12_345_678], dtype=np.int64)
    d = cfg.d
    got = oracle.table_rows(oracle.GEN_UNIFORM, cfg.fill_seed, cfg.fill_scale, d, rows)
    idx = (rows[:, None] * d + np.arange(d)).astype(np.uint64)
    h = W.splitmix64(np.uint64(cfg.fill_seed) ^ idx)
    c = (h >> np.uint64(40)).astype(np.int64) - (1 << 23)
    ref = c.astype(np.float32) * np.float32(cfg.fill_scale)
    np.testing.assert_array_equal(got, ref)
    assert oracle.splitmix64(12345) == int(W.splitmix64(np.uint64(12345)))


def test_table_generator_statistics(oracle):
    cfg = W.CONFIGS["dlrm_fp32"]
    v = oracle.table_rows(oracle.GEN_UNIFORM, cfg.fill_seed, cfg.fill_scale, 128, np.arange(4000)).ravel()
    assert v.min() >= -0.01 and v.max() < 0.01
    assert abs(v.mean()) < 2e-4 and abs(v.var() - 0.01 ** 2 / 3) < 1e-6
    c3 = W.CONFIGS["bf16_large"]
    b = oracle.table_rows(oracle.GEN_NORMAL4, c3.fill_seed, c3.fill_scale, 64, np.arange(8000))
    x = W.bf16_bits_to_f32(b).ravel().astype(np.float64)
    assert abs(x.mean()) < 2e-4 and abs(x.std() - 0.01) < 2e-4
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(kurt - 2.7) < 0.1       # Irwin-Hall(4): excess kurtosis -0.3


def test_zipf_sampler_matches_pmf():
    rng = W._rng(123, 0)
    for alpha, n in ((1.05, 20), (1.2, 40)):
        k = W.zipf_ranks(rng, alpha, n, 400_000)
        assert k.min() >= 1 and k.max() <= n
        p = np.arange(1, n + 1, dtype=float) ** -alpha
        p /= p.sum()
        e = p * k.size
        c = np.bincount(k, minlength=n + 1)[1:]
        chi2 = ((c - e) ** 2 / e).sum()
        assert chi2 < (n - 1) + 6 * np.sqrt(2 * (n - 1))   # ~ 4.2 sigma above the mean
