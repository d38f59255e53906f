"""Seeded synthetic workloads for the CTR embedding + interaction path.

This module only draws inputs: bag lengths, categorical IDs, dense vectors and
upstream gradients, plus the parameters of the counter-based table generator.
It holds none of the method's arithmetic (no pooling, no dedup, no dot
products, no update), so it can feed both the CUDA path and the CPU oracle.

Workload shapes follow the page "Meta DLRM" (section 05: the benchmark draws
random synthetic inputs whose categorical features come from distributions; the
public ads set has 26 categorical fields) and the page "DHEN" (section 2.1:
one trainable d-vector per categorical term).  The five named workloads are the
tiny reference case, a DLRM-shaped fp32 forward, a large-batch bf16 forward, a
TensorNet-style dedup + sparse backward on one hashed table, and the full step
at scale.  No dataset record is used.

Every array comes from its own numpy stream,
``Generator(PCG64(SeedSequence([seed, stream, ...])))``.

Embedding tables are never materialised here.  Their values come from a
counter-based generator built on splitmix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) that both the CUDA
library and the oracle implement on their own from that definition:

* ``uniform``: h = splitmix64(S xor idx); v = fp32(int(h >> 40) - 2^23) * scale,
  scale = fp32(hi) * 2^-23.  One IEEE rounding, so host and device agree bit
  for bit.  Values lie in [-hi, hi).
* ``normal4``: an Irwin-Hall sum of four 22-bit uniforms taken from
  h1 = splitmix64(S xor 2*idx) and h2 = splitmix64(S xor (2*idx + 1)),
  centred (exact in fp32), times scale = fp32(sigma * sqrt(3) * 2^-22), then
  rounded to bf16 (round to nearest even).  Mean 0, standard deviation sigma.

idx is the global element index row * d + c and S = splitmix64(seed).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np

U64 = np.uint64
_MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_HASH_MULT = 2654435761  # odd, not a multiple of 5: a bijection mod 2^a * 5^b


# --------------------------------------------------------------------------
# splitmix64 (Steele, Lea, Flood 2014), vectorised over uint64 with wraparound
# --------------------------------------------------------------------------
def splitmix64(x) -> np.ndarray:
    """splitmix64 output function applied to state+gamma, elementwise."""
    with np.errstate(over="ignore"):
        z = np.asarray(x, dtype=U64) + U64(GOLDEN_GAMMA)
        z = (z ^ (z >> U64(30))) * U64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> U64(27))) * U64(0x94D049BB133111EB)
        return z ^ (z >> U64(31))


def splitmix64_int(x: int) -> int:
    return int(splitmix64(np.array([x & _MASK64], dtype=U64))[0])


# --------------------------------------------------------------------------
# Truncated Zipf sampling by rejection-inversion (Hormann and Derflinger,
# "Rejection-inversion to generate variates from monotone discrete
# distributions", ACM TOMACS 1996).  Exact for P(k) ~ k^-alpha, k = 1..n.
# --------------------------------------------------------------------------
def _h(alpha: float, x):
    return np.exp(-alpha * np.log(x))


def _H(alpha: float, x):
    # integral of t^-alpha from 1 to x, stable near alpha = 1
    lx = np.log(x)
    t = (1.0 - alpha) * lx
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(np.abs(t) > 1e-8, np.expm1(t) / np.where(t == 0, 1, t), 1.0 + t / 2.0)
    return r * lx


def _H_inv(alpha: float, y):
    t = np.maximum(y * (1.0 - alpha), -1.0 + 1e-16)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(np.abs(t) > 1e-8, np.log1p(t) / np.where(t == 0, 1, t), 1.0 - t / 2.0)
    return np.exp(r * y)


def zipf_ranks(rng: np.random.Generator, alpha: float, n: int, size: int) -> np.ndarray:
    """Draw `size` ranks in [1, n] with P(k) proportional to k^-alpha."""
    if size == 0:
        return np.zeros(0, dtype=np.int64)
    h_x1 = float(_H(alpha, 1.5)) - 1.0
    h_n = float(_H(alpha, n + 0.5))
    s = 2.0 - float(_H_inv(alpha, _H(alpha, 2.5) - _h(alpha, 2.0)))
    out = np.empty(size, dtype=np.int64)
    filled = 0
    while filled < size:
        m = size - filled
        m = int(m * 1.05) + 64
        u = h_n + rng.random(m) * (h_x1 - h_n)
        x = _H_inv(alpha, u)
        k = np.clip(np.floor(x + 0.5), 1, n)
        ok = (k - x <= s) | (u >= _H(alpha, k + 0.5) - _h(alpha, k))
        acc = k[ok].astype(np.int64)
        take = min(acc.size, size - filled)
        out[filled:filled + take] = acc[:take]
        filled += take
    return out


# --------------------------------------------------------------------------
# bf16 bit helpers for generated inputs (round to nearest even)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# Workload configurations
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    seed: int
    batch: int
    num_fields: int
    field_to_table: Tuple[int, ...]
    rows_per_table: Tuple[int, ...]
    d: int
    dtype: str                      # "f32" | "bf16"  (table, pooled and interaction dtype)
    table_init: Tuple               # ("uniform", hi) | ("normal4", sigma)
    bag_len: Tuple                  # ("fixed", L) | ("uniform", lo, hi) | ("poisson", mean, lo, hi)
    ids: Tuple                      # ("uniform",) | ("zipf", alpha) | ("zipf_hashed", alpha, raw_space, row_bits)
    pool: str                       # "sum" | "mean"
    interaction: bool
    backward: str                   # "none" | "pooled_grad" | "full"
    lr: float
    dedup_gather: bool = False      # pool from the batch-sized unique-row matrix via the inverse map
    interaction_mode: str = "cross"  # "cross" (i > j) | "with_self" (i >= j) | "full" (n x n Gram matrix)

    @property
    def num_tables(self) -> int:
        return len(self.rows_per_table)

    @property
    def row_base(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(np.asarray(self.rows_per_table, dtype=np.int64))]).astype(np.int64)

    @property
    def total_rows(self) -> int:
        return int(sum(self.rows_per_table))

    @property
    def n_vectors(self) -> int:
        return self.num_fields + 1

    @property
    def out_width(self) -> int:
        """Interaction output row: [dense | products i > j], [dense | products i >= j] or the n x n Gram matrix."""
        n = self.n_vectors
        if self.interaction_mode == "full":
            return n * n
        return self.d + (n * (n - 1) // 2 if self.interaction_mode == "cross" else n * (n + 1) // 2)

    @property
    def fill_seed(self) -> int:
        return splitmix64_int(self.seed)

    @property
    def fill_scale(self) -> float:
        kind, p = self.table_init
        if kind == "uniform":
            return float(np.float32(np.float32(p) * np.float32(2.0 ** -23)))
        if kind == "normal4":
            return float(np.float32(p * math.sqrt(3.0) * 2.0 ** -22))
        raise ValueError(kind)

    @property
    def fill_kind(self) -> int:
        return {"uniform": 0, "normal4": 1}[self.table_init[0]]

    def shrink(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


def _tables(n: int, rows: int) -> Tuple[int, ...]:
    return tuple([rows] * n)


CONFIGS: Dict[str, Config] = {
    # 1. tiny reference: 4 fp32 tables 1000 x 16, one uniform ID per bag, SGD step
    "tiny": Config("tiny", 0, 64, 4, (0, 1, 2, 3), _tables(4, 1000), 16, "f32",
                   ("uniform", 0.05), ("fixed", 1), ("uniform",), "sum", True, "pooled_grad", 0.01),
    # 2. DLRM-shaped fp32 forward
    "dlrm_fp32": Config("dlrm_fp32", 2, 2048, 26, tuple(range(26)), _tables(26, 500_000), 128, "f32",
                        ("uniform", 0.01), ("uniform", 1, 20), ("zipf", 1.05), "sum", True, "none", 0.01),
    # 3. bf16 tables, large batch, mean pooling, tensor-core interaction
    "bf16_large": Config("bf16_large", 3, 65536, 26, tuple(range(26)), _tables(26, 4_000_000), 64, "bf16",
                         ("normal4", 0.01), ("poisson", 30, 1, 100), ("zipf", 1.2), "mean", True, "none", 0.01),
    # 4. TensorNet-style: 100 fields share one 2^26-row table of hashed 64-bit IDs
    "tensornet": Config("tensornet", 4, 16384, 100, tuple([0] * 100), (1 << 26,), 32, "f32",
                        ("uniform", 0.01), ("uniform", 1, 10), ("zipf_hashed", 1.1, 10 ** 9, 26), "sum", False,
                        "pooled_grad", 0.01, dedup_gather=True),
    # 5. full step at scale: 26 x 8M x 128 fp32 (106.5 GB of tables)
    "full_step": Config("full_step", 5, 131072, 26, tuple(range(26)), _tables(26, 8_000_000), 128, "f32",
                        ("uniform", 0.01), ("uniform", 1, 50), ("zipf", 1.05), "sum", True, "full", 0.01),
}


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def bag_lengths(cfg: Config) -> np.ndarray:
    """Lengths of the F*B bags, field-major: bag (f, b) is entry f*B + b."""
    n = cfg.num_fields * cfg.batch
    rng = _rng(cfg.seed, 1)
    kind = cfg.bag_len[0]
    if kind == "fixed":
        return np.full(n, cfg.bag_len[1], dtype=np.int64)
    if kind == "uniform":
        return rng.integers(cfg.bag_len[1], cfg.bag_len[2] + 1, size=n, dtype=np.int64)
    if kind == "poisson":
        return np.clip(rng.poisson(cfg.bag_len[1], size=n), cfg.bag_len[2], cfg.bag_len[3]).astype(np.int64)
    raise ValueError(kind)


def _batch_stream(batch_index: int, *stream: int):
    """Stream key of one array of batch `batch_index` (batch 0 keeps the original keys)."""
    return (*stream, batch_index) if batch_index else stream


def draw_ids(cfg: Config, lengths: np.ndarray, batch_index: int = 0) -> np.ndarray:
    """Table-local row IDs for every bag occurrence, field-major CSR order.

    Batches with another `batch_index` draw new IDs from the same distribution
    (the same hot rows: the rank -> row map is a property of the table)."""
    B = cfg.batch
    per_field = lengths.reshape(cfg.num_fields, B).sum(axis=1)
    ids = np.empty(int(per_field.sum()), dtype=np.int64)
    pos = 0
    kind = cfg.ids[0]
    off_rng = _rng(cfg.seed, 5)
    table_shift = off_rng.integers(0, np.asarray(cfg.rows_per_table, dtype=np.int64))
    for f in range(cfg.num_fields):
        t = cfg.field_to_table[f]
        nrows = cfg.rows_per_table[t]
        m = int(per_field[f])
        rng = _rng(cfg.seed, *_batch_stream(batch_index, 2, f))
        if kind == "uniform":
            v = rng.integers(0, nrows, size=m, dtype=np.int64)
        elif kind == "zipf":
            k = zipf_ranks(rng, cfg.ids[1], nrows, m) - 1
            # scatter hot ranks over the table like hashed IDs: k -> (k*A + c_t) mod N
            v = (k * _HASH_MULT + int(table_shift[t])) % nrows  # k < 2^32, no int64 overflow
        elif kind == "zipf_hashed":
            _, alpha, raw_space, row_bits = cfg.ids
            k = zipf_ranks(rng, alpha, raw_space, m)
            v = (splitmix64(k.astype(U64)) & U64((1 << row_bits) - 1)).astype(np.int64)
        else:
            raise ValueError(kind)
        ids[pos:pos + m] = v
        pos += m
    return ids


def make_workload(cfg: Config, with_grads: bool = True, batch_index: int = 0) -> Dict[str, np.ndarray]:
    """All host-side inputs of one step for `cfg` (tables excluded).

    `batch_index` > 0 gives another batch of the same workload: new IDs, dense
    vectors and upstream gradients, with the same bag lengths (so every batch
    has the same ID count, which a captured step fixes)."""
    lengths = bag_lengths(cfg)
    offsets = np.zeros(lengths.size + 1, dtype=np.int64)
    np.cumsum(lengths, out=offsets[1:])
    w = {
        "offsets": offsets,
        "ids": draw_ids(cfg, lengths, batch_index),
        "bag_to_table": np.asarray(cfg.field_to_table, dtype=np.int32),
        "row_base": cfg.row_base,
    }
    drng = _rng(cfg.seed, *_batch_stream(batch_index, 3))
    dense = drng.standard_normal((cfg.batch, cfg.d)).astype(np.float32)
    w["dense"] = f32_to_bf16_bits(dense) if cfg.dtype == "bf16" else dense
    if with_grads:
        grng = _rng(cfg.seed, *_batch_stream(batch_index, 4))
        if cfg.backward == "pooled_grad":
            w["grad_pooled"] = grng.standard_normal((cfg.batch, cfg.num_fields, cfg.d)).astype(np.float32)
        elif cfg.backward == "full":
            w["dout"] = grng.standard_normal((cfg.batch, cfg.out_width)).astype(np.float32)
    return w


def table_rows_host_bytes(cfg: Config) -> int:
    return cfg.total_rows * cfg.d * (2 if cfg.dtype == "bf16" else 4)


def describe(cfg: Config) -> Dict:
    return {
        "workload": cfg.name, "batch": cfg.batch, "fields": cfg.num_fields, "tables": cfg.num_tables,
        "rows_per_table": cfg.rows_per_table[0], "d": cfg.d, "dtype": cfg.dtype, "pool": cfg.pool,
        "bag_len": list(cfg.bag_len), "ids": list(cfg.ids), "lr": cfg.lr,
    }
