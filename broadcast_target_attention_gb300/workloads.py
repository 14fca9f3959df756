"""Seeded synthetic workloads for IKBO target attention.

This module draws inputs and nothing else: the candidate count of each user,
the user sequence lengths, the ``cand_to_user`` map, the jagged
``user_offsets`` and the bf16 bits of q, k and v.  It holds none of the
attention arithmetic, so the CUDA path's tests and bench and the CPU oracle
can both take their inputs from it.

Shapes (the layout the library's C ABI documents):

* ``q``            bf16 bits ``uint16[n_cand, H, Lq, D]``
* ``k``, ``v``     bf16 bits ``uint16[T, H, D]``, user sequences packed back to
                   back (jagged, no padding tokens), ``T = user_offsets[-1]``
* ``user_offsets`` ``int32[n_user + 1]``, ``user_offsets[0] = 0``, non-decreasing
* ``cand_to_user`` ``int32[n_cand]``, values in ``[0, n_user)``

The named configurations follow the workload shapes of "In-Kernel Broadcast
Optimization: Co-Designing Kernels for RecSys Inference" (§1.1: about 15
users behind 1024 candidates, a ~70x replication; §3: target attention over
the user history) with the jagged packing of "Optimizing Jagged Flash
Attention with TLX" (introduction: sequences packed with an offsets tensor).
The pages name no public dataset; these seeded draws stand in for their
production traffic.

Every draw uses numpy's PCG64 generator, whose output is the same on x86_64
and aarch64 (structure from one stream seeded by the config's seed, values
from per-chunk streams), and floats are rounded to bf16 with integer arithmetic
(round-to-nearest-even), so the bits are identical on every machine.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

from dataclasses import dataclass, field
from typing import Sequence

import numpy as np

# Values are drawn in chunks of this many elements so that very large tensors
# never need a float32 temporary of their full size.
_CHUNK = 1 << 24


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Finite inputs only (the generators below never produce inf or NaN).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(seed: int, tensor_id: int, shape, std: float) -> np.ndarray:
    """N(0, std^2) values rounded to bf16.

    Chunk ``i`` of tensor ``tensor_id`` is drawn from its own PCG64 stream
    seeded by ``SeedSequence([seed, tensor_id, i])``, so chunks can be drawn
    on several threads and the result does not depend on the thread count.
    """
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)

    def fill(i: int) -> None:
        s = i * _CHUNK
        e = min(n, s + _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, i])))
        x = g.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(x)

    n_chunks = (n + _CHUNK - 1) // _CHUNK
    if n_chunks <= 1:
        for i in range(n_chunks):
            fill(i)
    else:
        workers = min(n_chunks, os.cpu_count() or 1)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


@dataclass(frozen=True)
class Config:
    """A workload recipe.  ``counts``/``lens`` pick how the structure is drawn.

    counts: "multinomial" -> every user gets 1 + Multinomial(n_cand - n_user, uniform)
            "zipf"        -> Zipf(s) weights, with the last users forced to ``forced_counts``
            a tuple       -> explicit per-user counts
    lens:   "uniform"     -> integers uniform in [len_lo, len_hi]
            "loguniform"  -> round(exp(U[ln len_lo, ln len_hi]))
            a tuple       -> explicit per-user lengths
    """

    name: str
    n_cand: int
    n_user: int
    H: int
    D: int
    Lq: int
    seed: int
    std: float = 1.0
    counts: object = "multinomial"
    lens: object = "uniform"
    len_lo: int = 0
    len_hi: int = 0
    zipf_s: float = 1.1
    forced_counts: Sequence[int] = ()
    shuffle: bool = False
    description: str = ""


@dataclass
class Workload:
    cfg: Config
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    user_offsets: np.ndarray
    cand_to_user: np.ndarray
    scale: float
    counts: np.ndarray = field(repr=False, default=None)
    lens: np.ndarray = field(repr=False, default=None)

    @property
    def n_cand(self) -> int:
        return int(self.cand_to_user.shape[0])

    @property
    def n_user(self) -> int:
        return int(self.user_offsets.shape[0] - 1)

    @property
    def T(self) -> int:
        return int(self.user_offsets[-1])

    @property
    def S(self) -> int:
        """Total keys visited: sum over candidates of their user's length."""
        L = np.diff(self.user_offsets.astype(np.int64))
        return int(L[self.cand_to_user.astype(np.int64)].sum())


def _draw_counts(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    if isinstance(cfg.counts, (tuple, list)):
        c = np.asarray(cfg.counts, dtype=np.int64)
        assert c.shape == (cfg.n_user,) and int(c.sum()) == cfg.n_cand
        return c
    if cfg.counts == "multinomial":
        extra = rng.multinomial(cfg.n_cand - cfg.n_user, [1.0 / cfg.n_user] * cfg.n_user)
        return 1 + extra.astype(np.int64)
    if cfg.counts == "zipf":
        forced = np.asarray(cfg.forced_counts, dtype=np.int64)
        n_free = cfg.n_user - forced.size
        w = (np.arange(1, n_free + 1, dtype=np.float64)) ** (-cfg.zipf_s)
        w /= w.sum()
        extra = rng.multinomial(cfg.n_cand - int(forced.sum()) - n_free, w)
        return np.concatenate([1 + extra.astype(np.int64), forced])
    raise ValueError(f"unknown counts recipe {cfg.counts!r}")


def _draw_lens(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    if isinstance(cfg.lens, (tuple, list)):
        L = np.asarray(cfg.lens, dtype=np.int64)
        assert L.shape == (cfg.n_user,)
        return L
    if cfg.lens == "uniform":
        return rng.integers(cfg.len_lo, cfg.len_hi + 1, size=cfg.n_user).astype(np.int64)
    if cfg.lens == "loguniform":
        x = rng.uniform(np.log(cfg.len_lo), np.log(cfg.len_hi), size=cfg.n_user)
        return np.clip(np.round(np.exp(x)), cfg.len_lo, cfg.len_hi).astype(np.int64)
    raise ValueError(f"unknown lens recipe {cfg.lens!r}")


def generate(cfg: Config) -> Workload:
    """Draw one workload.  The same ``cfg`` always gives the same bits."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    counts = _draw_counts(cfg, rng)
    lens = _draw_lens(cfg, rng)
    c2u = np.repeat(np.arange(cfg.n_user, dtype=np.int32), counts)
    if cfg.shuffle:
        c2u = c2u[rng.permutation(c2u.shape[0])]
    offsets = np.zeros(cfg.n_user + 1, dtype=np.int64)
    np.cumsum(lens, out=offsets[1:])
    assert offsets[-1] < 2**31
    T = int(offsets[-1])
    q = _normal_bf16(cfg.seed, 0, (cfg.n_cand, cfg.H, cfg.Lq, cfg.D), cfg.std)
    k = _normal_bf16(cfg.seed, 1, (T, cfg.H, cfg.D), cfg.std)
    v = _normal_bf16(cfg.seed, 2, (T, cfg.H, cfg.D), cfg.std)
    return Workload(cfg=cfg, q=q, k=k, v=v,
                    user_offsets=offsets.astype(np.int32),
                    cand_to_user=c2u.astype(np.int32),
                    scale=float(1.0 / np.sqrt(cfg.D)),
                    counts=counts, lens=lens)


def custom(n_user: int, counts: Sequence[int], lens: Sequence[int], H: int, D: int, Lq: int,
           seed: int = 0, std: float = 1.0, shuffle: bool = False, name: str = "custom") -> Workload:
    """A workload with explicit per-user candidate counts and sequence lengths."""
    cfg = Config(name=name, n_cand=int(sum(counts)), n_user=n_user, H=H, D=D, Lq=Lq, seed=seed,
                 std=std, counts=tuple(int(c) for c in counts), lens=tuple(int(x) for x in lens),
                 shuffle=shuffle)
    return generate(cfg)


def user_queries(wl: Workload) -> np.ndarray:
    """Queries of the user sequence for self-attention: bf16 bits ``uint16[T, H, D]``, drawn
    like ``k`` and ``v`` (same seed, their own stream, the config's std)."""
    cfg = wl.cfg
    T = int(wl.user_offsets[-1])
    return _normal_bf16(cfg.seed, 3, (T, cfg.H, cfg.D), cfg.std)


def sample_rows(wl: Workload, max_count: int) -> np.ndarray:
    """A deterministic subset of sequence rows for large workloads: every user's first and
    last row, plus an even stride over all rows, capped near ``max_count``; sorted, unique."""
    T = int(wl.user_offsets[-1])
    if T <= max_count:
        return np.arange(T, dtype=np.int64)
    picks = set(np.linspace(0, T - 1, num=max_count, dtype=np.int64).tolist())
    off = wl.user_offsets.astype(np.int64)
    for u in range(off.shape[0] - 1):
        if off[u + 1] > off[u]:
            picks.add(int(off[u]))
            picks.add(int(off[u + 1] - 1))
    return np.asarray(sorted(picks), dtype=np.int64)


def sample_candidates(wl: Workload, max_count: int) -> np.ndarray:
    """A deterministic subset of candidate indices for large workloads.

    Every user's first and last candidate, plus an even stride over all
    candidates, capped near ``max_count``; sorted, unique, int64.
    """
    n = wl.n_cand
    if n <= max_count:
        return np.arange(n, dtype=np.int64)
    c2u = wl.cand_to_user.astype(np.int64)
    picks = set(np.linspace(0, n - 1, num=max_count, dtype=np.int64).tolist())
    first = {}
    last = {}
    for i, u in enumerate(c2u.tolist()):
        first.setdefault(u, i)
        last[u] = i
    picks.update(first.values())
    picks.update(last.values())
    return np.asarray(sorted(picks), dtype=np.int64)


# ---------------------------------------------------------------------------
# IKBO linear compression ("In-Kernel Broadcast Optimization", §2): each
# candidate's K input embeddings (its user's K_user, then its own K_cand, each
# of N values) are compressed to M by a learned W [M, K].  The library takes
# the decomposed operands, each K block zero-padded to a multiple of 8 (§2.2:
# padding is exact and keeps every row 16-byte aligned).

def round_up8(x: int) -> int:
    return (int(x) + 7) // 8 * 8


@dataclass
class LceConfig:
    name: str
    n_cand: int
    n_user: int
    M: int
    K_user: int          # user embeddings (before padding)
    K_cand: int          # candidate embeddings (before padding)
    N: int
    seed: int
    description: str = ""


@dataclass
class LceWorkload:
    cfg: LceConfig
    W_user: np.ndarray       # bf16 bits [M, Ku8]   (Ku8 = K_user rounded up to 8; zero columns past K_user)
    W_cand: np.ndarray       # bf16 bits [M, Kc8]
    X_user: np.ndarray       # bf16 bits [n_user, Ku8, N]  (zero rows past K_user)
    X_cand: np.ndarray       # bf16 bits [n_cand, Kc8, N]
    cand_to_user: np.ndarray  # int32 [n_cand], sorted
    counts: np.ndarray = field(repr=False, default=None)


def lce_generate(cfg: LceConfig) -> LceWorkload:
    """One seeded LCE workload: candidates per user 1 + Multinomial (uniform), sorted map;
    X ~ N(0, 1), W ~ N(0, (0.5 / sqrt(K))^2) so that outputs are O(1)."""
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    counts = 1 + rng.multinomial(cfg.n_cand - cfg.n_user, np.full(cfg.n_user, 1.0 / cfg.n_user))
    c2u = np.repeat(np.arange(cfg.n_user, dtype=np.int32), counts)
    ku, kc = round_up8(cfg.K_user), round_up8(cfg.K_cand)
    std_w = 0.5 / np.sqrt(cfg.K_user + cfg.K_cand)

    def padded(tid, shape, pad_axis, valid, std):
        x = _normal_bf16(cfg.seed, tid, shape, std).reshape(shape)
        idx = [slice(None)] * len(shape)
        idx[pad_axis] = slice(valid, None)
        x[tuple(idx)] = 0
        return x

    W_user = padded(10, (cfg.M, ku), 1, cfg.K_user, std_w)
    W_cand = padded(11, (cfg.M, kc), 1, cfg.K_cand, std_w)
    X_user = padded(12, (cfg.n_user, ku, cfg.N), 1, cfg.K_user, 1.0)
    X_cand = padded(13, (cfg.n_cand, kc, cfg.N), 1, cfg.K_cand, 1.0)
    return LceWorkload(cfg=cfg, W_user=W_user, W_cand=W_cand, X_user=X_user, X_cand=X_cand,
                       cand_to_user=c2u.astype(np.int32), counts=counts)


LCE_CONFIGS = {
    "lce_tiny_8x3": LceConfig(name="lce_tiny_8x3", n_cand=8, n_user=3, M=37, K_user=13, K_cand=21,
                              N=64, seed=20,
                              description="8 candidates over 3 users, M=37, K=13+21 (padded 16+24), N=64"),
    "lce_1024x15": LceConfig(name="lce_1024x15", n_cand=1024, n_user=15, M=433, K_user=1022,
                             K_cand=1022, N=256, seed=21,
                             description="1024 candidates over 15 users (~70:1), M=433, "
                                         "K=1022+1022 (padded 1024+1024), N=256"),
}


# ---------------------------------------------------------------------------
# Multi-level broadcast ("In-Kernel Broadcast Optimization", §5): a user sees
# several ads vendors and every vendor offers several ads items, so two nested
# broadcast relations with independent, uneven ratios.  The structure is drawn
# top-down: vendors per user, then items per vendor, each 1 + a multinomial
# with Dirichlet(1) weights (uneven, independent at the two levels).  The maps
# the library takes are item_to_vendor and vendor_to_user; ``item_user`` is the
# user of every item as drawn (the structure itself, not a composition of the
# maps), which the oracle's own walk of the maps is checked against.

def draw_hierarchy(n_item: int, n_vendor: int, n_user: int, seed: int, shuffle: bool = False):
    """Returns (item_to_vendor, vendor_to_user, item_user, vendors_per_user, items_per_vendor).

    Unshuffled, both maps are sorted (vendors grouped by user, items by vendor).
    ``shuffle`` relabels the vendors and reorders the items with seeded permutations.
    """
    assert 1 <= n_user <= n_vendor <= n_item
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x4D4C])))
    vpu = 1 + rng.multinomial(n_vendor - n_user, rng.dirichlet(np.ones(n_user)))
    ipv = 1 + rng.multinomial(n_item - n_vendor, rng.dirichlet(np.ones(n_vendor)))
    v2u = np.repeat(np.arange(n_user, dtype=np.int64), vpu)
    i2v = np.repeat(np.arange(n_vendor, dtype=np.int64), ipv)
    vstart = np.concatenate([[0], np.cumsum(vpu)])
    items_of_user = np.array([ipv[vstart[u]:vstart[u + 1]].sum() for u in range(n_user)])
    item_user = np.repeat(np.arange(n_user, dtype=np.int64), items_of_user)
    if shuffle:
        relabel = rng.permutation(n_vendor)          # vendor j becomes relabel[j]
        v2u_new = np.empty_like(v2u)
        v2u_new[relabel] = v2u
        v2u, i2v = v2u_new, relabel[i2v]
        order = rng.permutation(n_item)
        i2v, item_user = i2v[order], item_user[order]
    return (i2v.astype(np.int32), v2u.astype(np.int32), item_user.astype(np.int32),
            vpu.astype(np.int64), ipv.astype(np.int64))


@dataclass(frozen=True)
class MlConfig:
    """Target attention over a user -> vendor -> item hierarchy: every item is a candidate
    with Lq query tokens; the keys and values are the user sequences (lengths uniform in
    [len_lo, len_hi])."""
    name: str
    n_item: int
    n_vendor: int
    n_user: int
    H: int
    D: int
    Lq: int
    seed: int
    len_lo: int
    len_hi: int
    std: float = 1.0
    shuffle: bool = False
    description: str = ""


@dataclass
class MlWorkload:
    cfg: MlConfig
    wl: Workload                 # items as candidates; wl.cand_to_user is ``item_user`` as drawn
    item_to_vendor: np.ndarray   # int32 [n_item]
    vendor_to_user: np.ndarray   # int32 [n_vendor]
    vendors_per_user: np.ndarray = field(repr=False, default=None)
    items_per_vendor: np.ndarray = field(repr=False, default=None)


def ml_generate(cfg: MlConfig) -> MlWorkload:
    """One seeded multi-level workload (q, k, v drawn as ``generate`` draws them)."""
    i2v, v2u, item_user, vpu, ipv = draw_hierarchy(cfg.n_item, cfg.n_vendor, cfg.n_user, cfg.seed,
                                                    cfg.shuffle)
    counts = np.bincount(item_user, minlength=cfg.n_user)
    base = Config(name=cfg.name, n_cand=cfg.n_item, n_user=cfg.n_user, H=cfg.H, D=cfg.D, Lq=cfg.Lq,
                  seed=cfg.seed, std=cfg.std, counts=tuple(int(c) for c in counts), lens="uniform",
                  len_lo=cfg.len_lo, len_hi=cfg.len_hi, description=cfg.description)
    wl = generate(base)
    wl.cand_to_user = item_user.copy()               # the drawn order (sorted unless shuffled)
    return MlWorkload(cfg=cfg, wl=wl, item_to_vendor=i2v, vendor_to_user=v2u,
                      vendors_per_user=vpu, items_per_vendor=ipv)


@dataclass
class LceMlConfig:
    name: str
    n_item: int
    n_vendor: int
    n_user: int
    M: int
    K_user: int
    K_vendor: int
    K_item: int
    N: int
    seed: int
    shuffle: bool = False
    description: str = ""


@dataclass
class LceMlWorkload:
    cfg: LceMlConfig
    W_user: np.ndarray        # bf16 bits [M, Ku8]
    W_vendor: np.ndarray      # bf16 bits [M, Kv8]
    W_item: np.ndarray        # bf16 bits [M, Ki8]
    X_user: np.ndarray        # bf16 bits [n_user, Ku8, N]
    X_vendor: np.ndarray      # bf16 bits [n_vendor, Kv8, N]
    X_item: np.ndarray        # bf16 bits [n_item, Ki8, N]
    item_to_vendor: np.ndarray
    vendor_to_user: np.ndarray
    item_user: np.ndarray = field(repr=False, default=None)


def lce_ml_generate(cfg: LceMlConfig) -> LceMlWorkload:
    """Linear compression over a user -> vendor -> item hierarchy: an item's K input
    embeddings are its user's block, its vendor's block and its own, each zero-padded to a
    multiple of 8; X ~ N(0, 1), W ~ N(0, (0.5 / sqrt(K))^2)."""
    i2v, v2u, item_user, _, _ = draw_hierarchy(cfg.n_item, cfg.n_vendor, cfg.n_user, cfg.seed,
                                               cfg.shuffle)
    std_w = 0.5 / np.sqrt(max(cfg.K_user + cfg.K_vendor + cfg.K_item, 1))

    def padded(tid, shape, pad_axis, valid, std):
        x = _normal_bf16(cfg.seed, tid, shape, std).reshape(shape)
        idx = [slice(None)] * len(shape)
        idx[pad_axis] = slice(valid, None)
        x[tuple(idx)] = 0
        return x

    ku, kv, ki = round_up8(cfg.K_user), round_up8(cfg.K_vendor), round_up8(cfg.K_item)
    return LceMlWorkload(
        cfg=cfg,
        W_user=padded(30, (cfg.M, ku), 1, cfg.K_user, std_w),
        W_vendor=padded(31, (cfg.M, kv), 1, cfg.K_vendor, std_w),
        W_item=padded(32, (cfg.M, ki), 1, cfg.K_item, std_w),
        X_user=padded(33, (cfg.n_user, ku, cfg.N), 1, cfg.K_user, 1.0),
        X_vendor=padded(34, (cfg.n_vendor, kv, cfg.N), 1, cfg.K_vendor, 1.0),
        X_item=padded(35, (cfg.n_item, ki, cfg.N), 1, cfg.K_item, 1.0),
        item_to_vendor=i2v, vendor_to_user=v2u, item_user=item_user)


ML_CONFIGS = {
    "ml_tiny_12x5x2": MlConfig(name="ml_tiny_12x5x2", n_item=12, n_vendor=5, n_user=2, H=2, D=64,
                               Lq=1, seed=50, len_lo=16, len_hi=40,
                               description="12 items over 5 vendors over 2 users, L~U[16,40], "
                                           "H=2 D=64 Lq=1"),
    "ml_1024x60x15": MlConfig(name="ml_1024x60x15", n_item=1024, n_vendor=60, n_user=15, H=4,
                              D=128, Lq=1, seed=51, len_lo=256, len_hi=1024,
                              description="1024 items over 60 vendors over 15 users (uneven "
                                          "ratios), L~U[256,1024], H=4 D=128 Lq=1"),
}

LCE_ML_CONFIGS = {
    "lce_ml_tiny_12x5x2": LceMlConfig(name="lce_ml_tiny_12x5x2", n_item=12, n_vendor=5, n_user=2,
                                      M=37, K_user=13, K_vendor=9, K_item=21, N=64, seed=52,
                                      description="12 items over 5 vendors over 2 users, M=37, "
                                                  "K=13+9+21 (padded 16+16+24), N=64"),
    "lce_ml_1024x60x15": LceMlConfig(name="lce_ml_1024x60x15", n_item=1024, n_vendor=60,
                                     n_user=15, M=433, K_user=1022, K_vendor=510, K_item=1022,
                                     N=256, seed=53,
                                     description="1024 items over 60 vendors over 15 users, "
                                                 "M=433, K=1022+510+1022 (padded 1024+512+1024), "
                                                 "N=256"),
}


CONFIGS = {
    "tiny_8x2": Config(
        name="tiny_8x2", n_cand=8, n_user=2, H=2, D=64, Lq=1, seed=0,
        counts=(5, 3), lens=(16, 24),
        description="2 users, 8 candidates (cand_to_user 0,0,0,0,0,1,1,1), L=16/24, H=2 D=64 Lq=1"),
    "ratio_1024x15": Config(
        name="ratio_1024x15", n_cand=1024, n_user=15, H=4, D=128, Lq=1, seed=1,
        counts="multinomial", lens="uniform", len_lo=256, len_hi=1024,
        description="1024 candidates over 15 users (~70:1), sorted, L~U[256,1024], H=4 D=128 Lq=1"),
    "odd_groups_2048x16": Config(
        name="odd_groups_2048x16", n_cand=2048, n_user=16, H=8, D=128, Lq=4, seed=2,
        counts="zipf", zipf_s=1.1, forced_counts=(1, 1, 3), lens="uniform", len_lo=64, len_hi=4096,
        description="2048 candidates over 16 users, Zipf(1.1) counts with users at 1,1,3, "
                    "L~U[64,4096], H=8 D=128 Lq=4"),
    "extreme_4096x4": Config(
        name="extreme_4096x4", n_cand=4096, n_user=4, H=8, D=128, Lq=8, seed=3, std=0.5,
        counts="multinomial", lens="uniform", len_lo=1024, len_hi=2048,
        description="4096 candidates over 4 users (~1000:1), L~U[1024,2048], H=8 D=128 Lq=8, N(0,0.5)"),
}
for _D in (64, 128):
    for _Lq in (1, 4):
        _n = f"sweep_16384x64_d{_D}_lq{_Lq}"
        CONFIGS[_n] = Config(
            name=_n, n_cand=16384, n_user=64, H=16, D=_D, Lq=_Lq, seed=4,
            counts="multinomial", lens="loguniform", len_lo=128, len_hi=8192,
            description=f"16384 candidates over 64 users, L log-uniform [128,8192], H=16 D={_D} Lq={_Lq}")

# Batches of few users, beside the table above.  Three have fewer units (user, head,
# query tile) than SMs and one unit much longer than the others, so that how a
# unit's keys are spread over SMs decides the time (the key-interleaved kernel,
# ikbo_set_kernel(4), is built for these); the fourth, one user with many
# candidates and short keys, is their counterpart with many short units.
# Explicit counts and lengths; values N(0, 1).
LONG_CONFIGS = {
    "long_user_5000": Config(
        name="long_user_5000", n_cand=1, n_user=1, H=2, D=128, Lq=1, seed=3,
        counts=(1,), lens=(5000,),
        description="1 candidate of 1 user with 5000 keys, H=2 D=128 Lq=1"),
    "long_user_65000": Config(
        name="long_user_65000", n_cand=7, n_user=2, H=2, D=128, Lq=3, seed=77,
        counts=(5, 2), lens=(65000, 300),
        description="7 candidates over 2 users with 65000 and 300 keys, H=2 D=128 Lq=3"),
    "one_user_10000x700": Config(
        name="one_user_10000x700", n_cand=10000, n_user=1, H=4, D=128, Lq=1, seed=9,
        counts=(10000,), lens=(700,),
        description="10000 candidates of 1 user with 700 keys, H=4 D=128 Lq=1"),
    "few_long_82x4": Config(
        name="few_long_82x4", n_cand=82, n_user=4, H=4, D=128, Lq=1, seed=10,
        counts=(20, 50, 3, 9), lens=(12000, 3000, 8000, 500),
        description="82 candidates over 4 users with 12000, 3000, 8000 and 500 keys, "
                    "H=4 D=128 Lq=1"),
}


def attention_config(name: str) -> Config:
    """A target-attention configuration by name, from the table or the long-user set."""
    if name in CONFIGS:
        return CONFIGS[name]
    return LONG_CONFIGS[name]


# The configuration the headline metric is quoted on (1024 candidates / 15 users).
HEADLINE = "ratio_1024x15"
