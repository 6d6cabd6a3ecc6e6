"""Seeded synthetic workloads shaped like the InferScale evaluation.

The pages (InferScale, arXiv 2607.27090, "Results"/"Resultados"/"결과") evaluate
on LoCoMo with Llama-3.1-8B, Mistral-7B and Qwen2.5-7B, retrieval budgets k from
5 to 50 and up to 100 concurrent users.  LoCoMo and trained weights are not
available, so the five workloads below stand in for it with the same KV shapes,
fact lengths of tens of tokens, the same k and the same concurrency.

Everything here is input generation: lengths, unit embeddings, query
embeddings, segment start positions and block tables come from
``numpy.random.default_rng(seed)``; keys and values come from the counter-based
generator in ``synth.kvgen`` (host) / ``synth/csrc/synthgen.cu`` (device).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

from . import kvgen


@dataclass(frozen=True)
class RopeSpec:
    theta: float
    style: int = 0            # 0 = NeoX half split (i, i + D/2), 1 = interleaved (2i, 2i+1)
    scaling: int = 0          # 0 = none, 1 = Llama-3.1 frequency scaling
    factor: float = 1.0
    low_freq_factor: float = 1.0
    high_freq_factor: float = 1.0
    original_max_pos: int = 0


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_layers: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str                      # "f32" | "bf16" | "f16"
    rope: RopeSpec
    n_users: int
    facts_per_user: int
    length_dist: tuple                 # ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    emb_dim: int
    emb_dtype: str                     # "f16" | "f32"
    n_queries: int
    k: int
    query_kind: str                    # "random" | "planted"
    start: tuple                       # ("const", s) | ("uniform", lo, hi)
    block_size: int
    tokens_cap: int                    # per-request segment capacity the block table covers
    block_layout: str                  # "permutation" | "free_list"
    seed: int
    query_noise: float = 0.1
    queries_share_user: bool = False   # all queries ask the same user's store
    num_blocks_fixed: int = 0          # only for block_layout == "permutation"

    @property
    def n_facts(self) -> int:
        return self.n_users * self.facts_per_user

    @property
    def token_elems(self) -> int:
        """Elements of K (or of V) per token: L * H * D."""
        return self.num_layers * self.num_kv_heads * self.head_dim

    @property
    def elt_bytes(self) -> int:
        return 4 if self.kv_dtype == "f32" else 2

    def with_(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


LLAMA31_ROPE = RopeSpec(theta=5.0e5, style=0, scaling=1, factor=8.0,
                        low_freq_factor=1.0, high_freq_factor=4.0, original_max_pos=8192)

SPECS = {
    # Tiny CPU-checkable case.
    "tiny": WorkloadSpec(
        name="tiny", num_layers=1, num_kv_heads=2, head_dim=64, kv_dtype="f32",
        rope=RopeSpec(theta=1.0e4), n_users=1, facts_per_user=64,
        length_dist=("uniform", 4, 16), emb_dim=64, emb_dtype="f32", n_queries=1, k=4,
        query_kind="random", start=("const", 8), block_size=16, tokens_cap=4 * 16,
        block_layout="permutation", num_blocks_fixed=32, seed=1),
    # Llama-3.1-8B KV shape, one request, k = 50.
    "llama31_8b": WorkloadSpec(
        name="llama31_8b", num_layers=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
        rope=LLAMA31_ROPE, n_users=1, facts_per_user=2000, length_dist=("uniform", 10, 40),
        emb_dim=1024, emb_dtype="f16", n_queries=1, k=50, query_kind="planted",
        start=("const", 32), block_size=16, tokens_cap=50 * 40, block_layout="free_list",
        seed=2),
    # Mistral-7B KV shape, one request, k swept over {5, 10, 20, 50}.
    "mistral_7b": WorkloadSpec(
        name="mistral_7b", num_layers=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
        rope=RopeSpec(theta=1.0e6), n_users=1, facts_per_user=2000,
        length_dist=("uniform", 10, 40), emb_dim=1024, emb_dtype="f16", n_queries=1, k=50,
        query_kind="planted", start=("const", 32), block_size=16, tokens_cap=50 * 40,
        block_layout="free_list", seed=3),
    # Qwen2.5-7B KV shape, 100 users with their own stores, one query each.
    "qwen25_7b_100u": WorkloadSpec(
        name="qwen25_7b_100u", num_layers=28, num_kv_heads=4, head_dim=128, kv_dtype="bf16",
        rope=RopeSpec(theta=1.0e6), n_users=100, facts_per_user=300,
        length_dist=("uniform", 10, 40), emb_dim=1024, emb_dtype="f16", n_queries=100, k=50,
        query_kind="planted", start=("const", 32), block_size=16, tokens_cap=50 * 40,
        block_layout="free_list", seed=4),
    # Qwen3-14B KV shape (the pages' larger model): 40 layers, 8 KV heads,
    # head_dim 128, theta 1e6, otherwise as the Llama-3.1-8B request.
    "qwen3_14b": WorkloadSpec(
        name="qwen3_14b", num_layers=40, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
        rope=RopeSpec(theta=1.0e6), n_users=1, facts_per_user=2000,
        length_dist=("uniform", 10, 40), emb_dim=1024, emb_dtype="f16", n_queries=1, k=50,
        query_kind="planted", start=("const", 32), block_size=16, tokens_cap=50 * 40,
        block_layout="free_list", seed=6),
    # Capacity stress on the Llama-3.1-8B KV shape (~105 GB store).
    "capacity": WorkloadSpec(
        name="capacity", num_layers=32, num_kv_heads=8, head_dim=128, kv_dtype="bf16",
        rope=LLAMA31_ROPE, n_users=1, facts_per_user=32000,
        length_dist=("lognormal", 20.0, 0.668, 4, 128), emb_dim=1024, emb_dtype="f16",
        n_queries=64, k=200, query_kind="planted", start=("uniform", 0, 4096), block_size=16,
        tokens_cap=8192, block_layout="free_list", queries_share_user=True, seed=5),
}


@dataclass
class Workload:
    spec: WorkloadSpec
    lengths: np.ndarray          # int32 [n_facts], global fact order (user-major)
    fact_user: np.ndarray        # int32 [n_facts]
    tok_base: np.ndarray         # int64 [n_facts], generator token index of each fact's first token
    emb: np.ndarray              # [n_facts][E], float16 or float32
    queries: np.ndarray          # [Q][E], float16 or float32
    users: np.ndarray            # int32 [Q]
    planted: np.ndarray          # int32 [Q], source fact of a planted query (-1 if random)
    seg_start: np.ndarray        # int32 [Q]
    block_table: np.ndarray      # int32 [Q][max_blocks]; -1 = unassigned
    num_blocks: int
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.lengths.sum())

    def user_facts(self, u: int) -> np.ndarray:
        """Global fact indices of user u, in insertion order."""
        return np.nonzero(self.fact_user == u)[0].astype(np.int64)

    def token_kv(self, f: int, t: int, stream: int) -> np.ndarray:
        """K (stream 0) or V (stream 1) of token t of fact f: [L][H][D] in storage encoding."""
        s = self.spec
        first = (int(self.tok_base[f]) + int(t)) * s.token_elems
        flat = kvgen.kv_elements(s.seed, stream, first, s.token_elems, s.kv_dtype)
        return flat.reshape(s.num_layers, s.num_kv_heads, s.head_dim)

    def fact_kv(self, f: int, stream: int) -> np.ndarray:
        """K (stream 0) or V (stream 1) of fact f: [len][L][H][D] in storage encoding."""
        s = self.spec
        n = int(self.lengths[f]) * s.token_elems
        flat = kvgen.kv_elements(s.seed, stream, int(self.tok_base[f]) * s.token_elems, n,
                                 s.kv_dtype)
        return flat.reshape(int(self.lengths[f]), s.num_layers, s.num_kv_heads, s.head_dim)


def _lengths(spec: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    d = spec.length_dist
    n = spec.n_facts
    if d[0] == "uniform":
        return rng.integers(d[1], d[2] + 1, size=n).astype(np.int32)
    if d[0] == "lognormal":
        _, median, sigma, lo, hi = d
        x = rng.lognormal(mean=np.log(median), sigma=sigma, size=n)
        return np.clip(np.rint(x), lo, hi).astype(np.int32)
    raise ValueError(d)


def _unit_rows(rng: np.random.Generator, n: int, e: int, dtype) -> np.ndarray:
    out = np.empty((n, e), dtype=dtype)
    for s in range(0, n, 4096):
        z = rng.standard_normal((min(n, s + 4096) - s, e))
        z /= np.linalg.norm(z, axis=1, keepdims=True)
        out[s:s + z.shape[0]] = z.astype(dtype)
    return out


def generate(spec: WorkloadSpec) -> Workload:
    rng = np.random.default_rng(spec.seed)
    lengths = _lengths(spec, rng)
    fact_user = np.repeat(np.arange(spec.n_users, dtype=np.int32), spec.facts_per_user)
    tok_base = np.zeros(spec.n_facts, dtype=np.int64)
    tok_base[1:] = np.cumsum(lengths[:-1].astype(np.int64))
    edt = np.float16 if spec.emb_dtype == "f16" else np.float32
    emb = _unit_rows(rng, spec.n_facts, spec.emb_dim, edt)

    Q = spec.n_queries
    if spec.queries_share_user or spec.n_users == 1:
        users = np.zeros(Q, dtype=np.int32)
    else:
        assert Q == spec.n_users
        users = np.arange(Q, dtype=np.int32)
    planted = np.full(Q, -1, dtype=np.int32)
    if spec.query_kind == "random":
        queries = _unit_rows(rng, Q, spec.emb_dim, edt)
    else:
        queries = np.empty((Q, spec.emb_dim), dtype=edt)
        for q in range(Q):
            u = int(users[q])
            f = u * spec.facts_per_user + int(rng.integers(0, spec.facts_per_user))
            planted[q] = f
            z = emb[f].astype(np.float64) + rng.normal(0.0, spec.query_noise, spec.emb_dim)
            queries[q] = (z / np.linalg.norm(z)).astype(edt)

    if spec.start[0] == "const":
        seg_start = np.full(Q, spec.start[1], dtype=np.int32)
    else:
        seg_start = rng.integers(spec.start[1], spec.start[2], size=Q).astype(np.int32)

    bs = spec.block_size
    if spec.block_layout == "permutation":
        num_blocks = spec.num_blocks_fixed
        block_table = np.stack([rng.permutation(num_blocks).astype(np.int32) for _ in range(Q)])
    else:
        max_blocks = int((int(seg_start.max()) + spec.tokens_cap - 1) // bs + 1)
        first = seg_start // bs
        last = (seg_start + spec.tokens_cap - 1) // bs
        counts = (last - first + 1).astype(np.int64)
        num_blocks = int(1 + counts.sum())            # physical block 0 is the shared dummy
        free_list = rng.permutation(np.arange(1, num_blocks, dtype=np.int32))
        block_table = np.full((Q, max_blocks), -1, dtype=np.int32)
        pos = 0
        for r in range(Q):
            wholly_before = np.arange(max_blocks) * bs + bs <= seg_start[r]
            block_table[r, wholly_before] = 0
            c = int(counts[r])
            block_table[r, first[r]:first[r] + c] = free_list[pos:pos + c]
            pos += c
    return Workload(spec=spec, lengths=lengths, fact_user=fact_user, tok_base=tok_base,
                    emb=emb, queries=queries, users=users, planted=planted,
                    seg_start=seg_start, block_table=block_table, num_blocks=num_blocks)


def get(name: str, **overrides) -> Workload:
    spec = SPECS[name]
    if overrides:
        spec = spec.with_(**overrides)
    return generate(spec)


def cache_shape(spec: WorkloadSpec, num_blocks: int) -> tuple:
    """Paged KV cache [L][2][num_blocks][block_size][H][D] (vLLM-style, K then V per layer)."""
    return (spec.num_layers, 2, num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim)


CANARY_BITS = {"bf16": 0x7FA5, "f16": 0x7E5A, "f32": 0x7FC0A5A5, "e4m3": 0x7F}
"""Bit pattern every cache element holds before injection (a NaN payload that
no finite rotated key or copied value can equal)."""
