"""Seeded synthetic inputs for the paged KV cache hot path.

This module is shared by the CUDA path's tests and benchmark and by the oracle's
tests.  It draws random numbers and lays out block tables, slots and copy-on-write
pairs; it contains none of the attention arithmetic.

Every workload describes one decode step:

1. ``cow_pairs`` (src, dst) -- the copy-on-write copies made before the step writes
   into a block it shares ("anthology-of-the-sota note-023", Concepts).
2. ``k_new``/``v_new`` go to ``slot_mapping`` -- one new token per sequence at logical
   position ``context_lens[s] - 1`` ("Efficient Memory Management ... with
   PagedAttention", How It Works: blocks of e.g. 16 tokens, filled as tokens are
   generated).
3. decode attention of ``q`` over ``context_lens[s]`` tokens through ``block_tables``.

Layouts: pools ``[num_blocks, num_kv_heads, block_size, head_dim]``; q ``[S, Hq, D]``;
block_tables int32 ``[S, max_blocks]`` padded with -1; context_lens int32 ``[S]``;
slot = physical_block * block_size + row, int64.

Values: q, K and V are N(0, 1) drawn in float32 and rounded to the workload dtype.
Physical blocks are handed out by a seeded ``randperm`` over a pool 1.25x the blocks
in use (64 blocks for the tiny case).  With ``canary=True`` every pool row that no
sequence owns before the step (including the tail of each partly filled block, the
slot the append will write, and copy-on-write destinations) is NaN, so any read of
a row that should not be read poisons the result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEED_BASE = 310_000

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}

# The five workloads, numbered as in the method's test plan.
CONFIGS = {
    1: dict(name="tiny decode: 4 seqs, lens {1,15,16,33}+1, bs16, 64-block pool, 4/4 heads, D64, f32",
            kind="tiny", num_q_heads=4, num_kv_heads=4, head_dim=64, dtype="f32", block_size=16),
    2: dict(name="Llama-2-7B-like decode: 64 seqs, 32/32 heads, D128, bf16, lens U[128,2048], bs16",
            kind="uniform", num_seqs=64, lo=128, hi=2048, num_q_heads=32, num_kv_heads=32,
            head_dim=128, dtype="bf16", block_size=16),
    3: dict(name="GQA-70B-like decode: 128 seqs, 64/8 heads, D128, bf16, lens U[512,4096], bs16",
            kind="uniform", num_seqs=128, lo=512, hi=4096, num_q_heads=64, num_kv_heads=8,
            head_dim=128, dtype="bf16", block_size=16),
    4: dict(name="shared 4000-token prefix x10 + 8 beam trees x4 with copy-on-write, 32/8 heads, D128, bf16, bs16",
            kind="shared", num_q_heads=32, num_kv_heads=8, head_dim=128, dtype="bf16", block_size=16),
    5: dict(name="long-context mix: 256 seqs, lognormal(median 1024, sigma 1) in [1,32768], bs32, 32/8 heads, D128, f16",
            kind="lognormal", num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
            dtype="f16", block_size=32),
}


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: torch.Tensor      # int32 [S], tokens attended (after the append)
    block_tables: torch.Tensor      # int32 [S, max_blocks], -1 padded
    q: torch.Tensor                 # [S, Hq, D]
    k_cache: torch.Tensor           # [NB, Hkv, bs, D], state before the step
    v_cache: torch.Tensor
    k_new: torch.Tensor             # [T, Hkv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # int64 [T]
    cow_pairs: torch.Tensor         # int64 [n, 2] (src, dst)
    scale: float
    unique_blocks: int = 0          # physical blocks referenced by any table
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.numel())

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    def to(self, device) -> "Workload":
        fields = {k: getattr(self, k) for k in self.__dataclass_fields__}
        for k, v in fields.items():
            if isinstance(v, torch.Tensor):
                fields[k] = v.to(device)
        return Workload(**fields)

    def kv_bytes(self) -> int:
        """K+V bytes decode reads once per step: sum_s L_s * 2 * Hkv * D * elem."""
        e = torch.empty((), dtype=self.dtype).element_size()
        return int(self.context_lens.sum()) * 2 * self.num_kv_heads * self.head_dim * e


def _randn(shape, gen, dtype, device="cpu"):
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(dtype)


def build_from_layout(*, name, seed, dtype, num_q_heads, num_kv_heads, head_dim, block_size,
                      ctx, block_keys, owned_rows, cow, num_blocks=None, canary=True,
                      pool_device="cpu", gen=None, meta=None, shuffle=True) -> Workload:
    """Materialise a workload from a logical layout.

    ctx[s]          -- tokens sequence s attends over (its append writes position ctx[s]-1).
    block_keys[s]   -- one hashable key per logical block of s; equal keys share one
                       physical block.
    owned_rows[key] -- rows of that block holding valid K/V before the step.
    cow             -- list of (src_key, dst_key) copied before the append.
    """
    g = gen if gen is not None else torch.Generator().manual_seed(seed)
    tdtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
    S = len(ctx)
    order = []
    seen = set()
    for keys in block_keys:
        for k in keys:
            if k not in seen:
                seen.add(k)
                order.append(k)
    for _, dst in cow:
        assert dst in seen, "copy-on-write destinations must appear in a table"
    unique = len(order)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(1.25 * unique))
    assert num_blocks >= unique
    # shuffle=False lays blocks out in logical order: each sequence contiguous, the
    # identity-table arrangement used to measure what the indirection costs
    perm = torch.randperm(num_blocks, generator=g) if shuffle else torch.arange(num_blocks)
    phys = {k: int(perm[i]) for i, k in enumerate(order)}

    max_blocks = max((len(k) for k in block_keys), default=1)
    tables = torch.full((S, max(1, max_blocks)), -1, dtype=torch.int32)
    for s, keys in enumerate(block_keys):
        assert len(keys) == math.ceil(ctx[s] / block_size), (s, len(keys), ctx[s])
        for i, k in enumerate(keys):
            tables[s, i] = phys[k]

    q = _randn((S, num_q_heads, head_dim), g, tdtype)
    k_new = _randn((S, num_kv_heads, head_dim), g, tdtype)
    v_new = _randn((S, num_kv_heads, head_dim), g, tdtype)
    slots = torch.full((S,), -1, dtype=torch.int64)
    for s in range(S):
        if ctx[s] == 0:
            continue
        pos = ctx[s] - 1
        slots[s] = phys[block_keys[s][pos // block_size]] * block_size + pos % block_size

    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    if pool_device == "cpu":
        pool_gen = g
    else:
        pool_gen = torch.Generator(device=pool_device).manual_seed(seed + 7919)
    k_cache = torch.empty(shape, dtype=tdtype, device=pool_device)
    v_cache = torch.empty(shape, dtype=tdtype, device=pool_device)
    step = max(1, (64 << 20) // (num_kv_heads * block_size * head_dim))
    for cache in (k_cache, v_cache):
        for b0 in range(0, num_blocks, step):
            b1 = min(num_blocks, b0 + step)
            cache[b0:b1] = _randn((b1 - b0,) + shape[1:], pool_gen, tdtype, pool_device)
    if canary:
        owned = torch.zeros((num_blocks, block_size), dtype=torch.bool)
        for k, rows in owned_rows.items():
            owned[phys[k], list(rows)] = True
        mask = (~owned).to(pool_device)[:, None, :, None].expand(shape)
        k_cache.masked_fill_(mask, float("nan"))
        v_cache.masked_fill_(mask, float("nan"))

    pairs = torch.tensor([[phys[a], phys[b]] for a, b in cow], dtype=torch.int64).reshape(-1, 2)
    return Workload(name=name, dtype=tdtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, block_size=block_size, num_blocks=num_blocks,
                    context_lens=torch.tensor(ctx, dtype=torch.int32), block_tables=tables, q=q,
                    k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new, slot_mapping=slots,
                    cow_pairs=pairs, scale=1.0 / math.sqrt(head_dim), unique_blocks=unique,
                    meta=dict(meta or {}))


def private_layout(ctx, block_size):
    """Each sequence owns its blocks; rows before position ctx-1 are valid."""
    keys, owned = [], {}
    for s, n in enumerate(ctx):
        ks = [("seq", s, i) for i in range(math.ceil(n / block_size))]
        keys.append(ks)
        for i, k in enumerate(ks):
            owned[k] = [r for r in range(block_size) if i * block_size + r < n - 1]
    return keys, owned


def make_workload(config: int, *, canary: bool = True, pool_device="cpu", shuffle: bool = True,
                  **overrides) -> Workload:
    """One of the five numbered workloads (seed 310000 + config).

    overrides replace fields of the workload (e.g. block_size); shuffle=False assigns
    physical blocks in logical order instead of by a seeded permutation.
    """
    c = dict(CONFIGS[config])
    c.update(overrides)
    seed = SEED_BASE + config
    g = torch.Generator().manual_seed(seed)
    bs = c["block_size"]
    # a workload with fields changed is named as such (its figures are not the base one's)
    changed = {k: v for k, v in sorted(overrides.items()) if CONFIGS[config].get(k) != v}
    name = c["name"]
    if changed:
        name += " [with " + ", ".join(f"{k}={v}" for k, v in changed.items()) + "]"
    common = dict(name=name, seed=seed, dtype=c["dtype"], num_q_heads=c["num_q_heads"],
                  num_kv_heads=c["num_kv_heads"], head_dim=c["head_dim"], block_size=bs,
                  canary=canary, pool_device=pool_device, gen=g, shuffle=shuffle)
    kind = c["kind"]
    if kind == "tiny":
        before = [1, 15, 16, 33]
        ctx = [n + 1 for n in before]
        keys, owned = private_layout(ctx, bs)
        return build_from_layout(ctx=ctx, block_keys=keys, owned_rows=owned, cow=[],
                                 num_blocks=64, meta=dict(lens_before_append=before), **common)
    if kind == "uniform":
        S = c["num_seqs"]
        ctx = torch.randint(c["lo"], c["hi"] + 1, (S,), generator=g).tolist()
        keys, owned = private_layout(ctx, bs)
        return build_from_layout(ctx=ctx, block_keys=keys, owned_rows=owned, cow=[], **common)
    if kind == "lognormal":
        S = c["num_seqs"]
        z = torch.randn(S, generator=g, dtype=torch.float64)
        ctx = [int(min(32768, max(1, round(math.exp(math.log(1024.0) + 1.0 * float(x)))))) for x in z]
        keys, owned = private_layout(ctx, bs)
        return build_from_layout(ctx=ctx, block_keys=keys, owned_rows=owned, cow=[], **common)
    if kind == "shared":
        return _shared_prefix(c, g, common)
    raise ValueError(kind)


def _shared_prefix(c, g, common) -> Workload:
    """Ten sequences sharing a 4000-token system prompt plus eight 4-wide beam trees.

    The prompt is 250 full blocks of 16 tokens shared by reference; each sequence's
    suffix (uniform 1..512 tokens) and its new token live in private blocks.  Each
    beam tree's prompt (uniform 100..2000 tokens, redrawn while a multiple of 16) ends
    in a partly filled shared block; the new token goes into that block, so beams
    0..2 first copy it (copy-on-write, the copy happens while another beam still
    shares it) and beam 3 writes the original.
    """
    bs = c["block_size"]
    prefix, n_users, n_trees, width = 4000, 10, 8, 4
    keys, owned, ctx, cow = [], {}, [], []
    n_prefix_blocks = prefix // bs
    for i in range(n_prefix_blocks):
        owned[("prefix", i)] = list(range(bs))
    suffix = torch.randint(1, 513, (n_users,), generator=g).tolist()
    for u in range(n_users):
        n = prefix + suffix[u] + 1
        ks = [("prefix", i) for i in range(n_prefix_blocks)]
        for i in range(n_prefix_blocks, math.ceil(n / bs)):
            k = ("user", u, i)
            ks.append(k)
            owned[k] = [r for r in range(bs) if i * bs + r < n - 1]
        keys.append(ks)
        ctx.append(n)
    prompts = []
    for t in range(n_trees):
        p = int(torch.randint(100, 2001, (1,), generator=g))
        while p % bs == 0:
            p = int(torch.randint(100, 2001, (1,), generator=g))
        prompts.append(p)
        nb = math.ceil(p / bs)
        for i in range(nb):
            owned[("tree", t, i)] = [r for r in range(bs) if i * bs + r < p]
        for w in range(width):
            ks = [("tree", t, i) for i in range(nb)]
            if w < width - 1:
                dst = ("cow", t, w)
                cow.append((("tree", t, nb - 1), dst))
                ks[-1] = dst
                owned.setdefault(dst, [])
            keys.append(ks)
            ctx.append(p + 1)
    meta = dict(prefix_tokens=prefix, users=n_users, suffix=suffix, beam_prompts=prompts,
                beam_width=width)
    return build_from_layout(ctx=ctx, block_keys=keys, owned_rows=owned, cow=cow, meta=meta, **common)


def random_workload(seed, *, num_seqs, max_len, num_q_heads, num_kv_heads, head_dim, block_size,
                    dtype="f32", min_len=0, canary=True, extra_blocks=3) -> Workload:
    """A small random workload for edge-case tests (lengths uniform in [min_len, max_len]).

    A sequence of length 0 has no blocks and its new token has the padding slot -1.
    """
    g = torch.Generator().manual_seed(seed)
    ctx = torch.randint(min_len, max_len + 1, (num_seqs,), generator=g).tolist()
    keys, owned = private_layout(ctx, block_size)
    unique = sum(len(k) for k in keys)
    return build_from_layout(name=f"random seed {seed}", seed=seed, dtype=dtype,
                             num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                             block_size=block_size, ctx=ctx, block_keys=keys, owned_rows=owned,
                             cow=[], num_blocks=unique + extra_blocks, canary=canary, gen=g)


def prefill_workload(seed, *, num_seqs, max_len, num_q_heads, num_kv_heads, head_dim=128, block_size=16,
                     dtype="bf16", min_len=1, new_tokens=None, canary=True, pool_device="cpu"):
    """A pool whose every context row is valid, plus new tokens for multi-token attention.

    Context lengths are uniform in [min_len, max_len]; sequence s brings
    new_tokens(s, L) new tokens (default: uniform in [1, L]), the last ones of its
    context.  Returns (workload, q [T, Hq, D], query_start int32 [S+1]).
    """
    g = torch.Generator().manual_seed(seed)
    tdtype = DTYPES[dtype]
    ctx = torch.randint(min_len, max_len + 1, (num_seqs,), generator=g).tolist()
    keys, _ = private_layout(ctx, block_size)
    owned = {}
    for s, n in enumerate(ctx):
        for i, k in enumerate(keys[s]):
            owned[k] = [r for r in range(block_size) if i * block_size + r < n]
    unique = sum(len(k) for k in keys)
    w = build_from_layout(name=f"prefill seed {seed}", seed=seed, dtype=dtype, num_q_heads=num_q_heads,
                          num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=block_size, ctx=ctx,
                          block_keys=keys, owned_rows=owned, cow=[], num_blocks=unique + 3, canary=canary,
                          gen=g, pool_device=pool_device)
    if new_tokens is None:
        nq = [int(torch.randint(0, n, (1,), generator=g)) + 1 if n else 0 for n in ctx]
    else:
        nq = [min(n, int(new_tokens(s, n))) for s, n in enumerate(ctx)]
    qs = [0]
    for n in nq:
        qs.append(qs[-1] + n)
    q = _randn((qs[-1], num_q_heads, head_dim), g, tdtype)
    return w, q, torch.tensor(qs, dtype=torch.int32)
