"""Pins of the float64 oracle to things other than itself (CPU only).

Each test ties the oracle to something the pages or mathematics fix: exhaustive
element decoding against numpy/torch, a pure-Python brute force that builds each
sequence's K/V contiguously first, a library softmax for identity block tables, closed
forms (one token, two tokens, uniform keys, hand-worked golden files) and the
invariants paging must keep (physical placement, sharing by reference, copy-on-write).
"""
import math
import os
import random

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pool(dtype, NB, Hkv, bs, D, fill=float("nan")):
    return torch.full((NB, Hkv, bs, D), fill, dtype=dtype)


# --------------------------------------------------------------------------------------
# element decoders: exhaustive over all 2^16 bit patterns

def test_f16_decoder_exhaustive():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.float16)
    got = oracle.decode_elements(t)
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_bf16_decoder_exhaustive():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    got = oracle.decode_elements(t)
    ref = t.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_f32_decoder_sample():
    t = torch.randn(10000, generator=torch.Generator().manual_seed(1))
    assert np.array_equal(oracle.decode_elements(t), t.double().numpy())


# --------------------------------------------------------------------------------------
# pure-Python brute force: contiguous per-sequence K/V first, blocks assigned after

def _brute_case(rng, dtype):
    S = rng.randint(1, 4)
    bs = rng.choice([1, 2, 4, 16])
    G = rng.choice([1, 2, 4])
    Hkv = rng.randint(1, 2)
    Hq = Hkv * G
    D = rng.choice([1, 3, 8])
    lens = [rng.randint(0, 40) for _ in range(S)]
    nblocks = [math.ceil(n / bs) for n in lens]
    NB = sum(nblocks) + rng.randint(0, 5)
    phys = list(range(NB))
    rng.shuffle(phys)
    # contiguous logical K/V per sequence, values exactly representable in the dtype
    gen = torch.Generator().manual_seed(rng.randint(0, 2**31))

    def draw(*shape):
        return torch.randn(shape, generator=gen).to(dtype)

    q = draw(S, Hq, D)
    Kc = [draw(Hkv, n, D) for n in lens]
    Vc = [draw(Hkv, n, D) for n in lens]
    kc, vc = _pool(dtype, NB, Hkv, bs, D), _pool(dtype, NB, Hkv, bs, D)
    MB = max(1, max(nblocks))
    tables = torch.full((S, MB), -1, dtype=torch.int32)
    it = iter(phys)
    for s in range(S):
        for i in range(nblocks[s]):
            b = next(it)
            tables[s, i] = b
            for r in range(bs):
                j = i * bs + r
                if j < lens[s]:
                    kc[b, :, r, :] = Kc[s][:, j, :]
                    vc[b, :, r, :] = Vc[s][:, j, :]
    scale = rng.choice([1.0 / math.sqrt(D), 0.7, 1.3])
    return dict(q=q, Kc=Kc, Vc=Vc, kc=kc, vc=vc, tables=tables,
                lens=torch.tensor(lens, dtype=torch.int32), scale=scale, G=G)


def _brute_attention(case):
    q = case["q"].double().tolist()
    S, Hq = len(q), len(q[0])
    out = []
    for s in range(S):
        K = case["Kc"][s].double().tolist()
        V = case["Vc"][s].double().tolist()
        rows = []
        for h in range(Hq):
            g = h // case["G"]
            n = len(K[g])
            D = len(q[s][h])
            if n == 0:
                rows.append([0.0] * D)
                continue
            sc = [case["scale"] * math.fsum(q[s][h][d] * K[g][j][d] for d in range(D)) for j in range(n)]
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            l = math.fsum(w)
            rows.append([math.fsum(w[j] * V[g][j][d] for j in range(n)) / l for d in range(D)])
        out.append(rows)
    return np.array(out, dtype=np.float64)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_bruteforce_random_tiny(dtype):
    rng = random.Random({torch.float32: 310_101, torch.float16: 310_102, torch.bfloat16: 310_103}[dtype])
    for _ in range(70):
        c = _brute_case(rng, dtype)
        got = oracle.attention_decode(c["q"], c["kc"], c["vc"], c["tables"], c["lens"], c["scale"])
        ref = _brute_attention(c)
        assert got.shape == ref.shape
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_bruteforce_config1():
    w = workloads.make_workload(1)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    got = oracle.attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    # rebuild contiguous K/V per sequence by walking the table in Python
    G = w.num_q_heads // w.num_kv_heads
    Kc, Vc = [], []
    for s in range(w.num_seqs):
        n = int(w.context_lens[s])
        rows_k = torch.stack([kc[int(w.block_tables[s, j // w.block_size]), :, j % w.block_size, :]
                              for j in range(n)], dim=1)
        rows_v = torch.stack([vc[int(w.block_tables[s, j // w.block_size]), :, j % w.block_size, :]
                              for j in range(n)], dim=1)
        Kc.append(rows_k)
        Vc.append(rows_v)
    ref = _brute_attention(dict(q=w.q, Kc=Kc, Vc=Vc, scale=w.scale, G=G))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    assert np.isfinite(got).all()


# --------------------------------------------------------------------------------------
# identity block table == plain attention on a contiguous buffer (library softmax)

@pytest.mark.parametrize("G,bs,M,lens", [(1, 4, 6, [5, 24, 13]), (4, 4, 6, [5, 24, 13]), (2, 64, 3, [5, 130, 64])],
                         ids=["G1-bs4", "G4-bs4", "G2-bs64"])
def test_identity_table_matches_library_attention(G, bs, M, lens):
    gen = torch.Generator().manual_seed(310_201)
    S, Hkv, D = 3, 2, 16
    Hq = Hkv * G
    lens = torch.tensor(lens, dtype=torch.int32)
    kc = torch.randn(S * M, Hkv, bs, D, generator=gen, dtype=torch.float64).float()
    vc = torch.randn(S * M, Hkv, bs, D, generator=gen, dtype=torch.float64).float()
    q = torch.randn(S, Hq, D, generator=gen).float()
    tables = torch.arange(S * M, dtype=torch.int32).reshape(S, M)
    got = oracle.attention_decode(q, kc, vc, tables, lens, 0.25)
    for s in range(S):
        n = int(lens[s])
        # contiguous view: sequence s occupies blocks s*M .. s*M+M-1 in order
        K = kc[s * M:(s + 1) * M].permute(1, 0, 2, 3).reshape(Hkv, M * bs, D)[:, :n].double().numpy()
        V = vc[s * M:(s + 1) * M].permute(1, 0, 2, 3).reshape(Hkv, M * bs, D)[:, :n].double().numpy()
        for h in range(Hq):
            p = scipy.special.softmax(0.25 * (K[h // G] @ q[s, h].double().numpy()))
            np.testing.assert_allclose(got[s, h], p @ V[h // G], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------------------
# invariants of paging

def test_permutation_invariance_bit_exact():
    w = workloads.make_workload(4)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.block_copy(w.cow_pairs, kc, vc)
    oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    sel = slice(0, 12)
    base = oracle.attention_decode(w.q[sel], kc, vc, w.block_tables[sel], w.context_lens[sel], w.scale)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(5))
    kp, vp = torch.empty_like(kc), torch.empty_like(vc)
    kp[perm] = kc
    vp[perm] = vc
    bt = w.block_tables.clone()
    ok = bt >= 0
    bt[ok] = perm[bt[ok].long()].to(torch.int32)
    moved = oracle.attention_decode(w.q[sel], kp, vp, bt[sel], w.context_lens[sel], w.scale)
    assert np.array_equal(base, moved)
    assert np.isfinite(base).all()


def test_shared_vs_copied_bit_exact():
    """Ten tables pointing at one prefix read it exactly as ten private copies would."""
    w = workloads.make_workload(4)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    users = w.meta["users"]
    nprefix = w.meta["prefix_tokens"] // w.block_size
    bt = w.block_tables[:users].clone()
    assert (bt[:, :nprefix] == bt[0, :nprefix]).all()
    shared = oracle.attention_decode(w.q[:users], kc, vc, bt, w.context_lens[:users], w.scale)
    # give every user but the first private copies of the prefix blocks
    extra = (users - 1) * nprefix
    NB = w.num_blocks
    kx = torch.cat([kc, torch.empty((extra,) + tuple(kc.shape[1:]), dtype=kc.dtype)])
    vx = torch.cat([vc, torch.empty((extra,) + tuple(vc.shape[1:]), dtype=vc.dtype)])
    pairs = []
    for u in range(1, users):
        for i in range(nprefix):
            dst = NB + (u - 1) * nprefix + i
            pairs.append((int(bt[u, i]), dst))
            bt[u, i] = dst
    oracle.block_copy(torch.tensor(pairs), kx, vx)
    copied = oracle.attention_decode(w.q[:users], kx, vx, bt, w.context_lens[:users], w.scale)
    assert np.array_equal(shared, copied)


def test_copy_on_write_divergence():
    """After the copy and the writer's append, sharers still see the old block."""
    w = workloads.make_workload(4)
    users = w.meta["users"]
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.block_copy(w.cow_pairs, kc, vc)
    # beams 0..2 of tree 0 write into copies; beam 3 writes the original last block
    beams = slice(users, users + 4)
    before_lens = w.context_lens[beams] - 1
    pre = oracle.attention_decode(w.q[beams], kc, vc, w.block_tables[beams], before_lens, w.scale)
    # all four beams see identical K/V before anyone writes
    first = oracle.gather(kc, vc, w.block_tables[beams][0:1], before_lens[0:1])
    for b in range(1, 4):
        other = oracle.gather(kc, vc, w.block_tables[beams][b:b + 1], before_lens[b:b + 1])
        for x, y in zip(first, other):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    # beam 0 alone appends into its private copy
    k1, v1 = kc.clone(), vc.clone()
    oracle.kv_append(w.k_new[users:users + 1], w.v_new[users:users + 1], w.slot_mapping[users:users + 1], k1, v1)
    post = oracle.attention_decode(w.q[beams], k1, v1, w.block_tables[beams], before_lens, w.scale)
    assert np.array_equal(pre, post)  # nobody's first L tokens changed
    after = oracle.attention_decode(w.q[beams][:1], k1, v1, w.block_tables[beams][:1],
                                    w.context_lens[beams][:1], w.scale)
    assert np.isfinite(after).all() and not np.array_equal(after[0], pre[0])
    # the other beams' copies still hold NaN in the written row: they did not see it
    slot = int(w.slot_mapping[users])
    for b in (1, 2, 3):
        other = int(w.slot_mapping[users + b])
        assert other != slot
        blk, row = divmod(other, w.block_size)
        assert torch.isnan(k1[blk, :, row]).all()


# --------------------------------------------------------------------------------------
# closed forms

def test_single_token_returns_v0_exactly():
    gen = torch.Generator().manual_seed(3)
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        kc = torch.randn(5, 2, 8, 32, generator=gen).to(dtype)
        vc = torch.randn(5, 2, 8, 32, generator=gen).to(dtype)
        q = torch.randn(3, 4, 32, generator=gen).to(dtype)
        tables = torch.tensor([[3], [0], [4]], dtype=torch.int32)
        out = oracle.attention_decode(q, kc, vc, tables, torch.tensor([1, 1, 1], dtype=torch.int32), 0.3)
        for s in range(3):
            for h in range(4):
                assert np.array_equal(out[s, h], vc[int(tables[s, 0]), h // 2, 0].double().numpy())


def test_two_tokens_closed_form():
    gen = torch.Generator().manual_seed(4)
    kc = torch.randn(4, 1, 2, 16, generator=gen)
    vc = torch.randn(4, 1, 2, 16, generator=gen)
    q = torch.randn(1, 1, 16, generator=gen)
    tables = torch.tensor([[2]], dtype=torch.int32)
    out = oracle.attention_decode(q, kc, vc, tables, torch.tensor([2], dtype=torch.int32), 0.5)
    qd = q[0, 0].double()
    s0 = 0.5 * float(qd @ kc[2, 0, 0].double())
    s1 = 0.5 * float(qd @ kc[2, 0, 1].double())
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    ref = sig(s0 - s1) * vc[2, 0, 0].double().numpy() + sig(s1 - s0) * vc[2, 0, 1].double().numpy()
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-13, atol=1e-14)


def test_uniform_keys_give_mean_of_values():
    gen = torch.Generator().manual_seed(6)
    n, bs = 37, 8
    kc = torch.randn(6, 1, bs, 24, generator=gen)
    kc[:] = kc[0, 0, 0]  # every key identical
    vc = torch.randn(6, 1, bs, 24, generator=gen)
    q = torch.randn(2, 1, 24, generator=gen)
    tables = torch.tensor([[5, 1, 3, 0, 2], [4, 0, 1, 2, 3]], dtype=torch.int32)
    out = oracle.attention_decode(q, kc, vc, tables, torch.tensor([n, 9], dtype=torch.int32), 0.09)
    for s, m in ((0, n), (1, 9)):
        rows = [vc[int(tables[s, j // bs]), 0, j % bs].double().numpy() for j in range(m)]
        np.testing.assert_allclose(out[s, 0], np.mean(rows, axis=0), rtol=1e-12, atol=1e-14)
    # scale 0 makes any keys uniform
    kr = torch.randn(6, 1, bs, 24, generator=gen)
    out0 = oracle.attention_decode(q, kr, vc, tables, torch.tensor([n, 9], dtype=torch.int32), 0.0)
    np.testing.assert_allclose(out0, out, rtol=1e-12, atol=1e-14)


def test_empty_context_gives_zeros():
    q = torch.randn(2, 2, 8)
    kc = torch.full((3, 2, 4, 8), float("nan"))
    out = oracle.attention_decode(q, kc, kc.clone(), torch.full((2, 1), -1, dtype=torch.int32),
                                  torch.tensor([0, 0], dtype=torch.int32), 1.0)
    assert np.array_equal(out, np.zeros((2, 2, 8)))


def _read_golden(name):
    d = {"k": [], "v": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, val = [x.strip() for x in line.split("=")]
            if key in ("k", "v"):
                d[key].append([float(x) for x in val.split()])
            else:
                d[key] = [float(x) for x in val.split()]
    return d


def test_golden_worked_example():
    g = _read_golden("worked_two_block_gqa.txt")
    NB, bs, D = int(g["num_blocks"][0]), int(g["block_size"][0]), int(g["head_dim"][0])
    kc = _pool(torch.float32, NB, 1, bs, D)
    vc = _pool(torch.float32, NB, 1, bs, D)
    for rows, pool in ((g["k"], kc), (g["v"], vc)):
        for tok, b, r, *vals in rows:
            pool[int(b), 0, int(r)] = torch.tensor(vals)
    q = torch.tensor([[g["q0"], g["q1"]]], dtype=torch.float32)
    tables = torch.tensor([[int(x) for x in g["table"]]], dtype=torch.int32)
    out = oracle.attention_decode(q, kc, vc, tables, torch.tensor([int(g["context_len"][0])], dtype=torch.int32),
                                  g["scale"][0])
    np.testing.assert_allclose(out[0, 0], g["expect0"], rtol=0, atol=g["tolerance0"][0])
    np.testing.assert_allclose(out[0, 1], g["expect1"], rtol=0, atol=g["tolerance1"][0])


def test_golden_shared_system_prompt_layout():
    g = _read_golden("shared_system_prompt.txt")
    w = workloads.make_workload(4)
    users, n = int(g["users"][0]), int(g["shared_blocks"][0])
    assert w.meta["users"] == users and w.meta["prefix_tokens"] == int(g["prompt_tokens"][0])
    assert w.block_size == int(g["block_size"][0])
    prefix = w.block_tables[:users, :n]
    assert (prefix == prefix[0]).all() and len(set(prefix[0].tolist())) == n
    # stored once: the prefix occupies n physical blocks, not users * n
    assert len(set(prefix.flatten().tolist())) == n
    assert users * n == int(g["blocks_without_sharing"][0])
    assert (w.block_tables[:users, n] != w.block_tables[0, n]).sum() == users - 1


# --------------------------------------------------------------------------------------
# partition merge

@pytest.mark.parametrize("part", [1, 5, 16, 64, 1000])
def test_partition_merge_matches_single_pass(part):
    w = workloads.random_workload(310_300 + part, num_seqs=5, max_len=150, num_q_heads=4, num_kv_heads=2,
                                  head_dim=32, block_size=8, dtype="bf16")
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    full = oracle.attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    m, l, o = oracle.attention_partitions(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, part)
    merged = oracle.merge_partitions(m, l, o)
    np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-13)
    # a partition's own normalised output is attention over its token range alone
    s = int(torch.argmax(w.context_lens))
    if int(w.context_lens[s]) > part:
        np.testing.assert_array_less(0, l[s, :, 0])


# --------------------------------------------------------------------------------------
# append, block copy and gather against a dictionary model of the pool

def test_append_and_copy_match_dictionary_model():
    rng = random.Random(7)
    NB, Hkv, bs, D = 9, 2, 4, 8
    for dtype in (torch.float32, torch.bfloat16, torch.float16):
        kc = torch.randn(NB, Hkv, bs, D).to(dtype)
        vc = torch.randn(NB, Hkv, bs, D).to(dtype)
        model_k = {(b, g, r): kc[b, g, r].clone() for b in range(NB) for g in range(Hkv) for r in range(bs)}
        model_v = {(b, g, r): vc[b, g, r].clone() for b in range(NB) for g in range(Hkv) for r in range(bs)}
        T = 6
        slots = rng.sample(range(NB * bs), T - 1) + [-1]
        k = torch.randn(T, Hkv, D).to(dtype)
        v = torch.randn(T, Hkv, D).to(dtype)
        for t, sl in enumerate(slots):
            if sl >= 0:
                for g in range(Hkv):
                    model_k[(sl // bs, g, sl % bs)] = k[t, g].clone()
                    model_v[(sl // bs, g, sl % bs)] = v[t, g].clone()
        oracle.kv_append(k, v, torch.tensor(slots), kc, vc)
        pairs = [(1, 4), (7, 0), (4, 2)]  # applied in order: 2 receives the new 4
        for src, dst in pairs:
            for g in range(Hkv):
                for r in range(bs):
                    model_k[(dst, g, r)] = model_k[(src, g, r)].clone()
                    model_v[(dst, g, r)] = model_v[(src, g, r)].clone()
        oracle.block_copy(torch.tensor(pairs), kc, vc)
        for key, val in model_k.items():
            assert torch.equal(kc[key].view(torch.int16 if dtype != torch.float32 else torch.int32),
                               val.view(torch.int16 if dtype != torch.float32 else torch.int32))
        for key, val in model_v.items():
            assert torch.equal(vc[key], val) or (torch.isnan(vc[key]) & torch.isnan(val)).all()


def test_append_rejects_out_of_range_slot():
    kc = torch.zeros(2, 1, 4, 8)
    with pytest.raises(ValueError):
        oracle.kv_append(torch.zeros(1, 1, 8), torch.zeros(1, 1, 8), torch.tensor([8]), kc, kc.clone())


def test_gather_walks_block_table():
    w = workloads.random_workload(11, num_seqs=4, max_len=30, num_q_heads=2, num_kv_heads=2, head_dim=8,
                                  block_size=4, dtype="f16", min_len=1)
    kg, vg = oracle.gather(w.k_cache, w.v_cache, w.block_tables, w.context_lens)
    for s in range(w.num_seqs):
        for j in range(int(w.context_lens[s])):
            b = int(w.block_tables[s, j // 4])
            assert torch.equal(kg[s, :, j].view(torch.int16), w.k_cache[b, :, j % 4].view(torch.int16))
            assert torch.equal(vg[s, :, j].view(torch.int16), w.v_cache[b, :, j % 4].view(torch.int16))
        assert (kg[s, :, int(w.context_lens[s]):] == 0).all()


def test_nan_canaries_never_read():
    """Every unowned row is NaN; the oracle's outputs stay finite on every workload shape."""
    for cfg in (1, 4):
        w = workloads.make_workload(cfg)
        kc, vc = w.k_cache.clone(), w.v_cache.clone()
        oracle.block_copy(w.cow_pairs, kc, vc)
        oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
        sel = slice(0, min(w.num_seqs, 14))
        out = oracle.attention_decode(w.q[sel], kc, vc, w.block_tables[sel], w.context_lens[sel], w.scale)
        assert np.isfinite(out).all()
        # without the append, the last token's slot is NaN and poisons the output
        bad = oracle.attention_decode(w.q[sel], w.k_cache, w.v_cache, w.block_tables[sel],
                                      w.context_lens[sel], w.scale)
        assert np.isnan(bad).any()


def test_config_shapes_follow_the_pages():
    w1 = workloads.make_workload(1)
    assert w1.context_lens.tolist() == [2, 16, 17, 34] and w1.num_blocks == 64
    w4 = workloads.make_workload(4)
    assert w4.cow_pairs.shape == (24, 2)
    assert all(p % 16 for p in w4.meta["beam_prompts"])
    assert len(set(w4.cow_pairs[:, 1].tolist())) == 24
