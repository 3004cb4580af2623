"""Pins of the oracle's causal multi-token (prefill) attention (CPU only)."""
import math
import random

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads


def _case(seed, dtype="bf16", S=3, max_ctx=70, Hq=4, Hkv=2, D=16, bs=8):
    """A random pool plus, per sequence, a number of new tokens at the end of its context."""
    w = workloads.random_workload(seed, num_seqs=S, max_len=max_ctx, min_len=1, num_q_heads=Hq, num_kv_heads=Hkv,
                                  head_dim=D, block_size=bs, dtype=dtype, canary=True)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    oracle.kv_append(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    rng = random.Random(seed)
    # every row of the context must be valid: fill the NaN canaries of owned rows
    lens = w.context_lens.tolist()
    g = torch.Generator().manual_seed(seed)
    for s, L in enumerate(lens):
        for j in range(L):
            b = int(w.block_tables[s, j // bs])
            if torch.isnan(kc[b, :, j % bs].float()).any():
                kc[b, :, j % bs] = torch.randn(Hkv, D, generator=g).to(kc.dtype)
                vc[b, :, j % bs] = torch.randn(Hkv, D, generator=g).to(vc.dtype)
    nq = [rng.randint(1, L) for L in lens]
    qs = torch.tensor([0] + list(np.cumsum(nq)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), Hq, D, generator=g).to(kc.dtype)
    return w, kc, vc, q, qs


def test_one_new_token_is_decode():
    w, kc, vc, _, _ = _case(310_800)
    qs = torch.arange(w.num_seqs + 1, dtype=torch.int32)
    pre = oracle.attention_prefill(w.q, kc, vc, w.block_tables, w.context_lens, qs, w.scale)
    dec = oracle.attention_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    assert np.array_equal(pre, dec)


@pytest.mark.parametrize("seed", range(5))
def test_prefill_bruteforce(seed):
    # the last case has 64-token blocks, contexts of 146 and 103 tokens (three and two)
    w, kc, vc, q, qs = _case([310_810, 310_811, 310_812, 310_813, 310_821][seed],
                             dtype=["f32", "bf16", "f16", "bf16", "f16"][seed],
                             Hq=[2, 4, 4, 8, 4][seed], Hkv=[2, 1, 2, 2, 2][seed], S=[3, 3, 3, 3, 2][seed],
                             max_ctx=[70, 70, 70, 70, 150][seed], bs=[8, 8, 8, 8, 64][seed])
    got = oracle.attention_prefill(q, kc, vc, w.block_tables, w.context_lens, qs, w.scale)
    G = w.num_q_heads // w.num_kv_heads
    bs = w.block_size
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        n = int(qs[s + 1] - qs[s])
        K = [[kc[int(w.block_tables[s, j // bs]), g, j % bs].double().tolist() for j in range(L)]
             for g in range(w.num_kv_heads)]
        V = [[vc[int(w.block_tables[s, j // bs]), g, j % bs].double().tolist() for j in range(L)]
             for g in range(w.num_kv_heads)]
        for i in range(n):
            pos = L - n + i
            for h in range(w.num_q_heads):
                qv = q[int(qs[s]) + i, h].double().tolist()
                sc = [w.scale * math.fsum(a * b for a, b in zip(qv, K[h // G][j])) for j in range(pos + 1)]
                m = max(sc)
                e = [math.exp(x - m) for x in sc]
                l = math.fsum(e)
                want = [math.fsum(e[j] * V[h // G][j][d] for j in range(pos + 1)) / l for d in range(w.head_dim)]
                np.testing.assert_allclose(got[int(qs[s]) + i, h], want, rtol=1e-12, atol=1e-12)


def test_causality():
    """Changing K/V after position p leaves the output of the token at p unchanged."""
    w, kc, vc, q, qs = _case(310_820, max_ctx=60)
    base = oracle.attention_prefill(q, kc, vc, w.block_tables, w.context_lens, qs, w.scale)
    s = int(torch.argmax(w.context_lens))
    L, n = int(w.context_lens[s]), int(qs[s + 1] - qs[s])
    assert n >= 2
    cut = L - 1  # perturb the last token only
    b, r = int(w.block_tables[s, cut // w.block_size]), cut % w.block_size
    k2, v2 = kc.clone(), vc.clone()
    k2[b, :, r] += 1.0
    v2[b, :, r] -= 2.0
    moved = oracle.attention_prefill(q, k2, v2, w.block_tables, w.context_lens, qs, w.scale)
    rows_before = slice(int(qs[s]), int(qs[s + 1]) - 1)
    assert np.array_equal(base[rows_before], moved[rows_before])
    assert not np.array_equal(base[int(qs[s + 1]) - 1], moved[int(qs[s + 1]) - 1])


def test_identity_tables_match_library_masked_softmax():
    g = torch.Generator().manual_seed(310_830)
    bs, M, D, Hq, Hkv = 4, 8, 8, 2, 1
    L, n = 29, 11
    kc = torch.randn(M, Hkv, bs, D, generator=g)
    vc = torch.randn(M, Hkv, bs, D, generator=g)
    q = torch.randn(n, Hq, D, generator=g)
    tables = torch.arange(M, dtype=torch.int32)[None]
    got = oracle.attention_prefill(q, kc, vc, tables, torch.tensor([L], dtype=torch.int32),
                                   torch.tensor([0, n], dtype=torch.int32), 0.3)
    K = kc.permute(1, 0, 2, 3).reshape(Hkv, M * bs, D)[:, :L].double().numpy()
    V = vc.permute(1, 0, 2, 3).reshape(Hkv, M * bs, D)[:, :L].double().numpy()
    pos = np.arange(L - n, L)
    mask = np.arange(L)[None, :] > pos[:, None]                  # key after the query: hidden
    for h in range(Hq):
        sc = 0.3 * q[:, h].double().numpy() @ K[0].T
        sc[mask] = -np.inf
        np.testing.assert_allclose(got[:, h], scipy.special.softmax(sc, axis=1) @ V[0], rtol=1e-12, atol=1e-13)
