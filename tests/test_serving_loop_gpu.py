"""Decode steps driven by the host block manager, on the GPU, checked end to end.

The manager hands out slots and copy-on-write pairs; the library's kernels apply them
and decode.  Independently, the test keeps every sequence's K/V history as a plain
contiguous tensor; the oracle's attention over those histories (identity block tables
on a freshly built pool) is the reference.  Sequences are forked (parallel sampling),
finished (their blocks reused) and started during the run.
"""
import random

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_310_gb300 as pkv
from paged_kv_cache_310_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu

BS, HKV, HQ, D = 16, 4, 16, 128
DT = torch.bfloat16


def reference(histories, q, ids):
    """Oracle attention over contiguous histories laid out with identity block tables."""
    lens = [histories[s][0].shape[1] for s in ids]
    nblk = [-(-n // BS) for n in lens]
    kc = torch.full((max(1, sum(nblk)), HKV, BS, D), float("nan"), dtype=DT)
    vc = kc.clone()
    tables = torch.full((len(ids), max(nblk)), -1, dtype=torch.int32)
    base = 0
    for i, s in enumerate(ids):
        K, V = histories[s]
        for j in range(nblk[i]):
            rows = min(BS, lens[i] - j * BS)
            kc[base + j, :, :rows] = K[:, j * BS:j * BS + rows]
            vc[base + j, :, :rows] = V[:, j * BS:j * BS + rows]
            tables[i, j] = base + j
        base += nblk[i]
    return oracle.attention_decode(q, kc, vc, tables, torch.tensor(lens, dtype=torch.int32), D ** -0.5)


@pytest.mark.parametrize("path", [pkv.PATH_CUDA_CORE, pkv.PATH_TENSOR_CORE], ids=["cuda_core", "tensor_core"])
def test_block_manager_driven_decode_steps(path):
    rng = random.Random(310_600)
    gen = torch.Generator().manual_seed(310_601)
    NB = 400
    bm = BlockManager(NB, BS)
    kc = torch.full((NB, HKV, BS, D), float("nan"), dtype=DT, device="cuda")
    vc = kc.clone()
    hist = {}
    next_id = 0

    def new_sequence(n):
        nonlocal next_id
        s = next_id
        next_id += 1
        bm.add_sequence(s, n)
        K = torch.randn(HKV, n, D, generator=gen).to(DT)
        V = torch.randn(HKV, n, D, generator=gen).to(DT)
        hist[s] = (K, V)
        # write the prompt through the append kernel, one slot per prompt token
        tables, _ = bm.block_tables([s])
        slots = torch.tensor([int(tables[0, j // BS]) * BS + j % BS for j in range(n)], dtype=torch.int64)
        if n:
            pkv.paged_kv_append(K.permute(1, 0, 2).contiguous().cuda(), V.permute(1, 0, 2).contiguous().cuda(),
                                slots.cuda(), kc, vc)

    for _ in range(5):
        new_sequence(rng.randint(1, 300))
    copies = 0
    for step in range(14):
        live = sorted(hist)
        if step % 3 == 1:                       # parallel sampling: fork two sequences
            for parent in rng.sample(live, 2):
                bm.fork(parent, next_id)
                hist[next_id] = tuple(t.clone() for t in hist[parent])
                next_id += 1
        if step % 4 == 3:                       # one finishes, a new request arrives
            done = rng.choice(live)
            bm.free_sequence(done)
            del hist[done]
            new_sequence(rng.randint(1, 200))
        ids = sorted(hist)
        slots, pairs = bm.append(ids)
        copies += pairs.shape[0]
        if pairs.numel():
            pkv.paged_block_copy(pairs.cuda(), kc, vc, host_pairs=pairs)
        k_new = torch.randn(len(ids), HKV, D, generator=gen).to(DT)
        v_new = torch.randn(len(ids), HKV, D, generator=gen).to(DT)
        pkv.paged_kv_append(k_new.cuda(), v_new.cuda(), slots.cuda(), kc, vc)
        for i, s in enumerate(ids):
            K, V = hist[s]
            hist[s] = (torch.cat([K, k_new[i][:, None]], 1), torch.cat([V, v_new[i][:, None]], 1))
        q = torch.randn(len(ids), HQ, D, generator=gen).to(DT)
        tables, lens = bm.block_tables(ids)
        out = torch.empty((len(ids), HQ, D), dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode(q.cuda(), kc, vc, tables.cuda(), lens.cuda(), D ** -0.5, out,
                                   max_context_len=int(lens.max()), path=path, partition_tokens=128)
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        ref = reference(hist, q, ids)
        err = np.abs(out.cpu().double().numpy() - ref).max()
        assert err <= 2e-3, f"step {step}: max-abs error {err:.3g}"
        st = bm.stats()
        assert st["logical_tokens"] == sum(h[0].shape[1] for h in hist.values())
    assert copies > 0                            # forks made sharers write into shared blocks
