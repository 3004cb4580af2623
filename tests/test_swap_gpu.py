"""Swap of blocks between the device pool and pinned CPU memory (preemption), on the GPU.

Round trips are bit-exact; a sequence preempted while its blocks are reused by another
request decodes, once restored into different blocks, to exactly the same bits.
"""
import pytest
import torch

import paged_kv_cache_310_gb300 as pkv
from paged_kv_cache_310_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu


def same_bytes(a, b):
    return torch.equal(a.contiguous().cpu().view(torch.uint8), b.contiguous().cpu().view(torch.uint8))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_swap_round_trip_bit_exact(dtype):
    g = torch.Generator(device="cuda").manual_seed(310_700)
    NB, H, BS, D = 50, 4, 16, 64 if dtype == torch.float32 else 128
    kc = torch.randn((NB, H, BS, D), generator=g, device="cuda").to(dtype)
    vc = torch.randn((NB, H, BS, D), generator=g, device="cuda").to(dtype)
    kc[3, 1, 5, 7] = float("nan")  # payloads survive as bytes
    k0, v0 = kc.clone(), vc.clone()
    ids = torch.tensor([7, 3, 41, 0, 19], dtype=torch.int64)
    hk = torch.empty((5, H, BS, D), dtype=dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    pkv.paged_block_swap_out(ids.cuda(), kc, vc, hk, hv)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    assert same_bytes(hk, k0[ids.cuda()]) and same_bytes(hv, v0[ids.cuda()])
    kc[ids.cuda()] = float("nan")
    vc[ids.cuda()] = float("nan")
    new_ids = torch.tensor([44, 2, 3, 30, 8], dtype=torch.int64)   # restore elsewhere, overlapping 3
    pkv.paged_block_swap_in(new_ids.cuda(), hk, hv, kc, vc)
    torch.cuda.synchronize()
    assert same_bytes(kc[new_ids.cuda()], k0[ids.cuda()]) and same_bytes(vc[new_ids.cuda()], v0[ids.cuda()])


def test_swap_refuses_pageable_memory():
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    pageable = torch.empty((1, 2, 16, 128), dtype=torch.bfloat16)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_block_swap_out(torch.tensor([1], device="cuda"), kc, kc.clone(), pageable, pageable.clone())
    assert "pageable" in str(e.value)


@pytest.mark.parametrize("path", [pkv.PATH_CUDA_CORE, pkv.PATH_TENSOR_CORE], ids=["cuda_core", "tensor_core"])
def test_preempt_and_resume_exactly(path):
    gen = torch.Generator().manual_seed(310_701)
    NB, H, HQ, BS, D = 200, 2, 8, 16, 128
    bm = BlockManager(NB, BS)
    kc = torch.full((NB, H, BS, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()

    def fill(seq, n):
        bm.add_sequence(seq, n)
        t, _ = bm.block_tables([seq])
        slots = torch.tensor([int(t[0, j // BS]) * BS + j % BS for j in range(n)], dtype=torch.int64)
        k = torch.randn(n, H, D, generator=gen).bfloat16()
        v = torch.randn(n, H, D, generator=gen).bfloat16()
        pkv.paged_kv_append(k.cuda(), v.cuda(), slots.cuda(), kc, vc)

    for s, n in ((1, 700), (2, 333), (3, 901)):
        fill(s, n)
    q = torch.randn(3, HQ, D, generator=gen).bfloat16().cuda()

    def decode(ids):
        tables, lens = bm.block_tables(ids)
        out = torch.empty((len(ids), HQ, D), dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode(q[: len(ids)], kc, vc, tables.cuda(), lens.cuda(), D ** -0.5, out,
                                   max_context_len=int(lens.max()), path=path, partition_tokens=256)
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        return out

    before = decode([1, 2, 3])
    # preempt sequence 2: its blocks go to pinned CPU memory and back to the free list
    blocks = bm.swap_out(2)
    ids = torch.tensor(blocks, dtype=torch.int64)
    hk = torch.empty((len(blocks), H, BS, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    pkv.paged_block_swap_out(ids.cuda(), kc, vc, hk, hv)
    # a new request takes (and overwrites) the freed blocks
    fill(4, 600)
    taken, _ = bm.block_tables([4])
    assert set(blocks) & set(taken[0].tolist())
    # restore into whatever blocks are free now
    fresh = bm.swap_in(2)
    assert fresh != blocks
    pkv.paged_block_swap_in(torch.tensor(fresh, dtype=torch.int64).cuda(), hk, hv, kc, vc)
    after = decode([1, 2, 3])
    assert torch.equal(before, after)       # bit-identical: placement never changes the result
    assert bm.stats()["swapped"] == 0
