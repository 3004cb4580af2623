"""Prepared calls (PreparedCall): arguments checked and marshalled once, then replayed.
A replay must do exactly what the plain call does -- the same kernels on the same
buffers -- so its results are compared bit for bit with the plain call's, after the
inputs' contents change between replays and on another stream."""
import pytest
import torch

import paged_kv_cache_310_gb300 as pkv
import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,path", [("bf16", pkv.PATH_AUTO), ("f32", pkv.PATH_TENSOR_CORE),
                                        ("f16", pkv.PATH_CUDA_CORE)])
def test_prepared_step_matches_plain_calls(dtype, path):
    w = workloads.make_workload(4, canary=False)  # copy-on-write pairs, shared prefix, beams
    if dtype != "bf16":
        w = workloads.random_workload(310_700, num_seqs=9, max_len=1500, min_len=1, num_q_heads=32, num_kv_heads=4,
                                      head_dim=128, block_size=16, dtype=dtype, canary=False)
    a, b = w.to("cuda"), w.to("cuda")
    out_a = torch.empty(a.q.shape, dtype=torch.float32, device="cuda")
    out_b = torch.empty_like(out_a)
    L = w.max_context_len
    calls = []
    if b.cow_pairs.numel():
        calls.append(pkv.prepare_block_copy(b.cow_pairs, b.k_cache, b.v_cache, host_pairs=w.cow_pairs))
    calls.append(pkv.prepare_kv_append(b.k_new, b.v_new, b.slot_mapping, b.k_cache, b.v_cache))
    calls.append(pkv.prepare_attention_decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.context_lens, b.scale,
                                              out_b, max_context_len=L, path=path))
    side = torch.cuda.Stream()
    for step in range(3):
        # new queries and new tokens each step, written into the same buffers
        gen = torch.Generator(device="cuda").manual_seed(step)
        for x_a, x_b in ((a.q, b.q), (a.k_new, b.k_new), (a.v_new, b.v_new)):
            x_a.copy_(torch.randn(x_a.shape, generator=gen, device="cuda").to(x_a.dtype))
            x_b.copy_(x_a)
        if a.cow_pairs.numel():
            pkv.paged_block_copy(a.cow_pairs, a.k_cache, a.v_cache, host_pairs=w.cow_pairs)
        pkv.paged_kv_append(a.k_new, a.v_new, a.slot_mapping, a.k_cache, a.v_cache)
        pkv.paged_attention_decode(a.q, a.k_cache, a.v_cache, a.block_tables, a.context_lens, a.scale, out_a,
                                   max_context_len=L, path=path)
        torch.cuda.synchronize()
        if step == 1:  # replay on another stream, given as a raw handle
            side.wait_stream(torch.cuda.current_stream())
            for call in calls:
                call(side.cuda_stream)
            torch.cuda.current_stream().wait_stream(side)
        else:
            for call in calls:
                call()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.equal(out_a, out_b)
        assert torch.equal(a.k_cache.view(torch.uint8), b.k_cache.view(torch.uint8))
        assert torch.equal(a.v_cache.view(torch.uint8), b.v_cache.view(torch.uint8))


def test_prepared_decode_requires_a_host_bound():
    w = workloads.random_workload(310_701, num_seqs=2, max_len=64, min_len=1, num_q_heads=8, num_kv_heads=2,
                                  head_dim=128, block_size=16, dtype="bf16", canary=False)
    g = w.to("cuda")
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(pkv.PagedKVError):
        pkv.prepare_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                                     max_context_len=None)
    with pytest.raises(pkv.PagedKVError):  # argument checks happen when the call is prepared
        pkv.prepare_kv_append(g.k_new, g.v_new, g.slot_mapping.to(torch.int32), g.k_cache, g.v_cache)
