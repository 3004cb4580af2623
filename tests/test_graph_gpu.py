"""The library's calls inside a CUDA graph: a decode step (append, decode with split-K
partitions and the merge, on both paths) and a chunked-prefill call are captured once
and replayed with new query values; every replay must match an eager call on the same
inputs bit for bit (the kernels are deterministic).  Small batches are launch-bound,
and a captured step is how a serving loop removes the per-call host cost."""
import pytest
import torch

import paged_kv_cache_310_gb300 as pkv
import workloads

pytestmark = pytest.mark.gpu


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the capture: first-call setup happens here
        fn()
        fn()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("path", [pkv.PATH_CUDA_CORE, pkv.PATH_TENSOR_CORE], ids=["cuda_core", "tensor_core"])
def test_decode_step_replays_in_a_graph(path, head_dim):
    w = workloads.random_workload(310_470, num_seqs=9, max_len=1500, min_len=1, num_q_heads=16, num_kv_heads=4,
                                  head_dim=head_dim, block_size=16, dtype="bf16", canary=False)
    g = w.to("cuda")
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")

    def step():
        pkv.paged_kv_append(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
        pkv.paged_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, w.scale, out,
                                   max_context_len=w.max_context_len, path=path, partition_tokens=256)

    graph = capture(step)
    gen = torch.Generator(device="cuda").manual_seed(310_471)
    for _ in range(3):
        g.q.copy_(torch.randn(g.q.shape, generator=gen, device="cuda").to(g.q.dtype))
        graph.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        step()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.equal(replayed, out)


def test_prefill_replays_in_a_graph():
    w, q, qs = workloads.prefill_workload(310_472, num_seqs=4, max_len=600, min_len=50, num_q_heads=32,
                                          num_kv_heads=4, block_size=16, dtype="bf16", new_tokens=None,
                                          canary=False)
    g = w.to("cuda")
    qd, qsd = q.cuda(), qs.cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")

    def call():
        pkv.paged_attention_prefill(qd, g.k_cache, g.v_cache, g.block_tables, g.context_lens, qsd, w.scale, out,
                                    max_context_len=w.max_context_len)

    graph = capture(call)
    gen = torch.Generator(device="cuda").manual_seed(310_473)
    for _ in range(3):
        qd.copy_(torch.randn(qd.shape, generator=gen, device="cuda").to(qd.dtype))
        graph.replay()
        torch.cuda.synchronize()
        replayed = out.clone()
        call()
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert torch.equal(replayed, out)
