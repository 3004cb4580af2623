"""Back-to-back calls on unchanged inputs give bit-identical outputs: the kernels are
deterministic, and a race in their pipelines (a stage reused too early, a buffer read
before it landed) would show up as a differing repeat.  Decode runs on the GQA-70B-like
batch (tensor cores, dependent launches after the append) and with split-K partitions
on both paths at both head sizes (at head_dim 64 also with 16 query heads per KV head:
the 32-column paired-heads instance); prefill on a chunked-prefill batch.  With
head_dim-128 operands (head_dim 128, and two paired KV heads per item at 64) the
tensor-core CTAs claim their items as they get free, so which CTA computes an item
changes from call to call: equal bits also show that the result does not depend on
where an item runs."""
import pytest
import torch

import paged_kv_cache_310_gb300 as pkv
import workloads

pytestmark = pytest.mark.gpu


def repeat_equal(call, out, n):
    call()
    torch.cuda.synchronize()
    first = out.clone()
    for i in range(n):
        call()
        torch.cuda.synchronize()
        assert torch.equal(out, first), f"repeat {i} differs"
    assert pkv.device_error() == 0


def test_decode_steps_repeat_bit_identically():
    w = workloads.make_workload(3, canary=False, pool_device="cuda")
    g = w.to("cuda")
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")

    def step():
        pkv.paged_kv_append(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
        pkv.paged_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, w.scale, out,
                                   max_context_len=w.max_context_len)

    repeat_equal(step, out, 60)


@pytest.mark.parametrize("head_dim,num_q_heads", [(128, 32), (64, 32), (64, 128)], ids=["d128", "d64", "d64_g16"])
@pytest.mark.parametrize("path", [pkv.PATH_CUDA_CORE, pkv.PATH_TENSOR_CORE], ids=["cuda_core", "tensor_core"])
def test_split_decode_repeats_bit_identically(path, head_dim, num_q_heads):
    if path == pkv.PATH_CUDA_CORE and num_q_heads // 8 > 8:
        pytest.skip("the CUDA-core path takes up to 8 query heads per KV head")
    w = workloads.random_workload(310_480, num_seqs=24, max_len=3000, min_len=1, num_q_heads=num_q_heads,
                                  num_kv_heads=8, head_dim=head_dim, block_size=16, dtype="bf16", canary=False)
    g = w.to("cuda")
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")

    def call():
        pkv.paged_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, w.scale, out,
                                   max_context_len=w.max_context_len, path=path, partition_tokens=256)

    repeat_equal(call, out, 40)


def test_prefill_repeats_bit_identically():
    w, q, qs = workloads.prefill_workload(310_481, num_seqs=8, max_len=2000, min_len=300, num_q_heads=64,
                                          num_kv_heads=8, block_size=16, dtype="bf16", new_tokens=None,
                                          canary=False)
    g = w.to("cuda")
    qd, qsd = q.cuda(), qs.cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")

    def call():
        pkv.paged_attention_prefill(qd, g.k_cache, g.v_cache, g.block_tables, g.context_lens, qsd, w.scale, out,
                                    max_context_len=w.max_context_len)

    repeat_equal(call, out, 20)
