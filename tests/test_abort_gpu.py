"""The decode and prefill kernels' abort path, forced without any fault.

Every pipeline wait in those kernels is bounded; when one runs out the kernel stops
issuing work, waits (each wait again bounded) for the copies and MMAs it still has in
flight, frees its tensor memory, records PKV_ERR_DEVICE_TIMEOUT in the device flag and
returns.  Here the bound is lowered to 1 us through the library's diagnostic setter,
far below what a healthy pipeline wait takes, so a normal call on valid inputs gives
up part-way.  The test checks that the call returns promptly with the timeout status
and that the next call with the normal bound, on the same context, matches the oracle.
"""
import time

import pytest
import torch

import oracle
import paged_kv_cache_310_gb300 as pkv
import workloads
from parity_bounds import check_close

pytestmark = pytest.mark.gpu

FORCED_LIMIT_NS = 1_000


def _decode(w, g, path, part):
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                               max_context_len=w.max_context_len, path=path, partition_tokens=part)
    return out


# (path, dtype, head_dim, query heads, KV heads): at head_dim 64 two KV heads share an item
# (16 S columns at 4 query heads per KV head, 32 columns and two K stages at 16), and an
# odd number of KV heads keeps one head per item in the fixed order
CASES = [(pkv.PATH_CUDA_CORE, "bf16", 128, 16, 4), (pkv.PATH_TENSOR_CORE, "bf16", 128, 16, 4),
         (pkv.PATH_TENSOR_CORE, "f32", 128, 16, 4), (pkv.PATH_TENSOR_CORE, "bf16", 64, 16, 4),
         (pkv.PATH_TENSOR_CORE, "bf16", 64, 64, 4), (pkv.PATH_TENSOR_CORE, "bf16", 64, 48, 3)]


@pytest.mark.parametrize("path,dtype,head_dim,hq,hkv", CASES,
                         ids=["cuda_core", "tensor_core", "tensor_core_f32", "tensor_core_d64_paired",
                              "tensor_core_d64_paired_32cols", "tensor_core_d64_one_head"])
def test_decode_gives_up_and_the_context_survives(path, dtype, head_dim, hq, hkv):
    w = workloads.random_workload(310_480, num_seqs=8, max_len=2500, min_len=300, num_q_heads=hq, num_kv_heads=hkv,
                                  head_dim=head_dim, block_size=16, dtype=dtype, canary=False)
    g = w.to("cuda")
    assert pkv.device_error() == 0
    pkv.set_wait_limit(FORCED_LIMIT_NS)
    try:
        t0 = time.perf_counter()
        _decode(w, g, path, 512)
        status = pkv.device_error()  # synchronises the stream
        elapsed = time.perf_counter() - t0
    finally:
        pkv.set_wait_limit(0)
    assert status == 6, f"expected PKV_ERR_DEVICE_TIMEOUT, got {status}"
    assert elapsed < 10.0
    assert pkv.device_error() == 0  # read-and-clear
    # the same call with the normal bound, on the same context
    ref = oracle.attention_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    out = _decode(w, g, path, 512)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    check_close(out, ref, w.dtype)


def test_prefill_gives_up_and_the_context_survives():
    w, q, qs = workloads.prefill_workload(310_481, num_seqs=5, max_len=1500, min_len=300, num_q_heads=32,
                                          num_kv_heads=4, block_size=16, dtype="bf16", canary=False)
    g = w.to("cuda")
    qd, qsd = q.cuda(), qs.cuda()

    def run():
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        pkv.paged_attention_prefill(qd, g.k_cache, g.v_cache, g.block_tables, g.context_lens, qsd, w.scale, out,
                                    max_context_len=w.max_context_len)
        return out

    assert pkv.device_error() == 0
    pkv.set_wait_limit(FORCED_LIMIT_NS)
    try:
        t0 = time.perf_counter()
        run()
        status = pkv.device_error()
        elapsed = time.perf_counter() - t0
    finally:
        pkv.set_wait_limit(0)
    assert status == 6, f"expected PKV_ERR_DEVICE_TIMEOUT, got {status}"
    assert elapsed < 10.0
    ref = oracle.attention_prefill(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, qs, w.scale)
    out = run()
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    check_close(out, ref, w.dtype)


def test_wait_limit_setter_rejects_too_long():
    with pytest.raises(pkv.PagedKVError):
        pkv.set_wait_limit(6_000_000_000)
    pkv.set_wait_limit(0)
