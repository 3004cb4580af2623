"""paged_attention_decode_no_alloc: decode for callers that must not allocate device
memory (allocator callbacks, serving paths that may not hit out-of-memory, runtimes
that only hand over pre-registered buffers).  Its scratch is the library's built-in
per-GPU array, so two calls in a row must each give the same result as the
workspace-taking entry point on the same inputs.

This file is collected last on purpose: when it fails, a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_310_gb300 as pkv
import workloads

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}


def _with_workspace(w, g, path, part):
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                               max_context_len=w.max_context_len, path=path, partition_tokens=part)
    return out


def _no_alloc_via_c_abi(w, g, path, part):
    """Direct C-ABI call (ctypes), no workspace argument."""
    lib = pkv.library()
    out = torch.full(g.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    desc = pkv.cache_desc(g.k_cache)
    cfg = pkv.DecodeConfig(path, part)
    S, Hq, _ = g.q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.paged_attention_decode_no_alloc(
        ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(g.k_cache.data_ptr()), ctypes.c_void_p(g.v_cache.data_ptr()),
        ctypes.c_void_p(g.block_tables.data_ptr()), g.block_tables.shape[1], ctypes.c_void_p(g.context_lens.data_ptr()),
        S, Hq, w.max_context_len, g.scale, ctypes.c_void_p(out.data_ptr()), pkv.F32, ctypes.byref(desc),
        ctypes.byref(cfg), stream)
    assert rc == 0, lib.paged_kv_last_error().decode()
    return out


@pytest.mark.parametrize("path", [pkv.PATH_CUDA_CORE, pkv.PATH_TENSOR_CORE], ids=["cuda_core", "tensor_core"])
def test_no_alloc_matches_workspace_entry_point_twice(path):
    # two different problems back to back, both split into several partitions, so the
    # second call runs over what the first one left in the shared array
    cases = [
        workloads.random_workload(310_900, num_seqs=9, max_len=3000, min_len=700, num_q_heads=32, num_kv_heads=4,
                                  head_dim=128, block_size=16, dtype="bf16", canary=False),
        workloads.random_workload(310_901, num_seqs=5, max_len=2200, min_len=1, num_q_heads=16, num_kv_heads=2,
                                  head_dim=128, block_size=32, dtype="f16", canary=False),
        workloads.random_workload(310_903, num_seqs=7, max_len=1800, min_len=1, num_q_heads=16, num_kv_heads=4,
                                  head_dim=64, block_size=16, dtype="bf16", canary=False),
        # f32 caches, 8 query heads per KV head: the tf32 kernel on the tensor-core path
        workloads.random_workload(310_905, num_seqs=6, max_len=2000, min_len=300, num_q_heads=16, num_kv_heads=2,
                                  head_dim=128, block_size=16, dtype="f32", canary=False),
    ]
    for w in cases:
        g = w.to("cuda")
        need = pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.max_context_len, g.k_cache,
                                                   path=path, partition_tokens=256)
        assert 0 < need <= pkv.paged_attention_no_alloc_limit()
        ref = _with_workspace(w, g, path, 256)
        got = _no_alloc_via_c_abi(w, g, path, 256)
        torch.cuda.synchronize()
        assert pkv.device_error() == 0
        assert np.isfinite(got.cpu().numpy()).all()
        err = (got - ref).abs().max().item()
        assert err <= TOL[w.dtype], f"max-abs difference {err:.3g}"
        # the same kernels with the same plan, only the scratch address differs: the
        # kernels are deterministic, so the two outputs agree bit for bit
        assert torch.equal(got, ref), f"outputs differ (max-abs {err:.3g})"


def test_python_wrapper_allocates_nothing():
    """Through the Python binding too, the call takes no device memory from torch's
    allocator: the counters of allocations do not move over two calls."""
    w = workloads.random_workload(310_904, num_seqs=6, max_len=2500, min_len=600, num_q_heads=16, num_kv_heads=2,
                                  head_dim=128, block_size=16, dtype="bf16", canary=False)
    g = w.to("cuda")
    out = torch.empty(g.q.shape, dtype=torch.float32, device="cuda")
    ref = _with_workspace(w, g, pkv.PATH_AUTO, 256)
    torch.cuda.synchronize()
    before = torch.cuda.memory_stats()
    for _ in range(2):
        pkv.paged_attention_decode_no_alloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                                            max_context_len=w.max_context_len, partition_tokens=256)
    torch.cuda.synchronize()
    after = torch.cuda.memory_stats()
    for key in ("allocation.all.allocated", "segment.all.allocated", "allocated_bytes.all.allocated"):
        assert after.get(key, 0) == before.get(key, 0), f"{key}: {before.get(key, 0)} -> {after.get(key, 0)}"
    assert pkv.device_error() == 0
    assert torch.equal(out, ref)
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_attention_decode_no_alloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale, out,
                                            max_context_len=None)


def test_no_alloc_rejects_more_than_the_array():
    w = workloads.random_workload(310_902, num_seqs=4, max_len=64, min_len=8, num_q_heads=8, num_kv_heads=1,
                                  head_dim=128, block_size=16, dtype="bf16", canary=False)
    g = w.to("cuda")
    # a claimed max length this large needs far more partition space than the array holds
    big = 1 << 22
    need = pkv.paged_attention_workspace_bytes(64, 8, big, g.k_cache, path=pkv.PATH_CUDA_CORE,
                                               partition_tokens=128)
    assert need > pkv.paged_attention_no_alloc_limit()
    tables = torch.zeros((64, big // 16), dtype=torch.int32, device="cuda")
    lens = torch.ones(64, dtype=torch.int32, device="cuda")
    q = torch.zeros((64, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode_no_alloc(q, g.k_cache, g.v_cache, tables, lens, 1.0, out, max_context_len=big,
                                            path=pkv.PATH_CUDA_CORE, partition_tokens=128)
    assert e.value.status == 3 and "built-in array" in str(e.value)
