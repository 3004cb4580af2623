"""The C ABI without a GPU: the library builds, loads, exports what the header
declares, and its host-side argument checks answer before any device work."""
import ctypes
import subprocess

import pytest

import paged_kv_cache_310_gb300 as pkv
from paged_kv_cache_310_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.library()


def test_header_declares_the_three_calls():
    names = pkv.declared_functions()
    for n in ("paged_kv_append", "paged_attention_decode", "paged_block_copy"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in pkv.declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version(lib):
    assert lib.paged_kv_version().decode().count(".") == 2


def _desc(num_blocks=64, block_size=16, num_kv_heads=8, head_dim=128, dtype=pkv.BF16):
    return pkv.CacheDesc(num_blocks, block_size, num_kv_heads, head_dim, dtype)


def _ws(lib, S, Hq, L, desc, part=0, path=0):
    cfg = pkv.DecodeConfig(path, part)
    return lib.paged_attention_workspace_bytes(S, Hq, L, ctypes.byref(desc), ctypes.byref(cfg))


def test_workspace_sizes(lib):
    d = _desc()
    core, tensor = pkv.PATH_CUDA_CORE, pkv.PATH_TENSOR_CORE
    assert _ws(lib, 64, 32, 512, d, path=core) == 0      # one partition: no workspace
    n = _ws(lib, 64, 32, 2048, d, path=core)             # 4 partitions of 512
    rows = 64 * 32 * 4
    assert n == -(-rows * 8 // 256) * 256 + rows * 128 * 4
    assert _ws(lib, 64, 32, 2048, d, part=1024, path=core) < n
    # the tensor-core path (chosen automatically for groups >= 2) splits at 1024 tokens
    assert _ws(lib, 64, 32, 2048, d) == _ws(lib, 64, 32, 2048, d, path=tensor)
    # one partition: the tensor-core path still needs its work list (16 B per item + header)
    assert _ws(lib, 64, 32, 1024, d, path=tensor, part=1024) == 256 + -(-64 * 8 * 16 // 256) * 256
    assert _ws(lib, 64, 32, 2048, d, path=tensor, part=8192) == 0  # partitions <= 4096 on tensor cores
    assert _ws(lib, 64, 32, 2048, d, part=100) == 0       # invalid partition size
    assert _ws(lib, 64, 30, 2048, d) == 0                 # heads not a multiple of kv heads
    assert _ws(lib, 4, 8, 2048, _desc(dtype=pkv.F32), path=tensor) > 0   # f32: the tf32 kernel's work list
    assert _ws(lib, 4, 8 * 9, 2048, _desc(dtype=pkv.F32), path=tensor) == 0  # f32 groups above 8: none


@pytest.mark.parametrize("field,value,status", [
    ("block_size", 7, 2), ("head_dim", 96, 2), ("dtype", 5, 2), ("num_blocks", 0, 1), ("num_kv_heads", 0, 1),
])
def test_cache_descriptor_checks(lib, field, value, status):
    d = _desc()
    setattr(d, field, value)
    rc = lib.paged_kv_append(None, None, None, 1, None, None, ctypes.byref(d), None)
    assert rc == status
    assert lib.paged_kv_last_error()


def test_argument_checks_before_device_work(lib):
    d = _desc()
    assert lib.paged_kv_append(None, None, None, -1, None, None, ctypes.byref(d), None) == 1
    assert lib.paged_kv_append(None, None, None, 0, None, None, ctypes.byref(d), None) == 0
    assert lib.paged_kv_append(None, None, None, 3, None, None, ctypes.byref(d), None) == 1
    assert b"NULL" in lib.paged_kv_last_error()
    odd = ctypes.c_void_p(0x1008)
    assert lib.paged_kv_append(odd, odd, odd, 3, odd, odd, ctypes.byref(d), None) == 1
    assert b"aligned" in lib.paged_kv_last_error()
    cfg = pkv.DecodeConfig(0, 0)
    # a group of 17 query heads per kv head is outside the supported set; 16 only on tensor cores
    assert lib.paged_attention_decode(None, None, None, None, 0, None, 4, 136, 16, 1.0, None, 2, None, 0,
                                      ctypes.byref(d), ctypes.byref(cfg), None) == 2
    core = pkv.DecodeConfig(pkv.PATH_CUDA_CORE, 0)
    assert lib.paged_attention_decode(None, None, None, None, 0, None, 4, 128, 16, 1.0, None, 2, None, 0,
                                      ctypes.byref(d), ctypes.byref(core), None) == 2
    # workspace too small for a split decode
    a = ctypes.c_void_p(0x10000)
    rc = lib.paged_attention_decode(a, a, a, a, 256, a, 4, 32, 4096, 1.0, a, 2, None, 0, ctypes.byref(d),
                                    ctypes.byref(cfg), None)
    assert rc == 3, lib.paged_kv_last_error()
    # too few table columns for the stated max length
    rc = lib.paged_attention_decode(a, a, a, a, 10, a, 4, 32, 4096, 1.0, a, 2, a, 1 << 30, ctypes.byref(d),
                                    ctypes.byref(cfg), None)
    assert rc == 1 and b"max_blocks_per_seq" in lib.paged_kv_last_error()
    # out dtype f16 for bf16 caches
    rc = lib.paged_attention_decode(a, a, a, a, 256, a, 4, 32, 4096, 1.0, a, 1, a, 1 << 30, ctypes.byref(d),
                                    ctypes.byref(cfg), None)
    assert rc == 2


def test_block_copy_pair_checks(lib):
    d = _desc(num_blocks=10)
    a = ctypes.c_void_p(0x10000)

    def run(pairs):
        arr = (ctypes.c_int64 * (2 * len(pairs)))(*[x for p in pairs for x in p])
        return lib.paged_block_copy(a, arr, len(pairs), a, a, ctypes.byref(d), None)

    assert run([(1, 1)]) == 1                  # onto itself
    assert run([(1, 2), (3, 2)]) == 1          # destination twice
    assert run([(1, 2), (2, 3)]) == 1          # destination also a source
    assert run([(1, 10)]) == 1                 # out of range
    assert run([(-1, 2)]) == 1


def test_binding_fails_loudly_without_a_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    k = torch.zeros(2, 1, 16, 64)
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_kv_append(k[:, 0, :1], k[:, 0, :1], torch.zeros(2, dtype=torch.int64), k, k)


def test_plan_reports_path_partitions_and_launches(lib):
    k16 = __import__("torch").empty((1, 8, 16, 128), dtype=__import__("torch").bfloat16)
    p = pkv.paged_attention_plan(128, 64, 4096, k16)            # GQA group 8 -> tensor cores
    assert p["path"] == pkv.PATH_TENSOR_CORE and p["partition_tokens"] % 128 == 0
    assert p["partition_tokens"] <= 4096 and p["kernel_launches"] == 2 + (p["max_partitions"] > 1)
    p1 = pkv.paged_attention_plan(64, 8, 2048, k16, path=pkv.PATH_CUDA_CORE)   # 512-token partitions
    assert p1["path"] == pkv.PATH_CUDA_CORE and p1["partition_tokens"] == 512 and p1["max_partitions"] == 4
    assert p1["kernel_launches"] == 2
    assert pkv.paged_attention_plan(64, 8, 300, k16, path=pkv.PATH_CUDA_CORE)["kernel_launches"] == 1
    assert pkv.paged_attention_plan(64, 8, 2048, k16)["path"] == pkv.PATH_TENSOR_CORE  # automatic, bf16 D128
    k32 = __import__("torch").empty((1, 8, 16, 64), dtype=__import__("torch").float32)
    assert pkv.paged_attention_plan(64, 8, 2048, k32)["path"] == pkv.PATH_CUDA_CORE   # f32, D64
    torch = __import__("torch")
    k16d64 = torch.empty((1, 8, 16, 64), dtype=torch.float16)
    assert pkv.paged_attention_plan(64, 8, 2048, k16d64)["path"] == pkv.PATH_TENSOR_CORE  # f16, D64
    # head_dim 64 on the 16-bit tensor-core kernel: an even number of KV heads pairs up,
    # two KV heads per work item (any group size); otherwise one
    assert pkv.paged_attention_plan(64, 8, 2048, k16d64)["kv_heads_per_item"] == 2       # 8 KV heads, G = 1
    assert pkv.paged_attention_plan(64, 128, 2048, k16d64)["kv_heads_per_item"] == 2     # G = 16
    k16d64odd = torch.empty((1, 3, 16, 64), dtype=torch.bfloat16)
    assert pkv.paged_attention_plan(64, 48, 2048, k16d64odd)["kv_heads_per_item"] == 1   # 3 KV heads
    assert pkv.paged_attention_plan(64, 8, 2048, k16)["kv_heads_per_item"] == 1          # head_dim 128
    assert pkv.paged_attention_plan(64, 64, 2048, k32)["kv_heads_per_item"] == 1          # f32, tf32 kernel
    assert pkv.paged_attention_plan(64, 8, 2048, k16d64, path=pkv.PATH_CUDA_CORE)["kv_heads_per_item"] == 1
    k16b64 = torch.empty((1, 8, 64, 128), dtype=torch.bfloat16)
    assert pkv.paged_attention_plan(128, 8, 2048, k16b64)["path"] == pkv.PATH_TENSOR_CORE  # 64-token blocks
    k32b64 = torch.empty((1, 8, 64, 128), dtype=torch.float32)
    assert pkv.paged_attention_plan(32, 8, 2048, k32b64)["path"] == pkv.PATH_CUDA_CORE
    # f32: at head_dim 128 CUDA cores up to 4 query heads per KV head, the tf32
    # tensor-core kernel from 5 to 8; at head_dim 64 CUDA cores up to 8 (either path on
    # request up to 8), nothing above 8
    k32d128 = torch.empty((1, 8, 16, 128), dtype=torch.float32)
    assert pkv.paged_attention_plan(64, 8, 2048, k32, path=pkv.PATH_TENSOR_CORE)["path"] == pkv.PATH_TENSOR_CORE
    assert pkv.paged_attention_plan(64, 32, 2048, k32d128)["path"] == pkv.PATH_CUDA_CORE  # group 4
    assert pkv.paged_attention_plan(64, 40, 2048, k32d128)["path"] == pkv.PATH_TENSOR_CORE  # group 5
    assert pkv.paged_attention_plan(64, 64, 2048, k32d128)["path"] == pkv.PATH_TENSOR_CORE  # group 8
    assert pkv.paged_attention_plan(64, 24, 2048, k32d128)["path"] == pkv.PATH_CUDA_CORE  # group 3
    assert pkv.paged_attention_plan(64, 40, 2048, k32)["path"] == pkv.PATH_CUDA_CORE     # head_dim 64, group 5
    assert pkv.paged_attention_plan(64, 64, 2048, k32)["path"] == pkv.PATH_CUDA_CORE     # head_dim 64, group 8
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_attention_plan(64, 72, 2048, k32, path=pkv.PATH_TENSOR_CORE)          # group 9
    with pytest.raises(pkv.PagedKVError):   # f32 at group 16: above the CUDA-core path's 8
        pkv.paged_attention_plan(4, 128, 2048, k32b64)
    assert pkv.paged_attention_plan(4, 128, 2048, k16b64)["path"] == pkv.PATH_TENSOR_CORE  # bf16 at group 16
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_attention_plan(64, 8, 2048, k16, path=pkv.PATH_TENSOR_CORE, partition_tokens=8192)


def test_prefill_argument_checks_before_device_work(lib):
    a = ctypes.c_void_p(0x10000)

    def run(desc, Hq=64, T=100, S=4, L=4096, mbps=256, out_dtype=pkv.BF16, ws=None, wsb=0, q=a, scale=0.1):
        return lib.paged_attention_prefill(q, a, a, a, mbps, a, a, S, Hq, T, L, scale, a, out_dtype, ws, wsb,
                                           ctypes.byref(desc), None)

    d = _desc()
    need = lib.paged_attention_prefill_workspace_bytes(4, 64, 100, ctypes.byref(d))
    assert need > 256
    assert run(_desc(dtype=pkv.F32)) == 2                       # f32 has no prefill path
    assert run(_desc(head_dim=96)) == 2                          # head_dim outside {64, 128}
    assert run(d, Hq=8 * 17) == 2                               # group 17
    assert run(_desc(num_kv_heads=4096), Hq=4096) == 2           # KV head packed in 12 bits
    assert b"4095" in lib.paged_kv_last_error()
    assert run(d, Hq=60) == 1                                   # not a multiple of the KV heads
    assert run(d, ws=None) == 3                                 # no workspace
    assert run(d, ws=ctypes.c_void_p(0x10100), wsb=need - 256) == 3
    assert run(d, ws=ctypes.c_void_p(0x10080), wsb=need) == 1   # workspace not 256-byte aligned
    assert run(d, q=ctypes.c_void_p(0x10008), ws=a, wsb=need) == 1  # q not 16-byte aligned
    assert run(d, mbps=255, ws=a, wsb=need) == 1                # table narrower than max length needs
    assert run(d, out_dtype=pkv.F16, ws=a, wsb=need) == 2       # out must be the cache dtype or f32
    assert run(d, scale=float("inf"), ws=a, wsb=need) == 1
    assert run(d, T=0) == 0 and run(d, S=0) == 0                # nothing to do
