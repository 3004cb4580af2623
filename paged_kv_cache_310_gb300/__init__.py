"""Python binding of libpagedkv.so -- the paged KV cache hot path on one GB300.

Argument marshalling only: every step runs in the library's CUDA kernels.  PyTorch
supplies device memory and the current stream.  The calls mirror the C ABI in
``include/pagedkv.h``:

* :func:`paged_kv_append`        -- new tokens' K/V into their cache slots
* :func:`paged_block_copy`       -- copy-on-write block copies
* :func:`paged_attention_decode` -- single-token decode attention through block tables
* :func:`paged_kv_gather`        -- the block-table gather alone (indexing checks)

If the library has not been built the import still succeeds, but every call raises:
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

__all__ = [
    "PagedKVError", "CacheDesc", "DecodeConfig", "DecodePlan", "paged_attention_plan", "library", "library_path", "cache_desc",
    "paged_kv_append", "paged_block_copy", "paged_attention_decode",
    "paged_attention_workspace_bytes", "paged_attention_decode_no_alloc", "paged_attention_no_alloc_limit",
    "paged_kv_gather", "paged_block_swap_out", "paged_block_swap_in", "paged_attention_prefill", "device_error", "declared_functions",
    "PATH_AUTO", "PATH_CUDA_CORE", "PATH_TENSOR_CORE",
    "PreparedCall", "prepare_kv_append", "prepare_block_copy", "prepare_attention_decode", "set_wait_limit",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpagedkv.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pagedkv.h")

F32, F16, BF16 = 0, 1, 2
DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
PATH_AUTO, PATH_CUDA_CORE, PATH_TENSOR_CORE = 0, 1, 2

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_WORKSPACE",
          4: "PKV_ERR_CUDA", 5: "PKV_ERR_DEVICE_INDEX", 6: "PKV_ERR_DEVICE_TIMEOUT", 7: "PKV_ERR_OUT_OF_BLOCKS"}


class PagedKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class DecodeConfig(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("partition_tokens", ctypes.c_int32)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("partition_tokens", ctypes.c_int32),
                ("max_partitions", ctypes.c_int32), ("kernel_launches", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("kv_heads_per_item", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def declared_functions(header: str = HEADER) -> list[str]:
    """Names of the functions include/pagedkv.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:paged|pkv)_\w+)\s*\(", text)))


def library():
    """The loaded libpagedkv.so (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(library_path):
            raise PagedKVError(4, f"{library_path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(library_path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        desc_p, cfg_p = ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeConfig)
        sig = {
            "paged_kv_append": [vp, vp, vp, i32, vp, vp, desc_p, vp],
            "paged_block_copy": [vp, vp, i32, vp, vp, desc_p, vp],
            "paged_attention_workspace_bytes": [i32, i32, i32, desc_p, cfg_p],
            "paged_attention_plan": [i32, i32, i32, desc_p, cfg_p, ctypes.POINTER(DecodePlan)],
            "paged_attention_decode": [vp, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp, i32,
                                       vp, sz, desc_p, cfg_p, vp],
            "paged_kv_gather": [vp, vp, vp, i32, vp, i32, i32, vp, vp, desc_p, vp],
            "paged_block_swap_out": [vp, i32, vp, vp, vp, vp, desc_p, vp],
            "paged_attention_prefill": [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp, i32,
                                        vp, sz, desc_p, vp],
            "paged_attention_prefill_workspace_bytes": [i32, i32, i32, desc_p],
            "paged_block_swap_in": [vp, i32, vp, vp, vp, vp, desc_p, vp],
            "paged_attention_decode_no_alloc": [vp, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp,
                                                i32, desc_p, cfg_p, vp],
            "paged_attention_no_alloc_limit": [],
            "paged_kv_device_error": [vp],
            "paged_kv_selftest_wait_timeout": [ctypes.c_uint64, vp],
            "paged_kv_set_wait_limit": [ctypes.c_uint64],
            "paged_kv_last_error": [],
            "paged_kv_version": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.paged_attention_workspace_bytes.restype = sz
        lib.paged_attention_no_alloc_limit.restype = sz
        lib.paged_attention_prefill_workspace_bytes.restype = sz
        lib.paged_kv_last_error.restype = ctypes.c_char_p
        lib.paged_kv_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != 0:
        raise PagedKVError(status, library().paged_kv_last_error().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (t.device.type != "cuda" or not t.is_contiguous()):
            raise PagedKVError(1, "tensors must be contiguous CUDA tensors")


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """Descriptor of a pool shaped [num_blocks, num_kv_heads, block_size, head_dim]."""
    if k_cache.dim() != 4:
        raise PagedKVError(1, "cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    if k_cache.dtype not in DTYPE_CODE:
        raise PagedKVError(2, f"cache dtype {k_cache.dtype}")
    return CacheDesc(nb, bs, hkv, d, DTYPE_CODE[k_cache.dtype])


class PreparedCall:
    """One library call whose arguments were checked and marshalled once.

    Calling it enqueues the same work again on `stream` (a torch.cuda.Stream or a raw
    cudaStream_t handle; default: the device's current stream), with none of the
    per-call argument checks and ctypes conversions of the plain functions -- what a
    serving loop that replays the same buffers every step wants.  The tensors it was
    made from stay referenced by it; their contents may change between calls, their
    storage must not (no reallocation, resize or reshaping in place)."""

    __slots__ = ("_fn", "_args", "_device", "_keep")

    def __init__(self, fn, args, device, keep):
        self._fn, self._args, self._device, self._keep = fn, tuple(args), device, keep

    def __call__(self, stream=None) -> None:
        if stream is None:
            handle = torch.cuda.current_stream(self._device).cuda_stream
        else:
            handle = stream if isinstance(stream, int) else stream.cuda_stream
        status = self._fn(*self._args, ctypes.c_void_p(handle))
        if status != 0:
            raise PagedKVError(status, library().paged_kv_last_error().decode())


def _run(prepared: PreparedCall) -> None:
    prepared()


def _append_call(k, v, slot_mapping, k_cache, v_cache) -> PreparedCall:
    _need_cuda(k, v, slot_mapping, k_cache, v_cache)
    if slot_mapping.dtype != torch.int64 or k.dtype != k_cache.dtype or v.dtype != k_cache.dtype:
        raise PagedKVError(1, "slot_mapping must be int64 and k/v must have the cache dtype")
    if k.shape != v.shape or k.dim() != 3 or k.shape[0] != slot_mapping.numel() \
            or tuple(k.shape[1:]) != (k_cache.shape[1], k_cache.shape[3]) or k_cache.shape != v_cache.shape:
        raise PagedKVError(1, "shape mismatch between k, v, slot_mapping and the caches")
    desc = cache_desc(k_cache)
    args = (_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache),
            ctypes.byref(desc))
    return PreparedCall(library().paged_kv_append, args, k_cache.device, (k, v, slot_mapping, k_cache, v_cache, desc))


def paged_kv_append(k, v, slot_mapping, k_cache, v_cache) -> None:
    """k, v [T, Hkv, D] -> k_cache/v_cache rows given by slot_mapping (int64 [T])."""
    _run(_append_call(k, v, slot_mapping, k_cache, v_cache))


def prepare_kv_append(k, v, slot_mapping, k_cache, v_cache) -> PreparedCall:
    """paged_kv_append with its arguments bound once (see PreparedCall)."""
    return _append_call(k, v, slot_mapping, k_cache, v_cache)


def _block_copy_call(src_dst_pairs, k_cache, v_cache, host_pairs) -> PreparedCall:
    _need_cuda(src_dst_pairs, k_cache, v_cache)
    if src_dst_pairs.dtype != torch.int64 or (src_dst_pairs.numel() % 2):
        raise PagedKVError(1, "src_dst_pairs must be int64 [n, 2]")
    if host_pairs is not None:
        host_pairs = host_pairs.to(torch.int64).contiguous()
        if host_pairs.device.type != "cpu" or host_pairs.numel() != src_dst_pairs.numel():
            raise PagedKVError(1, "host_pairs must be a CPU copy of src_dst_pairs")
    desc = cache_desc(k_cache)
    n = src_dst_pairs.numel() // 2
    args = (_ptr(src_dst_pairs), _ptr(host_pairs), n, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc))
    return PreparedCall(library().paged_block_copy, args, k_cache.device,
                        (src_dst_pairs, host_pairs, k_cache, v_cache, desc))


def paged_block_copy(src_dst_pairs, k_cache, v_cache, host_pairs: torch.Tensor | None = None) -> None:
    """Copy block src to block dst for each row of src_dst_pairs (device int64 [n, 2]).

    host_pairs (CPU int64 [n, 2], optional) lets the library validate the pairs.
    """
    _run(_block_copy_call(src_dst_pairs, k_cache, v_cache, host_pairs))


def prepare_block_copy(src_dst_pairs, k_cache, v_cache, host_pairs: torch.Tensor | None = None) -> PreparedCall:
    """paged_block_copy with its arguments bound once (see PreparedCall); the pairs are
    validated against host_pairs, when given, at every call."""
    return _block_copy_call(src_dst_pairs, k_cache, v_cache, host_pairs)


def _swap_buffers(ids, k_cache, host_k, host_v):
    _need_cuda(ids, k_cache)
    if ids.dtype != torch.int64:
        raise PagedKVError(1, "block ids must be int64")
    shape = (ids.numel(),) + tuple(k_cache.shape[1:])
    for h in (host_k, host_v):
        if tuple(h.shape) != shape or h.dtype != k_cache.dtype or not h.is_contiguous():
            raise PagedKVError(1, f"swap buffers must be contiguous {shape} in the cache dtype")


def paged_block_swap_out(block_ids, k_cache, v_cache, host_k, host_v) -> None:
    """host_k/v[i] <- pool block block_ids[i] (device int64 ids; pinned host buffers)."""
    _swap_buffers(block_ids, k_cache, host_k, host_v)
    desc = cache_desc(k_cache)
    _check(library().paged_block_swap_out(_ptr(block_ids), block_ids.numel(), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(host_k), _ptr(host_v), ctypes.byref(desc), _stream(k_cache)))


def paged_block_swap_in(block_ids, host_k, host_v, k_cache, v_cache) -> None:
    """pool block block_ids[i] <- host_k/v[i]."""
    _swap_buffers(block_ids, k_cache, host_k, host_v)
    desc = cache_desc(k_cache)
    _check(library().paged_block_swap_in(_ptr(block_ids), block_ids.numel(), _ptr(host_k), _ptr(host_v),
                                         _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _stream(k_cache)))


def _config(path: int, partition_tokens: int) -> DecodeConfig:
    return DecodeConfig(int(path), int(partition_tokens))


def paged_attention_workspace_bytes(num_seqs, num_q_heads, max_context_len, k_cache, *, path=PATH_AUTO,
                                    partition_tokens=0) -> int:
    desc = cache_desc(k_cache)
    cfg = _config(path, partition_tokens)
    return int(library().paged_attention_workspace_bytes(num_seqs, num_q_heads, max_context_len,
                                                         ctypes.byref(desc), ctypes.byref(cfg)))


def paged_attention_plan(num_seqs, num_q_heads, max_context_len, k_cache, *, path=PATH_AUTO,
                         partition_tokens=0) -> dict:
    """The path, partition size, partition count, kernel launches and workspace bytes
    paged_attention_decode uses for these sizes."""
    desc = cache_desc(k_cache)
    cfg = _config(path, partition_tokens)
    plan = DecodePlan()
    _check(library().paged_attention_plan(num_seqs, num_q_heads, max_context_len, ctypes.byref(desc),
                                          ctypes.byref(cfg), ctypes.byref(plan)))
    return {f: getattr(plan, f) for f, _ in DecodePlan._fields_}


_ws_cache: dict = {}


def _workspace(device, nbytes: int) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    key = (device.type, device.index)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, *,
                           max_context_len: int | None = None, workspace: torch.Tensor | None = None,
                           path: int = PATH_AUTO, partition_tokens: int = 0) -> torch.Tensor:
    """out[s, h] = softmax(scale * q[s, h] . K_j) V_j over the context_lens[s] tokens of s.

    q [S, Hq, D]; caches [NB, Hkv, bs, D]; block_tables int32 [S, max_blocks];
    context_lens int32 [S]; out [S, Hq, D] in q's dtype or float32.
    max_context_len: host upper bound on context_lens (computed with a device sync
    when omitted).  workspace: uint8 device buffer, allocated and cached when omitted.
    """
    _run(_decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len,
                      workspace, path, partition_tokens))
    return out


def prepare_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, *,
                             max_context_len: int, workspace: torch.Tensor | None = None,
                             path: int = PATH_AUTO, partition_tokens: int = 0) -> PreparedCall:
    """paged_attention_decode with its arguments bound once (see PreparedCall).
    max_context_len stays the bound of every later call."""
    if max_context_len is None:
        raise PagedKVError(1, "max_context_len is required for a prepared decode")
    return _decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len, workspace,
                        path, partition_tokens)


def _decode_call(q, k_cache, v_cache, block_tables, context_lens, scale, out, max_context_len, workspace, path,
                 partition_tokens) -> PreparedCall:
    _need_cuda(q, k_cache, v_cache, block_tables, context_lens, out, workspace)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PagedKVError(1, "block_tables and context_lens must be int32")
    if q.dim() != 3 or out.shape != q.shape or q.dtype != k_cache.dtype or v_cache.shape != k_cache.shape \
            or v_cache.dtype != k_cache.dtype or q.shape[2] != k_cache.shape[3]:
        raise PagedKVError(1, "shape/dtype mismatch between q, out and the caches")
    S, Hq, _ = q.shape
    if context_lens.numel() != S or block_tables.dim() != 2 or block_tables.shape[0] != S:
        raise PagedKVError(1, "block_tables must be [S, max_blocks] and context_lens [S]")
    if out.dtype not in DTYPE_CODE:
        raise PagedKVError(2, f"out dtype {out.dtype}")
    if max_context_len is None:
        max_context_len = int(context_lens.max()) if S else 0
    desc = cache_desc(k_cache)
    cfg = _config(path, partition_tokens)
    lib = library()
    need = int(lib.paged_attention_workspace_bytes(S, Hq, max_context_len, ctypes.byref(desc),
                                                   ctypes.byref(cfg)))
    if workspace is None:
        workspace = _workspace(q.device, need)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            S, Hq, max_context_len, ctypes.c_float(float(scale)), _ptr(out), DTYPE_CODE[out.dtype], _ptr(workspace),
            ws_bytes, ctypes.byref(desc), ctypes.byref(cfg))
    return PreparedCall(lib.paged_attention_decode, args, q.device,
                        (q, k_cache, v_cache, block_tables, context_lens, out, workspace, desc, cfg))


def paged_attention_decode_no_alloc(q, k_cache, v_cache, block_tables, context_lens, scale, out, *,
                                    max_context_len: int, path: int = PATH_AUTO,
                                    partition_tokens: int = 0) -> torch.Tensor:
    """paged_attention_decode without a workspace argument, for callers that cannot
    allocate device memory: the scratch is the library's built-in array of
    ``paged_attention_no_alloc_limit()`` bytes per GPU, shared by every call (calls
    that overlap on the GPU race on it).

    max_context_len (a host bound on context_lens) is required here: working it out
    from the device tensor would run a reduction that allocates its result."""
    _need_cuda(q, k_cache, v_cache, block_tables, context_lens, out)
    if q.dim() != 3 or out.shape != q.shape or q.dtype != k_cache.dtype or block_tables.dtype != torch.int32 \
            or context_lens.dtype != torch.int32:
        raise PagedKVError(1, "shape/dtype mismatch between q, out, the caches and the tables")
    if max_context_len is None:
        raise PagedKVError(1, "max_context_len is required: computing it on the device would allocate")
    S, Hq, _ = q.shape
    desc = cache_desc(k_cache)
    cfg = _config(path, partition_tokens)
    _check(library().paged_attention_decode_no_alloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), S, Hq,
        max_context_len, float(scale), _ptr(out), DTYPE_CODE[out.dtype], ctypes.byref(desc), ctypes.byref(cfg),
        _stream(q)))
    return out


def paged_attention_no_alloc_limit() -> int:
    """Bytes of the built-in workspace array used by paged_attention_decode_no_alloc."""
    return int(library().paged_attention_no_alloc_limit())


def paged_attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, out, *,
                            max_context_len: int | None = None,
                            workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Causal attention of several new tokens per sequence (prefill / chunked prefill).

    q, out [T, Hq, D]: sequence s's new tokens are rows query_start[s]..query_start[s+1]-1,
    the last ones of its context_lens[s] tokens (K/V already appended).  query_start:
    int32 [S+1] on the device.
    """
    _need_cuda(q, k_cache, v_cache, block_tables, context_lens, query_start, out, workspace)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or query_start.dtype != torch.int32:
        raise PagedKVError(1, "block_tables, context_lens and query_start must be int32")
    if q.dim() != 3 or out.shape != q.shape or q.dtype != k_cache.dtype or q.shape[2] != k_cache.shape[3]:
        raise PagedKVError(1, "shape/dtype mismatch between q, out and the caches")
    T, Hq, _ = q.shape
    S = context_lens.numel()
    if query_start.numel() != S + 1 or block_tables.shape[0] != S:
        raise PagedKVError(1, "query_start must be [S+1] and block_tables [S, max_blocks]")
    if out.dtype not in DTYPE_CODE:
        raise PagedKVError(2, f"out dtype {out.dtype}")
    if max_context_len is None:
        max_context_len = int(context_lens.max()) if S else 0
    desc = cache_desc(k_cache)
    lib = library()
    need = int(lib.paged_attention_prefill_workspace_bytes(S, Hq, T, ctypes.byref(desc)))
    if workspace is None:
        workspace = _workspace(q.device, need)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.paged_attention_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       block_tables.shape[1], _ptr(context_lens), _ptr(query_start), S, Hq, T,
                                       max_context_len, float(scale), _ptr(out), DTYPE_CODE[out.dtype],
                                       _ptr(workspace), ws_bytes, ctypes.byref(desc), _stream(q)))
    return out


def paged_kv_gather(k_cache, v_cache, block_tables, context_lens, k_out, v_out, *,
                    max_context_len: int | None = None) -> None:
    """k_out/v_out [S, Hkv, max_len, D] <- each sequence's rows through its block table."""
    _need_cuda(k_cache, v_cache, block_tables, context_lens, k_out, v_out)
    S = context_lens.numel()
    if max_context_len is None:
        max_context_len = k_out.shape[2]
    if k_out.shape != (S, k_cache.shape[1], max_context_len, k_cache.shape[3]) or v_out.shape != k_out.shape \
            or k_out.dtype != k_cache.dtype or v_out.dtype != k_cache.dtype:
        raise PagedKVError(1, "k_out/v_out must be [S, Hkv, max_len, D] in the cache dtype")
    desc = cache_desc(k_cache)
    _check(library().paged_kv_gather(_ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                     _ptr(context_lens), S, max_context_len, _ptr(k_out), _ptr(v_out),
                                     ctypes.byref(desc), _stream(k_cache)))


def selftest_wait_timeout(limit_ns: int = 50_000_000) -> None:
    """Run the bounded-wait self-test kernel on the current stream (see the header)."""
    stream = torch.cuda.current_stream()
    _check(library().paged_kv_selftest_wait_timeout(int(limit_ns), ctypes.c_void_p(stream.cuda_stream)))


def set_wait_limit(limit_ns: int = 0) -> None:
    """Bound of the decode and prefill kernels' pipeline waits for later launches
    (0 = the default 2 s).  A tiny bound forces their abort path; see the header."""
    _check(library().paged_kv_set_wait_limit(int(limit_ns)))


def device_error(device=None) -> int:
    """Synchronise the current stream and read-and-clear the device error flag (0 = none)."""
    stream = torch.cuda.current_stream(device)
    return int(library().paged_kv_device_error(ctypes.c_void_p(stream.cuda_stream)))
