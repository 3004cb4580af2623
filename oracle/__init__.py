"""Float64 CPU oracle for the paged KV cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product library never calls it and it never calls the
product library: the two share no code.

The arithmetic lives in ``pagedkv_oracle.c`` (plain loops in double precision, built
with gcc, OpenMP over (sequence, query head) when available).  This module only
builds that file, marshals CPU tensors to it and converts results back.

What each function computes, and where the pages state it:

* :func:`attention_decode` -- softmax(scale * q K^T) V over each sequence's tokens,
  K/V gathered through its block table ("anthology-of-the-sota note-023", Method and
  Concepts; "Paged Attention" glossary, paragraph 4: the attention arithmetic is
  unchanged, only where K/V live).
* :func:`attention_prefill` -- several new tokens per sequence with a causal mask
  (prefill / chunked prefill); one new token is exactly decode.
* :func:`attention_partitions` / :func:`merge_partitions` -- the same softmax over
  consecutive token ranges and their exact recombination.  Not on the pages; it is
  the split over context partitions that long sequences need, pinned against the
  single pass.
* :func:`kv_append` -- a new token's K/V written into its slot of a fixed-size block
  ("Efficient Memory Management ... with PagedAttention", How It Works: pages are
  allocated as tokens are generated).
* :func:`block_copy` -- copy-on-write: the writer gets its own copy of a shared block
  (note-023, Concepts; same page, How It Works).
* :func:`gather` -- the block-table lookup alone, materialised contiguously.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_STATUS = {0: "ok", 1: "invalid argument", 2: "block or slot index out of range", 3: "out of memory"}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the compiler supports it).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded on both
    x86-64 and aarch64, so the oracle gives identical doubles on x86 and Arm.
    """
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC,
            "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # PKV_ORACLE_LIB points the pins at another build of this file (the
            # mutation tests use it to show that planted mistakes are caught)
            lib = ctypes.CDLL(os.environ.get("PKV_ORACLE_LIB") or build())
            i32, i64, dbl, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.pkvo_decode.argtypes = [i32, vp, i64, vp]
            lib.pkvo_max_threads.restype = i32
            lib.pkvo_attention_decode.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                                  i32, i32, dbl, i32, vp]
            lib.pkvo_attention_partitions.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                                      i32, i32, i32, dbl, i32, i32, vp, vp, vp]
            lib.pkvo_merge_partitions.argtypes = [vp, vp, vp, i64, i32, i32, vp]
            lib.pkvo_attention_prefill.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, i32, i32, i32,
                                                   i32, i32, dbl, i32, vp]
            lib.pkvo_kv_append.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32]
            lib.pkvo_block_copy.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, i32]
            lib.pkvo_gather.argtypes = [vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, vp]
            for name in ("pkvo_decode", "pkvo_attention_decode", "pkvo_attention_partitions", "pkvo_attention_prefill",
                         "pkvo_merge_partitions", "pkvo_kv_append", "pkvo_block_copy", "pkvo_gather"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: {_STATUS.get(rc, rc)}")


def _cpu(t: torch.Tensor, dtype=None) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes CPU tensors")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.contiguous()


def max_threads() -> int:
    """Threads the oracle uses when not told otherwise (OpenMP default)."""
    return int(_load().pkvo_max_threads())


def decode_elements(t: torch.Tensor) -> np.ndarray:
    """The oracle's exact float64 value of every element of a f32/f16/bf16 tensor."""
    t = _cpu(t)
    out = np.empty(t.numel(), dtype=np.float64)
    _check(_load().pkvo_decode(DTYPE_CODE[t.dtype], t.data_ptr(), t.numel(), out.ctypes.data),
           "decode")
    return out.reshape(tuple(t.shape))


def attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, num_threads=0):
    """float64 [S, Hq, D]: softmax(scale * q K^T) V per (sequence, query head).

    q [S, Hq, D]; k_cache, v_cache [NB, Hkv, bs, D] (same dtype as q);
    block_tables int32 [S, max_blocks]; context_lens int32 [S].
    """
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache, q.dtype), _cpu(v_cache, q.dtype)
    bt, cl = _cpu(block_tables, torch.int32), _cpu(context_lens, torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch")
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().pkvo_attention_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       DTYPE_CODE[q.dtype], bt.data_ptr(), bt.shape[1] if bt.dim() == 2 else 0,
                                       cl.data_ptr(), S, Hq, Hkv, D, bs, NB, float(scale),
                                       int(num_threads), out.ctypes.data)
    _check(rc, "attention_decode")
    return out


def attention_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, num_threads=0):
    """float64 [T, Hq, D]: causal attention of each sequence's new tokens.

    Sequence s's new tokens are rows query_start[s]..query_start[s+1]-1 of q and the last
    (query_start[s+1] - query_start[s]) of its context_lens[s] tokens; the token at
    position p attends to positions 0..p.
    """
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache, q.dtype), _cpu(v_cache, q.dtype)
    bt, cl = _cpu(block_tables, torch.int32), _cpu(context_lens, torch.int32)
    qs = _cpu(query_start, torch.int32)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = cl.numel()
    if qs.numel() != S + 1 or int(qs[-1]) != T:
        raise ValueError("query_start must be [S+1] ending at the number of query rows")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = _load().pkvo_attention_prefill(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), DTYPE_CODE[q.dtype],
                                        bt.data_ptr(), bt.shape[1], cl.data_ptr(), qs.data_ptr(), S, Hq, Hkv, D, bs,
                                        NB, float(scale), int(num_threads), out.ctypes.data)
    _check(rc, "attention_prefill")
    return out


def attention_partitions(q, k_cache, v_cache, block_tables, context_lens, scale, part_tokens):
    """Per-partition (m, l, o) of the softmax; shapes [S,Hq,P], [S,Hq,P], [S,Hq,P,D]."""
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache, q.dtype), _cpu(v_cache, q.dtype)
    bt, cl = _cpu(block_tables, torch.int32), _cpu(context_lens, torch.int32)
    S, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    max_len = int(cl.max()) if S else 0
    P = max(1, -(-max_len // part_tokens))
    m = np.empty((S, Hq, P)); l = np.empty((S, Hq, P)); o = np.empty((S, Hq, P, D))
    rc = _load().pkvo_attention_partitions(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           DTYPE_CODE[q.dtype], bt.data_ptr(), bt.shape[1], cl.data_ptr(),
                                           S, Hq, Hkv, D, bs, NB, float(scale), int(part_tokens), P,
                                           m.ctypes.data, l.ctypes.data, o.ctypes.data)
    _check(rc, "attention_partitions")
    return m, l, o


def merge_partitions(m, l, o):
    """Recombine per-partition (m, l, o) into normalised outputs [..., D]."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    P, D = o.shape[-2], o.shape[-1]
    rows = int(np.prod(o.shape[:-2]))
    out = np.empty(o.shape[:-2] + (D,))
    _check(_load().pkvo_merge_partitions(m.ctypes.data, l.ctypes.data, o.ctypes.data, rows, P, D,
                                         out.ctypes.data), "merge_partitions")
    return out


def kv_append(k, v, slot_mapping, k_cache, v_cache):
    """In place on the CPU pools: k/v [T, Hkv, D] rows go to slot_mapping [T] (int64)."""
    k, v = _cpu(k, k_cache.dtype), _cpu(v, k_cache.dtype)
    sm = _cpu(slot_mapping, torch.int64)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("pools must be contiguous")
    NB, Hkv, bs, D = k_cache.shape
    _check(_load().pkvo_kv_append(k.data_ptr(), v.data_ptr(), sm.data_ptr(), sm.numel(),
                                  k_cache.data_ptr(), v_cache.data_ptr(), DTYPE_CODE[k_cache.dtype],
                                  NB, Hkv, bs, D), "kv_append")


def block_copy(pairs, k_cache, v_cache):
    """In place on the CPU pools: block dst := block src for each (src, dst) row of pairs."""
    pairs = _cpu(pairs, torch.int64).reshape(-1, 2)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("pools must be contiguous")
    NB, Hkv, bs, D = k_cache.shape
    _check(_load().pkvo_block_copy(pairs.data_ptr(), pairs.shape[0], k_cache.data_ptr(),
                                   v_cache.data_ptr(), DTYPE_CODE[k_cache.dtype], NB, Hkv, bs, D),
           "block_copy")


def gather(k_cache, v_cache, block_tables, context_lens, max_len=None):
    """Contiguous copies [S, Hkv, max_len, D] of each sequence's K and V (zeros past its length)."""
    k_cache, v_cache = _cpu(k_cache), _cpu(v_cache, k_cache.dtype)
    bt, cl = _cpu(block_tables, torch.int32), _cpu(context_lens, torch.int32)
    NB, Hkv, bs, D = k_cache.shape
    S = cl.numel()
    if max_len is None:
        max_len = int(cl.max()) if S else 0
    k_out = torch.zeros((S, Hkv, max_len, D), dtype=k_cache.dtype)
    v_out = torch.zeros_like(k_out)
    _check(_load().pkvo_gather(k_cache.data_ptr(), v_cache.data_ptr(), DTYPE_CODE[k_cache.dtype],
                               bt.data_ptr(), bt.shape[1], cl.data_ptr(), S, NB, Hkv, bs, D, max_len,
                               k_out.data_ptr(), v_out.data_ptr()), "gather")
    return k_out, v_out
