"""Multi-token causal (prefill / chunked-prefill) attention on the GPU against the
float64 oracle.  Tolerances as for decode: max-abs <= 2e-3 on fp32 outputs; an output
in the cache dtype lies within one rounding of the oracle's value (|ref| * 2^-8 +
1e-4 for bf16, |ref| * 2^-11 + 1e-4 for f16) and is exactly the RNE rounding of the
same call's fp32 output."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_310_gb300 as pkv
import workloads
from parity_bounds import check_in_dtype

pytestmark = pytest.mark.gpu

CASES = [
    # dtype, bs, Hq, Hkv, max_len, min_len, new tokens (None = uniform 1..L)
    ("bf16", 16, 8, 8, 300, 1, None), ("f16", 16, 32, 4, 700, 100, None), ("bf16", 8, 64, 8, 900, 300, None),
    ("bf16", 32, 16, 1, 600, 1, None), ("f16", 16, 12, 4, 500, 1, None), ("bf16", 16, 32, 2, 400, 1, None),
    ("bf16", 16, 8, 2, 2000, 1500, lambda s, L: 128), ("f16", 32, 32, 8, 1200, 1, lambda s, L: (s * 37) % 5),
    ("bf16", 8, 4, 4, 3000, 2000, lambda s, L: L),
    # query-head groups that do not divide 16: 5, 6 and 7 heads per KV head
    ("bf16", 16, 40, 8, 800, 1, None), ("f16", 16, 12, 2, 600, 100, None), ("bf16", 32, 28, 4, 900, 200, None),
    # 64-token blocks: one block per 64-key chunk
    ("bf16", 64, 32, 8, 1200, 1, None), ("f16", 64, 8, 1, 900, 400, lambda s, L: 100),
]
# head_dim 64: dtype, bs, Hq, Hkv, max_len, min_len, new tokens
CASES_D64 = [
    ("bf16", 16, 32, 8, 900, 1, None), ("f16", 8, 16, 1, 700, 300, None), ("bf16", 32, 12, 4, 1500, 1, None),
    ("f16", 16, 8, 8, 2000, 1200, lambda s, L: 64), ("bf16", 16, 64, 4, 600, 1, lambda s, L: L),
    ("bf16", 64, 16, 2, 1000, 1, None),
]


def run(w, q, qs, out_dtype=torch.float32):
    g = w.to("cuda")
    kc, vc = g.k_cache, g.v_cache
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    pkv.paged_attention_prefill(q.cuda(), kc, vc, g.block_tables, g.context_lens, qs.cuda(), w.scale, out,
                                max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    return out


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-bs{c[1]}-{c[2]}x{c[3]}-L{c[4]}" for c in CASES])
def test_prefill_parity(case):
    dt, bs, Hq, Hkv, max_len, min_len, nt = case
    w, q, qs = workloads.prefill_workload(310_900 + CASES.index(case), num_seqs=6, max_len=max_len, min_len=min_len,
                                          num_q_heads=Hq, num_kv_heads=Hkv, block_size=bs, dtype=dt, new_tokens=nt)
    if int(qs[-1]) == 0:
        pytest.skip("no new tokens")
    ref = oracle.attention_prefill(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, qs, w.scale)
    out = run(w, q, qs)
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= 2e-3, f"max-abs {err:.3g}"
    low = run(w, q, qs, w.dtype)
    check_in_dtype(low, ref)
    assert torch.equal(low.cpu().view(torch.uint8), out.to(w.dtype).cpu().view(torch.uint8))


@pytest.mark.parametrize("case", CASES_D64, ids=[f"{c[0]}-bs{c[1]}-{c[2]}x{c[3]}-L{c[4]}" for c in CASES_D64])
def test_prefill_parity_head_dim_64(case):
    dt, bs, Hq, Hkv, max_len, min_len, nt = case
    w, q, qs = workloads.prefill_workload(310_940 + CASES_D64.index(case), num_seqs=6, max_len=max_len,
                                          min_len=min_len, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=64,
                                          block_size=bs, dtype=dt, new_tokens=nt)
    if int(qs[-1]) == 0:
        pytest.skip("no new tokens")
    ref = oracle.attention_prefill(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, qs, w.scale)
    out = run(w, q, qs)
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= 2e-3, f"max-abs {err:.3g}"
    low = run(w, q, qs, w.dtype)
    check_in_dtype(low, ref)
    assert torch.equal(low.cpu().view(torch.uint8), out.to(w.dtype).cpu().view(torch.uint8))


@pytest.mark.parametrize("scale", [-0.3, 0.0, 0.6], ids=["negative", "zero", "sharp"])
def test_prefill_scales_other_than_inverse_sqrt_d(scale):
    """A negative scale takes the minimum-score branch of the row maximum; zero gives the
    mean of the visible values; a large scale gives a sharp distribution."""
    w, q, qs = workloads.prefill_workload(310_960, num_seqs=5, max_len=700, min_len=1, num_q_heads=24,
                                          num_kv_heads=4, block_size=16, dtype="bf16", new_tokens=None)
    g = w.to("cuda")
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    pkv.paged_attention_prefill(q.cuda(), g.k_cache, g.v_cache, g.block_tables, g.context_lens, qs.cuda(), scale, out,
                                max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    ref = oracle.attention_prefill(q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, qs, scale)
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 2e-3


def test_one_new_token_matches_decode():
    w, q, qs = workloads.prefill_workload(310_950, num_seqs=9, max_len=1500, min_len=1, num_q_heads=32,
                                          num_kv_heads=8, new_tokens=lambda s, L: 1)
    out = run(w, q, qs)
    g = w.to("cuda")
    dec = torch.empty_like(out)
    pkv.paged_attention_decode(q.cuda(), g.k_cache, g.v_cache, g.block_tables, g.context_lens, w.scale, dec,
                               max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert (out - dec).abs().max().item() <= 2e-3


def test_bench_prefill_workload_sampled():
    """The chunked-prefill workload bench.py times (same seed, sizes and launch): every
    output computed on the GPU in one call, two whole sequences' outputs checked against
    the oracle, the rest checked finite."""
    dev = torch.device("cuda")
    nq = 512
    w, q, qs = workloads.prefill_workload(310_990, num_seqs=32, max_len=4096, min_len=1024, num_q_heads=64,
                                          num_kv_heads=8, block_size=16, dtype="bf16",
                                          new_tokens=lambda s, L: nq, canary=False, pool_device=dev)
    g = w.to(dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    pkv.paged_attention_prefill(q.to(dev), g.k_cache, g.v_cache, g.block_tables, g.context_lens, qs.to(dev),
                                w.scale, out, max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    got = out.cpu()
    assert torch.isfinite(got).all()
    kc, vc = w.k_cache.cpu(), w.v_cache.cpu()
    tables, lens, qh = w.block_tables.cpu(), w.context_lens.cpu(), q.cpu()
    for s in (0, 17):
        rows = slice(int(qs[s]), int(qs[s + 1]))
        ref = oracle.attention_prefill(qh[rows], kc, vc, tables[s:s + 1], lens[s:s + 1],
                                       torch.tensor([0, nq], dtype=torch.int32), w.scale)
        err = np.abs(got[rows].double().numpy() - ref).max()
        assert err <= 2e-3, f"sequence {s}: max-abs {err:.3g}"
