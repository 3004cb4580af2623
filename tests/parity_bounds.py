"""Parity bounds shared by the GPU parity tests (the CUDA path against the float64
oracle).

* fp32 outputs: max-abs error against the oracle within 1e-5 for f32 inputs and
  2e-3 for f16/bf16 inputs (fp32 accumulation).
* outputs stored in the 16-bit input dtype: every element within one rounding of the
  oracle's value plus a small absolute term for the fp32 accumulation,
  ``|ref| * 2^-8 + 1e-4`` for bf16 (8 significant bits: round-to-nearest moves a value
  in [2^e, 2^(e+1)) by at most 2^(e-8) <= |ref| * 2^-8) and ``|ref| * 2^-11 + 1e-4``
  for f16 (11 significant bits; the 1e-4 also covers the subnormal range).  A max-abs
  bound cannot hold there: a bf16 value in [1, 2) is already rounded by up to 3.9e-3.

The attention arithmetic is the plain one ("Paged Attention" glossary, paragraph 4:
paging changes where K/V live, not what attention computes), so the oracle's float64
value is the reference for both.
"""
import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.float16: 2e-3, torch.bfloat16: 2e-3}
REL = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
ABS_LOWP = 1e-4


def check_close(out, ref, dtype):
    """fp32 outputs: max-abs error against the oracle <= TOL[input dtype]."""
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= TOL[dtype], f"max-abs error {err.max():.3g} > {TOL[dtype]}"
    return float(err.max())


def check_in_dtype(out_lowp, ref):
    """An f16/bf16 output: each element within |ref| * 2^-p + 1e-4 of the oracle."""
    got = out_lowp.cpu().double().numpy()
    assert np.isfinite(got).all()
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.abs(ref) * REL[out_lowp.dtype] + ABS_LOWP
    over = np.abs(got - ref) > bound
    if over.any():
        i = np.unravel_index(np.argmax(np.abs(got - ref) - bound), ref.shape)
        raise AssertionError(f"{int(over.sum())} of {over.size} {out_lowp.dtype} outputs outside "
                             f"|ref|*2^-p + 1e-4; worst at {i}: got {got[i]!r}, oracle {ref[i]!r}")
    return float((np.abs(got - ref) / bound).max())
