"""Shared tolerance checks for GPU-vs-oracle parity (bf16 inputs, fp32 accumulation).

The bar: max |out - ref| <= 1e-2, mean |out - ref| <= 1e-3, max |lse - ref| <= 1e-3, where
the reference is the fp64 oracle evaluated on the very same rounded inputs.  Rows the oracle
marks as empty (lse = -inf) must come back as out == 0 and lse == -inf exactly.
"""
import math

import torch

MAX_ERR = 1e-2
MEAN_ERR = 1e-3
LSE_ERR = 1e-3


def check(out, lse, ref_out, ref_lse, *, max_err=MAX_ERR, mean_err=MEAN_ERR, lse_err=LSE_ERR,
          what=""):
    out = out.detach().to("cpu", torch.float64).reshape(ref_out.shape)
    ref_out = ref_out.to(torch.float64)
    assert torch.isfinite(out).all(), f"{what}: non-finite output"
    d = (out - ref_out).abs()
    assert d.max().item() <= max_err, f"{what}: max |err| {d.max().item():.3e} > {max_err}"
    assert d.mean().item() <= mean_err, f"{what}: mean |err| {d.mean().item():.3e} > {mean_err}"
    if lse is not None:
        lse = lse.detach().to("cpu", torch.float64).reshape(ref_lse.shape)
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse)), f"{what}: lse finiteness differs"
        assert torch.all(lse[~fin] == -math.inf), f"{what}: empty rows need lse = -inf"
        if fin.any():
            dl = (lse[fin] - ref_lse[fin]).abs().max().item()
            assert dl <= lse_err, f"{what}: max |lse err| {dl:.3e} > {lse_err}"
        empty = ~fin
        if empty.any():
            assert torch.all(out[empty] == 0), f"{what}: empty rows need out = 0"
    return d.max().item(), d.mean().item()
