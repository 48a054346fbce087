"""GPU parity of the dense prefill kernel against the fp64 oracle, through the C ABI.

Shapes span several 128-row tiles and KV tiles with ragged tails, every supported head
dimension, grouped-query packings, causal alignment with Lq < Lkv and Lq > Lkv (empty rows),
forced KV splits (merge path), additive masks, fp16 and fp32 inputs, and the two full-size
workloads on sampled rows.
"""
import math

import pytest
import torch

import oracle
import softmax_attention_gb300 as fa
import workloads
from tests._parity import check
from tests._guard import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    yield
    assert fa.fa_get_device_status() == fa.FA_OK, fa.fa_last_error()


def _run(c: workloads.DenseCase, *, mask=None, num_splits=0, short_form=False, rows=None):
    q, k, v = workloads.dense_inputs(c)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = None if mask is None else mask.to(dev)
    og, lg = Guarded(qd.shape, qd.dtype), Guarded(qd.shape[:-1], torch.float32)
    if short_form:
        out, lse = fa.fa_prefill(qd, kd, vd, causal=c.causal, scale=c.sm_scale, out=og.view,
                                 lse=lg.view)
    else:
        out, lse = fa.fa_prefill_ex(qd, kd, vd, causal=c.causal, scale=c.sm_scale, mask=md,
                                    num_splits=num_splits, out=og.view, lse=lg.view)
    torch.cuda.synchronize()
    og.assert_intact("prefill out")
    lg.assert_intact("prefill lse")
    ref_o, ref_l = oracle.attention(q, k, v, causal=c.causal, scale=c.sm_scale, mask=mask,
                                    rows=rows)
    if rows is not None:
        out = out.reshape(-1, c.dv)[torch.as_tensor(rows, device=dev)]
        lse = lse.reshape(-1)[torch.as_tensor(rows, device=dev)]
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_fp32(causal):
    """B=1, Hq=Hkv=2, Lq=Lkv=64, D=64, fp32 N(0,1), scale 1/8."""
    c = workloads.tiny_dense(causal)
    out, lse, ro, rl = _run(c)
    assert out.dtype == torch.float32
    check(out, lse, ro, rl, what=f"tiny causal={causal}")


def _fp32_range_case(q_mag, k_mag, v_mag, seed):
    c = workloads.DenseCase(B=1, Hq=4, Hkv=2, Lq=70, Lkv=300, D=64, causal=True,
                            dtype=torch.float32, sigma=1.0, seed=seed)
    q, k, v = workloads.dense_inputs(c)
    return c, q * q_mag, k * k_mag, v * v_mag


@pytest.mark.parametrize("q_mag,k_mag,v_mag", [(1e5, 1e-5, 1e5), (1e-20, 1e20, 1e-30),
                                               (1.0, 1.0, 3e37)])
def test_fp32_keeps_range_and_precision(q_mag, k_mag, v_mag):
    # magnitudes fp16 cannot hold (above 65504, below its subnormals): fp32 inputs are not
    # narrowed, so the result matches the oracle to fp32 precision relative to its scale
    c, q, k, v = _fp32_range_case(q_mag, k_mag, v_mag, seed=17)
    dev = torch.device("cuda")
    og, lg = Guarded(q.shape, torch.float32), Guarded(q.shape[:-1], torch.float32)
    out, lse = fa.fa_prefill_ex(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=c.sm_scale,
                                out=og.view, lse=lg.view)
    torch.cuda.synchronize()
    og.assert_intact("fp32 out")
    lg.assert_intact("fp32 lse")
    ro, rl = oracle.attention(q, k, v, causal=True, scale=c.sm_scale)
    o64 = out.double().cpu()
    assert torch.isfinite(o64).all()
    rel = ((o64 - ro).abs().max() / ro.abs().max()).item()
    assert rel <= 1e-5, f"relative max error {rel:.3e}"
    assert (lse.double().cpu() - rl).abs().max().item() <= 1e-4


CASES = [
    # B, Hq, Hkv, Lq, Lkv, D, causal
    (1, 4, 4, 200, 333, 64, False),
    (2, 8, 2, 130, 260, 128, True),     # GQA 4, ragged q and kv tails
    (1, 32, 8, 96, 1100, 128, True),    # Llama-like packing, chunk at the end of context
    (1, 8, 1, 40, 700, 256, True),      # MQA, D=256
    (2, 6, 3, 77, 77, 128, True),       # G=2, square causal
    (1, 12, 4, 50, 129, 64, False),     # G=3: 42 queries per tile, 126 rows
    (1, 2, 2, 300, 40, 128, True),      # Lq > Lkv: the first 260 rows see no key
    (1, 16, 1, 33, 515, 128, False),    # G=16
    (3, 2, 1, 1, 513, 128, True),       # single query per sequence
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,D,causal", CASES)
def test_parity_shapes(B, Hq, Hkv, Lq, Lkv, D, causal):
    c = workloads.DenseCase(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lkv=Lkv, D=D, causal=causal,
                            sigma=0.5, seed=B * 7 + Lq)
    out, lse, ro, rl = _run(c)
    check(out, lse, ro, rl, what=str(c))


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_forced_splits(splits):
    c = workloads.DenseCase(B=1, Hq=8, Hkv=2, Lq=100, Lkv=900, D=128, causal=True, sigma=0.5,
                            seed=3)
    out, lse, ro, rl = _run(c, num_splits=splits)
    check(out, lse, ro, rl, what=f"splits={splits}")


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,D,causal,splits", [
    (1, 12, 4, 50, 700, 64, False, 5),    # G=3: 42 queries x 3 heads per tile; last split empty
    (2, 16, 1, 33, 515, 128, True, 4),    # G=16: 8 queries per tile, ragged last query tile
    (1, 8, 1, 37, 900, 256, True, 9),     # MQA, D=256: 16 queries x 8 heads, ragged tail
    (1, 6, 6, 300, 300, 128, True, 3),    # square causal: the early query tiles' later splits are empty
])
def test_forced_splits_shapes(B, Hq, Hkv, Lq, Lkv, D, causal, splits):
    """Split partial states of tiles whose rows are not a power of two of queries per head,
    ragged query tiles and empty splits (O = 0, lse = -inf), through the merge."""
    c = workloads.DenseCase(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lkv=Lkv, D=D, causal=causal, sigma=0.5,
                            seed=11 * splits + D)
    out, lse, ro, rl = _run(c, num_splits=splits)
    check(out, lse, ro, rl, what=f"{c} splits={splits}")


def test_short_form_matches_oracle():
    c = workloads.DenseCase(B=1, Hq=8, Hkv=2, Lq=256, Lkv=1024, D=128, causal=True, sigma=0.5)
    out, lse, ro, rl = _run(c, short_form=True)
    check(out, lse, ro, rl, what="fa_prefill short form")


@pytest.mark.parametrize("mask_dtype,mask_b", [(torch.float32, 1), (torch.bfloat16, 2)])
def test_additive_mask(mask_dtype, mask_b):
    c = workloads.DenseCase(B=2, Hq=4, Hkv=2, Lq=70, Lkv=300, D=128, causal=False, sigma=0.5)
    mask = workloads.additive_mask(mask_b, c.Lq, c.Lkv, seed=9, p_masked=0.3, dtype=mask_dtype)
    mask[..., 5, :] = float("-inf")  # a fully masked query row
    out, lse, ro, rl = _run(c, mask=mask)
    check(out, lse, ro, rl, what="mask")


@pytest.mark.parametrize("D,causal,splits", [(64, False, 0), (128, False, 0), (128, True, 3),
                                              (256, False, 0), (256, True, 2)])
def test_running_max_rises_every_tile(D, causal, splits):
    """Scores that grow along the keys by ~12 (log2 units) per key tile: every tile moves the
    running max past the lazy-rescale threshold, so O and the row sum are rescaled each time;
    with splits, the parts' log-sum-exps differ by hundreds."""
    c = workloads.DenseCase(B=1, Hq=4, Hkv=2, Lq=96, Lkv=1100, D=D, causal=causal, sigma=0.5,
                            seed=D + 5)
    q, k, v = workloads.dense_inputs(c)
    bn = 64 if D == 256 else 128
    ramp = 12.0 / (bn * 2.0 * c.sm_scale * 1.4426950408889634)  # per key, in raw score units
    q[..., 0] = 2.0
    k[..., 0] = (k[..., 0].float() + ramp * torch.arange(c.Lkv, dtype=torch.float32)).to(k.dtype)
    dev = torch.device("cuda")
    out, lse = fa.fa_prefill_ex(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=c.sm_scale,
                                num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = oracle.attention(q, k, v, causal=causal, scale=c.sm_scale)
    check(out, lse, ro, rl, what=f"rising scores D={D} causal={causal} splits={splits}")


def test_fp16_inputs():
    c = workloads.DenseCase(B=1, Hq=4, Hkv=1, Lq=150, Lkv=400, D=128, causal=True,
                            dtype=torch.float16, sigma=0.5)
    out, lse, ro, rl = _run(c)
    assert out.dtype == torch.float16
    check(out, lse, ro, rl, what="fp16")


def test_empty_kv():
    c = workloads.DenseCase(B=1, Hq=2, Hkv=2, Lq=5, Lkv=0, D=64, causal=False)
    out, lse, ro, rl = _run(c)
    assert torch.all(out == 0) and torch.all(lse == -math.inf)


def _sample_rows(total, n, seed):
    g = torch.Generator().manual_seed(seed)
    rows = torch.randperm(total, generator=g)[:n]
    return torch.sort(rows).values.tolist()


def test_gqa_prefill_chunk_full_size_sampled():
    """Llama-8B-like chunk: Hq=32, Hkv=8, D=128, Lq=512 at 15872..16383 of a 16K cache."""
    c = workloads.gqa_prefill_chunk()
    total = c.B * c.Hq * c.Lq
    rows = _sample_rows(total, 192, seed=21) + [0, total - 1]
    out, lse, ro, rl = _run(c, rows=rows)
    check(out, lse, ro, rl, what="gqa prefill chunk (sampled)")


@pytest.mark.parametrize("Lq", workloads.MQA_SWEEP_LQ)
def test_mqa_sweep_full_size_sampled(Lq):
    c = workloads.mqa_prefill(Lq)
    total = c.B * c.Hq * c.Lq
    rows = _sample_rows(total, min(total, 96), seed=Lq)
    out, lse, ro, rl = _run(c, rows=rows)
    check(out, lse, ro, rl, what=f"mqa Lq={Lq} (sampled)")
