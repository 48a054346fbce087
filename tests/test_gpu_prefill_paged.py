"""GPU parity of the paged prefill (a query chunk at the end of each sequence, K/V read
through a page table) against the fp64 oracle, through the C ABI.

Cases cover every head dimension and page size class, grouped-query packings, ragged
sequence lengths including sequences shorter than the chunk (rows with no key) and empty
ones, causal and non-causal, the full-size workload on sampled rows, bit-exact equality with
the dense kernel on the gathered cache, and device-side bounds errors.
"""
import pytest
import torch

import oracle
import softmax_attention_gb300 as fa
import workloads
from tests._guard import Guarded
from tests._parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    yield
    assert fa.fa_get_device_status() == fa.FA_OK, fa.fa_last_error()


def _run(c: workloads.PagedPrefillCase, rows=None):
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    qd, kd, vd, td, ld = (t.cuda() for t in (q, kp, vp, table, lens))
    max_len = int(lens.max()) if c.B else 0
    og, lg = Guarded(qd.shape, qd.dtype), Guarded(qd.shape[:-1], torch.float32)
    out, lse = fa.fa_prefill_paged(qd, kd, vd, td, ld, max_len, causal=c.causal,
                                   scale=c.sm_scale, out=og.view, lse=lg.view)
    torch.cuda.synchronize()
    og.assert_intact("paged prefill out")
    lg.assert_intact("paged prefill lse")
    ro, rl = oracle.prefill_paged(q, kp, vp, table, lens, causal=c.causal, scale=c.sm_scale,
                                  rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, device="cuda")
        out, lse = out.reshape(-1, c.D)[idx], lse.reshape(-1)[idx]
    return out, lse, ro, rl


CASES = [
    # B, Hq, Hkv, Lq, lens, D, page_size, causal
    (2, 8, 2, 100, [700, 150], 128, 16, True),
    (3, 4, 4, 64, [64, 1000, 10], 64, 8, True),        # a sequence shorter than the chunk
    (1, 8, 1, 40, [333], 256, 64, True),               # D = 256 (64-key tiles)
    (2, 32, 8, 33, [2049, 0], 128, 128, False),        # non-causal, an empty sequence
    (4, 12, 4, 50, [129, 128, 127, 1], 64, 32, True),  # G = 3, lengths around a tile
    (1, 16, 1, 7, [4000], 128, 16, True),              # G = 16
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,lens,D,ps,causal", CASES)
def test_parity_shapes(B, Hq, Hkv, Lq, lens, D, ps, causal):
    need = sum(-(-n // ps) for n in lens)
    c = workloads.PagedPrefillCase(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, page_size=ps,
                                   num_pages=need + 7, min_len=0, max_len=max(lens),
                                   causal=causal, seq_lens=lens, seed=B + Lq + ps)
    out, lse, ro, rl = _run(c)
    check(out, lse, ro, rl, what=f"paged prefill {lens} D={D} ps={ps}")


def test_full_size_sampled():
    c = workloads.paged_gqa_prefill()
    rows = list(range(0, c.B * c.Hq * c.Lq, 613))
    out, lse, ro, rl = _run(c, rows=rows)
    check(out, lse, ro, rl, what="paged_gqa_prefill (sampled)")


def test_paged_equals_dense_on_gathered_cache_bit_exact():
    """One sequence: the paged call and the dense call on the same keys in order run the
    same plan and arithmetic, so they agree bit for bit."""
    c = workloads.PagedPrefillCase(B=1, Hq=8, Hkv=2, Lq=200, D=128, page_size=16,
                                   num_pages=200, min_len=0, max_len=1500, seq_lens=[1500],
                                   seed=3)
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    n = int(lens[0])
    pages = table[0, : -(-n // c.page_size)].long()
    kd = kp[pages].permute(1, 0, 2, 3).reshape(1, c.Hkv, -1, c.D)[:, :, :n].contiguous()
    vd = vp[pages].permute(1, 0, 2, 3).reshape(1, c.Hkv, -1, c.D)[:, :, :n].contiguous()
    o1, l1 = fa.fa_prefill_paged(*(t.cuda() for t in (q, kp, vp, table, lens)), n, causal=True,
                                 scale=c.sm_scale)
    o2, l2 = fa.fa_prefill_ex(q.cuda(), kd.cuda(), vd.cuda(), causal=True, scale=c.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_out_of_range_page_is_reported():
    c = workloads.PagedPrefillCase(B=2, Hq=4, Hkv=2, Lq=16, D=64, page_size=8, num_pages=40,
                                   min_len=0, max_len=100, seq_lens=[100, 30], seed=4)
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    bad = table.clone()
    bad[1, 2] = c.num_pages  # a page inside sequence 1 (its keys 16..23)
    fa.fa_prefill_paged(*(t.cuda() for t in (q, kp, vp, bad, lens)), 100, scale=c.sm_scale)
    assert fa.fa_get_device_status() == fa.FA_ERR_BOUNDS
    assert fa.fa_get_device_status() == fa.FA_OK
    long = lens.clone()
    long[0] = table.shape[1] * c.page_size + 1  # longer than its page table can hold
    fa.fa_prefill_paged(*(t.cuda() for t in (q, kp, vp, table, long)), 100, scale=c.sm_scale)
    assert fa.fa_get_device_status() == fa.FA_ERR_BOUNDS
    assert fa.fa_get_device_status() == fa.FA_OK
