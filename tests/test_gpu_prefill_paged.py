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
    (2, 8, 2, 30, [515, 90], 256, 8, True),            # D = 256, eight pages a tile
    (1, 4, 1, 20, [300], 128, 8, False),               # 8-key pages, one row group each
    (2, 8, 4, 10, [260, 129], 64, 128, True),          # D = 64, a page per tile
    (4, 8, 2, 24, [500, 500, 200, 500], 128, 16, True),  # equal lengths (ties in the order)
    (70, 4, 2, 3, [(37 * i) % 300 + 1 for i in range(70)], 64, 8, True),  # > 64 sequences:
                                                        # no longest-first order
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,lens,D,ps,causal", CASES)
def test_parity_shapes(B, Hq, Hkv, Lq, lens, D, ps, causal):
    need = sum(-(-n // ps) for n in lens)
    c = workloads.PagedPrefillCase(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, D=D, page_size=ps,
                                   num_pages=need + 7, min_len=0, max_len=max(lens),
                                   causal=causal, seq_lens=lens, seed=B + Lq + ps)
    out, lse, ro, rl = _run(c)
    check(out, lse, ro, rl, what=f"paged prefill {lens} D={D} ps={ps}")


@pytest.mark.parametrize("D,ps", [(128, 16), (256, 64)])
def test_running_max_rises_every_tile(D, ps):
    """Scores that grow along each sequence's keys by ~12 (log2 units) per key tile, so every
    tile moves the running max past the lazy-rescale threshold (the paged instantiations
    reduce the tile max differently from the dense one)."""
    c = workloads.PagedPrefillCase(B=2, Hq=8, Hkv=2, Lq=40, D=D, page_size=ps, num_pages=120,
                                   min_len=0, max_len=1100, seq_lens=[1100, 700], causal=True,
                                   seed=D + ps)
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    bn = 64 if D == 256 else 128
    ramp = 12.0 / (bn * 2.0 * c.sm_scale * 1.4426950408889634)  # per key, in raw score units
    q[..., 0] = 2.0
    for b in range(c.B):
        n = int(lens[b])
        for pi in range(-(-n // ps)):
            keys = pi * ps + torch.arange(ps, dtype=torch.float32)
            page = int(table[b, pi])
            kp[page, :, :, 0] = (kp[page, :, :, 0].float() + ramp * keys).to(kp.dtype)
    qd, kd, vd, td, ld = (t.cuda() for t in (q, kp, vp, table, lens))
    out, lse = fa.fa_prefill_paged(qd, kd, vd, td, ld, int(lens.max()), causal=True,
                                   scale=c.sm_scale)
    torch.cuda.synchronize()
    ro, rl = oracle.prefill_paged(q, kp, vp, table, lens, causal=True, scale=c.sm_scale)
    check(out, lse, ro, rl, what=f"paged rising scores D={D} page={ps}")


def test_full_size_sampled():
    c = workloads.paged_gqa_prefill()
    rows = list(range(0, c.B * c.Hq * c.Lq, 613))
    out, lse, ro, rl = _run(c, rows=rows)
    check(out, lse, ro, rl, what="paged_gqa_prefill (sampled)")


def test_paged_equals_dense_gathered_bit_exact():
    """Page-table indexing, bit for bit: the sequence's pages reached through a permuted page
    table and the same pages laid out in order (identity table) give identical results, with
    the same split count.  The dense call on the gathered keys agrees within the parity
    tolerance (the dense and paged instantiations may tile the keys differently)."""
    c = workloads.PagedPrefillCase(B=1, Hq=8, Hkv=2, Lq=200, D=128, page_size=16,
                                   num_pages=200, min_len=0, max_len=1500, seq_lens=[1500],
                                   seed=3)
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    n = int(lens[0])
    np_ = -(-n // c.page_size)
    pages = table[0, :np_].long()
    id_table = torch.full_like(table, -1)
    id_table[0, :np_] = torch.arange(np_, dtype=torch.int32)
    kg, vg = kp[pages].contiguous(), vp[pages].contiguous()
    o1, l1 = fa.fa_prefill_paged(*(t.cuda() for t in (q, kp, vp, table, lens)), n, causal=True,
                                 scale=c.sm_scale, num_splits=3)
    o2, l2 = fa.fa_prefill_paged(*(t.cuda() for t in (q, kg, vg, id_table, lens)), n,
                                 causal=True, scale=c.sm_scale, num_splits=3)
    kd = kg.permute(1, 0, 2, 3).reshape(1, c.Hkv, -1, c.D)[:, :, :n].contiguous()
    vd = vg.permute(1, 0, 2, 3).reshape(1, c.Hkv, -1, c.D)[:, :, :n].contiguous()
    o3, l3 = fa.fa_prefill_ex(q.cuda(), kd.cuda(), vd.cuda(), causal=True, scale=c.sm_scale,
                              num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    check(o1, l1, o3.cpu().double(), l3.cpu().double(), what="paged vs dense on gathered keys")


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


def _inputs_on_gpu(c):
    q, kp, vp, table, lens = workloads.paged_prefill_inputs(c)
    return (q, kp, vp, table, lens), [t.cuda() for t in (q, kp, vp, table, lens)]


def test_fp16():
    c = workloads.PagedPrefillCase(B=2, Hq=8, Hkv=2, Lq=70, D=128, page_size=16, num_pages=120,
                                   min_len=0, max_len=900, seq_lens=[900, 60],
                                   dtype=torch.float16, seed=6)
    (q, kp, vp, table, lens), dev = _inputs_on_gpu(c)
    out, lse = fa.fa_prefill_paged(*dev, 900, scale=c.sm_scale)
    torch.cuda.synchronize()
    assert out.dtype == torch.float16
    ro, rl = oracle.prefill_paged(q, kp, vp, table, lens, scale=c.sm_scale)
    check(out, lse, ro, rl, what="paged prefill fp16")


@pytest.mark.parametrize("mask_dtype,per_seq", [(torch.bfloat16, True), (torch.float32, False)])
def test_additive_mask(mask_dtype, per_seq):
    """A llama.cpp-style explicit mask [1 or B, Lq, max_len] (here non-causal with -inf
    holes and finite biases), the paged counterpart of small-batch decode with a KQ mask."""
    c = workloads.PagedPrefillCase(B=3, Hq=8, Hkv=4, Lq=6, D=64, page_size=8, num_pages=100,
                                   min_len=0, max_len=500, seq_lens=[500, 37, 6], causal=False,
                                   seed=8)
    (q, kp, vp, table, lens), dev = _inputs_on_gpu(c)
    g = torch.Generator().manual_seed(11)
    mb = c.B if per_seq else 1
    mask = (torch.randn(mb, c.Lq, c.max_len, generator=g) * 0.5).to(mask_dtype)
    mask[:, :, 5::7] = -float("inf")
    out, lse = fa.fa_prefill_paged(*dev, c.max_len, causal=False, scale=c.sm_scale,
                                   mask=mask.cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.prefill_paged(q, kp, vp, table, lens, causal=False, scale=c.sm_scale,
                                  mask=mask)
    check(out, lse, ro, rl, what=f"paged prefill mask {mask_dtype} per_seq={per_seq}")


@pytest.mark.parametrize("splits", [2, 5])
def test_forced_splits(splits):
    c = workloads.PagedPrefillCase(B=2, Hq=8, Hkv=2, Lq=40, D=128, page_size=32, num_pages=90,
                                   min_len=0, max_len=1200, seq_lens=[1200, 300], seed=9)
    (q, kp, vp, table, lens), dev = _inputs_on_gpu(c)
    out, lse = fa.fa_prefill_paged(*dev, 1200, scale=c.sm_scale, num_splits=splits)
    torch.cuda.synchronize()
    ro, rl = oracle.prefill_paged(q, kp, vp, table, lens, scale=c.sm_scale)
    check(out, lse, ro, rl, what=f"paged prefill splits={splits}")


def test_positional_entry_point_matches_the_struct_one():
    c = workloads.PagedPrefillCase(B=2, Hq=8, Hkv=2, Lq=50, D=128, page_size=16, num_pages=90,
                                   min_len=0, max_len=1000, seq_lens=[1000, 200], seed=10)
    _, (qd, kd, vd, td, ld) = _inputs_on_gpu(c)
    lib = fa.load_library()
    o1, l1 = fa.fa_prefill_paged(qd, kd, vd, td, ld, 1000, scale=c.sm_scale)
    o2 = torch.empty_like(qd)
    l2 = torch.empty(c.B, c.Hq, c.Lq, dtype=torch.float32, device="cuda")
    n = lib.fa_prefill_paged_workspace_size(c.B, c.Hq, c.Hkv, c.Lq, c.D, 1000)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    rc = lib.fa_prefill_paged(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), td.data_ptr(),
                              ld.data_ptr(), o2.data_ptr(), l2.data_ptr(), c.B, c.Hq, c.Hkv,
                              c.Lq, c.D, c.page_size, td.shape[1], c.num_pages, 1000, 1,
                              c.sm_scale, ws.data_ptr(), n,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK, fa.fa_last_error()
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
