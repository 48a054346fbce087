"""GPU parity of MLA paged decode (latent form: ckv is K and V, kpe adds the rope term)
against the fp64 oracle, through the C ABI; bit-exact paging; the bounds-error path."""
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


def _run(c: workloads.MlaCase, rows=None):
    qn, qp, ckv, kpe, table, lens = workloads.mla_inputs(c)
    dev = [t.cuda() for t in (qn, qp, ckv, kpe, table, lens)]
    og, lg = Guarded(dev[0].shape, dev[0].dtype), Guarded(dev[0].shape[:-1], torch.float32)
    out, lse = fa.mla_decode_paged(*dev, c.max_len, c.scale, out=og.view, lse=lg.view)
    torch.cuda.synchronize()
    og.assert_intact("mla out")
    lg.assert_intact("mla lse")
    ro, rl = oracle.mla_decode_paged(qn, qp, ckv, kpe, table, lens, scale=c.scale, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, device="cuda")
        out, lse = out.reshape(-1, c.Dc)[idx], lse.reshape(-1)[idx]
    return out, lse, ro, rl


@pytest.mark.parametrize("lens,ps", [
    ([1, 31, 32, 33], 1),
    ([63, 64, 65, 700], 1),
    ([511, 512, 513, 1500], 1),
    ([0, 5, 1024], 1),
    ([17, 300, 1030], 16),
    ([200, 64], 64),
    ([0, 100], 1),          # one chunk per sequence: final output written directly
    ([40, 200, 31], 8),     # 8-token pages: four TMA page slices per stage
    ([100, 500, 33], 32),   # a stage is one 32-token page
    ([300, 129], 128),      # a stage is a slice of a page
])
def test_parity_shapes(lens, ps):
    c = workloads.MlaCase(B=len(lens), H=64, seq_len=None, seq_lens=lens, page_size=ps,
                          seed=len(lens) + ps)
    out, lse, ro, rl = _run(c)
    check(out, lse, ro, rl, what=f"mla {lens} ps={ps}")


@pytest.mark.parametrize("ps", [1, 64])
def test_running_max_rises_every_tile(ps):
    """Scores that grow along each sequence by ~0.2 (log2 units) per token, ~13 per 64-token
    tile: every tile moves the running max past the lazy-rescale threshold.  The ramp is put
    on the rope part (kpe, q_pe), which enters the scores but not the values."""
    c = workloads.MlaCase(B=2, H=64, seq_len=None, seq_lens=[2000, 900], page_size=ps, seed=ps + 3)
    qn, qp, ckv, kpe, table, lens = workloads.mla_inputs(c)
    ramp = 0.2 / (2.0 * c.scale * 1.4426950408889634)  # per token, in raw score units
    qp[..., 0] = 2.0
    for b in range(c.B):
        n = int(lens[b])
        for pi in range(-(-n // ps)):
            toks = pi * ps + torch.arange(ps, dtype=torch.float32)
            page = int(table[b, pi])
            kpe[page, :, 0] = (kpe[page, :, 0].float() + ramp * toks).to(kpe.dtype)
    dev = [t.cuda() for t in (qn, qp, ckv, kpe, table, lens)]
    out, lse = fa.mla_decode_paged(*dev, c.max_len, c.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.mla_decode_paged(qn, qp, ckv, kpe, table, lens, scale=c.scale)
    check(out, lse, ro, rl, what=f"mla rising scores ps={ps}")


@pytest.mark.parametrize("H,lens,ps", [
    (16, [100, 700, 0], 1),      # one tensor-parallel shard's heads: a partial head group
    (32, [513, 64], 16),
    (128, [300, 1500, 65], 1),   # two head groups per sequence
    (96, [200, 129], 64),        # a full and a partial group
    (128, [4000, 100], 1),       # several chunks per sequence, merged
    (1, [77], 1),
])
def test_head_counts(H, lens, ps):
    c = workloads.MlaCase(B=len(lens), H=H, seq_len=None, seq_lens=lens, page_size=ps,
                          seed=H + len(lens))
    out, lse, ro, rl = _run(c)
    check(out, lse, ro, rl, what=f"mla H={H} {lens} ps={ps}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_short_last_wave_is_split(dtype):
    """More sequences than SMs, one chunk each: the sequences of the short last wave are cut
    into chunks and merged, the others written directly.  The cut ones include an empty
    sequence and lengths around the 64-token tile and the chunk."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tail = [0, 1, 63, 64, 65, 129, 130, 100]
    lens = [130 - (i % 7) for i in range(sms)] + tail
    c = workloads.MlaCase(B=len(lens), H=64, seq_len=None, seq_lens=lens, dtype=dtype, seed=3)
    assert fa.load_library().mla_decode_workspace_size(c.B, c.H, c.Dc, c.max_len) > 0
    out, lse, ro, rl = _run(c)
    check(out, lse, ro, rl, what=f"mla short last wave {dtype}")


@pytest.mark.parametrize("batch,seq", [(128, 2048), (768, 1024), (64, 1024), (64, 2048),
                                       (128, 1024), (768, 2048)])
def test_mla_full_size_sampled(batch, seq):
    """The MLA grid of the flashinfer PR's results section, on sampled (sequence, head) rows."""
    c = workloads.mla_decode(batch, seq)
    rows = list(range(0, c.B * c.H, 97 if batch == 768 else 41))
    out, lse, ro, rl = _run(c, rows=rows)
    check(out, lse, ro, rl, what=f"mla b{batch} s{seq} (sampled)")


@pytest.mark.parametrize("ps", [8, 16, 64])
def test_page_copies_equal_row_gathers_bit_exact(ps):
    """Full stages of pages >= 8 tokens are copied with TMA boxes, pages of one token are
    gathered row by row; both fill the stage ring with the same bytes, so the same tokens
    give bit-identical results either way."""
    c = workloads.MlaCase(B=3, H=64, seq_len=None, seq_lens=[700, 1500, 65], page_size=ps,
                          seed=ps)
    qn, qp, ckv, kpe, table, lens = workloads.mla_inputs(c)
    P = ckv.shape[0]
    ckv1 = ckv.reshape(P * ps, 1, c.Dc)
    kpe1 = kpe.reshape(P * ps, 1, c.Dr)
    t = torch.arange(c.max_len)
    table1 = torch.full((c.B, c.max_len), -1, dtype=torch.int32)
    for b in range(c.B):
        n = int(lens[b])
        pages = table[b, (t[:n] // ps)].long()
        table1[b, :n] = (pages * ps + t[:n] % ps).to(torch.int32)
    o1, l1 = fa.mla_decode_paged(*[x.cuda() for x in (qn, qp, ckv, kpe, table, lens)],
                                 c.max_len, c.scale)
    o2, l2 = fa.mla_decode_paged(*[x.cuda() for x in (qn, qp, ckv1, kpe1, table1, lens)],
                                 c.max_len, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mla_64_token_pages_full_size_sampled():
    c = workloads.mla_decode(128, 2048, page_size=64)
    rows = list(range(0, c.B * c.H, 53))
    out, lse, ro, rl = _run(c, rows=rows)
    check(out, lse, ro, rl, what="mla b128 s2048 ps64 (sampled)")


def test_paged_equals_dense_gathered_bit_exact():
    c = workloads.MlaCase(B=4, H=64, seq_len=None, seq_lens=[900, 1, 1025, 333], seed=7)
    qn, qp, ckv, kpe, table, lens = workloads.mla_inputs(c)
    order, id_table, pos = [], torch.full_like(table, -1), 0
    for b in range(c.B):
        n = int(lens[b])
        order.append(table[b, :n].long())
        id_table[b, :n] = torch.arange(pos, pos + n, dtype=torch.int32)
        pos += n
    order = torch.cat(order)
    o1, l1 = fa.mla_decode_paged(*[t.cuda() for t in (qn, qp, ckv, kpe, table, lens)],
                                 c.max_len, c.scale)
    o2, l2 = fa.mla_decode_paged(*[t.cuda() for t in (qn, qp, ckv[order].contiguous(),
                                                      kpe[order].contiguous(), id_table, lens)],
                                 c.max_len, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_states_then_merge_equals_full_call():
    c = workloads.MlaCase(B=3, H=64, seq_len=None, seq_lens=[1300, 40, 0], seed=9)
    dev = [t.cuda() for t in workloads.mla_inputs(c)]
    out, lse = fa.mla_decode_paged(*dev, c.max_len, c.scale)
    op, ol, chunk = fa.mla_decode_paged_states(*dev, c.max_len, c.scale)
    lens = dev[5].long().cpu()
    n = torch.repeat_interleave((lens + chunk - 1) // chunk, c.H).to(torch.int32)
    out2, lse2 = fa.fa_merge_states(op, ol, n.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out.reshape(-1, c.Dc), out2) and torch.equal(lse.reshape(-1), lse2)


def test_out_of_range_page_is_reported():
    c = workloads.MlaCase(B=2, H=64, seq_len=None, seq_lens=[100, 50], seed=3)
    qn, qp, ckv, kpe, table, lens = workloads.mla_inputs(c)
    table[0, 10] = 10 ** 7
    fa.mla_decode_paged(*[t.cuda() for t in (qn, qp, ckv, kpe, table, lens)], c.max_len, c.scale)
    assert fa.fa_get_device_status() == fa.FA_ERR_BOUNDS
    assert fa.fa_get_device_status() == fa.FA_OK


@pytest.mark.parametrize("lens", [[300, 1, 2048], [100, 0]])
def test_fp16(lens):
    """fp16 operands (the tensor cores' f16 kind with fp16 on both sides); the first case
    splits sequences into chunks and merges, the second writes the output directly."""
    c = workloads.MlaCase(B=len(lens), H=64, seq_len=None, seq_lens=lens, page_size=1,
                          dtype=torch.float16, seed=len(lens) + 17)
    out, lse, ro, rl = _run(c)
    assert out.dtype == torch.float16
    check(out, lse, ro, rl, what=f"mla fp16 {lens}")
