"""GPU parity of split-KV paged GQA decode against the fp64 oracle, through the C ABI, on
both decode kernels (the chunked CUDA-core kernel with its merge, and the paged attention
kernel on the tensor cores), plus the bit-exact paging check: the same kernel on a page pool
with a random table and on the dense-gathered cache with an identity table must give
identical bytes."""
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


def _gpu(*ts):
    return [t.to("cuda") for t in ts]


AUTO, CC, TC = fa.FA_DECODE_AUTO, fa.FA_DECODE_CUDA_CORES, fa.FA_DECODE_TENSOR_CORES


def _run(c: workloads.PagedCase, rows=None, path=AUTO):
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    qd, kd, vd, td, ld = _gpu(q, kp, vp, table, lens)
    max_len = int(lens.max()) if c.B else 0
    og, lg = Guarded(qd.shape, qd.dtype), Guarded(qd.shape[:-1], torch.float32)
    out, lse = fa.fa_decode_paged(qd, kd, vd, td, ld, max_len, c.sm_scale, out=og.view, lse=lg.view,
                                  path=path)
    torch.cuda.synchronize()
    og.assert_intact("decode out")
    lg.assert_intact("decode lse")
    ro, rl = oracle.decode_paged(q, kp, vp, table, lens, scale=c.sm_scale, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, device="cuda")
        out, lse = out.reshape(-1, c.D)[idx], lse.reshape(-1)[idx]
    return out, lse, ro, rl


CASES = [
    # B, Hq, Hkv, D, page_size, lens
    (4, 32, 8, 128, 16, [1, 15, 16, 17]),
    (3, 8, 2, 128, 16, [1023, 1024, 1025]),
    (5, 16, 4, 128, 16, [0, 5, 513, 2048, 4096]),
    (2, 8, 8, 128, 16, [300, 77]),        # G = 1
    (2, 16, 2, 128, 32, [600, 1031]),     # G = 8, 32-token pages
    (2, 8, 2, 64, 16, [129, 1000]),
    (2, 8, 2, 256, 16, [129, 700]),
    (3, 8, 1, 64, 64, [64, 65, 2000]),    # G = 8, D = 64
    (2, 4, 2, 128, 8, [9, 100]),          # pages smaller than a 16-token block
    (2, 4, 2, 128, 1, [3, 40]),           # page_size 1
    (2, 16, 1, 64, 16, [200, 33]),        # G = 16
    (2, 4, 2, 256, 4, [50, 17]),          # G = 2, D = 256, 4-token pages
    (1, 8, 4, 128, 256, [600]),           # pages larger than a 16-token block
    # groups only the tensor-core kernel takes
    (2, 12, 4, 128, 16, [700, 129]),      # G = 3
    (2, 64, 4, 128, 16, [1000, 1]),       # G = 16 at D = 128
    (1, 40, 8, 128, 32, [2049]),          # G = 5
    (2, 48, 1, 64, 8, [300, 77]),         # G = 48
    (1, 32, 1, 256, 64, [900]),           # G = 32 at D = 256
]


def _supports(B, Hq, Hkv, D, ps, path):
    G = Hq // Hkv
    if path == CC:
        return G <= 16 and (G & (G - 1)) == 0 and G * D <= 1024
    if path == TC:
        return 8 <= ps <= (64 if D == 256 else 128)
    return True


@pytest.mark.parametrize("path", [AUTO, CC, TC], ids=["auto", "cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("B,Hq,Hkv,D,ps,lens", CASES)
def test_parity_shapes(B, Hq, Hkv, D, ps, lens, path):
    if not _supports(B, Hq, Hkv, D, ps, path):
        pytest.skip("shape outside this kernel's range")
    need = sum(-(-n // ps) for n in lens)
    c = workloads.PagedCase(B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, num_pages=need + 7,
                            min_len=0, max_len=max(lens), seq_lens=lens, seed=B + D)
    out, lse, ro, rl = _run(c, path=path)
    check(out, lse, ro, rl, what=f"{lens} path {path}")


@pytest.mark.parametrize("path", [CC, TC], ids=["cuda_cores", "tensor_cores"])
def test_running_max_rises_every_tile(path):
    """Scores that grow along each sequence by ~0.2 (log2 units) per token: every key tile
    (and every CUDA-core chunk) moves the running max past the lazy-rescale threshold."""
    c = workloads.PagedCase(B=3, Hq=32, Hkv=8, D=128, page_size=16, num_pages=200, min_len=1,
                            max_len=1500, seq_lens=[1500, 900, 40], seed=17)
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    ramp = 0.2 / (2.0 * c.sm_scale * 1.4426950408889634)  # per token, in raw score units
    q[..., 0] = 2.0
    for b in range(c.B):
        n = int(lens[b])
        for pi in range(-(-n // c.page_size)):
            toks = pi * c.page_size + torch.arange(c.page_size, dtype=torch.float32)
            page = int(table[b, pi])
            kp[page, :, :, 0] = (kp[page, :, :, 0].float() + ramp * toks).to(kp.dtype)
    out, lse = fa.fa_decode_paged(*_gpu(q, kp, vp, table, lens), int(lens.max()), c.sm_scale,
                                  path=path)
    torch.cuda.synchronize()
    ro, rl = oracle.decode_paged(q, kp, vp, table, lens, scale=c.sm_scale)
    check(out, lse, ro, rl, what=f"decode rising scores path {path}")


@pytest.mark.parametrize("path", [CC, TC], ids=["cuda_cores", "tensor_cores"])
def test_paged_equals_dense_gathered_bit_exact(path):
    c = workloads.PagedCase(B=6, Hq=32, Hkv=8, D=128, page_size=16, num_pages=2000, min_len=1,
                            max_len=3000, seed=5)
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    # dense-gathered pool: sequence b's pages laid out in order, identity page table
    pages = []
    id_table = torch.full_like(table, -1)
    pos = 0
    for b in range(c.B):
        n = -(-int(lens[b]) // c.page_size)
        pages.append(table[b, :n].long())
        id_table[b, :n] = torch.arange(pos, pos + n, dtype=torch.int32)
        pos += n
    order = torch.cat(pages)
    kd_pool, vd_pool = kp[order].contiguous(), vp[order].contiguous()
    max_len = int(lens.max())
    o1, l1 = fa.fa_decode_paged(*_gpu(q, kp, vp, table, lens), max_len, c.sm_scale, path=path)
    o2, l2 = fa.fa_decode_paged(*_gpu(q, kd_pool, vd_pool, id_table, lens), max_len, c.sm_scale,
                                path=path)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("path", [AUTO, CC], ids=["auto", "cuda_cores"])
def test_paged_gqa_decode_full_size(path):
    """batch 128, Hq=32, Hkv=8, D=128, lens ~ U{1024..4096}, page_size 16, 40000-page pool."""
    c = workloads.paged_gqa_decode()
    rows = list(range(0, c.B * c.Hq, 7))
    out, lse, ro, rl = _run(c, rows=rows, path=path)
    check(out, lse, ro, rl, what=f"paged decode full size (every 7th row), path {path}")


def test_full_size_plan_is_the_tensor_core_kernel_unsplit():
    c = workloads.paged_gqa_decode()
    q, kp, vp, table, lens = _gpu(*workloads.paged_inputs(c))
    plan = fa.fa_decode_get_plan(q, kp, vp, table, lens, int(lens.max()))
    assert plan == {"path": TC, "n_splits": 1, "launches": 1, "workspace_bytes": 0}


@pytest.mark.parametrize("path", [CC, TC], ids=["cuda_cores", "tensor_cores"])
def test_out_of_range_page_is_reported_not_read(path):
    c = workloads.PagedCase(B=2, Hq=8, Hkv=2, D=128, page_size=16, num_pages=64, min_len=0,
                            max_len=200, seq_lens=[100, 200], seed=2)
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    bad = table.clone()
    bad[1, 3] = 10 ** 6
    fa.fa_decode_paged(*_gpu(q, kp, vp, bad, lens), 200, c.sm_scale, path=path)
    assert fa.fa_get_device_status() == fa.FA_ERR_BOUNDS
    assert fa.fa_get_device_status() == fa.FA_OK  # the status is cleared by reading it


def test_states_then_merge_equals_full_call():
    c = workloads.PagedCase(B=5, Hq=16, Hkv=4, D=128, page_size=16, num_pages=900, min_len=0,
                            max_len=2500, seed=11)
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    args = _gpu(q, kp, vp, table, lens)
    max_len = int(lens.max())
    out, lse = fa.fa_decode_paged(*args, max_len, c.sm_scale, path=CC)
    op, ol, chunk = fa.fa_decode_paged_states(*args, max_len, c.sm_scale)
    n = torch.repeat_interleave((lens.long() + chunk - 1) // chunk, c.Hq).to(torch.int32)
    out2, lse2 = fa.fa_merge_states(op, ol, n.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out.reshape(-1, c.D), out2) and torch.equal(lse.reshape(-1), lse2)


@pytest.mark.parametrize("path", [CC, TC], ids=["cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("D,Hq,Hkv,ps", [(128, 32, 8, 16), (64, 8, 1, 32)])
def test_fp16(D, Hq, Hkv, ps, path):
    c = workloads.PagedCase(B=5, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, num_pages=400, min_len=0,
                            max_len=1500, dtype=torch.float16, seed=D + Hq)
    out, lse, ro, rl = _run(c, path=path)
    assert out.dtype == torch.float16
    check(out, lse, ro, rl, what=f"decode fp16 D={D}")
