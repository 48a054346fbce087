"""The no-allocation paged decode entry point, for callers that cannot allocate device memory
(an arena allocator that owns all of it, a serving loop that must not allocate).

fa_decode_paged_noalloc takes the split-KV scratch from the library's fixed device array
instead of a caller workspace.  Called through the C ABI it must give what fa_decode_paged
(the workspace entry point) gives, within the parity tolerance, on two calls in a row -- the
second one running over the scratch the first one left behind -- and agree with the fp64
oracle on sampled rows.  Every case here takes a plan that uses scratch (a split KV loop and a
merge), on each of the two decode kernels.  The outputs sit in guarded buffers (NaN-filled,
canaries on both sides), so an element the call never writes or a write past an output fails.
It must also refuse a problem whose scratch would not fit, and check its arguments before
that.  This file is collected last so that a run stopping at its first failure has already
run every other test.
"""
import ctypes

import pytest
import torch

import oracle
import softmax_attention_gb300 as fa
import workloads
from tests._guard import Guarded
from tests._parity import check

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kp, vp, table, lens, max_len, scale, out, lse):
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = kp.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.fa_decode_paged_noalloc(p(q), p(kp), p(vp), p(table), p(lens), p(out), p(lse), B,
                                       Hq, Hkv, D, page_size, table.shape[1], num_pages, max_len,
                                       scale,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # a few long sequences: the chunked CUDA-core kernel, chunk states in the scratch
    workloads.PagedCase(B=4, Hq=32, Hkv=8, D=128, page_size=16, num_pages=1200, min_len=1,
                        max_len=4096, seed=31),
    # an empty sequence among them
    workloads.PagedCase(B=7, Hq=16, Hkv=2, D=128, page_size=16, num_pages=900, min_len=0,
                        max_len=1500, seed=32),
    # a group of three heads: the tensor-core kernel with a split KV loop
    workloads.PagedCase(B=2, Hq=12, Hkv=4, D=128, page_size=16, num_pages=700, min_len=3000,
                        max_len=5000, seed=33),
]


@pytest.mark.parametrize("c", CASES, ids=["cuda_cores", "with_empty", "tensor_cores_split"])
def test_noalloc_matches_workspace_entry_point_twice(c):
    lib = fa.load_library()
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    qd, kd, vd, td, ld = (t.cuda() for t in (q, kp, vp, table, lens))
    max_len = int(lens.max())
    plan = fa.fa_decode_get_plan(qd, kd, vd, td, ld, max_len)
    assert plan["launches"] == 2 and plan["workspace_bytes"] > 0  # the scratch is used
    ref_out, ref_lse = fa.fa_decode_paged(qd, kd, vd, td, ld, max_len, c.sm_scale)
    rows = list(range(0, c.B * c.Hq, 5))
    o64, l64 = oracle.decode_paged(q, kp, vp, table, lens, scale=c.sm_scale, rows=rows)
    idx = torch.as_tensor(rows, device="cuda")
    for call in range(2):  # two calls in a row over the same scratch array
        og, lg = Guarded(qd.shape, qd.dtype), Guarded(qd.shape[:-1], torch.float32)
        rc = _noalloc(lib, qd, kd, vd, td, ld, max_len, c.sm_scale, og.view, lg.view)
        assert rc == fa.FA_OK, fa.fa_last_error()
        torch.cuda.synchronize()
        og.assert_intact(f"noalloc out, call {call}")
        lg.assert_intact(f"noalloc lse, call {call}")
        check(og.view, lg.view, ref_out.double().cpu(), ref_lse.double().cpu(),
              what=f"noalloc vs workspace B={c.B}, call {call}")
        check(og.view.reshape(-1, c.D)[idx], lg.view.reshape(-1)[idx], o64, l64,
              what=f"noalloc vs oracle B={c.B}, call {call}")
    assert fa.fa_get_device_status() == fa.FA_OK, fa.fa_last_error()


def test_noalloc_refuses_problems_larger_than_its_scratch():
    lib = fa.load_library()
    t = torch.empty(64, dtype=torch.bfloat16, device="cuda")  # valid pointers; nothing runs
    p = ctypes.c_void_p(t.data_ptr())
    # 1024 sequences x 64 heads x 32K tokens in 1-token pages: the chunked kernel's states
    # need far more than the fixed array
    rc = lib.fa_decode_paged_noalloc(p, p, p, p, p, p, p, 1024, 64, 8, 128, 1, 32768, 1, 32768,
                                     0.1, None)
    assert rc == fa.FA_ERR_WORKSPACE
    assert b"scratch" in lib.fa_last_error()
    # a malformed call is refused for its bad argument, not for the scratch
    rc = lib.fa_decode_paged_noalloc(p, p, p, p, p, None, p, 1024, 64, 8, 128, 1, 32768, 1,
                                     32768, 0.1, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    rc = lib.fa_decode_paged_noalloc(p, p, p, p, p, p, p, 1024, 64, 8, 96, 1, 32768, 1, 32768,
                                     0.1, None)
    assert rc == fa.FA_ERR_UNSUPPORTED
