"""The no-allocation paged decode entry point, for callers that cannot allocate device memory
(an arena allocator that owns all of it, a serving loop that must not allocate).

fa_decode_paged_noalloc takes the split-KV scratch from the library's fixed device array
instead of a caller workspace.  Called through the C ABI it must give what fa_decode_paged
(the workspace entry point) gives, within the parity tolerance, on two calls in a row -- the
second one running over the scratch the first one left behind -- and it must refuse a problem
whose scratch would not fit.  This file is collected last so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import softmax_attention_gb300 as fa
import workloads
from tests._parity import check

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kp, vp, table, lens, max_len, scale):
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = kp.shape
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.fa_decode_paged_noalloc(p(q), p(kp), p(vp), p(table), p(lens), p(out), p(lse), B,
                                     Hq, Hkv, D, page_size, table.shape[1], num_pages, max_len,
                                     scale, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_OK, fa.fa_last_error()
    return out, lse


def test_noalloc_matches_workspace_entry_point_twice():
    lib = fa.load_library()
    cases = [
        workloads.PagedCase(B=16, Hq=32, Hkv=8, D=128, page_size=16, num_pages=5000,
                            min_len=1, max_len=4096, seed=31),
        workloads.PagedCase(B=7, Hq=16, Hkv=2, D=128, page_size=16, num_pages=900,
                            min_len=0, max_len=1500, seed=32),
    ]
    for c in cases:  # two calls in a row over the same scratch array
        q, kp, vp, table, lens = (t.cuda() for t in workloads.paged_inputs(c))
        max_len = int(lens.max())
        ref_out, ref_lse = fa.fa_decode_paged(q, kp, vp, table, lens, max_len, c.sm_scale)
        out, lse = _noalloc(lib, q, kp, vp, table, lens, max_len, c.sm_scale)
        torch.cuda.synchronize()
        check(out, lse, ref_out.double().cpu(), ref_lse.double().cpu(),
              what=f"noalloc vs workspace B={c.B}")
    assert fa.fa_get_device_status() == fa.FA_OK, fa.fa_last_error()


def test_noalloc_refuses_problems_larger_than_its_scratch():
    lib = fa.load_library()
    # 1024 sequences x 64 heads x 32K tokens needs far more than the fixed array
    rc = lib.fa_decode_paged_noalloc(None, None, None, None, None, None, None, 1024, 64, 8, 128,
                                     16, 2048, 1, 32768, 0.1, None)
    assert rc == fa.FA_ERR_WORKSPACE
    assert b"scratch" in lib.fa_last_error()
