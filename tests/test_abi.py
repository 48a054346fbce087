"""Host-side checks of the C ABI: the library builds, loads and exports every symbol that
include/fa.h declares, and rejects malformed arguments before touching a device."""
import ctypes
import os
import re

import pytest
import torch

import softmax_attention_gb300 as fa
from softmax_attention_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert len(declared) >= 12
    assert sorted(fa.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.fa_version() == 400  # 0.4.0: the decode path field and fa_decode_get_plan


def _args(**kw):
    a = fa.PrefillArgs()
    a.B, a.Hq, a.Hkv, a.Lq, a.Lkv, a.D = 1, 4, 2, 8, 8, 128
    a.scale = 0.1
    a.dtype = fa.FA_BF16
    a.q = a.k = a.v = a.out = 4096
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Lq=-1), fa.FA_ERR_INVALID_ARG),
    (dict(Hq=256, Hkv=1), fa.FA_ERR_UNSUPPORTED),
    (dict(q=4097), fa.FA_ERR_INVALID_ARG),
    (dict(out=None), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
    (dict(mask=8192, mask_batches=3, B=2), fa.FA_ERR_INVALID_ARG),
    (dict(num_splits=-2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_arguments(lib, kw, code):
    a = _args(**kw)
    rc = lib.fa_prefill_ex(ctypes.byref(a), None)
    assert rc == code, (rc, lib.fa_last_error())
    assert lib.fa_last_error()


def test_prefill_short_form_rejects_bad_head_dim(lib):
    rc = lib.fa_prefill(4096, 4096, 4096, 4096, None, 1, 2, 2, 4, 4, 80, 0, 0.1, None)
    assert rc == fa.FA_ERR_UNSUPPORTED
    assert b"D must be" in lib.fa_last_error()


def test_empty_work_is_ok_without_device(lib):
    a = _args(B=0)
    assert lib.fa_prefill_ex(ctypes.byref(a), None) == fa.FA_OK
    a = _args(Lq=0)
    assert lib.fa_prefill_ex(ctypes.byref(a), None) == fa.FA_OK
    assert lib.fa_prefill_workspace_size(ctypes.byref(a)) == 0


def test_workspace_sizes_are_consistent(lib):
    # fp32 inputs run unsplit in fp32 (no workspace, even when a split is asked for); forced
    # splits of 16-bit inputs need partial states
    a = _args(dtype=fa.FA_FP32, num_splits=4, Lkv=4096)
    assert lib.fa_prefill_workspace_size(ctypes.byref(a)) == 0
    assert lib.fa_prefill_num_splits(ctypes.byref(a)) == 1
    a = _args(num_splits=4, Lkv=4096)
    assert lib.fa_prefill_num_splits(ctypes.byref(a)) == 4
    assert lib.fa_prefill_workspace_size(ctypes.byref(a)) >= 1 * 4 * 8 * 4 * (128 + 1) * 4
    assert lib.fa_decode_workspace_size(128, 32, 128, 4096) >= 128 * 32 * (128 + 1) * 4
    assert lib.fa_decode_workspace_size(0, 32, 128, 4096) == 0
    # MLA: one chunk per sequence writes the output directly (no workspace); sequences split
    # into chunks need partial states for their rows only
    assert lib.mla_decode_workspace_size(128, 64, 512, 2048) == 0
    assert lib.mla_decode_workspace_size(64, 64, 512, 2048) >= 64 * 64 * 2 * (512 + 1) * 4
    tail = lib.mla_decode_workspace_size(768, 64, 512, 1024)  # a short last wave is split
    assert 0 < tail < 768 * 64 * (512 + 1) * 4


def test_prefill_split_plan(lib):
    """The automatic KV split: none while the (query tile, kv head, batch) units cover half the
    SMs; otherwise as many parts as still fit one wave, each of at least four KV tiles, never
    more parts than KV tiles; and a forced count is taken as given (capped by the KV tiles)."""
    sms = (torch.cuda.get_device_properties(0).multi_processor_count
           if torch.cuda.is_available() else 148)
    for B, Hq, Hkv, Lq, Lkv, D in ((1, 8, 1, 16, 16384, 256), (1, 8, 1, 64, 16384, 256),
                                   (1, 8, 1, 256, 16384, 256), (1, 8, 1, 1024, 16384, 256),
                                   (1, 32, 8, 512, 16384, 128), (2, 4, 4, 1, 300, 64),
                                   (1, 4, 1, 8, 100, 128), (4, 16, 2, 100, 8192, 128)):
        a = _args(B=B, Hq=Hq, Hkv=Hkv, Lq=Lq, Lkv=Lkv, D=D)
        n = lib.fa_prefill_num_splits(ctypes.byref(a))
        G = Hq // Hkv
        q_per_tile = 128 // G
        units = -(-Lq // q_per_tile) * Hkv * B
        bn = 64 if D == 256 else 128
        kv_tiles = -(-Lkv // bn)
        assert 1 <= n <= max(1, kv_tiles), (B, Hq, Hkv, Lq, Lkv, D, n)
        if units * 2 > sms:
            assert n == 1, (Lq, n)
        else:
            assert n * units <= sms, (Lq, n)
            assert n == 1 or kv_tiles // n >= 4, (Lq, n)
            # as many parts as fit, unless the four-tile floor or the KV tiles cap it
            assert n == min(sms // units, max(1, kv_tiles // 4)), (Lq, n)
        ws = lib.fa_prefill_workspace_size(ctypes.byref(a))
        assert (ws > 0) == (n > 1)
        if n > 1:
            assert ws >= B * Hq * Lq * n * (D + 1) * 4
    a = _args(Lkv=300, num_splits=7)  # 3 KV tiles of 128 keys: seven parts become three
    assert lib.fa_prefill_num_splits(ctypes.byref(a)) == 3


@pytest.mark.parametrize("args,code", [
    (dict(D=80), fa.FA_ERR_UNSUPPORTED),
    (dict(Hq=32, Hkv=1, page_size=4, max_pages=1024), fa.FA_ERR_UNSUPPORTED),  # G=32
    (dict(Hq=12, Hkv=4, page_size=256), fa.FA_ERR_UNSUPPORTED),  # G=3: tensor cores only
    (dict(Hq=256, Hkv=1), fa.FA_ERR_UNSUPPORTED),   # G > 128
    (dict(page_size=12), fa.FA_ERR_INVALID_ARG),
    (dict(max_seq_len=5000), fa.FA_ERR_INVALID_ARG),  # > max_pages * page_size
    (dict(ws_bytes=16), fa.FA_ERR_WORKSPACE),
])
def test_decode_rejects_bad_arguments(lib, args, code):
    p = dict(B=2, Hq=8, Hkv=2, D=128, page_size=16, max_pages=256, num_pages=600,
             max_seq_len=4096, ws_bytes=1 << 30)
    p.update(args)
    rc = lib.fa_decode_paged(4096, 4096, 4096, 4096, 4096, 4096, None, p["B"], p["Hq"], p["Hkv"],
                             p["D"], p["page_size"], p["max_pages"], p["num_pages"],
                             p["max_seq_len"], 0.1, 4096 if p["ws_bytes"] > 16 else 4096,
                             p["ws_bytes"], None)
    assert rc == code, (rc, lib.fa_last_error())


def test_mla_rejects_unsupported_shapes(lib):
    for H, Dc, Dr in ((2048, 512, 64), (64, 256, 64), (64, 512, 32)):
        rc = lib.mla_decode_paged(*([4096] * 7), None, 2, H, Dc, Dr, 1, 16, 32, 16, 0.1, 4096,
                                  1 << 30, None)
        assert rc == fa.FA_ERR_UNSUPPORTED, (H, Dc, Dr)


def test_merge_rejects_bad_arguments(lib):
    assert lib.fa_merge_states(4096, 4096, None, 4096, None, 4, 6, 2, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_merge_states(4096, 4096, None, 4096, None, 4, 8, 2, 9, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_merge_states(None, None, None, 4096, None, 0, 8, 2, 0, None) == fa.FA_OK
    assert lib.fa_merge_states(4096, 4096, None, 4096, None, 4, 516, 2, 0, None) == fa.FA_ERR_UNSUPPORTED


def test_size_queries_ignore_pointers(lib):
    a = _args(num_splits=3, Lkv=4096, q=None, k=None, v=None, out=None)
    assert lib.fa_prefill_workspace_size(ctypes.byref(a)) > 0
    assert lib.fa_prefill_num_splits(ctypes.byref(a)) == 3


def test_selftest_rejects_bad_timeouts(lib):
    # validated on the host, before any device is touched
    for t in (0, 2_000_001, 10**9):
        assert lib.fa_selftest_wait_timeout(t, None) == fa.FA_ERR_INVALID_ARG
        assert "timeout_us" in fa.fa_last_error()


def test_binding_checks_element_types(lib):
    # the C entry points take raw pointers, so the binding checks dtypes before anything else
    q = torch.zeros(1, 2, 8, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="bfloat16"):
        fa.fa_prefill(q, q, q)
    qb = q.to(torch.bfloat16)
    with pytest.raises(ValueError, match="bfloat16"):
        fa.fa_prefill_ex(qb, q, qb)
    with pytest.raises(ValueError, match="int32"):
        fa.fa_decode_paged(qb[0], qb, qb, torch.zeros(1, 1, dtype=torch.int64),
                           torch.zeros(1, dtype=torch.int32), 8)
    with pytest.raises(ValueError, match="float32"):
        fa.fa_merge_states(torch.zeros(1, 1, 4, dtype=torch.bfloat16), torch.zeros(1, 1), None)


def test_prefill_paged_rejects_bad_arguments(lib):
    def call(ps=16, max_pages=4, num_pages=4, max_len=64, D=128, Hq=4, Hkv=2):
        return lib.fa_prefill_paged(None, None, None, None, None, None, None, 1, Hq, Hkv, 8, D,
                                    ps, max_pages, num_pages, max_len, 1, 0.1, None, 0, None)
    assert call(ps=4) == fa.FA_ERR_UNSUPPORTED          # below 8 rows per page
    assert call(ps=24) == fa.FA_ERR_UNSUPPORTED         # not a power of two
    assert call(ps=256) == fa.FA_ERR_UNSUPPORTED        # wider than a key tile
    assert call(ps=128, D=256) == fa.FA_ERR_UNSUPPORTED  # D = 256 tiles are 64 keys
    assert call(max_len=65) == fa.FA_ERR_INVALID_ARG    # more than max_pages * page_size
    assert call(Hq=3) == fa.FA_ERR_INVALID_ARG
    assert call() == fa.FA_ERR_INVALID_ARG              # null pointers
    assert "null" in fa.fa_last_error()


def test_prefill_ex_paged_mode_validation(lib):
    # page_size > 0 switches fa_prefill_ex to paged K/V
    a = _args(page_size=16, max_pages=4, num_pages=4, Lkv=64)
    a.dtype = fa.FA_FP32
    assert lib.fa_prefill_ex(ctypes.byref(a), None) == fa.FA_ERR_UNSUPPORTED
    a = _args(page_size=16, max_pages=4, num_pages=4, Lkv=64)
    assert lib.fa_prefill_ex(ctypes.byref(a), None) == fa.FA_ERR_INVALID_ARG  # no page table
    a = _args(page_size=16, max_pages=4, num_pages=4, Lkv=65)
    assert lib.fa_prefill_workspace_size(ctypes.byref(a)) == 0  # invalid: Lkv > 64 slots
    a = _args(page_size=-1)
    assert lib.fa_prefill_ex(ctypes.byref(a), None) == fa.FA_ERR_INVALID_ARG


def test_prefill_paged_workspace_follows_the_dense_plan(lib):
    # one 128-row tile per kv head and long keys: the planner splits, so a workspace exists
    assert lib.fa_prefill_paged_workspace_size(1, 8, 1, 16, 128, 16384) > 0
    assert lib.fa_prefill_paged_workspace_size(0, 8, 1, 16, 128, 16384) == 0
    assert lib.fa_prefill_paged_workspace_size(1, 8, 1, 16, 128, 0) == 0


def _decode_args(**kw):
    a = fa.DecodeArgs()
    a.B, a.Hq, a.Hkv, a.D, a.page_size = 128, 32, 8, 128, 16
    a.max_pages_per_seq, a.num_pages, a.max_seq_len = 256, 40000, 4096
    a.scale, a.dtype = 0.1, fa.FA_BF16
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _plan(lib, **kw):
    pl = fa.DecodePlan()
    rc = lib.fa_decode_get_plan(ctypes.byref(_decode_args(**kw)), ctypes.byref(pl))
    return rc, pl


def test_decode_plan_chooses_a_kernel(lib):
    # 128 sequences x 8 kv heads fill the GPU: tensor cores, unsplit, no workspace
    rc, pl = _plan(lib)
    assert rc == fa.FA_OK
    assert (pl.path, pl.n_splits, pl.launches, pl.workspace_bytes) == \
        (fa.FA_DECODE_TENSOR_CORES, 1, 1, 0)
    # few sequences: the chunked CUDA-core kernel and the merge, chunk states in the workspace
    rc, pl = _plan(lib, B=2)
    assert rc == fa.FA_OK and pl.path == fa.FA_DECODE_CUDA_CORES and pl.launches == 2
    assert pl.workspace_bytes >= 2 * 32 * pl.n_splits * (128 + 1) * 4
    # a group the CUDA-core kernel cannot take goes to the tensor cores even when small
    rc, pl = _plan(lib, B=2, Hq=12, Hkv=4)
    assert rc == fa.FA_OK and pl.path == fa.FA_DECODE_TENSOR_CORES
    # page sizes the tensor-core kernel cannot take go to the CUDA cores
    rc, pl = _plan(lib, page_size=1, max_pages_per_seq=4096)
    assert rc == fa.FA_OK and pl.path == fa.FA_DECODE_CUDA_CORES
    # forced paths, and their refusals
    rc, pl = _plan(lib, path=fa.FA_DECODE_CUDA_CORES)
    assert rc == fa.FA_OK and pl.path == fa.FA_DECODE_CUDA_CORES
    assert _plan(lib, path=fa.FA_DECODE_TENSOR_CORES, page_size=4, max_pages_per_seq=1024)[0] \
        == fa.FA_ERR_UNSUPPORTED
    assert _plan(lib, path=fa.FA_DECODE_CUDA_CORES, Hq=24, Hkv=8)[0] == fa.FA_ERR_UNSUPPORTED
    assert _plan(lib, path=7)[0] == fa.FA_ERR_INVALID_ARG


def test_decode_workspace_size_bounds_every_plan(lib):
    for B, Hq, Hkv, D, ps, L in ((2, 32, 8, 128, 16, 4096), (1, 12, 4, 128, 16, 9000),
                                 (3, 8, 1, 256, 64, 20000), (128, 32, 8, 128, 16, 4096),
                                 (5, 64, 4, 64, 8, 3000), (2, 8, 2, 128, 1, 1000)):
        bound = lib.fa_decode_workspace_size(B, Hq, D, L)
        for path in (fa.FA_DECODE_AUTO, fa.FA_DECODE_CUDA_CORES, fa.FA_DECODE_TENSOR_CORES):
            rc, pl = _plan(lib, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=ps,
                           max_pages_per_seq=-(-L // ps), num_pages=4096, max_seq_len=L,
                           path=path)
            if rc == fa.FA_OK:
                assert pl.workspace_bytes <= bound, (B, Hq, Hkv, D, ps, L, path)
