"""The device failure path shared by every kernel: a bounded wait that runs out records
FA_ERR_TIMEOUT in the sticky status word and the kernel ends; the host reads the status, it
is cleared by the read, and the device keeps working (a prefill run afterwards matches the
oracle).  The wait is on a barrier that nothing arrives on, with a 20 ms limit."""
import time

import pytest
import torch

import oracle
import softmax_attention_gb300 as fa
import workloads
from tests._parity import check

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_the_device_stays_usable():
    fa.load_library()
    assert fa.fa_get_device_status() == fa.FA_OK, fa.fa_last_error()
    t0 = time.monotonic()
    assert fa.fa_selftest_wait_timeout(20_000) == fa.FA_OK, fa.fa_last_error()
    assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    assert time.monotonic() - t0 < 10.0
    assert "bounded wait" in fa.fa_last_error()
    assert fa.fa_get_device_status() == fa.FA_OK  # cleared by the read

    c = workloads.DenseCase(B=1, Hq=4, Hkv=2, Lq=70, Lkv=200, D=64, causal=True, sigma=0.5)
    q, k, v = workloads.dense_inputs(c)
    out, lse = fa.fa_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=c.sm_scale)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(q, k, v, causal=True, scale=c.sm_scale)
    check(out, lse, ref_o, ref_l, what="prefill after the timeout self-test")
    assert fa.fa_get_device_status() == fa.FA_OK
