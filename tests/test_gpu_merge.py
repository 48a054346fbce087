"""GPU parity of the split-state merge against the oracle's merge."""
import math

import pytest
import torch

import oracle
import softmax_attention_gb300 as fa
from tests._parity import check
from tests._guard import Guarded

pytestmark = pytest.mark.gpu


# (rows, parts, D): one to eight warps per row (parts <= 8, 16, 32, more), one to four 16-byte
# vectors per lane, D not a multiple of 128, row counts that leave a CTA partly empty; 128 rows
# of 64 parts at D=256 is the shape of the multi-query sweep's shortest size.
@pytest.mark.parametrize("rows,S,D", [(37, 5, 128), (8, 40, 512), (3, 1, 64), (21, 12, 256),
                                      (9, 30, 384), (5, 150, 100), (50, 16, 200), (17, 8, 4),
                                      (128, 64, 256), (7, 33, 128)])
def test_merge_parity(rows, S, D):
    g = torch.Generator().manual_seed(rows * S)
    o = torch.randn(rows, S, D, generator=g)
    lse = torch.randn(rows, S, generator=g) * 3
    lse[0, :] = -math.inf                  # a row with no key at all
    if S > 1:
        lse[1, 0] = -math.inf              # an empty part
    n = torch.full((rows,), S, dtype=torch.int32)
    if rows > 2:
        n[2] = max(1, S // 2)              # a row with fewer valid parts
    ro, rl = oracle.merge(o, lse)
    if rows > 2:
        o2, l2 = oracle.merge(o[2:3, : int(n[2])], lse[2:3, : int(n[2])])
        ro[2], rl[2] = o2[0], l2[0]
    og, lg = Guarded((rows, D), torch.float32), Guarded((rows,), torch.float32)
    out, lse_g = fa.fa_merge_states(o.cuda(), lse.cuda(), n.cuda(), out_dtype=torch.float32,
                                    out=og.view, lse=lg.view)
    torch.cuda.synchronize()
    og.assert_intact("merge out")
    lg.assert_intact("merge lse")
    check(out, lse_g, ro, rl, max_err=1e-5, mean_err=1e-6, lse_err=1e-5, what="merge")


def test_merge_bf16_output():
    rows, S, D = 33, 9, 128
    g = torch.Generator().manual_seed(5)
    o = torch.randn(rows, S, D, generator=g)
    lse = torch.randn(rows, S, generator=g) * 3
    ro, rl = oracle.merge(o, lse)
    og, lg = Guarded((rows, D), torch.bfloat16), Guarded((rows,), torch.float32)
    out, lse_g = fa.fa_merge_states(o.cuda(), lse.cuda(), None, out_dtype=torch.bfloat16,
                                    out=og.view, lse=lg.view)
    torch.cuda.synchronize()
    og.assert_intact("merge out")
    lg.assert_intact("merge lse")
    assert out.dtype == torch.bfloat16
    check(out, lse_g, ro, rl, what="merge bf16")
