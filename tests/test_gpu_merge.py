"""GPU parity of the split-state merge against the oracle's merge."""
import math

import pytest
import torch

import oracle
import softmax_attention_gb300 as fa
from tests._parity import check
from tests._guard import Guarded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,S,D", [(37, 5, 128), (8, 40, 512), (3, 1, 64)])
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
