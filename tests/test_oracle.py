"""Pins for the fp64 oracle, against things other than itself.

* hand-derived closed forms (tests/golden/closed_forms.json);
* library routines: torch's CPU scaled_dot_product_attention in fp64 (with its own
  lower-right causal bias and grouped-query broadcast) and torch.logsumexp;
* invariants of the method: constant scores give the mean of V, a dominant key returns
  its V row, key order does not matter without a mask, MLA equals expanded multi-head
  attention (two ways), decode equals prefill on the gathered cache, split-KV merging
  equals the unsplit result, exact widening of bf16/fp16 storage.
"""
import json
import math
import os

import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def _t(x):
    def conv(v):
        if isinstance(v, list):
            return [conv(e) for e in v]
        if isinstance(v, str):
            return float(v)
        return v
    return torch.tensor(conv(x), dtype=torch.float64)


def _golden():
    with open(os.path.join(HERE, "golden", "closed_forms.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_closed_forms(case):
    kind = case["kind"]
    if kind == "attention":
        mask = _t(case["mask"]) if "mask" in case else None
        out, lse = oracle.attention(_t(case["q"]), _t(case["k"]), _t(case["v"]),
                                    causal=case["causal"], scale=case["scale"], mask=mask)
    elif kind == "decode_paged":
        out, lse = oracle.decode_paged(_t(case["q"]), _t(case["k_pages"]), _t(case["v_pages"]),
                                       torch.tensor(case["page_table"], dtype=torch.int32),
                                       torch.tensor(case["seq_lens"], dtype=torch.int32),
                                       scale=case["scale"])
    elif kind == "mla_decode_paged":
        out, lse = oracle.mla_decode_paged(
            _t(case["q_nope"]), _t(case["q_pe"]), _t(case["ckv"]), _t(case["kpe"]),
            torch.tensor(case["page_table"], dtype=torch.int32),
            torch.tensor(case["seq_lens"], dtype=torch.int32), scale=case["scale"])
    elif kind == "merge":
        out, lse = oracle.merge(_t(case["o_parts"]), _t(case["lse_parts"]))
    else:
        raise AssertionError(kind)
    exp_out, exp_lse = _t(case["out"]), _t(case["lse"])
    assert out.shape == exp_out.shape
    torch.testing.assert_close(out, exp_out, rtol=0, atol=1e-12)
    fin = torch.isfinite(exp_lse)
    assert torch.equal(fin, torch.isfinite(lse))
    torch.testing.assert_close(lse[fin], exp_lse[fin], rtol=0, atol=1e-12)
    assert torch.all(lse[~fin] == -math.inf)


# --------------------------------------------------------------------------------------
# Library routine: torch SDPA in fp64
# --------------------------------------------------------------------------------------
SDPA_CASES = [
    # B, Hq, Hkv, Lq, Lkv, Dk, Dv, causal, use_mask
    (1, 2, 2, 5, 5, 8, 8, False, False),
    (2, 2, 2, 7, 7, 16, 16, True, False),
    (1, 8, 2, 3, 11, 16, 16, True, False),   # GQA, chunk at the end of a longer context
    (2, 6, 1, 4, 9, 8, 12, False, True),     # MQA, Dk != Dv, additive mask
    (1, 4, 4, 6, 6, 32, 32, True, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,Dk,Dv,causal,use_mask", SDPA_CASES)
def test_matches_torch_sdpa(B, Hq, Hkv, Lq, Lkv, Dk, Dv, causal, use_mask):
    g = torch.Generator().manual_seed(B * 1000 + Hq * 100 + Lq * 10 + Lkv)
    q = torch.randn(B, Hq, Lq, Dk, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Lkv, Dk, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Lkv, Dv, generator=g, dtype=torch.float64)
    scale = 0.37
    mask = None
    if use_mask:
        mask = workloads.additive_mask(1, Lq, Lkv, seed=5, p_masked=0.2, dtype=torch.float64)
        # keep at least one visible key per row so SDPA's output is defined
        mask[..., 0] = 0.25
    out, lse = oracle.attention(q, k, v, causal=causal, scale=scale, mask=mask)
    if causal:
        bias = causal_lower_right(Lq, Lkv)
        if mask is not None:
            keep = bias._materialize(torch.device("cpu"))
            attn_mask = mask[0].masked_fill(~keep, float("-inf"))
        else:
            attn_mask = bias
    else:
        attn_mask = None if mask is None else mask[0]
    ref = F.scaled_dot_product_attention(q, k, v, attn_mask=attn_mask, scale=scale,
                                         enable_gqa=(Hq != Hkv))
    torch.testing.assert_close(out, ref, rtol=0, atol=1e-12)


def test_lse_matches_logsumexp():
    g = torch.Generator().manual_seed(7)
    q = torch.randn(1, 4, 6, 16, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, 10, 16, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, 10, 16, generator=g, dtype=torch.float64)
    _, lse = oracle.attention(q, k, v, causal=True, scale=0.5)
    kk = k.repeat_interleave(2, dim=1)
    s = torch.matmul(q, kk.transpose(-1, -2)) * 0.5
    s = s.masked_fill(~causal_lower_right(6, 10)._materialize(torch.device("cpu")),
                      float("-inf"))
    torch.testing.assert_close(lse, torch.logsumexp(s, dim=-1), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------------------
def test_constant_scores_give_mean_of_v():
    g = torch.Generator().manual_seed(3)
    q = torch.zeros(1, 2, 4, 8, dtype=torch.float64)
    k = torch.randn(1, 2, 9, 8, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, 9, 5, generator=g, dtype=torch.float64)
    out, lse = oracle.attention(q, k, v, scale=1.0)
    torch.testing.assert_close(out, v.mean(dim=2, keepdim=True).expand_as(out), rtol=0, atol=1e-12)
    torch.testing.assert_close(lse, torch.full_like(lse, math.log(9)), rtol=0, atol=1e-12)


def test_scale_zero_gives_mean_and_log_n():
    g = torch.Generator().manual_seed(4)
    q = torch.randn(1, 1, 3, 8, generator=g, dtype=torch.float64)
    k = torch.randn(1, 1, 5, 8, generator=g, dtype=torch.float64)
    v = torch.randn(1, 1, 5, 8, generator=g, dtype=torch.float64)
    out, lse = oracle.attention(q, k, v, scale=0.0, causal=True)
    # bottom-right causal: row i sees 5-3+i+1 keys
    for i in range(3):
        n = 5 - 3 + i + 1
        torch.testing.assert_close(out[0, 0, i], v[0, 0, :n].mean(0), rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i].item() - math.log(n)) < 1e-12


def test_one_hot_dominant_key():
    g = torch.Generator().manual_seed(5)
    D = 16
    q = torch.randn(1, 1, 1, D, generator=g, dtype=torch.float64)
    k = torch.randn(1, 1, 12, D, generator=g, dtype=torch.float64) * 0.01
    k[0, 0, 7] = q[0, 0, 0] * 40.0
    v = torch.randn(1, 1, 12, D, generator=g, dtype=torch.float64)
    out, lse = oracle.attention(q, k, v, scale=1.0)
    s = (k[0, 0] @ q[0, 0, 0])
    gap = (s[7] - torch.cat([s[:7], s[8:]]).max()).item()
    assert gap > 30
    err = (out[0, 0, 0] - v[0, 0, 7]).abs().max().item()
    assert err <= 12 * math.exp(-gap) * v.abs().max().item() + 1e-15
    assert abs(lse.item() - s[7].item()) < 1e-10


def test_key_permutation_invariance():
    g = torch.Generator().manual_seed(6)
    q = torch.randn(2, 4, 5, 8, generator=g, dtype=torch.float64)
    k = torch.randn(2, 2, 13, 8, generator=g, dtype=torch.float64)
    v = torch.randn(2, 2, 13, 8, generator=g, dtype=torch.float64)
    perm = torch.randperm(13, generator=g)
    o1, l1 = oracle.attention(q, k, v, scale=0.3)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], scale=0.3)
    torch.testing.assert_close(o1, o2, rtol=0, atol=1e-12)
    torch.testing.assert_close(l1, l2, rtol=0, atol=1e-12)


def test_causal_first_row_is_v0():
    g = torch.Generator().manual_seed(8)
    q = torch.randn(1, 2, 6, 8, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, 6, 8, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, 6, 8, generator=g, dtype=torch.float64)
    out, lse = oracle.attention(q, k, v, causal=True, scale=0.7)
    torch.testing.assert_close(out[:, :, 0], v[:, :, 0], rtol=0, atol=1e-15)
    s00 = 0.7 * (q[:, :, 0] * k[:, :, 0]).sum(-1)
    torch.testing.assert_close(lse[:, :, 0], s00, rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_heads():
    g = torch.Generator().manual_seed(9)
    q = torch.randn(2, 8, 4, 8, generator=g, dtype=torch.float64)
    k = torch.randn(2, 2, 7, 8, generator=g, dtype=torch.float64)
    v = torch.randn(2, 2, 7, 8, generator=g, dtype=torch.float64)
    o1, l1 = oracle.attention(q, k, v, causal=True, scale=0.4)
    o2, l2 = oracle.attention(q, k.repeat_interleave(4, 1), v.repeat_interleave(4, 1),
                              causal=True, scale=0.4)
    torch.testing.assert_close(o1, o2, rtol=0, atol=0)
    torch.testing.assert_close(l1, l2, rtol=0, atol=0)


def test_row_subset_matches_full():
    g = torch.Generator().manual_seed(10)
    q = torch.randn(2, 4, 5, 8, generator=g, dtype=torch.float64)
    k = torch.randn(2, 2, 9, 8, generator=g, dtype=torch.float64)
    v = torch.randn(2, 2, 9, 8, generator=g, dtype=torch.float64)
    o, l = oracle.attention(q, k, v, causal=True, scale=0.4)
    rows = [0, 7, 39, 13]
    os_, ls = oracle.attention(q, k, v, causal=True, scale=0.4, rows=rows)
    torch.testing.assert_close(os_, o.reshape(-1, 8)[rows], rtol=0, atol=0)
    torch.testing.assert_close(ls, l.reshape(-1)[rows], rtol=0, atol=0)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, rows=[40])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_storage_widening_is_exact(dtype):
    g = torch.Generator().manual_seed(11)
    q = (torch.randn(1, 2, 3, 16, generator=g) * 3).to(dtype)
    k = (torch.randn(1, 2, 5, 16, generator=g) * 3).to(dtype)
    v = (torch.randn(1, 2, 5, 16, generator=g) * 3).to(dtype)
    if dtype == torch.float16:  # include subnormals and large values
        v[0, 0, 0, :4] = torch.tensor([6e-8, -3e-6, 6.0e4, -1.0e-5], dtype=torch.float16)
    o1, l1 = oracle.attention(q, k, v, causal=True, scale=0.25)
    o2, l2 = oracle.attention(q.double(), k.double(), v.double(), causal=True, scale=0.25)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _dense_from_pages(k_pages, page_table, seq_len, b):
    """Dense [Hkv, L, D] keys of sequence b, gathered with torch indexing."""
    ps = k_pages.shape[2]
    t = torch.arange(seq_len)
    pages = page_table[b, t // ps].long()
    return k_pages[pages, :, t % ps].permute(1, 0, 2)


def test_decode_equals_prefill_on_gathered_cache():
    c = workloads.PagedCase(B=3, Hq=8, Hkv=2, D=16, page_size=4, num_pages=20,
                            min_len=1, max_len=17, dtype=torch.float64, seed=12,
                            seq_lens=[17, 1, 9])
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    out, lse = oracle.decode_paged(q, kp, vp, table, lens, scale=0.3)
    for b in range(c.B):
        n = int(lens[b])
        kd = _dense_from_pages(kp, table, n, b).unsqueeze(0)
        vd = _dense_from_pages(vp, table, n, b).unsqueeze(0)
        o2, l2 = oracle.attention(q[b:b + 1].unsqueeze(2), kd, vd, scale=0.3)
        torch.testing.assert_close(out[b], o2[0, :, 0], rtol=0, atol=1e-12)
        torch.testing.assert_close(lse[b], l2[0, :, 0], rtol=0, atol=1e-12)


def test_decode_empty_sequence_and_bad_page():
    c = workloads.PagedCase(B=2, Hq=2, Hkv=1, D=8, page_size=2, num_pages=4, min_len=0,
                            max_len=4, dtype=torch.float64, seq_lens=[0, 3], seed=13)
    q, kp, vp, table, lens = workloads.paged_inputs(c)
    out, lse = oracle.decode_paged(q, kp, vp, table, lens)
    assert torch.all(out[0] == 0) and torch.all(lse[0] == -math.inf)
    assert torch.isfinite(lse[1]).all()
    bad = table.clone()
    bad[1, 0] = 4
    with pytest.raises(ValueError):
        oracle.decode_paged(q, kp, vp, bad, lens)


def _mla_case():
    c = workloads.MlaCase(B=3, H=4, seq_len=None, Dc=32, Dr=8, page_size=1,
                          dtype=torch.float64, seq_lens=[7, 1, 12], seed=14, scale=0.2)
    return c, workloads.mla_inputs(c)


def test_mla_equals_expanded_mha_concat_form():
    c, (qn, qp, ckv, kpe, table, lens) = _mla_case()
    out, lse = oracle.mla_decode_paged(qn, qp, ckv, kpe, table, lens, scale=c.scale)
    for b in range(c.B):
        n = int(lens[b])
        idx = table[b, :n].long()
        kc = ckv[idx, 0]          # [n, Dc]
        kr = kpe[idx, 0]          # [n, Dr]
        K = torch.cat([kc, kr], -1)[None, None]            # one kv head, 576-style concat
        Q = torch.cat([qn[b], qp[b]], -1)[None, :, None]   # [1,H,1,Dc+Dr]
        ref = F.scaled_dot_product_attention(Q, K.expand(1, c.H, n, -1),
                                             kc[None, None].expand(1, c.H, n, -1),
                                             scale=c.scale)
        torch.testing.assert_close(out[b], ref[0, :, 0], rtol=0, atol=1e-12)
        s = torch.einsum("hd,nd->hn", torch.cat([qn[b], qp[b]], -1), K[0, 0]) * c.scale
        torch.testing.assert_close(lse[b], torch.logsumexp(s, -1), rtol=0, atol=1e-12)


def test_mla_equals_unabsorbed_multihead_form():
    """With per-head up-projections W_UK_h [Dc,dn] and W_UV_h [Dc,dv], multi-head attention
    over k_h = ckv W_UK_h (plus the shared rope part) and v_h = ckv W_UV_h, queried with
    q_h, equals the latent form queried with q_nope_h = W_UK_h q_h, after projecting the
    latent output by W_UV_h."""
    c, (_, qp, ckv, kpe, table, lens) = _mla_case()
    g = torch.Generator().manual_seed(15)
    dn, dv = 6, 5
    W_UK = torch.randn(c.H, c.Dc, dn, generator=g, dtype=torch.float64) * 0.3
    W_UV = torch.randn(c.H, c.Dc, dv, generator=g, dtype=torch.float64) * 0.3
    q_h = torch.randn(c.B, c.H, dn, generator=g, dtype=torch.float64)
    q_nope = torch.einsum("hcd,bhd->bhc", W_UK, q_h)
    lat, _ = oracle.mla_decode_paged(q_nope, qp, ckv, kpe, table, lens, scale=c.scale)
    for b in range(c.B):
        n = int(lens[b])
        idx = table[b, :n].long()
        kc, kr = ckv[idx, 0], kpe[idx, 0]
        for h in range(c.H):
            k_h = torch.cat([kc @ W_UK[h], kr], -1)        # [n, dn+Dr]
            v_h = kc @ W_UV[h]                              # [n, dv]
            qq = torch.cat([q_h[b, h], qp[b, h]])
            ref = F.scaled_dot_product_attention(qq[None, None, None], k_h[None, None],
                                                 v_h[None, None], scale=c.scale)[0, 0, 0]
            got = lat[b, h] @ W_UV[h]
            torch.testing.assert_close(got, ref, rtol=0, atol=1e-10)


def test_merge_of_partition_equals_whole():
    g = torch.Generator().manual_seed(16)
    q = torch.randn(1, 4, 3, 8, generator=g, dtype=torch.float64)
    k = torch.randn(1, 4, 20, 8, generator=g, dtype=torch.float64)
    v = torch.randn(1, 4, 20, 8, generator=g, dtype=torch.float64)
    whole_o, whole_l = oracle.attention(q, k, v, scale=0.5)
    cuts = [0, 3, 4, 11, 20]
    parts_o, parts_l = [], []
    for a, e in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.attention(q, k[:, :, a:e], v[:, :, a:e], scale=0.5)
        parts_o.append(o.reshape(-1, 8))
        parts_l.append(l.reshape(-1))
    # an empty part (no keys) carries lse = -inf and must not change the result
    parts_o.append(torch.full_like(parts_o[0], 7.0))
    parts_l.append(torch.full_like(parts_l[0], -math.inf))
    o, l = oracle.merge(torch.stack(parts_o, 1), torch.stack(parts_l, 1))
    torch.testing.assert_close(o, whole_o.reshape(-1, 8), rtol=0, atol=1e-12)
    torch.testing.assert_close(l, whole_l.reshape(-1), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------------------
# Paged prefill: each sequence's chunk attends to its gathered cache
# ---------------------------------------------------------------------------------------
def _paged_prefill_case(**kw):
    args = dict(B=4, Hq=6, Hkv=2, Lq=5, D=16, page_size=4, num_pages=40, min_len=0, max_len=23,
                dtype=torch.float64, seed=21, seq_lens=[23, 5, 3, 0])
    args.update(kw)
    c = workloads.PagedPrefillCase(**args)
    return c, workloads.paged_prefill_inputs(c)


def test_prefill_paged_equals_dense_attention_on_the_gathered_cache():
    c, (q, kp, vp, table, lens) = _paged_prefill_case()
    for causal in (True, False):
        out, lse = oracle.prefill_paged(q, kp, vp, table, lens, causal=causal, scale=0.4)
        for b in range(c.B):
            n = int(lens[b])
            kd = _dense_from_pages(kp, table, n, b).unsqueeze(0)
            vd = _dense_from_pages(vp, table, n, b).unsqueeze(0)
            o2, l2 = oracle.attention(q[b:b + 1], kd, vd, causal=causal, scale=0.4)
            torch.testing.assert_close(out[b], o2[0], rtol=0, atol=1e-12)
            torch.testing.assert_close(lse[b], l2[0], rtol=0, atol=1e-12)


def test_prefill_paged_single_query_equals_paged_decode():
    # one query per sequence sits at the sequence's last position: the decode definition,
    # computed by the oracle's separate C routine that walks the page table itself
    c, (q, kp, vp, table, lens) = _paged_prefill_case(Lq=1, seq_lens=[23, 5, 3, 1])
    out, lse = oracle.prefill_paged(q, kp, vp, table, lens, causal=True, scale=0.4)
    o2, l2 = oracle.decode_paged(q[:, :, 0], kp, vp, table, lens, scale=0.4)
    torch.testing.assert_close(out[:, :, 0], o2, rtol=0, atol=1e-12)
    torch.testing.assert_close(lse[:, :, 0], l2, rtol=0, atol=1e-12)


def test_prefill_paged_is_invariant_to_page_placement():
    c, (q, kp, vp, table, lens) = _paged_prefill_case()
    out, lse = oracle.prefill_paged(q, kp, vp, table, lens, causal=True)
    perm = torch.randperm(c.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    kp2, vp2 = kp[perm], vp[perm]          # page p of the new pool is old page perm[p]
    t2 = torch.where(table >= 0, inv[table.clamp(min=0).long()].to(torch.int32), table)
    out2, lse2 = oracle.prefill_paged(q, kp2, vp2, t2, lens, causal=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_prefill_paged_rows_without_keys_are_empty():
    # sequence lengths 3 and 0 with Lq = 5: causally the first 2 (resp. all 5) queries of
    # those sequences have no key
    c, (q, kp, vp, table, lens) = _paged_prefill_case()
    out, lse = oracle.prefill_paged(q, kp, vp, table, lens, causal=True)
    assert torch.all(lse[2, :, :2] == -math.inf) and torch.all(out[2, :, :2] == 0)
    assert torch.isfinite(lse[2, :, 2:]).all()
    assert torch.all(lse[3] == -math.inf) and torch.all(out[3] == 0)


def test_prefill_paged_mask_equals_dense_with_the_mask_columns():
    c, (q, kp, vp, table, lens) = _paged_prefill_case()
    g = torch.Generator().manual_seed(9)
    mask = torch.randn(c.B, c.Lq, c.max_len, generator=g, dtype=torch.float64)
    mask[:, :, 3] = -math.inf
    out, lse = oracle.prefill_paged(q, kp, vp, table, lens, causal=False, mask=mask)
    for b in range(c.B):
        n = int(lens[b])
        kd = _dense_from_pages(kp, table, n, b).unsqueeze(0)
        vd = _dense_from_pages(vp, table, n, b).unsqueeze(0)
        o2, l2 = oracle.attention(q[b:b + 1], kd, vd, mask=mask[b:b + 1, :, :n])
        torch.testing.assert_close(out[b], o2[0], rtol=0, atol=1e-12)
        torch.testing.assert_close(lse[b], l2[0], rtol=0, atol=1e-12)
