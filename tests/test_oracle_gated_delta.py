"""Pins for the fp64 gated-delta oracle (oracle.gated_delta), against things other than itself.

The recurrence is the gated delta rule (Gated Delta Networks, 2024) that the hip-ep page
"perf(kernels): speed up linear-attention prefill ~2.6x" names but does not write out:

    S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T,  o_t = S_t (scale q_t)

Pins, each computed without the oracle's own loop:
* closed forms: with beta = 0 the state only decays (o_t = exp(sum g) S_0 q_t); along one
  repeated unit key the state's value y_t = S_t k obeys the scalar recursion
  y_t = alpha_t (1 - beta_t) y_{t-1} + beta_t v_t; with alpha = beta = 1 and q = k every
  token reads back exactly its own value (the delta rule's overwrite);
* a textbook routine: with orthonormal keys and alpha = beta = 1 the rule is causal linear
  attention, tril(Q K^T) V (a torch matmul);
* a different algorithm: the chunked (WY) form, one triangular solve per chunk (torch),
  equals the recurrence in general position;
* invariants: running T tokens equals running a prefix and then the rest from the prefix's
  final state; grouped value heads equal repeated query/key heads.
Mistakes planted in a private copy of the oracle must fail at least one of these
(tests/test_oracle_gated_delta_mutations.py).
"""
import math

import pytest
import torch

import oracle

F64 = torch.float64


def _unit(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.nn.functional.normalize(torch.randn(*shape, generator=g, dtype=F64), dim=-1)


def _rand(*shape, seed, lo=None, hi=None):
    g = torch.Generator().manual_seed(seed)
    if lo is None:
        return torch.randn(*shape, generator=g, dtype=F64)
    return lo + (hi - lo) * torch.rand(*shape, generator=g, dtype=F64)


def test_no_write_only_decays_the_initial_state():
    B, Hk, Hv, T, dk, dv = 1, 2, 4, 9, 6, 5
    q = _rand(B, Hk, T, dk, seed=1)
    k = _unit(B, Hk, T, dk, seed=2)
    v = _rand(B, Hv, T, dv, seed=3)
    g = _rand(B, Hv, T, seed=4, lo=-0.7, hi=-0.01)
    beta = torch.zeros(B, Hv, T, dtype=F64)
    s0 = _rand(B, Hv, dv, dk, seed=5)
    scale = 0.37
    out, st = oracle.gated_delta(q, k, v, g, beta, scale=scale, initial_state=s0)
    decay = torch.exp(torch.cumsum(g, dim=-1))                        # [B,Hv,T]
    qh = q.repeat_interleave(Hv // Hk, dim=1)                         # value head -> q head
    want = decay[..., None] * torch.einsum("bhij,bhtj->bhti", s0, scale * qh)
    assert torch.allclose(out, want, rtol=1e-12, atol=1e-13)
    assert torch.allclose(st, decay[..., -1, None, None] * s0, rtol=1e-12, atol=1e-13)


def test_repeated_key_follows_the_scalar_recursion():
    # one unit key k for every token: y_t = S_t k obeys y_t = alpha_t (1 - beta_t) y_{t-1}
    # + beta_t v_t, and with q_t = k, o_t = scale * y_t
    T, dk, dv, scale = 40, 8, 3, 0.5
    kk = _unit(dk, seed=11)
    k = kk.expand(1, 1, T, dk).contiguous()
    v = _rand(1, 1, T, dv, seed=12)
    g = _rand(1, 1, T, seed=13, lo=-0.5, hi=0.0)
    beta = _rand(1, 1, T, seed=14, lo=0.0, hi=1.0)
    s0 = _rand(1, 1, dv, dk, seed=15)
    out, st = oracle.gated_delta(k, k, v, g, beta, scale=scale, initial_state=s0)
    y = s0[0, 0] @ kk
    for t in range(T):
        a, b = math.exp(g[0, 0, t]), beta[0, 0, t]
        y = a * (1 - b) * y + b * v[0, 0, t]
        assert torch.allclose(out[0, 0, t], scale * y, rtol=1e-11, atol=1e-12), t
    assert torch.allclose(st[0, 0] @ kk, y, rtol=1e-11, atol=1e-12)


def test_full_write_reads_back_each_tokens_own_value():
    # alpha = beta = 1 and unit keys: S_t k_t = v_t exactly, whatever came before
    B, Hk, Hv, T, dk, dv = 2, 1, 1, 30, 16, 7
    k = _unit(B, Hk, T, dk, seed=21)
    v = _rand(B, Hv, T, dv, seed=22)
    g = torch.zeros(B, Hv, T, dtype=F64)
    beta = torch.ones(B, Hv, T, dtype=F64)
    s0 = _rand(B, Hv, dv, dk, seed=23)
    out, _ = oracle.gated_delta(k, k, v, g, beta, scale=1.0, initial_state=s0)
    assert torch.allclose(out, v, rtol=1e-10, atol=1e-11)


def test_orthonormal_keys_give_causal_linear_attention():
    T, dk, dv = 12, 16, 6
    g0 = torch.Generator().manual_seed(31)
    basis, _ = torch.linalg.qr(torch.randn(dk, dk, generator=g0, dtype=F64))
    k = basis[:T].reshape(1, 1, T, dk).contiguous()                   # orthonormal rows
    q = _rand(1, 1, T, dk, seed=32)
    v = _rand(1, 1, T, dv, seed=33)
    g = torch.zeros(1, 1, T, dtype=F64)
    beta = torch.ones(1, 1, T, dtype=F64)
    scale = 0.25
    out, st = oracle.gated_delta(q, k, v, g, beta, scale=scale)
    want = torch.tril(scale * q[0, 0] @ k[0, 0].T) @ v[0, 0]
    assert torch.allclose(out[0, 0], want, rtol=1e-12, atol=1e-13)
    assert torch.allclose(st[0, 0], v[0, 0].T @ k[0, 0], rtol=1e-12, atol=1e-13)


def _chunked(q, k, v, g, beta, scale, s0, C):
    """The chunked (WY) form of the rule for one head, with a triangular solve per chunk:
    U = (I + A)^-1 (beta * (V - Gamma K S^T)) with A = strictly lower beta_i Gamma_i/Gamma_j
    k_i.k_j, O = Gamma Q S^T + (Q K^T * Gamma_i/Gamma_j, lower incl. diagonal) U and
    S <- Gamma_C S + U^T (Gamma_C/Gamma_j K)."""
    T = q.shape[0]
    S = s0.clone()
    out = torch.empty(T, v.shape[1], dtype=F64)
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        K, Q, V = k[sl], scale * q[sl], v[sl]
        gam = torch.cumsum(g[sl], 0)
        ratio = torch.exp(gam[:, None] - gam[None, :])
        A = torch.tril(beta[sl, None] * ratio * (K @ K.T), -1)
        rhs = beta[sl, None] * (V - torch.exp(gam)[:, None] * (K @ S.T))
        U = torch.linalg.solve_triangular(torch.eye(len(gam), dtype=F64) + A, rhs, upper=False,
                                          unitriangular=True)
        out[sl] = torch.exp(gam)[:, None] * (Q @ S.T) + torch.tril(ratio * (Q @ K.T)) @ U
        S = torch.exp(gam[-1]) * S + (torch.exp(gam[-1] - gam)[:, None] * U).T @ K
    return out, S


@pytest.mark.parametrize("C", [1, 4, 16])
def test_chunked_form_equals_the_recurrence(C):
    B, Hk, Hv, T, dk, dv = 1, 2, 2, 37, 8, 6
    q = _unit(B, Hk, T, dk, seed=41)
    k = _unit(B, Hk, T, dk, seed=42)
    v = _rand(B, Hv, T, dv, seed=43)
    g = _rand(B, Hv, T, seed=44, lo=-0.4, hi=-0.001)
    beta = _rand(B, Hv, T, seed=45, lo=0.0, hi=1.0)
    s0 = _rand(B, Hv, dv, dk, seed=46)
    scale = dk ** -0.5
    out, st = oracle.gated_delta(q, k, v, g, beta, scale=scale, initial_state=s0)
    for h in range(Hv):
        o_c, s_c = _chunked(q[0, h], k[0, h], v[0, h], g[0, h], beta[0, h], scale, s0[0, h], C)
        assert torch.allclose(out[0, h], o_c, rtol=1e-10, atol=1e-12)
        assert torch.allclose(st[0, h], s_c, rtol=1e-10, atol=1e-12)


def test_state_passing_splits_the_sequence():
    B, Hk, Hv, T, dk, dv, T1 = 2, 1, 2, 25, 8, 8, 11
    q, k = _rand(B, Hk, T, dk, seed=51), _unit(B, Hk, T, dk, seed=52)
    v = _rand(B, Hv, T, dv, seed=53)
    g = _rand(B, Hv, T, seed=54, lo=-0.3, hi=0.0)
    beta = _rand(B, Hv, T, seed=55, lo=0.0, hi=1.0)
    s0 = _rand(B, Hv, dv, dk, seed=56)
    out, st = oracle.gated_delta(q, k, v, g, beta, initial_state=s0)
    o1, s1 = oracle.gated_delta(q[:, :, :T1].contiguous(), k[:, :, :T1].contiguous(),
                                v[:, :, :T1].contiguous(), g[:, :, :T1].contiguous(),
                                beta[:, :, :T1].contiguous(), initial_state=s0)
    o2, s2 = oracle.gated_delta(q[:, :, T1:].contiguous(), k[:, :, T1:].contiguous(),
                                v[:, :, T1:].contiguous(), g[:, :, T1:].contiguous(),
                                beta[:, :, T1:].contiguous(), initial_state=s1)
    assert torch.allclose(torch.cat([o1, o2], dim=2), out, rtol=1e-12, atol=1e-13)
    assert torch.allclose(s2, st, rtol=1e-12, atol=1e-13)


def test_grouped_value_heads_equal_repeated_query_key_heads():
    B, Hk, Hv, T, dk, dv = 1, 2, 4, 10, 8, 4
    q, k = _rand(B, Hk, T, dk, seed=61), _unit(B, Hk, T, dk, seed=62)
    v = _rand(B, Hv, T, dv, seed=63)
    g = _rand(B, Hv, T, seed=64, lo=-0.3, hi=0.0)
    beta = _rand(B, Hv, T, seed=65, lo=0.0, hi=1.0)
    out, st = oracle.gated_delta(q, k, v, g, beta)
    rq = q.repeat_interleave(2, dim=1).contiguous()   # value head h reads q/k head h // 2
    rk = k.repeat_interleave(2, dim=1).contiguous()
    out2, st2 = oracle.gated_delta(rq, rk, v, g, beta)
    assert torch.equal(out, out2) and torch.equal(st, st2)


def test_storage_types_are_widened_exactly():
    B, Hk, Hv, T, dk, dv = 1, 1, 1, 6, 8, 8
    q, k = _rand(B, Hk, T, dk, seed=71), _unit(B, Hk, T, dk, seed=72)
    v = _rand(B, Hv, T, dv, seed=73)
    g = _rand(B, Hv, T, seed=74, lo=-0.3, hi=0.0).float()
    beta = _rand(B, Hv, T, seed=75, lo=0.0, hi=1.0).float()
    for dt in (torch.bfloat16, torch.float16):
        qs, ks, vs = q.to(dt), k.to(dt), v.to(dt)
        a, sa = oracle.gated_delta(qs, ks, vs, g, beta)
        b, sb = oracle.gated_delta(qs.double(), ks.double(), vs.double(), g.double(),
                                   beta.double())
        assert torch.equal(a, b) and torch.equal(sa, sb)
