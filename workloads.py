"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the attention
arithmetic.  Both the fp64 oracle (via the tests and the CPU baseline) and the CUDA path
(via the tests and the benchmark) take their inputs from here, so that the two sides see the
same bits.

Recipe: a ``torch.Generator('cpu')`` seeded per call draws fp32 N(0,1) values, which are
multiplied by sigma and rounded to the storage dtype (round-to-nearest-even for bf16/fp16).
Integer structure (sequence lengths, page permutations) comes from the same generator.

The shapes follow the workloads on the pages: a Llama-8B-like grouped-query prefill chunk
against a 16K-token cache and a Gemma-2B-like multi-query sweep (llama.cpp PR "CUDA: fix FA
occupancy, optimize tile kernel", performance table: gemma 2B / llama 8B, pp16384, ubatch
16..16384), paged decode over a page pool, and MLA decode with 64 heads at page_size 1
(flashinfer PR "perf: FlashAttention-3 style MLA PageAttention", results section:
batch 128 / 768, seq_len 2048 / 1024).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, sigma: float, dtype: torch.dtype, gen: torch.Generator,
           chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1)*sigma drawn in fp32, then rounded to ``dtype``.  Drawn in chunks so that
    multi-GB pools do not need a full fp32 copy."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=dtype)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        out[s:e] = x.to(dtype)
    return out.view(*shape)


# ----------------------------------------------------------------------------------------
# Dense prefill inputs
# ----------------------------------------------------------------------------------------
@dataclass
class DenseCase:
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lkv: int
    D: int
    causal: bool
    dtype: torch.dtype = torch.bfloat16
    sigma: float = 1.0
    seed: int = 1
    Dv: int | None = None
    scale: float | None = None

    @property
    def dv(self) -> int:
        return self.Dv if self.Dv is not None else self.D

    @property
    def sm_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)


def dense_inputs(c: DenseCase):
    """q [B,Hq,Lq,D], k [B,Hkv,Lkv,D], v [B,Hkv,Lkv,Dv] on the CPU."""
    g = _gen(c.seed)
    q = normal((c.B, c.Hq, c.Lq, c.D), c.sigma, c.dtype, g)
    k = normal((c.B, c.Hkv, c.Lkv, c.D), c.sigma, c.dtype, g)
    v = normal((c.B, c.Hkv, c.Lkv, c.dv), c.sigma, c.dtype, g)
    return q, k, v


def additive_mask(Bm: int, Lq: int, Lkv: int, seed: int, p_masked: float = 0.25,
                  dtype=torch.float32) -> torch.Tensor:
    """An additive mask [Bm,Lq,Lkv]: -inf with probability p_masked, else N(0,1)*0.5."""
    g = _gen(seed)
    vals = torch.randn(Bm, Lq, Lkv, generator=g) * 0.5
    drop = torch.rand(Bm, Lq, Lkv, generator=g) < p_masked
    vals[drop] = float("-inf")
    return vals.to(dtype)


# ----------------------------------------------------------------------------------------
# Paged decode inputs
# ----------------------------------------------------------------------------------------
@dataclass
class PagedCase:
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    min_len: int
    max_len: int
    dtype: torch.dtype = torch.bfloat16
    sigma: float = 0.5
    seed: int = 1
    seq_lens: list | None = None  # explicit lengths override min_len/max_len

    @property
    def max_pages(self) -> int:
        return -(-self.max_len // self.page_size)

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def paged_inputs(c: PagedCase):
    """q [B,Hq,D]; k_pages, v_pages [num_pages,Hkv,page_size,D]; page_table
    [B,max_pages] int32 (unused slots = -1); seq_lens [B] int32.

    Pages are assigned from one seeded permutation of the pool: sequence b takes the next
    ceil(len_b / page_size) entries, in order."""
    g = _gen(c.seed)
    if c.seq_lens is not None:
        lens = torch.tensor(c.seq_lens, dtype=torch.int32)
        assert lens.numel() == c.B
    else:
        lens = torch.randint(c.min_len, c.max_len + 1, (c.B,), generator=g, dtype=torch.int64)
        lens = lens.to(torch.int32)
    need = [-(-int(n) // c.page_size) for n in lens.tolist()]
    if sum(need) > c.num_pages:
        raise ValueError(f"pool of {c.num_pages} pages is smaller than the {sum(need)} needed")
    perm = torch.randperm(c.num_pages, generator=g, dtype=torch.int64).to(torch.int32)
    table = torch.full((c.B, c.max_pages), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    q = normal((c.B, c.Hq, c.D), c.sigma, c.dtype, g)
    kp = normal((c.num_pages, c.Hkv, c.page_size, c.D), c.sigma, c.dtype, g)
    vp = normal((c.num_pages, c.Hkv, c.page_size, c.D), c.sigma, c.dtype, g)
    return q, kp, vp, table, lens


# ----------------------------------------------------------------------------------------
# Paged prefill inputs (a query chunk at the end of each sequence's cached context)
# ----------------------------------------------------------------------------------------
@dataclass
class PagedPrefillCase:
    B: int
    Hq: int
    Hkv: int
    Lq: int
    D: int
    page_size: int
    num_pages: int
    min_len: int
    max_len: int
    causal: bool = True
    dtype: torch.dtype = torch.bfloat16
    sigma: float = 0.5
    seed: int = 1
    seq_lens: list | None = None  # explicit lengths (chunk included) override min/max

    @property
    def max_pages(self) -> int:
        return max(1, -(-self.max_len // self.page_size))

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def paged_prefill_inputs(c: PagedPrefillCase):
    """q [B,Hq,Lq,D]; k_pages, v_pages [num_pages,Hkv,page_size,D]; page_table
    [B,max_pages] int32 (unused slots = -1); seq_lens [B] int32 (the chunk included).
    Pages come from one seeded permutation of the pool, as in paged_inputs."""
    dc = PagedCase(B=c.B, Hq=c.Hq, Hkv=c.Hkv, D=c.D, page_size=c.page_size,
                   num_pages=c.num_pages, min_len=c.min_len, max_len=c.max_len, dtype=c.dtype,
                   sigma=c.sigma, seed=c.seed, seq_lens=c.seq_lens)
    _, kp, vp, table, lens = paged_inputs(dc)
    g = _gen(c.seed + 7919)
    q = normal((c.B, c.Hq, c.Lq, c.D), c.sigma, c.dtype, g)
    return q, kp, vp, table, lens


def paged_prefill_flops(c: PagedPrefillCase, lens) -> float:
    """Algorithmic FLOPs (4 * D per visible (query, key) pair per query head)."""
    total = 0
    for n in (int(x) for x in lens):
        for i in range(c.Lq):
            pos = n - c.Lq + i
            total += max(0, min(n, pos + 1)) if c.causal else n
    return 4.0 * c.D * c.Hq * total


# ----------------------------------------------------------------------------------------
# MLA paged decode inputs
# ----------------------------------------------------------------------------------------
@dataclass
class MlaCase:
    B: int
    H: int
    seq_len: int | None
    Dc: int = 512
    Dr: int = 64
    page_size: int = 1
    dtype: torch.dtype = torch.bfloat16
    sigma: float = 0.3
    seed: int = 1
    seq_lens: list | None = None
    scale: float = 1.0 / math.sqrt(192.0)

    def lens(self) -> list:
        return list(self.seq_lens) if self.seq_lens is not None else [self.seq_len] * self.B

    @property
    def max_len(self) -> int:
        return max(self.lens()) if self.B > 0 else 0

    @property
    def max_pages(self) -> int:
        return max(1, -(-self.max_len // self.page_size))


def mla_inputs(c: MlaCase):
    """q_nope [B,H,Dc], q_pe [B,H,Dr]; ckv [P,page_size,Dc], kpe [P,page_size,Dr];
    page_table [B,max_pages] int32 (unused = -1); seq_lens [B] int32.  The pool holds
    exactly the pages the batch needs, handed out by one seeded permutation."""
    g = _gen(c.seed)
    lens = c.lens()
    need = [-(-n // c.page_size) for n in lens]
    P = max(1, sum(need))
    perm = torch.randperm(P, generator=g, dtype=torch.int64).to(torch.int32)
    table = torch.full((c.B, c.max_pages), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[pos:pos + n]
        pos += n
    q_nope = normal((c.B, c.H, c.Dc), c.sigma, c.dtype, g)
    q_pe = normal((c.B, c.H, c.Dr), c.sigma, c.dtype, g)
    ckv = normal((P, c.page_size, c.Dc), c.sigma, c.dtype, g)
    kpe = normal((P, c.page_size, c.Dr), c.sigma, c.dtype, g)
    return q_nope, q_pe, ckv, kpe, table, torch.tensor(lens, dtype=torch.int32)


# ----------------------------------------------------------------------------------------
# The named workloads
# ----------------------------------------------------------------------------------------
def tiny_dense(causal: bool, seed: int = 1) -> DenseCase:
    """B=1, Hq=Hkv=2, Lq=Lkv=64, D=64, fp32 N(0,1), scale 1/8."""
    return DenseCase(B=1, Hq=2, Hkv=2, Lq=64, Lkv=64, D=64, causal=causal,
                     dtype=torch.float32, sigma=1.0, seed=seed)


def gqa_prefill_chunk(seed: int = 1, Lq: int = 512, Lkv: int = 16384) -> DenseCase:
    """Llama-8B-like: B=1, Hq=32, Hkv=8, D=128, 16K cache, a 512-query chunk at the end
    of the context (positions 15872..16383), causal, bf16 N(0,1)*0.5, scale 1/sqrt(128)."""
    return DenseCase(B=1, Hq=32, Hkv=8, Lq=Lq, Lkv=Lkv, D=128, causal=True,
                     dtype=torch.bfloat16, sigma=0.5, seed=seed)


def paged_gqa_decode(seed: int = 1) -> PagedCase:
    """batch 128, Hq=32, Hkv=8, D=128, bf16 N(0,1)*0.5, seq_lens ~ U{1024..4096},
    page_size 16, a 40000-page pool handed out by a seeded permutation."""
    return PagedCase(B=128, Hq=32, Hkv=8, D=128, page_size=16, num_pages=40000,
                     min_len=1024, max_len=4096, sigma=0.5, seed=seed)


def mla_decode(batch: int = 128, seq_len: int = 2048, seed: int = 1,
               page_size: int = 1) -> MlaCase:
    """64 heads, ckv 512 (K and V), kpe 64, bf16 N(0,1)*0.3, scale 1/sqrt(192), page_size 1
    unless given; batch 128 x seq 2048 or batch 768 x seq 1024 (and the grid around them)."""
    return MlaCase(B=batch, H=64, seq_len=seq_len, seed=seed, page_size=page_size)


MQA_SWEEP_LQ = (16, 64, 256, 1024, 4096, 16384)


def paged_gqa_prefill(seed: int = 1) -> PagedPrefillCase:
    """Chunked prefill against a paged cache, Llama-8B-like heads: 8 sequences, Hq=32,
    Hkv=8, D=128, a 512-query chunk at the end of each sequence's context of U{2048..8192}
    tokens (chunk included), page_size 16, causal, bf16 N(0,1)*0.5, scale 1/sqrt(128)."""
    return PagedPrefillCase(B=8, Hq=32, Hkv=8, Lq=512, D=128, page_size=16, num_pages=6000,
                            min_len=2048, max_len=8192, seed=seed)


def mqa_prefill(Lq: int, seed: int = 1) -> DenseCase:
    """Gemma-2B-like: B=1, Hq=8, Hkv=1, D=256, 16K context, causal, bf16 N(0,1)*0.5,
    Lq queries at the end of the context, scale 1/16."""
    return DenseCase(B=1, Hq=8, Hkv=1, Lq=Lq, Lkv=16384, D=256, causal=True,
                     dtype=torch.bfloat16, sigma=0.5, seed=seed)


def causal_pairs(Lq: int, Lkv: int) -> int:
    """Number of (query, key) pairs a bottom-right causal mask leaves visible."""
    off = Lkv - Lq
    total = 0
    for i in range(Lq):
        total += max(0, min(Lkv, i + off + 1))
    return total


# ----------------------------------------------------------------------------------------
# Gated-delta linear-attention prefill inputs (a second workload, not softmax attention)
# ----------------------------------------------------------------------------------------
@dataclass
class GatedDeltaCase:
    """q, k [B,Hk,T,dk] and v [B,Hv,T,dv] in `dtype`; g (log decay) and beta [B,Hv,T] fp32;
    an optional fp32 initial state [B,Hv,dv,dk]."""
    B: int
    T: int
    Hk: int
    Hv: int
    dk: int = 128
    dv: int = 128
    dtype: torch.dtype = torch.bfloat16
    sigma_v: float = 1.0
    g_min: float = -0.25
    g_max: float = -0.005
    with_state: bool = False
    seed: int = 1

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)


def gated_delta_inputs(c: GatedDeltaCase):
    """Returns (q, k, v, g, beta, initial_state or None).  Query and key rows are drawn
    N(0,1), scaled to unit L2 norm in fp32 (the model normalises them before the recurrence)
    and then rounded to `dtype`; v ~ N(0,1)*sigma_v; g ~ U(g_min, g_max) (decays
    alpha = e^g of about 0.78..0.995); beta = sigmoid(N(0,1)); the initial state, when asked
    for, ~ N(0,1)*0.1."""
    g_ = _gen(c.seed)

    def unit_rows(shape):
        x = torch.randn(*shape, generator=g_, dtype=torch.float32)
        return (x / x.norm(dim=-1, keepdim=True)).to(c.dtype)

    q = unit_rows((c.B, c.Hk, c.T, c.dk))
    k = unit_rows((c.B, c.Hk, c.T, c.dk))
    v = normal((c.B, c.Hv, c.T, c.dv), c.sigma_v, c.dtype, g_)
    g = c.g_min + (c.g_max - c.g_min) * torch.rand(c.B, c.Hv, c.T, generator=g_,
                                                   dtype=torch.float32)
    beta = torch.sigmoid(torch.randn(c.B, c.Hv, c.T, generator=g_, dtype=torch.float32))
    s0 = None
    if c.with_state:
        s0 = normal((c.B, c.Hv, c.dv, c.dk), 0.1, torch.float32, g_)
    return q, k, v, g, beta, s0


def gated_delta_prefill(seed: int = 1) -> GatedDeltaCase:
    """Chunked linear-attention prefill of the hip-ep PR's shape class: one 1842-token
    sequence, dk = dv = 128, 16 query/key heads and 32 value heads, bf16, fp32 gates."""
    return GatedDeltaCase(B=1, T=1842, Hk=16, Hv=32, seed=seed)
