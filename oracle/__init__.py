"""fp64 CPU oracle for softmax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library never calls it, and it never calls the CUDA library.

The arithmetic lives in ``fa_oracle.c`` (plain fp64 C, OpenMP over rows); this module builds
it with gcc on first use and marshals torch CPU tensors to it.  Every function returns fp64
torch tensors.  Definitions (see the C file for the readings taken where the pages are
silent):

* ``attention``: out = softmax(scale * q k^T + mask) v with bottom-right causal masking and
  grouped-query head mapping h -> h // (Hq // Hkv); lse = natural log-sum-exp of the scaled,
  masked scores.
* ``decode_paged``: the same with one query per sequence and keys gathered through a page
  table from a [num_pages, Hkv, page_size, D] cache.
* ``prefill_paged``: ``attention`` per sequence, with the sequence's keys and values gathered
  in order through its page table and its queries at its last Lq positions.
* ``mla_decode_paged``: latent-form MLA, where ckv serves as K and V and q_pe . kpe is added
  to each score ("perf: FlashAttention-3 style MLA PageAttention", change list item 4).
* ``merge``: combination of attention states over disjoint key sets.
* ``gated_delta``: the gated delta rule of gated-delta linear attention, evaluated one token
  after another (``gdn_oracle.c``; "perf(kernels): speed up linear-attention prefill ~2.6x",
  hip-ep PR, Test plan: the per-token oracle its chunked prefill kernel is checked against).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_GD_SRC = os.path.join(_HERE, "gdn_oracle.c")
_GD_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_gdn.so")
_lock = threading.Lock()
_lib = None
_gd_lib = None

_DTYPE_CODE = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2, torch.float64: 3}

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def _build_one(src: str, lib: str, force: bool) -> str:
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
        os.replace(tmp, lib)
    return lib


def build(force: bool = False) -> str:
    """Compile fa_oracle.c and gdn_oracle.c into shared libraries (gcc, -O2, OpenMP); return
    the attention oracle's path."""
    _build_one(_GD_SRC, _GD_LIB_PATH, force)
    return _build_one(_SRC, _LIB_PATH, force)


def _load_gd():
    global _gd_lib
    with _lock:
        if _gd_lib is None:
            # GDN_ORACLE_LIB lets the oracle's own mutation test point at a deliberately
            # broken build of gdn_oracle.c; nothing else sets it.
            path = os.environ.get("GDN_ORACLE_LIB") or _build_one(_GD_SRC, _GD_LIB_PATH, False)
            lib = ctypes.CDLL(path)
            lib.oracle_gated_delta.restype = ctypes.c_int
            lib.oracle_gated_delta.argtypes = [
                _p, _p, _p, ctypes.c_int, _p, _p, ctypes.c_int, _p,
                _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_double, _p, _p]
            _gd_lib = lib
    return _gd_lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # FA_ORACLE_LIB lets the oracle's own mutation test point at a deliberately
            # broken build of fa_oracle.c; nothing else sets it.
            path = os.environ.get("FA_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [
                _p, _p, _p, ctypes.c_int, _p, ctypes.c_int, _i64,
                _i64, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_double,
                _p, _i64, _p, _p]
            lib.oracle_decode_paged.restype = ctypes.c_int
            lib.oracle_decode_paged.argtypes = [
                _p, _p, _p, ctypes.c_int, _p, _p,
                _i64, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                _p, _i64, _p, _p]
            lib.oracle_mla_decode_paged.restype = ctypes.c_int
            lib.oracle_mla_decode_paged.argtypes = [
                _p, _p, _p, _p, ctypes.c_int, _p, _p,
                _i64, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                _p, _i64, _p, _p]
            lib.oracle_merge.restype = ctypes.c_int
            lib.oracle_merge.argtypes = [_p, _p, ctypes.c_int, _i64, _i64, _i64, _p, _p]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes CPU tensors")
    return t.contiguous()


def _code(t: torch.Tensor) -> int:
    try:
        return _DTYPE_CODE[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _rows(rows):
    if rows is None:
        return None, 0
    r = torch.as_tensor(rows, dtype=torch.int64).contiguous()
    return r, r.numel()


def num_threads() -> int:
    """Threads the oracle's parallel loops use (OMP_NUM_THREADS or all cores)."""
    return _load().oracle_num_threads()


def attention(q, k, v, *, causal=False, scale=None, mask=None, rows=None):
    """Dense attention.  q [B,Hq,Lq,Dk]; k [B,Hkv,Lkv,Dk]; v [B,Hkv,Lkv,Dv] (one dtype);
    mask optional additive [Bm,Lq,Lkv] with Bm in {1,B}.  Returns (out, lse) in fp64:
    out [B,Hq,Lq,Dv] and lse [B,Hq,Lq], or [n,Dv] / [n] for the flat row ids in ``rows``."""
    lib = _load()
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    B, Hq, Lq, Dk = q.shape
    _, Hkv, Lkv, Dv = v.shape
    if k.shape != (B, Hkv, Lkv, Dk) or v.shape[:3] != (B, Hkv, Lkv):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = Dk ** -0.5
    m_ptr, m_code, m_b = None, 0, 0
    if mask is not None:
        mask = _cpu(mask)
        if mask.dim() == 2:
            mask = mask.unsqueeze(0)
        if mask.shape[1:] != (Lq, Lkv) or mask.shape[0] not in (1, B):
            raise ValueError("mask must be [1 or B, Lq, Lkv]")
        m_ptr, m_code, m_b = mask.data_ptr(), _code(mask), mask.shape[0]
    r, n = _rows(rows)
    n_out = n if r is not None else B * Hq * Lq
    out = torch.empty(n_out, Dv, dtype=torch.float64)
    lse = torch.empty(n_out, dtype=torch.float64)
    rc = lib.oracle_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), _code(q),
                              m_ptr, m_code, m_b, B, Hq, Hkv, Lq, Lkv, Dk, Dv,
                              int(bool(causal)), float(scale),
                              r.data_ptr() if r is not None else None, n,
                              out.data_ptr(), lse.data_ptr())
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    if r is None:
        return out.view(B, Hq, Lq, Dv), lse.view(B, Hq, Lq)
    return out, lse


def decode_paged(q, k_pages, v_pages, page_table, seq_lens, *, scale=None, rows=None):
    """Paged GQA decode.  q [B,Hq,D]; k_pages/v_pages [num_pages,Hkv,page_size,D];
    page_table [B,max_pages] int32; seq_lens [B] int32.  Returns fp64 (out [B,Hq,D],
    lse [B,Hq]) or per-row results for flat ids b*Hq + h in ``rows``."""
    lib = _load()
    q, kp, vp = _cpu(q), _cpu(k_pages), _cpu(v_pages)
    pt = _cpu(page_table).to(torch.int32)
    sl = _cpu(seq_lens).to(torch.int32)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = kp.shape
    if scale is None:
        scale = D ** -0.5
    r, n = _rows(rows)
    n_out = n if r is not None else B * Hq
    out = torch.empty(n_out, D, dtype=torch.float64)
    lse = torch.empty(n_out, dtype=torch.float64)
    rc = lib.oracle_decode_paged(q.data_ptr(), kp.data_ptr(), vp.data_ptr(), _code(q),
                                 pt.data_ptr(), sl.data_ptr(), B, Hq, Hkv, D, page_size,
                                 pt.shape[1], num_pages, float(scale),
                                 r.data_ptr() if r is not None else None, n,
                                 out.data_ptr(), lse.data_ptr())
    if rc != 0:
        raise ValueError("oracle_decode_paged rejected its arguments")
    if r is None:
        return out.view(B, Hq, D), lse.view(B, Hq)
    return out, lse


def prefill_paged(q, k_pages, v_pages, page_table, seq_lens, *, causal=True, scale=None,
                  mask=None, rows=None):
    """Chunked prefill against a paged cache.  q [B,Hq,Lq,D]; k_pages/v_pages
    [num_pages,Hkv,page_size,D]; page_table [B,max_pages]; seq_lens [B] (the chunk included);
    optional additive mask [1 or B, Lq, >= max seq_lens].  For each sequence b the first
    seq_lens[b] cached tokens are gathered in page order into dense [1,Hkv,seq_lens[b],D]
    keys and values and ``attention`` runs on them (with the mask's first seq_lens[b]
    columns), so the Lq queries sit at the sequence's last Lq positions.  Returns fp64 (out [B,Hq,Lq,D],
    lse [B,Hq,Lq]) or per-row results for flat ids (b*Hq + h)*Lq + i in ``rows``."""
    q, kp, vp = _cpu(q), _cpu(k_pages), _cpu(v_pages)
    pt, sl = _cpu(page_table).to(torch.int64), _cpu(seq_lens).to(torch.int64)
    B, Hq, Lq, D = q.shape
    num_pages, Hkv, page_size, _ = kp.shape
    per_b = Hq * Lq
    if mask is not None:
        mask = _cpu(mask)
        if mask.dim() == 2:
            mask = mask.unsqueeze(0)
    outs, lses, where = [], [], []
    sel = None if rows is None else torch.as_tensor(rows, dtype=torch.int64).reshape(-1)
    for b in range(B):
        n = int(sl[b])
        n_pages = -(-n // page_size)
        ids = pt[b, :n_pages]
        if n_pages and (int(ids.min()) < 0 or int(ids.max()) >= num_pages):
            raise ValueError("page id out of range")
        # [n_pages, Hkv, page_size, D] -> [1, Hkv, n_pages * page_size, D], first n tokens
        kb = kp[ids].permute(1, 0, 2, 3).reshape(1, Hkv, n_pages * page_size, D)[:, :, :n]
        vb = vp[ids].permute(1, 0, 2, 3).reshape(1, Hkv, n_pages * page_size, D)[:, :, :n]
        kb, vb = kb.contiguous(), vb.contiguous()
        mb = None
        if mask is not None:
            mb = mask[0 if mask.shape[0] == 1 else b, :, :n].unsqueeze(0).contiguous()
        if sel is None:
            o, l = attention(q[b:b + 1], kb, vb, causal=causal, scale=scale, mask=mb)
            outs.append(o[0])
            lses.append(l[0])
        else:
            pos = torch.nonzero((sel >= b * per_b) & (sel < (b + 1) * per_b)).reshape(-1)
            if pos.numel():
                o, l = attention(q[b:b + 1], kb, vb, causal=causal, scale=scale, mask=mb,
                                 rows=(sel[pos] - b * per_b).tolist())
                outs.append(o)
                lses.append(l)
                where.append(pos)
    if sel is None:
        return torch.stack(outs), torch.stack(lses)
    o = torch.empty(sel.numel(), D, dtype=torch.float64)
    l = torch.empty(sel.numel(), dtype=torch.float64)
    if where:
        idx = torch.cat(where)
        o[idx] = torch.cat(outs)
        l[idx] = torch.cat(lses)
    return o, l


def mla_decode_paged(q_nope, q_pe, ckv, kpe, page_table, seq_lens, *, scale, rows=None):
    """MLA paged decode (latent form).  q_nope [B,H,Dc]; q_pe [B,H,Dr];
    ckv [num_pages,page_size,Dc]; kpe [num_pages,page_size,Dr]; page_table [B,max_pages];
    seq_lens [B].  Returns fp64 (out [B,H,Dc], lse [B,H]) or per-row results."""
    lib = _load()
    qn, qp, c, kr = _cpu(q_nope), _cpu(q_pe), _cpu(ckv), _cpu(kpe)
    pt = _cpu(page_table).to(torch.int32)
    sl = _cpu(seq_lens).to(torch.int32)
    B, H, Dc = qn.shape
    Dr = qp.shape[2]
    num_pages, page_size = c.shape[0], c.shape[1]
    r, n = _rows(rows)
    n_out = n if r is not None else B * H
    out = torch.empty(n_out, Dc, dtype=torch.float64)
    lse = torch.empty(n_out, dtype=torch.float64)
    rc = lib.oracle_mla_decode_paged(qn.data_ptr(), qp.data_ptr(), c.data_ptr(),
                                     kr.data_ptr(), _code(qn), pt.data_ptr(), sl.data_ptr(),
                                     B, H, Dc, Dr, page_size, pt.shape[1], num_pages,
                                     float(scale), r.data_ptr() if r is not None else None,
                                     n, out.data_ptr(), lse.data_ptr())
    if rc != 0:
        raise ValueError("oracle_mla_decode_paged rejected its arguments")
    if r is None:
        return out.view(B, H, Dc), lse.view(B, H)
    return out, lse


def merge(o_parts, lse_parts):
    """Merge attention states.  o_parts [rows,S,D], lse_parts [rows,S] (fp32 or fp64).
    Returns fp64 (out [rows,D], lse [rows])."""
    lib = _load()
    o = _cpu(o_parts)
    l = _cpu(lse_parts).to(o.dtype)
    rows, S, D = o.shape
    out = torch.empty(rows, D, dtype=torch.float64)
    lse = torch.empty(rows, dtype=torch.float64)
    rc = lib.oracle_merge(o.data_ptr(), l.data_ptr(), _code(o), rows, S, D,
                          out.data_ptr(), lse.data_ptr())
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return out, lse


def gated_delta(q, k, v, g, beta, *, scale=None, initial_state=None):
    """Gated delta rule, token by token.  q, k [B,Hk,T,dk]; v [B,Hv,T,dv] (one dtype);
    g (log decay), beta [B,Hv,T]; initial_state [B,Hv,dv,dk] or None (zero).  Value head h
    reads query/key head h // (Hv // Hk).  Returns fp64 (out [B,Hv,T,dv], final state
    [B,Hv,dv,dk])."""
    lib = _load_gd()
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    g, beta = _cpu(g), _cpu(beta)
    if not (q.dtype == k.dtype == v.dtype) or g.dtype != beta.dtype:
        raise TypeError("q, k, v must share a dtype, and g, beta another")
    B, Hk, T, dk = q.shape
    Hv, dv = v.shape[1], v.shape[3]
    if k.shape != q.shape or v.shape != (B, Hv, T, dv) or g.shape != (B, Hv, T) or \
            beta.shape != (B, Hv, T) or Hv % Hk:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = dk ** -0.5
    s0 = None
    if initial_state is not None:
        s0 = _cpu(initial_state).to(torch.float64)
        if s0.shape != (B, Hv, dv, dk):
            raise ValueError("initial_state must be [B,Hv,dv,dk]")
    out = torch.empty(B, Hv, T, dv, dtype=torch.float64)
    st = torch.empty(B, Hv, dv, dk, dtype=torch.float64)
    rc = lib.oracle_gated_delta(q.data_ptr(), k.data_ptr(), v.data_ptr(), _code(q),
                                g.data_ptr(), beta.data_ptr(), _code(g),
                                s0.data_ptr() if s0 is not None else None,
                                B, T, Hk, Hv, dk, dv, float(scale), out.data_ptr(), st.data_ptr())
    if rc != 0:
        raise ValueError("oracle_gated_delta rejected its arguments")
    return out, st
