"""GB300 (sm_103a) fused softmax-attention forward: Python binding of libfa.so.

Argument marshalling only.  Every step of the computation runs in the CUDA kernels behind
the C ABI in ``include/fa.h``; PyTorch provides device memory and the current stream.  There
is no fallback: if the library is missing or a call fails, an exception is raised.

Entry points (same names as the C ABI):
    fa_prefill(q, k, v, causal, scale)                       bf16, spec signature
    fa_prefill_ex(q, k, v, causal=..., scale=..., mask=..., num_splits=..., dtype from q)
    fa_decode_paged(q, k_pages, v_pages, page_table, seq_lens, max_seq_len, scale)
    mla_decode_paged(q_nope, q_pe, ckv, kpe, page_table, seq_lens, max_seq_len, scale)
    fa_merge_states(o_parts, lse_parts, n_splits=None, out_dtype=torch.bfloat16)
    fa_get_device_status()
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT, \
    FA_ERR_BOUNDS = range(7)
FA_BF16, FA_FP16, FA_FP32 = 0, 1, 2
_DT = {torch.bfloat16: FA_BF16, torch.float16: FA_FP16, torch.float32: FA_FP32}

# Every symbol include/fa.h declares.
EXPORTS = (
    "fa_prefill", "fa_prefill_ex", "fa_prefill_workspace_size", "fa_prefill_num_splits",
    "fa_prefill_paged", "fa_prefill_paged_workspace_size",
    "fa_decode_paged", "fa_decode_paged_ex", "fa_decode_workspace_size", "fa_decode_chunk_tokens",
    "fa_decode_get_plan",
    "fa_decode_paged_noalloc",
    "fa_decode_paged_states", "mla_decode_paged", "mla_decode_workspace_size",
    "mla_decode_chunk_tokens", "mla_decode_paged_states", "mla_decode_paged_ex", "fa_merge_states",
    "fa_get_device_status", "fa_selftest_wait_timeout", "fa_last_error", "fa_version",
    "gated_delta_prefill", "gated_delta_workspace_size",
)


class FAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[fa status {code}] {msg}")
        self.code = code


class PrefillArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Lq", ctypes.c_int),
        ("Lkv", ctypes.c_int), ("D", ctypes.c_int), ("causal", ctypes.c_int),
        ("scale", ctypes.c_float), ("dtype", ctypes.c_int), ("mask", ctypes.c_void_p),
        ("mask_dtype", ctypes.c_int), ("mask_batches", ctypes.c_int),
        ("num_splits", ctypes.c_int), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("page_size", ctypes.c_int), ("max_pages", ctypes.c_int), ("num_pages", ctypes.c_int),
    ]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
        ("page_size", ctypes.c_int), ("max_pages_per_seq", ctypes.c_int),
        ("num_pages", ctypes.c_int), ("max_seq_len", ctypes.c_int),
        ("scale", ctypes.c_float), ("dtype", ctypes.c_int), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("path", ctypes.c_int),
    ]


class DecodePlan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("n_splits", ctypes.c_int), ("launches", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t)]


# fa_decode_path
FA_DECODE_AUTO, FA_DECODE_CUDA_CORES, FA_DECODE_TENSOR_CORES = 0, 1, 2


class MlaArgs(ctypes.Structure):
    _fields_ = [
        ("q_nope", ctypes.c_void_p), ("q_pe", ctypes.c_void_p),
        ("ckv_pages", ctypes.c_void_p), ("kpe_pages", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("Dc", ctypes.c_int), ("Dr", ctypes.c_int),
        ("page_size", ctypes.c_int), ("max_pages_per_seq", ctypes.c_int),
        ("num_pages", ctypes.c_int), ("max_seq_len", ctypes.c_int),
        ("scale", ctypes.c_float), ("dtype", ctypes.c_int), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class GatedDeltaArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("initial_state", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("final_state", ctypes.c_void_p),
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
        ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("scale", ctypes.c_float),
        ("dtype", ctypes.c_int), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_lock = threading.Lock()
_lib = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def load_library(path: str | None = None):
    """Load libfa.so (built by ``softmax_attention_gb300.build``).  Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} not found: build it with `python -m softmax_attention_gb300.build`")
        lib = ctypes.CDLL(p)
        lib.fa_prefill.restype = _i
        lib.fa_prefill.argtypes = [_vp, _vp, _vp, _vp, _vp] + [_i] * 7 + [_f, _vp]
        lib.fa_prefill_ex.restype = _i
        lib.fa_prefill_ex.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
        lib.fa_prefill_workspace_size.restype = _sz
        lib.fa_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
        lib.fa_prefill_num_splits.restype = _i
        lib.fa_prefill_num_splits.argtypes = [ctypes.POINTER(PrefillArgs)]
        lib.fa_prefill_paged.restype = _i
        lib.fa_prefill_paged.argtypes = [_vp] * 7 + [_i] * 10 + [_f, _vp, _sz, _vp]
        lib.fa_prefill_paged_workspace_size.restype = _sz
        lib.fa_prefill_paged_workspace_size.argtypes = [_i] * 6
        lib.fa_decode_paged.restype = _i
        lib.fa_decode_paged.argtypes = [_vp] * 7 + [_i] * 8 + [_f, _vp, _sz, _vp]
        lib.fa_decode_paged_ex.restype = _i
        lib.fa_decode_paged_ex.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
        lib.fa_decode_get_plan.restype = _i
        lib.fa_decode_get_plan.argtypes = [ctypes.POINTER(DecodeArgs), ctypes.POINTER(DecodePlan)]
        lib.mla_decode_paged_ex.restype = _i
        lib.mla_decode_paged_ex.argtypes = [ctypes.POINTER(MlaArgs), _vp]
        lib.fa_decode_workspace_size.restype = _sz
        lib.fa_decode_workspace_size.argtypes = [_i] * 4
        lib.fa_decode_paged_noalloc.restype = _i
        lib.fa_decode_paged_noalloc.argtypes = [_vp] * 7 + [_i] * 8 + [_f, _vp]
        lib.fa_decode_chunk_tokens.restype = _i
        lib.fa_decode_chunk_tokens.argtypes = [_i] * 3
        lib.fa_decode_paged_states.restype = _i
        lib.fa_decode_paged_states.argtypes = [_vp] * 7 + [_i] * 9 + [_f, _vp]
        lib.mla_decode_chunk_tokens.restype = _i
        lib.mla_decode_chunk_tokens.argtypes = [_i] * 3
        lib.mla_decode_paged_states.restype = _i
        lib.mla_decode_paged_states.argtypes = [_vp] * 8 + [_i] * 9 + [_f, _vp]
        lib.mla_decode_paged.restype = _i
        lib.mla_decode_paged.argtypes = [_vp] * 8 + [_i] * 8 + [_f, _vp, _sz, _vp]
        lib.mla_decode_workspace_size.restype = _sz
        lib.mla_decode_workspace_size.argtypes = [_i] * 4
        lib.fa_merge_states.restype = _i
        lib.fa_merge_states.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
        lib.fa_get_device_status.restype = _i
        lib.fa_get_device_status.argtypes = [_vp]
        lib.fa_selftest_wait_timeout.restype = _i
        lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, _vp]
        lib.fa_last_error.restype = ctypes.c_char_p
        lib.fa_last_error.argtypes = []
        lib.fa_version.restype = _i
        lib.fa_version.argtypes = []
        lib.gated_delta_prefill.restype = _i
        lib.gated_delta_prefill.argtypes = [ctypes.POINTER(GatedDeltaArgs), _vp]
        lib.gated_delta_workspace_size.restype = _sz
        lib.gated_delta_workspace_size.argtypes = [ctypes.POINTER(GatedDeltaArgs)]
        _lib = lib
        return lib


def _check(rc: int):
    if rc != FA_OK:
        raise FAError(rc, load_library().fa_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_dtype(dtype, *ts):
    """The C entry points take raw pointers; element types are checked here."""
    for t in ts:
        if t is not None and t.dtype != dtype:
            raise ValueError(f"expected {dtype}, got {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _workspace(nbytes: int, device, workspace):
    if nbytes == 0:
        return None
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------------------------------
def fa_prefill(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
               stream=None):
    """bf16 dense attention through the short-form entry point (no KV split)."""
    lib = load_library()
    _need_dtype(torch.bfloat16, q, k, v, out)
    _need_dtype(torch.float32, lse)
    _need_cuda(q, k, v, out, lse)
    B, Hq, Lq, D = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Lq, dtype=torch.float32, device=q.device)
    _check(lib.fa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Lq, Lkv, D,
                          int(bool(causal)), float(scale), _stream(stream)))
    return out, lse


def prefill_args(q, k, v, *, causal=False, scale=None, out=None, lse=None, mask=None,
                 num_splits=0, workspace=None, page_table=None, seq_lens=None,
                 max_seq_len=None) -> PrefillArgs:
    """Argument struct of fa_prefill_ex.  Dense: k, v [B,Hkv,Lkv,D].  Paged (page_table
    given): k, v are pages [num_pages,Hkv,page_size,D] and Lkv = max_seq_len."""
    B, Hq, Lq, D = q.shape
    if page_table is None:
        Hkv, Lkv = k.shape[1], k.shape[2]
    else:
        Hkv, Lkv = k.shape[1], int(max_seq_len)
    a = PrefillArgs()
    if page_table is not None:
        a.page_table = page_table.data_ptr()
        a.seq_lens = seq_lens.data_ptr()
        a.num_pages, a.page_size = k.shape[0], k.shape[2]
        a.max_pages = page_table.shape[1]
    a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    a.out = out.data_ptr() if out is not None else None
    a.lse = lse.data_ptr() if lse is not None else None
    a.B, a.Hq, a.Hkv, a.Lq, a.Lkv, a.D = B, Hq, Hkv, Lq, Lkv, D
    a.causal = int(bool(causal))
    a.scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    if q.dtype not in _DT:
        raise TypeError(f"unsupported dtype {q.dtype}")
    a.dtype = _DT[q.dtype]
    if mask is not None:
        m = mask if mask.dim() == 3 else mask.unsqueeze(0)
        a.mask = m.data_ptr()
        a.mask_dtype = _DT[m.dtype]
        a.mask_batches = m.shape[0]
    a.num_splits = int(num_splits)
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def fa_prefill_ex(q, k, v, *, causal=False, scale=None, mask=None, num_splits=0, out=None,
                  lse=None, workspace=None, stream=None):
    """Dense attention, any supported dtype (bf16/fp16/fp32), optional additive mask
    [1 or B, Lq, Lkv], optional KV split (0 = library's choice)."""
    lib = load_library()
    _need_dtype(q.dtype, k, v, out)
    _need_dtype(torch.float32, lse)
    _need_cuda(q, k, v, mask, out, lse)
    B, Hq, Lq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Lq, dtype=torch.float32, device=q.device)
    a = prefill_args(q, k, v, causal=causal, scale=scale, out=out, lse=lse, mask=mask,
                     num_splits=num_splits)
    need = lib.fa_prefill_workspace_size(ctypes.byref(a))
    ws = _workspace(need, q.device, workspace)
    if ws is not None:
        a.workspace = ws.data_ptr()
        a.workspace_bytes = ws.numel() * ws.element_size()
    _check(lib.fa_prefill_ex(ctypes.byref(a), _stream(stream)))
    return out, lse


def prefill_workspace_size(q, k, v, **kw) -> int:
    return load_library().fa_prefill_workspace_size(ctypes.byref(prefill_args(q, k, v, **kw)))


def prefill_num_splits(q, k, v, **kw) -> int:
    return load_library().fa_prefill_num_splits(ctypes.byref(prefill_args(q, k, v, **kw)))


def fa_prefill_paged_workspace_size(B, Hq, Hkv, Lq, D, max_seq_len) -> int:
    return load_library().fa_prefill_paged_workspace_size(B, Hq, Hkv, Lq, D, max_seq_len)


def fa_prefill_paged(q, k_pages, v_pages, page_table, seq_lens, max_seq_len: int,
                     causal: bool = True, scale: float | None = None, mask=None, num_splits=0,
                     out=None, lse=None, workspace=None, stream=None):
    """Chunked prefill against a paged cache (fa_prefill_ex with a page table).
    q [B,Hq,Lq,D] bf16 or fp16 (each sequence's last Lq positions); pages
    [num_pages,Hkv,page_size,D] in q's dtype; page_table [B,max_pages] int32; seq_lens [B]
    int32 (device): each sequence's cached tokens, the chunk included; optional additive
    mask [1 or B, Lq, max_seq_len]."""
    lib = load_library()
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"expected bfloat16 or float16, got {q.dtype}")
    _need_dtype(q.dtype, k_pages, v_pages, out)
    _need_dtype(torch.int32, page_table, seq_lens)
    _need_dtype(torch.float32, lse)
    _need_cuda(q, k_pages, v_pages, page_table, seq_lens, mask, out, lse)
    B, Hq, Lq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Lq, dtype=torch.float32, device=q.device)
    a = prefill_args(q, k_pages, v_pages, causal=causal, scale=scale, out=out, lse=lse,
                     mask=mask, num_splits=num_splits, page_table=page_table,
                     seq_lens=seq_lens, max_seq_len=max_seq_len)
    ws = _workspace(lib.fa_prefill_workspace_size(ctypes.byref(a)), q.device, workspace)
    if ws is not None:
        a.workspace = ws.data_ptr()
        a.workspace_bytes = ws.numel() * ws.element_size()
    _check(lib.fa_prefill_ex(ctypes.byref(a), _stream(stream)))
    return out, lse


def fa_decode_workspace_size(B, Hq, D, max_seq_len) -> int:
    return load_library().fa_decode_workspace_size(B, Hq, D, max_seq_len)


def decode_args(q, k_pages, v_pages, page_table, seq_lens, max_seq_len: int,
                scale: float | None = None, out=None, lse=None, workspace=None,
                path: int = FA_DECODE_AUTO) -> DecodeArgs:
    """Argument struct of fa_decode_paged_ex (sizes from the tensors' shapes)."""
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"expected bfloat16 or float16, got {q.dtype}")
    return DecodeArgs(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(seq_lens),
                      _ptr(out), _ptr(lse), B, Hq, Hkv, D, page_size, page_table.shape[1],
                      num_pages, int(max_seq_len), float(scale), _DT[q.dtype], _ptr(workspace),
                      0 if workspace is None else workspace.numel() * workspace.element_size(),
                      int(path))


def fa_decode_get_plan(q, k_pages, v_pages, page_table, seq_lens, max_seq_len: int,
                       path: int = FA_DECODE_AUTO) -> dict:
    """What a decode call with these tensors does: {"path", "n_splits", "launches",
    "workspace_bytes"} (path 1 = CUDA cores, 2 = tensor cores)."""
    lib = load_library()
    a = decode_args(q, k_pages, v_pages, page_table, seq_lens, max_seq_len, path=path)
    pl = DecodePlan()
    _check(lib.fa_decode_get_plan(ctypes.byref(a), ctypes.byref(pl)))
    return {"path": pl.path, "n_splits": pl.n_splits, "launches": pl.launches,
            "workspace_bytes": pl.workspace_bytes}


def fa_decode_paged(q, k_pages, v_pages, page_table, seq_lens, max_seq_len: int,
                    scale: float | None = None, out=None, lse=None, workspace=None, stream=None,
                    path: int = FA_DECODE_AUTO):
    """Split-KV paged GQA decode.  q [B,Hq,D] bf16 or fp16; pages [num_pages,Hkv,page_size,D]
    in q's dtype; page_table [B,max_pages] int32; seq_lens [B] int32 (device).  path: 0 the
    library's choice, 1 the CUDA-core kernel, 2 the tensor-core kernel."""
    lib = load_library()
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"expected bfloat16 or float16, got {q.dtype}")
    _need_dtype(q.dtype, k_pages, v_pages)
    _need_dtype(torch.int32, page_table, seq_lens)
    _need_cuda(q, k_pages, v_pages, page_table, seq_lens)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    _need_dtype(q.dtype, out)
    _need_dtype(torch.float32, lse)
    _need_cuda(out, lse)
    need = fa_decode_get_plan(q, k_pages, v_pages, page_table, seq_lens, max_seq_len,
                              path)["workspace_bytes"]
    ws = _workspace(need, q.device, workspace)
    a = decode_args(q, k_pages, v_pages, page_table, seq_lens, max_seq_len, scale, out, lse, ws,
                    path)
    _check(lib.fa_decode_paged_ex(ctypes.byref(a), _stream(stream)))
    return out, lse


def fa_decode_paged_noalloc(q, k_pages, v_pages, page_table, seq_lens, max_seq_len: int,
                            scale: float | None = None, out=None, lse=None, stream=None):
    """fa_decode_paged without a workspace, for callers that cannot allocate: the library's
    fixed device scratch is used instead (problems needing more than it holds are refused).
    Calls that overlap on the GPU share that scratch and race."""
    lib = load_library()
    _need_dtype(torch.bfloat16, q, k_pages, v_pages, out)
    _need_dtype(torch.int32, page_table, seq_lens)
    _need_dtype(torch.float32, lse)
    _need_cuda(q, k_pages, v_pages, page_table, seq_lens, out, lse)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    _check(lib.fa_decode_paged_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                       _ptr(seq_lens), _ptr(out), _ptr(lse), B, Hq, Hkv, D,
                                       page_size, page_table.shape[1], num_pages,
                                       int(max_seq_len), float(scale), _stream(stream)))
    return out, lse


def fa_decode_chunk_tokens(B, Hq, max_seq_len) -> int:
    return load_library().fa_decode_chunk_tokens(B, Hq, max_seq_len)


def fa_decode_paged_states(q, k_pages, v_pages, page_table, seq_lens, max_seq_len: int,
                           scale: float | None = None, o_parts=None, lse_parts=None, stream=None):
    """Per-chunk split-KV states of paged decode (no merge).  Returns (o_parts
    [B*Hq, n_chunks, D] fp32, lse_parts [B*Hq, n_chunks] fp32, chunk)."""
    lib = load_library()
    _need_dtype(torch.bfloat16, q, k_pages, v_pages)
    _need_dtype(torch.int32, page_table, seq_lens)
    _need_cuda(q, k_pages, v_pages, page_table, seq_lens)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_pages.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    chunk = lib.fa_decode_chunk_tokens(B, Hq, max_seq_len)
    n = -(-max_seq_len // chunk)
    if o_parts is None:
        o_parts = torch.empty(B * Hq, n, D, dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty(B * Hq, n, dtype=torch.float32, device=q.device)
    _check(lib.fa_decode_paged_states(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                      _ptr(seq_lens), _ptr(o_parts), _ptr(lse_parts), n, B, Hq,
                                      Hkv, D, page_size, page_table.shape[1], num_pages,
                                      int(max_seq_len), float(scale), _stream(stream)))
    return o_parts, lse_parts, chunk


def mla_decode_chunk_tokens(B, H, max_seq_len) -> int:
    return load_library().mla_decode_chunk_tokens(B, H, max_seq_len)


def mla_decode_paged_states(q_nope, q_pe, ckv, kpe, page_table, seq_lens, max_seq_len: int,
                            scale: float, o_parts=None, lse_parts=None, stream=None):
    """Per-chunk split-KV states of MLA decode (no merge).  Returns (o_parts, lse_parts,
    chunk)."""
    lib = load_library()
    _need_dtype(torch.bfloat16, q_nope, q_pe, ckv, kpe)
    _need_dtype(torch.int32, page_table, seq_lens)
    _need_cuda(q_nope, q_pe, ckv, kpe, page_table, seq_lens)
    B, H, Dc = q_nope.shape
    Dr = q_pe.shape[2]
    num_pages, page_size = ckv.shape[0], ckv.shape[1]
    chunk = lib.mla_decode_chunk_tokens(B, H, max_seq_len)
    n = -(-max_seq_len // chunk)
    if o_parts is None:
        o_parts = torch.empty(B * H, n, Dc, dtype=torch.float32, device=q_nope.device)
    if lse_parts is None:
        lse_parts = torch.empty(B * H, n, dtype=torch.float32, device=q_nope.device)
    _check(lib.mla_decode_paged_states(_ptr(q_nope), _ptr(q_pe), _ptr(ckv), _ptr(kpe),
                                       _ptr(page_table), _ptr(seq_lens), _ptr(o_parts),
                                       _ptr(lse_parts), n, B, H, Dc, Dr, page_size,
                                       page_table.shape[1], num_pages, int(max_seq_len),
                                       float(scale), _stream(stream)))
    return o_parts, lse_parts, chunk


def mla_decode_workspace_size(B, H, Dc, max_seq_len) -> int:
    return load_library().mla_decode_workspace_size(B, H, Dc, max_seq_len)


def mla_decode_paged(q_nope, q_pe, ckv, kpe, page_table, seq_lens, max_seq_len: int,
                     scale: float, out=None, lse=None, workspace=None, stream=None):
    """MLA paged decode (latent form).  q_nope [B,H,512], q_pe [B,H,64] bf16 or fp16;
    ckv [P,page_size,512], kpe [P,page_size,64] in that dtype; page_table [B,max_pages];
    seq_lens [B]."""
    lib = load_library()
    if q_nope.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"expected bfloat16 or float16, got {q_nope.dtype}")
    _need_dtype(q_nope.dtype, q_pe, ckv, kpe)
    _need_dtype(torch.int32, page_table, seq_lens)
    _need_cuda(q_nope, q_pe, ckv, kpe, page_table, seq_lens)
    B, H, Dc = q_nope.shape
    Dr = q_pe.shape[2]
    num_pages, page_size = ckv.shape[0], ckv.shape[1]
    if out is None:
        out = torch.empty_like(q_nope)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q_nope.device)
    _need_dtype(q_nope.dtype, out)
    _need_dtype(torch.float32, lse)
    _need_cuda(out, lse)
    ws = _workspace(lib.mla_decode_workspace_size(B, H, Dc, max_seq_len), q_nope.device, workspace)
    a = MlaArgs(_ptr(q_nope), _ptr(q_pe), _ptr(ckv), _ptr(kpe), _ptr(page_table), _ptr(seq_lens),
                _ptr(out), _ptr(lse), B, H, Dc, Dr, page_size, page_table.shape[1], num_pages,
                int(max_seq_len), float(scale), _DT[q_nope.dtype], _ptr(ws),
                0 if ws is None else ws.numel())
    _check(lib.mla_decode_paged_ex(ctypes.byref(a), _stream(stream)))
    return out, lse


def fa_merge_states(o_parts, lse_parts, n_splits=None, out_dtype=torch.bfloat16, out=None,
                    lse=None, stream=None):
    """Merge partial states: o_parts [rows,S,D] fp32, lse_parts [rows,S] fp32."""
    lib = load_library()
    _need_dtype(torch.float32, o_parts, lse_parts, lse)
    _need_dtype(torch.int32, n_splits)
    _need_cuda(o_parts, lse_parts, n_splits, out, lse)
    rows, S, D = o_parts.shape
    if out is None:
        out = torch.empty(rows, D, dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=o_parts.device)
    _check(lib.fa_merge_states(_ptr(o_parts), _ptr(lse_parts), _ptr(n_splits), _ptr(out),
                               _ptr(lse), rows, D, S, _DT[out.dtype], _stream(stream)))
    return out, lse


def fa_get_device_status(stream=None) -> int:
    """Synchronise, return and clear the library's sticky device status (0 = OK)."""
    return load_library().fa_get_device_status(_stream(stream))


def fa_selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    """Enqueue the failure-path self-test (a bounded wait that runs out); returns the call's
    status.  Read the result with fa_get_device_status(): FA_ERR_TIMEOUT."""
    return load_library().fa_selftest_wait_timeout(int(timeout_us), _stream(stream))


def fa_last_error() -> str:
    return load_library().fa_last_error().decode(errors="replace")


def gated_delta_args(q, k, v, g, beta, *, scale=None, initial_state=None, out=None,
                     final_state=None, workspace=None) -> GatedDeltaArgs:
    """Argument struct of gated_delta_prefill (sizes from the tensors' shapes)."""
    B, Hk, T, dk = q.shape
    Hv, dv = v.shape[1], v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    if q.dtype not in _DT:
        raise TypeError(f"unsupported dtype {q.dtype}")
    return GatedDeltaArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                          _ptr(out), _ptr(final_state), B, T, Hk, Hv, dk, dv, float(scale),
                          _DT[q.dtype], _ptr(workspace),
                          0 if workspace is None else workspace.numel() * workspace.element_size())


def gated_delta_workspace_size(q, k, v, g, beta) -> int:
    return load_library().gated_delta_workspace_size(
        ctypes.byref(gated_delta_args(q, k, v, g, beta)))


def gated_delta_prefill(q, k, v, g, beta, *, scale=None, initial_state=None, out=None,
                        final_state=None, want_state=True, workspace=None, stream=None):
    """Chunked prefill of gated-delta linear attention.  q, k [B,Hk,T,dk] bf16; v [B,Hv,T,dv]
    bf16; g (log decay), beta [B,Hv,T] fp32; initial_state [B,Hv,dv,dk] fp32 or None.
    Returns (out [B,Hv,T,dv] bf16, final state [B,Hv,dv,dk] fp32 or None)."""
    lib = load_library()
    _need_dtype(torch.bfloat16, q, k, v, out)
    _need_dtype(torch.float32, g, beta, initial_state, final_state)
    _need_cuda(q, k, v, g, beta, initial_state, out, final_state)
    B, Hk, T, dk = q.shape
    Hv, dv = v.shape[1], v.shape[3]
    if out is None:
        out = torch.empty(B, Hv, T, dv, dtype=torch.bfloat16, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty(B, Hv, dv, dk, dtype=torch.float32, device=q.device)
    a = gated_delta_args(q, k, v, g, beta, scale=scale, initial_state=initial_state, out=out,
                         final_state=final_state)
    ws = _workspace(lib.gated_delta_workspace_size(ctypes.byref(a)), q.device, workspace)
    if ws is not None:
        a.workspace = ws.data_ptr()
        a.workspace_bytes = ws.numel() * ws.element_size()
    _check(lib.gated_delta_prefill(ctypes.byref(a), _stream(stream)))
    return out, final_state
