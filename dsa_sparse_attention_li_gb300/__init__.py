"""DSA hot path on GB300: fused Lightning Indexer top-K and Sparse Flash Attention.

A thin ctypes binding over the C-ABI library ``libdsa.so`` (declared in ``include/dsa.h``).
Every step of the path runs in the library's CUDA kernels; this module only marshals torch
tensors (device pointers, the current stream) into the C argument structs and allocates output
tensors when the caller does not pass them.  There is no CPU or framework fallback: if the
library cannot be built or loaded, ``load()`` raises.

Functions (same names as the C entry points, without the ``dsa_`` prefix):
    li_topk(...)             -> (idx [n_q, K] int32, cnt [n_q] int32)
    sfa_decode(...)          -> (out [n_q, H, 512] bf16, lse [n_q, H] fp32)
    sfa_prefill(...)         -> same
    sfa_workspace_bytes(...) -> int
    page_bytes(dtype, rows, dim), page_table_validate(...), cache_write(...)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")
HOOKS_LIB_PATH = os.path.join(_PKG, "libdsa_testhooks.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_DEVICE_CHECK, DSA_ERR_TIMEOUT = range(6)
DSA_BF16, DSA_FP8_E4M3, DSA_MXFP8_E4M3 = 0, 1, 2

SYMBOLS = ["dsa_status_string", "dsa_last_error", "dsa_abi_version", "dsa_li_workspace_bytes", "dsa_li_topk",
           "dsa_sfa_workspace_bytes", "dsa_sfa_decode", "dsa_sfa_prefill",
           "dsa_sfa_decode_static", "dsa_page_bytes", "dsa_page_table_validate",
           "dsa_cache_write", "dsa_prolog_workspace_bytes", "dsa_indexer_prolog", "dsa_topk_merge"]

# Capacity of the library's fixed scratch array used by dsa_sfa_decode_static.
SFA_STATIC_SCRATCH_BYTES = 20 * 1024 * 1024


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        super().__init__("%s: %s%s" % (where, status_string(code) if _lib else code,
                                       (" -- " + detail) if detail else ""))


class LiArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "n_q", "H_I", "d_I", "K", "page_size", "max_pages", "num_pages", "max_seq_len",
        "max_q_per_seq", "dtype")] + [(n, ctypes.c_void_p) for n in (
            "q", "q_scale", "w", "k_pool", "k_scale", "page_table", "seq_lens", "q_start",
            "out_idx", "out_cnt", "status", "q_sf", "k_sf", "out_score", "workspace")] + [
        ("workspace_bytes", ctypes.c_size_t)]


class MergeArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("S", "n_q", "K_in", "K")] + [
        (n, ctypes.c_void_p) for n in ("cand_idx", "cand_score", "shard_offset", "out_idx", "out_cnt")]


class PrologArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_q", "B", "d_q", "d_model", "H_I", "d_I", "dtype", "page_size", "max_pages",
        "num_pages")] + [("ln_eps", ctypes.c_float), ("w_scale", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in (
            "xq", "x", "w_q", "w_k", "w_w", "ln_gamma", "ln_beta", "page_table", "seq_lens",
            "q_start", "q_out", "q_sf", "w_out", "k_pool", "k_sf", "workspace")] + [
        ("workspace_bytes", ctypes.c_size_t), ("status", ctypes.c_void_p)]


class SfaArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "n_q", "H", "d_qk", "d_v", "K", "page_size", "max_pages", "num_pages", "max_seq_len",
        "max_q_per_seq")] + [("softmax_scale", ctypes.c_float)] + [(n, ctypes.c_void_p) for n in (
            "q", "kv_pool", "page_table", "seq_lens", "q_start", "idx", "out", "lse", "status",
            "workspace")] + [("workspace_bytes", ctypes.c_size_t), ("kv_dtype", ctypes.c_int),
                             ("row_splits", ctypes.c_int)]


_lib = None
_hooks = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) libdsa.so.  Raises if it cannot."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdsa.so not built (run __graft_entry__.build())")
    _lib = _configure(ctypes.CDLL(LIB_PATH))
    return _lib


def load_testhooks(build_if_missing: bool = True) -> ctypes.CDLL:
    """The test build libdsa_testhooks.so (short device-side wait limits and
    dsa_test_inject_stall; include/dsa_testhooks.h).  For the failure-handling tests only."""
    global _hooks
    if _hooks is not None:
        return _hooks
    if build_if_missing and not _build.up_to_date(HOOKS_LIB_PATH):
        _build.build(hooks=True)
    if not os.path.exists(HOOKS_LIB_PATH):
        raise RuntimeError("libdsa_testhooks.so not built (run __graft_entry__.build())")
    lib = _configure(ctypes.CDLL(HOOKS_LIB_PATH))
    lib.dsa_test_inject_stall.argtypes = [ctypes.c_int]
    lib.dsa_test_inject_stall.restype = None
    _hooks = lib
    return lib


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_last_error.restype = ctypes.c_char_p
    lib.dsa_abi_version.restype = ctypes.c_int
    lib.dsa_li_topk.argtypes = [ctypes.POINTER(LiArgs), P]
    lib.dsa_li_topk.restype = ctypes.c_int
    lib.dsa_li_workspace_bytes.argtypes = [ctypes.POINTER(LiArgs)]
    lib.dsa_li_workspace_bytes.restype = ctypes.c_size_t
    for f in (lib.dsa_sfa_decode, lib.dsa_sfa_prefill, lib.dsa_sfa_decode_static):
        f.argtypes = [ctypes.POINTER(SfaArgs), P]
        f.restype = ctypes.c_int
    lib.dsa_sfa_workspace_bytes.argtypes = [ctypes.POINTER(SfaArgs)]
    lib.dsa_sfa_workspace_bytes.restype = ctypes.c_size_t
    lib.dsa_page_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.dsa_page_bytes.restype = ctypes.c_size_t
    lib.dsa_page_table_validate.argtypes = [P, ctypes.c_int, ctypes.c_int, P, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int]
    lib.dsa_page_table_validate.restype = ctypes.c_int
    lib.dsa_topk_merge.argtypes = [ctypes.POINTER(MergeArgs), P]
    lib.dsa_topk_merge.restype = ctypes.c_int
    lib.dsa_prolog_workspace_bytes.argtypes = [ctypes.POINTER(PrologArgs)]
    lib.dsa_prolog_workspace_bytes.restype = ctypes.c_size_t
    lib.dsa_indexer_prolog.argtypes = [ctypes.POINTER(PrologArgs), P]
    lib.dsa_indexer_prolog.restype = ctypes.c_int
    lib.dsa_cache_write.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    P, ctypes.c_int, ctypes.c_int, P, P, P, P, ctypes.c_int, P, P]
    lib.dsa_cache_write.restype = ctypes.c_int
    return lib


def status_string(code: int) -> str:
    return load().dsa_status_string(int(code)).decode()


def last_error() -> str:
    return load().dsa_last_error().decode()


def _check(code: int, where: str):
    if code != DSA_OK:
        raise DsaError(code, where, last_error())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the DSA library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _host_max(seq_lens: torch.Tensor, q_start: torch.Tensor, max_seq_len, max_q_per_seq):
    """The host-known bounds that size a launch.  Reading them from device tensors would be a
    hidden device-to-host synchronisation, so a caller with device tensors must pass them."""
    if max_seq_len is None:
        if seq_lens.is_cuda:
            raise ValueError("max_seq_len is required with device tensors (reading it back "
                             "would synchronise the stream)")
        max_seq_len = int(seq_lens.max())
    if max_q_per_seq is None:
        if q_start.is_cuda:
            raise ValueError("max_q_per_seq is required with device tensors (reading it back "
                             "would synchronise the stream)")
        max_q_per_seq = int((q_start[1:] - q_start[:-1]).max())
    return int(max_seq_len), int(max_q_per_seq)


def li_topk_args(q, w, k_pool, page_table, seq_lens, q_start, K, *, q_scale=None, k_scale=None,
                 max_seq_len=None, max_q_per_seq=None, out_idx=None, out_cnt=None, status=None,
                 q_sf=None, k_sf=None, out_score=None, workspace=None):
    """Fill the C argument struct of dsa_li_topk (tensors must outlive the call).  e4m3 q/k take
    either fp32 q_scale/k_scale (FP8) or uint8 E8M0 group scales q_sf/k_sf (MXFP8);
    ``workspace`` holds li_workspace_bytes() bytes when that is not 0."""
    fp8 = q.dtype == torch.float8_e4m3fn
    n_q, H_I, d_I = q.shape
    max_seq_len, max_q_per_seq = _host_max(seq_lens, q_start, max_seq_len, max_q_per_seq)
    a = LiArgs()
    a.B = seq_lens.shape[0]
    a.n_q, a.H_I, a.d_I, a.K = n_q, H_I, d_I, int(K)
    a.page_size = k_pool.shape[1]
    a.max_pages = page_table.shape[1]
    a.num_pages = k_pool.shape[0]
    a.max_seq_len, a.max_q_per_seq = max_seq_len, max_q_per_seq
    a.dtype = (DSA_MXFP8_E4M3 if q_sf is not None else DSA_FP8_E4M3) if fp8 else DSA_BF16
    a.q, a.q_scale, a.w, a.k_pool, a.k_scale = _ptr(q), _ptr(q_scale), _ptr(w), _ptr(k_pool), _ptr(k_scale)
    a.page_table, a.seq_lens, a.q_start = _ptr(page_table), _ptr(seq_lens), _ptr(q_start)
    a.out_idx, a.out_cnt, a.status = _ptr(out_idx), _ptr(out_cnt), _ptr(status)
    a.q_sf, a.k_sf = _ptr(q_sf), _ptr(k_sf)
    a.out_score = _ptr(out_score)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return a


def li_workspace_bytes(B: int, K: int, max_seq_len: int, max_q_per_seq: int) -> int:
    """Scratch bytes dsa_li_topk needs for a batch of this shape (0: none)."""
    a = LiArgs()
    a.B, a.K, a.max_seq_len, a.max_q_per_seq = int(B), int(K), int(max_seq_len), int(max_q_per_seq)
    return int(load().dsa_li_workspace_bytes(ctypes.byref(a)))


def li_topk(q, w, k_pool, page_table, seq_lens, q_start, K, *, q_scale=None, k_scale=None,
            max_seq_len=None, max_q_per_seq=None, out_idx=None, out_cnt=None, status=None,
            stream=None, q_sf=None, k_sf=None, out_score=None, workspace=None):
    """Fused indexer scoring + top-K.  Returns (idx [n_q, K] int32, cnt [n_q] int32); with
    ``out_score`` ([n_q, K] fp32) also the score of every selected position.  The scratch for
    sequences split into position units is allocated here unless ``workspace`` is given."""
    lib = load()
    n_q = q.shape[0]
    if out_idx is None:
        out_idx = torch.empty((n_q, K), dtype=torch.int32, device=q.device)
    if out_cnt is None:
        out_cnt = torch.empty((n_q,), dtype=torch.int32, device=q.device)
    max_seq_len, max_q_per_seq = _host_max(seq_lens, q_start, max_seq_len, max_q_per_seq)
    if workspace is None:
        nbytes = li_workspace_bytes(seq_lens.shape[0], K, max_seq_len, max_q_per_seq)
        if nbytes:
            workspace = torch.empty((nbytes,), dtype=torch.uint8, device=q.device)
    a = li_topk_args(q, w, k_pool, page_table, seq_lens, q_start, K, q_scale=q_scale,
                     k_scale=k_scale, max_seq_len=max_seq_len, max_q_per_seq=max_q_per_seq,
                     out_idx=out_idx, out_cnt=out_cnt, status=status, q_sf=q_sf, k_sf=k_sf,
                     out_score=out_score, workspace=workspace)
    _check(lib.dsa_li_topk(ctypes.byref(a), _stream(stream)), "dsa_li_topk")
    return out_idx, out_cnt


def sfa_args(q, kv_pool, page_table, seq_lens, q_start, idx, *, softmax_scale, max_seq_len=None,
             max_q_per_seq=None, out=None, lse=None, status=None, workspace=None, row_splits=0):
    n_q, H, d_qk = q.shape
    max_seq_len, max_q_per_seq = _host_max(seq_lens, q_start, max_seq_len, max_q_per_seq)
    a = SfaArgs()
    a.B = seq_lens.shape[0]
    a.n_q, a.H, a.d_qk, a.d_v, a.K = n_q, H, d_qk, 512, idx.shape[1]
    a.page_size, a.max_pages, a.num_pages = kv_pool.shape[1], page_table.shape[1], kv_pool.shape[0]
    a.max_seq_len, a.max_q_per_seq = max_seq_len, max_q_per_seq
    a.softmax_scale = float(softmax_scale)
    a.q, a.kv_pool, a.page_table, a.seq_lens, a.q_start = (_ptr(q), _ptr(kv_pool), _ptr(page_table),
                                                          _ptr(seq_lens), _ptr(q_start))
    a.idx, a.out, a.lse, a.status = _ptr(idx), _ptr(out), _ptr(lse), _ptr(status)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    # a uint8 pool holds FP8 rows (576 e4m3 codes + 5 fp32 tile scales + padding = 608 bytes)
    a.kv_dtype = DSA_FP8_E4M3 if kv_pool.dtype == torch.uint8 else DSA_BF16
    a.row_splits = int(row_splits)
    return a


def sfa_workspace_bytes(q, idx, row_splits=0) -> int:
    """Scratch bytes dsa_sfa_decode needs for a batch of this shape."""
    a = SfaArgs()
    a.n_q, a.H, a.K, a.d_qk, a.d_v = q.shape[0], q.shape[1], idx.shape[1], q.shape[2], 512
    a.row_splits = int(row_splits)
    return int(load().dsa_sfa_workspace_bytes(ctypes.byref(a)))


def new_workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    """A zeroed workspace buffer (the arrival counters inside it must start at zero)."""
    if nbytes == 0:
        return None
    return torch.zeros((nbytes,), dtype=torch.uint8, device=device)


def _sfa(entry, name, q, kv_pool, page_table, seq_lens, q_start, idx, *, softmax_scale,
         max_seq_len=None, max_q_per_seq=None, out=None, lse=None, status=None, workspace=None,
         stream=None, row_splits=0):
    lib = load()
    n_q, H, _ = q.shape
    if out is None:
        out = torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((n_q, H), dtype=torch.float32, device=q.device)
    if workspace is None and entry == "dsa_sfa_decode":
        workspace = new_workspace(sfa_workspace_bytes(q, idx, row_splits), q.device)
    a = sfa_args(q, kv_pool, page_table, seq_lens, q_start, idx, softmax_scale=softmax_scale,
                 max_seq_len=max_seq_len, max_q_per_seq=max_q_per_seq, out=out, lse=lse,
                 status=status, workspace=workspace, row_splits=row_splits)
    _check(getattr(lib, entry)(ctypes.byref(a), _stream(stream)), entry)
    return out, lse


def sfa_decode(q, kv_pool, page_table, seq_lens, q_start, idx, **kw):
    """Sparse attention for few tokens per sequence (row splits merged through a workspace)."""
    return _sfa("dsa_sfa_decode", "sfa_decode", q, kv_pool, page_table, seq_lens, q_start, idx, **kw)


def sfa_decode_static(q, kv_pool, page_table, seq_lens, q_start, idx, *, softmax_scale,
                      max_seq_len=None, max_q_per_seq=None, out=None, lse=None, status=None,
                      stream=None, row_splits=0):
    """sfa_decode for callers that cannot allocate: the split-merge scratch is the library's own
    fixed device array (SFA_STATIC_SCRATCH_BYTES, shared by every call on the device, so calls
    must not overlap on the GPU).  Only the outputs are allocated here, and only when not given."""
    lib = load()
    n_q, H, _ = q.shape
    if out is None:
        out = torch.empty((n_q, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((n_q, H), dtype=torch.float32, device=q.device)
    a = sfa_args(q, kv_pool, page_table, seq_lens, q_start, idx, softmax_scale=softmax_scale,
                 max_seq_len=max_seq_len, max_q_per_seq=max_q_per_seq, out=out, lse=lse,
                 status=status, workspace=None, row_splits=row_splits)
    _check(lib.dsa_sfa_decode_static(ctypes.byref(a), _stream(stream)), "dsa_sfa_decode_static")
    return out, lse


def sfa_prefill(q, kv_pool, page_table, seq_lens, q_start, idx, **kw):
    """Sparse attention for many tokens per sequence (no workspace)."""
    return _sfa("dsa_sfa_prefill", "sfa_prefill", q, kv_pool, page_table, seq_lens, q_start, idx, **kw)


def page_bytes(dtype: int, rows: int, dim: int) -> int:
    return int(load().dsa_page_bytes(int(dtype), int(rows), int(dim)))


def page_table_validate(page_table: torch.Tensor, seq_lens: torch.Tensor, page_size: int,
                        num_pages: int, require_unique: bool = False) -> None:
    """Host-side page-table check; raises DsaError with the reason on failure."""
    pt = page_table.detach().to("cpu", torch.int32).contiguous()
    sl = seq_lens.detach().to("cpu", torch.int32).contiguous()
    code = load().dsa_page_table_validate(_ptr(pt), pt.shape[0], pt.shape[1], _ptr(sl),
                                          int(page_size), int(num_pages), int(require_unique))
    _check(code, "dsa_page_table_validate")


def cache_write(pool, page_table, seq, pos, rows, *, scale_pool=None, row_scales=None,
                status=None, stream=None) -> None:
    """Scatter rows [n, dim] into pool [num_pages, page_size, dim] at (seq[i], pos[i])."""
    lib = load()
    num_pages, page_size, dim = pool.shape
    code = lib.dsa_cache_write(_ptr(pool), _ptr(scale_pool), num_pages, page_size, dim,
                               pool.element_size(), _ptr(page_table), page_table.shape[1],
                               page_table.shape[0], _ptr(seq), _ptr(pos), _ptr(rows),
                               _ptr(row_scales), rows.shape[0], _ptr(status), _stream(stream))
    _check(code, "dsa_cache_write")


def topk_merge(cand_idx, cand_score, shard_offset, K, *, out_idx=None, out_cnt=None, stream=None):
    """Merge S shards' candidates ([S, n_q, K_in] shard-local positions and scores; position +
    shard_offset[s] is the sequence position) into the top-K by (score desc, position asc),
    ascending positions with -1 padding.  Returns (idx [n_q, K], cnt [n_q])."""
    lib = load()
    S, n_q, K_in = cand_idx.shape
    dev = cand_idx.device
    if out_idx is None:
        out_idx = torch.empty((n_q, K), dtype=torch.int32, device=dev)
    if out_cnt is None:
        out_cnt = torch.empty((n_q,), dtype=torch.int32, device=dev)
    a = MergeArgs()
    a.S, a.n_q, a.K_in, a.K = S, n_q, K_in, int(K)
    a.cand_idx, a.cand_score, a.shard_offset = _ptr(cand_idx), _ptr(cand_score), _ptr(shard_offset)
    a.out_idx, a.out_cnt = _ptr(out_idx), _ptr(out_cnt)
    _check(lib.dsa_topk_merge(ctypes.byref(a), _stream(stream)), "dsa_topk_merge")
    return out_idx, out_cnt


def prolog_args(inp: dict, *, q_out, q_sf, w_out, workspace=None, status=None):
    """Fill the C argument struct of dsa_indexer_prolog from a ``dsa_inputs.generate_prolog``
    dict (device tensors; the key cache in it is written in place)."""
    wl = inp["wl"]
    a = PrologArgs()
    a.n_q, a.B, a.d_q, a.d_model = inp["xq"].shape[0], inp["seq_lens"].shape[0], \
        inp["xq"].shape[1], inp["x"].shape[1]
    a.H_I, a.d_I = inp["w_w"].shape[0], inp["w_k"].shape[0]
    a.dtype = DSA_MXFP8_E4M3 if inp.get("k_sf") is not None else DSA_BF16
    a.page_size, a.max_pages, a.num_pages = inp["k_pool"].shape[1], inp["pt_k"].shape[1], \
        inp["k_pool"].shape[0]
    a.ln_eps, a.w_scale = float(inp["ln_eps"]), float(inp["w_scale"])
    for k in ("xq", "x", "w_q", "w_k", "w_w", "ln_gamma", "ln_beta", "seq_lens", "q_start",
              "k_pool", "k_sf"):
        setattr(a, k, _ptr(inp.get(k)))
    a.page_table = _ptr(inp["pt_k"])
    a.q_out, a.q_sf, a.w_out = _ptr(q_out), _ptr(q_sf), _ptr(w_out)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.status = _ptr(status)
    del wl
    return a


def prolog_workspace_bytes(inp: dict) -> int:
    a = prolog_args(inp, q_out=None, q_sf=None, w_out=None)
    return int(load().dsa_prolog_workspace_bytes(ctypes.byref(a)))


def indexer_prolog(inp: dict, *, q_out=None, q_sf=None, w_out=None, workspace=None, status=None,
                   stream=None):
    """Indexer Prolog of the new tokens: returns (q, q_sf or None, w) and writes the new keys into
    inp["k_pool"] (and inp["k_sf"]).  ``workspace``: optional; prolog_workspace_bytes(inp) is 0
    (the input slices of a tile meet in distributed shared memory)."""
    lib = load()
    n_q, H_I, d_I = inp["xq"].shape[0], inp["w_w"].shape[0], inp["w_k"].shape[0]
    dev = inp["xq"].device
    mx = inp.get("k_sf") is not None
    if q_out is None:
        q_out = torch.empty((n_q, H_I, d_I), dtype=torch.float8_e4m3fn if mx else torch.bfloat16,
                            device=dev)
    if q_sf is None and mx:
        q_sf = torch.empty((n_q, H_I, d_I // 32), dtype=torch.uint8, device=dev)
    if w_out is None:
        w_out = torch.empty((n_q, H_I), dtype=torch.float32, device=dev)
    nb = prolog_workspace_bytes(inp)
    if workspace is None and nb:
        workspace = torch.zeros(nb, dtype=torch.uint8, device=dev)
    a = prolog_args(inp, q_out=q_out, q_sf=q_sf, w_out=w_out, workspace=workspace, status=status)
    _check(lib.dsa_indexer_prolog(ctypes.byref(a), _stream(stream)), "dsa_indexer_prolog")
    return q_out, q_sf, w_out


def decode_step(inp: dict, *, idx=None, cnt=None, out=None, lse=None, workspace=None, status=None,
                stream=None, max_seq_len=None, max_q_per_seq=None, prefill: bool = False,
                row_splits: int = 0, li_workspace=None):
    """One pass of the whole hot path over a batch laid out as ``dsa_inputs.generate`` does:
    li_topk followed by sfa_decode (or sfa_prefill) on the same stream."""
    wl = inp["wl"]
    ms = max_seq_len if max_seq_len is not None else max(wl.seq_lens)
    mq = max_q_per_seq if max_q_per_seq is not None else max(wl.n_new)
    idx, cnt = li_topk(inp["q_li"], inp["w"], inp["k_pool"], inp["pt_k"], inp["seq_lens"],
                       inp["q_start"], wl.K, q_scale=inp.get("q_scale"), k_scale=inp.get("k_scale"),
                       max_seq_len=ms, max_q_per_seq=mq, out_idx=idx, out_cnt=cnt, status=status,
                       stream=stream, q_sf=inp.get("q_sf"), k_sf=inp.get("k_sf"),
                       workspace=li_workspace)
    f = sfa_prefill if prefill else sfa_decode
    kv = inp["kv8_pool"] if getattr(wl, "kv_dtype", "bf16") == "fp8" else inp["kv_pool"]
    out, lse = f(inp["q_sfa"], kv, inp["pt_kv"], inp["seq_lens"], inp["q_start"], idx,
                 softmax_scale=inp["softmax_scale"], max_seq_len=ms, max_q_per_seq=mq, out=out,
                 lse=lse, status=status, workspace=workspace, stream=stream,
                 row_splits=row_splits)
    return idx, cnt, out, lse
