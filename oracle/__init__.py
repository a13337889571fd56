"""CPU oracle of the DSA hot path (Lightning Indexer top-K + Sparse Flash Attention), fp64.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. It shares no code with the CUDA library; it reads the same input
tensors (CPU, contiguous) and nothing else.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64). This wrapper only marshals arguments.
Functions:
  li_scores(inp, t)          -> (s[0..p], mag[0..p]) float64 for query token t
  li_topk(inp, tokens)       -> (idx [n, K] int32, cnt [n] int32, kth [n] float64)
  sfa(inp, idx, tokens)      -> (out [n, H, d_v] float64, lse [n, H] float64)
  prolog(inp)                -> Indexer Prolog outputs (projections, LayerNorm, quantisation)
  mx_quantize(v)             -> OCP MX e4m3 codes and E8M0 scale bytes of a vector
  decode_kv8(row, d)         -> element d of one FP8 latent-cache row (608 bytes)
``inp`` is the dict produced by ``dsa_inputs.generate`` (tensors moved to the CPU on demand).
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build

_lib = None


class _Li(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "n_q", "H_I", "d_I", "K", "page_size", "max_pages", "num_pages", "fp8")] + [
        ("q", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("k_pool", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("q_start", ctypes.c_void_p), ("q_sf", ctypes.c_void_p), ("k_sf", ctypes.c_void_p)]


class _Sfa(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "n_q", "H", "d_qk", "d_v", "K", "page_size", "max_pages", "num_pages")] + [
        ("scale", ctypes.c_double), ("q", ctypes.c_void_p), ("kv_pool", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("q_start", ctypes.c_void_p), ("kv_fp8", ctypes.c_int), ("kv8_pool", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        _lib.oracle_li_scores.argtypes = [P, ctypes.c_int, P, P]
        _lib.oracle_li_topk.argtypes = [P, ctypes.c_int, P, P, P, P]
        _lib.oracle_sfa.argtypes = [P, ctypes.c_int, P, P, P, P]
    return _lib


def _cpu(t):
    if t is None:
        return None
    return t.detach().to("cpu").contiguous()


class _Keep:
    """Holds CPU copies alive while a C call runs."""

    def __init__(self):
        self.items = []

    def ptr(self, t):
        if t is None:
            return None
        t = _cpu(t)
        self.items.append(t)
        return ctypes.c_void_p(t.data_ptr())


def _li_struct(inp, keep):
    wl = inp["wl"]
    s = _Li()
    s.B, s.n_q, s.H_I, s.d_I, s.K = wl.B, wl.n_q, wl.H_I, wl.d_I, wl.K
    s.page_size, s.max_pages = wl.page_size, int(inp["pt_k"].shape[1])
    s.num_pages = int(inp["k_pool"].shape[0])
    s.fp8 = {"bf16": 0, "fp8": 1, "mxfp8": 2}[wl.li_dtype]
    s.q = keep.ptr(inp["q_li"])
    s.q_scale = keep.ptr(inp.get("q_scale"))
    s.w = keep.ptr(inp["w"])
    s.k_pool = keep.ptr(inp["k_pool"])
    s.k_scale = keep.ptr(inp.get("k_scale"))
    s.page_table = keep.ptr(inp["pt_k"])
    s.seq_lens = keep.ptr(inp["seq_lens"])
    s.q_start = keep.ptr(inp["q_start"])
    s.q_sf = keep.ptr(inp.get("q_sf"))
    s.k_sf = keep.ptr(inp.get("k_sf"))
    return s


def _sfa_struct(inp, K, keep):
    wl = inp["wl"]
    s = _Sfa()
    s.B, s.n_q, s.H, s.d_qk, s.d_v, s.K = wl.B, wl.n_q, wl.H, wl.d_qk, wl.d_v, K
    s.page_size, s.max_pages = wl.page_size, int(inp["pt_kv"].shape[1])
    s.num_pages = int(inp["kv_pool"].shape[0])
    s.scale = float(inp["softmax_scale"])
    s.q = keep.ptr(inp["q_sfa"])
    s.kv_pool = keep.ptr(inp["kv_pool"])
    s.page_table = keep.ptr(inp["pt_kv"])
    s.seq_lens = keep.ptr(inp["seq_lens"])
    s.q_start = keep.ptr(inp["q_start"])
    s.kv_fp8 = 1 if getattr(wl, "kv_dtype", "bf16") == "fp8" else 0
    s.kv8_pool = keep.ptr(inp.get("kv8_pool"))
    return s


def _tokens(inp, tokens):
    if tokens is None:
        tokens = range(inp["wl"].n_q)
    return torch.tensor(list(tokens), dtype=torch.int32)


def li_scores(inp, t):
    keep = _Keep()
    s = _li_struct(inp, keep)
    L = int(inp["seq_lens"].max())
    sc = np.zeros(L, dtype=np.float64)
    mag = np.zeros(L, dtype=np.float64)
    n = lib().oracle_li_scores(ctypes.byref(s), int(t), sc.ctypes.data, mag.ctypes.data)
    if n < 0:
        raise ValueError("oracle_li_scores failed: %d" % n)
    return sc[:n], mag[:n]


def li_topk(inp, tokens=None):
    keep = _Keep()
    s = _li_struct(inp, keep)
    toks = _tokens(inp, tokens)
    K = inp["wl"].K
    idx = np.zeros((len(toks), K), dtype=np.int32)
    cnt = np.zeros(len(toks), dtype=np.int32)
    kth = np.zeros(len(toks), dtype=np.float64)
    rc = lib().oracle_li_topk(ctypes.byref(s), len(toks), toks.data_ptr(), idx.ctypes.data,
                              cnt.ctypes.data, kth.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_li_topk failed: %d" % rc)
    return idx, cnt, kth


def sfa(inp, idx, tokens=None):
    keep = _Keep()
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    K = idx.shape[1]
    s = _sfa_struct(inp, K, keep)
    toks = _tokens(inp, tokens)
    assert idx.shape[0] == len(toks)
    wl = inp["wl"]
    out = np.zeros((len(toks), wl.H, wl.d_v), dtype=np.float64)
    lse = np.zeros((len(toks), wl.H), dtype=np.float64)
    rc = lib().oracle_sfa(ctypes.byref(s), len(toks), toks.data_ptr(), idx.ctypes.data,
                          out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_sfa failed: %d" % rc)
    return out, lse


class _Prolog(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_q", "B", "d_q", "d_model", "H_I", "d_I", "mx")] + [
        (n, ctypes.c_void_p) for n in ("xq", "x", "w_q", "w_k", "w_w", "ln_gamma", "ln_beta")] + [
        ("ln_eps", ctypes.c_double), ("w_scale", ctypes.c_double), ("page_table", ctypes.c_void_p),
        ("max_pages", ctypes.c_int), ("page_size", ctypes.c_int), ("seq_lens", ctypes.c_void_p),
        ("q_start", ctypes.c_void_p)]


def prolog(inp):
    """Indexer Prolog of every new token (``inp`` from ``dsa_inputs.generate_prolog``).  Returns
    q_val [n_q, H_I*d_I], k_val [n_q, d_I] (fp64 before rounding), w [n_q, H_I], the encoded q
    (uint8 e4m3 codes or uint16 bf16 bits) with q_sf, the encoded k with k_sf, and k_row [n_q]."""
    wl = inp["wl"]
    keep = _Keep()
    s = _Prolog()
    s.n_q, s.B, s.d_q, s.d_model, s.H_I, s.d_I = wl.n_q, wl.B, wl.d_q, wl.d_model, wl.H_I, wl.d_I
    mx = wl.li_dtype == "mxfp8"
    s.mx = 1 if mx else 0
    for k in ("xq", "x", "w_q", "w_k", "w_w", "ln_gamma", "ln_beta"):
        setattr(s, k, keep.ptr(inp[k]))
    s.ln_eps, s.w_scale = float(inp["ln_eps"]), float(inp["w_scale"])
    s.page_table = keep.ptr(inp["pt_k"])
    s.max_pages, s.page_size = int(inp["pt_k"].shape[1]), wl.page_size
    s.seq_lens, s.q_start = keep.ptr(inp["seq_lens"]), keep.ptr(inp["q_start"])
    n, F, D = wl.n_q, wl.H_I * wl.d_I, wl.d_I
    r = {"q_val": np.zeros((n, F)), "k_val": np.zeros((n, D)), "w": np.zeros((n, wl.H_I)),
         "q_enc": np.zeros((n, F), dtype=np.uint8 if mx else np.uint16),
         "k_enc": np.zeros((n, D), dtype=np.uint8 if mx else np.uint16),
         "q_sf": np.zeros((n, F // 32), dtype=np.uint8), "k_sf": np.zeros((n, D // 32), dtype=np.uint8),
         "k_row": np.zeros(n, dtype=np.int64)}
    f = lib().oracle_prolog
    f.argtypes = [ctypes.c_void_p] * 9
    rc = f(ctypes.byref(s), *(ctypes.c_void_p(r[k].ctypes.data) for k in
                              ("q_val", "k_val", "w", "q_enc", "q_sf", "k_enc", "k_sf", "k_row")))
    if rc != 0:
        raise ValueError("oracle_prolog failed: %d" % rc)
    return r


def mx_quantize(v):
    """OCP MX quantisation of a float64 vector (length a multiple of 32): (codes, scale bytes)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    codes = np.zeros(v.shape[0], dtype=np.uint8)
    sf = np.zeros(v.shape[0] // 32, dtype=np.uint8)
    f = lib().oracle_mx_quantize
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    rc = f(v.ctypes.data, v.shape[0], codes.ctypes.data, sf.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_mx_quantize failed: %d" % rc)
    return codes, sf


def decode_bf16(bits: int) -> float:
    f = lib().orc_bf16
    f.argtypes = [ctypes.c_uint16]
    f.restype = ctypes.c_double
    return f(bits)


def decode_kv8(row, d: int) -> float:
    """Element d of one FP8 latent-cache row (608 bytes: 576 e4m3 codes, 5 fp32 tile scales)."""
    row = np.ascontiguousarray(np.asarray(row, dtype=np.uint8))
    assert row.shape == (608,)
    f = lib().orc_kv8_element
    f.argtypes = [ctypes.c_void_p, ctypes.c_int]
    f.restype = ctypes.c_double
    return f(row.ctypes.data, d)


def decode_e8m0(bits: int) -> float:
    f = lib().orc_e8m0
    f.argtypes = [ctypes.c_uint8]
    f.restype = ctypes.c_double
    return f(bits)


def decode_e4m3(bits: int) -> float:
    f = lib().orc_e4m3
    f.argtypes = [ctypes.c_uint8]
    f.restype = ctypes.c_double
    return f(bits)
