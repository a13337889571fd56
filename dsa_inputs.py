"""Seeded synthetic inputs for the DSA hot path (Lightning Indexer top-K + Sparse Flash Attention).

This module draws random tensors, builds random page tables and lays the values out in paged
caches. It contains none of the method's arithmetic (no scoring, no selection, no attention):
the same bytes it produces are consumed by the CPU oracle (``oracle/``) and by the CUDA library
(``dsa_sparse_attention_li_gb300``), and neither of those imports the other.

Layouts (all row-major, C order):

* ``q_li``     [n_q, H_I, d_I]  bf16, or float8_e4m3fn for the quantised indexer paths
* ``q_scale``  [n_q, H_I]       fp32 (fp8 only; one scale per query token, replicated over heads)
* ``q_sf``     [n_q, H_I, d_I/32] uint8 E8M0 block scales (mxfp8 only: one per 32 elements)
* ``w``        [n_q, H_I]       fp32 index-head weights
* ``k_pool``   [pages_k, 64, d_I]  paged index-key cache (bf16 or e4m3)
* ``k_scale``  [pages_k, 64]    fp32 per-row key scale (fp8 only)
* ``k_sf``     [pages_k, 64, d_I/32] uint8 E8M0 block scales of the key rows (mxfp8 only)
* ``pt_k``     [B, max_pages]   int32 page table of the key cache
* ``q_sfa``    [n_q, H, 576]    bf16 attention queries (512 latent + 64 rope)
* ``kv_pool``  [pages_kv, 64, 576] bf16 paged MLA latent cache; the value is its first 512 columns
* ``kv8_pool`` [pages_kv, 64, 608] uint8 FP8 latent cache (kv_dtype "fp8"): per row 576 e4m3
               codes, then one fp32 scale per 128-column tile (5; the last tile is the 64 rope
               columns), then 12 zero bytes
* ``pt_kv``    [B, max_pages]   int32 page table of the latent cache
* ``seq_lens`` [B] int32 positions per sequence, new tokens included
* ``q_start``  [B+1] int32 prefix offsets of each sequence's query tokens

Logical position ``j`` of sequence ``b`` lives at physical row ``pt[b][j // 64] * 64 + j % 64``.
Rows of a partially filled last page that lie past ``seq_lens[b]`` are filled with values four
times larger than the real ones, so that a missing length mask shows up as a wrong selection.
Unused page-table entries hold 0 (a valid page), never an out-of-range id.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

PAGE = 64
D_QK = 576
D_V = 512
FP8_MAX = 448.0


@dataclass
class Workload:
    name: str
    seq_lens: List[int]
    n_new: List[int]
    H_I: int
    d_I: int
    K: int
    H: int
    li_dtype: str = "bf16"          # "bf16" | "fp8" | "mxfp8"
    values: str = "normal"          # "normal" (N(0,1)) | "int4" (integers uniform in [-4, 4])
    w_values: str = "normal"        # "normal" (N(0,1)/sqrt(H_I)) | "int14" (integers in [1, 4])
    seed: int = 0
    d_qk: int = D_QK
    d_v: int = D_V
    page_size: int = PAGE
    softmax_scale: float = field(default=1.0 / math.sqrt(D_QK))
    d_q: int = 1536                 # Indexer Prolog: input width of the Q projection
    d_model: int = 7168             # Indexer Prolog: input width of the K / head-weight projections
    kv_dtype: str = "bf16"          # latent cache: "bf16" | "fp8" (per-token, 128-column tiles)

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def n_q(self) -> int:
        return sum(self.n_new)

    def pages(self) -> List[int]:
        return [(L + self.page_size - 1) // self.page_size for L in self.seq_lens]

    @property
    def max_pages(self) -> int:
        return max(self.pages())

    @property
    def num_pages(self) -> int:
        return sum(self.pages())

    def describe(self) -> dict:
        return {
            "workload": self.name, "B": self.B, "n_q": self.n_q, "H_I": self.H_I, "d_I": self.d_I,
            "K": self.K, "H": self.H, "d_qk": self.d_qk, "d_v": self.d_v, "page": self.page_size,
            "li_dtype": self.li_dtype, "kv_dtype": self.kv_dtype, "values": self.values,
            "seq_len_min": min(self.seq_lens), "seq_len_max": max(self.seq_lens),
            "positions": sum(self.seq_lens), "seed": self.seed,
        }


def _log_uniform_lengths(B: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(B, generator=g, dtype=torch.float64)
    lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return [int(min(max(v, lo), hi)) for v in lens.tolist()]


def preset(name: str) -> Workload:
    """The five synthetic workloads of the method's decode / speculative / prefill regimes.

    decode_int_4k   : 1 sequence, 1 token, L=4096, 8x64 index heads, K=256, 16 SFA heads,
                      integer-valued bf16 inputs (scores exact in fp32)
    decode_32k      : 32 sequences x 1 token, L=32768, 64x128 index heads, K=2048, 128 heads
    decode_32k_fp8  : decode_32k with e4m3 index q/k and per-token fp32 scales
    decode_32k_mxfp8: decode_32k with MXFP8 index q/k (e4m3 elements, one E8M0 scale per 32)
    decode_32k_kv8  : decode_32k with the FP8 latent cache (per-token 128-column tile scales)
    prolog_decode_32k: the Indexer Prolog of decode_32k_mxfp8's 32 new tokens (Q projection from
                      a 1536-wide query input, K and head weights from a 7168-wide hidden state)
    specdec_ragged  : 64 sequences x 2 tokens (verified + draft), L log-uniform in [1024, 131072]
    prefill_64k     : 1 sequence, 4096 new tokens appended to a 61440-token prefix
    """
    if name == "decode_int_4k":
        return Workload(name, [4096], [1], H_I=8, d_I=64, K=256, H=16, values="int4",
                        w_values="int14", seed=1001)
    if name == "decode_32k":
        return Workload(name, [32768] * 32, [1] * 32, H_I=64, d_I=128, K=2048, H=128, seed=1002)
    if name == "decode_32k_fp8":
        return Workload(name, [32768] * 32, [1] * 32, H_I=64, d_I=128, K=2048, H=128,
                        li_dtype="fp8", seed=1003)
    if name == "decode_32k_mxfp8":
        return Workload(name, [32768] * 32, [1] * 32, H_I=64, d_I=128, K=2048, H=128,
                        li_dtype="mxfp8", seed=1006)
    if name == "prolog_decode_32k":
        return Workload(name, [32768] * 32, [1] * 32, H_I=64, d_I=128, K=2048, H=128,
                        li_dtype="mxfp8", seed=1007)
    if name == "decode_32k_kv8":
        return Workload(name, [32768] * 32, [1] * 32, H_I=64, d_I=128, K=2048, H=128,
                        kv_dtype="fp8", seed=1008)
    if name == "specdec_ragged":
        lens = _log_uniform_lengths(64, 1024, 131072, seed=1004)
        return Workload(name, lens, [2] * 64, H_I=64, d_I=128, K=2048, H=128, seed=1004)
    if name == "prefill_64k":
        return Workload(name, [65536], [4096], H_I=64, d_I=128, K=2048, H=128, seed=1005)
    raise KeyError(name)


PRESETS = ["decode_int_4k", "decode_32k", "decode_32k_fp8", "decode_32k_mxfp8", "decode_32k_kv8",
           "specdec_ragged", "prefill_64k"]


def small(name: str, **over) -> Workload:
    """A reduced copy of a preset with the same heads/dims/value recipe, for quick parity runs."""
    wl = preset(name)
    return replace(wl, name=name + "_small", **over)


# --------------------------------------------------------------------------------------------
# drawing
# --------------------------------------------------------------------------------------------

def _draw(shape, kind: str, g: torch.Generator, device) -> torch.Tensor:
    if kind == "int4":
        return torch.randint(-4, 5, shape, generator=g, device=device).to(torch.float32)
    if kind == "normal":
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    raise ValueError(kind)


def _quant_e4m3(x: torch.Tensor, dim: int):
    """Per-slice symmetric e4m3 quantisation: scale = amax/448 (1 if amax == 0), RNE, clamped."""
    amax = x.abs().amax(dim=dim, keepdim=True)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    q = (x / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q, scale.squeeze(dim).to(torch.float32)


MX_GROUP = 32
E4M3_EMAX = 8  # exponent of the largest normal e4m3 value (448 = 1.75 * 2^8)


def _quant_mx(x: torch.Tensor):
    """MX quantisation of the last dimension in groups of 32 (OCP Microscaling Formats v1.0):
    shared scale X = 2^(floor(log2(amax)) - 8) stored as an E8M0 byte (exponent + 127; 127 when
    amax == 0), elements x / X rounded to nearest-even e4m3 and clamped to +-448."""
    shape = x.shape
    g = x.reshape(*shape[:-1], shape[-1] // MX_GROUP, MX_GROUP)
    amax = g.abs().amax(dim=-1, keepdim=True)
    _, e = torch.frexp(amax)                     # amax = m * 2^e, m in [0.5, 1)
    shared = torch.where(amax > 0, e - 1 - E4M3_EMAX, torch.zeros_like(e)).clamp(-127, 127)
    q = (g / torch.ldexp(torch.ones_like(amax), shared)).clamp(-FP8_MAX, FP8_MAX)
    q = q.to(torch.float8_e4m3fn).reshape(shape)
    return q, (shared.squeeze(-1) + 127).to(torch.uint8)


def _int_mx(x: torch.Tensor, g: torch.Generator):
    """Integer-valued elements (exact in e4m3) with E8M0 scales drawn from {2^-1, 2^0, 2^1}."""
    sf = torch.randint(126, 129, (*x.shape[:-1], x.shape[-1] // MX_GROUP), generator=g,
                       device=x.device).to(torch.uint8)
    return x.to(torch.float8_e4m3fn), sf


KV8_ROW = 608
KV8_TILE = 128


def _quant_kv8(rows: torch.Tensor) -> torch.Tensor:
    """FP8 latent-cache rows from fp32 rows [N, 576]: per row and 128-column tile, scale =
    amax/448 (1 when amax == 0), codes = e4m3(x / scale) (nearest even, clamped); packed as 576
    code bytes, 5 fp32 scales, 12 zero bytes."""
    n, d = rows.shape
    out = torch.zeros((n, KV8_ROW), dtype=torch.uint8, device=rows.device)
    for i, c0 in enumerate(range(0, d, KV8_TILE)):
        tile = rows[:, c0:c0 + KV8_TILE]
        amax = tile.abs().amax(1, keepdim=True)
        scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
        codes = (tile / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
        out[:, c0:c0 + tile.shape[1]] = codes.view(torch.uint8)
        out[:, d + 4 * i:d + 4 * i + 4] = scale.to(torch.float32).view(torch.uint8).view(n, 4)
    return out


def _page_table(pages: List[int], max_pages: int, g: torch.Generator) -> torch.Tensor:
    total = sum(pages)
    perm = torch.randperm(total, generator=g).to(torch.int32)
    pt = torch.zeros((len(pages), max_pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt


def _paged_fill(wl: Workload, pt: torch.Tensor, dim: int, kind: str, g: torch.Generator,
                device, chunk_rows: int = 1 << 22) -> torch.Tensor:
    """Random rows for every logical position, scattered into pages through ``pt``.

    Rows past a sequence's length inside its last page are drawn 4x larger (poison)."""
    P = wl.page_size
    pool = torch.empty((wl.num_pages * P, dim), dtype=torch.float32, device=device)
    # draw the whole pool in order of physical rows, then scale the poison rows
    r = 0
    while r < pool.shape[0]:
        n = min(chunk_rows, pool.shape[0] - r)
        pool[r:r + n] = _draw((n, dim), kind, g, device)
        r += n
    poison = []
    for b, L in enumerate(wl.seq_lens):
        if L % P:
            page = int(pt[b, (L - 1) // P])
            poison.append(torch.arange(page * P + L % P, page * P + P))
    if poison:
        rows = torch.cat(poison).to(device)
        pool[rows] *= 4.0
    return pool.view(wl.num_pages, P, dim)


def generate(wl: Workload, device="cpu") -> dict:
    """All inputs of one workload, seeded by ``wl.seed``; bulk values drawn on ``device``.

    Structure (page tables, lengths) always comes from a CPU generator, so it does not depend on
    the device; the values come from a generator on ``device``."""
    device = torch.device(device)
    gs = torch.Generator().manual_seed(wl.seed)
    gv = torch.Generator(device=device).manual_seed(wl.seed + 7919)
    pages = wl.pages()
    pt_k = _page_table(pages, wl.max_pages, gs)
    pt_kv = _page_table(pages, wl.max_pages, gs)
    n_q = wl.n_q
    out = {"wl": wl}

    # index queries, head weights and the key cache
    q = _draw((n_q, wl.H_I, wl.d_I), wl.values, gv, device)
    k = _paged_fill(wl, pt_k, wl.d_I, wl.values, gv, device)
    if wl.w_values == "int14":
        w = torch.randint(1, 5, (n_q, wl.H_I), generator=gv, device=device).to(torch.float32)
    else:
        w = torch.randn((n_q, wl.H_I), generator=gv, device=device) / math.sqrt(wl.H_I)
    if wl.li_dtype == "mxfp8":
        gm = torch.Generator(device=device).manual_seed(wl.seed + 104729)
        quant = (lambda x: _int_mx(x, gm)) if wl.values == "int4" else _quant_mx
        q8, qsf = quant(q)
        k8, ksf = quant(k)
        out["q_li"], out["q_sf"] = q8.contiguous(), qsf.contiguous()
        out["k_pool"], out["k_sf"] = k8.contiguous(), ksf.contiguous()
        out["q_scale"] = None
        out["k_scale"] = None
    elif wl.li_dtype == "fp8":
        q8, qs = _quant_e4m3(q.reshape(n_q, -1), dim=1)
        out["q_li"] = q8.view(n_q, wl.H_I, wl.d_I)
        out["q_scale"] = qs[:, None].expand(n_q, wl.H_I).contiguous()
        k8, ks = _quant_e4m3(k.reshape(-1, wl.d_I), dim=1)
        out["k_pool"] = k8.view(wl.num_pages, wl.page_size, wl.d_I)
        out["k_scale"] = ks.view(wl.num_pages, wl.page_size).contiguous()
    else:
        out["q_li"] = q.to(torch.bfloat16)
        out["k_pool"] = k.to(torch.bfloat16)
        out["q_scale"] = None
        out["k_scale"] = None
    out["w"] = w.contiguous()
    del q, k

    # attention queries and the latent cache
    out["q_sfa"] = _draw((n_q, wl.H, wl.d_qk), wl.values, gv, device).to(torch.bfloat16)
    kv = _paged_fill(wl, pt_kv, wl.d_qk, wl.values, gv, device)
    out["kv_pool"] = kv.to(torch.bfloat16)
    if wl.kv_dtype == "fp8":
        out["kv8_pool"] = _quant_kv8(kv.view(-1, wl.d_qk)).view(wl.num_pages, wl.page_size, KV8_ROW)
    del kv

    out["pt_k"] = pt_k.to(device)
    out["pt_kv"] = pt_kv.to(device)
    out["seq_lens"] = torch.tensor(wl.seq_lens, dtype=torch.int32, device=device)
    qs_ = [0]
    for n in wl.n_new:
        qs_.append(qs_[-1] + n)
    out["q_start"] = torch.tensor(qs_, dtype=torch.int32, device=device)
    out["softmax_scale"] = wl.softmax_scale
    return out


def redraw_queries(inp: dict, seed: int) -> dict:
    """The same caches and page tables with freshly drawn query-side inputs (indexer queries
    with their scales, head weights, attention queries), from ``seed``, by the recipes of
    ``generate``: another decode step over the same context.  The benchmark rotates several
    such sets so that every step selects, and gathers, other latent rows."""
    wl = inp["wl"]
    device = inp["q_sfa"].device
    gv = torch.Generator(device=device).manual_seed(seed)
    n_q = wl.n_q
    out = dict(inp)
    q = _draw((n_q, wl.H_I, wl.d_I), wl.values, gv, device)
    if wl.w_values == "int14":
        w = torch.randint(1, 5, (n_q, wl.H_I), generator=gv, device=device).to(torch.float32)
    else:
        w = torch.randn((n_q, wl.H_I), generator=gv, device=device) / math.sqrt(wl.H_I)
    if wl.li_dtype == "mxfp8":
        gm = torch.Generator(device=device).manual_seed(seed + 104729)
        quant = (lambda x: _int_mx(x, gm)) if wl.values == "int4" else _quant_mx
        q8, qsf = quant(q)
        out["q_li"], out["q_sf"] = q8.contiguous(), qsf.contiguous()
    elif wl.li_dtype == "fp8":
        q8, qs = _quant_e4m3(q.reshape(n_q, -1), dim=1)
        out["q_li"] = q8.view(n_q, wl.H_I, wl.d_I)
        out["q_scale"] = qs[:, None].expand(n_q, wl.H_I).contiguous()
    else:
        out["q_li"] = q.to(torch.bfloat16)
    out["w"] = w.contiguous()
    out["q_sfa"] = _draw((n_q, wl.H, wl.d_qk), wl.values, gv, device).to(torch.bfloat16)
    return out


def generate_prolog(wl: Workload, device="cpu") -> dict:
    """Inputs of the Indexer Prolog for the new tokens of ``wl``: activations, random projection
    weights (the model's weights are not available; the prolog's arithmetic does not depend on
    their values), LayerNorm parameters, and a key cache (random contents) with its page table,
    into which the prolog writes the new tokens' keys.

    values "normal": x ~ N(0, 1), weights ~ N(0, 1/fan_in), gamma ~ 1 + N(0, 0.1^2),
    beta ~ N(0, 0.1^2).  values "int4": x and weights integers in [-2, 2], gamma 1, beta 0 (every
    projection is then exact in fp32)."""
    device = torch.device(device)
    gs = torch.Generator().manual_seed(wl.seed)
    gv = torch.Generator(device=device).manual_seed(wl.seed + 15485863)
    n_q, F = wl.n_q, wl.H_I * wl.d_I

    def draw(shape, fan_in):
        if wl.values == "int4":
            return torch.randint(-2, 3, shape, generator=gv, device=device).to(torch.bfloat16)
        return (torch.randn(shape, generator=gv, device=device) / math.sqrt(fan_in)).to(torch.bfloat16)

    out = {"wl": wl}
    out["xq"] = draw((n_q, wl.d_q), 1)
    out["x"] = draw((n_q, wl.d_model), 1)
    out["w_q"] = draw((F, wl.d_q), wl.d_q)
    out["w_k"] = draw((wl.d_I, wl.d_model), wl.d_model)
    out["w_w"] = draw((wl.H_I, wl.d_model), wl.d_model)
    if wl.values == "int4":
        out["ln_gamma"] = torch.ones(wl.d_I, device=device)
        out["ln_beta"] = torch.zeros(wl.d_I, device=device)
    else:
        out["ln_gamma"] = 1 + 0.1 * torch.randn(wl.d_I, generator=gv, device=device)
        out["ln_beta"] = 0.1 * torch.randn(wl.d_I, generator=gv, device=device)
    out["ln_eps"] = 1e-6
    out["w_scale"] = 1.0 / math.sqrt(wl.H_I)
    pt_k = _page_table(wl.pages(), wl.max_pages, gs)
    out["pt_k"] = pt_k.to(device)
    rows = wl.num_pages * wl.page_size
    if wl.li_dtype == "mxfp8":
        codes = torch.randint(0, 256, (rows, wl.d_I), generator=gv, device=device).to(torch.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0  # no NaN codes in the old contents
        out["k_pool"] = codes.view(torch.float8_e4m3fn).view(wl.num_pages, wl.page_size, wl.d_I)
        out["k_sf"] = torch.randint(120, 135, (wl.num_pages, wl.page_size, wl.d_I // MX_GROUP),
                                    generator=gv, device=device).to(torch.uint8)
    else:
        out["k_pool"] = torch.randn((wl.num_pages, wl.page_size, wl.d_I), generator=gv,
                                    device=device).to(torch.bfloat16)
        out["k_sf"] = None
    out["seq_lens"] = torch.tensor(wl.seq_lens, dtype=torch.int32, device=device)
    qs_ = [0]
    for n in wl.n_new:
        qs_.append(qs_[-1] + n)
    out["q_start"] = torch.tensor(qs_, dtype=torch.int32, device=device)
    return out


def to_device(inp: dict, device) -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def token_positions(wl: Workload) -> List[int]:
    """Absolute position of every query token: the new tokens are the last ones of each sequence."""
    pos = []
    for L, n in zip(wl.seq_lens, wl.n_new):
        pos.extend(range(L - n, L))
    return pos


def repage(inp: dict, seed: int) -> dict:
    """The same logical caches under fresh random page tables (for permutation-invariance checks)."""
    wl = inp["wl"]
    g = torch.Generator().manual_seed(seed)
    out = dict(inp)
    for pool_key, pt_key, sc_keys in (("k_pool", "pt_k", ("k_scale", "k_sf")),
                                      ("kv_pool", "pt_kv", ("kv8_pool",))):
        old_pt = inp[pt_key].cpu()
        new_pt = _page_table(wl.pages(), wl.max_pages, g)
        pool = inp[pool_key]
        new_pool = torch.empty_like(pool)
        src = [int(old_pt[b, p]) for b, n in enumerate(wl.pages()) for p in range(n)]
        dst = [int(new_pt[b, p]) for b, n in enumerate(wl.pages()) for p in range(n)]
        src_t = torch.tensor(src, device=pool.device)
        dst_t = torch.tensor(dst, device=pool.device)
        new_pool.view(pool.shape[0], -1)[dst_t] = pool.view(pool.shape[0], -1)[src_t]
        out[pool_key] = new_pool
        for sc_key in sc_keys:
            if inp.get(sc_key) is None:
                continue
            sc = inp[sc_key]
            new_sc = torch.empty_like(sc)
            new_sc[dst_t] = sc[src_t]
            out[sc_key] = new_sc
        out[pt_key] = new_pt.to(pool.device)
    return out
