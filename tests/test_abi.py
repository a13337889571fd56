"""The C-ABI library builds, loads without a GPU, exports every symbol include/dsa.h declares,
and rejects bad arguments on the host before touching CUDA (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

import dsa_sparse_attention_li_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = dsa.load()
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(dsa.SYMBOLS)


def test_abi_version_and_status_strings():
    lib = dsa.load()
    assert lib.dsa_abi_version() == 7
    assert dsa.status_string(0) == "DSA_OK"
    assert dsa.status_string(5) == "DSA_ERR_TIMEOUT"
    assert dsa.status_string(77) == "DSA_ERR_UNKNOWN"


def test_struct_layouts_match_header():
    """ctypes mirrors of the argument structs have the C sizes (x86_64 / aarch64 LP64)."""
    assert ctypes.sizeof(dsa.LiArgs) == 11 * 4 + 4 + 15 * 8 + 8
    assert ctypes.sizeof(dsa.MergeArgs) == 4 * 4 + 5 * 8
    assert ctypes.sizeof(dsa.SfaArgs) == 12 * 4 + 10 * 8 + 8 + 8
    assert ctypes.sizeof(dsa.PrologArgs) == 10 * 4 + 2 * 4 + 16 * 8 + 8 + 8


def test_static_scratch_covers_every_automatic_decode_plan():
    """20 MiB of static scratch holds the split-merge workspace of every decode plan the library
    chooses by itself (row_splits = 0) for K <= 2048, at the SM count the plan sees here (the
    152-SM default without a GPU); an explicit row_splits may exceed it."""
    worst = 0
    for n_q in list(range(1, 161)) + [256, 1024]:
        q = torch.empty((n_q, 128, 576), dtype=torch.bfloat16, device="meta")
        for K in (1, 63, 64, 65, 128, 500, 1000, 1024, 2047, 2048):
            idx = torch.empty((n_q, K), dtype=torch.int32, device="meta")
            worst = max(worst, dsa.sfa_workspace_bytes(q, idx))
    assert 0 < worst <= dsa.SFA_STATIC_SCRATCH_BYTES
    q = torch.empty((32, 128, 576), dtype=torch.bfloat16, device="meta")
    idx = torch.empty((32, 2048), dtype=torch.int32, device="meta")
    assert dsa.sfa_workspace_bytes(q, idx, row_splits=32) > dsa.SFA_STATIC_SCRATCH_BYTES


def test_li_workspace_bytes_for_position_units():
    """Scratch for the indexer's position units: none unless a decode or two-token group's
    sequence can exceed one cluster's span (32768 positions) and the batch has at most 256
    sequences, then one K-row of positions and one of scores per (sequence, unit, token) and
    the unit plan's item list, each array padded to 256 bytes."""
    assert dsa.li_workspace_bytes(32, 2048, 32768, 1) == 0
    assert dsa.li_workspace_bytes(1, 2048, 131072, 4096) == 0      # prefill: no units
    assert dsa.li_workspace_bytes(64, 2048, 131072, 3) == 0        # groups of 4: no units
    half = lambda n: (n * 4 + 255) // 256 * 256
    # + the item list of the unit plan: a count and one word per (sequence, unit)
    assert dsa.li_workspace_bytes(64, 2048, 131072, 2) == 2 * half(64 * 4 * 2 * 2048) + half(1 + 64 * 4)
    assert dsa.li_workspace_bytes(3, 256, 70000, 1) == 2 * half(3 * 3 * 256) + half(1 + 3 * 3)
    assert dsa.li_workspace_bytes(2, 2048, 32769, 1) == 2 * half(2 * 2 * 2048) + half(1 + 2 * 2)
    assert dsa.li_workspace_bytes(257, 2048, 65536, 1) == 0  # more sequences than the plan orders


def test_page_bytes():
    assert dsa.page_bytes(dsa.DSA_BF16, 64, 576) == 64 * 576 * 2
    assert dsa.page_bytes(dsa.DSA_FP8_E4M3, 64, 128) == 64 * 128
    assert dsa.page_bytes(dsa.DSA_BF16, -1, 4) == 0


def test_page_table_validate():
    pt = torch.tensor([[3, 1, 0], [2, 0, 0]], dtype=torch.int32)
    sl = torch.tensor([130, 64], dtype=torch.int32)
    dsa.page_table_validate(pt, sl, 64, 4, require_unique=True)
    with pytest.raises(dsa.DsaError) as e:
        dsa.page_table_validate(pt, sl, 64, 3)          # page 3 out of range
    assert "out of" in str(e.value)
    with pytest.raises(dsa.DsaError):
        dsa.page_table_validate(torch.tensor([[1, 1, 0], [2, 0, 0]], dtype=torch.int32), sl, 64, 4,
                                require_unique=True)    # page 1 used twice
    with pytest.raises(dsa.DsaError):
        dsa.page_table_validate(pt, torch.tensor([200, 1], dtype=torch.int32), 64, 4)  # > max_pages


def _li(**over):
    a = dsa.LiArgs()
    a.B, a.n_q, a.H_I, a.d_I, a.K, a.page_size, a.max_pages, a.num_pages = 1, 1, 64, 128, 2048, 64, 8, 8
    a.max_seq_len, a.max_q_per_seq, a.dtype = 512, 1, dsa.DSA_BF16
    for n in ("q", "w", "k_pool", "page_table", "seq_lens", "q_start", "out_idx"):
        setattr(a, n, 4096)  # fake, aligned, never dereferenced on these error paths
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    ({"K": 0}, dsa.DSA_ERR_INVALID_ARG),
    ({"B": 0}, dsa.DSA_ERR_INVALID_ARG),
    ({"dtype": 7}, dsa.DSA_ERR_INVALID_ARG),
    ({"q": None}, dsa.DSA_ERR_INVALID_ARG),
    ({"dtype": dsa.DSA_FP8_E4M3}, dsa.DSA_ERR_INVALID_ARG),   # no scales
    ({"max_seq_len": 8 * 64 + 1}, dsa.DSA_ERR_INVALID_ARG),
    ({"q": 4097}, dsa.DSA_ERR_INVALID_ARG),                    # misaligned
    ({"K": 4096}, dsa.DSA_ERR_UNSUPPORTED),
    ({"page_size": 32, "max_pages": 16}, dsa.DSA_ERR_UNSUPPORTED),
])
def test_li_topk_host_validation(over, code):
    lib = dsa.load()
    rc = lib.dsa_li_topk(ctypes.byref(_li(**over)), None)
    assert rc == code, dsa.last_error()
    assert dsa.last_error()


def test_li_topk_null_args_and_empty_batch():
    lib = dsa.load()
    assert lib.dsa_li_topk(None, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_li_topk(ctypes.byref(_li(n_q=0)), None) == dsa.DSA_OK


def _sfa(**over):
    a = dsa.SfaArgs()
    a.B, a.n_q, a.H, a.d_qk, a.d_v, a.K, a.page_size, a.max_pages, a.num_pages = 1, 1, 128, 576, 512, 2048, 64, 8, 8
    a.max_seq_len, a.max_q_per_seq, a.softmax_scale = 512, 1, 1 / 24
    for n in ("q", "kv_pool", "page_table", "seq_lens", "q_start", "idx", "out"):
        setattr(a, n, 4096)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    ({"H": 0}, dsa.DSA_ERR_INVALID_ARG),
    ({"softmax_scale": 0.0}, dsa.DSA_ERR_INVALID_ARG),
    ({"softmax_scale": float("nan")}, dsa.DSA_ERR_INVALID_ARG),
    ({"idx": None}, dsa.DSA_ERR_INVALID_ARG),
    ({"out": 4100}, dsa.DSA_ERR_INVALID_ARG),
    ({"d_qk": 512}, dsa.DSA_ERR_UNSUPPORTED),
    ({"H": 256}, dsa.DSA_ERR_UNSUPPORTED),
    ({"K": 4096}, dsa.DSA_ERR_UNSUPPORTED),
    ({"kv_dtype": dsa.DSA_MXFP8_E4M3}, dsa.DSA_ERR_UNSUPPORTED),  # latent cache: bf16 or FP8 rows
])
@pytest.mark.parametrize("entry", ["dsa_sfa_decode", "dsa_sfa_prefill"])
def test_sfa_host_validation(over, code, entry):
    lib = dsa.load()
    rc = getattr(lib, entry)(ctypes.byref(_sfa(**over)), None)
    assert rc == code, dsa.last_error()


def test_cache_write_host_validation():
    lib = dsa.load()
    P = 4096
    assert lib.dsa_cache_write(P, None, 4, 64, 576, 3, P, 4, 1, P, P, P, None, 1, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_cache_write(P, None, 4, 64, 4, 2, P, 4, 1, P, P, P, None, 1, None, None) == dsa.DSA_ERR_UNSUPPORTED
    assert lib.dsa_cache_write(P, P, 4, 64, 576, 2, P, 4, 1, P, P, P, None, 1, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_cache_write(P, None, 4, 64, 576, 2, P, 4, 1, P, P, P, None, 0, None, None) == dsa.DSA_OK


def _prolog(**over):
    a = dsa.PrologArgs()
    a.n_q, a.B, a.d_q, a.d_model, a.H_I, a.d_I = 4, 2, 1536, 7168, 64, 128
    a.dtype, a.page_size, a.max_pages, a.num_pages = dsa.DSA_MXFP8_E4M3, 64, 8, 16
    a.ln_eps, a.w_scale = 1e-6, 0.125
    for n in ("xq", "x", "w_q", "w_k", "w_w", "ln_gamma", "ln_beta", "page_table", "seq_lens",
              "q_start", "q_out", "q_sf", "w_out", "k_pool", "k_sf", "workspace"):
        setattr(a, n, 4096)  # fake, aligned, never dereferenced on these error paths
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,code", [
    ({"B": 0}, dsa.DSA_ERR_INVALID_ARG),
    ({"n_q": -1}, dsa.DSA_ERR_INVALID_ARG),
    ({"H_I": 32}, dsa.DSA_ERR_UNSUPPORTED),
    ({"d_I": 64}, dsa.DSA_ERR_UNSUPPORTED),
    ({"dtype": dsa.DSA_FP8_E4M3}, dsa.DSA_ERR_UNSUPPORTED),   # per-token FP8 is not produced
    ({"d_q": 1540}, dsa.DSA_ERR_UNSUPPORTED),                 # row stride not a multiple of 16 B
    ({"k_sf": None}, dsa.DSA_ERR_INVALID_ARG),                # MXFP8 needs the scale arrays
    ({"x": 4100}, dsa.DSA_ERR_INVALID_ARG),                   # misaligned
])
def test_indexer_prolog_host_validation(over, code):
    lib = dsa.load()
    a = _prolog(**over)
    assert lib.dsa_indexer_prolog(ctypes.byref(a), None) == code
    assert dsa.last_error()
    if code == dsa.DSA_ERR_UNSUPPORTED or over.get("B") == 0 or "n_q" in over:
        assert lib.dsa_prolog_workspace_bytes(ctypes.byref(a)) == 0
    assert lib.dsa_indexer_prolog(None, None) == dsa.DSA_ERR_INVALID_ARG


def test_topk_merge_host_validation():
    lib = dsa.load()
    a = dsa.MergeArgs()
    a.S, a.n_q, a.K_in, a.K = 2, 3, 2048, 2048
    for n in ("cand_idx", "cand_score", "shard_offset", "out_idx"):
        setattr(a, n, 4096)
    assert lib.dsa_topk_merge(None, None) == dsa.DSA_ERR_INVALID_ARG
    a.S = 9
    assert lib.dsa_topk_merge(ctypes.byref(a), None) == dsa.DSA_ERR_UNSUPPORTED  # 9 x 2048 > 16384
    a.S, a.cand_idx = 2, None
    assert lib.dsa_topk_merge(ctypes.byref(a), None) == dsa.DSA_ERR_INVALID_ARG
    a.n_q = 0
    assert lib.dsa_topk_merge(ctypes.byref(a), None) == dsa.DSA_OK  # nothing to merge


def test_test_hook_symbol_only_in_the_test_build():
    """dsa_test_inject_stall (include/dsa_testhooks.h) exists in libdsa_testhooks.so only."""
    assert not hasattr(dsa.load(), "dsa_test_inject_stall")
    hooks = dsa.load_testhooks()
    assert hasattr(hooks, "dsa_test_inject_stall")
    for n in dsa.SYMBOLS:
        assert hasattr(hooks, n), n
