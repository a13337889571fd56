"""Parity of the CUDA path (called through the C ABI) with the CPU oracle on seeded inputs.

Small cases span several 128-key tiles, several CTAs of a cluster and ragged tails; the six
full-size workloads run in the launch configuration the benchmark times and are checked on
sampled tokens.  Index sets are bit-exact on the integer-valued configs; elsewhere differences
must be certified near-ties.  Attention outputs stay within max-abs 2e-2 / mean-rel 5e-3 (bf16)
of the fp64 oracle on the GPU's own index sets, and within 5e-2 / 1e-2 end to end on the FP8
indexer path.
"""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_li_gb300 as dsa
import oracle
from parity import (BF16_TOL, FP8_TOL, check_end_to_end, check_indices, check_sfa, integer_fp8,
                    report, run_gpu, sample_tokens)

pytestmark = pytest.mark.gpu


def _small(name, **over):
    wl = di.small(name, **over)
    inp_cpu = di.generate(wl)
    return inp_cpu, di.to_device(inp_cpu, "cuda")


def _check_path(inp_cpu, g, toks, exact, tol=BF16_TOL):
    """Index sets, attention on the GPU's own sets, and the whole path end to end."""
    n_exact, ties, oidx = check_indices(inp_cpu, g, toks, exact=exact, return_oracle=True)
    check_sfa(inp_cpu, g, toks)
    check_end_to_end(inp_cpu, g, toks, oidx, tol)
    return n_exact, ties


# ------------------------------------------------------------------ indexer + attention, small

@pytest.mark.parametrize("lens,new", [([4096], [1]), ([300, 4096, 1000], [1, 2, 3]),
                                      ([70, 129, 2500], [1, 1, 1]), ([63], [1])])
def test_integer_config_bit_exact(cuda_lib, lens, new):
    inp_cpu, inp = _small("decode_int_4k", seq_lens=lens, n_new=new)
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    n_exact, ties = check_indices(inp_cpu, g, toks, exact=True)
    assert n_exact == len(toks)
    check_sfa(inp_cpu, g, toks)


@pytest.mark.parametrize("K", [1, 17, 64, 200])
def test_integer_config_small_k_bit_exact(cuda_lib, K):
    """Top-K of one position, of fewer rows than one 64-row attention tile, of exactly one tile
    and of a ragged number of tiles, beside a sequence of a single position: exact index sets,
    and the attention reads only the selected rows."""
    inp_cpu, inp = _small("decode_int_4k", seq_lens=[4096, 300, 1], n_new=[1, 2, 1], K=K)
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    n_exact, ties = check_indices(inp_cpu, g, toks, exact=True)
    assert n_exact == len(toks)
    check_sfa(inp_cpu, g, toks)


@pytest.mark.parametrize("lens,new", [([5000, 2100, 777], [1, 1, 1]), ([9000, 3000], [2, 2]),
                                      ([2047, 2048, 2049], [1, 2, 1])])
def test_bf16_indexer_and_attention_small(cuda_lib, lens, new):
    inp_cpu, inp = _small("decode_32k", seq_lens=lens, n_new=new)
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    _check_path(inp_cpu, g, toks, exact=False)


@pytest.mark.parametrize("lens,new", [([6000, 2500, 300], [1, 2, 1]), ([3000], [9]),
                                      ([4100, 700], [5, 3])])
def test_fp8_integer_unit_case_bit_exact(cuda_lib, lens, new):
    """Per-token FP8: integer e4m3 codes with their per-token scales, for single tokens and for
    groups of two and four tokens that share the key stream (each token's own query scale)."""
    inp_cpu, _ = _small("decode_32k_fp8", seq_lens=lens, n_new=new)
    inp_cpu = integer_fp8(inp_cpu, seed=3)
    inp = di.to_device(inp_cpu, "cuda")
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    n_exact, _ = check_indices(inp_cpu, g, toks, exact=True)
    assert n_exact == len(toks)


def test_fp8_normal_small(cuda_lib):
    inp_cpu, inp = _small("decode_32k_fp8", seq_lens=[7000, 3100], n_new=[1, 2])
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    _check_path(inp_cpu, g, toks, exact=False, tol=FP8_TOL)


@pytest.mark.parametrize("lens,new", [([6000, 2500, 300], [1, 2, 1]), ([4100, 129], [1, 1]),
                                      ([3000], [9])])
def test_mxfp8_integer_unit_case_bit_exact(cuda_lib, lens, new):
    """MXFP8: integer e4m3 codes with group scales 2^-1..2^1 keep every fp32 step exact."""
    inp_cpu, inp = _small("decode_32k_mxfp8", seq_lens=lens, n_new=new, values="int4",
                          w_values="int14")
    assert set(torch.unique(inp_cpu["k_sf"]).tolist()) == {126, 127, 128}
    g = run_gpu(inp, prefill=False)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    n_exact, _ = check_indices(inp_cpu, g, toks, exact=True)
    assert n_exact == len(toks)


@pytest.mark.parametrize("lens,new", [([7000, 3100], [1, 2]), ([5000], [40])])
def test_mxfp8_normal_small(cuda_lib, lens, new):
    inp_cpu, inp = _small("decode_32k_mxfp8", seq_lens=lens, n_new=new)
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = sample_tokens(inp_cpu["wl"], 12, seed=2)
    _check_path(inp_cpu, g, toks, exact=False, tol=FP8_TOL)


def test_prefill_small(cuda_lib):
    inp_cpu, inp = _small("prefill_64k", seq_lens=[3000], n_new=[300], K=256)
    g = run_gpu(inp, prefill=True)
    assert g["status"] == 0
    toks = sample_tokens(inp_cpu["wl"], 12, seed=1)
    _check_path(inp_cpu, g, toks, exact=False)


@pytest.mark.parametrize("splits", [2, 4])
def test_integer_config_row_splits_16_heads(cuda_lib, splits):
    """16 SFA heads (padded to 128 on chip) through the cluster merge of two splits and the
    last-CTA merge of four, on the integer-exact indexer config."""
    inp_cpu, inp = _small("decode_int_4k", seq_lens=[4096, 700], n_new=[1, 2])
    g = run_gpu(inp, prefill=False, row_splits=splits)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    n_exact, _ = check_indices(inp_cpu, g, toks, exact=True)
    assert n_exact == len(toks)
    check_sfa(inp_cpu, g, toks)


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_decode_row_split_counts(cuda_lib, splits):
    """One split (no merge), two (the splits of a token share a cluster of four and each finalises
    half of the heads) and three (the last CTA merges all partials) give the oracle's attention
    on the same index sets."""
    inp_cpu, inp = _small("decode_32k", seq_lens=[5000, 3000, 129], n_new=[1, 2, 1])
    g = run_gpu(inp, prefill=False, row_splits=splits)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    check_indices(inp_cpu, g, toks, exact=False)
    check_sfa(inp_cpu, g, toks)


def test_decode_and_prefill_attention_agree(cuda_lib):
    inp_cpu, inp = _small("decode_32k", seq_lens=[4000, 5000], n_new=[1, 1])
    a = run_gpu(inp, prefill=False)
    b = run_gpu(inp, prefill=True)
    assert np.array_equal(a["idx"], b["idx"])
    d = (a["out"] - b["out"]).abs().max().item()
    assert d <= 2e-2, d


@pytest.mark.parametrize("prefill", [False, True])
def test_sequence_without_new_tokens(cuda_lib, prefill):
    """A sequence of the batch with no query tokens (equal consecutive q_start) contributes no
    rows and does not disturb its neighbours."""
    inp_cpu, inp = _small("decode_32k", seq_lens=[3000, 2000, 4000], n_new=[1, 0, 2])
    g = run_gpu(inp, prefill=prefill)
    assert g["status"] == 0
    toks = list(range(inp_cpu["wl"].n_q))
    check_indices(inp_cpu, g, toks, exact=False)
    check_sfa(inp_cpu, g, toks)


def test_k_covers_context_selects_everything(cuda_lib):
    inp_cpu, inp = _small("decode_32k", seq_lens=[1500, 64, 2048], n_new=[1, 2, 1])
    g = run_gpu(inp)
    pos = di.token_positions(inp_cpu["wl"])
    for t, p in enumerate(pos):
        assert g["idx"][t].tolist() == list(range(p + 1)) + [-1] * (2048 - p - 1)
    check_sfa(inp_cpu, g, list(range(len(pos))))


# ------------------------------------------------------------------ invariants on the GPU

def test_page_permutation_invariance_and_determinism(cuda_lib):
    inp_cpu, inp = _small("decode_32k", seq_lens=[6000, 3000], n_new=[1, 2])
    a = run_gpu(inp)
    a2 = run_gpu(inp)
    assert np.array_equal(a["idx"], a2["idx"]) and torch.equal(a["out"], a2["out"])
    inp_r = di.to_device(di.repage(inp_cpu, seed=77), "cuda")
    b = run_gpu(inp_r)
    assert np.array_equal(a["idx"], b["idx"])
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["lse"], b["lse"])


def test_bad_page_id_sets_status_without_fault(cuda_lib):
    inp_cpu, inp = _small("decode_32k", seq_lens=[3000], n_new=[1])
    pt = inp["pt_k"].clone()
    pt[0, 5] = inp["k_pool"].shape[0] + 100
    inp = dict(inp, pt_k=pt)
    g = run_gpu(inp)
    assert g["status"] == dsa.DSA_ERR_DEVICE_CHECK
    torch.cuda.synchronize()  # the context is still usable


def test_sequence_longer_than_page_table_sets_status_without_fault(cuda_lib):
    """A sequence length past what the page table covers is reported, never read past."""
    inp_cpu, inp = _small("decode_32k", seq_lens=[3000], n_new=[1])
    wl = inp["wl"]
    pt_k, pt_kv = inp["pt_k"][:, :20].contiguous(), inp["pt_kv"][:, :20].contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.full((wl.n_q, wl.K), -1, dtype=torch.int32, device="cuda")
    dsa.li_topk(inp["q_li"], inp["w"], inp["k_pool"], pt_k, inp["seq_lens"], inp["q_start"], wl.K,
                max_seq_len=20 * 64, max_q_per_seq=1, out_idx=idx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == dsa.DSA_ERR_DEVICE_CHECK
    status.zero_()
    idx[:, :8] = torch.arange(1272, 1280 + 7 * 8, 8, dtype=torch.int32)  # last 7 past coverage
    dsa.sfa_decode(inp["q_sfa"], inp["kv_pool"], pt_kv, inp["seq_lens"], inp["q_start"], idx,
                   softmax_scale=wl.softmax_scale, max_seq_len=20 * 64, max_q_per_seq=1,
                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == dsa.DSA_ERR_DEVICE_CHECK


def test_unit_length_beyond_bound_sets_status_without_fault(cuda_lib):
    """With position units, a sequence longer than max_seq_len (units x span) is reported and
    skipped by the plan, the indexer and the merge; the other sequences are still exact."""
    inp_cpu, inp = _small("decode_int_4k", seq_lens=[40000, 70000], n_new=[1, 1])
    wl = inp_cpu["wl"]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.full((wl.n_q, wl.K), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.n_q,), dtype=torch.int32, device="cuda")
    assert dsa.li_workspace_bytes(2, wl.K, 40000, 1) > 0
    dsa.li_topk(inp["q_li"], inp["w"], inp["k_pool"], inp["pt_k"], inp["seq_lens"], inp["q_start"],
                wl.K, max_seq_len=40000, max_q_per_seq=1, out_idx=idx, out_cnt=cnt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == dsa.DSA_ERR_DEVICE_CHECK
    g = {"idx": idx.cpu().numpy(), "cnt": cnt.cpu().numpy()}
    n_exact, _ = check_indices(inp_cpu, g, [0], exact=True)
    assert n_exact == 1
    assert np.all(g["idx"][1] == -7)  # the skipped token's row is left as it was


def test_cache_write_roundtrip(cuda_lib):
    inp_cpu, inp = _small("decode_32k", seq_lens=[200, 100], n_new=[1, 1])
    pool = torch.zeros_like(inp["kv_pool"])
    seq = torch.tensor([0, 0, 1, 1], dtype=torch.int32, device="cuda")
    pos = torch.tensor([0, 199, 5, 99], dtype=torch.int32, device="cuda")
    rows = torch.randn(4, 576, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.cache_write(pool, inp["pt_kv"], seq, pos, rows, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pt = inp["pt_kv"].cpu()
    for r in range(4):
        b, j = int(seq[r]), int(pos[r])
        assert torch.equal(pool[int(pt[b, j // 64]), j % 64], rows[r])


def test_cuda_graph_replay_matches_eager(cuda_lib):
    inp_cpu, inp = _small("decode_32k", seq_lens=[5000, 4000], n_new=[1, 1])
    eager = run_gpu(inp)
    wl = inp["wl"]
    idx = torch.empty((wl.n_q, wl.K), dtype=torch.int32, device="cuda")
    cnt = torch.empty((wl.n_q,), dtype=torch.int32, device="cuda")
    out = torch.empty((wl.n_q, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.n_q, wl.H), dtype=torch.float32, device="cuda")
    ws = dsa.new_workspace(dsa.sfa_workspace_bytes(inp["q_sfa"], idx), "cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dsa.decode_step(inp, idx=idx, cnt=cnt, out=out, lse=lse, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dsa.decode_step(inp, idx=idx, cnt=cnt, out=out, lse=lse, workspace=ws)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), eager["idx"])
    assert torch.equal(out.float().cpu(), eager["out"])


# ------------------------------------------------------------------ full-size workloads

# (workload, index sets bit-exact, end-to-end attention tolerance of its indexer path)
FULL = [("decode_int_4k", True, BF16_TOL), ("decode_32k", False, BF16_TOL),
        ("decode_32k_fp8", False, FP8_TOL), ("decode_32k_mxfp8", False, FP8_TOL),
        ("decode_32k_kv8", False, BF16_TOL), ("specdec_ragged", False, BF16_TOL),
        ("prefill_64k", False, BF16_TOL)]


def full_size_sample(wl):
    """Tokens checked at full size: every token of the decode and speculative batches; for the
    4096-token prefill chunk its first and last 8 tokens plus 48 drawn from the rest."""
    if wl.n_q <= 128:
        return list(range(wl.n_q))
    g = np.random.default_rng(11)
    pick = set(range(8)) | set(range(wl.n_q - 8, wl.n_q))
    while len(pick) < 64:
        pick.add(int(g.integers(8, wl.n_q - 8)))
    return sorted(pick)


@pytest.mark.parametrize("name,exact,tol", FULL, ids=[f[0] for f in FULL])
def test_full_size_workload_sampled(cuda_lib, name, exact, tol):
    """Full-size workloads in the benchmark's launch configuration.  Index sets: bit-exact on the
    integer-valued workload, certified near-ties elsewhere (every one is recorded).  Attention:
    on the GPU's own index sets within the bf16 tolerance, and end to end (GPU pipeline against
    the oracle's selection followed by the oracle's attention) within the indexer path's
    tolerance."""
    wl = di.preset(name)
    inp = di.generate(wl, device="cuda")
    g = run_gpu(inp)
    assert g["status"] == 0
    inp_cpu = di.to_device(inp, "cpu")
    del inp
    toks = full_size_sample(wl)
    n_exact, ties, oidx = check_indices(inp_cpu, g, toks, exact=exact, return_oracle=True)
    own = check_sfa(inp_cpu, g, toks)
    e2e = check_end_to_end(inp_cpu, g, toks, oidx, tol)
    report({"test": "full_size", "workload": name, "tokens": len(toks), "exact_rows": n_exact,
            "near_ties": [[int(t), int(n), round(float(r), 4)] for t, n, r in ties],
            "own_indices": {"max_abs": own[0], "mean_rel": own[1], "lse_abs": own[2]},
            "end_to_end": {"max_abs": e2e[0], "mean_rel": e2e[1], "lse_abs": e2e[2],
                           "tol": list(tol)}})


# ------------------------------------------------------------------ context-parallel indexer

@pytest.mark.parametrize("name,L,B,S", [("decode_int_4k", 4096, 2, 2), ("decode_32k", 9000, 2, 3),
                                        ("decode_32k_mxfp8", 12800, 1, 4), ("decode_32k_fp8", 5000, 3, 2)])
def test_context_parallel_shards_merge_to_the_full_selection(cuda_lib, name, L, B, S):
    """Each shard (a page-aligned range of every sequence's positions, same for all sequences)
    selects its own top-K with scores; merging the shards' candidates gives exactly the
    unsharded selection (a position's score does not depend on the split).  Decode: the query
    is the last position, so every shard's positions are visible to it."""
    inp_cpu, inp = _small(name, seq_lens=[L] * B, n_new=[1] * B)
    wl = inp_cpu["wl"]
    full = run_gpu(inp)
    pages = (L + 63) // 64
    cuts = [round(pages * s / S) for s in range(S + 1)]
    cand_idx = torch.empty((S, wl.n_q, wl.K), dtype=torch.int32, device="cuda")
    cand_score = torch.empty((S, wl.n_q, wl.K), dtype=torch.float32, device="cuda")
    offsets = []
    for s in range(S):
        lo, hi = cuts[s] * 64, min(L, cuts[s + 1] * 64)
        offsets.append(lo)
        pt = inp["pt_k"][:, cuts[s]:cuts[s + 1]].contiguous()
        seq = torch.full((B,), hi - lo, dtype=torch.int32, device="cuda")
        dsa.li_topk(inp["q_li"], inp["w"], inp["k_pool"], pt, seq, inp["q_start"], wl.K,
                    q_scale=inp.get("q_scale"), k_scale=inp.get("k_scale"), q_sf=inp.get("q_sf"),
                    k_sf=inp.get("k_sf"), out_idx=cand_idx[s], out_score=cand_score[s],
                    max_seq_len=hi - lo, max_q_per_seq=1)
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    idx, cnt = dsa.topk_merge(cand_idx, cand_score, off, wl.K)
    torch.cuda.synchronize()
    merged = {"idx": idx.cpu().numpy(), "cnt": cnt.cpu().numpy()}
    assert np.array_equal(merged["idx"], full["idx"])
    assert np.array_equal(merged["cnt"], full["cnt"])
    # the merged selection against the oracle's unsharded one: bit-exact on the integer-valued
    # config, certified near-ties elsewhere
    toks = list(range(wl.n_q))
    n_exact, ties = check_indices(inp_cpu, merged, toks, exact=name == "decode_int_4k")
    report({"test": "context_parallel_merge", "workload": name, "shards": S, "tokens": len(toks),
            "exact_rows": n_exact, "near_ties": [[int(t), int(n), round(float(r), 4)]
                                                 for t, n, r in ties]})
    # the scores a shard reports are the oracle's (exact on the integer-valued config)
    if name == "decode_int_4k":
        s_or, _ = oracle.li_scores(inp_cpu, 0)
        ci, cs = cand_idx[0, 0].cpu().numpy(), cand_score[0, 0].cpu().numpy()
        assert np.array_equal(cs[ci >= 0], s_or[ci[ci >= 0]])


# ------------------------------------------------------------------ position units

@pytest.mark.parametrize("name,lens,new,exact", [
    ("decode_int_4k", [40000, 3000, 70000], [1, 2, 1], True),
    ("decode_32k", [33000, 5000, 65600], [2, 1, 2], False),
    ("decode_32k_mxfp8", [40000, 900], [1, 1], False),
    ("decode_32k_fp8", [98400, 32769], [1, 2], False)])
def test_position_units_long_and_short_sequences(cuda_lib, name, lens, new, exact):
    """Sequences longer than one cluster's span (32768 positions) are split into units whose
    local top-K candidates are merged on the GPU; the batch mixes them with short ones.  The
    selection equals the oracle's over the whole sequence (bit-exact on the integer config,
    certified near-ties elsewhere), the attention follows, and the scores reported with
    out_score are the oracle's (exact on the integer config)."""
    inp_cpu, inp = _small(name, seq_lens=lens, n_new=new)
    wl = inp_cpu["wl"]
    assert dsa.li_workspace_bytes(len(lens), wl.K, max(lens), max(new)) > 0
    g = run_gpu(inp)
    assert g["status"] == 0
    toks = list(range(wl.n_q))
    n_exact, ties = _check_path(inp_cpu, g, toks, exact=exact,
                                tol=FP8_TOL if wl.li_dtype != "bf16" else BF16_TOL)
    report({"test": "position_units", "workload": name, "lens": lens, "tokens": len(toks),
            "exact_rows": n_exact, "near_ties": [[int(t), int(n), round(float(r), 4)]
                                                 for t, n, r in ties]})
    # the same selection with scores requested (scores of the merged candidates)
    score = torch.empty((wl.n_q, wl.K), dtype=torch.float32, device="cuda")
    idx2, cnt2 = dsa.li_topk(inp["q_li"], inp["w"], inp["k_pool"], inp["pt_k"], inp["seq_lens"],
                             inp["q_start"], wl.K, q_scale=inp.get("q_scale"),
                             k_scale=inp.get("k_scale"), q_sf=inp.get("q_sf"), k_sf=inp.get("k_sf"),
                             out_score=score, max_seq_len=max(lens), max_q_per_seq=max(new))
    torch.cuda.synchronize()
    assert np.array_equal(idx2.cpu().numpy(), g["idx"])
    sc = score.cpu().numpy()
    assert np.all(np.isneginf(sc[g["idx"] < 0]))
    if exact:
        for t in toks:
            s_or, _ = oracle.li_scores(inp_cpu, t)
            row = g["idx"][t]
            assert np.array_equal(sc[t][row >= 0], s_or[row[row >= 0]])


# ------------------------------------------------------------------ FP8 latent cache

@pytest.mark.parametrize("name,lens,new,prefill,K", [
    ("decode_32k", [5000, 2100, 777], [1, 2, 1], False, None),
    ("decode_int_4k", [4096, 700], [1, 2], False, None),
    ("prefill_64k", [3000], [300], True, 256)])
def test_fp8_latent_cache_attention(cuda_lib, name, lens, new, prefill, K):
    """Attention over FP8 latent rows (e4m3 codes, fp32 scale per 128-column tile) against the
    oracle on the same rows, de-quantised as bf16(fp32(code * scale))."""
    over = dict(seq_lens=lens, n_new=new, kv_dtype="fp8")
    if K:
        over["K"] = K
    inp_cpu, inp = _small(name, **over)
    g = run_gpu(inp, prefill=prefill)
    assert g["status"] == 0
    toks = sample_tokens(inp_cpu["wl"], 12, seed=4)
    check_indices(inp_cpu, g, toks, exact=name == "decode_int_4k")
    check_sfa(inp_cpu, g, toks)


@pytest.mark.parametrize("li_dtype", ["fp8", "mxfp8"])
def test_quantised_indexer_with_fp8_latent_cache(cuda_lib, li_dtype):
    """The fully quantised path: an e4m3 indexer (per-token or MX group scales) selects the rows
    and the attention reads them from the FP8 latent cache; index sets are certified against the
    oracle, and the output is checked on the GPU's own sets and end to end against the oracle's
    selection and attention, within the FP8 indexer path's tolerance."""
    inp_cpu, inp = _small("decode_32k_kv8", seq_lens=[5000, 2100, 777], n_new=[1, 2, 1],
                          li_dtype=li_dtype)
    g = run_gpu(inp)
    assert g["status"] == 0
    _check_path(inp_cpu, g, list(range(inp_cpu["wl"].n_q)), exact=False, tol=FP8_TOL)
