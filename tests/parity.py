"""Comparison helpers: the CUDA path (through the C ABI) against the CPU oracle.

Index sets: bit-exact where the inputs make every fp32 step exact (integer-valued configs);
otherwise every difference must be a certified near-tie: both the dropped and the added position
have oracle scores within the fp32 forward-error bound of the oracle's K-th score.

Attention outputs are checked twice, within the stated tolerances (max-abs, mean-relative):
  - on the GPU's own index sets, which isolates attention from selection (bf16 tolerance: the
    attention arithmetic is bf16 on every path);
  - end to end: the GPU pipeline (its own selection, then its attention) against the oracle's
    pipeline (the oracle's selection, then the oracle's attention), with the tolerance of the
    indexer path (bf16, or the wider one of the FP8 indexer paths).
``report`` appends one JSON line per checked workload to the file named by the environment
variable DSA_PARITY_REPORT (test bookkeeping: exact rows, certified near-ties, errors).
"""
import json
import math
import os

import numpy as np
import torch

import dsa_inputs as di
import dsa_sparse_attention_li_gb300 as dsa
import oracle

# fp32 unit roundoff of a truncating adder (tensor-core accumulation order and rounding are
# not specified, so the bound assumes the worse of round-to-nearest and truncation)
U32 = 2.0 ** -23
BF16_TOL = (2e-2, 5e-3)   # max-abs, mean-rel
FP8_TOL = (5e-2, 1e-2)


def run_gpu(inp, prefill=None, workspace=None, row_splits=0):
    """li_topk then sfa_{decode,prefill} on the current stream; returns CPU tensors + status."""
    wl = inp["wl"]
    if prefill is None:
        prefill = max(wl.n_new) > 2
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, cnt, out, lse = dsa.decode_step(inp, status=status, prefill=prefill, workspace=workspace,
                                         row_splits=row_splits)
    torch.cuda.synchronize()
    return {"idx": idx.cpu().numpy(), "cnt": cnt.cpu().numpy(), "out": out.float().cpu(),
            "lse": lse.cpu(), "status": int(status.item())}


def sample_tokens(wl, n, seed=0):
    if wl.n_q <= n:
        return list(range(wl.n_q))
    g = np.random.default_rng(seed)
    pick = {0, wl.n_q - 1}
    while len(pick) < n:
        pick.add(int(g.integers(0, wl.n_q)))
    return sorted(pick)


def row_is_valid(row, cnt, p, K):
    sel = row[row >= 0]
    return (len(sel) == cnt and np.all(row[cnt:] == -1) and np.all(np.diff(sel) > 0)
            and (len(sel) == 0 or (sel[0] >= 0 and sel[-1] <= p)))


def check_indices(inp_cpu, g, tokens, exact, return_oracle=False):
    """Returns (n_exact, near_ties[, oracle index rows]); asserts validity, exactness or
    certification.  A near-tie entry is (token, positions swapped, max |s - s_K| / bound)."""
    wl = inp_cpu["wl"]
    pos = di.token_positions(wl)
    oidx, ocnt, okth = oracle.li_topk(inp_cpu, tokens)
    gamma = (wl.d_I + wl.H_I + 8) * U32
    n_exact, ties = 0, []
    for i, t in enumerate(tokens):
        grow, orow = g["idx"][t], oidx[i]
        assert g["cnt"][t] == ocnt[i], (t, g["cnt"][t], ocnt[i])
        assert row_is_valid(grow, ocnt[i], pos[t], wl.K), t
        if np.array_equal(grow, orow):
            n_exact += 1
            continue
        assert not exact, "token %d: index sets differ on an exact config" % t
        s, mag = oracle.li_scores(inp_cpu, t)
        gs, os_ = set(grow[grow >= 0].tolist()), set(orow[orow >= 0].tolist())
        kth = okth[i]
        # the position holding the K-th score in the oracle's order
        j_k = max((j for j in os_ if s[j] == kth))
        eps_k = gamma * mag[j_k]
        worst = 0.0
        for j in gs ^ os_:
            bound = gamma * mag[j] + eps_k
            assert abs(s[j] - kth) <= bound, (
                "token %d position %d: |s - s_K| = %g exceeds bound %g" %
                (t, j, abs(s[j] - kth), bound))
            worst = max(worst, abs(s[j] - kth) / bound)
        ties.append((t, len(gs - os_), worst))
    if return_oracle:
        return n_exact, ties, oidx
    return n_exact, ties


def sfa_errors(inp_cpu, g, tokens, idx=None):
    """(max_abs, mean_rel, max_lse_abs) of the GPU attention against the oracle's attention on
    the index rows ``idx`` (default: the GPU's own index sets)."""
    wl = inp_cpu["wl"]
    if idx is None:
        idx = np.stack([g["idx"][t] for t in tokens])
    ref, ref_lse = oracle.sfa(inp_cpu, idx, tokens)
    got = g["out"][tokens][:, :wl.H].double().numpy()
    diff = np.abs(got - ref)
    max_abs = float(diff.max())
    mean_rel = float(diff.sum() / max(np.abs(ref).sum(), 1e-300))
    gl = g["lse"][tokens][:, :wl.H].double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(gl))
    lse_err = float(np.abs(gl[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
    return max_abs, mean_rel, lse_err


def check_sfa(inp_cpu, g, tokens, tol=BF16_TOL, lse_tol=2e-3):
    """Attention alone: the GPU's output against the oracle's attention on the GPU's own index
    sets."""
    max_abs, mean_rel, lse_err = sfa_errors(inp_cpu, g, tokens)
    assert max_abs <= tol[0] and mean_rel <= tol[1], (max_abs, mean_rel)
    assert lse_err <= lse_tol, lse_err
    return max_abs, mean_rel, lse_err


def check_end_to_end(inp_cpu, g, tokens, oracle_idx, tol):
    """The whole path: the GPU's output (its selection, then its attention) against the oracle's
    attention on the oracle's own selection, within ``tol`` (max-abs, mean-rel).  The lse is
    reported, not bounded: a certified near-tie swap moves it by the swapped row's weight."""
    max_abs, mean_rel, lse_err = sfa_errors(inp_cpu, g, tokens, idx=oracle_idx)
    assert max_abs <= tol[0] and mean_rel <= tol[1], (max_abs, mean_rel, tol)
    return max_abs, mean_rel, lse_err


def report(record: dict):
    """Append one JSON line to $DSA_PARITY_REPORT (no-op when unset)."""
    path = os.environ.get("DSA_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps(record) + "\n")


def integer_fp8(inp, seed=0):
    """Replace the indexer inputs of a workload by e4m3 codes of integers in [-8, 8] with
    power-of-two scales: every product and every fp32 partial sum is then exact."""
    wl = inp["wl"]
    g = torch.Generator().manual_seed(seed)
    dev = inp["k_pool"].device
    q = torch.randint(-8, 9, tuple(inp["q_li"].shape), generator=g).float()
    k = torch.randint(-8, 9, tuple(inp["k_pool"].shape), generator=g).float()
    qs = (2.0 ** torch.randint(-3, 2, (wl.n_q,), generator=g).float())
    ks = (2.0 ** torch.randint(-3, 2, tuple(inp["k_pool"].shape[:2]), generator=g).float())
    w = torch.randint(1, 5, (wl.n_q, wl.H_I), generator=g).float()
    out = dict(inp)
    out["wl"] = di.Workload(**{**wl.__dict__, "li_dtype": "fp8", "name": wl.name + "_intfp8"})
    out["q_li"] = q.to(torch.float8_e4m3fn).to(dev)
    out["k_pool"] = k.to(torch.float8_e4m3fn).to(dev)
    out["q_scale"] = qs[:, None].expand(wl.n_q, wl.H_I).contiguous().to(dev)
    out["k_scale"] = ks.contiguous().to(dev)
    out["w"] = w.to(dev)
    return out
