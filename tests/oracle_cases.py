"""Hand-built tiny problems for the oracle pins (CPU tensors in the dsa_inputs layout)."""
import math

import torch

import dsa_inputs as di


def bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def li_problem(q, w, keys_by_pos, page_size, page_table, seq_len, n_new=1, K=4,
               fp8=None):
    """One sequence; every new token uses the same q [H_I, d_I] and w [H_I]."""
    q = torch.tensor(q, dtype=torch.float32)
    H_I, d_I = q.shape
    L = len(keys_by_pos)
    pages = (L + page_size - 1) // page_size
    wl = di.Workload("hand", [seq_len], [n_new], H_I=H_I, d_I=d_I, K=K, H=1,
                     li_dtype="fp8" if fp8 else "bf16", page_size=page_size)
    pool = torch.zeros((pages, page_size, d_I), dtype=torch.float32)
    for j, k in enumerate(keys_by_pos):
        pool[page_table[j // page_size], j % page_size] = torch.tensor(k, dtype=torch.float32)
    inp = {"wl": wl, "pt_k": torch.tensor([page_table], dtype=torch.int32),
           "seq_lens": torch.tensor([seq_len], dtype=torch.int32),
           "q_start": torch.tensor([0, n_new], dtype=torch.int32),
           "w": torch.tensor([w] * n_new, dtype=torch.float32)}
    if fp8:
        inp["q_li"] = torch.tensor([fp8["q_codes"]] * n_new, dtype=torch.uint8).view(torch.float8_e4m3fn)
        inp["q_scale"] = torch.full((n_new, H_I), fp8["q_scale"], dtype=torch.float32)
        kc = torch.zeros((pages, page_size, d_I), dtype=torch.uint8)
        for j, k in enumerate(fp8["k_codes_by_position"]):
            kc[page_table[j // page_size], j % page_size] = torch.tensor(k, dtype=torch.uint8)
        inp["k_pool"] = kc.view(torch.float8_e4m3fn)
        inp["k_scale"] = torch.full((pages, page_size), fp8["k_scale"], dtype=torch.float32)
    else:
        inp["q_li"] = q[None].expand(n_new, H_I, d_I).contiguous().to(torch.bfloat16)
        inp["k_pool"] = pool.to(torch.bfloat16)
        inp["q_scale"] = None
        inp["k_scale"] = None
    return inp


def li_problem_mx(q_blocks, w, k_blocks_by_pos, page_size, page_table, group, K=4):
    """One sequence, one new token at the last position, MXFP8 inputs: q_blocks[h][g] and
    k_blocks_by_pos[j][g] give the e4m3 code shared by all elements of group g and its E8M0
    scale byte."""
    H_I, n_grp = len(q_blocks), len(q_blocks[0])
    d_I = n_grp * group
    L = len(k_blocks_by_pos)
    pages = (L + page_size - 1) // page_size
    wl = di.Workload("hand_mx", [L], [1], H_I=H_I, d_I=d_I, K=K, H=1, li_dtype="mxfp8",
                     page_size=page_size)
    qc = torch.zeros((1, H_I, d_I), dtype=torch.uint8)
    qsf = torch.zeros((1, H_I, n_grp), dtype=torch.uint8)
    for h in range(H_I):
        for g, blk in enumerate(q_blocks[h]):
            qc[0, h, g * group:(g + 1) * group] = blk["code"]
            qsf[0, h, g] = blk["sf"]
    kc = torch.zeros((pages, page_size, d_I), dtype=torch.uint8)
    ksf = torch.full((pages, page_size, n_grp), 127, dtype=torch.uint8)
    for j, blocks in enumerate(k_blocks_by_pos):
        pg, r = page_table[j // page_size], j % page_size
        for g, blk in enumerate(blocks):
            kc[pg, r, g * group:(g + 1) * group] = blk["code"]
            ksf[pg, r, g] = blk["sf"]
    return {"wl": wl, "pt_k": torch.tensor([page_table], dtype=torch.int32),
            "seq_lens": torch.tensor([L], dtype=torch.int32),
            "q_start": torch.tensor([0, 1], dtype=torch.int32),
            "w": torch.tensor([w], dtype=torch.float32),
            "q_li": qc.view(torch.float8_e4m3fn), "q_sf": qsf,
            "k_pool": kc.view(torch.float8_e4m3fn), "k_sf": ksf,
            "q_scale": None, "k_scale": None}


def sfa_problem(q_heads, rows_by_pos, page_size, page_table, d_v, scale, n_new=1, K=2):
    """One sequence with len(rows_by_pos) positions; q_heads [H, d_qk] for every new token."""
    q = torch.tensor(q_heads, dtype=torch.float32)
    H, d_qk = q.shape
    L = len(rows_by_pos)
    pages = (L + page_size - 1) // page_size
    wl = di.Workload("hand", [L], [n_new], H_I=1, d_I=1, K=K, H=H, page_size=page_size,
                     d_qk=d_qk, d_v=d_v, softmax_scale=scale)
    pool = torch.zeros((pages, page_size, d_qk), dtype=torch.float32)
    for j, r in enumerate(rows_by_pos):
        pool[page_table[j // page_size], j % page_size] = torch.tensor(r, dtype=torch.float32)
    return {"wl": wl, "q_sfa": q[None].expand(n_new, H, d_qk).contiguous().to(torch.bfloat16),
            "kv_pool": pool.to(torch.bfloat16),
            "pt_kv": torch.tensor([page_table], dtype=torch.int32),
            "seq_lens": torch.tensor([L], dtype=torch.int32),
            "q_start": torch.tensor([0, n_new], dtype=torch.int32), "softmax_scale": scale}
