"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to a hand-worked value, a closed form, a library routine,
a brute-force check of the definition, or an invariant, chosen so that a plausible mistake
(a dropped ReLU or weight, a wrong index, a transposed operand, a reversed tie-break, an
off-by-one in the causal limit, a wrong page translation, a missing scale) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import dsa_inputs as di
import oracle
from oracle_cases import li_problem, li_problem_mx, sfa_problem

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- number formats

def test_bf16_decoder_matches_torch_on_every_pattern():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_bf16(b) for b in range(1 << 16)])
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[fin], got[fin])


def test_e4m3_decoder_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.decode_e4m3(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert oracle.decode_e4m3(0x7E) == 448.0 and oracle.decode_e4m3(0x01) == 2.0 ** -9


# ---------------------------------------------------------------- indexer: hand-worked example

def _hand(fp8=False, n_new=1, K=4, seq_len=None):
    g = _gold("li_hand_example.json")
    keys = g["keys_by_position"]
    return g, li_problem(g["q"], g["w"], keys, g["page_size"], g["page_table"],
                         seq_len or len(keys), n_new=n_new, K=K, fp8=g["fp8"] if fp8 else None)


@pytest.mark.parametrize("fp8", [False, True])
def test_indexer_hand_example_scores(fp8):
    g, inp = _hand(fp8)
    s, _ = oracle.li_scores(inp, 0)
    assert s.tolist() == g["scores"]


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6])
def test_indexer_hand_example_topk(fp8, K):
    g, inp = _hand(fp8, K=K)
    idx, cnt, _ = oracle.li_topk(inp)
    assert idx[0].tolist() == g["topk_full_context"][str(K)]
    assert cnt[0] == min(K, 5)


@pytest.mark.parametrize("K", [2, 4])
def test_indexer_hand_example_causal_two_tokens(K):
    g, inp = _hand(n_new=2, K=K)
    idx, cnt, _ = oracle.li_topk(inp)
    c = g["causal_two_tokens"]
    assert idx[0].tolist() == c["token0"][str(K)]
    assert idx[1].tolist() == c["token1"][str(K)]
    assert cnt.tolist() == [min(K, 4), min(K, 5)]


# ---------------------------------------------------------------- indexer: closed forms

def _random_li(seed, B=2, L=(70, 131), n_new=(1, 2), H_I=4, d_I=16, K=8, values="int4",
               page_size=8, li_dtype="bf16"):
    wl = di.Workload("t", list(L), list(n_new), H_I=H_I, d_I=d_I, K=K, H=2, values=values,
                     w_values="int14" if values == "int4" else "normal", seed=seed,
                     page_size=page_size, li_dtype=li_dtype, d_qk=32, d_v=16)
    return di.generate(wl)


def _key_rows(inp, b, n):
    """Logical key rows 0..n-1 of sequence b, read through the page table (float64)."""
    wl = inp["wl"]
    pt = inp["pt_k"][b]
    pool = inp["k_pool"].to(torch.float64)
    rows = [pool[int(pt[j // wl.page_size]), j % wl.page_size] for j in range(n)]
    out = torch.stack(rows)
    if inp.get("k_scale") is not None:
        ks = inp["k_scale"].to(torch.float64)
        out = out * torch.stack([ks[int(pt[j // wl.page_size]), j % wl.page_size]
                                 for j in range(n)])[:, None]
    return out


def test_indexer_unit_query_reads_one_key_coordinate():
    """q_h = e_d and w = one-hot(h) make s_j = w_h * max(0, k_j[d]): checks ReLU, head weight
    and the (head, dim) indexing without the dot-product formula."""
    inp = _random_li(11, H_I=4, d_I=16)
    wl = inp["wl"]
    for (h, d, wh) in [(0, 0, 3.0), (2, 5, 1.0), (3, 15, 2.0)]:
        q = torch.zeros(wl.n_q, wl.H_I, wl.d_I)
        q[:, h, d] = 1.0
        w = torch.zeros(wl.n_q, wl.H_I)
        w[:, h] = wh
        inp2 = dict(inp, q_li=q.to(torch.bfloat16), w=w)
        t = wl.n_q - 1  # last token of the last sequence sees all its positions
        s, _ = oracle.li_scores(inp2, t)
        keys = _key_rows(inp, wl.B - 1, len(s))
        expect = wh * torch.clamp(keys[:, d], min=0.0)
        assert np.array_equal(s, expect.numpy())


def test_indexer_scores_head_permutation_and_weight_scaling():
    inp = _random_li(12, values="normal")
    wl = inp["wl"]
    t = wl.n_q - 1
    s0, _ = oracle.li_scores(inp, t)
    perm = torch.tensor([2, 0, 3, 1])
    inp_p = dict(inp, q_li=inp["q_li"][:, perm].contiguous(), w=inp["w"][:, perm].contiguous())
    sp, _ = oracle.li_scores(inp_p, t)
    np.testing.assert_allclose(sp, s0, rtol=1e-12, atol=1e-12)
    inp_s = dict(inp, w=inp["w"] * 4.0)
    ss, _ = oracle.li_scores(inp_s, t)
    np.testing.assert_allclose(ss, 4.0 * s0, rtol=1e-12, atol=1e-12)
    # zero head weights give zero scores everywhere
    inp_n = dict(inp, w=torch.zeros_like(inp["w"]))
    sn, _ = oracle.li_scores(inp_n, t)
    assert not np.any(sn)


def test_indexer_scores_match_library_matmul_on_integers():
    """Integer inputs make every sum exact, so the oracle must equal a torch int64 matmul of the
    logical keys (a library routine) with ReLU and the weights applied."""
    inp = _random_li(13)
    wl = inp["wl"]
    for t, (b, p) in enumerate([(b, p) for b in range(wl.B)
                                for p in range(wl.seq_lens[b] - wl.n_new[b], wl.seq_lens[b])]):
        s, _ = oracle.li_scores(inp, t)
        assert len(s) == p + 1
        keys = _key_rows(inp, b, p + 1).to(torch.int64)
        q = inp["q_li"][t].to(torch.float64).to(torch.int64)
        dots = torch.matmul(keys, q.T)                       # [p+1, H_I]
        w = inp["w"][t].to(torch.float64).to(torch.int64)
        expect = (torch.clamp(dots, min=0) * w).sum(1)
        assert np.array_equal(s, expect.numpy().astype(np.float64))


def test_fp8_scores_equal_dequantised_bf16_scores():
    """e4m3 codes of small integers with power-of-two scales dequantise exactly; the fp8 oracle
    must then agree exactly with the bf16 oracle fed the dequantised values."""
    inp = _random_li(14)
    wl = inp["wl"]
    g = torch.Generator().manual_seed(5)
    qs = torch.tensor([0.5, 0.25, 2.0])[torch.randint(0, 3, (wl.n_q,), generator=g)]
    ks = torch.tensor([0.125, 1.0, 4.0])[torch.randint(0, 3, inp["k_pool"].shape[:2], generator=g)]
    q8 = (inp["q_li"].float() / qs[:, None, None]).to(torch.float8_e4m3fn)
    k8 = (inp["k_pool"].float() / ks[:, :, None]).to(torch.float8_e4m3fn)
    assert torch.equal(q8.float() * qs[:, None, None], inp["q_li"].float())
    assert torch.equal(k8.float() * ks[:, :, None], inp["k_pool"].float())
    wl8 = di.Workload(**{**wl.__dict__, "li_dtype": "fp8"})
    inp8 = dict(inp, wl=wl8, q_li=q8, k_pool=k8, q_scale=qs[:, None].expand(wl.n_q, wl.H_I).contiguous(),
                k_scale=ks.contiguous())
    a = oracle.li_topk(inp)
    b = oracle.li_topk(inp8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


# ---------------------------------------------------------------- indexer: MXFP8 inputs

def test_e8m0_decoder_matches_its_definition_on_every_code():
    """E8M0 (OCP Microscaling): 2^(code - 127), code 255 is NaN; torch's decoder where present."""
    got = np.array([oracle.decode_e8m0(c) for c in range(256)])
    assert np.isnan(got[255]) and not np.isnan(got[:255]).any()
    assert all(got[c] == math.ldexp(1.0, c - 127) for c in range(255))
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu)
        ref = ref.to(torch.float64).numpy()
        assert np.array_equal(ref[:255], got[:255]) and np.isnan(ref[255])


def _hand_mx(K=4):
    g = _gold("li_mx_hand_example.json")
    return g, li_problem_mx(g["q_blocks"], g["w"], g["k_blocks_by_position"], g["page_size"],
                            g["page_table"], g["group"], K=K)


def test_mx_hand_example_scores():
    g, inp = _hand_mx()
    s, _ = oracle.li_scores(inp, 0)
    assert s.tolist() == g["scores"]


@pytest.mark.parametrize("K", [1, 2, 3, 4, 5, 6])
def test_mx_hand_example_topk(K):
    g, inp = _hand_mx(K=K)
    idx, cnt, _ = oracle.li_topk(inp)
    assert idx[0].tolist() == g["topk_full_context"][str(K)]
    assert cnt[0] == min(K, 5)


def _mx_dequant(codes, sf):
    """Library decode (torch's e4m3) times 2^(sf - 127) repeated over each group of 32."""
    v = codes.to(torch.float64)
    e = sf.to(torch.int64) - 127
    return v * torch.pow(2.0, e.to(torch.float64)).repeat_interleave(32, dim=-1)


def test_mx_scores_match_library_matmul_on_integers():
    """Integer e4m3 codes and scales in 2^-1..2^1 keep every sum exact: the oracle equals a torch
    matmul of the library-dequantised logical keys with ReLU and the weights applied."""
    inp = _random_li(15, d_I=64, li_dtype="mxfp8")
    wl = inp["wl"]
    assert set(torch.unique(inp["k_sf"]).tolist()) <= {126, 127, 128}
    pt = inp["pt_k"]
    for t, (b, p) in enumerate([(b, p) for b in range(wl.B)
                                for p in range(wl.seq_lens[b] - wl.n_new[b], wl.seq_lens[b])]):
        s, _ = oracle.li_scores(inp, t)
        rows = [(int(pt[b, j // wl.page_size]), j % wl.page_size) for j in range(p + 1)]
        keys = torch.stack([_mx_dequant(inp["k_pool"][a, r], inp["k_sf"][a, r]) for a, r in rows])
        q = _mx_dequant(inp["q_li"][t], inp["q_sf"][t])          # [H_I, d_I]
        dots = keys @ q.T
        expect = (torch.clamp(dots, min=0) * inp["w"][t].to(torch.float64)).sum(1)
        assert np.array_equal(s, expect.numpy())


def test_mx_with_one_exponent_per_row_equals_per_token_fp8():
    """When all groups of a query token (every head) share one exponent and all groups of a key
    row share one, MXFP8 is the per-token/per-row scaled e4m3 format pinned above."""
    inp = _random_li(16, d_I=64, li_dtype="mxfp8")
    wl = inp["wl"]
    g = torch.Generator().manual_seed(7)
    eq = torch.randint(124, 131, (wl.n_q,), generator=g).to(torch.uint8)
    ek = torch.randint(124, 131, tuple(inp["k_pool"].shape[:2]), generator=g).to(torch.uint8)
    mx = dict(inp, q_sf=eq[:, None, None].expand(wl.n_q, wl.H_I, 2).contiguous(),
              k_sf=ek[:, :, None].expand(*ek.shape, 2).contiguous())
    wl8 = di.Workload(**{**wl.__dict__, "li_dtype": "fp8"})
    f8 = dict(inp, wl=wl8, q_sf=None, k_sf=None,
              q_scale=torch.pow(2.0, eq.double() - 127).float()[:, None].expand(wl.n_q, wl.H_I).contiguous(),
              k_scale=torch.pow(2.0, ek.double() - 127).float().contiguous())
    for t in range(wl.n_q):
        assert np.array_equal(oracle.li_scores(mx, t)[0], oracle.li_scores(f8, t)[0])
    a, b = oracle.li_topk(mx), oracle.li_topk(f8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


@pytest.mark.parametrize("grp", [0, 1])
def test_mx_group_scale_scales_only_its_own_group(grp):
    """One head, unit weight, non-negative codes (so s is the dot product itself): doubling the
    scale of group g of a key row adds exactly that group's share, which is what zeroing the
    group's codes removes.  Doubling group g of the query does the same for every key."""
    inp = _random_li(17, d_I=64, H_I=1, li_dtype="mxfp8")
    wl = inp["wl"]
    inp = dict(inp, q_li=inp["q_li"].float().abs().to(torch.float8_e4m3fn),
               k_pool=inp["k_pool"].float().abs().to(torch.float8_e4m3fn),
               w=torch.ones_like(inp["w"]))
    t = wl.n_q - 1
    s0, _ = oracle.li_scores(inp, t)
    kz = inp["k_pool"].float().clone()
    kz[..., grp * 32:(grp + 1) * 32] = 0
    s_without, _ = oracle.li_scores(dict(inp, k_pool=kz.to(torch.float8_e4m3fn)), t)
    share = s0 - s_without
    assert np.all(share >= 0) and np.any(share > 0)
    ksf = inp["k_sf"].clone()
    ksf[..., grp] += 1
    s_k, _ = oracle.li_scores(dict(inp, k_sf=ksf), t)
    assert np.array_equal(s_k, s0 + share)
    qsf = inp["q_sf"].clone()
    qsf[t, :, grp] += 1
    s_q, _ = oracle.li_scores(dict(inp, q_sf=qsf), t)
    assert np.array_equal(s_q, s0 + share)


def test_mx_generator_quantiser_follows_the_format():
    """The input generator's MX quantiser: each group's largest code lies in [256, 448] (the
    shared exponent is floor(log2 amax) - 8); codes below the clamp are within e4m3's half-ulp
    (2^-4 relative) of x / 2^shared, clamped ones are +-448."""
    x = torch.randn(6, 4, 128, generator=torch.Generator().manual_seed(3)).double()
    q, sf = di._quant_mx(x.float())
    codes = q.double()
    assert codes.view(6, 4, 4, 32).abs().amax(-1).min() >= 256
    assert codes.abs().max() <= 448
    scaled = x / torch.pow(2.0, sf.double() - 127).repeat_interleave(32, -1)
    clamped = scaled.abs() > 448
    assert torch.all(codes[clamped].abs() == 448)
    normal = ~clamped & (scaled.abs() >= 2.0 ** -6)
    assert torch.all((codes - scaled).abs()[normal] <= scaled.abs()[normal] * 2.0 ** -4)


# ---------------------------------------------------------------- Indexer Prolog

@pytest.mark.parametrize("case", range(4))
def test_mx_quantiser_hand_cases(case):
    c = _gold("mx_quant_hand_cases.json")["cases"][case]
    v = np.zeros(32)
    v[:len(c["values"])] = c["values"]
    codes, sf = oracle.mx_quantize(v)
    assert sf.tolist() == [c["sf"]]
    assert codes[:len(c["codes"])].tolist() == c["codes"]
    assert not codes[len(c["codes"]):].any()


def test_mx_quantiser_rounding_matches_torch_e4m3_conversion():
    """Element rounding against torch's float8_e4m3fn conversion (round to nearest even) of the
    values divided by the group scale, over groups spanning 2^-20 .. 2^20 in magnitude."""
    g = np.random.default_rng(4)
    v = g.standard_normal(32 * 64) * np.repeat(2.0 ** g.integers(-20, 21, 64), 32)
    codes, sf = oracle.mx_quantize(v)
    scale = np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32)
    y = torch.tensor(v / scale).clamp(-448, 448)
    ref = y.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()  # v/scale exact in fp32
    ref = np.where(ref == 0x80, 0, ref)  # -0 -> +0, as the quantiser emits
    assert np.array_equal(codes, ref)
    amax = np.abs(v).reshape(64, 32).max(1)
    assert np.all((amax / np.ldexp(1.0, sf.astype(np.int64) - 127) >= 256) &
                  (amax / np.ldexp(1.0, sf.astype(np.int64) - 127) < 512))


def _prolog_small(values="normal", li_dtype="mxfp8", **over):
    kw = dict(seq_lens=[300, 130, 65], n_new=[1, 2, 3], d_q=64, d_model=96, values=values,
              li_dtype=li_dtype)
    kw.update(over)
    wl = di.small("prolog_decode_32k", **kw)
    return di.generate_prolog(wl)


@pytest.mark.parametrize("values", ["int4", "normal"])
def test_prolog_projections_match_library_matmul(values):
    inp = _prolog_small(values)
    r = oracle.prolog(inp)
    q = (inp["xq"].double() @ inp["w_q"].double().T).numpy()
    w = inp["w_scale"] * (inp["x"].double() @ inp["w_w"].double().T).numpy()
    if values == "int4":
        assert np.array_equal(r["q_val"], q) and np.array_equal(r["w"], w)
    else:
        np.testing.assert_allclose(r["q_val"], q, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["w"], w, rtol=1e-12, atol=1e-14)


def test_prolog_layernorm_matches_torch():
    inp = _prolog_small()
    r = oracle.prolog(inp)
    z = inp["x"].double() @ inp["w_k"].double().T
    ref = torch.nn.functional.layer_norm(z, (z.shape[1],), inp["ln_gamma"].double(),
                                         inp["ln_beta"].double(), eps=inp["ln_eps"])
    np.testing.assert_allclose(r["k_val"], ref.numpy(), rtol=1e-11, atol=1e-12)


def test_prolog_layernorm_closed_forms():
    """Identical K-projection rows make every feature equal: the normalised key is beta.  With
    eps = 0, scaling the activations leaves the normalised key unchanged."""
    inp = _prolog_small()
    same = dict(inp, w_k=inp["w_k"][:1].expand_as(inp["w_k"]).contiguous())
    r = oracle.prolog(same)
    np.testing.assert_allclose(r["k_val"], np.broadcast_to(inp["ln_beta"].double().numpy(),
                                                           r["k_val"].shape), atol=1e-12)
    a = oracle.prolog(dict(inp, ln_eps=0.0))
    b = oracle.prolog(dict(inp, ln_eps=0.0, x=(inp["x"].float() * 4).to(torch.bfloat16)))
    np.testing.assert_allclose(a["k_val"], b["k_val"], rtol=1e-12, atol=1e-12)


def test_prolog_encodings_and_cache_rows():
    """MX outputs are the pinned quantiser applied per head / per key; bf16 outputs on
    integer inputs are the exact values; each token's key goes to its position's row."""
    inp = _prolog_small()
    wl = inp["wl"]
    r = oracle.prolog(inp)
    for t in range(wl.n_q):
        c, s = oracle.mx_quantize(r["q_val"][t])
        assert np.array_equal(c, r["q_enc"][t]) and np.array_equal(s, r["q_sf"][t])
        c, s = oracle.mx_quantize(r["k_val"][t])
        assert np.array_equal(c, r["k_enc"][t]) and np.array_equal(s, r["k_sf"][t])
    pos = di.token_positions(wl)
    seq = [b for b, n in enumerate(wl.n_new) for _ in range(n)]
    pt = inp["pt_k"]
    assert r["k_row"].tolist() == [int(pt[b, p // 64]) * 64 + p % 64 for b, p in zip(seq, pos)]
    ib = _prolog_small("int4", li_dtype="bf16")
    rb = oracle.prolog(ib)
    qb = torch.tensor(rb["q_val"]).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(rb["q_enc"], qb)  # integers below 2^8 are exact in bf16


# ---------------------------------------------------------------- FP8 latent cache

def test_kv8_row_hand_decoding():
    g = _gold("kv8_hand_row.json")
    row = np.zeros(608, dtype=np.uint8)
    row[576:596] = np.array(g["scales"], dtype=np.float32).view(np.uint8)
    for e in g["elements"]:
        row[e["d"]] = e["code"]
    for e in g["elements"]:
        assert oracle.decode_kv8(row, e["d"]) == e["value"], e
    assert oracle.decode_kv8(row, 2) == 0.0  # code 0


def test_sfa_on_fp8_cache_equals_bf16_cache_of_the_dequantised_values():
    """Power-of-two tile scales and small integer codes de-quantise exactly, so attention over
    the FP8 rows must equal the pinned bf16 attention over a cache holding those values."""
    wl = di.Workload("kv8", [70, 130], [1, 2], H_I=2, d_I=8, K=16, H=3, values="int4", seed=51,
                     kv_dtype="fp8")
    inp = di.generate(wl)
    g = torch.Generator().manual_seed(9)
    n = wl.num_pages * wl.page_size
    codes = torch.randint(-6, 7, (n, 576), generator=g).float()
    scales = 2.0 ** torch.randint(-3, 3, (n, 5), generator=g).float()
    rows = torch.zeros((n, 608), dtype=torch.uint8)
    rows[:, :576] = codes.to(torch.float8_e4m3fn).view(torch.uint8)
    rows[:, 576:596] = scales.contiguous().view(torch.uint8).view(n, 20)
    vals = codes * scales.repeat_interleave(128, 1)[:, :576]
    kv8 = dict(inp, kv8_pool=rows.view(wl.num_pages, wl.page_size, 608))
    bf = dict(inp, wl=di.Workload(**{**wl.__dict__, "kv_dtype": "bf16"}),
              kv_pool=vals.to(torch.bfloat16).view(wl.num_pages, wl.page_size, 576))
    assert torch.equal(vals.to(torch.bfloat16).float(), vals)  # exactly representable
    sets = [[0, 5, 33, 69, -1, 12], [129, 64, 1, -1, -1, 100], [7, 8, 9, 10, 128, 127]]
    a, b = oracle.sfa(kv8, sets), oracle.sfa(bf, sets)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_kv8_generator_tiles():
    """Each tile's largest code is +-448 (scale = amax / 448), and de-quantised rows stay within
    e4m3's half step (2^-4 relative) of the bf16 cache they were made from."""
    wl = di.small("decode_32k", seq_lens=[200], n_new=[1], kv_dtype="fp8")
    inp = di.generate(wl)
    rows = inp["kv8_pool"].view(-1, 608)
    codes = rows[:, :576].view(torch.float8_e4m3fn).float()
    for i in range(5):
        assert torch.all(codes[:, 128 * i:128 * (i + 1)].abs().amax(1) == 448)
    ref = inp["kv_pool"].view(-1, 576).float()
    r = rows[:4].numpy()
    got = torch.tensor([[oracle.decode_kv8(r[k], d) for d in range(576)] for k in range(4)])
    assert torch.all((got - ref[:4]).abs() <= ref[:4].abs() * 2.0 ** -4 * 1.01 + 2.0 ** -12)


# ---------------------------------------------------------------- top-K: definition by brute force

def _check_selection(s, idx_row, cnt, K):
    p1 = len(s)
    m = min(K, p1)
    assert cnt == m
    sel = [j for j in idx_row if j >= 0]
    assert len(sel) == m and list(idx_row[m:]) == [-1] * (K - m)
    assert sel == sorted(sel) and len(set(sel)) == m
    assert all(0 <= j < p1 for j in sel)
    chosen = np.zeros(p1, bool)
    chosen[sel] = True
    # every chosen position beats every other one: larger score, or equal score and lower index
    for j in np.nonzero(chosen)[0]:
        others = np.nonzero(~chosen)[0]
        if len(others) == 0:
            break
        assert np.all((s[j] > s[others]) | ((s[j] == s[others]) & (j < others)))
    # and the same set as a library sort (numpy lexsort: score descending, position ascending)
    order = np.lexsort((np.arange(p1), -s))
    assert sorted(order[:m].tolist()) == sel


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("K", [1, 5, 64, 200])
def test_topk_is_the_definition_on_random_tiny_cases(seed, K):
    inp = _random_li(100 + seed, K=K, values="int4" if seed % 2 == 0 else "normal")
    wl = inp["wl"]
    idx, cnt, _ = oracle.li_topk(inp)
    for t in range(wl.n_q):
        s, _ = oracle.li_scores(inp, t)
        _check_selection(s, idx[t], cnt[t], K)


def test_topk_all_scores_equal_takes_lowest_positions():
    inp = _random_li(21, K=10)
    inp = dict(inp, w=torch.zeros_like(inp["w"]))  # every score is exactly 0
    idx, cnt, _ = oracle.li_topk(inp)
    for t in range(inp["wl"].n_q):
        assert idx[t].tolist() == list(range(10))


def test_topk_relu_killed_scores_and_negative_zero():
    """Queries that make every dot product <= 0 give all-zero scores (some -0.0 after the
    weighting with negative weights): ties again resolve to the lowest positions."""
    inp = _random_li(22, K=7)
    keys_all = inp["k_pool"].float()
    inp = dict(inp, k_pool=keys_all.abs().to(torch.bfloat16),
               q_li=(-inp["q_li"].float().abs()).to(torch.bfloat16),
               w=-inp["w"].abs())
    idx, _, _ = oracle.li_topk(inp)
    for t in range(inp["wl"].n_q):
        assert idx[t].tolist() == list(range(7))


def test_topk_k_at_least_context_returns_every_visible_position():
    inp = _random_li(23, L=(20, 9), n_new=(2, 1), K=64, page_size=4)
    wl = inp["wl"]
    idx, cnt, _ = oracle.li_topk(inp)
    pos = di.token_positions(wl)
    for t in range(wl.n_q):
        assert idx[t].tolist() == list(range(pos[t] + 1)) + [-1] * (64 - pos[t] - 1)


def test_causal_draft_sees_last_position_verified_does_not():
    """Two new tokens; the key at the last position is made the best for both queries. The draft
    (second) token must select it, the verified (first) token must not."""
    inp = _random_li(24, L=(40,), n_new=(2,), K=3, page_size=8)
    wl = inp["wl"]
    k = inp["k_pool"].float()
    pt = inp["pt_k"][0]
    L = wl.seq_lens[0]
    k[int(pt[(L - 1) // 8]), (L - 1) % 8] = 4.0  # all-positive key: dot with int4 q is large
    q = inp["q_li"].float().abs()
    inp = dict(inp, k_pool=k.to(torch.bfloat16), q_li=q.to(torch.bfloat16))
    idx, _, _ = oracle.li_topk(inp)
    assert L - 1 in idx[1].tolist()
    assert all(j <= L - 2 for j in idx[0].tolist())


def test_page_table_permutation_invariance():
    inp = _random_li(25, L=(200, 77), n_new=(1, 3), K=16)
    inp2 = di.repage(inp, seed=99)
    assert not torch.equal(inp["pt_k"], inp2["pt_k"])
    a = oracle.li_topk(inp)
    b = oracle.li_topk(inp2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])
    oa = oracle.sfa(inp, a[0])
    ob = oracle.sfa(inp2, a[0])
    assert np.array_equal(oa[0], ob[0]) and np.array_equal(oa[1], ob[1])


def test_poisoned_rows_past_length_are_never_visible():
    """The generator makes rows past seq_len 4x larger; they must not change any score."""
    inp = _random_li(26, L=(61,), n_new=(1,), K=8, page_size=16)
    wl = inp["wl"]
    s, _ = oracle.li_scores(inp, 0)
    assert len(s) == 61
    k = inp["k_pool"].clone()
    pt = inp["pt_k"][0]
    k[int(pt[3]), 13:] = 0  # the poison rows of the last page
    s2, _ = oracle.li_scores(dict(inp, k_pool=k), 0)
    assert np.array_equal(s, s2)


# ---------------------------------------------------------------- SFA

def test_sfa_hand_example():
    g = _gold("sfa_hand_example.json")
    inp = sfa_problem([g["q"]], g["rows_by_position"], g["page_size"], g["page_table"],
                      g["d_v"], g["scale"], K=2)
    for case in g["cases"]:
        out, lse = oracle.sfa(inp, [case["idx"]])
        np.testing.assert_allclose(out[0, 0], case["out"], rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(lse[0, 0], case["lse"], rtol=1e-14, atol=1e-14)


def _random_sfa(seed, L=(50, 90), n_new=(1, 2), H=3, d_qk=24, d_v=16, page_size=8):
    wl = di.Workload("t", list(L), list(n_new), H_I=2, d_I=8, K=4, H=H, seed=seed,
                     page_size=page_size, d_qk=d_qk, d_v=d_v, softmax_scale=1 / math.sqrt(d_qk))
    return di.generate(wl)


def _latent_rows(inp, b, js):
    wl = inp["wl"]
    pt = inp["pt_kv"][b]
    pool = inp["kv_pool"].to(torch.float64)
    return torch.stack([pool[int(pt[j // wl.page_size]), j % wl.page_size] for j in js])


def test_sfa_zero_query_gives_mean_of_selected_values():
    inp = _random_sfa(31)
    inp = dict(inp, q_sfa=torch.zeros_like(inp["q_sfa"]))
    wl = inp["wl"]
    sets = [[0, 3, 17, -1, 40, -1], [5, -1, -1, -1, -1, -1], [1, 2, 3, 4, 5, 60]]
    out, lse = oracle.sfa(inp, sets)
    seq_of = [0, 1, 1]
    for t in range(3):
        js = [j for j in sets[t] if j >= 0]
        mean = _latent_rows(inp, seq_of[t], js)[:, :wl.d_v].mean(0)
        for h in range(wl.H):
            np.testing.assert_allclose(out[t, h], mean.numpy(), rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[t, h], math.log(len(js)), rtol=1e-14)


def test_sfa_single_row_returns_that_row():
    inp = _random_sfa(32)
    wl = inp["wl"]
    out, lse = oracle.sfa(inp, [[-1, 33, -1], [7, -1, -1], [-1, -1, 89]])
    for t, (b, j) in enumerate([(0, 33), (1, 7), (1, 89)]):
        row = _latent_rows(inp, b, [j])[0]
        for h in range(wl.H):
            assert np.array_equal(out[t, h], row[:wl.d_v].numpy())


def test_sfa_equals_library_dense_attention_when_k_covers_context():
    """K >= visible context: SFA is dense causal attention; compare with torch's
    scaled_dot_product_attention (fp64, CPU) over the logical rows."""
    inp = _random_sfa(33, L=(37, 64), n_new=(2, 3))
    wl = inp["wl"]
    pos = di.token_positions(wl)
    seq_of = [0, 0, 1, 1, 1]
    K = 64
    sets = [list(range(p + 1)) + [-1] * (K - p - 1) for p in pos]
    out, lse = oracle.sfa(inp, sets)
    for t in range(wl.n_q):
        rows = _latent_rows(inp, seq_of[t], range(pos[t] + 1))     # [n, d_qk]
        q = inp["q_sfa"][t].to(torch.float64)                        # [H, d_qk]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :], rows[None, None].expand(1, wl.H, -1, -1),
            rows[None, None, :, :wl.d_v].expand(1, wl.H, -1, -1), scale=wl.softmax_scale)
        np.testing.assert_allclose(out[t], ref[0, :, 0].numpy(), rtol=1e-11, atol=1e-12)
        z = wl.softmax_scale * (q @ rows.T)
        np.testing.assert_allclose(lse[t], torch.logsumexp(z, 1).numpy(), rtol=1e-12)


def test_sfa_two_rows_equal_logits_average():
    inp = _random_sfa(34, L=(16,), n_new=(1,), H=1, d_qk=8, d_v=4, page_size=4)
    q = inp["q_sfa"].clone()
    q[:, :, :4] = 0  # logits then depend on dims 4..7 only
    inp = dict(inp, q_sfa=q)
    kv = inp["kv_pool"].float()
    pt = inp["pt_kv"][0]
    # make rows 2 and 9 share their key part (equal logits) but differ in value
    r2 = kv[int(pt[0]), 2].clone()
    kv[int(pt[2]), 1, 4:] = r2[4:]
    inp = dict(inp, kv_pool=kv.to(torch.bfloat16))
    out, lse = oracle.sfa(inp, [[2, 9]])
    rows = _latent_rows(inp, 0, [2, 9])
    np.testing.assert_allclose(out[0, 0], rows[:, :4].mean(0).numpy(), rtol=1e-13, atol=1e-13)


def test_sfa_rejects_out_of_range_index():
    inp = _random_sfa(35)
    with pytest.raises(ValueError):
        oracle.sfa(inp, [[50, -1], [0, 1], [0, 1]])


def test_fp8_latent_cache_page_permutation_invariance():
    wl = di.Workload("kv8p", [90, 150], [1, 2], H_I=2, d_I=8, K=16, H=2, seed=61, d_qk=576,
                     d_v=512, page_size=16, kv_dtype="fp8")
    inp = di.generate(wl)
    inp2 = di.repage(inp, seed=5)
    assert not torch.equal(inp["pt_kv"], inp2["pt_kv"])
    sets = [[0, 3, 89, -1], [5, 149, 77, 100], [1, 2, 148, 149]]
    a, b = oracle.sfa(inp, sets), oracle.sfa(inp2, sets)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_kv8_decoding_matches_library_roundings_on_every_code():
    """bf16(fp32(code * scale)) for all 256 codes and many scales, against numpy's float32
    product and torch's round-to-nearest-even float32 -> bfloat16 conversion."""
    g = np.random.default_rng(8)
    scales = np.concatenate([g.uniform(1e-4, 3.0, 40), 2.0 ** g.integers(-20, 10, 8),
                             [1.0 / 3.0, 0.1, 448.0 / 7.0]]).astype(np.float32)
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    fin = ~np.isnan(vals)
    row = np.zeros(608, dtype=np.uint8)
    for sc in scales:
        prod = (vals[fin].astype(np.float32) * np.float32(sc)).astype(np.float32)
        ref = torch.from_numpy(prod).to(torch.bfloat16).double().numpy()
        row[576:580] = np.array([sc], dtype=np.float32).view(np.uint8)
        got = []
        for c in codes[fin]:
            row[0] = c
            got.append(oracle.decode_kv8(row, 0))
        assert np.array_equal(np.array(got), ref), sc
