"""Indexer Prolog on the GPU (through the C ABI) against the CPU oracle.

Integer-valued inputs make every projection exact in fp32, so the quantised queries, their
group scales and the head weights must match the oracle bit for bit.  The LayerNorm'd keys (and,
on normal-valued inputs, everything) are compared after dequantisation, within half an e4m3 step
of the oracle's value (the rounding decision itself may flip where fp32 and fp64 straddle a
midpoint) plus the fp32 evaluation error.  Key-cache rows other than the new tokens' must not
change.
"""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_li_gb300 as dsa
import oracle

pytestmark = pytest.mark.gpu


def _case(values="int4", li_dtype="mxfp8", **over):
    kw = dict(seq_lens=[300, 4100, 65], n_new=[1, 2, 3], d_q=1536, d_model=7168, values=values,
              li_dtype=li_dtype)
    kw.update(over)
    wl = di.small("prolog_decode_32k", **kw)
    cpu = di.generate_prolog(wl)
    return cpu, di.to_device(cpu, "cuda")


def _run(inp, workspace=None):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, qsf, w = dsa.indexer_prolog(inp, status=status, workspace=workspace)
    torch.cuda.synchronize()
    return q, qsf, w, int(status.item())


def _e4m3(codes):
    return torch.as_tensor(codes).contiguous().view(torch.float8_e4m3fn).double()


def _check_mx(c_got, s_got, c_ref, s_ref, val, rel, rel_group):
    """GPU MX codes against the oracle's: a group's scale byte may differ only where the
    oracle's amax sits at a power of two, and an element's code only where the oracle's scaled
    value sits at the midpoint of the two codes (the fp32 and fp64 evaluations straddle a
    rounding decision); both within the fp32 evaluation error (rel of the value, rel_group of
    the group's amax)."""
    val = torch.as_tensor(val, dtype=torch.float64).reshape(-1, 32)
    c_got, c_ref = torch.as_tensor(c_got).reshape(-1, 32), torch.as_tensor(c_ref).reshape(-1, 32)
    s_got, s_ref = torch.as_tensor(s_got).reshape(-1), torch.as_tensor(s_ref).reshape(-1)
    amax = val.abs().amax(1)
    diff_s = s_got != s_ref
    lg = torch.log2(amax[diff_s])
    assert torch.all((lg - lg.round()).abs() < 4 * rel), lg
    same = ~diff_s
    y = val[same] / torch.pow(2.0, s_ref[same].double() - 127)[:, None]
    vg, vr = _e4m3(c_got[same]), _e4m3(c_ref[same])
    d = vg != vr
    tol = rel * y.abs() + rel_group * y.abs().amax(1, keepdim=True)
    mid = (vg + vr) / 2
    assert torch.all(((y - mid).abs() <= tol)[d]), float(((y - mid).abs() - tol)[d].max())
    return int(diff_s.sum()), int(d.sum())


@pytest.mark.parametrize("li_dtype", ["mxfp8", "bf16"])
def test_prolog_integer_inputs(cuda_lib, li_dtype):
    cpu, inp = _case("int4", li_dtype)
    wl = cpu["wl"]
    before = inp["k_pool"].clone()
    ws = torch.zeros(max(dsa.prolog_workspace_bytes(inp), 256), dtype=torch.uint8, device="cuda")
    q, qsf, w, st = _run(inp, ws)
    assert st == 0
    r = oracle.prolog(cpu)
    assert np.array_equal(w.cpu().double().numpy(), r["w"])
    F = wl.H_I * wl.d_I
    if li_dtype == "mxfp8":
        assert np.array_equal(q.view(torch.uint8).cpu().numpy().reshape(wl.n_q, F), r["q_enc"])
        assert np.array_equal(qsf.cpu().numpy().reshape(wl.n_q, F // 32), r["q_sf"])
    else:
        assert np.array_equal(q.view(torch.int16).cpu().numpy().reshape(wl.n_q, F).astype(np.uint16),
                              r["q_enc"])
    rows = torch.tensor(r["k_row"])
    pool = inp["k_pool"].view(-1, wl.d_I)
    kv = torch.tensor(r["k_val"])
    if li_dtype == "mxfp8":
        ksf = inp["k_sf"].view(-1, wl.d_I // 32)[rows.cuda()].cpu()
        kc = pool.view(torch.uint8)[rows.cuda()].cpu()
        _check_mx(kc, ksf, r["k_enc"], r["k_sf"], kv, 1e-5, 1e-5)
    else:
        got = pool[rows.cuda()].cpu().double()
        assert torch.all((got - kv).abs() <= kv.abs() * 2.0 ** -8 + 1e-5)
    # no other cache row changed
    keep = torch.ones(pool.shape[0], dtype=torch.bool, device="cuda")
    keep[rows.cuda()] = False
    now_b = inp["k_pool"].view(torch.uint8).reshape(pool.shape[0], -1)
    before_b = before.view(torch.uint8).reshape(pool.shape[0], -1)
    assert torch.equal(now_b[keep], before_b[keep])
    # a second call gives the same bytes (the slices are added in a fixed order)
    q2, qsf2, w2, st2 = _run(inp, ws)
    assert st2 == 0 and torch.equal(q2.view(torch.uint8), q.view(torch.uint8)) and torch.equal(w2, w)


@pytest.mark.parametrize("n_new,d_q,d_model", [([1, 2, 3], 1536, 7168), ([150, 130, 20], 256, 512),
                                               ([7], 72, 200), ([32], 1536, 7168),
                                               ([300, 220], 1536, 7168)])
def test_prolog_normal_inputs(cuda_lib, n_new, d_q, d_model):
    cpu, inp = _case("normal", "mxfp8", n_new=n_new, d_q=d_q, d_model=d_model,
                     seq_lens=[300, 4100, 65][:len(n_new)] if len(n_new) > 1 else [3000])
    wl = cpu["wl"]
    q, qsf, w, st = _run(inp)
    assert st == 0
    r = oracle.prolog(cpu)
    F = wl.H_I * wl.d_I
    # fp32 accumulation of d_q bf16 products: relative error well below 1e-5 of the group's amax
    nq = _check_mx(q.view(torch.uint8).cpu(), qsf.cpu(), r["q_enc"], r["q_sf"], r["q_val"], 1e-6, 1e-5)
    np.testing.assert_allclose(w.cpu().double().numpy(), r["w"], rtol=1e-4,
                               atol=1e-5 * np.abs(r["w"]).max())
    rows = torch.tensor(r["k_row"]).cuda()
    ksf = inp["k_sf"].view(-1, wl.d_I // 32)[rows].cpu()
    kc = inp["k_pool"].view(torch.uint8).view(-1, wl.d_I)[rows].cpu()
    nk = _check_mx(kc, ksf, r["k_enc"], r["k_sf"], r["k_val"], 1e-5, 1e-5)
    print("prolog %s: rounding flips q %s, k %s of %d / %d elements" % (n_new, nq, nk, wl.n_q * F,
                                                                       wl.n_q * wl.d_I))


def test_prolog_bad_page_sets_status(cuda_lib):
    cpu, inp = _case("int4", "mxfp8")
    pt = inp["pt_k"].clone()
    pt[1, 4099 // 64] = inp["k_pool"].shape[0] + 5  # the page of sequence 1's new tokens
    q, qsf, w, st = _run(dict(inp, pt_k=pt))
    assert st == dsa.DSA_ERR_DEVICE_CHECK
    torch.cuda.synchronize()
