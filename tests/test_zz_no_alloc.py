"""dsa_sfa_decode_static: sparse-attention decode for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: an operator whose device memory is planned
entirely by a host framework that passes it only inputs and outputs, or a path where allocating
is not allowed.  For them the library keeps its own fixed scratch array and this entry point
uses it.  The test calls it through the C ABI, twice in a row (the shared scratch keeps the last
call's contents, so the second call must not depend on it), and checks each result against
dsa_sfa_decode with a caller workspace, within the attention tolerance of the parity tests.
It also checks that arguments needing more scratch than the fixed capacity are refused.

Kept in its own file, named to be collected last.
"""
import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_li_gb300 as dsa

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_REL = 2e-2, 5e-3


def _inputs():
    wl = di.small("decode_32k", seq_lens=[7000, 2600, 4500], n_new=[1, 2, 1])
    inp = di.to_device(di.generate(wl), "cuda")
    idx, _ = dsa.li_topk(inp["q_li"], inp["w"], inp["k_pool"], inp["pt_k"], inp["seq_lens"],
                         inp["q_start"], wl.K, max_seq_len=max(wl.seq_lens),
                         max_q_per_seq=max(wl.n_new))
    return wl, inp, idx


def _kw(wl, inp):
    return dict(softmax_scale=wl.softmax_scale, max_seq_len=max(wl.seq_lens),
                max_q_per_seq=max(wl.n_new))


def test_static_scratch_decode_matches_workspace_decode(cuda_lib):
    wl, inp, idx = _inputs()
    args = (inp["q_sfa"], inp["kv_pool"], inp["pt_kv"], inp["seq_lens"], inp["q_start"], idx)
    need = dsa.sfa_workspace_bytes(inp["q_sfa"], idx)
    assert 0 < need <= dsa.SFA_STATIC_SCRATCH_BYTES  # the split-merge path is exercised
    ref_out, ref_lse = dsa.sfa_decode(*args, **_kw(wl, inp))
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out, lse = dsa.sfa_decode_static(*args, status=status, **_kw(wl, inp))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        d = (out.float() - ref_out.float()).abs()
        assert d.max().item() <= MAX_ABS
        assert d.sum().item() <= MEAN_REL * ref_out.float().abs().sum().item()
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=0, atol=2e-3)


def test_static_scratch_rejects_arguments_beyond_capacity(cuda_lib):
    wl, inp, idx = _inputs()
    # 4 tokens x 2 halves x 32 splits of partials exceed the fixed capacity
    assert dsa.sfa_workspace_bytes(inp["q_sfa"], idx, row_splits=32) > dsa.SFA_STATIC_SCRATCH_BYTES
    with pytest.raises(dsa.DsaError) as e:
        dsa.sfa_decode_static(inp["q_sfa"], inp["kv_pool"], inp["pt_kv"], inp["seq_lens"],
                              inp["q_start"], idx, row_splits=32, **_kw(wl, inp))
    assert e.value.code == dsa.DSA_ERR_UNSUPPORTED
    assert "capacity" in str(e.value)
