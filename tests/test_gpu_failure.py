"""Failure handling on the GPU without a GPU fault: a bounded device-side wait that runs out.

The test build of the library (libdsa_testhooks.so, include/dsa_testhooks.h) gives every
device-side wait a 20 ms limit and can make the MMA-issuing thread of a kernel's first CTA wait
on an mbarrier that no thread ever arrives on.  That wait gives up: the kernel must store
DSA_ERR_TIMEOUT in the caller's status word, drain its copies, free its tensor memory and
complete -- and the next call on the same context must give the oracle's result.  Nothing here
traps, faults or waits without a bound.
"""
import ctypes

import numpy as np
import pytest
import torch

import dsa_inputs as di
import dsa_sparse_attention_li_gb300 as dsa
import oracle
from parity import BF16_TOL, sfa_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hooks(cuda_lib):
    return dsa.load_testhooks()


def _calls(lib, inp, status, prefill):
    """li_topk then sparse attention through the C ABI of ``lib``; returns the outputs."""
    wl = inp["wl"]
    ms, mq = max(wl.seq_lens), max(wl.n_new)
    idx = torch.full((wl.n_q, wl.K), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((wl.n_q,), dtype=torch.int32, device="cuda")
    out = torch.zeros((wl.n_q, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((wl.n_q, wl.H), dtype=torch.float32, device="cuda")
    ws = dsa.new_workspace(dsa.sfa_workspace_bytes(inp["q_sfa"], idx), "cuda")
    li = dsa.li_topk_args(inp["q_li"], inp["w"], inp["k_pool"], inp["pt_k"], inp["seq_lens"],
                          inp["q_start"], wl.K, max_seq_len=ms, max_q_per_seq=mq, out_idx=idx,
                          out_cnt=cnt, status=status)
    sa = dsa.sfa_args(inp["q_sfa"], inp["kv_pool"], inp["pt_kv"], inp["seq_lens"], inp["q_start"],
                      idx, softmax_scale=wl.softmax_scale, max_seq_len=ms, max_q_per_seq=mq,
                      out=out, lse=lse, status=status, workspace=ws)
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.dsa_li_topk(ctypes.byref(li), sp) == dsa.DSA_OK
    entry = lib.dsa_sfa_prefill if prefill else lib.dsa_sfa_decode
    assert entry(ctypes.byref(sa), sp) == dsa.DSA_OK
    torch.cuda.synchronize()
    return {"idx": idx.cpu().numpy(), "cnt": cnt.cpu().numpy(), "out": out.float().cpu(),
            "lse": lse.cpu()}


@pytest.mark.parametrize("kernel,prefill", [(1, False), (2, False), (2, True)],
                         ids=["indexer", "attention_decode", "attention_prefill"])
def test_timed_out_wait_is_reported_and_the_context_recovers(hooks, kernel, prefill):
    wl = di.small("decode_int_4k", seq_lens=[4096, 700], n_new=[1, 2])
    inp_cpu = di.generate(wl)
    inp = di.to_device(inp_cpu, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hooks.dsa_test_inject_stall(kernel)
    try:
        _calls(hooks, inp, status, prefill)
    finally:
        hooks.dsa_test_inject_stall(0)
    assert int(status.item()) == dsa.DSA_ERR_TIMEOUT
    # the same context, the same test build, no stall: the oracle's result
    status.zero_()
    g = _calls(hooks, inp, status, prefill)
    assert int(status.item()) == dsa.DSA_OK
    ref_idx, ref_cnt, _ = oracle.li_topk(inp_cpu)
    assert np.array_equal(g["idx"], ref_idx) and np.array_equal(g["cnt"], ref_cnt)
    max_abs, mean_rel, _ = sfa_errors(inp_cpu, g, list(range(wl.n_q)))
    assert max_abs <= BF16_TOL[0] and mean_rel <= BF16_TOL[1]
    # and the product library on the same context
    status.zero_()
    g2 = _calls(dsa.load(), inp, status, prefill)
    assert int(status.item()) == dsa.DSA_OK
    assert np.array_equal(g2["idx"], ref_idx)
