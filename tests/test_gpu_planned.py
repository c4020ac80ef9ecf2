"""The work plan made ahead (dcp_decode_plan, on a second stream beside the
step's cache write) and the attention on it (dcp_decode_attention_planned):
the fused call's result bit for bit, one plan serving several calls, a plan
for other arguments refused on the device, and requests that own no token
(their groups own no chunk) through both paths."""

import numpy as np
import pytest
import torch

import oracle
from dcp_workloads import config, make_workload

from gpu_common import assert_close_rows, f64, tol_for

pytestmark = pytest.mark.gpu

DEV_ERR_TOKEN = 0x2
DEV_ERR_PLAN = 0x40

CASES = {
    "gqa_bf16_ragged": config("gqa_llama8b", B=3, lengths=("list", [1000, 37, 513])),
    # more units than the planner keeps in shared memory
    "gqa_bf16_many_units": config("gqa_llama8b", B=160, lengths=("lognormal", 40, 0.8, 1, 300)),
    "gqa_toy_fp32": config("gqa_toy"),  # the CUDA-core kernel + segment merge
    "mla_bf16": config("mla_bf16_32k", B=2, lengths=("list", [700, 1531])),
    "mla_fp8_tq4": config("mla_fp8_1m", lengths=("list", [2000])),
}


def _dw(name, seed=1):
    from context_decode_attention_gb300.harness import DeviceWorkload
    wl = make_workload(CASES[name], seed=seed)
    return wl, DeviceWorkload(wl)


@pytest.mark.parametrize("name", list(CASES))
def test_planned_equals_fused_bit_exact(name):
    wl, dw = _dw(name)
    a, la = dw.decode()
    a, la = a.clone(), la.clone()
    b, lb = dw.step()  # plan beside the cache write, then the planned attention
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    assert torch.equal(a, b) and torch.equal(la, lb)
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(b).reshape(ref_o.shape), f64(lb).reshape(-1), ref_o, ref_l, tol_for(wl.cfg), name)


@pytest.mark.parametrize("name", ["gqa_bf16_ragged", "mla_fp8_tq4", "gqa_toy_fp32"])
def test_one_plan_serves_several_calls(name):
    """As a model's layers would: one plan, three attention calls on three
    query batches, each equal to the fused call on the same batch."""
    import context_decode_attention_gb300 as dcp
    wl, dw = _dw(name)
    q0 = dw.q.clone()
    dcp.dcp_decode_plan(dw.params, dw.seq_lens, dw.local_lens, int(dw.block_tables.shape[-1]), dw.workspace,
                        dw.stream)
    got = []
    for k in range(3):
        dw.q.copy_(q0 * (k + 1) if k < 2 else -q0)
        o, l = dw.decode_planned()
        got.append((o.clone(), l.clone()))
    for k in range(3):
        dw.q.copy_(q0 * (k + 1) if k < 2 else -q0)
        o, l = dw.decode()
        assert torch.equal(o, got[k][0]) and torch.equal(l, got[k][1]), k
    torch.cuda.synchronize()
    assert dw.error_bits() == 0


def test_plan_for_other_arguments_is_refused():
    import context_decode_attention_gb300 as dcp
    wl, dw = _dw("gqa_bf16_ragged")
    # a fresh workspace holds no plan
    dw.out.fill_(7.0)
    dw.decode_planned()
    torch.cuda.synchronize()
    assert dw.error_bits() == DEV_ERR_PLAN
    assert bool((dw.out == 7.0).all())
    # a fused call's plan is not one made ahead (it has no worker starts)
    dw.decode()
    dw.out.fill_(7.0)
    dw.decode_planned()
    torch.cuda.synchronize()
    assert dw.error_bits() == DEV_ERR_PLAN
    assert bool((dw.out == 7.0).all())
    # a plan for two of the three requests
    sl2 = dw.seq_lens[:2].clone()
    ll2 = dw.local_lens[:, :2].contiguous()
    dcp.dcp_decode_plan(dw.params, sl2, ll2, int(dw.block_tables.shape[-1]), dw.workspace, dw.stream)
    dw.decode_planned()
    torch.cuda.synchronize()
    assert dw.error_bits() == DEV_ERR_PLAN
    assert bool((dw.out == 7.0).all())
    # and the right plan is taken
    dcp.dcp_decode_plan(dw.params, dw.seq_lens, dw.local_lens, int(dw.block_tables.shape[-1]), dw.workspace,
                        dw.stream)
    out, lse = dw.decode_planned()
    torch.cuda.synchronize()
    assert dw.error_bits() == 0
    ref_o, ref_l = oracle.attention(wl)
    assert_close_rows(f64(out).reshape(ref_o.shape), f64(lse).reshape(-1), ref_o, ref_l, tol_for(wl.cfg),
                      "after refusals")


@pytest.mark.parametrize("name", ["gqa_bf16_ragged", "mla_bf16", "gqa_toy_fp32"])
@pytest.mark.parametrize("planned", [False, True])
def test_request_with_no_token(name, planned):
    """Request 0 set to length 0 on the device: its merge group owns no chunk,
    its rows come out as zeros and -inf (the planner lists the group, the
    attention kernel or the segment merge writes it), the length check
    raises DCP_DEV_ERR_TOKEN, and the other requests are unchanged."""
    import context_decode_attention_gb300 as dcp
    wl, dw = _dw(name)
    ref_o, ref_l = oracle.attention(wl)
    B, Tq, Hq = dw.B, dw.Tq, dw.Hq
    dw.seq_lens[0] = 0
    dcp.dcp_slot_mapping(dw.params, dw.seq_lens, local_lens=dw.local_lens, workspace=dw.workspace, stream=dw.stream)
    dw.out.fill_(7.0)
    dw.lse.fill_(7.0)
    if planned:
        dcp.dcp_decode_plan(dw.params, dw.seq_lens, dw.local_lens, int(dw.block_tables.shape[-1]), dw.workspace,
                            dw.stream)
        out, lse = dw.decode_planned()
    else:
        out, lse = dw.decode()
    torch.cuda.synchronize()
    assert dw.error_bits() == DEV_ERR_TOKEN
    o = f64(out).reshape(B, Tq * Hq, -1)
    l = f64(lse).reshape(B, Tq * Hq)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))
    ro = ref_o.reshape(B, Tq * Hq, -1)
    rl = ref_l.reshape(B, Tq * Hq)
    assert_close_rows(o[1:].reshape(-1, o.shape[-1]), l[1:].reshape(-1), ro[1:].reshape(-1, ro.shape[-1]),
                      rl[1:].reshape(-1), tol_for(wl.cfg), f"{name} other requests")
