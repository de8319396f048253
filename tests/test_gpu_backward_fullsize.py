"""Full-size parity of the attention backward at the causal benchmark shapes,
against the float64 oracle computed in the background from the session's
start (tests/fullsize_oracle.py):

* dq on 512 seeded query rows (block edges included) of every query head
  (oracle.attention_backward_rows);
* dk, dv on sampled key rows of every key/value head: every query that sees
  them enters with its full softmax statistics, summed over the query heads
  of the group (oracle.attention_backward_keys); at halfmil_512k (one
  document of 524288 tokens in 16 striped blocks) the sampled keys are the
  last 64 tokens, the only ones whose observers the oracle can afford;
* sum rules that hold at any size, on the whole tensors: the rows of dS sum
  to zero, so sum_j dk_j = 0; the rows of P sum to one, so sum_j dv_j equals
  the sum of dout over the group's query heads.
out and lse come from our forward, as in a training step."""

import numpy as np
import pytest
import torch

from fullsize_oracle import BACKWARD_DQ_ROWS, backward_dout
from helpers import check_grad, np32
import workloads

pytestmark = pytest.mark.gpu

SUM_RULE_TOL = 1e-3  # |sum| relative to sum of |.| per column (bf16 storage)


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


@pytest.mark.parametrize("name,workload,order", [
    pytest.param("bwd_llama8b_32k", "llama8b_32k", "contiguous",
                 marks=pytest.mark.fullsize_oracle("bwd_llama8b_32k")),
    pytest.param("bwd_packed_128k_striped", "packed_128k", "striped",
                 marks=pytest.mark.fullsize_oracle("bwd_packed_128k_striped")),
    pytest.param("bwd_halfmil_512k_striped", "halfmil_512k", "striped",
                 marks=pytest.mark.fullsize_oracle("bwd_halfmil_512k_striped")),
])
def test_backward_full_size(sp, fullsize_oracle, name, workload, order):
    cfg = workloads.CONFIGS[workload]
    B, S, Hq, Hkv, d, P = (cfg[x] for x in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    dout = backward_dout(cfg)
    pos = workloads.position_ids(cfg)
    tpos = torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    dq, dk, dv = sp.blockwise_attention_backward(q, k, v, out, dout, lse, P, order, tpos)
    torch.cuda.synchronize()
    del out, lse, q, k, v

    # sum rules over every key row
    G = Hq // Hkv
    dk64 = dk.double().sum(dim=1)                       # [B][Hkv][d]
    dv64 = dv.double().sum(dim=1)
    do64 = dout.double().sum(dim=1).view(B, Hkv, G, d).sum(dim=2)
    dk_abs = dk.double().abs().sum(dim=1)
    dv_abs = dv.double().abs().sum(dim=1)
    assert (dk64.abs() <= SUM_RULE_TOL * dk_abs).all(), f"{name}: sum of dk is not 0"
    assert ((dv64 - do64).abs() <= SUM_RULE_TOL * dv_abs).all(), f"{name}: sum of dv"

    rows, ref_dq, keys, ref_dk, ref_dv = fullsize_oracle.backward_result(name)
    assert len(rows) == BACKWARD_DQ_ROWS
    trows, tkeys = torch.from_numpy(rows).cuda(), torch.from_numpy(keys).cuda()
    e = check_grad(np32(dq.index_select(1, trows)), ref_dq, "bf16", f"dq {name}")
    print(f"PARITY-GRAD {name}: dq {len(rows)} rows x {Hq} heads max=%.3e mean=%.3e" % e)
    e = check_grad(np32(dk.index_select(1, tkeys)), ref_dk, "bf16", f"dk {name}")
    print(f"PARITY-GRAD {name}: dk {len(keys)} keys x {Hkv} heads max=%.3e mean=%.3e" % e)
    e = check_grad(np32(dv.index_select(1, tkeys)), ref_dv, "bf16", f"dv {name}")
    print(f"PARITY-GRAD {name}: dv {len(keys)} keys x {Hkv} heads max=%.3e mean=%.3e" % e)


@pytest.mark.parametrize("workload,order", [("llama8b_32k", "contiguous"),
                                            ("packed_128k", "striped"),
                                            ("halfmil_512k", "striped")])
def test_backward_forms_agree_everywhere(sp, workload, order):
    """Every element of both forms of the bf16 backward at full size: dk and
    dv bit-identical (the same products in the same order); dq within one
    bf16 step of the two-kernel form plus 1e-4 of the tensor's largest
    magnitude -- the fused form adds dQ's per-key-tile pieces (up to 4096
    at halfmil_512k) in float32 in no fixed order, and where those pieces
    cancel, the reassociation error of the float32 sum can exceed one bf16
    step of a small result.  The default (fused) form is the one compared
    with the oracle above on sampled rows and keys; this extends the check
    to every row."""
    from sequence_parallelism_gb300 import _lib
    cfg = workloads.CONFIGS[workload]
    B, S, Hq, Hkv, d, P = (cfg[x] for x in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    dout = backward_dout(cfg)
    tpos = torch.from_numpy(workloads.position_ids(cfg)).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    grads = {}
    for form in (True, False):
        prev = _lib.sp_set_bwd_dq_reduction(form)
        try:
            grads[form] = sp.blockwise_attention_backward(q, k, v, out, dout, lse, P, order, tpos)
        finally:
            _lib.sp_set_bwd_dq_reduction(prev)
    torch.cuda.synchronize()
    (dq_f, dk_f, dv_f), (dq_r, dk_r, dv_r) = grads[True], grads[False]
    assert torch.equal(dk_f, dk_r), f"{workload}: dk differs between the forms"
    assert torch.equal(dv_f, dv_r), f"{workload}: dv differs between the forms"
    a, b = dq_f.float(), dq_r.float()
    scale = float(b.abs().max())
    step = torch.maximum(a.abs(), b.abs()) * 2.0 ** -7
    excess = ((a - b).abs() - step).clamp(min=0.0)
    beyond = int((excess > 1e-6 * scale).sum())
    diff = int((a != b).sum())
    worst = float(excess.max()) / scale
    print(f"PARITY-FORMS {workload} {order}: dq elements differing {diff} of {a.numel()}, "
          f"beyond one bf16 step + 1e-6 of max |dq| {beyond} (largest excess {worst:.2e})")
    assert worst <= 1e-4, f"{workload}: dq differs beyond one bf16 step by {worst:.2e} of max |dq|"
