"""GPU parity of the attention backward (dq, dk, dv) against the float64
oracle's derivatives, through the C ABI.  The kernel takes out and lse from
our forward, as a training step would."""

import numpy as np
import pytest
import torch

import oracle
from helpers import check_grad, np32
import workloads
from test_gpu_attention import _positions

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


@pytest.fixture(params=["dq_reduction", "dq_recompute"])
def dq_form(request):
    """Both forms of the bf16 backward: dQ summed by reductions in the fused
    kernel (the default) and dQ recomputed by its own kernel."""
    from sequence_parallelism_gb300 import _lib
    prev = _lib.sp_set_bwd_dq_reduction(request.param == "dq_reduction")
    yield request.param
    _lib.sp_set_bwd_dq_reduction(prev)


def _run_bwd(sp, dtype, B, S, Hq, Hkv, d, P, order, pos_kind, seed):
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, seed, dtype)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    pos = _positions(pos_kind, B, S, seed)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    dq, dk, dv = sp.blockwise_attention_backward(q, k, v, out, dout, lse, P, order, tpos)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attention_backward(np32(q), np32(k), np32(v), np32(dout), pos)
    tag = f"{dtype} S={S} P={P} {order} {pos_kind}"
    check_grad(np32(dq), rq, dtype, "dq " + tag)
    check_grad(np32(dk), rk, dtype, "dk " + tag)
    check_grad(np32(dv), rv, dtype, "dv " + tag)


@pytest.mark.parametrize("B,S,Hq,Hkv,d,P,order,pos", [
    (1, 32, 1, 1, 16, 4, "contiguous", "none"),     # the Ring Attention page's shape
    (1, 96, 4, 2, 64, 3, "contiguous", "causal"),
    (2, 64, 2, 1, 32, 4, "striped", "packed"),
    (1, 80, 2, 2, 100, 2, "striped", "causal"),
])
def test_backward_f32(sp, B, S, Hq, Hkv, d, P, order, pos):
    _run_bwd(sp, "f32", B, S, Hq, Hkv, d, P, order, pos, 800 + S)


@pytest.mark.parametrize("B,S,Hq,Hkv,P,order,pos", [
    (1, 512, 4, 2, 2, "contiguous", "causal"),
    (1, 768, 2, 2, 4, "striped", "packed"),
    (2, 256, 2, 1, 1, "contiguous", "none"),
    (1, 1000, 2, 1, 2, "striped", "none"),          # ragged blocks of 500
    (1, 2048, 8, 2, 4, "contiguous", "packed"),     # GQA group of 4, documents across blocks
    (1, 1416, 4, 4, 3, "striped", "causal"),        # ragged tiles: blocks of 472 rows
])
def test_backward_bf16(sp, dq_form, B, S, Hq, Hkv, P, order, pos):
    _run_bwd(sp, "bf16", B, S, Hq, Hkv, 128, P, order, pos, 850 + S)


@pytest.mark.parametrize("dtype,B,S,Hq,Hkv,P,order,pos", [
    ("bf16", 2, 1, 2, 1, 1, "contiguous", "causal"),     # a single token
    ("bf16", 1, 256, 2, 1, 256, "striped", "causal"),    # one token per block
    ("f32", 1, 1, 1, 1, 1, "contiguous", "none"),
    ("f32", 1, 64, 2, 1, 64, "striped", "packed"),
])
def test_backward_degenerate_shapes(sp, dq_form, dtype, B, S, Hq, Hkv, P, order, pos):
    _run_bwd(sp, dtype, B, S, Hq, Hkv, 128 if dtype == "bf16" else 16, P, order, pos,
             950 + S + P)


@pytest.mark.parametrize("pos_kind,fused,ring_blocks", [("causal", False, None),
                                                      ("packed", False, None),
                                                      ("none", True, None),
                                                      ("causal", False, 2)])
def test_ulysses_layer_backward(sp, pos_kind, fused, ring_blocks):
    """Gradients of a whole Ulysses layer (seq->head, blockwise attention per
    head group, head->seq; GQA with one key/value head per group) against the
    oracle's derivatives of plain attention on the sequence-sharded tensors.
    ring_blocks=2 is the Ulysses + Ring hybrid (4 head groups x 2 ring
    blocks)."""
    B, S, Hq, Hkv, d, P = 1, 768, 8, 4, 128, 4
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 990, "bf16")
    g = torch.Generator(device="cuda")
    g.manual_seed(991)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    pos = _positions(pos_kind, B, S, 992)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out, ctx = sp.ulysses_attention(q, k, v, P, ring_blocks=ring_blocks, position_ids=tpos,
                                    fused=fused, return_context=True)
    dq, dk, dv = sp.ulysses_attention_backward(ctx, dout)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attention_backward(np32(q), np32(k), np32(v), np32(dout), pos)
    tag = f"ulysses {pos_kind} fused={fused} ring_blocks={ring_blocks}"
    check_grad(np32(dq), rq, "bf16", "dq " + tag)
    check_grad(np32(dk), rk, "bf16", "dk " + tag)
    check_grad(np32(dv), rv, "bf16", "dv " + tag)
