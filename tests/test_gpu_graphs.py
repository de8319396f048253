"""The library's calls inside CUDA graphs: a causal attention call, the
Ulysses layer (seq->head of q, k, v, attention per head group, head->seq)
and the backward are captured once and replayed with new inputs copied into
the captured buffers; every replay must give the same bits as the same calls
run eagerly (the kernels are deterministic; the backward's dq only when it is
recomputed by its own kernel: summed by reductions, it matches to float32
rounding of the sum), and the device error word must stay clear.  Every call's first use happens before capture (it sets kernel
attributes and looks up driver entry points on the host)."""

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def _new_inputs(seed, shapes):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return [torch.randn(s, generator=g, device="cuda").to(torch.bfloat16) for s in shapes]


@pytest.mark.parametrize("dq_reduction", [True, False])
def test_causal_attention_and_backward_replay(sp, dq_reduction):
    from sequence_parallelism_gb300 import _lib
    prev = _lib.sp_set_bwd_dq_reduction(dq_reduction)
    try:
        _replay_attention_and_backward(sp, _lib, dq_reduction)
    finally:
        _lib.sp_set_bwd_dq_reduction(prev)


def _replay_attention_and_backward(sp, _lib, dq_reduction):
    B, S, Hq, Hkv, d, P = 1, 2048, 4, 2, 128, 4
    shapes = [(B, S, Hq, d), (B, S, Hkv, d), (B, S, Hkv, d), (B, S, Hq, d)]
    q, k, v, do = _new_inputs(1, shapes)
    pos = torch.from_numpy(workloads.position_ids_from_lengths(
        workloads.doc_lengths(S, 4, 3))[None].astype("int32")).cuda()
    ws = sp.attention_workspace(B, S, True)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    bws = torch.empty(_lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, True),
                      dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        _lib.sp_blockwise_attn_fwd(q, k, v, pos, P, "striped", 0.0, out, lse, ws)
        _lib.sp_blockwise_attn_bwd(q, k, v, out, do, lse, pos, P, "striped", 0.0, dq, dk, dv,
                                   bws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # first use outside capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (11, 12):
        new = _new_inputs(seed, shapes)
        for dst, src in zip((q, k, v, do), new):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (out, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), got, (out, lse, dq, dk, dv)):
            if name == "dq" and dq_reduction:
                # bf16 of two float32 sums of the same pieces in different
                # orders: at most one bf16 step apart
                err = (a.float() - b.float()).abs()
                assert float(err.max()) <= float(b.float().abs().max()) * 2.0 ** -7, name
            else:
                assert torch.equal(a, b), name
    assert _lib.sp_get_device_error(ws) == (0, 0)
    assert _lib.sp_get_device_error(bws) == (0, 0)


def test_ulysses_layer_replay(sp):
    from sequence_parallelism_gb300 import _lib
    B, S, H, d, P = 1, 1024, 8, 128, 4
    G = H // P
    shapes = [(B, S, H, d)] * 3
    q, k, v = _new_inputs(2, shapes)
    yq = torch.empty((P, B, S, G, d), dtype=torch.bfloat16, device="cuda")
    yk, yv, yo = torch.empty_like(yq), torch.empty_like(yq), torch.empty_like(yq)
    ylse = torch.empty((P * B, G, S), dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    ws = sp.attention_workspace(P * B, S, False)

    def layer():
        _lib.sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, P)
        _lib.sp_blockwise_attn_fwd(yq.view(P * B, S, G, d), yk.view(P * B, S, G, d),
                                   yv.view(P * B, S, G, d), None, P, "contiguous", 0.0,
                                   yo.view(P * B, S, G, d), ylse, ws)
        _lib.sp_ulysses_head_to_seq(yo, out, P)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()
    for seed in (21, 22):
        for dst, src in zip((q, k, v), _new_inputs(seed, shapes)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone(), ylse.clone()
        layer()
        torch.cuda.synchronize()
        assert torch.equal(got[0], out) and torch.equal(got[1], ylse)
    assert _lib.sp_get_device_error(ws) == (0, 0)
