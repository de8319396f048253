"""Out-of-bounds write checks for every entry point that writes device memory.

compute-sanitizer is not available on the GPU pool, so each output (and each
workspace) is placed in the middle of a larger buffer whose bytes all start
as 0xFF: after the call the 64 KiB guard bands on both sides must still hold
0xFF byte for byte (a write past either end of any buffer shows there), and
the outputs themselves must hold no NaN -- 0xFF.. is a NaN in bf16 and fp32,
so an element the kernel never wrote would show up -- and must match the
float64 oracle as the parity tests require."""

import numpy as np
import pytest
import torch

import oracle
from helpers import BF16_MAX_ABS, F32_MAX_ABS, check_attention, check_grad, np32
import workloads
from sequence_parallelism_gb300 import _lib
from test_gpu_attention import _positions

pytestmark = pytest.mark.gpu

GUARD = 1 << 16  # bytes on each side; a multiple of every alignment the calls need


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


class Guarded:
    """A tensor of `shape` in the middle of a 0xFF-filled byte buffer."""

    def __init__(self, shape, dtype):
        el = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * el
        self.buf = torch.full((2 * GUARD + n,), 0xFF, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)

    def intact(self):
        return bool((self.buf[:GUARD] == 0xFF).all()) and bool((self.buf[-GUARD:] == 0xFF).all())


def _workspace(nbytes):
    return Guarded((nbytes,), torch.uint8)


def _assert_guarded(what, *gs):
    torch.cuda.synchronize()
    for name, g in gs:
        assert g.intact(), f"{what}: a write landed outside {name}"


def _no_nan(what, **ts):
    for name, t in ts.items():
        assert not torch.isnan(t.float()).any(), f"{what}: {name} has elements never written"


@pytest.mark.parametrize("dtype,B,S,Hq,Hkv,d,P,order,pos_kind", [
    ("bf16", 2, 1000, 4, 2, 128, 2, "contiguous", "none"),    # tail split + ragged tail
    ("bf16", 1, 1536, 2, 1, 128, 3, "striped", "packed"),
    ("bf16", 1, 2048, 2, 2, 128, 4, "contiguous", "causal"),
    ("f32", 2, 96, 4, 2, 64, 3, "striped", "packed"),
])
def test_attention_writes_stay_inside_out_lse_workspace(sp, dtype, B, S, Hq, Hkv, d, P, order,
                                                         pos_kind):
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 700 + S, dtype)
    pos = _positions(pos_kind, B, S, 700 + S)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out = Guarded(q.shape, q.dtype)
    lse = Guarded((B, Hq, S), torch.float32)
    ws = _workspace(_lib.sp_blockwise_attn_split_workspace_bytes(B, S, tpos is not None))
    sp.blockwise_attention(q, k, v, P, order, tpos, out=out.t, lse=lse.t, workspace=ws.t)
    what = f"attention {dtype} S={S} P={P} {order} {pos_kind}"
    _assert_guarded(what, ("out", out), ("lse", lse), ("workspace", ws))
    _no_nan(what, out=out.t)
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    check_attention(np32(out.t), lse.t.cpu().numpy(), ref_out, ref_lse, dtype, what)


@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_ring_step_writes_stay_inside(sp, order):
    B, S, Hq, Hkv, d, P = 1, 1024, 2, 1, 128, 4
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 710, "bf16")
    pos = _positions("packed", B, S, 710)
    tpos = torch.from_numpy(pos).cuda()
    for step in range(P):
        out = Guarded(q.shape, q.dtype)
        lse = Guarded((B, Hq, S), torch.float32)
        ws = _workspace(_lib.sp_blockwise_attn_workspace_bytes(B, S, True))
        sp.ring_step(q, k, v, P, step, order, tpos, out=out.t, lse=lse.t, workspace=ws.t)
        _assert_guarded(f"ring step {step} {order}", ("out", out), ("lse", lse), ("workspace", ws))
        _no_nan(f"ring step {step} {order}", out=out.t)
        ro, rl = oracle.ring_partial(np32(q), np32(k), np32(v), P, step, order, pos)
        check_attention(np32(out.t), lse.t.cpu().numpy(), ro, rl, "bf16",
                        f"ring step {step} {order}")


@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_accumulating_ring_step_writes_stay_inside(sp, order):
    """Each device's ring on 200-row blocks (one 256-row unit whose last 56
    rows lie past the block: the running output's TMA load reads them as
    zeros, the store drops them): step 0 writes the guarded running result,
    steps 1..P-1 fold into it; nothing lands outside out, lse or the
    workspace, and the result is block i's rows of full attention."""
    B, S, Hq, Hkv, d, P = 2, 600, 2, 1, 128, 3
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 720, "bf16")
    pos = _positions("packed", B, S, 720)
    tpos = torch.from_numpy(pos).cuda()
    full_o, full_l = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    blocks = [oracle.block_tokens(S, P, p_, order) for p_ in range(P)]
    blk = lambda t, p_: t[:, torch.from_numpy(blocks[p_]).cuda()].contiguous()
    for i in range(P):
        out = Guarded((B, S // P, Hq, d), q.dtype)
        lse = Guarded((B, Hq, S // P), torch.float32)
        ws = _workspace(_lib.sp_blockwise_attn_workspace_bytes(B, S, True))
        for s_ in range(P):
            j = (i - s_) % P
            call = _lib.sp_ring_block_step if s_ == 0 else _lib.sp_ring_block_step_accumulate
            call(blk(q, i), blk(k, j), blk(v, j), tpos, S, P, order, i, j, 0.0, out.t, lse.t,
                 ws.t)
        what = f"accumulating ring {order} device {i}"
        _assert_guarded(what, ("out", out), ("lse", lse), ("workspace", ws))
        _no_nan(what, out=out.t)
        check_attention(np32(out.t), lse.t.cpu().numpy(), full_o[:, blocks[i]],
                        full_l[:, :, blocks[i]], "bf16", what)


@pytest.fixture(params=["tma_staged", "default"])
def path(request):
    """Every permutation that meets the bulk-copy rules on the TMA-staged
    kernel, or the default size threshold (these small ones on the vector
    kernel)."""
    prev = _lib.sp_permute_set_bulk_min_bytes(0 if request.param == "tma_staged" else 128 << 20)
    yield request.param
    _lib.sp_permute_set_bulk_min_bytes(prev)


@pytest.mark.parametrize("dtype,B,S,H,d,P", [
    ("bf16", 2, 300, 12, 128, 4),   # 768 B chunks, 10 rows per item
    ("bf16", 1, 292, 12, 128, 4),   # the last item of each head group is partial
    ("bf16", 2, 300, 6, 40, 2),     # 240 B chunks: vector kernel only
    ("f32", 2, 300, 8, 24, 4),      # 192 B chunks: vector kernel only
    ("f32", 1, 260, 8, 64, 4),      # 512 B chunks, partial last item
])
def test_permutation_writes_stay_inside(sp, path, dtype, B, S, H, d, P):
    g = torch.Generator(device="cuda")
    g.manual_seed(720 + H)
    x = torch.randn((B, S, H, d), generator=g, device="cuda").to(
        torch.bfloat16 if dtype == "bf16" else torch.float32)
    y = Guarded((P, B, S, H // P, d), x.dtype)
    sp.seq_to_head(x, P, out=y.t)
    _assert_guarded("seq_to_head", ("y", y))
    assert np.array_equal(np32(y.t), oracle.seq_to_head(np32(x), P))
    back = Guarded(x.shape, x.dtype)
    sp.head_to_seq(y.t, out=back.t)
    _assert_guarded("head_to_seq", ("x", back))
    assert torch.equal(back.t, x)


def test_qkv_permutation_writes_stay_inside(path):
    B, S, H, d, P = 1, 520, 8, 128, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(730)
    xs = [torch.randn((B, S, H, d), generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(3)]
    ys = [Guarded((P, B, S, H // P, d), torch.bfloat16) for _ in range(3)]
    _lib.sp_ulysses_seq_to_head_qkv(xs[0], xs[1], xs[2], ys[0].t, ys[1].t, ys[2].t, P)
    _assert_guarded("seq_to_head_qkv", *[(f"y{i}", y) for i, y in enumerate(ys)])
    for x, y in zip(xs, ys):
        assert np.array_equal(np32(y.t), oracle.seq_to_head(np32(x), P))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_writes_stay_inside(sp, dtype):
    P, B, S, H, d = 3, 2, 41, 3, 64
    g = torch.Generator(device="cuda")
    g.manual_seed(740)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    outs = torch.randn((P, B, S, H, d), generator=g, device="cuda").to(tdt)
    lses = torch.randn((P, B, H, S), generator=g, device="cuda") * 2
    out = Guarded((B, S, H, d), tdt)
    lse = Guarded((B, H, S), torch.float32)
    sp.merge_partials(outs, lses, out=out.t, lse=lse.t)
    _assert_guarded(f"merge {dtype}", ("out", out), ("lse", lse))
    _no_nan(f"merge {dtype}", out=out.t)
    ro, rl = oracle.merge_partials(np32(outs).astype(np.float64), lses.cpu().numpy())
    # bf16 outputs reach |x| ~ 3, where half a bf16 ulp is already 0.008
    tol = F32_MAX_ABS if dtype == "f32" else BF16_MAX_ABS
    assert np.abs(np32(out.t) - ro).max() <= tol
    assert np.abs(lse.t.cpu().numpy() - rl).max() <= 1e-4


def test_doc_starts_writes_stay_inside():
    B, S = 2, 3000
    pos = _positions("packed", B, S, 750)
    tpos = torch.from_numpy(pos).cuda()
    ds = Guarded((B, S), torch.int32)
    ws = _workspace(_lib.sp_segment_starts_workspace_bytes(B, S))
    _lib.sp_segment_starts(tpos, ds.t, ws.t)
    _assert_guarded("doc_starts", ("doc_start", ds), ("workspace", ws))
    assert np.array_equal(ds.t.cpu().numpy(), oracle.doc_starts(pos))


@pytest.mark.parametrize("dtype,order,pos_kind", [
    ("bf16", "contiguous", "causal"),
    ("bf16", "striped", "packed"),
    ("f32", "contiguous", "none"),
])
@pytest.mark.parametrize("dq_reduction", [True, False])
def test_backward_writes_stay_inside(sp, dq_reduction, dtype, order, pos_kind):
    B, S, Hq, Hkv, P = 1, 640 if dtype == "bf16" else 96, 4, 2, 2
    d = 128 if dtype == "bf16" else 32
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 760, dtype)
    g = torch.Generator(device="cuda")
    g.manual_seed(761)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    pos = _positions(pos_kind, B, S, 760)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    dq, dk, dv = (Guarded(t.shape, t.dtype) for t in (q, k, v))
    ws = _workspace(_lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, tpos is not None))
    prev = _lib.sp_set_bwd_dq_reduction(dq_reduction)
    try:
        _lib.sp_blockwise_attn_bwd(q, k, v, out, dout, lse, tpos, P, order, 0.0, dq.t, dk.t, dv.t,
                                   ws.t)
    finally:
        _lib.sp_set_bwd_dq_reduction(prev)
    what = f"backward {dtype} {order} {pos_kind} dq_reduction={dq_reduction}"
    _assert_guarded(what, ("dq", dq), ("dk", dk), ("dv", dv), ("workspace", ws))
    _no_nan(what, dq=dq.t, dk=dk.t, dv=dv.t)
    rq, rk, rv = oracle.attention_backward(np32(q), np32(k), np32(v), np32(dout), pos)
    check_grad(np32(dq.t), rq, dtype, "dq " + what)
    check_grad(np32(dk.t), rk, dtype, "dk " + what)
    check_grad(np32(dv.t), rv, dtype, "dv " + what)


def test_hybrid_writes_stay_inside(sp):
    B, S, Hq, Hkv, d, P_u, P_r = 1, 1024, 4, 2, 128, 2, 2
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 770, "bf16")
    pos = _positions("causal", B, S, 770)
    tpos = torch.from_numpy(pos).cuda()
    out = Guarded(q.shape, q.dtype)
    lse = Guarded((P_u, B, Hq // P_u, S), torch.float32)
    ws = _workspace(_lib.sp_ulysses_ring_attn_workspace_bytes(B, S, Hq, Hkv, d, True,
                                                              _lib._dtype(q)))
    sp.ulysses_ring_attention(q, k, v, P_u, P_r, "striped", tpos, out=out.t, lse=lse.t,
                              workspace=ws.t)
    _assert_guarded("hybrid", ("out", out), ("lse", lse), ("workspace", ws))
    _no_nan("hybrid", out=out.t)
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    # lse in the head-sharded layout: group r holds heads r*Hq/P_u ...
    ref_lse_h = ref_lse.reshape(B, P_u, Hq // P_u, S).transpose(1, 0, 2, 3)
    check_attention(np32(out.t), lse.t.cpu().numpy(), ref_out, ref_lse_h, "bf16", "hybrid")


def test_noalloc_writes_stay_inside_out_lse():
    """The allocation-free entry point keeps its scratch in a static device
    array; its outputs must still be written exactly within out and lse."""
    B, S, Hq, Hkv, d, P = 1, 1536, 2, 1, 128, 3
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 780, "bf16")
    pos = _positions("packed", B, S, 780)
    tpos = torch.from_numpy(pos).cuda()
    out = Guarded(q.shape, q.dtype)
    lse = Guarded((B, Hq, S), torch.float32)
    _lib.sp_blockwise_attn_fwd_noalloc(q, k, v, tpos, P, "striped", 0.0, out.t, lse.t)
    _assert_guarded("noalloc", ("out", out), ("lse", lse))
    _no_nan("noalloc", out=out.t)
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    check_attention(np32(out.t), lse.t.cpu().numpy(), ref_out, ref_lse, "bf16", "noalloc")
