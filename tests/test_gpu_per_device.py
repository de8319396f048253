"""GPU parity of the per-device entry points against the float64 oracle.

A device of a real ring holds only its query block and, at each step, one
key/value block ("Ring Attention", "Cómo funciona la atención en anillo"):
sp_ring_block_step computes that block pair from block tensors, with the
mask in global token indices.  Every (i, j) pair must equal block i's rows of
the oracle's ring partial at step (i - j) mod P, merging device i's P steps
must give block i's rows of full attention, and sp_query_block_attn_fwd (the
all-gathered variant: query block i against the whole K, V) must give those
rows directly.  The backward of a ring step (sp_ring_block_step_bwd) must
give every pair's gradient parts, and their sums the whole gradients.
Shapes span ragged 128-row tiles, GQA, packed documents and both block
orders."""

import numpy as np
import pytest
import torch

import oracle
from helpers import check_attention, check_grad, np32
import workloads
from test_gpu_attention import _positions

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


CASES = [
    # dtype, B, S, Hq, Hkv, d, P, order, pos_kind
    ("bf16", 1, 1024, 4, 2, 128, 4, "contiguous", "causal"),
    ("bf16", 1, 1024, 4, 2, 128, 4, "striped", "packed"),
    ("bf16", 2, 600, 2, 1, 128, 3, "contiguous", "packed"),
    ("bf16", 1, 768, 2, 2, 128, 3, "striped", "none"),
    ("f32", 1, 96, 2, 1, 32, 3, "contiguous", "packed"),
    ("f32", 2, 64, 2, 2, 16, 4, "striped", "causal"),
]


def _block(t, tokens):
    return t[:, torch.from_numpy(tokens).to(t.device)].contiguous()


@pytest.mark.parametrize("case", CASES)
def test_ring_block_step_every_pair(sp, case):
    from sequence_parallelism_gb300 import _lib
    dtype, B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4100 + S, dtype)
    pos = _positions(pos_kind, B, S, 77)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    qn, kn, vn = np32(q), np32(k), np32(v)
    ws = sp.attention_workspace(B, S, pos is not None, minimal=True)
    blocks = [oracle.block_tokens(S, P, p, order) for p in range(P)]
    partials = {}
    for s in range(P):
        ref_o, ref_l = oracle.ring_partial(qn, kn, vn, P, s, order, pos)
        for i in range(P):
            j = (i - s) % P
            out = torch.full((B, S // P, Hq, d), float("nan"), dtype=q.dtype, device="cuda")
            lse = torch.full((B, Hq, S // P), float("nan"), dtype=torch.float32, device="cuda")
            _lib.sp_ring_block_step(_block(q, blocks[i]), _block(k, blocks[j]), _block(v, blocks[j]),
                                    tpos, S, P, order, i, j, 0.0, out, lse, ws)
            torch.cuda.synchronize()
            check_attention(np32(out), lse.cpu().numpy(), ref_o[:, blocks[i]],
                            ref_l[:, :, blocks[i]], dtype, f"{case} i={i} j={j}")
            partials[(i, s)] = (out, lse)
    # device i merges its P steps: block i's rows of full attention
    full_o, full_l = oracle.full_attention(qn, kn, vn, pos)
    for i in range(P):
        outs = torch.stack([partials[(i, s)][0] for s in range(P)])
        lses = torch.stack([partials[(i, s)][1] for s in range(P)])
        mo, ml = sp.merge_partials(outs, lses)
        torch.cuda.synchronize()
        check_attention(np32(mo), ml.cpu().numpy(), full_o[:, blocks[i]], full_l[:, :, blocks[i]],
                        dtype, f"{case} merged device {i}")


@pytest.mark.parametrize("case", [c for c in CASES if c[0] == "bf16"])
def test_ring_block_step_accumulate_every_device(sp, case):
    """Each device i folds its P steps, in ring order, into one running
    result with sp_ring_block_step_accumulate, starting from lse = -inf and
    an output of NaNs (which must not be read).  After every step the running
    result equals the oracle's merge of the partials so far, and after the
    last one block i's rows of full attention; contiguous causal pairs with
    j > i launch nothing and leave the result bit for bit."""
    from sequence_parallelism_gb300 import _lib
    dtype, B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4300 + S, dtype)
    pos = _positions(pos_kind, B, S, 79)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    qn, kn, vn = np32(q), np32(k), np32(v)
    ws = sp.attention_workspace(B, S, pos is not None)
    blocks = [oracle.block_tokens(S, P, p, order) for p in range(P)]
    parts = [oracle.ring_partial(qn, kn, vn, P, s, order, pos) for s in range(P)]
    full_o, full_l = oracle.full_attention(qn, kn, vn, pos)
    for i in range(P):
        tok = blocks[i]
        out = torch.full((B, S // P, Hq, d), float("nan"), dtype=q.dtype, device="cuda")
        lse = torch.full((B, Hq, S // P), float("-inf"), dtype=torch.float32, device="cuda")
        for s in range(P):
            j = (i - s) % P
            before = (out.clone(), lse.clone())
            sp.ring_block_step_accumulate(_block(q, tok), _block(k, blocks[j]),
                                          _block(v, blocks[j]), P, i, j, out, lse, order, tpos,
                                          workspace=ws)
            torch.cuda.synchronize()
            if pos is not None and order == "contiguous" and j > i:
                assert _lib.sp_last_launch_count() == 0
                assert torch.equal(out.view(torch.int16), before[0].view(torch.int16))
                assert torch.equal(lse, before[1])
            ro, rl = oracle.merge_partials(np.stack([p_[0][:, tok] for p_ in parts[:s + 1]]),
                                           np.stack([p_[1][:, :, tok] for p_ in parts[:s + 1]]))
            fin = np.isfinite(rl)
            got = np32(out)
            assert not np.isnan(got[np.broadcast_to(fin.transpose(0, 2, 1)[..., None],
                                                    got.shape)]).any()
            check_attention(np.where(fin.transpose(0, 2, 1)[..., None], got, 0.0),
                            lse.cpu().numpy(), np.where(fin.transpose(0, 2, 1)[..., None], ro, 0.0),
                            rl, dtype, f"{case} device {i} after step {s}")
        check_attention(np32(out), lse.cpu().numpy(), full_o[:, tok], full_l[:, :, tok], dtype,
                        f"{case} device {i} accumulated")


@pytest.mark.parametrize("case", [c for c in CASES if c[0] == "bf16"])
def test_ring_block_step_accumulate_onto_any_running_result(sp, case):
    """A running result that is not a ring's own (random rows, random finite
    lse, some rows at -inf): every pair (i, j) folded onto it must equal the
    oracle's two-way merge of it with the pair's partial, and rows with no
    allowed key in block j keep their bits."""
    dtype, B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4400 + S, dtype)
    pos = _positions(pos_kind, B, S, 80)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    qn, kn, vn = np32(q), np32(k), np32(v)
    ws = sp.attention_workspace(B, S, pos is not None)
    blocks = [oracle.block_tokens(S, P, p, order) for p in range(P)]
    g = torch.Generator(device="cuda").manual_seed(4401 + S)
    Lb = S // P
    for s in range(P):
        part_o, part_l = oracle.ring_partial(qn, kn, vn, P, s, order, pos)
        for i in range(P):
            j = (i - s) % P
            tok = blocks[i]
            # |x| < 3: half a bf16 ulp stays below the output bar
            run_o = (torch.randn((B, Lb, Hq, d), generator=g, device="cuda") * 0.5).to(q.dtype)
            run_l = torch.randn((B, Hq, Lb), generator=g, device="cuda") * 4
            run_l[:, :, ::7] = float("-inf")
            run_o[:, ::7] = float("nan")   # not read: those rows' lse is -inf
            out, lse = run_o.clone(), run_l.clone()
            sp.ring_block_step_accumulate(_block(q, tok), _block(k, blocks[j]),
                                          _block(v, blocks[j]), P, i, j, out, lse, order, tpos,
                                          workspace=ws)
            torch.cuda.synchronize()
            rl_in = run_l.cpu().numpy()
            ro_in = np.where(np.isfinite(rl_in).transpose(0, 2, 1)[..., None],
                             np32(run_o), 0.0)
            ro, rl = oracle.merge_partials(np.stack([ro_in, part_o[:, tok]]),
                                           np.stack([rl_in, part_l[:, :, tok]]))
            fin = np.isfinite(rl)
            mask = fin.transpose(0, 2, 1)[..., None]
            check_attention(np.where(mask, np32(out), 0.0), lse.cpu().numpy(),
                            np.where(mask, ro, 0.0), rl, dtype, f"{case} i={i} j={j}")
            # rows with no key in block j: untouched, bit for bit
            keep = torch.from_numpy(~np.isfinite(part_l[:, :, tok])).cuda()  # [B][Hq][Lb]
            keep_rows = keep.transpose(1, 2)  # [B][Lb][Hq]
            assert torch.equal(lse[keep], run_l[keep])
            assert torch.equal(out.view(torch.int16)[keep_rows], run_o.view(torch.int16)[keep_rows])


@pytest.mark.parametrize("case", [CASES[1], CASES[4], CASES[5]])
def test_library_kernels_accumulate_both_paths(sp, case):
    """dist.LibraryKernels.ring_step_accumulate, as dist.ring_attention calls
    it: one accumulating call for bf16 with d = 128, else the step into a
    temporary and the merge.  Device i's ring folded step by step equals
    block i's rows of full attention."""
    from sequence_parallelism_gb300 import dist as spd
    dtype, B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4600 + S, dtype)
    pos = _positions(pos_kind, B, S, 82)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    full_o, full_l = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    kern = spd.LibraryKernels()
    blocks = [oracle.block_tokens(S, P, p, order) for p in range(P)]
    for i in range(P):
        tok = blocks[i]
        out = torch.empty((B, S // P, Hq, d), dtype=q.dtype, device="cuda")
        lse = torch.empty((B, Hq, S // P), dtype=torch.float32, device="cuda")
        for s in range(P):
            j = (i - s) % P
            args = (_block(q, tok), _block(k, blocks[j]), _block(v, blocks[j]), tpos, S, P,
                    order, i, j, out, lse)
            if s == 0:
                kern.ring_step(*args)
            else:
                kern.ring_step_accumulate(*args)
        torch.cuda.synchronize()
        check_attention(np32(out), lse.cpu().numpy(), full_o[:, tok], full_l[:, :, tok], dtype,
                        f"{case} device {i}")


@pytest.mark.parametrize("case", CASES)
def test_query_block_against_whole_sequence(sp, case):
    from sequence_parallelism_gb300 import _lib
    dtype, B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4200 + S, dtype)
    pos = _positions(pos_kind, B, S, 78)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    full_o, full_l = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    ws = sp.attention_workspace(B, S, pos is not None)
    ref_out, ref_lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    for i in range(P):
        tok = oracle.block_tokens(S, P, i, order)
        out = torch.full((B, S // P, Hq, d), float("nan"), dtype=q.dtype, device="cuda")
        lse = torch.full((B, Hq, S // P), float("nan"), dtype=torch.float32, device="cuda")
        _lib.sp_query_block_attn_fwd(_block(q, tok), k, v, tpos, P, order, i, 0.0, out, lse, ws)
        torch.cuda.synchronize()
        check_attention(np32(out), lse.cpu().numpy(), full_o[:, tok], full_l[:, :, tok], dtype,
                        f"{case} query block {i}")
        if pos is not None:
            # causal calls visit the same tiles in the same order as the
            # whole-sequence call: the same bits
            ti = torch.from_numpy(tok).cuda()
            assert torch.equal(out, ref_out[:, ti]) and torch.equal(lse, ref_lse[:, :, ti])


@pytest.mark.parametrize("case", [c for c in CASES if c[0] == "bf16"])
def test_ring_block_step_backward_every_pair(sp, case):
    """Every (query block i, key/value block j) pair's gradient parts against
    oracle.ring_partial_backward on the same inputs (our forward's out and
    lse, as a training step would use), then the sums -- dq over j, dk and
    dv over i -- against the whole gradients of the oracle and against the
    whole-sequence backward on the GPU."""
    from sequence_parallelism_gb300 import _lib
    dtype, B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4500 + S, dtype)
    g = torch.Generator(device="cuda").manual_seed(4501 + S)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(q.dtype)
    pos = _positions(pos_kind, B, S, 81)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    Lb = S // P
    blocks = [oracle.block_tokens(S, P, p, order) for p in range(P)]
    ws = torch.empty(_lib.sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, pos is not None),
                     dtype=torch.uint8, device="cuda")
    tl = lambda t, p: t[:, :, torch.from_numpy(blocks[p]).cuda()].contiguous()
    dq = torch.zeros((B, S, Hq, d), dtype=torch.float64)
    dk = torch.zeros((B, S, Hkv, d), dtype=torch.float64)
    dv = torch.zeros((B, S, Hkv, d), dtype=torch.float64)
    for i in range(P):
        for j in range(P):
            acc = [torch.zeros((B, Lb, h, d), dtype=torch.float32, device="cuda")
                   for h in (Hq, Hkv, Hkv)]
            args = (_block(q, blocks[i]), _block(k, blocks[j]), _block(v, blocks[j]),
                    _block(out, blocks[i]), _block(dout, blocks[i]), tl(lse, i))
            _lib.sp_ring_block_step_bwd(*args, tpos, S, P, order, i, j, 0.0, *acc, ws)
            torch.cuda.synchronize()
            if pos is not None and order == "contiguous" and j > i:
                assert _lib.sp_last_launch_count() == 0   # nothing allowed: no launch
            ref = oracle.ring_partial_backward(*(np32(a) for a in args[:5]),
                                               args[5].cpu().numpy(), S, P, i, j, order, pos)
            for name, got, r in zip(("dq", "dk", "dv"), acc, ref):
                check_grad(got.cpu().numpy(), r, "bf16", f"{case} pair ({i}, {j}) {name}")
            dq[:, blocks[i]] += acc[0].cpu().double()
            dk[:, blocks[j]] += acc[1].cpu().double()
            dv[:, blocks[j]] += acc[2].cpu().double()
    assert _lib.sp_get_device_error(ws) == (0, 0)
    ref_g = oracle.attention_backward(np32(q), np32(k), np32(v), np32(dout), pos)
    whole = sp.blockwise_attention_backward(q, k, v, out, dout, lse, P, order, tpos)
    torch.cuda.synchronize()
    for name, got, r, w in zip(("dq", "dk", "dv"), (dq, dk, dv), ref_g, whole):
        check_grad(got.numpy(), r, "bf16", f"{case} summed {name}")
        # the same products summed in another order: within bf16 rounding of the whole call
        check_grad(got.numpy(), np32(w).astype(np.float64), "bf16", f"{case} vs whole {name}")


def test_ring_block_step_backward_helper_and_errors(sp):
    """sp.ring_block_step_backward gives the C call's bits; bad block indices,
    float32 tensors, float32-less accumulators and a short workspace are
    refused before any launch."""
    from sequence_parallelism_gb300 import _lib
    B, S, Hq, Hkv, d, P = 1, 512, 2, 1, 128, 4
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4600, "bf16")
    dout = torch.randn_like(q)
    tpos = torch.from_numpy(_positions("causal", B, S, 82)).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, "contiguous", tpos)
    blk = lambda t: t[:, 256:384].contiguous()
    lse_b = lse[:, :, 256:384].contiguous()
    args = (blk(q), blk(k), blk(v), blk(out), blk(dout), lse_b)
    h = sp.ring_block_step_backward(*args, P, 2, 2, "contiguous", tpos)
    ws = torch.empty(_lib.sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, True),
                     dtype=torch.uint8, device="cuda")
    acc = [torch.zeros_like(t, dtype=torch.float32) for t in (blk(q), blk(k), blk(v))]
    _lib.sp_ring_block_step_bwd(*args, tpos, S, P, "contiguous", 2, 2, 0.0, *acc, ws)
    torch.cuda.synchronize()
    for a_, b_ in zip(h, acc):
        assert torch.equal(a_, b_)
    for i, j in ((4, 0), (0, 4), (-1, 0)):
        with pytest.raises(_lib.SPError):
            _lib.sp_ring_block_step_bwd(*args, tpos, S, P, "contiguous", i, j, 0.0, *acc, ws)
    f32 = [t.float() for t in args[:5]]
    with pytest.raises(_lib.SPError, match="not supported|unsupported"):
        _lib.sp_ring_block_step_bwd(*f32, lse_b, tpos, S, P, "contiguous", 0, 0, 0.0, *acc, ws)
    with pytest.raises(ValueError):
        _lib.sp_ring_block_step_bwd(*args, tpos, S, P, "contiguous", 0, 0, 0.0, acc[0].double(),
                                    acc[1], acc[2], ws)
    with pytest.raises(_lib.SPError):
        _lib.sp_ring_block_step_bwd(*args, tpos, S, P, "contiguous", 0, 0, 0.0, *acc, ws[:256])
    assert _lib.sp_last_launch_count() == 0


def test_package_helpers_match_the_c_calls(sp):
    """sp.ring_block_step / sp.query_block_attention allocate their outputs
    and give the same bits as the C entry points."""
    from sequence_parallelism_gb300 import _lib
    B, S, Hq, Hkv, d, P = 1, 768, 2, 1, 128, 3
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4400, "bf16")
    pos = torch.from_numpy(_positions("packed", B, S, 80)).cuda()
    blocks = [oracle.block_tokens(S, P, p, "striped") for p in range(P)]
    o1, l1 = sp.ring_block_step(_block(q, blocks[2]), _block(k, blocks[0]), _block(v, blocks[0]),
                                P, 2, 0, "striped", pos)
    ws = sp.attention_workspace(B, S, True)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    _lib.sp_ring_block_step(_block(q, blocks[2]), _block(k, blocks[0]), _block(v, blocks[0]), pos,
                            S, P, "striped", 2, 0, 0.0, o2, l2, ws)
    o3, l3 = sp.query_block_attention(_block(q, blocks[1]), k, v, P, 1, "striped", pos)
    o4, l4 = sp.blockwise_attention(q, k, v, P, "striped", pos)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    t1 = torch.from_numpy(blocks[1]).cuda()
    assert torch.equal(o3, o4[:, t1]) and torch.equal(l3, l4[:, :, t1])


def test_per_device_argument_errors(sp):
    from sequence_parallelism_gb300 import _lib
    q, k, v = workloads.small_case(1, 512, 2, 1, 128, 5, "bf16")
    blk = lambda t: t[:, :128].contiguous()
    ws = sp.attention_workspace(1, 512, False)
    out = torch.empty_like(blk(q))
    lse = torch.empty((1, 2, 128), dtype=torch.float32, device="cuda")
    for i, j in ((4, 0), (0, 4), (-1, 0)):
        with pytest.raises(_lib.SPError):
            _lib.sp_ring_block_step(blk(q), blk(k), blk(v), None, 512, 4, "contiguous", i, j, 0.0,
                                    out, lse, ws)
    with pytest.raises(_lib.SPError):
        _lib.sp_query_block_attn_fwd(blk(q), k, v, None, 4, "contiguous", 4, 0.0, out, lse, ws)
    assert _lib.sp_last_launch_count() == 0


def test_data_plane_on_one_rank_runs_the_library_kernels(sp):
    """sequence_parallelism_gb300.dist with its default kernels on a
    one-rank NCCL group (the only group one GPU allows): the ring, the
    all-gathered variant and the Ulysses layer reduce to their per-device
    calls and must match the oracle.  The exchanges between ranks are
    covered by tests/test_dist_cpu.py on gloo ranks."""
    import socket
    import torch.distributed as dist
    from sequence_parallelism_gb300 import dist as spd
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        B, S, Hq, Hkv, d = 1, 640, 4, 2, 128
        q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 4300, "bf16")
        pos = _positions("packed", B, S, 79)
        tpos = torch.from_numpy(pos).cuda()
        ref_o, ref_l = oracle.full_attention(np32(q), np32(k), np32(v), pos)
        for fn in (spd.ring_attention, spd.allgather_kv_attention):
            out, lse = fn(q, k, v, tpos, "contiguous")
            torch.cuda.synchronize()
            check_attention(np32(out), lse.cpu().numpy(), ref_o, ref_l, "bf16", fn.__name__)
        out, ctx = spd.ulysses_attention(q, k, v, tpos, ring_blocks=2, return_context=True)
        torch.cuda.synchronize()
        err = np.abs(np32(out).astype(np.float64) - ref_o)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3
        g = torch.Generator(device="cuda").manual_seed(4301)
        dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
        grads = spd.ulysses_attention_backward(ctx, dout)
        torch.cuda.synchronize()
        ref_g = oracle.attention_backward(np32(q), np32(k), np32(v), np32(dout), pos)
        for name, got, ref in zip(("dq", "dk", "dv"), grads, ref_g):
            check_grad(np32(got), ref, "bf16", f"one-rank Ulysses {name}")
        out, lse = spd.ring_attention(q, k, v, tpos, "contiguous")
        grads = spd.ring_attention_backward(q, k, v, out, dout, lse, tpos, "contiguous")
        torch.cuda.synchronize()
        for name, got, ref in zip(("dq", "dk", "dv"), grads, ref_g):
            check_grad(np32(got), ref, "bf16", f"one-rank ring backward {name}")
    finally:
        dist.destroy_process_group()
