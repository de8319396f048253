"""GPU parity of blockwise attention (fp32 CUDA-core and bf16 tcgen05 paths),
of single ring steps and of the partial merge, against the float64 oracle on
the same seeded inputs.  Sizes span several 128-row tiles, ragged tails,
GQA, packed documents with length-1 documents, P from 1 to 16, both block
orders."""

import numpy as np
import pytest
import torch

import oracle
from helpers import BF16_MAX_ABS, F32_MAX_ABS, check_attention, np32, torch_dtype
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def _positions(kind, B, S, seed):
    if kind == "none":
        return None
    if kind == "causal":
        return np.tile(np.arange(S, dtype=np.int32), (B, 1))
    rows = []
    for b in range(B):  # packed documents, a few of length 1, not tile-aligned
        rng = np.random.default_rng(seed + b)
        cuts = np.sort(rng.choice(np.arange(1, S), 6, replace=False))
        cuts = np.unique(np.concatenate([cuts, [cuts[0] + 1, S - 1]]))
        lengths = np.diff(np.concatenate([[0], cuts, [S]]))
        rows.append(workloads.position_ids_from_lengths(lengths))
    return np.stack(rows).astype(np.int32)


def _run(sp, dtype, B, S, Hq, Hkv, d, P, order, pos_kind, seed):
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, seed, dtype)
    pos = _positions(pos_kind, B, S, seed)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    return check_attention(np32(out), lse.cpu().numpy(), ref_out, ref_lse, dtype,
                           f"{dtype} S={S} P={P} {order} {pos_kind}")


def test_ring_tiny_f32(sp):
    """The Ring Attention page's example: 4 blocks of 8 tokens, d = 16, fp32,
    matches full attention within 1e-5 (the page's allclose tolerance)."""
    qn, kn, vn = workloads.ring_tiny_arrays()
    as4 = lambda a: torch.from_numpy(a)[None, :, None, :].contiguous().cuda()
    q, k, v = as4(qn), as4(kn), as4(vn)
    out, lse = sp.blockwise_attention(q, k, v, 4, "contiguous")
    torch.cuda.synchronize()
    as4n = lambda a: a.astype(np.float64)[None, :, None, :]
    ref_out, ref_lse = oracle.full_attention(as4n(qn), as4n(kn), as4n(vn))
    check_attention(np32(out), lse.cpu().numpy(), ref_out, ref_lse, "f32", "ring_tiny")
    assert np.abs(np32(out) - ref_out).max() <= 1e-5


@pytest.mark.parametrize("B,S,Hq,Hkv,d,P,order,pos", [
    (1, 32, 1, 1, 16, 1, "contiguous", "none"),
    (2, 96, 4, 2, 64, 3, "contiguous", "causal"),
    (2, 96, 4, 2, 64, 3, "striped", "packed"),
    (1, 200, 3, 1, 100, 4, "striped", "causal"),
    (1, 160, 2, 2, 256, 8, "contiguous", "packed"),
    (1, 64, 2, 1, 7, 16, "striped", "none"),
])
def test_f32_parity(sp, B, S, Hq, Hkv, d, P, order, pos):
    _run(sp, "f32", B, S, Hq, Hkv, d, P, order, pos, 100 + S)


@pytest.mark.parametrize("B,S,Hq,Hkv,P,order,pos", [
    (1, 128, 1, 1, 1, "contiguous", "none"),      # one tile
    (1, 1024, 2, 2, 1, "contiguous", "none"),     # 4 Q tiles, 8 KV tiles
    (2, 1000, 4, 2, 2, "contiguous", "none"),     # ragged tail (500 rows per block), GQA
    (1, 1200, 4, 1, 4, "striped", "none"),        # MQA, striped, ragged
    (1, 2048, 4, 2, 4, "contiguous", "causal"),
    (1, 2048, 4, 2, 4, "striped", "causal"),
    (2, 1536, 2, 1, 2, "contiguous", "packed"),
    (2, 1536, 2, 1, 3, "striped", "packed"),
    (1, 4096, 2, 2, 16, "striped", "causal"),
    (1, 4096, 2, 2, 16, "contiguous", "causal"),
    (1, 768, 3, 3, 8, "contiguous", "packed"),    # blocks of 96 rows (< one tile)
])
def test_bf16_parity(sp, B, S, Hq, Hkv, P, order, pos):
    _run(sp, "bf16", B, S, Hq, Hkv, 128, P, order, pos, 200 + S + P)


@pytest.mark.parametrize("dtype,B,S,Hq,Hkv,P,order,pos", [
    ("bf16", 2, 1, 2, 1, 1, "contiguous", "causal"),     # a single token
    ("bf16", 1, 1, 1, 1, 1, "striped", "none"),
    ("bf16", 1, 256, 2, 1, 256, "contiguous", "causal"),  # one token per block
    ("bf16", 1, 256, 2, 2, 256, "striped", "packed"),
    ("bf16", 1, 256, 4, 1, 256, "striped", "none"),       # ... with the tail split
    ("f32", 2, 1, 2, 1, 1, "contiguous", "causal"),
    ("f32", 1, 64, 2, 1, 64, "striped", "packed"),
])
def test_degenerate_shapes(sp, dtype, B, S, Hq, Hkv, P, order, pos):
    """The smallest shapes the method admits: one token in all, and blocks of
    one token each (every ring step then brings a single key)."""
    _run(sp, dtype, B, S, Hq, Hkv, 128 if dtype == "bf16" else 16, P, order, pos, 900 + S + P)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_masked_scores_never_set_the_exponent_base(sp, dtype, order):
    """Causal rows t < 1000 share key tiles with keys j >= 1000 that they may
    not see and whose scores are about 102 (147 in log2 units) while every
    key they may see scores about N(0, 1).  Had a masked score entered a
    row's running max, the allowed weights (2^-140 and below) would flush to
    zero and the row would come out as zeros; rows t >= 1000 see the large
    keys and average their values uniformly."""
    B, S, H, d, P = 1, 2048, 1, 128, 2
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)
    q = torch.ones((B, S, H, d), device="cuda")
    k = torch.randn((B, S, H, d), generator=g, device="cuda")
    k[:, 1000:] = 9.0
    v = torch.randn((B, S, H, d), generator=g, device="cuda")
    q, k, v = (x.to(torch_dtype(dtype)).contiguous() for x in (q, k, v))
    pos = _positions("causal", B, S, 0)
    out, lse = sp.blockwise_attention(q, k, v, P, order, torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    o, l = np32(out), lse.cpu().numpy()
    check_attention(o[:, :1000], l[:, :, :1000], ref_out[:, :1000], ref_lse[:, :, :1000], dtype,
                    f"{dtype} {order} rows beside large masked scores")
    assert np.abs(o[0, 990:1000]).max() > 0.05
    # rows that see the large keys: lse near 105, compared relatively
    tol = BF16_MAX_ABS if dtype == "bf16" else F32_MAX_ABS
    assert np.abs(o[:, 1000:] - ref_out[:, 1000:]).max() <= tol
    rel = np.abs(l[:, :, 1000:] - ref_lse[:, :, 1000:]) / np.abs(ref_lse[:, :, 1000:])
    assert rel.max() <= 1e-5


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 32)])
@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_ring_steps_merge_to_full(sp, dtype, d, order):
    """Each ring step alone matches the oracle's per-step partial (rows with
    no key in that block give 0 / -inf), and merging the P partials on the
    GPU reproduces full attention."""
    B, S, Hq, Hkv, P = 1, 1024, 2, 1, 4
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 300, dtype)
    pos = _positions("packed", B, S, 300)
    tpos = torch.from_numpy(pos).cuda()
    qn, kn, vn = np32(q), np32(k), np32(v)
    outs = torch.empty((P, B, S, Hq, d), dtype=torch_dtype(dtype), device="cuda")
    lses = torch.empty((P, B, Hq, S), dtype=torch.float32, device="cuda")
    for s in range(P):
        sp.ring_step(q, k, v, P, s, order, tpos, out=outs[s], lse=lses[s])
        torch.cuda.synchronize()
        ro, rl = oracle.ring_partial(qn, kn, vn, P, s, order, pos)
        check_attention(np32(outs[s]), lses[s].cpu().numpy(), ro, rl, dtype, f"step {s}")
    out, lse = sp.merge_partials(outs, lses)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.full_attention(qn, kn, vn, pos)
    check_attention(np32(out), lse.cpu().numpy(), ref_out, ref_lse, dtype, "merged")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_merge_partials_parity(sp, dtype):
    P, B, S, H, d = 5, 2, 37, 3, 48
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    outs = torch.randn((P, B, S, H, d), generator=g, device="cuda").to(torch_dtype(dtype))
    lses = torch.randn((P, B, H, S), generator=g, device="cuda") * 3
    lses[1, :, :, :5] = float("-inf")   # empty partials get weight 0
    lses[:, 1, 2, 7] = float("-inf")    # a row with nothing at all
    out, lse = sp.merge_partials(outs, lses)
    torch.cuda.synchronize()
    ro, rl = oracle.merge_partials(np32(outs).astype(np.float64), lses.cpu().numpy())
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert np.abs(np32(out) - ro).max() <= tol
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin)
    assert np.abs(lse.cpu().numpy()[fin] - rl[fin]).max() <= 1e-5
    assert (np32(out)[1, 7, 2] == 0).all()


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 9])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("bf16", 256), ("bf16", 48),
                                     ("f32", 128), ("f32", 32)])
def test_merge_partials_every_form(sp, P, dtype, d):
    """Every kernel form of the merge (16-byte pieces with room for 2, 4 or 8
    partials; one warp per row for head sizes that do not split into pieces
    dividing a warp, or more than 8 partials) against the oracle's merge.
    The oracle gets the same rounded inputs, so the result differs from it
    only by float32 arithmetic and one rounding of the output: at most half
    an output ulp (at most 2^-8 of |x| for bf16's 8 significant bits, 2^-24
    for float32's 24) plus float32 noise."""
    B, S, H = 2, 97, 3   # 582 rows: several warps' worth of rows and a ragged tail
    g = torch.Generator(device="cuda")
    g.manual_seed(900 + 10 * P + d)
    outs = torch.randn((P, B, S, H, d), generator=g, device="cuda").to(torch_dtype(dtype))
    lses = torch.randn((P, B, H, S), generator=g, device="cuda") * 3
    lses[0, :, :, :6] = float("-inf")      # an empty partial gets weight 0
    lses[:, 1, 2, 50] = float("-inf")      # a row with nothing at all
    out, lse = sp.merge_partials(outs, lses)
    torch.cuda.synchronize()
    ro, rl = oracle.merge_partials(np32(outs).astype(np.float64), lses.cpu().numpy())
    got = np32(out).astype(np.float64)
    half_ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -24
    err = np.abs(got - ro) - (half_ulp * np.abs(ro) + 4e-6 * np.abs(ro).max())
    assert err.max() <= 0, f"P={P} {dtype} d={d}: excess {err.max():.3g}"
    fin = np.isfinite(rl)
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.abs(lg[fin] - rl[fin]).max() <= 1e-5
    assert (np32(out)[1, 50, 2] == 0).all()


def test_constant_values_give_ones(sp):
    """v = 1: every softmax row sums to one (bf16 P rounding is the only
    error)."""
    B, S, Hq, Hkv = 1, 2048, 2, 1
    q, k, _ = workloads.small_case(B, S, Hq, Hkv, 128, 400, "bf16")
    v = torch.ones((B, S, Hkv, 128), dtype=torch.bfloat16, device="cuda")
    pos = torch.from_numpy(_positions("packed", B, S, 400)).cuda()
    out, _ = sp.blockwise_attention(q, k, v, 4, "striped", pos)
    torch.cuda.synchronize()
    assert np.abs(np32(out) - 1.0).max() <= 1e-2


def test_zero_query_closed_form(sp):
    """q = 0: out = mean of the allowed values, lse = ln(position + 1)."""
    B, S, Hq, Hkv = 1, 1536, 2, 2
    _, k, v = workloads.small_case(B, S, Hq, Hkv, 128, 401, "bf16")
    q = torch.zeros((B, S, Hq, 128), dtype=torch.bfloat16, device="cuda")
    pos = _positions("packed", B, S, 401)
    out, lse = sp.blockwise_attention(q, k, v, 2, "contiguous", torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    expect = np.log(pos[0].astype(np.float64) + 1.0)
    assert np.abs(lse.cpu().numpy()[0] - expect[None, :]).max() <= 1e-3
    ref_out, _ = oracle.full_attention(np32(q), np32(k), np32(v), pos)
    assert np.abs(np32(out) - ref_out).max() <= 2e-2


def test_no_device_error_reported(sp):
    B, S = 1, 1024
    q, k, v = workloads.small_case(B, S, 2, 2, 128, 402, "bf16")
    ws = sp.attention_workspace(B, S, False, minimal=True)
    sp.blockwise_attention(q, k, v, 2, "contiguous", workspace=ws)
    from sequence_parallelism_gb300 import _lib
    st, code = _lib.sp_get_device_error(ws)
    assert st == 0 and code == 0
    assert _lib.sp_last_launch_count() == 1


def test_repeated_calls_share_one_workspace(sp):
    """Calls of different shapes and kinds, repeated and interleaved, through
    one workspace: each call resets the work counter and the error word it
    keeps there, so every repeat reproduces its first result bit for bit
    (the kernels are deterministic) and the first results match the oracle."""
    from sequence_parallelism_gb300 import _lib
    shapes = [  # (B, S, Hq, Hkv, P, order, pos kind)
        (1, 2048, 4, 2, 4, "contiguous", "causal"),
        (2, 1000, 4, 2, 2, "contiguous", "none"),     # takes the tail split
        (1, 1536, 2, 1, 3, "striped", "packed"),
    ]
    n = max(_lib.sp_blockwise_attn_split_workspace_bytes(B, S, pos != "none")
            for B, S, _, _, _, _, pos in shapes)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    cases, first = [], []
    for c, (B, S, Hq, Hkv, P, order, kind) in enumerate(shapes):
        q, k, v = workloads.small_case(B, S, Hq, Hkv, 128, 600 + c, "bf16")
        pos = _positions(kind, B, S, 600 + c)
        cases.append((q, k, v, P, order, None if pos is None else torch.from_numpy(pos).cuda(),
                      pos))
    for rep in range(4):
        for c, (q, k, v, P, order, tpos, pos) in enumerate(cases):
            out, lse = sp.blockwise_attention(q, k, v, P, order, tpos, workspace=ws)
            torch.cuda.synchronize()
            st, code = _lib.sp_get_device_error(ws)
            assert st == 0 and code == 0
            if rep == 0:
                first.append((out.clone(), lse.clone()))
                ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos)
                check_attention(np32(out), lse.cpu().numpy(), ref_out, ref_lse, "bf16",
                                f"shape {c}")
            else:
                assert torch.equal(out.view(torch.int16), first[c][0].view(torch.int16)), (rep, c)
                assert torch.equal(lse, first[c][1]), (rep, c)


def test_calls_on_a_side_stream(sp):
    """The binding launches on torch's current stream: work queued on a side
    stream is ordered after that stream's earlier work and gives the same
    result as on the default stream."""
    B, S, Hq, Hkv, P = 1, 2048, 4, 2, 4
    q, k, v = workloads.small_case(B, S, Hq, Hkv, 128, 610, "bf16")
    pos = _positions("causal", B, S, 610)
    tpos = torch.from_numpy(pos).cuda()
    out0, lse0 = sp.blockwise_attention(q, k, v, P, "contiguous", tpos)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        q2 = q.clone()             # produced on the side stream ...
        out1, lse1 = sp.blockwise_attention(q2, k, v, P, "contiguous", tpos)  # ... and read there
        y = sp.seq_to_head(q2, P)
        back = sp.head_to_seq(y)
    side.synchronize()
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
    assert torch.equal(lse1, lse0)
    assert torch.equal(back, q)


def test_fused_ulysses_is_bit_identical_to_permuted_pipeline(sp):
    """On one GPU, attention on the sequence-sharded tensors computes every
    Ulysses head group in place: same result, bit for bit, with no
    permutation traffic."""
    B, S, H, P = 1, 2048, 8, 4
    q, k, v = workloads.small_case(B, S, H, H, 128, 500, "bf16")
    piped = sp.ulysses_attention(q, k, v, P)
    fused = sp.ulysses_attention(q, k, v, P, fused=True)
    torch.cuda.synchronize()
    assert torch.equal(piped.view(torch.int16), fused.view(torch.int16))
    ref, _ = oracle.full_attention(np32(q), np32(k), np32(v))
    check_attention(np32(fused), np.zeros((B, H, S)), ref, np.zeros((B, H, S)), "bf16", "fused")


@pytest.mark.parametrize("B,S,Hq,Hkv,P_u,P_r,order,pos", [
    (1, 2048, 4, 4, 4, 2, "striped", "causal"),     # one head per Ulysses group
    (2, 1536, 4, 2, 2, 3, "contiguous", "packed"),  # GQA inside each group
    (1, 1024, 2, 2, 2, 4, "striped", "none"),
])
def test_ulysses_ring_hybrid_parity(sp, B, S, Hq, Hkv, P_u, P_r, order, pos):
    q, k, v = workloads.small_case(B, S, Hq, Hkv, 128, 600 + S, "bf16")
    pos_np = _positions(pos, B, S, 600)
    tpos = None if pos_np is None else torch.from_numpy(pos_np).cuda()
    out, lse = sp.ulysses_ring_attention(q, k, v, P_u, P_r, order, tpos)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v), pos_np)
    G = Hq // P_u
    lse_nat = lse.permute(1, 0, 2, 3).reshape(B, Hq, S).cpu().numpy()  # [P_u][B][G][S] -> [B][H][S]
    check_attention(np32(out), lse_nat, ref_out, ref_lse, "bf16", f"hybrid {P_u}x{P_r} {order}")
    assert G >= 1


@pytest.mark.parametrize("B,S,Hq,Hkv,P,order", [
    (2, 1000, 4, 2, 2, "contiguous"),   # 8 items: every item split into pieces
    (1, 4096, 10, 5, 4, "striped"),     # 160 items: a full wave plus 8 split items
])
def test_tail_split_and_single_launch_agree_with_oracle(sp, B, S, Hq, Hkv, P, order):
    """Non-causal calls with the larger workspace split the items of their
    last wave and merge fp32 partials; with the minimal workspace every item
    runs whole in one launch.  Both match the oracle."""
    from sequence_parallelism_gb300 import _lib
    q, k, v = workloads.small_case(B, S, Hq, Hkv, 128, 700 + S, "bf16")
    ref_out, ref_lse = oracle.full_attention(np32(q), np32(k), np32(v))
    launches = {}
    for minimal in (True, False):
        ws = sp.attention_workspace(B, S, False, minimal=minimal)
        out, lse = sp.blockwise_attention(q, k, v, P, order, workspace=ws)
        launches[minimal] = _lib.sp_last_launch_count()
        torch.cuda.synchronize()
        check_attention(np32(out), lse.cpu().numpy(), ref_out, ref_lse, "bf16",
                        f"minimal={minimal}")
    assert launches[True] == 1 and launches[False] >= 2


def test_barrier_timeout_is_reported_and_context_survives(sp):
    """A wait that can never complete ends after its limit with the timeout
    code in the workspace error word (SP_ERR_DEVICE_TIMEOUT), and the
    context keeps working: no fault, no hang."""
    from sequence_parallelism_gb300 import _lib
    ws = sp.attention_workspace(1, 1024, False, minimal=True)
    _lib.sp_check_barrier_timeout(ws, 20000)  # 20 ms
    st, code = _lib.sp_get_device_error(ws)
    assert st == _lib.SP_ERR_DEVICE_TIMEOUT and code == 0x1F0
    st, code = _lib.sp_get_device_error(ws)     # reading clears the word
    assert st == 0 and code == 0
    _run(sp, "bf16", 1, 1024, 2, 2, 128, 2, "contiguous", "causal", 901)
