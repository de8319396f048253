"""A seeded random sweep of shapes against the float64 oracle: batch size,
number of ring blocks P (1 to 16), rows per block (ragged, from 1 up), GQA
ratio, head size (f32), block order and mask kind (none, causal, packed
documents) drawn together, so that combinations the hand-picked cases miss
are exercised too.  The draws are fixed by the seed; each case prints its
shape when it fails."""

import numpy as np
import pytest

from test_gpu_attention import _run
from test_gpu_backward import _run_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def _draw(rng, dtype, max_tokens):
    P = int(rng.integers(1, 17))
    Lb = int(rng.integers(1, max(2, max_tokens // P)))
    S = P * Lb
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    d = 128 if dtype == "bf16" else int(rng.choice([16, 40, 64, 128, 200]))
    order = str(rng.choice(["contiguous", "striped"]))
    # packed documents need at least seven tokens to cut
    pos = str(rng.choice(["none", "causal", "packed"] if S >= 8 else ["none", "causal"]))
    return B, S, Hq, Hkv, d, P, order, pos


def _cases(seed, dtype, n, max_tokens):
    rng = np.random.default_rng(seed)
    return [_draw(rng, dtype, max_tokens) for _ in range(n)]


def _id(case):
    B, S, Hq, Hkv, d, P, order, pos = case
    return f"B{B}-S{S}-H{Hq}x{Hkv}-d{d}-P{P}-{order}-{pos}"


@pytest.mark.parametrize("case", _cases(2024, "bf16", 40, 2400), ids=_id)
def test_random_bf16_forward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run(sp, "bf16", B, S, Hq, Hkv, d, P, order, pos, 1300 + S)


@pytest.mark.parametrize("case", _cases(2025, "f32", 20, 300), ids=_id)
def test_random_f32_forward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run(sp, "f32", B, S, Hq, Hkv, d, P, order, pos, 1400 + S)


@pytest.mark.parametrize("case", _cases(2026, "bf16", 12, 700), ids=_id)
def test_random_bf16_backward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run_bwd(sp, "bf16", B, S, Hq, Hkv, d, P, order, pos, 1500 + S)


@pytest.mark.parametrize("case", _cases(2027, "f32", 10, 160), ids=_id)
def test_random_f32_backward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run_bwd(sp, "f32", B, S, Hq, Hkv, d, P, order, pos, 1600 + S)


def _perm_draw(rng):
    P = int(rng.integers(1, 9))
    G = int(rng.integers(1, 5))       # heads per group
    d = int(rng.choice([16, 24, 64, 96, 128, 200]))
    dtype = str(rng.choice(["bf16", "f32"]))
    B = int(rng.integers(1, 3))
    S = P * int(rng.integers(1, 300))
    n = int(rng.choice([1, 3]))       # tensors per launch (3: q, k, v with their own groups)
    Gk = int(rng.integers(1, G + 1))
    return B, S, G * P, Gk * P, d, P, dtype, n


@pytest.mark.parametrize("case", [_perm_draw(np.random.default_rng(2028 + i)) for i in range(30)],
                         ids=lambda c: "B{}-S{}-H{}x{}-d{}-P{}-{}-n{}".format(*c))
def test_random_permutation_both_kernels(sp, case):
    """Seeded shapes through both permutation kernels (the TMA-staged one
    wherever its rules hold), bit-exact against the oracle's index loops,
    with a round trip; three-tensor launches move q, k, v together."""
    import torch
    import oracle
    from sequence_parallelism_gb300 import _lib
    B, S, Hq, Hkv, d, P, dtype, n = case
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    bits = torch.int16 if dtype == "bf16" else torch.int32
    g = torch.Generator(device="cuda").manual_seed(S + d)
    xs = [torch.randn((B, S, H, d), generator=g, device="cuda").to(tdt)
          for H in ((Hq, Hkv, Hkv) if n == 3 else (Hq,))]
    for threshold in (0, 128 << 20):
        prev = _lib.sp_permute_set_bulk_min_bytes(threshold)
        try:
            ys = [torch.empty((P, B, S, x.shape[2] // P, d), dtype=tdt, device="cuda") for x in xs]
            if n == 3:
                _lib.sp_ulysses_seq_to_head_qkv(*xs, *ys, P)
            else:
                _lib.sp_ulysses_seq_to_head(xs[0], ys[0], P)
            backs = [torch.empty_like(x) for x in xs]
            for y, bk in zip(ys, backs):
                _lib.sp_ulysses_head_to_seq(y, bk, P)
            torch.cuda.synchronize()
        finally:
            _lib.sp_permute_set_bulk_min_bytes(prev)
        for x, y, bk in zip(xs, ys, backs):
            ref = oracle.seq_to_head(x.view(bits).cpu().numpy(), P)
            assert np.array_equal(y.view(bits).cpu().numpy(), ref), (case, threshold)
            assert torch.equal(bk.view(bits), x.view(bits)), (case, threshold)
    assert _lib.sp_get_permute_error() == (0, 0)


@pytest.mark.parametrize("case", _cases(2029, "bf16", 10, 1600), ids=_id)
def test_random_ring_block_pairs(sp, case):
    """Seeded shapes through sp_ring_block_step for two random (i, j) block
    pairs each, against the oracle's ring partial of that step."""
    import torch
    import oracle
    import workloads
    from helpers import check_attention, np32
    from test_gpu_attention import _positions
    B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 1700 + S, "bf16")
    pos = _positions(pos_kind, B, S, 90 + S)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    rng = np.random.default_rng(S)
    qn, kn, vn = np32(q), np32(k), np32(v)
    for _ in range(2):
        i, j = int(rng.integers(P)), int(rng.integers(P))
        ti, tj = oracle.block_tokens(S, P, i, order), oracle.block_tokens(S, P, j, order)
        blk = lambda t, tok: t[:, torch.from_numpy(tok).cuda()].contiguous()
        out, lse = sp.ring_block_step(blk(q, ti), blk(k, tj), blk(v, tj), P, i, j, order, tpos)
        torch.cuda.synchronize()
        ro, rl = oracle.ring_partial(qn, kn, vn, P, (i - j) % P, order, pos)
        check_attention(np32(out), lse.cpu().numpy(), ro[:, ti], rl[:, :, ti], "bf16",
                        f"{_id(case)} i={i} j={j}")


@pytest.mark.parametrize("case", _cases(2030, "bf16", 10, 700), ids=_id)
def test_random_ring_block_pairs_backward(sp, case):
    """Seeded shapes through sp_ring_block_step_bwd for two random (i, j)
    block pairs each, accumulated twice into the same accumulators (the
    second call adds the first call's parts again, to float32 rounding: dq's
    per-key-tile pieces and dk/dv's per-query-head pieces are summed in no
    fixed order), against the oracle's ring step backward on our forward's
    out and lse."""
    import torch
    import oracle
    import workloads
    from helpers import check_grad, np32
    from test_gpu_attention import _positions
    B, S, Hq, Hkv, d, P, order, pos_kind = case
    q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 1800 + S, "bf16")
    g = torch.Generator(device="cuda").manual_seed(1801 + S)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    pos = _positions(pos_kind, B, S, 95 + S)
    tpos = None if pos is None else torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    rng = np.random.default_rng(S + 1)
    for _ in range(2):
        i, j = int(rng.integers(P)), int(rng.integers(P))
        ti, tj = oracle.block_tokens(S, P, i, order), oracle.block_tokens(S, P, j, order)
        blk = lambda t, tok: t[:, torch.from_numpy(tok).cuda()].contiguous()
        lse_i = lse[:, :, torch.from_numpy(ti).cuda()].contiguous()
        args = (blk(q, ti), blk(k, tj), blk(v, tj), blk(out, ti), blk(dout, ti), lse_i)
        acc = sp.ring_block_step_backward(*args, P, i, j, order, tpos)
        once = [a.clone() for a in acc]
        sp.ring_block_step_backward(*args, P, i, j, order, tpos, dq_acc=acc[0], dk_acc=acc[1],
                                    dv_acc=acc[2])
        torch.cuda.synchronize()
        ref = oracle.ring_partial_backward(*(np32(a) for a in args[:5]), lse_i.cpu().numpy(), S,
                                           P, i, j, order, pos)
        for name, got, first, r in zip(("dq", "dk", "dv"), acc, once, ref):
            tol = 1e-5 * float(first.abs().max()) + 1e-30
            assert float((got - 2 * first).abs().max()) <= tol, f"{_id(case)} {name} not additive"
            check_grad(first.cpu().numpy(), r, "bf16", f"{_id(case)} i={i} j={j} {name}")
