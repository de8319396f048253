"""Pins for the CPU oracle, against things other than the oracle itself.

Each test ties an oracle function to a fact fixed by the pages or by the
mathematics: the Ring Attention page's worked example, a library routine
(torch's scaled_dot_product_attention in float64), closed forms, brute force
on tiny inputs, and invariants (independence of P and block order, merge
identities, permutation round trips).  The last group plants plausible
mistakes in copies of oracle functions and checks that the pins catch them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _packed_positions(lengths):
    return np.concatenate([np.arange(L) for L in lengths])[None, :]


def _mask_from_lengths(lengths):
    """Block-diagonal lower-triangular mask, built from document lengths only."""
    S = sum(lengths)
    m = np.zeros((S, S), dtype=bool)
    o = 0
    for L in lengths:
        for i in range(L):
            m[o + i, o:o + i + 1] = True
        o += L
    return m


# --------------------------------------------------------------------------
# The Ring Attention page's worked example (4 devices x block 8, d = 16).
# --------------------------------------------------------------------------

def _load_ring_tiny():
    with open(os.path.join(GOLDEN, "ring_tiny_seed0.json"), encoding="utf-8") as f:
        doc = json.load(f)
    q, k, v = (np.array(doc[n], dtype=np.float32) for n in ("q", "k", "v"))
    return doc, q, k, v


def test_fixture_is_the_pages_draw():
    """The frozen inputs are torch.manual_seed(0); torch.randn(3, 32, 16)."""
    doc, q, k, v = _load_ring_tiny()
    torch.manual_seed(0)
    qkv = torch.randn(3, 32, 16)
    # torch's CPU generator is stable across versions in practice; if it ever
    # changes, the frozen fixture stays the reference.
    if not np.array_equal(qkv[0].numpy(), q):
        pytest.skip("this torch build draws different numbers for seed 0")
    assert np.array_equal(qkv[1].numpy(), k) and np.array_equal(qkv[2].numpy(), v)
    facts = doc["page_facts"]
    assert (facts["n_devices"] * facts["block"], facts["dim"]) == q.shape == (32, 16)


def test_ring_page_example_matches_full_attention():
    """The page prints 'Matches full attention: True' (allclose, atol 1e-5)."""
    doc, q, k, v = _load_ring_tiny()
    facts = doc["page_facts"]
    blockwise = oracle.ring_unstabilised_f32(q, k, v, facts["n_devices"])
    as4 = lambda a: a.astype(np.float64)[None, :, None, :]
    full, _ = oracle.full_attention(as4(q), as4(k), as4(v))
    assert np.allclose(blockwise, full[0, :, 0, :], atol=facts["allclose_atol"]) == facts[
        "matches_full_attention"]
    # stored expectation (written by the fixture script from the oracle)
    want = np.array([[float(x) for x in r] for r in doc["expected_out_oracle_f64"]])
    assert np.abs(full[0, :, 0, :] - want).max() < 1e-12
    # each device's score block is block x block; the full matrix n x n
    blk = facts["block"]
    assert (q[:blk] @ k[:blk].T).shape == tuple(facts["score_block"])
    assert (q @ k.T).shape == tuple(facts["full_matrix"])


@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_ring_page_example_every_block_count(order):
    """Exactness is independent of the number of devices and of the order."""
    _, q, k, v = _load_ring_tiny()
    as4 = lambda a: a.astype(np.float64)[None, :, None, :]
    full, lse = oracle.full_attention(as4(q), as4(k), as4(v))
    for P in (1, 2, 4, 8, 16, 32):
        out, l2 = oracle.blockwise_ring_attention(as4(q), as4(k), as4(v), P, order)
        assert np.abs(out - full).max() < 1e-12
        assert np.abs(l2 - lse).max() < 1e-12


# --------------------------------------------------------------------------
# Library routine: torch SDPA in float64 on the CPU.
# --------------------------------------------------------------------------

def _sdpa(q, k, v, mask):
    B, S, Hq, d = q.shape
    g = Hq // k.shape[2]
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(np.repeat(k, g, axis=2)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(np.repeat(v, g, axis=2)).permute(0, 2, 1, 3)
    am = None if mask is None else torch.from_numpy(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am)
    return o.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("case", ["noncausal", "causal", "packed"])
def test_full_attention_matches_sdpa(case):
    B, S, Hq, Hkv, d = 2, 37, 6, 2, 8
    q, k, v = (_rand((B, S, h, d), s) for s, h in ((1, Hq), (2, Hkv), (3, Hkv)))
    if case == "noncausal":
        pos, mask = None, None
    elif case == "causal":
        pos = np.tile(np.arange(S), (B, 1))
        mask = np.tril(np.ones((S, S), dtype=bool))
    else:
        lengths = [9, 1, 14, 13]
        pos = np.tile(_packed_positions(lengths), (B, 1))
        mask = _mask_from_lengths(lengths)
    out, _ = oracle.full_attention(q, k, v, pos)
    ref = _sdpa(q, k, v, mask)
    assert np.abs(out - ref).max() < 1e-12


def test_scale_argument_matches_sdpa():
    q, k, v = (_rand((1, 16, 2, 4), s) for s in (4, 5, 6))
    out, _ = oracle.full_attention(q, k, v, None, scale=0.3)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.3)
    assert np.abs(out - ref.permute(0, 2, 1, 3).numpy()).max() < 1e-12


# --------------------------------------------------------------------------
# Closed forms.
# --------------------------------------------------------------------------

def test_zero_query_gives_mean_and_log_count():
    """q = 0: every allowed score is 0, so out = mean of the allowed v and
    lse = ln(#allowed) = ln(position within document + 1)."""
    lengths = [5, 1, 7, 3, 16]
    S = sum(lengths)
    pos = _packed_positions(lengths)
    q = np.zeros((1, S, 4, 16))
    k = _rand((1, S, 2, 16), 7)
    v = _rand((1, S, 2, 16), 8)
    out, lse = oracle.full_attention(q, k, v, pos)
    expect_lse = np.log(pos[0] + 1.0)
    for h in range(4):
        assert np.abs(lse[0, h] - expect_lse).max() < 1e-12
    o = 0
    for L in lengths:
        for i in range(L):
            mean = v[0, o:o + i + 1].mean(axis=0)  # [Hkv][d]
            for h in range(4):
                assert np.abs(out[0, o + i, h] - mean[h // 2]).max() < 1e-12
        o += L


def test_zero_query_noncausal_is_global_mean():
    S = 20
    q = np.zeros((1, S, 1, 8))
    k, v = _rand((1, S, 1, 8), 9), _rand((1, S, 1, 8), 10)
    out, lse = oracle.full_attention(q, k, v)
    assert np.abs(out[0, :, 0] - v[0, :, 0].mean(axis=0)).max() < 1e-12
    assert np.abs(lse - math.log(S)).max() < 1e-12


def test_constant_values_give_constant_output():
    """v = 1: softmax rows sum to one, so out = 1 everywhere."""
    lengths = [3, 11, 2]
    pos = _packed_positions(lengths)
    S = sum(lengths)
    q, k = _rand((1, S, 2, 8), 11), _rand((1, S, 1, 8), 12)
    out, _ = oracle.full_attention(q, k, np.ones((1, S, 1, 8)), pos)
    assert np.abs(out - 1.0).max() < 1e-12


def test_document_first_token_sees_only_itself():
    lengths = [4, 6, 5]
    pos = _packed_positions(lengths)
    S = sum(lengths)
    q, k, v = _rand((1, S, 1, 8), 13), _rand((1, S, 1, 8), 14), _rand((1, S, 1, 8), 15)
    out, lse = oracle.full_attention(q, k, v, pos)
    for t in (0, 4, 10):
        assert np.abs(out[0, t, 0] - v[0, t, 0]).max() < 1e-12
        assert abs(lse[0, 0, t] - q[0, t, 0] @ k[0, t, 0] / math.sqrt(8)) < 1e-12


# --------------------------------------------------------------------------
# Brute force on tiny inputs (pure Python, math.exp).
# --------------------------------------------------------------------------

def _brute(q, k, v, pos):
    B, S, Hq, d = q.shape
    g = Hq // k.shape[2]
    out = np.zeros(q.shape[:3] + (v.shape[3],))
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for i in range(S):
            # document of i: walk back while positions step by one
            start = i
            if pos is not None:
                while start > 0 and pos[b][start] == pos[b][start - 1] + 1:
                    start -= 1
            keys = range(S) if pos is None else range(start, i + 1)
            for h in range(Hq):
                sc = {j: sum(q[b, i, h, c] * k[b, j, h // g, c] for c in range(d)) / math.sqrt(d)
                      for j in keys}
                mx = max(sc.values())
                w = {j: math.exp(s - mx) for j, s in sc.items()}
                tot = sum(w.values())
                for c in range(v.shape[3]):
                    out[b, i, h, c] = sum(w[j] * v[b, j, h // g, c] for j in w) / tot
                lse[b, h, i] = mx + math.log(tot)
    return out, lse


@pytest.mark.parametrize("pos", [None, [[0, 1, 2, 0, 1, 2, 3, 0, 0, 1, 2]],
                                 [[5, 6, 7, 8, 2, 3, 4, 4, 5, 9, 10]]])
def test_brute_force_tiny(pos):
    S = 11
    q, k, v = _rand((1, S, 4, 3), 16), _rand((1, S, 2, 3), 17), _rand((1, S, 2, 5), 18)
    p = None if pos is None else np.array(pos)
    out, lse = oracle.full_attention(q, k, v, p)
    bo, bl = _brute(q, k, v, p)
    assert np.abs(out - bo).max() < 1e-12
    assert np.abs(lse - bl).max() < 1e-12
    rows = np.array([10, 0, 7, 3])
    ro, rl = oracle.attention_rows(q, k, v, rows, p)
    assert np.abs(ro - bo[:, rows]).max() < 1e-12
    assert np.abs(rl - bl[:, :, rows]).max() < 1e-12


# --------------------------------------------------------------------------
# position_ids reading.
# --------------------------------------------------------------------------

def test_segments_hand_example():
    pos = np.array([[0, 1, 2, 0, 1, 0, 1, 2, 3]])
    assert oracle.segment_ids(pos).tolist() == [[1, 1, 1, 2, 2, 3, 3, 3, 3]]
    assert oracle.doc_starts(pos).tolist() == [[0, 0, 0, 3, 3, 5, 5, 5, 5]]
    # a document may start at any position value; a repeat also starts one
    pos = np.array([[7, 8, 9, 9, 10, 3]])
    assert oracle.segment_ids(pos).tolist() == [[1, 1, 1, 2, 2, 3]]
    assert oracle.doc_starts(pos).tolist() == [[0, 0, 0, 3, 3, 5]]


def test_allowed_mask_matches_lengths():
    lengths = [3, 1, 6, 2]
    m = oracle.allowed_mask(_packed_positions(lengths), 1, sum(lengths))
    assert np.array_equal(m[0], _mask_from_lengths(lengths))
    assert oracle.allowed_mask(None, 2, 5).all()


def test_plain_causal_is_lower_triangle():
    S = 9
    m = oracle.allowed_mask(np.arange(S)[None, :], 1, S)
    assert np.array_equal(m[0], np.tril(np.ones((S, S), dtype=bool)))


# --------------------------------------------------------------------------
# Invariants of the blockwise method.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("order", ["contiguous", "striped"])
@pytest.mark.parametrize("causal", [False, True])
def test_blockwise_independent_of_P_and_order(order, causal):
    S = 48
    lengths = [7, 1, 18, 22]
    pos = _packed_positions(lengths) if causal else None
    q, k, v = _rand((1, S, 4, 8), 20), _rand((1, S, 2, 8), 21), _rand((1, S, 2, 8), 22)
    full, lse = oracle.full_attention(q, k, v, pos)
    for P in (1, 2, 3, 4, 6, 8, 12, 16, 24, 48):
        out, l2 = oracle.blockwise_ring_attention(q, k, v, P, order, pos)
        assert np.abs(out - full).max() < 1e-12, P
        assert np.abs(l2 - lse).max() < 1e-12, P


@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_merge_of_ring_steps_is_full_attention(order):
    S, P = 40, 4
    pos = _packed_positions([13, 2, 25])
    q, k, v = _rand((2, S, 2, 8), 23), _rand((2, S, 1, 8), 24), _rand((2, S, 1, 8), 25)
    pos = np.tile(pos, (2, 1))
    parts = [oracle.ring_partial(q, k, v, P, s, order, pos) for s in range(P)]
    out, lse = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    full, flse = oracle.full_attention(q, k, v, pos)
    assert np.abs(out - full).max() < 1e-12
    assert np.abs(lse - flse).max() < 1e-12
    # in contiguous causal order, step s > i leaves block i with nothing
    if order == "contiguous":
        o1, l1 = parts[1]
        assert np.isneginf(l1[:, :, :S // P]).all() and (o1[:, :S // P] == 0).all()


def test_merge_identities():
    rng = np.random.default_rng(30)
    outs = rng.standard_normal((3, 1, 5, 2, 4))
    lses = rng.standard_normal((3, 1, 2, 5))
    o_all, l_all = oracle.merge_partials(outs, lses)
    # associativity: merge(merge(0,1), 2) == merge(0,1,2)
    o01, l01 = oracle.merge_partials(outs[:2], lses[:2])
    o_b, l_b = oracle.merge_partials([o01, outs[2]], [l01, lses[2]])
    assert np.abs(o_b - o_all).max() < 1e-12 and np.abs(l_b - l_all).max() < 1e-12
    # an empty partial (0, -inf) is the identity
    o_e, l_e = oracle.merge_partials([outs[0], np.zeros_like(outs[0])],
                                     [lses[0], np.full_like(lses[0], -np.inf)])
    assert np.abs(o_e - outs[0]).max() < 1e-12 and np.abs(l_e - lses[0]).max() < 1e-12
    # all empty -> 0 / -inf
    o_z, l_z = oracle.merge_partials(np.zeros((2, 1, 3, 1, 2)), np.full((2, 1, 1, 3), -np.inf))
    assert (o_z == 0).all() and np.isneginf(l_z).all()
    # equal lse: plain average, lse + ln 2
    o_h, l_h = oracle.merge_partials([outs[0], outs[1]], [lses[0], lses[0]])
    assert np.abs(o_h - 0.5 * (outs[0] + outs[1])).max() < 1e-12
    assert np.abs(l_h - (lses[0] + math.log(2))).max() < 1e-12


def test_gqa_is_repeated_heads():
    S = 16
    q, k, v = _rand((1, S, 6, 8), 31), _rand((1, S, 2, 8), 32), _rand((1, S, 2, 8), 33)
    pos = np.arange(S)[None, :]
    o1, l1 = oracle.full_attention(q, k, v, pos)
    o2, l2 = oracle.full_attention(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2), pos)
    assert np.abs(o1 - o2).max() == 0 and np.abs(l1 - l2).max() == 0


# --------------------------------------------------------------------------
# The permutation.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_permutation_roundtrip_and_bijection(P):
    B, S, H, d = 2, 8, 8, 3
    x = np.arange(B * S * H * d, dtype=np.int64).reshape(B, S, H, d)
    y = oracle.seq_to_head(x, P)
    assert y.shape == (P, B, S, H // P, d)
    assert np.array_equal(np.sort(y.ravel()), x.ravel())  # every element exactly once
    assert np.array_equal(oracle.head_to_seq(y), x)
    # rank r holds every position of its own heads and nothing else
    for r in range(P):
        heads = {int(val) // d % H for val in y[r].ravel()}
        assert heads == set(range(r * H // P, (r + 1) * H // P))
        toks = {int(val) // (H * d) % S for val in y[r].ravel()}
        assert toks == set(range(S))


def test_permutation_elementwise_tiny():
    B, S, H, d, P = 1, 6, 6, 2, 3
    x = _rand((B, S, H, d), 40)
    y = oracle.seq_to_head(x, P)
    G = H // P
    for r in range(P):
        for b in range(B):
            for t in range(S):
                for hl in range(G):
                    for c in range(d):
                        assert y[r, b, t, hl, c] == x[b, t, r * G + hl, c]


def test_block_tokens_partition():
    """Both block orders cut the tokens 0..S-1 into P blocks of S/P tokens:
    contiguous block p is [p*S/P, (p+1)*S/P) (GPU i holds [i*n/P,
    (i+1)*n/P) on the Ulysses pages); striped block p is {t : t mod P = p}
    (tokens spread uniformly, stripe width 1)."""
    S, P = 24, 4
    for order in ("contiguous", "striped"):
        blocks = [oracle.block_tokens(S, P, p, order) for p in range(P)]
        assert sorted(np.concatenate(blocks).tolist()) == list(range(S))
        assert all(len(b) == S // P for b in blocks)
        assert all(np.all(np.diff(b) > 0) for b in blocks)  # natural order inside a block
    assert oracle.block_tokens(S, P, 1, "contiguous").tolist() == list(range(6, 12))
    assert oracle.block_tokens(S, P, 1, "striped").tolist() == [1, 5, 9, 13, 17, 21]
    with pytest.raises(ValueError):
        oracle.block_tokens(10, 4, 0, "striped")


def test_permutation_rejects_indivisible():
    with pytest.raises(ValueError):
        oracle.seq_to_head(np.zeros((1, 4, 6, 2)), 4)
    with pytest.raises(ValueError):
        oracle.seq_to_head(np.zeros((1, 6, 8, 2)), 4)


# --------------------------------------------------------------------------
# Planted mistakes: copies of oracle code with one plausible error each must
# fail the pins above.
# --------------------------------------------------------------------------

def _sdpa_pin(fn):
    q, k, v = (_rand((1, 21, 4, 8), s) for s in (50, 51, 52))
    k, v = k[:, :, :2], v[:, :, :2]
    lengths = [6, 15]
    out, _ = fn(q, k, v, np.tile(_packed_positions(lengths), (1, 1)))
    return np.abs(out - _sdpa(q, k, v, _mask_from_lengths(lengths))).max() < 1e-12


def test_planted_mistakes_are_caught(monkeypatch):
    assert _sdpa_pin(oracle.full_attention)

    def wrong_scale(qrows, keys, vals, allowed, scale):
        return oa.__dict__["_orig_attend"](qrows, keys, vals, allowed, scale * scale)

    def transposed_mask(qrows, keys, vals, allowed, scale):
        if allowed.shape[0] == allowed.shape[1]:
            allowed = allowed.T
        return oa.__dict__["_orig_attend"](qrows, keys, vals, allowed, scale)

    def dropped_max(qrows, keys, vals, allowed, scale):  # keeps the right answer
        return oa.__dict__["_orig_attend"](qrows, keys, vals, allowed, scale)

    monkeypatch.setitem(oa.__dict__, "_orig_attend", oa._softmax_attend)
    for bad, caught in ((wrong_scale, True), (transposed_mask, True), (dropped_max, False)):
        monkeypatch.setattr(oa, "_softmax_attend", bad)
        assert _sdpa_pin(oa.full_attention) != caught
    monkeypatch.setattr(oa, "_softmax_attend", oa.__dict__["_orig_attend"])

    # wrong GQA mapping (h % Hkv instead of h // g) breaks the repeat pin
    q, k, v = _rand((1, 12, 4, 4), 53), _rand((1, 12, 2, 4), 54), _rand((1, 12, 2, 4), 55)
    good, _ = oracle.full_attention(q, k, v)
    kk = k[:, :, [0, 1, 0, 1]]
    vv = v[:, :, [0, 1, 0, 1]]
    wrong, _ = oracle.full_attention(q, kk, vv)
    assert np.abs(good - wrong).max() > 1e-3

    # a segment reading that only compares positions (pos_j <= pos_i) leaks
    # across packed documents and fails the closed form
    pos = _packed_positions([4, 4])
    leaky = (pos[0][None, :] <= pos[0][:, None])
    assert not np.array_equal(leaky, oracle.allowed_mask(pos, 1, 8)[0])
