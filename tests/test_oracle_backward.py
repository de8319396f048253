"""Pins for oracle.attention_backward against things other than itself:
torch autograd in float64 on an explicitly written masked softmax attention,
central finite differences, closed forms and the GQA sum rule."""

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _packed(lengths):
    return np.concatenate([np.arange(L) for L in lengths])[None, :]


def _torch_grads(q, k, v, dout, mask, scale):
    """Autograd through softmax(scale q k^T masked) v, per head, GQA by
    repeat_interleave (so the key/value gradients sum over the group)."""
    g = q.shape[2] // k.shape[2]
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    kk = torch.repeat_interleave(tk, g, dim=2)
    vv = torch.repeat_interleave(tv, g, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", tq, kk) * scale
    if mask is not None:
        s = s.masked_fill(~torch.from_numpy(mask)[None, None], float("-inf"))
    p = torch.softmax(s, dim=-1)
    o = torch.einsum("bhij,bjhc->bihc", p, vv)
    o.backward(torch.tensor(dout, dtype=torch.float64))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("case", ["noncausal", "causal", "packed"])
def test_backward_matches_autograd(case):
    B, S, Hq, Hkv, d = 1, 29, 4, 2, 8
    q, k, v, do = (_rand((B, S, h, d), s) for s, h in ((1, Hq), (2, Hkv), (3, Hkv), (4, Hq)))
    if case == "noncausal":
        pos, mask = None, None
    elif case == "causal":
        pos = np.arange(S)[None, :]
        mask = np.tril(np.ones((S, S), dtype=bool))
    else:
        lengths = [7, 1, 12, 9]
        pos = _packed(lengths)
        mask = oracle.allowed_mask(pos, 1, S)[0]
        # the mask itself is pinned in test_oracle.py; rebuild it here from lengths
        ref = np.zeros((S, S), dtype=bool)
        o = 0
        for L in lengths:
            for i in range(L):
                ref[o + i, o:o + i + 1] = True
            o += L
        assert np.array_equal(mask, ref)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos)
    tq, tk, tv = _torch_grads(q, k, v, do, mask, 1 / np.sqrt(d))
    for a, b_ in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.abs(a - b_).max() < 1e-12


def test_backward_matches_finite_differences():
    B, S, H, d = 1, 9, 1, 4
    q, k, v, do = (_rand((B, S, H, d), s) for s in (5, 6, 7, 8))
    pos = _packed([4, 5])
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos)
    loss = lambda q_, k_, v_: float((oracle.full_attention(q_, k_, v_, pos)[0] * do).sum())
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0, 0), (0, 3, 0, 2), (0, 5, 0, 1), (0, 8, 0, 3)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7, (name, idx)


def test_backward_closed_forms():
    B, S, Hq, Hkv, d = 1, 17, 2, 1, 8
    q, k, do = _rand((B, S, Hq, d), 9), _rand((B, S, Hkv, d), 10), _rand((B, S, Hq, d), 11)
    pos = _packed([6, 11])
    # constant values: out does not depend on q or k, so their gradients vanish,
    # and every query row's dout is spread over its keys with weights summing to 1
    v = np.ones((B, S, Hkv, d)) * 3.0
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv.sum(axis=1) - do.sum(axis=(1, 2))[:, None, :]).max() < 1e-12
    # zero upstream gradient: zero gradients
    z = oracle.attention_backward(q, k, v, np.zeros_like(do), pos)
    assert all(np.abs(t).max() == 0 for t in z)
    # a document's first token attends only itself: its dv row collects only
    # the dout of the rows that see it
    dq, dk, dv = oracle.attention_backward(q, k, _rand((B, S, Hkv, d), 12), do, np.arange(S)[None] * 0)
    # position 0 everywhere: every token is its own document
    assert np.abs(dv[0, :, 0] - do[0].sum(axis=1)).max() < 1e-12
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_backward_gqa_is_sum_over_repeated_heads():
    B, S, d = 1, 13, 4
    q, k, v, do = _rand((B, S, 6, d), 13), _rand((B, S, 2, d), 14), _rand((B, S, 2, d), 15), \
        _rand((B, S, 6, d), 16)
    pos = np.arange(S)[None, :]
    dq, dk, dv = oracle.attention_backward(q, k, v, do, pos)
    dq2, dk2, dv2 = oracle.attention_backward(q, np.repeat(k, 3, axis=2), np.repeat(v, 3, axis=2),
                                              do, pos)
    assert np.abs(dq - dq2).max() < 1e-12
    assert np.abs(dk - dk2.reshape(B, S, 2, 3, d).sum(axis=3)).max() < 1e-12
    assert np.abs(dv - dv2.reshape(B, S, 2, 3, d).sum(axis=3)).max() < 1e-12


def test_backward_planted_mistakes_are_caught():
    """Plausible slips in the backward -- dropping the D term of dS, or a
    transposed dS in dK -- disagree with autograd while the oracle agrees."""
    q, k, v, do = (_rand((1, 11, 1, 4), s) for s in (20, 21, 22, 23))
    scale = 0.5
    tq, tk, _ = _torch_grads(q, k, v, do, None, scale)
    dq, dk, _ = oracle.attention_backward(q, k, v, do, None, scale)
    assert np.abs(dq - tq).max() < 1e-12 and np.abs(dk - tk).max() < 1e-12
    qh, kh, vh, doh = q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0]
    s_ = scale * qh @ kh.T
    p_ = np.exp(s_ - s_.max(axis=1, keepdims=True))
    p_ /= p_.sum(axis=1, keepdims=True)
    dp = doh @ vh.T
    no_d = p_ * dp                                      # D term dropped
    assert np.abs(scale * no_d @ kh - tq[0, :, 0]).max() > 1e-3
    D = (doh * (p_ @ vh)).sum(axis=1)
    ds = p_ * (dp - D[:, None])
    assert np.abs(scale * ds @ qh - tk[0, :, 0]).max() > 1e-3   # dS instead of dS^T


@pytest.mark.parametrize("case", ["noncausal", "causal", "packed"])
def test_sampled_rows_and_keys_match_autograd(case):
    """The sampled-row (dq) and sampled-key (dk, dv) forms against float64
    autograd on the whole problem, GQA group of 3."""
    B, S, Hq, Hkv, d = 2, 37, 6, 2, 8
    q, k, v, do = (_rand((B, S, h, d), s) for s, h in ((11, Hq), (12, Hkv), (13, Hkv), (14, Hq)))
    if case == "noncausal":
        pos, mask = None, None
    elif case == "causal":
        pos = np.tile(np.arange(S)[None, :], (B, 1))
        mask = np.tril(np.ones((S, S), dtype=bool))
    else:
        pos = np.tile(_packed([10, 1, 15, 11]), (B, 1))
        mask = oracle.allowed_mask(pos, 1, S)[0]
    scale = 0.3
    tq, tk, tv = _torch_grads(q, k, v, do, mask, scale)
    rows = np.array([0, 5, 10, 11, 20, 36])
    keys = np.array([0, 9, 10, 11, 25, 36])
    dq = oracle.attention_backward_rows(q, k, v, do, rows, pos, scale, max_chunk_elems=64)
    assert np.abs(dq - tq[:, rows]).max() < 1e-12
    dk, dv = oracle.attention_backward_keys(q, k, v, do, keys, pos, scale, max_chunk_elems=64)
    assert np.abs(dk - tk[:, keys]).max() < 1e-12
    assert np.abs(dv - tv[:, keys]).max() < 1e-12
    dk1, dv1 = oracle.attention_backward_keys(q, k, v, do, keys, pos, scale, kv_heads=[1])
    assert np.abs(dk1[:, :, 1] - tk[:, keys, 1]).max() < 1e-12
    assert not dk1[:, :, 0].any() and not dv1[:, :, 0].any()


def _blocks(x, S, P, p, order, axis=1):
    return np.take(x, oracle.block_tokens(S, P, p, order), axis=axis)


@pytest.mark.parametrize("case,order,P", [("noncausal", "contiguous", 3), ("causal", "striped", 4),
                                          ("packed", "contiguous", 4), ("packed", "striped", 3)])
def test_ring_partial_backward_sums_to_autograd(case, order, P):
    """The per-device ring-step gradient parts, scattered back to token order
    and summed over every (query block i, key/value block j) pair, equal
    float64 autograd on the whole problem (GQA group of 3); using each
    block pair's own log-sum-exp instead of the whole row's -- a plausible
    slip -- does not."""
    B, S, Hq, Hkv, d = 2, 36, 6, 2, 8
    q, k, v, do = (_rand((B, S, h, d), s) for s, h in ((31, Hq), (32, Hkv), (33, Hkv), (34, Hq)))
    if case == "noncausal":
        pos, mask = None, None
    elif case == "causal":
        pos = np.tile(np.arange(S)[None, :], (B, 1))
        mask = np.tril(np.ones((S, S), dtype=bool))
    else:
        pos = np.tile(_packed([10, 1, 14, 11]), (B, 1))
        mask = oracle.allowed_mask(pos, 1, S)[0]
    scale = 0.3
    tq, tk, tv = _torch_grads(q, k, v, do, mask, scale)
    out, lse = oracle.full_attention(q, k, v, pos, scale)
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for i in range(P):
        ti = oracle.block_tokens(S, P, i, order)
        for j in range(P):
            tj = oracle.block_tokens(S, P, j, order)
            pq, pk, pv = oracle.ring_partial_backward(
                _blocks(q, S, P, i, order), _blocks(k, S, P, j, order), _blocks(v, S, P, j, order),
                _blocks(out, S, P, i, order), _blocks(do, S, P, i, order),
                _blocks(lse, S, P, i, order, axis=2), S, P, i, j, order, pos, scale)
            dq[:, ti] += pq
            dk[:, tj] += pk
            dv[:, tj] += pv
    assert np.abs(dq - tq).max() < 1e-10
    assert np.abs(dk - tk).max() < 1e-10
    assert np.abs(dv - tv).max() < 1e-10
    # planted slip: the pair's own lse (softmax over block j only)
    i, j = P - 1, 0
    _, lse_pair = oracle.ring_partial(q, k, v, P, (i - j) % P, order, pos, scale)
    ti = oracle.block_tokens(S, P, i, order)
    pq_wrong, _, _ = oracle.ring_partial_backward(
        _blocks(q, S, P, i, order), _blocks(k, S, P, j, order), _blocks(v, S, P, j, order),
        _blocks(out, S, P, i, order), _blocks(do, S, P, i, order),
        _blocks(lse_pair, S, P, i, order, axis=2), S, P, i, j, order, pos, scale)
    pq_right, _, _ = oracle.ring_partial_backward(
        _blocks(q, S, P, i, order), _blocks(k, S, P, j, order), _blocks(v, S, P, j, order),
        _blocks(out, S, P, i, order), _blocks(do, S, P, i, order),
        _blocks(lse, S, P, i, order, axis=2), S, P, i, j, order, pos, scale)
    if np.abs(pq_right).max() > 0:
        assert np.abs(pq_wrong - pq_right).max() > 1e-3
