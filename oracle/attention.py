"""Reference attention for the blockwise / ring path (float64, NumPy).

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA library never
imports this module.

Layouts (the same as the library's, but nothing is shared with it):
    q               [B][S][Hq][d]
    k, v            [B][S][Hkv][d]
    position_ids    [B][S] integers, or None for non-causal attention
    out             [B][S][Hq][d]
    lse             [B][Hq][S]   natural log-sum-exp of the scaled scores
"""

import numpy as np

NEG_INF = -np.inf


def segment_ids(position_ids):
    """Document index of every token, from position_ids alone.

    "Ulysses SPで100万トークン学習" (aitoolresearcher review), section 3: the
    causal mask is carried by position_ids (O(n)) instead of a 4D mask.  The
    page does not spell out packed documents; the reading taken here is that a
    new document starts at token 0 and wherever position_ids does not continue
    by +1.  seg(t) = number of such starts at or before t (so the first
    document is 1).
    """
    pos = np.asarray(position_ids, dtype=np.int64)
    if pos.ndim == 1:
        pos = pos[None, :]
    starts = np.ones(pos.shape, dtype=np.int64)
    starts[:, 1:] = (pos[:, 1:] != pos[:, :-1] + 1).astype(np.int64)
    return np.cumsum(starts, axis=1)


def doc_starts(position_ids):
    """First token index of every token's document: [B][S] int64.

    Same reading as segment_ids; the token where the document numbered
    seg(t) begins.
    """
    seg = segment_ids(position_ids)
    B, S = seg.shape
    first = np.zeros((B, S), dtype=np.int64)
    for b in range(B):
        start_of = {}
        for t in range(S):
            start_of.setdefault(int(seg[b, t]), t)
            first[b, t] = start_of[int(seg[b, t])]
    return first


def allowed_mask(position_ids, B, S):
    """allowed[b, i, j]: may query token i attend key token j?

    None -> every pair (non-causal).  Otherwise same document and j <= i.
    Materialises B*S*S booleans: small sizes only.
    """
    if position_ids is None:
        return np.ones((B, S, S), dtype=bool)
    seg = segment_ids(position_ids)
    idx = np.arange(S)
    causal = idx[None, :] <= idx[:, None]
    same = seg[:, :, None] == seg[:, None, :]
    return same & causal[None, :, :]


def _softmax_attend(qrows, keys, vals, allowed, scale):
    """Exact attention of some query rows over a key set.

    qrows [R][d], keys [K][d], vals [K][dv], allowed [R][K] bool.  Follows the
    textbook definition: s = scale * q.k; m = max over allowed keys;
    w = exp(s - m); out = sum w v / sum w; lse = m + ln(sum w).  A row with no
    allowed key gives out = 0 and lse = -inf.
    """
    s = scale * (qrows @ keys.T)
    s = np.where(allowed, s, NEG_INF)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], NEG_INF)
    any_allowed = np.isfinite(m)
    m_safe = np.where(any_allowed, m, 0.0)
    w = np.where(allowed, np.exp(s - m_safe[:, None]), 0.0)
    l = w.sum(axis=1)
    num = w @ vals
    out = np.zeros((qrows.shape[0], vals.shape[1]), dtype=np.float64)
    out[any_allowed] = num[any_allowed] / l[any_allowed, None]
    lse = np.full(qrows.shape[0], NEG_INF)
    lse[any_allowed] = m[any_allowed] + np.log(l[any_allowed])
    return out, lse


def _check_shapes(q, k, v):
    B, S, Hq, d = q.shape
    Bk, Sk, Hkv, dk = k.shape
    if (Bk, Sk, dk) != (B, S, d) or v.shape[:3] != k.shape[:3]:
        raise ValueError("q/k/v shapes disagree")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, S, Hq, Hkv, d


def attention_rows(q, k, v, rows=None, position_ids=None, scale=None, max_chunk_elems=1 << 25):
    """Exact softmax attention for the given query token indices.

    Returns out [B][R][Hq][dv] and lse [B][Hq][R] for R = len(rows) (all rows
    when rows is None).  GQA: query head h reads key/value head h // (Hq/Hkv).
    Rows are evaluated independently, a few at a time to bound memory; for a
    causal mask only keys up to the largest row of the group are formed (the
    others are masked anyway).
    """
    B, S, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    dv = v.shape[3]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    R = rows.shape[0]
    out = np.zeros((B, R, Hq, dv), dtype=np.float64)
    lse = np.full((B, Hq, R), NEG_INF)
    seg = None if position_ids is None else segment_ids(position_ids)
    for b in range(B):
        for kvh in range(Hkv):
            keys_all = np.asarray(k[b, :, kvh, :], dtype=np.float64)
            vals_all = np.asarray(v[b, :, kvh, :], dtype=np.float64)
            for h in range(kvh * g, (kvh + 1) * g):
                step = max(1, max_chunk_elems // max(S, 1))
                for c0 in range(0, R, step):
                    c1 = min(R, c0 + step)
                    sel = rows[c0:c1]
                    kmax = S if seg is None else int(sel.max()) + 1
                    if seg is None:
                        allowed = np.ones((sel.shape[0], kmax), dtype=bool)
                    else:
                        j = np.arange(kmax)
                        allowed = (seg[b, :kmax][None, :] == seg[b, sel][:, None]) & (
                            j[None, :] <= sel[:, None])
                    qrows = np.asarray(q[b, sel, h, :], dtype=np.float64)
                    o, l_ = _softmax_attend(qrows, keys_all[:kmax], vals_all[:kmax], allowed, scale)
                    out[b, c0:c1, h, :] = o
                    lse[b, h, c0:c1] = l_
    return out, lse


def full_attention(q, k, v, position_ids=None, scale=None):
    """softmax(scale * Q K^T + mask) V for every query row, with its lse.

    This is the result the Ring Attention page says the blockwise computation
    reaches exactly ("Ring Attention", section "Cómo funciona la atención en
    anillo": the four-device simulation matches full attention).
    """
    return attention_rows(q, k, v, None, position_ids, scale)


def block_tokens(S, P, p, order):
    """Token indices of sequence block p out of P.

    contiguous: tokens [p*S/P, (p+1)*S/P) -- the sequence sharding of the
    Ulysses pages (GPU i holds [i*n/P, (i+1)*n/P)).
    striped: tokens t with t mod P == p -- Striped Attention as described on
    the Ring Attention page (each device's tokens spread uniformly over the
    sequence; stripe width 1 is the reading taken).
    """
    if S % P:
        raise ValueError("S must be a multiple of P")
    if order == "contiguous":
        Lb = S // P
        return np.arange(p * Lb, (p + 1) * Lb)
    if order == "striped":
        return np.arange(p, S, P)
    raise ValueError(f"unknown block order {order!r}")


def _allowed_between(seg_b, ti, tj):
    if seg_b is None:
        return np.ones((ti.shape[0], tj.shape[0]), dtype=bool)
    return (seg_b[ti][:, None] == seg_b[tj][None, :]) & (tj[None, :] <= ti[:, None])


def blockwise_ring_attention(q, k, v, P, order="contiguous", position_ids=None, scale=None):
    """Ring attention simulated on one machine, P blocks, online softmax.

    "Ring Attention", section "Cómo funciona la atención en anillo": block i
    of the queries stays put; at step s it meets key/value block
    j = (i - s) mod P; a running sum of exponentiated scores (denominator)
    and of weighted values (numerator) is kept and divided at the end.  The
    same page notes that production kernels also subtract a running maximum,
    which is done here: when the maximum grows from m to m', the running sums
    are multiplied by exp(m - m').

    An independent restatement of full_attention, used to pin it.
    """
    B, S, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    dv = v.shape[3]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    seg = None if position_ids is None else segment_ids(position_ids)
    out = np.zeros((B, S, Hq, dv))
    lse = np.full((B, Hq, S), NEG_INF)
    blocks = [block_tokens(S, P, p, order) for p in range(P)]
    for b in range(B):
        seg_b = None if seg is None else seg[b]
        for h in range(Hq):
            kvh = h // g
            for i in range(P):
                ti = blocks[i]
                qi = np.asarray(q[b, ti, h, :], dtype=np.float64)
                m = np.full(ti.shape[0], NEG_INF)
                den = np.zeros(ti.shape[0])
                num = np.zeros((ti.shape[0], dv))
                for step in range(P):
                    j = (i - step) % P
                    tj = blocks[j]
                    kj = np.asarray(k[b, tj, kvh, :], dtype=np.float64)
                    vj = np.asarray(v[b, tj, kvh, :], dtype=np.float64)
                    ok = _allowed_between(seg_b, ti, tj)
                    s = np.where(ok, scale * (qi @ kj.T), NEG_INF)
                    m_new = np.maximum(m, s.max(axis=1))
                    live = np.isfinite(m_new)
                    base = np.where(live, m_new, 0.0)
                    # rows that had no allowed key so far carry zero sums
                    alpha = np.where(np.isfinite(m), np.exp(m - base), 0.0)
                    p = np.where(ok, np.exp(s - base[:, None]), 0.0)
                    den = alpha * den + p.sum(axis=1)
                    num = alpha[:, None] * num + p @ vj
                    m = m_new
                live = den > 0
                out[b, ti[live], h, :] = num[live] / den[live, None]
                lse[b, h, ti[live]] = m[live] + np.log(den[live])
    return out, lse


def ring_partial(q, k, v, P, step, order="contiguous", position_ids=None, scale=None):
    """What every simulated device holds after attending one ring step only.

    For each query block i, attention restricted to the key/value block
    j = (i - step) mod P ("Ring Attention", "Cómo funciona la atención en
    anillo").  Returned in natural token order: out [B][S][Hq][dv] and
    lse [B][Hq][S]; rows with no allowed key in that block give 0 / -inf.
    merge_partials over step = 0..P-1 recovers full_attention.
    """
    B, S, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    dv = v.shape[3]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    seg = None if position_ids is None else segment_ids(position_ids)
    out = np.zeros((B, S, Hq, dv))
    lse = np.full((B, Hq, S), NEG_INF)
    blocks = [block_tokens(S, P, p, order) for p in range(P)]
    for b in range(B):
        seg_b = None if seg is None else seg[b]
        for h in range(Hq):
            kvh = h // g
            for i in range(P):
                ti = blocks[i]
                tj = blocks[(i - step) % P]
                o, l_ = _softmax_attend(np.asarray(q[b, ti, h, :], dtype=np.float64),
                                        np.asarray(k[b, tj, kvh, :], dtype=np.float64),
                                        np.asarray(v[b, tj, kvh, :], dtype=np.float64),
                                        _allowed_between(seg_b, ti, tj), scale)
                out[b, ti, h, :] = o
                lse[b, h, ti] = l_
    return out, lse


def merge_partials(outs, lses):
    """Combine per-block partial results by their log-sum-exp weights.

    The cross-device combine of ring attention ("Ring Attention", "Cómo
    funciona la atención en anillo": partial results are combined by the
    cumulative softmax).  With lse = ln sum_j exp(lse_j):
        out = sum_j exp(lse_j - lse) * out_j.
    A partial with lse_j = -inf has weight 0; if all are -inf the result is
    out = 0, lse = -inf.

    outs [P][B][S][H][dv], lses [P][B][H][S] -> out [B][S][H][dv], lse [B][H][S].
    """
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = lses.max(axis=0)                               # [B][H][S]
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe[None]), 0.0)  # [P][B][H][S]
    total = w.sum(axis=0)
    lse = np.where(live, m_safe + np.log(np.where(live, total, 1.0)), NEG_INF)
    coef = np.where(live[None], w / np.where(live, total, 1.0)[None], 0.0)  # [P][B][H][S]
    coef = np.transpose(coef, (0, 1, 3, 2))[..., None]  # [P][B][S][H][1]
    out = (coef * outs).sum(axis=0)
    return out, lse


def ring_unstabilised_f32(q, k, v, n_blocks):
    """The Ring Attention page's four-device simulation, in float32.

    Single head, batch 1, q/k/v [n][d], contiguous blocks.  Device i keeps
    query block i; at step s it takes block j = (i - s) mod n, adds
    exp(q_i k_j^T / sqrt(d)) v_j to a numerator and the row sums of
    exp(q_i k_j^T / sqrt(d)) to a denominator -- without subtracting a
    maximum, as in the page's example -- and finally divides.
    """
    q = np.asarray(q, dtype=np.float32)
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    n, d = q.shape
    blk = n // n_blocks
    root_d = np.float32(np.sqrt(np.float32(d)))
    outs = []
    for i in range(n_blocks):
        qi = q[i * blk:(i + 1) * blk]
        num = np.zeros((blk, v.shape[1]), dtype=np.float32)
        den = np.zeros((blk, 1), dtype=np.float32)
        for step in range(n_blocks):
            j = (i - step) % n_blocks
            kj = k[j * blk:(j + 1) * blk]
            vj = v[j * blk:(j + 1) * blk]
            e = np.exp((qi @ kj.T) / root_d).astype(np.float32)
            num += e @ vj
            den += e.sum(axis=1, keepdims=True)
        outs.append(num / den)
    return np.concatenate(outs, axis=0)


def attention_backward(q, k, v, dout, position_ids=None, scale=None):
    """Gradients of out = softmax(scale * Q K^T + mask) V with respect to q,
    k, v for an upstream gradient dout (same layout as out).

    The pages' use case is training ("Ulysses SP: entrenar modelos con
    millones de tokens"; the ring keeps running sums per block, "Ring
    Attention", "Cómo funciona la atención en anillo") but they print no
    backward formulas; these are the derivatives of the definition:
        P  = softmax(S) over the allowed keys,   S = scale * Q K^T
        dV = P^T dO
        dP = dO V^T
        dS = P * (dP - D),   D_i = sum_c dO[i, c] * O[i, c]  (= sum_j P_ij dP_ij)
        dQ = scale * dS K,   dK = scale * dS^T Q
    GQA: the query heads of a group add into their shared key/value head.
    Rows with no allowed key contribute nothing.  Full score matrices per
    head: small sizes only.  Returns dq, dk, dv in float64.
    """
    B, S, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    allowed = allowed_mask(position_ids, B, S)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            qh = np.asarray(q[b, :, h, :], dtype=np.float64)
            kh = np.asarray(k[b, :, kvh, :], dtype=np.float64)
            vh = np.asarray(v[b, :, kvh, :], dtype=np.float64)
            doh = np.asarray(dout[b, :, h, :], dtype=np.float64)
            s = np.where(allowed[b], scale * (qh @ kh.T), NEG_INF)
            m = s.max(axis=1)
            live = np.isfinite(m)
            w = np.where(allowed[b], np.exp(s - np.where(live, m, 0.0)[:, None]), 0.0)
            l = w.sum(axis=1)
            p = np.zeros_like(w)
            p[live] = w[live] / l[live, None]
            o = p @ vh
            dv[b, :, kvh, :] += p.T @ doh
            dp = doh @ vh.T
            D = (doh * o).sum(axis=1)
            ds = p * (dp - D[:, None])
            dq[b, :, h, :] = scale * (ds @ kh)
            dk[b, :, kvh, :] += scale * (ds.T @ qh)
    return dq, dk, dv


def ring_partial_backward(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, S, P, i, j,
                          order="contiguous", position_ids=None, scale=None):
    """The gradient parts of one ring step on one device: the device holding
    query block i ("Ring Attention", "Cómo funciona la atención en anillo")
    after receiving key/value block j.  Block tensors in local row order
    (q_blk, out_blk, dout_blk [B][S/P][Hq][d]; k_blk, v_blk [B][S/P][Hkv][d];
    lse_blk [B][Hq][S/P], the forward's lse of block i's rows over the whole
    sequence); position_ids of the whole sequence.  The derivatives of the
    definition (as in attention_backward), restricted to the pair:
        P_ij  = exp(scale * Q_i K_j^T - lse_i)   on the allowed pairs
        D_i   = sum_c dO_i[:, c] * O_i[:, c]
        dS_ij = P_ij * (dO_i V_j^T - D_i)
        dq part = scale * dS_ij K_j,  dk part = scale * dS_ij^T Q_i,
        dv part = P_ij^T dO_i
    Summed over j (dq) and over i (dk, dv) these give attention_backward.
    Returns the three parts in float64, block-shaped.
    """
    B, Lb, Hq, d = q_blk.shape
    Hkv = k_blk.shape[2]
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    ti = block_tokens(S, P, i, order)
    tj = block_tokens(S, P, j, order)
    seg = None if position_ids is None else segment_ids(position_ids)
    dq = np.zeros((B, Lb, Hq, d))
    dk = np.zeros((B, Lb, Hkv, d))
    dv = np.zeros((B, Lb, Hkv, v_blk.shape[3]))
    for b in range(B):
        allowed = _allowed_between(None if seg is None else seg[b], ti, tj)
        for h in range(Hq):
            kvh = h // g
            qh = np.asarray(q_blk[b, :, h, :], dtype=np.float64)
            kh = np.asarray(k_blk[b, :, kvh, :], dtype=np.float64)
            vh = np.asarray(v_blk[b, :, kvh, :], dtype=np.float64)
            oh = np.asarray(out_blk[b, :, h, :], dtype=np.float64)
            doh = np.asarray(dout_blk[b, :, h, :], dtype=np.float64)
            lse = np.asarray(lse_blk[b, h, :], dtype=np.float64)
            live = allowed & np.isfinite(lse)[:, None]
            s = scale * (qh @ kh.T)
            p = np.where(live, np.exp(np.where(live, s - lse[:, None], 0.0)), 0.0)
            D = (doh * oh).sum(axis=1)
            ds = p * (doh @ vh.T - D[:, None])
            dq[b, :, h, :] += scale * (ds @ kh)
            dk[b, :, kvh, :] += scale * (ds.T @ qh)
            dv[b, :, kvh, :] += p.T @ doh
    return dq, dk, dv


def attention_backward_rows(q, k, v, dout, rows, position_ids=None, scale=None,
                            max_chunk_elems=1 << 24):
    """dq for the given query tokens only, every query head.

    The same derivatives as attention_backward, restricted to one query row
    t at a time: p = softmax of row t over its allowed keys, o = p V,
    D = dO_t . o, dS = p * (dO_t V^T - D), dq_t = scale * dS K.  A row needs
    only its own scores, so this runs at full sequence lengths.  Returns
    [B][R][Hq][d] in float64 for R = len(rows).
    """
    B, S, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = np.asarray(rows, dtype=np.int64)
    R = rows.shape[0]
    dq = np.zeros((B, R, Hq, d))
    seg = None if position_ids is None else segment_ids(position_ids)
    step = max(1, max_chunk_elems // max(S, 1))
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            for c0 in range(0, R, step):
                sel = rows[c0:c0 + step]
                kmax = S if seg is None else int(sel.max()) + 1
                keys = np.asarray(k[b, :kmax, kvh, :], dtype=np.float64)
                vals = np.asarray(v[b, :kmax, kvh, :], dtype=np.float64)
                if seg is None:
                    allowed = np.ones((sel.shape[0], kmax), dtype=bool)
                else:
                    j = np.arange(kmax)
                    allowed = (seg[b, :kmax][None, :] == seg[b, sel][:, None]) & (
                        j[None, :] <= sel[:, None])
                qr = np.asarray(q[b, sel, h, :], dtype=np.float64)
                dor = np.asarray(dout[b, sel, h, :], dtype=np.float64)
                o, lse = _softmax_attend(qr, keys, vals, allowed, scale)
                live = np.isfinite(lse)
                s = np.where(allowed, scale * (qr @ keys.T), NEG_INF)
                p = np.where(allowed & live[:, None],
                             np.exp(s - np.where(live, lse, 0.0)[:, None]), 0.0)
                D = (dor * o).sum(axis=1)
                ds = p * (dor @ vals.T - D[:, None])
                dq[b, c0:c0 + sel.shape[0], h, :] = scale * (ds @ keys)
    return dq


def attention_backward_keys(q, k, v, dout, keys, position_ids=None, scale=None, kv_heads=None,
                            max_chunk_elems=1 << 24):
    """dk and dv for the given key tokens only.

    dv_j = sum_t P_tj dO_t and dk_j = scale * sum_t dS_tj q_t over every
    query t allowed to see key j, in every query head of j's group.  Each
    such query enters with its full softmax statistics (lse_t and o_t over
    all its allowed keys, from attention_rows), then only the score columns
    of the sampled keys are formed.  kv_heads restricts the key/value heads
    computed (the others stay zero).  Returns dk, dv [B][J][Hkv][d] in
    float64 for J = len(keys).
    """
    B, S, Hq, Hkv, d = _check_shapes(q, k, v)
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    keys = np.asarray(keys, dtype=np.int64)
    J = keys.shape[0]
    dk = np.zeros((B, J, Hkv, d))
    dv = np.zeros((B, J, Hkv, v.shape[3]))
    heads = range(Hkv) if kv_heads is None else kv_heads
    seg = None if position_ids is None else segment_ids(position_ids)
    for b in range(B):
        # queries that see at least one sampled key
        if seg is None:
            qset = np.arange(S)
        else:
            t = np.arange(S)
            seen = np.zeros(S, dtype=bool)
            for j in keys:
                seen |= (t >= j) & (seg[b] == seg[b, j])
            qset = np.nonzero(seen)[0]
        if qset.shape[0] == 0:
            continue
        for kvh in heads:
            kj = np.asarray(k[b, keys, kvh, :], dtype=np.float64)
            vj = np.asarray(v[b, keys, kvh, :], dtype=np.float64)
            for h in range(kvh * g, (kvh + 1) * g):
                o, lse = attention_rows(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, kvh:kvh + 1],
                                        v[b:b + 1, :, kvh:kvh + 1], qset,
                                        None if position_ids is None
                                        else position_ids[b:b + 1], scale, max_chunk_elems)
                o, lse = o[0, :, 0, :], lse[0, 0, :]
                qr = np.asarray(q[b, qset, h, :], dtype=np.float64)
                dor = np.asarray(dout[b, qset, h, :], dtype=np.float64)
                if seg is None:
                    allowed = np.ones((qset.shape[0], J), dtype=bool)
                else:
                    allowed = (seg[b, qset][:, None] == seg[b, keys][None, :]) & (
                        keys[None, :] <= qset[:, None])
                live = np.isfinite(lse)
                s = scale * (qr @ kj.T)
                p = np.where(allowed & live[:, None],
                             np.exp(s - np.where(live, lse, 0.0)[:, None]), 0.0)
                D = (dor * o).sum(axis=1)
                ds = p * (dor @ vj.T - D[:, None])
                dv[b, :, kvh, :] += p.T @ dor
                dk[b, :, kvh, :] += scale * (ds.T @ qr)
    return dk, dv
