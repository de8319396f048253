"""Reference Ulysses sequence-shard <-> head-shard redistribution.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Ulysses SP: entrenar modelos con millones de tokens" (Keryc), section "Cómo
funciona Ulysses Sequence Parallelism (SP)": an all-to-all gives every GPU all
sequence positions but only a subset of the heads, and a second all-to-all
undoes it.  "DeepSpeed-Ulysses" (orangingq blog), section "Method": the split
changes from (N/P, d) to (N, d/P).

On one device the P sequence shards are the P consecutive slices of the
token axis of x [B][S][H][d]; what rank r would receive is every token of the
heads r*H/P ... (r+1)*H/P - 1, stored as y[r] with shape [B][S][H/P][d]:

    y[r][b][t][hl][:] = x[b][t][r*H/P + hl][:]

The copy below walks the (rank, head) pairs one at a time and moves whole
[B][S][d] slices; head_to_seq is the same loop with the assignment reversed.
"""

import numpy as np


def _groups(H, P):
    if P < 1 or H % P:
        raise ValueError("H must be a multiple of P (Ulysses needs heads >= sp_size)")
    return H // P


def seq_to_head(x, P):
    """[B][S][H][d] -> [P][B][S][H/P][d] (bit copy, any dtype)."""
    x = np.asarray(x)
    B, S, H, d = x.shape
    if S % P:
        raise ValueError("S must be a multiple of P")
    G = _groups(H, P)
    y = np.empty((P, B, S, G, d), dtype=x.dtype)
    for r in range(P):
        for hl in range(G):
            y[r, :, :, hl, :] = x[:, :, r * G + hl, :]
    return y


def head_to_seq(y):
    """[P][B][S][H/P][d] -> [B][S][H][d]: the inverse redistribution."""
    y = np.asarray(y)
    P, B, S, G, d = y.shape
    x = np.empty((B, S, P * G, d), dtype=y.dtype)
    for r in range(P):
        for hl in range(G):
            x[:, :, r * G + hl, :] = y[r, :, :, hl, :]
    return x
