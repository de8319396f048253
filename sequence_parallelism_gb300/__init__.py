"""GB300-native blockwise (ring) attention and Ulysses layout permutation.

The compute runs in libsp_gb300.so (hand-written sm_103a CUDA, C ABI in
include/sp_gb300.h); this package only allocates outputs and workspace with
torch and calls the C entry points on the current stream.  Importing it
without the built library raises ImportError -- there is no CPU path.

    seq_to_head(x, P) / head_to_seq(y)         Ulysses redistribution
    blockwise_attention(q, k, v, P, ...)       ring-order online-softmax attention
    ring_step(q, k, v, P, step, ...)           one ring step's partial result
    merge_partials(outs, lses)                 log-sum-exp combine of partials
    ulysses_attention(q, k, v, P, ...)         permute -> attention -> permute back
    ulysses_attention_backward(ctx, dout)      its gradients (permute, backward, permute)
    ulysses_ring_attention(q, k, v, P_u, P_r)  Ulysses + Ring hybrid (heads < devices)
    blockwise_attention_backward(...)          dq, dk, dv from out, dout and lse
    doc_starts(position_ids)                   O(n) causal-mask carrier
    ring_block_step(q_blk, k_blk, v_blk, ...)  one device's ring step on block tensors
    ring_block_step_accumulate(...)            the same step folded into a running result
    ring_block_step_backward(...)              its gradient parts, into float32 accumulators
    query_block_attention(q_blk, k, v, ...)    one device's query block against all K/V

sequence_parallelism_gb300.dist runs the ring, all-gathered and Ulysses
exchanges across the ranks of a torch.distributed group (one GPU per rank).
"""

import torch

from . import _lib
from ._lib import SPError  # noqa: F401

__all__ = ["seq_to_head", "head_to_seq", "blockwise_attention", "ring_step", "merge_partials",
           "ulysses_attention", "ulysses_attention_backward", "ulysses_ring_attention",
           "blockwise_attention_backward",
           "doc_starts", "attention_workspace", "ring_block_step", "ring_block_step_accumulate",
           "ring_block_step_backward",
           "query_block_attention",
           "SPError"]


def seq_to_head(x, P, out=None):
    B, S, H, d = x.shape
    y = torch.empty((P, B, S, H // P, d), dtype=x.dtype, device=x.device) if out is None else out
    return _lib.sp_ulysses_seq_to_head(x, y, P)


def head_to_seq(y, out=None):
    P, B, S, G, d = y.shape
    x = torch.empty((B, S, P * G, d), dtype=y.dtype, device=y.device) if out is None else out
    return _lib.sp_ulysses_head_to_seq(y, x, P)


def attention_workspace(B, S, causal, device=None, minimal=False):
    """Workspace for the attention calls; by default large enough for the
    tail split of non-causal calls (minimal=True: the required minimum)."""
    if minimal:
        n = _lib.sp_blockwise_attn_workspace_bytes(B, S, causal)
    else:
        n = _lib.sp_blockwise_attn_split_workspace_bytes(B, S, causal)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _outputs(q, out, lse):
    B, S, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    return out, lse


def blockwise_attention(q, k, v, P, order="contiguous", position_ids=None, scale=0.0, out=None,
                        lse=None, workspace=None):
    """Exact attention over P ring blocks; returns (out, lse)."""
    B, S = q.shape[:2]
    out, lse = _outputs(q, out, lse)
    if workspace is None:
        workspace = attention_workspace(B, S, position_ids is not None, q.device)
    return _lib.sp_blockwise_attn_fwd(q, k, v, position_ids, P, order, scale, out, lse, workspace)


def ring_step(q, k, v, P, step, order="contiguous", position_ids=None, scale=0.0, out=None,
              lse=None, workspace=None):
    """Partial result of ring step `step` for every query block; (out, lse)."""
    B, S = q.shape[:2]
    out, lse = _outputs(q, out, lse)
    if workspace is None:
        workspace = attention_workspace(B, S, position_ids is not None, q.device)
    return _lib.sp_blockwise_attn_step(q, k, v, position_ids, P, order, step, scale, out, lse,
                                       workspace)


def _block_outputs(q_blk, out, lse):
    B, Lb, Hq, d = q_blk.shape
    if out is None:
        out = torch.empty_like(q_blk)
    if lse is None:
        lse = torch.empty((B, Hq, Lb), dtype=torch.float32, device=q_blk.device)
    return out, lse


def ring_block_step(q_blk, k_blk, v_blk, P, i, j, order="contiguous", position_ids=None,
                    scale=0.0, out=None, lse=None, workspace=None):
    """What device i of a ring computes at the step it holds key/value block
    j: query block i ([B][S/P][Hq][d]) against block j ([B][S/P][Hkv][d]),
    masks in global token indices (position_ids of the whole sequence, or
    None for non-causal).  Returns the partial (out, lse [B][Hq][S/P])."""
    B, Lb = q_blk.shape[:2]
    S = Lb * P
    out, lse = _block_outputs(q_blk, out, lse)
    if workspace is None:
        workspace = attention_workspace(B, S, position_ids is not None, q_blk.device)
    return _lib.sp_ring_block_step(q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, scale,
                                   out, lse, workspace)


def ring_block_step_accumulate(q_blk, k_blk, v_blk, P, i, j, out, lse, order="contiguous",
                               position_ids=None, scale=0.0, workspace=None):
    """ring_block_step folded into a running result: (out [B][S/P][Hq][d],
    lse [B][Hq][S/P] float32) hold the merge of the steps so far (rows with
    lse = -inf: none yet) and are updated in place by the log-sum-exp merge
    with pair (i, j)'s partial.  bf16, d = 128."""
    B, Lb = q_blk.shape[:2]
    S = Lb * P
    if workspace is None:
        workspace = attention_workspace(B, S, position_ids is not None, q_blk.device)
    return _lib.sp_ring_block_step_accumulate(q_blk, k_blk, v_blk, position_ids, S, P, order, i,
                                              j, scale, out, lse, workspace)


def ring_block_step_backward(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, P, i, j,
                             order="contiguous", position_ids=None, scale=0.0, dq_acc=None,
                             dk_acc=None, dv_acc=None, workspace=None):
    """The backward of one device's ring step: adds block pair (i, j)'s
    gradient parts into float32 accumulators (created zeroed when not
    given): dq_acc [B][S/P][Hq][d], dk_acc and dv_acc [B][S/P][Hkv][d].
    lse_blk is block i's forward lse over the whole sequence.  Returns the
    three accumulators."""
    B, Lb = q_blk.shape[:2]
    S = Lb * P
    f32 = lambda like, acc: acc if acc is not None else torch.zeros(
        like.shape, dtype=torch.float32, device=like.device)
    dq_acc, dk_acc, dv_acc = f32(q_blk, dq_acc), f32(k_blk, dk_acc), f32(v_blk, dv_acc)
    if workspace is None:
        n = _lib.sp_ring_block_step_bwd_workspace_bytes(B, S, q_blk.shape[2], P,
                                                        position_ids is not None)
        workspace = torch.empty(n, dtype=torch.uint8, device=q_blk.device)
    return _lib.sp_ring_block_step_bwd(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk,
                                       position_ids, S, P, order, i, j, scale, dq_acc, dk_acc,
                                       dv_acc, workspace)


def query_block_attention(q_blk, k, v, P, i, order="contiguous", position_ids=None, scale=0.0,
                          out=None, lse=None, workspace=None):
    """Query block i ([B][S/P][Hq][d]) against the whole sequence's k, v
    ([B][S][Hkv][d]) in ring order: block i's rows of blockwise_attention."""
    B, S = k.shape[:2]
    out, lse = _block_outputs(q_blk, out, lse)
    if workspace is None:
        workspace = attention_workspace(B, S, position_ids is not None, q_blk.device)
    return _lib.sp_query_block_attn_fwd(q_blk, k, v, position_ids, P, order, i, scale, out, lse,
                                        workspace)


def blockwise_attention_backward(q, k, v, out, dout, lse, P, order="contiguous",
                                 position_ids=None, scale=0.0, workspace=None):
    """Gradients (dq, dk, dv) of blockwise attention; lse from the forward."""
    B, S, Hq, d = q.shape
    if workspace is None:
        n = _lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, position_ids is not None)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    return _lib.sp_blockwise_attn_bwd(q, k, v, out, dout, lse, position_ids, P, order, scale, dq,
                                      dk, dv, workspace)


def merge_partials(outs, lses, out=None, lse=None):
    P, B, S, H, d = outs.shape
    if out is None:
        out = torch.empty((B, S, H, d), dtype=outs.dtype, device=outs.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=outs.device)
    return _lib.sp_attn_merge_partials(outs, lses, out, lse)


def doc_starts(position_ids):
    B, S = position_ids.shape
    ws = torch.empty(_lib.sp_segment_starts_workspace_bytes(B, S), dtype=torch.uint8,
                     device=position_ids.device)
    ds = torch.empty_like(position_ids)
    return _lib.sp_segment_starts(position_ids, ds, ws)


def ulysses_attention(q, k, v, P, ring_blocks=None, order="contiguous", scale=0.0, fused=False,
                      position_ids=None, return_context=False):
    """One Ulysses attention layer simulated on one GPU.

    q [B][S][Hq][d], k/v [B][S][Hkv][d] in sequence-sharded layout: permute to
    head groups ([P][B][S][H/P][d] = batch P*B), run blockwise attention with
    `ring_blocks` blocks per head group (default P), permute back.
    position_ids [B][S] (optional) makes it causal; every head group sees all
    positions, so each group uses the same rows.

    fused=True skips both permutations: on one GPU, attention on the
    sequence-sharded tensors computes every head group's result in place and
    writes the output already in sequence-sharded layout (bit-identical).

    return_context=True also returns what ulysses_attention_backward needs
    (the head-sharded q, k, v, output and lse).
    """
    B, S, Hq, d = q.shape
    rb = ring_blocks or P
    if fused:
        out, lse = blockwise_attention(q, k, v, rb, order, position_ids, scale)
        ctx = dict(fused=True, q=q, k=k, v=v, out=out, lse=lse, P=P, rb=rb, order=order,
                   pos=position_ids, scale=scale)
        return (out, ctx) if return_context else out
    G, Gk = Hq // P, k.shape[2] // P
    yq = torch.empty((P, B, S, G, d), dtype=q.dtype, device=q.device)
    yk = torch.empty((P, B, S, Gk, d), dtype=k.dtype, device=k.device)
    yv = torch.empty_like(yk)
    _lib.sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, P)
    ypos = None if position_ids is None else position_ids.repeat(P, 1)
    yo, ylse = blockwise_attention(yq.view(P * B, S, G, d), yk.view(P * B, S, Gk, d),
                                   yv.view(P * B, S, Gk, d), rb, order, ypos, scale)
    out = head_to_seq(yo.view(P, B, S, G, d))
    if not return_context:
        return out
    ctx = dict(fused=False, yq=yq, yk=yk, yv=yv, yo=yo, ylse=ylse, P=P, rb=rb, order=order,
               pos=ypos, scale=scale)
    return out, ctx


def ulysses_attention_backward(ctx, dout):
    """Gradients (dq, dk, dv) of a Ulysses layer, in sequence-sharded layout:
    dout goes to the head groups (the layer's second all-to-all, transposed),
    every group runs the blockwise attention backward, and the gradients come
    back (the first all-to-all, transposed)."""
    P, rb, order, pos, scale = ctx["P"], ctx["rb"], ctx["order"], ctx["pos"], ctx["scale"]
    if ctx["fused"]:
        return blockwise_attention_backward(ctx["q"], ctx["k"], ctx["v"], ctx["out"], dout,
                                            ctx["lse"], rb, order, pos, scale)
    yq, yk, yv, yo, ylse = ctx["yq"], ctx["yk"], ctx["yv"], ctx["yo"], ctx["ylse"]
    _, B, S, G, d = yq.shape
    Gk = yk.shape[3]
    ydo = seq_to_head(dout, P)
    dyq, dyk, dyv = blockwise_attention_backward(
        yq.view(P * B, S, G, d), yk.view(P * B, S, Gk, d), yv.view(P * B, S, Gk, d),
        yo.view(P * B, S, G, d), ydo.view(P * B, S, G, d), ylse, rb, order, pos, scale)
    return (head_to_seq(dyq.view(P, B, S, G, d)), head_to_seq(dyk.view(P, B, S, Gk, d)),
            head_to_seq(dyv.view(P, B, S, Gk, d)))


def ulysses_ring_attention(q, k, v, P_u, P_r, order="contiguous", position_ids=None, scale=0.0,
                           out=None, lse=None, workspace=None):
    """Ulysses + Ring hybrid: P_u head groups x P_r ring blocks; returns
    (out [B][S][Hq][d], lse [P_u][B][Hq/P_u][S])."""
    B, S, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((P_u, B, Hq // P_u, S), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = _lib.sp_ulysses_ring_attn_workspace_bytes(B, S, Hq, Hkv, d, position_ids is not None,
                                                      _lib._dtype(q))
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    return _lib.sp_ulysses_ring_attn_fwd(q, k, v, position_ids, P_u, P_r, order, scale, out, lse,
                                         workspace)
