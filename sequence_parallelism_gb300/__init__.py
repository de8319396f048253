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
    ulysses_ring_attention(q, k, v, P_u, P_r)  Ulysses + Ring hybrid (heads < devices)
    blockwise_attention_backward(...)          dq, dk, dv from out, dout and lse
    doc_starts(position_ids)                   O(n) causal-mask carrier
"""

import torch

from . import _lib
from ._lib import SPError  # noqa: F401

__all__ = ["seq_to_head", "head_to_seq", "blockwise_attention", "ring_step", "merge_partials",
           "ulysses_attention", "ulysses_ring_attention", "blockwise_attention_backward",
           "doc_starts", "attention_workspace",
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


def ulysses_attention(q, k, v, P, ring_blocks=None, order="contiguous", scale=0.0, fused=False):
    """One Ulysses attention layer simulated on one GPU.

    q [B][S][Hq][d], k/v [B][S][Hkv][d] in sequence-sharded layout: permute to
    head groups ([P][B][S][H/P][d] = batch P*B), run blockwise attention with
    `ring_blocks` blocks per head group (default P), permute back.  Non-causal.

    fused=True skips both permutations: on one GPU, attention on the
    sequence-sharded tensors computes every head group's result in place and
    writes the output already in sequence-sharded layout (bit-identical).
    """
    B, S, Hq, d = q.shape
    if fused:
        out, _ = blockwise_attention(q, k, v, ring_blocks or P, order, None, scale)
        return out
    G, Gk = Hq // P, k.shape[2] // P
    yq = torch.empty((P, B, S, G, d), dtype=q.dtype, device=q.device)
    yk = torch.empty((P, B, S, Gk, d), dtype=k.dtype, device=k.device)
    yv = torch.empty_like(yk)
    _lib.sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, P)
    yo, _ = blockwise_attention(yq.view(P * B, S, G, d), yk.view(P * B, S, Gk, d),
                                yv.view(P * B, S, Gk, d), ring_blocks or P, order, None, scale)
    return head_to_seq(yo.view(P, B, S, G, d))


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
