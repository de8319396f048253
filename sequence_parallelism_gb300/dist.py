"""The multi-device data plane: ring attention and Ulysses across the ranks of
a torch.distributed process group, one device per rank.

The pages describe three ways to spread one attention layer over P devices:

* Ring ("Ring Attention", "Cómo funciona la atención en anillo"): device i
  keeps query block i; at every step it sends the key/value block it holds to
  device i + 1 and receives one from device i - 1, so at step s it holds block
  j = (i - s) mod P; the partial results are combined by the cumulative
  softmax.  ring_attention() below: P - 1 point-to-point exchanges, the next
  block in flight while the current one is multiplied; its gradients in
  ring_attention_backward(), where each key/value block travels with its
  dK/dV accumulators.
* Ulysses ("Ulysses SP: entrenar modelos con millones de tokens", "Cómo
  funciona Ulysses Sequence Parallelism (SP)"; "DeepSpeed-Ulysses",
  "Method"): an all-to-all turns every device's sequence shard of all heads
  into the whole sequence of a head group, attention runs per head group, and
  a second all-to-all turns the result back.  ulysses_attention() below,
  and its gradients (the same exchanges transposed around the per-group
  backward) in ulysses_attention_backward().
* All-gathered K/V ("Ulysses序列并行技术详解：ms-swift如何降低长序列显存占用"):
  K and V reach every rank through two all-gathers and each rank attends its
  own query block against the whole sequence.  allgather_kv_attention() below.

torch.distributed moves the bytes (NCCL between GPUs); every arithmetic step
runs in the library's kernels through `kernels`, an object with the per-device
operations (LibraryKernels by default: the C entry points on the current CUDA
stream).  Remote blocks always land in this device's memory before a kernel
reads them.  Shapes: B batch rows, S the whole sequence, P = world size, Lb =
S / P rows per block, block rows in block order (row u of block p is token
p*Lb + u in the contiguous order, u*P + p in the striped one); position_ids is
the whole sequence's [B][S] on every rank (O(S) integers: the mask needs
global token indices).
"""

import torch
import torch.distributed as dist

from . import _lib


class LibraryKernels:
    """The per-device operations, on the library's kernels.  Each writes its
    result into the tensors it is given."""

    def __init__(self):
        self._ws = {}

    def workspace(self, B, S, causal, device):
        key = (B, S, bool(causal), str(device))
        if key not in self._ws:
            n = _lib.sp_blockwise_attn_split_workspace_bytes(B, S, causal)
            self._ws[key] = torch.empty(n, dtype=torch.uint8, device=device)
        return self._ws[key]

    def ring_step(self, q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, out, lse):
        ws = self.workspace(q_blk.shape[0], S, position_ids is not None, q_blk.device)
        _lib.sp_ring_block_step(q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, 0.0, out,
                                lse, ws)

    def ring_step_accumulate(self, q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, out,
                             lse):
        """Folds pair (i, j)'s partial into the running (out, lse): one call
        for bf16 with d = 128, else the step into a temporary and the merge
        (both on the library's kernels)."""
        ws = self.workspace(q_blk.shape[0], S, position_ids is not None, q_blk.device)
        if q_blk.dtype == torch.bfloat16 and q_blk.shape[3] == 128:
            _lib.sp_ring_block_step_accumulate(q_blk, k_blk, v_blk, position_ids, S, P, order,
                                               i, j, 0.0, out, lse, ws)
            return
        outs = torch.empty((2,) + tuple(out.shape), dtype=out.dtype, device=out.device)
        lses = torch.empty((2,) + tuple(lse.shape), dtype=lse.dtype, device=lse.device)
        outs[0].copy_(out)
        lses[0].copy_(lse)
        _lib.sp_ring_block_step(q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, 0.0,
                                outs[1], lses[1], ws)
        _lib.sp_attn_merge_partials(outs, lses, out, lse)

    def ring_step_backward(self, q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, position_ids,
                           S, P, order, i, j, dq_acc, dk_acc, dv_acc):
        B, _, Hq, _ = q_blk.shape
        causal = position_ids is not None
        key = ("ring_bwd", B, S, Hq, P, causal, str(q_blk.device))
        if key not in self._ws:
            n = _lib.sp_ring_block_step_bwd_workspace_bytes(B, S, Hq, P, causal)
            self._ws[key] = torch.empty(n, dtype=torch.uint8, device=q_blk.device)
        _lib.sp_ring_block_step_bwd(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, position_ids,
                                    S, P, order, i, j, 0.0, dq_acc, dk_acc, dv_acc, self._ws[key])

    def merge(self, outs, lses, out, lse):
        _lib.sp_attn_merge_partials(outs, lses, out, lse)

    def query_block(self, q_blk, k, v, position_ids, P, order, i, out, lse):
        ws = self.workspace(q_blk.shape[0], k.shape[1], position_ids is not None, q_blk.device)
        _lib.sp_query_block_attn_fwd(q_blk, k, v, position_ids, P, order, i, 0.0, out, lse, ws)

    def seq_to_head(self, x, y, P):
        _lib.sp_ulysses_seq_to_head(x, y, P)

    def head_to_seq(self, y, x, P):
        _lib.sp_ulysses_head_to_seq(y, x, P)

    def attention(self, q, k, v, position_ids, P, order, out, lse):
        ws = self.workspace(q.shape[0], q.shape[1], position_ids is not None, q.device)
        _lib.sp_blockwise_attn_fwd(q, k, v, position_ids, P, order, 0.0, out, lse, ws)

    def attention_backward(self, q, k, v, out, dout, lse, position_ids, P, order, dq, dk, dv):
        B, S, Hq, _ = q.shape
        key = ("bwd", B, S, Hq, P, position_ids is not None, str(q.device))
        if key not in self._ws:
            n = _lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, position_ids is not None)
            self._ws[key] = torch.empty(n, dtype=torch.uint8, device=q.device)
        _lib.sp_blockwise_attn_bwd(q, k, v, out, dout, lse, position_ids, P, order, 0.0, dq, dk,
                                   dv, self._ws[key])


_DEFAULT = None


def _kernels(kernels):
    global _DEFAULT
    if kernels is not None:
        return kernels
    if _DEFAULT is None:
        _DEFAULT = LibraryKernels()
    return _DEFAULT


def _lse_dtype(t):
    """lse is float32 for the library's bf16 and fp32 tensors (float64 data,
    which only a caller's own kernels can take, keeps float64)."""
    return torch.float64 if t.dtype == torch.float64 else torch.float32


def _world(group):
    return dist.get_world_size(group), dist.get_rank(group)


def _peer(group, r):
    """Global rank of rank r of `group` (point-to-point ops take global ranks)."""
    return r if group is None else dist.get_global_rank(group, r)


def ring_attention(q_blk, k_blk, v_blk, position_ids, order="contiguous", group=None,
                   kernels=None):
    """Ring attention across the group: this rank (i of P) holds query,
    key and value block i ([B][Lb][H][d]); returns its rows of the exact
    attention, (out [B][Lb][Hq][d], lse [B][Hq][Lb]).

    Step s: the partial of query block i against the key/value block held,
    j = (i - s) mod P, is folded into the running result by the log-sum-exp
    merge (step 0 writes it, the later steps accumulate into it); meanwhile
    the held block goes to rank i + 1 and the next one arrives from rank
    i - 1 into the second of two buffers.
    """
    kn = _kernels(kernels)
    P, i = _world(group)
    B, Lb, Hq, d = q_blk.shape
    S = Lb * P
    nxt_rank, prv_rank = _peer(group, (i + 1) % P), _peer(group, (i - 1) % P)
    kv = [(k_blk, v_blk), (torch.empty_like(k_blk), torch.empty_like(v_blk))]
    out = torch.empty((B, Lb, Hq, d), dtype=q_blk.dtype, device=q_blk.device)
    lse = torch.empty((B, Hq, Lb), dtype=_lse_dtype(q_blk), device=q_blk.device)
    for s in range(P):
        j = (i - s) % P
        reqs = []
        if s + 1 < P:
            ck, cv = kv[s % 2]
            nk, nv = kv[(s + 1) % 2]
            reqs = dist.batch_isend_irecv([
                dist.P2POp(dist.isend, ck, nxt_rank, group),
                dist.P2POp(dist.isend, cv, nxt_rank, group),
                dist.P2POp(dist.irecv, nk, prv_rank, group),
                dist.P2POp(dist.irecv, nv, prv_rank, group)])
        hk, hv = kv[s % 2]
        if s == 0:
            kn.ring_step(q_blk, hk, hv, position_ids, S, P, order, i, j, out, lse)
        else:
            kn.ring_step_accumulate(q_blk, hk, hv, position_ids, S, P, order, i, j, out, lse)
        for r in reqs:
            r.wait()
    return out, lse


def ring_attention_backward(q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, position_ids,
                            order="contiguous", group=None, kernels=None):
    """Gradients of ring_attention across the group.  This rank (i of P)
    holds block i of q, k, v, of the forward's out and lse, and of dout;
    returns (dq, dk, dv) for its blocks in the inputs' dtypes.

    Step s: with key/value block j = (i - s) mod P and that block's dK/dV
    accumulators (float32; float64 for float64 data), add pair (i, j)'s
    gradient parts -- dq locally, dk and dv into the travelling
    accumulators -- then pass K_j, V_j and the accumulators to rank i + 1.
    K/V of the next step are in flight while the step is computed; the
    accumulators can leave only after it, and make one last hop after step
    P - 1, which brings every block's accumulators back to the rank that
    holds it.
    """
    kn = _kernels(kernels)
    P, i = _world(group)
    B, Lb, Hq, d = q_blk.shape
    S = Lb * P
    nxt_rank, prv_rank = _peer(group, (i + 1) % P), _peer(group, (i - 1) % P)
    acc_dtype = torch.float64 if q_blk.dtype == torch.float64 else torch.float32
    dev = q_blk.device
    dq = torch.zeros((B, Lb, Hq, d), dtype=acc_dtype, device=dev)
    kv = [(k_blk, v_blk), (torch.empty_like(k_blk), torch.empty_like(v_blk))]
    acc = [(torch.zeros(k_blk.shape, dtype=acc_dtype, device=dev),
            torch.zeros(v_blk.shape, dtype=acc_dtype, device=dev)),
           (torch.empty(k_blk.shape, dtype=acc_dtype, device=dev),
            torch.empty(v_blk.shape, dtype=acc_dtype, device=dev))]
    for s in range(P):
        j = (i - s) % P
        reqs = []
        if s + 1 < P:
            (ck, cv), (nk, nv) = kv[s % 2], kv[(s + 1) % 2]
            reqs = dist.batch_isend_irecv([
                dist.P2POp(dist.isend, ck, nxt_rank, group),
                dist.P2POp(dist.isend, cv, nxt_rank, group),
                dist.P2POp(dist.irecv, nk, prv_rank, group),
                dist.P2POp(dist.irecv, nv, prv_rank, group)])
        hk, hv = kv[s % 2]
        ak, av = acc[s % 2]
        kn.ring_step_backward(q_blk, hk, hv, out_blk, dout_blk, lse_blk, position_ids, S, P,
                              order, i, j, dq, ak, av)
        (nak, nav) = acc[(s + 1) % 2]
        reqs += dist.batch_isend_irecv([
            dist.P2POp(dist.isend, ak, nxt_rank, group),
            dist.P2POp(dist.isend, av, nxt_rank, group),
            dist.P2POp(dist.irecv, nak, prv_rank, group),
            dist.P2POp(dist.irecv, nav, prv_rank, group)])
        for r in reqs:
            r.wait()
    dk, dv = acc[P % 2]
    return dq.to(q_blk.dtype), dk.to(k_blk.dtype), dv.to(v_blk.dtype)


def allgather_kv_attention(q_blk, k_blk, v_blk, position_ids, order="contiguous", group=None,
                           kernels=None):
    """The all-gathered variant: K and V of every rank are gathered (two
    all-gathers), then this rank's query block attends the whole sequence.
    Contiguous order only (the gathered blocks are then the sequence in
    token order).  Returns (out [B][Lb][Hq][d], lse [B][Hq][Lb])."""
    if order != "contiguous":
        raise ValueError("the all-gathered variant takes the contiguous order")
    kn = _kernels(kernels)
    P, i = _world(group)
    B, Lb, Hkv, d = k_blk.shape
    S = Lb * P
    k = torch.empty((B, S, Hkv, d), dtype=k_blk.dtype, device=k_blk.device)
    v = torch.empty_like(k)
    for b in range(B):  # [P][Lb] of batch row b is its whole sequence
        dist.all_gather_into_tensor(k[b], k_blk[b].contiguous(), group=group)
        dist.all_gather_into_tensor(v[b], v_blk[b].contiguous(), group=group)
    out = torch.empty_like(q_blk)
    lse = torch.empty((B, q_blk.shape[2], Lb), dtype=_lse_dtype(q_blk), device=q_blk.device)
    kn.query_block(q_blk, k, v, position_ids, P, order, i, out, lse)
    return out, lse


def _to_head_groups(t, P, kn, group):
    """[B][S/P][H][d] sequence shard of every rank -> this rank's head group
    for the whole sequence, [B][S][H/P][d]: local seq->head, then an
    all-to-all (one batch row at a time; recv[p] = rank p's tokens)."""
    B, Sl, H, d = t.shape
    gh = H // P
    y = torch.empty((P, B, Sl, gh, d), dtype=t.dtype, device=t.device)
    kn.seq_to_head(t, y, P)
    f = torch.empty((B, Sl * P, gh, d), dtype=t.dtype, device=t.device)
    for b in range(B):
        dist.all_to_all_single(f[b].view(P, Sl, gh, d), y[:, b].contiguous(), group=group)
    return f


def _to_seq_shards(f, P, kn, group):
    """The inverse: this rank's head group for the whole sequence,
    [B][S][G][d] -> its sequence shard of every head, [B][S/P][G*P][d]
    (all-to-all sending shard p to rank p, then local head->seq)."""
    B, S, G, d = f.shape
    Sl = S // P
    back = torch.empty((P, B, Sl, G, d), dtype=f.dtype, device=f.device)
    for b in range(B):
        if B == 1:  # back[:, 0] is contiguous: receive in place
            dist.all_to_all_single(back[:, 0], f[0].view(P, Sl, G, d), group=group)
        else:
            recv = torch.empty((P, Sl, G, d), dtype=f.dtype, device=f.device)
            dist.all_to_all_single(recv, f[b].view(P, Sl, G, d), group=group)
            back[:, b] = recv
    out = torch.empty((B, Sl, G * P, d), dtype=f.dtype, device=f.device)
    kn.head_to_seq(back, out, P)
    return out


def ulysses_attention(q, k, v, position_ids=None, ring_blocks=1, order="contiguous", group=None,
                      kernels=None, return_context=False):
    """One Ulysses attention layer across the group: this rank holds the
    sequence shard r (tokens [r*S/P, (r+1)*S/P)) of every head, q
    [B][S/P][Hq][d], k/v [B][S/P][Hkv][d]; returns its shard of the output
    [B][S/P][Hq][d] (and, with return_context, what
    ulysses_attention_backward needs).

    seq->head on the shard gives P head-group slices; the first all-to-all
    sends slice g to rank g, so this rank holds head group r for the whole
    sequence; attention (ring_blocks blocks, `order`) runs on it; the result
    is cut into P sequence shards and the second all-to-all sends shard p back
    to rank p, where head->seq restores [S/P][H].
    """
    kn = _kernels(kernels)
    P, r = _world(group)
    B, Sl, Hq, d = q.shape
    Hkv = k.shape[2]
    if Hq % P or Hkv % P:
        raise ValueError("Ulysses needs the head counts divisible by the group size")
    S = Sl * P
    G = Hq // P
    fq, fk, fv = (_to_head_groups(t, P, kn, group) for t in (q, k, v))
    out_g = torch.empty_like(fq)
    lse_g = torch.empty((B, G, S), dtype=_lse_dtype(q), device=q.device)
    kn.attention(fq, fk, fv, position_ids, ring_blocks, order, out_g, lse_g)
    out = _to_seq_shards(out_g, P, kn, group)
    if not return_context:
        return out
    return out, dict(q=fq, k=fk, v=fv, out=out_g, lse=lse_g, pos=position_ids, rb=ring_blocks,
                     order=order)


def ulysses_attention_backward(ctx, dout, group=None, kernels=None):
    """Gradients of ulysses_attention across the group: dout, this rank's
    sequence shard [B][S/P][Hq][d], goes to the head groups like q did (the
    transpose of the second all-to-all), every rank runs the blockwise
    attention backward on its head group for the whole sequence, and dq, dk,
    dv come back to sequence shards (the transpose of the first all-to-all).
    Returns (dq, dk, dv), this rank's shards."""
    kn = _kernels(kernels)
    P, _ = _world(group)
    fdo = _to_head_groups(dout, P, kn, group)
    dq_g, dk_g, dv_g = (torch.empty_like(ctx[n]) for n in ("q", "k", "v"))
    kn.attention_backward(ctx["q"], ctx["k"], ctx["v"], ctx["out"], fdo, ctx["lse"], ctx["pos"],
                          ctx["rb"], ctx["order"], dq_g, dk_g, dv_g)
    return tuple(_to_seq_shards(g, P, kn, group) for g in (dq_g, dk_g, dv_g))
