"""The multi-device data plane (sequence_parallelism_gb300.dist) on CPU
ranks of a gloo process group.

What runs here is the exchange logic -- who sends which block to whom at
which step, where received blocks land, how partials are merged and how the
all-to-alls reassemble head groups and sequence shards.  The per-device
arithmetic is supplied by the float64 oracle in place of the kernels (the
GPU tests check the kernels against the same oracle), and every supplied
step first checks that the block it was handed is the one the ring schedule
names ("Ring Attention", "Cómo funciona la atención en anillo": at step s
device i holds key/value block j = (i - s) mod P).  Each rank's result must
equal its rows of full attention, or of its gradients; in the ring backward
every step also checks that the dK/dV accumulators it is handed hold exactly
the parts of the ranks the block has visited so far."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(B, S, Hq, Hkv, d, causal, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, S, Hq, d))
    k = rng.standard_normal((B, S, Hkv, d))
    v = rng.standard_normal((B, S, Hkv, d))
    pos = None
    if causal == "packed":
        pos = np.stack([workloads.position_ids_from_lengths(workloads.doc_lengths(S, 4, seed + b))
                        for b in range(B)]).astype(np.int32)
    elif causal == "causal":
        pos = np.tile(np.arange(S, dtype=np.int32), (B, 1))
    return q, k, v, pos


class OracleKernels:
    """The per-device operations of dist.LibraryKernels computed by the
    oracle on CPU tensors, each step checking the blocks it is handed."""

    def __init__(self, q, k, v, pos, order, log):
        self.q, self.k, self.v, self.pos, self.order, self.log = q, k, v, pos, order, log

    def ring_step(self, q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, out, lse):
        ti, tj = oracle.block_tokens(S, P, i, order), oracle.block_tokens(S, P, j, order)
        assert np.array_equal(q_blk.numpy(), self.q[:, ti])
        assert np.array_equal(k_blk.numpy(), self.k[:, tj]), f"device {i} holds the wrong block"
        assert np.array_equal(v_blk.numpy(), self.v[:, tj])
        self.log.append((i, j))
        step = (i - j) % P
        o, l_ = oracle.ring_partial(self.q, self.k, self.v, P, step, order, self.pos)
        out.copy_(torch.from_numpy(o[:, ti]))
        lse.copy_(torch.from_numpy(l_[:, :, ti]))

    def ring_step_accumulate(self, q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, out,
                             lse):
        """Checks that the running result handed in is the merge of the steps
        device i has taken so far (j' = i, i - 1, ..., j + 1), then folds in
        pair (i, j)'s partial."""
        ti = oracle.block_tokens(S, P, i, order)
        step = (i - j) % P
        parts = [oracle.ring_partial(self.q, self.k, self.v, P, s_, order, self.pos)
                 for s_ in range(step)]
        ro, rl = oracle.merge_partials(np.stack([p_[0][:, ti] for p_ in parts]),
                                       np.stack([p_[1][:, :, ti] for p_ in parts]))
        assert np.abs(out.numpy() - ro).max() < 1e-12, "running result out of step"
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(lse.numpy()), fin)
        assert np.abs(lse.numpy()[fin] - rl[fin]).max() < 1e-12
        part_o, part_l = torch.empty_like(out), torch.empty_like(lse)
        self.ring_step(q_blk, k_blk, v_blk, position_ids, S, P, order, i, j, part_o, part_l)
        self.merge(torch.stack([out, part_o]), torch.stack([lse, part_l]), out, lse)

    def _pair_parts(self, S, P, order, i, j):
        ti, tj = oracle.block_tokens(S, P, i, order), oracle.block_tokens(S, P, j, order)
        return oracle.ring_partial_backward(
            self.q[:, ti], self.k[:, tj], self.v[:, tj], self.out[:, ti], self.dout[:, ti],
            self.lse[:, :, ti], S, P, i, j, order, self.pos)

    def ring_step_backward(self, q_blk, k_blk, v_blk, out_blk, dout_blk, lse_blk, position_ids,
                           S, P, order, i, j, dq_acc, dk_acc, dv_acc):
        ti, tj = oracle.block_tokens(S, P, i, order), oracle.block_tokens(S, P, j, order)
        assert np.array_equal(q_blk.numpy(), self.q[:, ti])
        assert np.array_equal(out_blk.numpy(), self.out[:, ti])
        assert np.array_equal(dout_blk.numpy(), self.dout[:, ti])
        assert np.array_equal(lse_blk.numpy(), self.lse[:, :, ti])
        assert np.array_equal(k_blk.numpy(), self.k[:, tj]), f"device {i} holds the wrong block"
        assert np.array_equal(v_blk.numpy(), self.v[:, tj])
        # block j started at rank j and has visited ranks j, ..., i - 1
        seen_k, seen_v = np.zeros(k_blk.shape), np.zeros(v_blk.shape)
        for r in range(j, j + (i - j) % P):
            _, pk, pv = self._pair_parts(S, P, order, r % P, j)
            seen_k += pk
            seen_v += pv
        assert np.abs(dk_acc.numpy() - seen_k).max() < 1e-12, "dK accumulator out of step"
        assert np.abs(dv_acc.numpy() - seen_v).max() < 1e-12, "dV accumulator out of step"
        self.log.append((i, j))
        pq, pk, pv = self._pair_parts(S, P, order, i, j)
        dq_acc += torch.from_numpy(pq)
        dk_acc += torch.from_numpy(pk)
        dv_acc += torch.from_numpy(pv)

    def merge(self, outs, lses, out, lse):
        o, l_ = oracle.merge_partials(outs.numpy(), lses.numpy())
        out.copy_(torch.from_numpy(o))
        lse.copy_(torch.from_numpy(l_))

    def query_block(self, q_blk, k, v, position_ids, P, order, i, out, lse):
        S = k.shape[1]
        ti = oracle.block_tokens(S, P, i, order)
        assert np.array_equal(k.numpy(), self.k) and np.array_equal(v.numpy(), self.v)
        qf = np.zeros_like(self.q)
        qf[:, ti] = q_blk.numpy()
        o, l_ = oracle.attention_rows(qf, k.numpy(), v.numpy(), ti, self.pos)
        out.copy_(torch.from_numpy(o))
        lse.copy_(torch.from_numpy(l_))

    def seq_to_head(self, x, y, P):
        y.copy_(torch.from_numpy(oracle.seq_to_head(x.numpy(), P)))

    def head_to_seq(self, y, x, P):
        x.copy_(torch.from_numpy(oracle.head_to_seq(y.numpy())))

    def attention_backward(self, q, k, v, out, dout, lse, position_ids, P, order, dq, dk, dv):
        g = oracle.attention_backward(q.numpy(), k.numpy(), v.numpy(), dout.numpy(), self.pos)
        for dst, src in zip((dq, dk, dv), g):
            dst.copy_(torch.from_numpy(src))

    def attention(self, q, k, v, position_ids, P, order, out, lse):
        o, l_ = oracle.blockwise_ring_attention(q.numpy(), k.numpy(), v.numpy(), P, order,
                                                self.pos)
        out.copy_(torch.from_numpy(o))
        lse.copy_(torch.from_numpy(l_))


def _worker(rank, world, port, kind, params, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sequence_parallelism_gb300 import dist as spd
        B, S, Hq, Hkv, d, causal, order, seed = params
        q, k, v, pos = _problem(B, S, Hq, Hkv, d, causal, seed)
        log = []
        kn = OracleKernels(q, k, v, pos, order, log)
        tpos = None if pos is None else torch.from_numpy(pos)
        ref_o, ref_l = oracle.full_attention(q, k, v, pos)
        if kind == "ring_bwd":
            t = oracle.block_tokens(S, world, rank, order)
            blk = lambda a, ax=1: torch.from_numpy(np.ascontiguousarray(np.take(a, t, axis=ax)))
            dout = np.random.default_rng(seed + 1).standard_normal(q.shape)
            kn.out, kn.lse, kn.dout = ref_o, ref_l, dout
            grads = spd.ring_attention_backward(blk(q), blk(k), blk(v), blk(ref_o), blk(dout),
                                                blk(ref_l, 2), tpos, order, kernels=kn)
            ref_g = oracle.attention_backward(q, k, v, dout, pos)
            err = max(np.abs(g_.numpy() - r_[:, t]).max() for g_, r_ in zip(grads, ref_g))
        elif kind in ("ring", "allgather"):
            t = oracle.block_tokens(S, world, rank, order)
            blk = lambda a: torch.from_numpy(np.ascontiguousarray(a[:, t]))
            fn = spd.ring_attention if kind == "ring" else spd.allgather_kv_attention
            out, lse = fn(blk(q), blk(k), blk(v), tpos, order, kernels=kn)
            err = max(np.abs(out.numpy() - ref_o[:, t]).max(),
                      np.abs(lse.numpy() - ref_l[:, :, t]).max())
        else:  # ulysses: sequence shards, contiguous; forward and backward
            Sl = S // world
            sh = lambda a: torch.from_numpy(np.ascontiguousarray(a[:, rank * Sl:(rank + 1) * Sl]))
            out, ctx = spd.ulysses_attention(sh(q), sh(k), sh(v), tpos, ring_blocks=2, order=order,
                                             kernels=kn, return_context=True)
            err = np.abs(out.numpy() - ref_o[:, rank * Sl:(rank + 1) * Sl]).max()
            dout = np.random.default_rng(seed + 1).standard_normal(q.shape)
            grads = spd.ulysses_attention_backward(ctx, sh(dout), kernels=kn)
            ref_g = oracle.attention_backward(q, k, v, dout, pos)
            for g_, r_ in zip(grads, ref_g):
                err = max(err, np.abs(g_.numpy() - r_[:, rank * Sl:(rank + 1) * Sl]).max())
        results[rank] = (float(err), log)
    finally:
        dist.destroy_process_group()


def _run(world, kind, params):
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, kind, params, results), nprocs=world, join=True)
        return dict(results)


@pytest.mark.parametrize("world,params", [
    (2, (1, 48, 2, 1, 8, "causal", "contiguous", 11)),
    (3, (2, 60, 2, 2, 8, "packed", "striped", 12)),
    (4, (1, 64, 4, 2, 8, "none", "contiguous", 13)),
])
def test_ring_exchange_order_and_merge(world, params):
    res = _run(world, "ring", params)
    for rank in range(world):
        err, log = res[rank]
        assert err < 1e-12, f"rank {rank}: {err}"
        assert log == [(rank, (rank - s) % world) for s in range(world)]


@pytest.mark.parametrize("world,params", [
    (2, (2, 48, 2, 1, 8, "packed", "contiguous", 21)),
    (3, (1, 60, 3, 3, 8, "causal", "contiguous", 22)),
])
def test_allgather_kv(world, params):
    res = _run(world, "allgather", params)
    for rank in range(world):
        assert res[rank][0] < 1e-12


@pytest.mark.parametrize("world,params", [
    (2, (1, 48, 4, 2, 8, "packed", "contiguous", 31)),
    (2, (2, 40, 2, 2, 8, "none", "striped", 32)),
    (4, (1, 64, 8, 4, 8, "causal", "contiguous", 33)),
])
def test_ulysses_all_to_all_forward_and_backward(world, params):
    res = _run(world, "ulysses", params)
    for rank in range(world):
        assert res[rank][0] < 1e-12


@pytest.mark.parametrize("world,params", [
    (2, (1, 48, 2, 1, 8, "causal", "contiguous", 41)),
    (3, (2, 60, 4, 2, 8, "packed", "striped", 42)),
    (4, (1, 64, 2, 2, 8, "none", "striped", 43)),
])
def test_ring_backward_exchange(world, params):
    """The ring backward: every rank sees key/value block j = (i - s) mod P at
    step s together with accumulators that hold the parts of exactly the
    ranks that block has visited, and ends with its own blocks' gradients
    (dq from its steps, dk/dv brought home by the last hop)."""
    res = _run(world, "ring_bwd", params)
    for rank in range(world):
        err, log = res[rank]
        assert err < 1e-10, f"rank {rank}: {err}"
        assert log == [(rank, (rank - s) % world) for s in range(world)]
