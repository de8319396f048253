"""Seeded synthetic workloads: shapes, inputs, document splits, sampled rows.

Input generation only -- nothing here computes attention or a permutation.
Tests and bench.py draw the inputs from here, so the CUDA path and the CPU
oracle always see the same numbers.  The module stands apart from both the
library package and oracle/: importing it loads neither the CUDA library nor
the oracle (torch is imported only by the functions that draw on a device).

The five workloads (q, k, v ~ N(0, 1), then rounded to the storage dtype):
  ring_tiny     P=4 blocks x 8 tokens, d=16, 1 head, fp32, non-causal; the Ring
                Attention page's own draw (torch.manual_seed(0);
                torch.randn(3, 32, 16)), frozen in tests/golden.
  ulysses_4k    B=1, S=4096, H=32, d=128, P=4, bf16, non-causal; the Ulysses
                layer: seq->head permute, blockwise attention per head group,
                head->seq permute.
  llama8b_32k   Llama-3.1-8B-shaped causal attention: S=32768, Hq=32, Hkv=8,
                d=128, bf16, position_ids 0..S-1, P=8 contiguous blocks.
  packed_128k   S=131072, Hq=32, Hkv=8, d=128, bf16, 8 packed documents with
                seeded lengths (position_ids restart per document), P=8,
                contiguous and striped.
  halfmil_512k  S=524288, Hq=Hkv=8, d=128, bf16, causal, P=16 striped; the
                oracle is checked on 4096 seeded query rows.
"""

import json
import os

import numpy as np

_ROOT = os.path.dirname(os.path.abspath(__file__))
GOLDEN_RING_TINY = os.path.join(_ROOT, "tests", "golden", "ring_tiny_seed0.json")

CONFIGS = {
    "ring_tiny": dict(B=1, S=32, Hq=1, Hkv=1, d=16, P=4, orders=("contiguous",), causal=False,
                      dtype="f32", seed=0),
    "ulysses_4k": dict(B=1, S=4096, Hq=32, Hkv=32, d=128, P=4, orders=("contiguous",),
                       causal=False, dtype="bf16", seed=1002, ulysses=True),
    "llama8b_32k": dict(B=1, S=32768, Hq=32, Hkv=8, d=128, P=8, orders=("contiguous",),
                        causal=True, dtype="bf16", seed=1003),
    "packed_128k": dict(B=1, S=131072, Hq=32, Hkv=8, d=128, P=8,
                        orders=("contiguous", "striped"), causal=True, dtype="bf16", seed=1004,
                        n_docs=8),
    "halfmil_512k": dict(B=1, S=524288, Hq=8, Hkv=8, d=128, P=16, orders=("striped",),
                         causal=True, dtype="bf16", seed=1005, sampled_rows=4096),
}


def ring_tiny_arrays():
    """q, k, v [32][16] float32 of the Ring Attention page's example."""
    with open(GOLDEN_RING_TINY, encoding="utf-8") as f:
        doc = json.load(f)
    return tuple(np.array(doc[n], dtype=np.float32) for n in ("q", "k", "v"))


def doc_lengths(S, n_docs, seed):
    """n_docs lengths summing to S: n_docs-1 distinct cut points drawn
    uniformly from 1..S-1 (not tile-aligned)."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, S), n_docs - 1, replace=False))
    return np.diff(np.concatenate([[0], cuts, [S]])).astype(np.int64)


def position_ids_from_lengths(lengths):
    return np.concatenate([np.arange(L, dtype=np.int32) for L in lengths])


def position_ids(cfg):
    """[B][S] int32 for a causal config (None for non-causal ones)."""
    if not cfg["causal"]:
        return None
    S, B = cfg["S"], cfg["B"]
    if cfg.get("n_docs"):
        row = position_ids_from_lengths(doc_lengths(S, cfg["n_docs"], cfg["seed"]))
    else:
        row = np.arange(S, dtype=np.int32)
    return np.tile(row[None, :], (B, 1)).astype(np.int32)


def sample_rows(S, P, n, seed, order="contiguous"):
    """n distinct query tokens: t = 0, S-1, the first and last token of every
    block in the given order, then seeded uniform draws without replacement."""
    must = {0, S - 1}
    Lb = S // P
    for p in range(P):
        if order == "striped":
            must.update({p, p + (Lb - 1) * P})
        else:
            must.update({p * Lb, (p + 1) * Lb - 1})
    must = sorted(must)
    rng = np.random.default_rng(seed)
    pool = np.setdiff1d(np.arange(S), np.array(must))
    extra = rng.choice(pool, max(0, n - len(must)), replace=False)
    return np.sort(np.concatenate([np.array(must), extra]).astype(np.int64))


def qkv_torch(B, S, Hq, Hkv, d, seed, dtype, device):
    """q [B][S][Hq][d], k/v [B][S][Hkv][d] ~ N(0,1) drawn on `device` from a
    seeded generator, then cast to `dtype` (torch)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for h in (Hq, Hkv, Hkv):
        t = torch.randn((B, S, h, d), generator=g, device=device, dtype=torch.float32)
        out.append(t.to(dtype))
    return tuple(out)


def small_case(B, S, Hq, Hkv, d, seed, dtype="bf16", device="cuda"):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return qkv_torch(B, S, Hq, Hkv, d, seed, tdt, device)
