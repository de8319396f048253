"""Full-size parity at the benchmark workloads, in the launch configuration
bench.py times, on seeded sampled query rows that the oracle computes one by
one (all heads of each sampled row)."""

import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import check_attention, np32
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def oracle_rows(qn, kn, vn, rows, pos):
    """oracle.attention_rows split over query heads on a thread pool (numpy
    releases the GIL inside exp / matmul)."""
    Hq, Hkv = qn.shape[2], kn.shape[2]
    g = Hq // Hkv

    def one(h):
        kv = h // g
        return oracle.attention_rows(qn[:, :, h:h + 1], kn[:, :, kv:kv + 1], vn[:, :, kv:kv + 1],
                                     rows, pos)

    workers = min(Hq, os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        parts = list(ex.map(one, range(Hq)))
    out = np.concatenate([p[0] for p in parts], axis=2)
    lse = np.concatenate([p[1] for p in parts], axis=1)
    return out, lse


def _inputs(cfg):
    q, k, v = workloads.qkv_torch(cfg["B"], cfg["S"], cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["seed"],
                                  torch.bfloat16, "cuda")
    return q, k, v


def test_ulysses_4k_pipeline(sp):
    cfg = workloads.CONFIGS["ulysses_4k"]
    B, S, H, d, P = cfg["B"], cfg["S"], cfg["Hq"], cfg["d"], cfg["P"]
    q, k, v = _inputs(cfg)
    G = H // P
    yq, yk, yv = sp.seq_to_head(q, P), sp.seq_to_head(k, P), sp.seq_to_head(v, P)
    yo, ylse = sp.blockwise_attention(yq.view(P * B, S, G, d), yk.view(P * B, S, G, d),
                                      yv.view(P * B, S, G, d), P, "contiguous")
    out = sp.head_to_seq(yo.view(P, B, S, G, d))
    torch.cuda.synchronize()
    rows = workloads.sample_rows(S, P, 512, cfg["seed"])
    ref_out, ref_lse = oracle_rows(np32(q), np32(k), np32(v), rows, None)
    lse = ylse.view(P, B, G, S).permute(1, 0, 2, 3).reshape(B, H, S)
    stats = check_attention(np32(out)[:, rows], lse.cpu().numpy()[:, :, rows], ref_out, ref_lse,
                            "bf16", "ulysses_4k")
    print("PARITY ulysses_4k contiguous max=%.3e mean=%.3e lse=%.3e" % stats)


@pytest.mark.parametrize("name,order", [("llama8b_32k", "contiguous"),
                                        ("packed_128k", "contiguous"),
                                        ("packed_128k", "striped"),
                                        ("halfmil_512k", "striped")])
def test_causal_full_size(sp, name, order):
    cfg = workloads.CONFIGS[name]
    q, k, v = _inputs(cfg)
    pos = workloads.position_ids(cfg)
    out, lse = sp.blockwise_attention(q, k, v, cfg["P"], order, torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    n = cfg.get("sampled_rows", 256)
    rows = workloads.sample_rows(cfg["S"], cfg["P"], n, cfg["seed"], order)
    got_out = np32(out[:, rows])
    got_lse = lse[:, :, rows].cpu().numpy()
    del out, lse
    ref_out, ref_lse = oracle_rows(np32(q), np32(k), np32(v), rows, pos)
    stats = check_attention(got_out, got_lse, ref_out, ref_lse, "bf16", f"{name} {order}")
    print(f"PARITY {name} {order} " + "max=%.3e mean=%.3e lse=%.3e" % stats)


def test_halfmil_ulysses_ring_hybrid(sp):
    """halfmil_512k has 8 heads for P = 16 devices (Ulysses alone would need
    16 heads): 8 Ulysses head groups x 2 striped ring blocks."""
    cfg = workloads.CONFIGS["halfmil_512k"]
    q, k, v = _inputs(cfg)
    pos = workloads.position_ids(cfg)
    out, lse = sp.ulysses_ring_attention(q, k, v, 8, 2, "striped", torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    rows = workloads.sample_rows(cfg["S"], 2, 512, cfg["seed"] + 1, "striped")
    got_out = np32(out[:, rows])
    got_lse = lse.permute(1, 0, 2, 3).reshape(1, cfg["Hq"], cfg["S"])[:, :, rows].cpu().numpy()
    del out, lse
    ref_out, ref_lse = oracle_rows(np32(q), np32(k), np32(v), rows, pos)
    stats = check_attention(got_out, got_lse, ref_out, ref_lse, "bf16", "halfmil hybrid 8x2")
    print("PARITY halfmil_512k hybrid-8x2 max=%.3e mean=%.3e lse=%.3e" % stats)
