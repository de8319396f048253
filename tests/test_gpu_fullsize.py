"""Full-size parity at the benchmark workloads, in the launch configuration
bench.py times, against the float64 oracle computed on the host cores
(tests/fullsize_oracle.py runs it in the background from the session's
start):

  ulysses_4k     every row of every head (4096 x 32), through the permute ->
                 attention -> permute pipeline;
  llama8b_32k    every row of every head (32768 x 32);
  packed_128k    every row of every head (131072 x 32), for the contiguous
                 and the striped order (the oracle runs document by
                 document);
  halfmil_512k   the workload's 4096 seeded sampled rows of every head, for the
                 plain 16-block striped call and the 8 x 2 Ulysses + Ring
                 hybrid.
"""

import numpy as np
import pytest
import torch

from helpers import check_attention
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def _inputs(cfg):
    return workloads.qkv_torch(cfg["B"], cfg["S"], cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["seed"],
                               torch.bfloat16, "cuda")


def _check(out, lse, result, what):
    """Compare out [B][S][Hq][d] (device) and lse [B][Hq][S] (device) with an
    oracle result on its rows and heads, one head at a time; returns the
    worst (max, mean, lse) over the heads."""
    rows, heads, ref_out, ref_lse = result
    trows = torch.from_numpy(rows).to(out.device)
    worst = [0.0, 0.0, 0.0]
    for i, h in enumerate(heads):
        got = out[:, :, h].index_select(1, trows).float().cpu().numpy()
        got_lse = lse[:, h].index_select(1, trows).cpu().numpy()
        st = check_attention(got, got_lse, ref_out[:, :, i], ref_lse[:, i], "bf16",
                             f"{what} head {h}")
        worst = [max(a, b) for a, b in zip(worst, st)]
    print(f"PARITY {what}: {len(rows)} rows x {len(heads)} heads "
          "max=%.3e worst-head-mean=%.3e lse=%.3e" % tuple(worst))
    return worst


@pytest.mark.fullsize_oracle("ulysses_4k")
def test_ulysses_4k_pipeline_every_row(sp, fullsize_oracle):
    cfg = workloads.CONFIGS["ulysses_4k"]
    B, S, H, d, P = cfg["B"], cfg["S"], cfg["Hq"], cfg["d"], cfg["P"]
    q, k, v = _inputs(cfg)
    G = H // P
    yq, yk, yv = sp.seq_to_head(q, P), sp.seq_to_head(k, P), sp.seq_to_head(v, P)
    yo, ylse = sp.blockwise_attention(yq.view(P * B, S, G, d), yk.view(P * B, S, G, d),
                                      yv.view(P * B, S, G, d), P, "contiguous")
    out = sp.head_to_seq(yo.view(P, B, S, G, d))
    lse = ylse.view(P, B, G, S).permute(1, 0, 2, 3).reshape(B, H, S)
    torch.cuda.synchronize()
    res = fullsize_oracle.result("ulysses_4k")
    assert len(res[0]) == S and len(res[1]) == H
    _check(out, lse, res, "ulysses_4k pipeline")


@pytest.mark.fullsize_oracle("llama8b_32k")
def test_llama8b_32k_every_row(sp, fullsize_oracle):
    cfg = workloads.CONFIGS["llama8b_32k"]
    q, k, v = _inputs(cfg)
    pos = torch.from_numpy(workloads.position_ids(cfg)).cuda()
    out, lse = sp.blockwise_attention(q, k, v, cfg["P"], "contiguous", pos)
    torch.cuda.synchronize()
    del q, k, v
    res = fullsize_oracle.result("llama8b_32k")
    assert len(res[0]) == cfg["S"] and len(res[1]) == cfg["Hq"]
    _check(out, lse, res, "llama8b_32k contiguous")


@pytest.mark.fullsize_oracle("packed_128k")
@pytest.mark.parametrize("order", ["contiguous", "striped"])
def test_packed_128k_every_row(sp, fullsize_oracle, order):
    cfg = workloads.CONFIGS["packed_128k"]
    q, k, v = _inputs(cfg)
    pos = torch.from_numpy(workloads.position_ids(cfg)).cuda()
    out, lse = sp.blockwise_attention(q, k, v, cfg["P"], order, pos)
    torch.cuda.synchronize()
    del q, k, v
    res = fullsize_oracle.result("packed_128k")
    assert len(res[0]) == cfg["S"] and len(res[1]) == cfg["Hq"]
    _check(out, lse, res, f"packed_128k {order}")


@pytest.mark.fullsize_oracle("halfmil_512k")
def test_halfmil_512k_striped(sp, fullsize_oracle):
    cfg = workloads.CONFIGS["halfmil_512k"]
    q, k, v = _inputs(cfg)
    pos = torch.from_numpy(workloads.position_ids(cfg)).cuda()
    out, lse = sp.blockwise_attention(q, k, v, cfg["P"], "striped", pos)
    torch.cuda.synchronize()
    del q, k, v
    res = fullsize_oracle.result("halfmil_512k")
    assert len(res[0]) == cfg["sampled_rows"] and len(res[1]) == cfg["Hq"]
    _check(out, lse, res, "halfmil_512k striped")


@pytest.mark.fullsize_oracle("halfmil_512k")
def test_halfmil_ulysses_ring_hybrid(sp, fullsize_oracle):
    """halfmil_512k has 8 heads for P = 16 devices (Ulysses alone would need
    16 heads): 8 Ulysses head groups x 2 striped ring blocks, on the same
    4096 sampled rows (they include the first and last token of every
    block of both the 16-block and the 2-block striped partitions)."""
    cfg = workloads.CONFIGS["halfmil_512k"]
    S = cfg["S"]
    q, k, v = _inputs(cfg)
    pos = torch.from_numpy(workloads.position_ids(cfg)).cuda()
    out, lse = sp.ulysses_ring_attention(q, k, v, 8, 2, "striped", pos)
    torch.cuda.synchronize()
    del q, k, v
    res = fullsize_oracle.result("halfmil_512k")
    assert {0, 1, S - 2, S - 1} <= set(res[0].tolist())
    lse = lse.permute(1, 0, 2, 3).reshape(1, cfg["Hq"], S)
    _check(out, lse, res, "halfmil_512k hybrid 8x2")
