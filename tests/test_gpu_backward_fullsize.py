"""Full-size parity of the attention backward at the causal benchmark shapes.

* dq on seeded sampled query rows, every head (attention_backward_rows);
* dk, dv on sampled key rows of one key/value head: every query that sees
  them enters with its full softmax statistics (attention_backward_keys);
* sum rules that hold at any size, on the whole tensors: the rows of dS sum
  to zero, so sum_j dk_j = 0; the rows of P sum to one, so sum_j dv_j equals
  the sum of dout over the group's query heads.
out and lse come from our forward, as in a training step."""

import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle
from helpers import check_grad, np32
import workloads

pytestmark = pytest.mark.gpu

SUM_RULE_TOL = 1e-3  # |sum| relative to sum of |.| per column (bf16 storage)


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def _pool(fn, items):
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(items),
                                                               os.cpu_count() or 1)) as ex:
        return list(ex.map(fn, items))


def _sampled_keys(pos, S, P, order):
    """Key tokens whose observers are cheap to enumerate: the last 16 tokens
    of every document, every token of documents up to 128 long, the first 16
    of documents up to 5000 long; for a single document, the last block."""
    seg_starts = np.nonzero(pos[0] == 0)[0]
    ends = np.append(seg_starts[1:], S)
    keys = set()
    for a, e in zip(seg_starts, ends):
        L = e - a
        keys.update(range(max(a, e - 16), e))
        if L <= 128:
            keys.update(range(a, e))
        elif L <= 5000:
            keys.update(range(a, a + 16))
    if len(seg_starts) == 1:
        Lb = S // P
        blk = oracle.block_tokens(S, P, P - 1, order)
        rng = np.random.default_rng(S)
        keys.update(int(t) for t in rng.choice(blk, 48, replace=False))
        keys.update(range(S - Lb, S - Lb + 8))
    return np.array(sorted(keys), dtype=np.int64)


@pytest.mark.parametrize("name,order", [("llama8b_32k", "contiguous"),
                                        ("packed_128k", "striped")])
def test_backward_full_size(sp, name, order):
    cfg = workloads.CONFIGS[name]
    B, S, Hq, Hkv, d, P = (cfg[x] for x in ("B", "S", "Hq", "Hkv", "d", "P"))
    q, k, v = workloads.qkv_torch(B, S, Hq, Hkv, d, cfg["seed"], torch.bfloat16, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(cfg["seed"] + 7)
    dout = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    pos = workloads.position_ids(cfg)
    tpos = torch.from_numpy(pos).cuda()
    out, lse = sp.blockwise_attention(q, k, v, P, order, tpos)
    dq, dk, dv = sp.blockwise_attention_backward(q, k, v, out, dout, lse, P, order, tpos)
    torch.cuda.synchronize()
    del out, lse

    # sum rules over every key row
    G = Hq // Hkv
    dk64 = dk.double().sum(dim=1)                       # [B][Hkv][d]
    dv64 = dv.double().sum(dim=1)
    do64 = dout.double().sum(dim=1).view(B, Hkv, G, d).sum(dim=2)
    dk_abs = dk.double().abs().sum(dim=1)
    dv_abs = dv.double().abs().sum(dim=1)
    assert (dk64.abs() <= SUM_RULE_TOL * dk_abs).all(), f"{name}: sum of dk is not 0"
    assert ((dv64 - do64).abs() <= SUM_RULE_TOL * dv_abs).all(), f"{name}: sum of dv"

    qn, kn, vn, don = np32(q), np32(k), np32(v), np32(dout)
    rows = workloads.sample_rows(S, P, 128, cfg["seed"] + 3, order)
    got_dq = np32(dq[:, rows])

    def dq_head(h):
        kv = h // G
        return oracle.attention_backward_rows(qn[:, :, h:h + 1], kn[:, :, kv:kv + 1],
                                              vn[:, :, kv:kv + 1], don[:, :, h:h + 1], rows, pos)

    ref_dq = np.concatenate(_pool(dq_head, list(range(Hq))), axis=2)
    e = check_grad(got_dq, ref_dq, "bf16", f"dq {name} {order}")
    print(f"PARITY-GRAD {name} {order} dq max=%.3e mean=%.3e" % e)

    keys = _sampled_keys(pos, S, P, order)
    kvh = 0

    def dkv_head(h):  # one query head of the group, summed below
        return oracle.attention_backward_keys(qn[:, :, h:h + 1], kn[:, :, kvh:kvh + 1],
                                              vn[:, :, kvh:kvh + 1], don[:, :, h:h + 1], keys,
                                              pos)

    parts = _pool(dkv_head, list(range(kvh * G, (kvh + 1) * G)))
    ref_dk = sum(p[0] for p in parts)[:, :, 0]
    ref_dv = sum(p[1] for p in parts)[:, :, 0]
    e = check_grad(np32(dk[:, keys, kvh]), ref_dk, "bf16", f"dk {name} {order}")
    print(f"PARITY-GRAD {name} {order} dk max=%.3e mean=%.3e" % e)
    e = check_grad(np32(dv[:, keys, kvh]), ref_dv, "bf16", f"dv {name} {order}")
    print(f"PARITY-GRAD {name} {order} dv max=%.3e mean=%.3e" % e)
