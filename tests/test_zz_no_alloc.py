"""The allocation-free attention entry point.

sp_blockwise_attn_fwd_noalloc serves callers that cannot allocate device
memory (code that must not call cudaMalloc, or whose allocator only hands out
the caller's own tensors): it keeps its workspace in a fixed array with
static storage on the device instead of taking one from the caller.  These
tests call it through the C ABI and check, on two calls in a row (the array
keeps the previous call's contents, which must not leak into the next
result), that it reproduces the ordinary entry point and that both match the
float64 oracle.  Non-causal bf16 calls use the fixed array as the scratch of
the tail split as well, which holds fewer pieces than the workspace the
ordinary entry point is given, so their split schedule differs: the oracle
comparison covers it.  The file name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import BF16_MAX_ABS, BF16_MEAN_ABS, F32_MAX_ABS, LSE_BF16, check_attention, np32
import workloads

pytestmark = pytest.mark.gpu


def _packed_positions(B, S, seed):
    rows = [workloads.position_ids_from_lengths(workloads.doc_lengths(S, 5, seed + b))
            for b in range(B)]
    return torch.from_numpy(np.stack(rows).astype(np.int32)).cuda()


def _compare(got, ref, got_lse, ref_lse, dtype):
    err = np.abs(np32(got).astype(np.float64) - np32(ref))
    if dtype == "bf16":
        assert err.max() <= BF16_MAX_ABS and err.mean() <= BF16_MEAN_ABS
    else:
        assert err.max() <= F32_MAX_ABS
    a, b = got_lse.cpu().numpy(), ref_lse.cpu().numpy()
    assert np.array_equal(np.isfinite(a), np.isfinite(b))
    fin = np.isfinite(b)
    assert np.abs(a[fin] - b[fin]).max() <= LSE_BF16


@pytest.mark.parametrize("case", [
    # (dtype, B, S, Hq, Hkv, d, P, order, causal)
    ("bf16", 1, 2048, 4, 2, 128, 4, "striped", True),
    ("bf16", 2, 1000, 2, 1, 128, 2, "contiguous", False),
    ("bf16", 1, 4096, 8, 8, 128, 4, "contiguous", False),
    ("f32", 1, 96, 2, 1, 32, 3, "contiguous", True),
])
def test_noalloc_matches_workspace_entry_point(case):
    from sequence_parallelism_gb300 import _lib
    import sequence_parallelism_gb300 as sp
    dtype, B, S, Hq, Hkv, d, P, order, causal = case
    for call in range(2):  # two calls in a row, different inputs each time
        q, k, v = workloads.small_case(B, S, Hq, Hkv, d, 900 + 10 * call, dtype)
        pos = _packed_positions(B, S, 50 + call) if causal else None
        ref, ref_lse = sp.blockwise_attention(q, k, v, P, order, pos)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
        _lib.sp_blockwise_attn_fwd_noalloc(q, k, v, pos, P, order, 0.0, out, lse)
        torch.cuda.synchronize()
        _compare(out, ref, lse, ref_lse, dtype)
        o64, l64 = oracle.full_attention(np32(q), np32(k), np32(v),
                                         None if pos is None else pos.cpu().numpy())
        check_attention(np32(out), lse.cpu().numpy(), o64, l64, dtype, f"noalloc {case}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from sequence_parallelism_gb300 import _lib
    lib = _lib._lib
    fake = ctypes.c_void_p(0x100000)
    # causal with 4M tokens needs ~16 MiB of doc_start: more than the array
    st = lib.sp_blockwise_attn_fwd_noalloc(fake, fake, fake, fake, 1, 1 << 22, 8, 8, 128, 1, 0,
                                           0.0, 0, fake, None, None)
    assert st == _lib.SP_ERR_WORKSPACE
    assert lib.sp_last_launch_count() == 0
