"""GPU parity of the Ulysses permutation and of doc_start: bit-exact against
the oracle's index loops / segment reading, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
from helpers import npi
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


@pytest.fixture(params=["tma_staged", "default"])
def path(request):
    """Runs a test twice: with every launch that meets the bulk-copy rules on
    the TMA-staged kernel, and with the default size threshold (small
    launches on the vector kernel, large ones on the TMA-staged kernel)."""
    from sequence_parallelism_gb300 import _lib
    prev = _lib.sp_permute_set_bulk_min_bytes(0 if request.param == "tma_staged" else 128 << 20)
    yield request.param
    _lib.sp_permute_set_bulk_min_bytes(prev)


def _rand_tensor(shape, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if dtype == torch.bfloat16 or dtype == torch.float32:
        return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(dtype)
    raise ValueError(dtype)


@pytest.mark.parametrize("B,S,H,d,P,dtype", [
    (1, 64, 8, 128, 4, torch.bfloat16),     # 512 B chunks: TMA-staged path
    (2, 42, 6, 16, 3, torch.float32),       # 128 B chunks: vector path
    (1, 12, 4, 3, 2, torch.bfloat16),       # 2-byte chunks: scalar path
    (1, 10, 5, 7, 5, torch.float32),        # one head per group, 4-byte path
    (3, 16, 16, 64, 1, torch.bfloat16),     # P = 1: plain reshape (2 KiB chunks)
    (1, 32, 16, 128, 16, torch.bfloat16),   # P = H: 256 B chunks, the bulk minimum
    (1, 1000, 8, 128, 4, torch.bfloat16),   # items straddle head groups; partial last item
    (2, 300, 64, 128, 2, torch.bfloat16),   # 8 KiB chunks: one chunk per item
    (1, 513, 12, 32, 3, torch.float32),     # odd row count, fp32 512 B chunks
    (1, 64, 64, 128, 1, torch.bfloat16),    # 16 KiB chunks: above a stage, vector path
    (1, 2048, 32, 128, 8, torch.bfloat16),  # more items than CTAs, several ring laps
    (1, 99, 12, 40, 3, torch.bfloat16),     # 320 B chunks: box rows of 320 B
])
def test_permutation_bit_exact(sp, path, B, S, H, d, P, dtype):
    x = _rand_tensor((B, S, H, d), dtype, 11 + P)
    y = sp.seq_to_head(x, P)
    torch.cuda.synchronize()
    bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
    ref = oracle.seq_to_head(npi(x.view(bits)), P)
    assert np.array_equal(npi(y.view(bits)), ref)
    back = sp.head_to_seq(y)
    torch.cuda.synchronize()
    assert torch.equal(back.view(bits), x.view(bits))
    assert np.array_equal(npi(back.view(bits)), oracle.head_to_seq(ref))


@pytest.mark.parametrize("shift", [(8, 0), (0, 8)])
def test_permutation_unaligned_pointers(sp, path, shift):
    """A source or destination that is not 16-byte aligned (8 bytes off)
    takes the vector path: still bit-exact both ways."""
    from sequence_parallelism_gb300 import _lib
    B, S, H, d, P = 1, 96, 8, 128, 4
    n = B * S * H * d
    xs, ys = shift[0] // 2, shift[1] // 2  # in bf16 elements
    xbuf = _rand_tensor((n + 16,), torch.bfloat16, 71)
    ybuf = torch.zeros(n + 16, dtype=torch.bfloat16, device="cuda")
    x = xbuf[xs:xs + n].view(B, S, H, d)
    y = ybuf[ys:ys + n].view(P, B, S, H // P, d)
    _lib.sp_ulysses_seq_to_head(x, y, P)
    torch.cuda.synchronize()
    ref = oracle.seq_to_head(npi(x.view(torch.int16)), P)
    assert np.array_equal(npi(y.view(torch.int16)), ref)
    back = torch.zeros_like(xbuf)[xs:xs + n].view(B, S, H, d)
    _lib.sp_ulysses_head_to_seq(y, back, P)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    assert _lib.sp_get_permute_error() == (0, 0)


def test_permutation_full_size_ulysses(sp, path):
    """ulysses_4k: q, k, v [1][4096][32][128] bf16, P = 4."""
    cfg = workloads.CONFIGS["ulysses_4k"]
    q, k, v = workloads.qkv_torch(cfg["B"], cfg["S"], cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["seed"],
                                  torch.bfloat16, "cuda")
    for t in (q, k, v):
        y = sp.seq_to_head(t, cfg["P"])
        torch.cuda.synchronize()
        assert np.array_equal(npi(y.view(torch.int16)),
                              oracle.seq_to_head(npi(t.view(torch.int16)), cfg["P"]))
        assert torch.equal(sp.head_to_seq(y).view(torch.int16), t.view(torch.int16))


def test_permutation_large_tensor_roundtrip(sp, path):
    """A 256 MiB tensor (the llama8b_32k q shape) round-trips bit-exactly and
    lands in the head-sharded slots the index formula names (both directions
    take the TMA-staged kernel under either threshold)."""
    x = _rand_tensor((1, 32768, 32, 128), torch.bfloat16, 5)
    y = sp.seq_to_head(x, 8)
    back = sp.head_to_seq(y)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    rng = np.random.default_rng(3)
    for _ in range(64):
        r, t, hl = int(rng.integers(8)), int(rng.integers(32768)), int(rng.integers(4))
        assert torch.equal(y[r, 0, t, hl].view(torch.int16), x[0, t, r * 4 + hl].view(torch.int16))


def _doc_start_ref(pos):
    return oracle.doc_starts(pos).astype(np.int32)


@pytest.mark.parametrize("lengths", [[1], [5, 1, 7], [1023, 1, 1025, 2047], [3000, 1, 1, 96]])
def test_doc_start_bit_exact(sp, lengths):
    pos = np.stack([workloads.position_ids_from_lengths(lengths),
                    workloads.position_ids_from_lengths(lengths[::-1])])
    ds = sp.doc_starts(torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(npi(ds), _doc_start_ref(pos))


def test_doc_start_irregular_positions(sp):
    rng = np.random.default_rng(9)
    pos = rng.integers(0, 5, size=(3, 5000)).astype(np.int32)  # many restarts and repeats
    pos[1] = np.arange(5000, dtype=np.int32) + 17               # one doc not starting at 0
    ds = sp.doc_starts(torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(npi(ds), _doc_start_ref(pos))


@pytest.mark.parametrize("name", ["packed_128k", "halfmil_512k"])
def test_doc_start_full_size(sp, name):
    cfg = workloads.CONFIGS[name]
    pos = workloads.position_ids(cfg)
    ds = sp.doc_starts(torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(npi(ds), _doc_start_ref(pos))


@pytest.mark.parametrize("B,S,Hq,Hkv,d,P,dtype", [
    (1, 4096, 32, 8, 128, 4, torch.bfloat16),   # GQA shapes, TMA-staged path
    (1, 96, 16, 2, 128, 2, torch.bfloat16),     # k/v chunks of 256 B (bulk minimum)
    (1, 64, 16, 4, 64, 4, torch.bfloat16),      # k/v chunks of 128 B: vector path for all
    (2, 24, 6, 3, 4, 3, torch.bfloat16),        # 8-byte chunks
    (1, 10, 4, 2, 3, 2, torch.float32),         # 12-byte chunks: 4-byte path
])
def test_qkv_permutation_one_launch_bit_exact(sp, path, B, S, Hq, Hkv, d, P, dtype):
    from sequence_parallelism_gb300 import _lib
    q = _rand_tensor((B, S, Hq, d), dtype, 31)
    k = _rand_tensor((B, S, Hkv, d), dtype, 32)
    v = _rand_tensor((B, S, Hkv, d), dtype, 33)
    yq = torch.empty((P, B, S, Hq // P, d), dtype=dtype, device="cuda")
    yk = torch.empty((P, B, S, Hkv // P, d), dtype=dtype, device="cuda")
    yv = torch.empty_like(yk)
    _lib.sp_ulysses_seq_to_head_qkv(q, k, v, yq, yk, yv, P)
    assert _lib.sp_last_launch_count() == 1
    torch.cuda.synchronize()
    bits = torch.int16 if dtype == torch.bfloat16 else torch.int32
    for x, y in ((q, yq), (k, yk), (v, yv)):
        assert np.array_equal(npi(y.view(bits)), oracle.seq_to_head(npi(x.view(bits)), P))
    assert _lib.sp_get_permute_error() == (0, 0)
