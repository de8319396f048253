"""The C ABI without a GPU: the library loads, exports every entry point that
include/sp_gb300.h declares, sizes its workspace, and rejects bad arguments
on the host before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sp_gb300.h")
LIB = os.path.join(ROOT, "sequence_parallelism_gb300", "libsp_gb300.so")

SP_OK, SP_ERR_INVALID_ARG, SP_ERR_UNSUPPORTED, SP_ERR_WORKSPACE = 0, 1, 2, 3
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
FAKE_WS = ctypes.c_void_p(0x20000)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    from sequence_parallelism_gb300 import _lib
    return _lib._lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sp_ulysses_seq_to_head", "sp_ulysses_head_to_seq", "sp_blockwise_attn_fwd",
              "sp_attn_merge_partials", "sp_blockwise_attn_step", "sp_segment_starts"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_export(lib):
    from sequence_parallelism_gb300 import _lib
    assert set(_lib.EXPORTS) == set(declared_functions())


def test_status_strings(lib):
    for s in range(6):
        assert lib.sp_status_string(s).decode().startswith("SP_")


def test_workspace_sizes(lib):
    assert lib.sp_blockwise_attn_workspace_bytes(1, 4096, 0) == 256
    n = lib.sp_blockwise_attn_workspace_bytes(2, 1000, 1)
    assert n >= 256 + 2 * 1000 * 4 and n % 256 == 0
    assert lib.sp_blockwise_attn_workspace_bytes(0, 10, 1) == 0
    assert lib.sp_segment_starts_workspace_bytes(1, 524288) >= 512 * 4


def _permute(lib, fn, x, y, B, S, H, d, P, dt=0):
    return getattr(lib, fn)(x, y, B, S, H, d, P, dt, None)


@pytest.mark.parametrize("fn", ["sp_ulysses_seq_to_head", "sp_ulysses_head_to_seq"])
def test_permute_rejects_bad_arguments(lib, fn):
    assert _permute(lib, fn, None, FAKE, 1, 8, 4, 16, 2) == SP_ERR_INVALID_ARG
    assert _permute(lib, fn, FAKE, None, 1, 8, 4, 16, 2) == SP_ERR_INVALID_ARG
    assert _permute(lib, fn, FAKE, FAKE, 1, 9, 4, 16, 2) == SP_ERR_INVALID_ARG   # S % P
    assert _permute(lib, fn, FAKE, FAKE, 1, 8, 6, 16, 4) == SP_ERR_INVALID_ARG   # H % P
    assert _permute(lib, fn, FAKE, FAKE, 0, 8, 4, 16, 2) == SP_ERR_INVALID_ARG
    assert _permute(lib, fn, FAKE, FAKE, 1, 8, 4, 16, 0) == SP_ERR_INVALID_ARG
    assert _permute(lib, fn, FAKE, FAKE, 1, 8, 4, 16, 2, dt=7) == SP_ERR_INVALID_ARG
    assert lib.sp_last_launch_count() == 0


def _attn(lib, q=FAKE, k=FAKE, v=FAKE, pos=None, B=1, S=256, Hq=4, Hkv=2, d=128, P=2, order=0,
          scale=0.0, dt=0, out=FAKE, ws=FAKE_WS, wsb=1 << 20, step=None):
    if step is None:
        return lib.sp_blockwise_attn_fwd(q, k, v, pos, B, S, Hq, Hkv, d, P, order, scale, dt, out,
                                         None, ws, wsb, None)
    return lib.sp_blockwise_attn_step(q, k, v, pos, B, S, Hq, Hkv, d, P, order, step, scale, dt,
                                      out, None, ws, wsb, None)


def test_attention_rejects_bad_arguments(lib):
    assert _attn(lib, q=None) == SP_ERR_INVALID_ARG
    assert _attn(lib, out=None) == SP_ERR_INVALID_ARG
    assert _attn(lib, S=255) == SP_ERR_INVALID_ARG            # S % P
    assert _attn(lib, Hq=6, Hkv=4) == SP_ERR_INVALID_ARG      # Hq % Hkv
    assert _attn(lib, order=2) == SP_ERR_INVALID_ARG
    assert _attn(lib, dt=5) == SP_ERR_INVALID_ARG
    assert _attn(lib, P=0) == SP_ERR_INVALID_ARG
    assert _attn(lib, S=0) == SP_ERR_INVALID_ARG              # empty sequence
    assert _attn(lib, B=0) == SP_ERR_INVALID_ARG              # empty batch
    assert _attn(lib, Hq=0, Hkv=0) == SP_ERR_INVALID_ARG      # no heads
    assert _attn(lib, scale=float("nan")) == SP_ERR_INVALID_ARG
    assert _attn(lib, d=64) == SP_ERR_UNSUPPORTED              # bf16 needs d == 128
    assert _attn(lib, d=512, dt=1) == SP_ERR_UNSUPPORTED       # f32 d <= 256
    assert _attn(lib, q=ctypes.c_void_p(0x10008)) == SP_ERR_INVALID_ARG  # TMA alignment
    assert _attn(lib, ws=None) == SP_ERR_WORKSPACE
    assert _attn(lib, ws=ctypes.c_void_p(0x20010)) == SP_ERR_WORKSPACE  # 256-byte alignment
    assert _attn(lib, pos=FAKE, wsb=256) == SP_ERR_WORKSPACE           # causal needs doc_start
    assert _attn(lib, step=2) == SP_ERR_INVALID_ARG
    assert _attn(lib, step=-1) == SP_ERR_INVALID_ARG
    assert lib.sp_last_launch_count() == 0


def test_merge_and_segments_reject_bad_arguments(lib):
    m = lib.sp_attn_merge_partials
    assert m(None, FAKE, 2, 1, 8, 2, 16, 0, FAKE, None, None) == SP_ERR_INVALID_ARG
    assert m(FAKE, FAKE, 0, 1, 8, 2, 16, 0, FAKE, None, None) == SP_ERR_INVALID_ARG
    assert m(FAKE, FAKE, 2, 1, 8, 2, 16, 9, FAKE, None, None) == SP_ERR_INVALID_ARG
    s = lib.sp_segment_starts
    assert s(None, FAKE, 1, 8, FAKE_WS, 1 << 12, None) == SP_ERR_INVALID_ARG
    assert s(FAKE, FAKE, 1, 8, None, 1 << 12, None) == SP_ERR_WORKSPACE
    assert s(FAKE, FAKE, 1, 8, FAKE_WS, 0, None) == SP_ERR_WORKSPACE
    assert lib.sp_get_device_error(None, None, None) == SP_ERR_INVALID_ARG


def test_hybrid_rejects_bad_arguments(lib):
    f = lib.sp_ulysses_ring_attn_fwd
    ws = lib.sp_ulysses_ring_attn_workspace_bytes(1, 64, 8, 8, 128, 0, 0)
    assert ws >= 4 * 64 * 8 * 128 * 2
    args = lambda **kw: dict(dict(q=FAKE, k=FAKE, v=FAKE, pos=None, B=1, S=64, Hq=8, Hkv=8, d=128,
                                  Pu=4, Pr=2, order=0, scale=0.0, dt=0, out=FAKE, ws=FAKE_WS,
                                  wsb=1 << 30), **kw)
    call = lambda a: f(a["q"], a["k"], a["v"], a["pos"], a["B"], a["S"], a["Hq"], a["Hkv"], a["d"],
                       a["Pu"], a["Pr"], a["order"], a["scale"], a["dt"], a["out"], None, a["ws"],
                       a["wsb"], None)
    assert call(args(q=None)) == SP_ERR_INVALID_ARG
    assert call(args(Hkv=2, Pu=4)) == SP_ERR_INVALID_ARG     # Hkv % P_u
    assert call(args(S=66, Pr=4)) == SP_ERR_INVALID_ARG      # S % P_r
    assert call(args(Pu=0)) == SP_ERR_INVALID_ARG
    assert call(args(wsb=1024)) == SP_ERR_WORKSPACE
    assert lib.sp_last_launch_count() == 0


def test_qkv_permutation_rejects_bad_arguments(lib):
    f = lib.sp_ulysses_seq_to_head_qkv
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 8, 6, 16, 4, 0, None) == SP_ERR_INVALID_ARG
    assert f(FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 8, 8, 4, 16, 4, 0, None) == SP_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 9, 8, 4, 16, 4, 0, None) == SP_ERR_INVALID_ARG
    assert lib.sp_last_launch_count() == 0


def test_barrier_check_rejects_bad_arguments(lib):
    f = lib.sp_check_barrier_timeout
    assert f(None, 1000, None) == SP_ERR_WORKSPACE
    assert f(ctypes.c_void_p(0x20010), 1000, None) == SP_ERR_WORKSPACE
    assert f(FAKE_WS, 0, None) == SP_ERR_INVALID_ARG
    assert f(FAKE_WS, 2000000, None) == SP_ERR_INVALID_ARG


def test_per_device_entry_points_reject_bad_arguments(lib):
    """sp_ring_block_step / sp_query_block_attn_fwd: block indices outside
    0 .. P-1, indivisible sizes and missing pointers fail on the host."""
    f32 = ctypes.c_float
    ring = lambda i, j, S=1024, P=4, q=FAKE: lib.sp_ring_block_step(
        q, FAKE, FAKE, None, 1, S, 2, 1, 128, P, 0, i, j, f32(0.0), 0, FAKE, None, FAKE_WS,
        ctypes.c_size_t(1 << 20), None)
    for i, j in ((4, 0), (0, 4), (-1, 0), (0, -1)):
        assert ring(i, j) == SP_ERR_INVALID_ARG
    assert ring(0, 0, S=1023) == SP_ERR_INVALID_ARG     # S % P
    assert ring(0, 0, P=0) == SP_ERR_INVALID_ARG
    assert ring(0, 0, q=None) == SP_ERR_INVALID_ARG
    qb = lambda i, P=4: lib.sp_query_block_attn_fwd(
        FAKE, FAKE, FAKE, None, 1, 1024, 2, 1, 128, P, 0, i, f32(0.0), 0, FAKE, None, FAKE_WS,
        ctypes.c_size_t(1 << 20), None)
    assert qb(4) == SP_ERR_INVALID_ARG and qb(-1) == SP_ERR_INVALID_ARG and qb(0, P=0) == \
        SP_ERR_INVALID_ARG
    assert lib.sp_last_launch_count() == 0


def test_accumulating_step_arguments(lib):
    """sp_ring_block_step_accumulate: the per-device checks, plus a required
    running lse and bf16 only; a contiguous causal pair with j > i adds
    nothing and returns SP_OK without a launch (checked here on pointers the
    call must not touch)."""
    f32 = ctypes.c_float
    acc = lambda i, j, dtype=0, lse=FAKE, pos=None, order=0, P=4: \
        lib.sp_ring_block_step_accumulate(
            FAKE, FAKE, FAKE, pos, 1, 1024, 2, 1, 128, P, order, i, j, f32(0.0), dtype, FAKE, lse,
            FAKE_WS, ctypes.c_size_t(1 << 20), None)
    for i, j in ((4, 0), (0, 4), (-1, 0), (0, -1)):
        assert acc(i, j) == SP_ERR_INVALID_ARG
    assert acc(1, 0, lse=None) == SP_ERR_INVALID_ARG
    assert acc(1, 0, dtype=1) == SP_ERR_UNSUPPORTED
    assert acc(0, 1, pos=FAKE) == SP_OK
    assert lib.sp_last_launch_count() == 0


def test_ring_step_backward_skips_pairs_without_allowed_keys(lib):
    """sp_ring_block_step_bwd: a contiguous causal pair with j > i returns
    SP_OK without a launch and without touching the (fake) tensors; block
    indices are still validated first."""
    f32 = ctypes.c_float
    bwd = lambda i, j, pos, order=0: lib.sp_ring_block_step_bwd(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, pos, 1, 1024, 2, 1, 128, 4, order, i, j, f32(0.0), 0,
        FAKE, FAKE, FAKE, FAKE_WS, ctypes.c_size_t(1 << 30), None)
    assert bwd(0, 1, FAKE) == SP_OK and bwd(2, 3, FAKE) == SP_OK
    assert lib.sp_last_launch_count() == 0
    assert bwd(0, 4, FAKE) == SP_ERR_INVALID_ARG


def test_permutation_threshold_setting_round_trips(lib):
    lib.sp_permute_set_bulk_min_bytes.restype = ctypes.c_size_t
    lib.sp_permute_set_bulk_min_bytes.argtypes = [ctypes.c_size_t]
    prev = lib.sp_permute_set_bulk_min_bytes(12345)
    assert lib.sp_permute_set_bulk_min_bytes(prev) == 12345


def test_backward_dq_form_setting_round_trips(lib):
    lib.sp_set_bwd_dq_reduction.restype = ctypes.c_int
    lib.sp_set_bwd_dq_reduction.argtypes = [ctypes.c_int]
    prev = lib.sp_set_bwd_dq_reduction(0)
    assert prev == 1                              # dQ by reductions is the default
    assert lib.sp_set_bwd_dq_reduction(7) == 0    # any non-zero value means on
    assert lib.sp_set_bwd_dq_reduction(prev) == 1


def test_backward_workspace_holds_the_dq_accumulator(lib):
    """The backward workspace includes the float32 dQ accumulator: B * Hq * P
    * Lbp * 128 floats, Lbp = S/P rounded up to a multiple of 128."""
    lib.sp_blockwise_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.sp_blockwise_attn_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 5
    for B, S, Hq, P, causal in [(1, 32768, 32, 8, 1), (2, 1000, 4, 2, 0), (1, 1416, 4, 3, 1)]:
        Lbp = -(-(S // P) // 128) * 128
        acc = B * Hq * P * Lbp * 128 * 4
        assert lib.sp_blockwise_attn_bwd_workspace_bytes(B, S, Hq, P, causal) >= acc
    assert lib.sp_blockwise_attn_bwd_workspace_bytes(1, 1000, 4, 3, 0) == 0   # S % P != 0
