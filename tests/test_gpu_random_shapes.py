"""A seeded random sweep of shapes against the float64 oracle: batch size,
number of ring blocks P (1 to 16), rows per block (ragged, from 1 up), GQA
ratio, head size (f32), block order and mask kind (none, causal, packed
documents) drawn together, so that combinations the hand-picked cases miss
are exercised too.  The draws are fixed by the seed; each case prints its
shape when it fails."""

import numpy as np
import pytest

from test_gpu_attention import _run
from test_gpu_backward import _run_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import sequence_parallelism_gb300 as m
    return m


def _draw(rng, dtype, max_tokens):
    P = int(rng.integers(1, 17))
    Lb = int(rng.integers(1, max(2, max_tokens // P)))
    S = P * Lb
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    d = 128 if dtype == "bf16" else int(rng.choice([16, 40, 64, 128, 200]))
    order = str(rng.choice(["contiguous", "striped"]))
    # packed documents need at least seven tokens to cut
    pos = str(rng.choice(["none", "causal", "packed"] if S >= 8 else ["none", "causal"]))
    return B, S, Hq, Hkv, d, P, order, pos


def _cases(seed, dtype, n, max_tokens):
    rng = np.random.default_rng(seed)
    return [_draw(rng, dtype, max_tokens) for _ in range(n)]


def _id(case):
    B, S, Hq, Hkv, d, P, order, pos = case
    return f"B{B}-S{S}-H{Hq}x{Hkv}-d{d}-P{P}-{order}-{pos}"


@pytest.mark.parametrize("case", _cases(2024, "bf16", 40, 2400), ids=_id)
def test_random_bf16_forward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run(sp, "bf16", B, S, Hq, Hkv, d, P, order, pos, 1300 + S)


@pytest.mark.parametrize("case", _cases(2025, "f32", 20, 300), ids=_id)
def test_random_f32_forward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run(sp, "f32", B, S, Hq, Hkv, d, P, order, pos, 1400 + S)


@pytest.mark.parametrize("case", _cases(2026, "bf16", 12, 700), ids=_id)
def test_random_bf16_backward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run_bwd(sp, "bf16", B, S, Hq, Hkv, d, P, order, pos, 1500 + S)


@pytest.mark.parametrize("case", _cases(2027, "f32", 10, 160), ids=_id)
def test_random_f32_backward(sp, case):
    B, S, Hq, Hkv, d, P, order, pos = case
    _run_bwd(sp, "f32", B, S, Hq, Hkv, d, P, order, pos, 1600 + S)
