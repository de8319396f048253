"""The full-size oracle harness (tests/fullsize_oracle.py) on the CPU.

It evaluates the oracle in pieces -- one query head, a run of rows, and for
causal attention only the rows' own document -- in spawned worker
processes.  That decomposition rests on one property of the definition: a
query row sees only the keys of its own document, so the documents are
independent problems.  Here the harness's assembled result, with pieces
forced small, must equal the whole-sequence oracle on packed documents, GQA,
sampled rows and a head subset, to 1e-12 (the same float64 arithmetic on the
same rows; only the summation order inside the matrix products differs)."""

import numpy as np
import pytest

import oracle
import workloads
from fullsize_oracle import FullSizeOracle, rotating_heads


@pytest.fixture(scope="module")
def pool():
    p = FullSizeOracle(workers=2, min_piece=64)
    yield p
    p.close()


def _case(S, Hq, Hkv, d, seed, n_docs):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, S, Hq, d)).astype(np.float32)
    k = rng.standard_normal((1, S, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((1, S, Hkv, d)).astype(np.float32)
    pos = None
    if n_docs:
        pos = workloads.position_ids_from_lengths(workloads.doc_lengths(S, n_docs, seed))[None]
    return q, k, v, pos


@pytest.mark.parametrize("n_docs,rows,heads", [
    (0, None, None),                    # non-causal, every row and head
    (1, None, None),                    # one causal document
    (5, None, None),                    # packed documents
    (5, "sampled", None),               # packed, sampled rows
    (6, None, "rotating"),              # packed, one head per key/value group
])
def test_pieces_equal_whole_sequence_oracle(pool, n_docs, rows, heads):
    S, Hq, Hkv, d = 300, 8, 2, 16
    q, k, v, pos = _case(S, Hq, Hkv, d, 11 + n_docs, n_docs)
    sel = workloads.sample_rows(S, 4, 40, 5, "striped") if rows == "sampled" else None
    hs = rotating_heads(Hq, Hkv) if heads == "rotating" else None
    name = f"cpu_{n_docs}_{rows}_{heads}"
    pool.submit_arrays(name, q, k, v, pos, sel, hs)
    got_rows, got_heads, out, lse = pool.result(name, timeout=600)
    assert len(pool.requests[name]["jobs"]) == 0
    ref_out, ref_lse = oracle.attention_rows(q, k, v, sel, pos)
    hs = list(range(Hq)) if hs is None else hs
    assert list(got_heads) == hs
    np.testing.assert_array_equal(got_rows, np.arange(S) if sel is None else sel)
    np.testing.assert_allclose(out, ref_out[:, :, hs], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse[:, hs], rtol=0, atol=1e-12)


def test_rotating_heads_cover_every_group_and_position():
    hs = rotating_heads(32, 8)
    assert [h // 4 for h in hs] == list(range(8))
    assert sorted({h % 4 for h in hs}) == [0, 1, 2, 3]


def test_bf16_inputs_travel_exactly(pool):
    """bf16 tensors are stored as bit patterns and widened in the worker:
    the result equals the oracle on the float32 values of the same tensors."""
    import torch
    g = torch.Generator().manual_seed(3)
    q = torch.randn((1, 200, 4, 32), generator=g).to(torch.bfloat16)
    k = torch.randn((1, 200, 2, 32), generator=g).to(torch.bfloat16)
    v = torch.randn((1, 200, 2, 32), generator=g).to(torch.bfloat16)
    pos = workloads.position_ids_from_lengths(workloads.doc_lengths(200, 3, 9))[None]
    pool.submit_arrays("cpu_bf16", q, k, v, pos)
    _, _, out, lse = pool.result("cpu_bf16", timeout=600)
    f = lambda t: t.float().numpy()
    ref_out, ref_lse = oracle.attention_rows(f(q), f(k), f(v), None, pos)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n_docs", [1, 4])
def test_backward_pieces_equal_whole_gqa_oracle(pool, n_docs):
    """dq per query head, and dk/dv per query head summed over each GQA
    group, equal the oracle's whole-tensor attention_backward_rows / _keys."""
    S, Hq, Hkv, d = 160, 4, 2, 16
    q, k, v, pos = _case(S, Hq, Hkv, d, 31 + n_docs, n_docs)
    dout = np.random.default_rng(5).standard_normal(q.shape).astype(np.float32)
    rows = workloads.sample_rows(S, 4, 24, 3, "contiguous")
    keys = np.array([0, 5, 77, 100, 159])
    name = f"cpu_bwd_{n_docs}"
    pool.submit_backward_arrays(name, q, k, v, dout, pos, rows, keys)
    got_rows, dq, got_keys, dk, dv = pool.backward_result(name, timeout=600)
    ref_dq = oracle.attention_backward_rows(q, k, v, dout, rows, pos)
    ref_dk, ref_dv = oracle.attention_backward_keys(q, k, v, dout, keys, pos)
    np.testing.assert_array_equal(got_rows, rows)
    np.testing.assert_array_equal(got_keys, keys)
    np.testing.assert_allclose(dq, ref_dq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, ref_dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, ref_dv, rtol=0, atol=1e-12)
