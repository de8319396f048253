"""CPU oracle for blockwise (ring) attention and the Ulysses layout permutation.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
constant, table or helper with the CUDA library in
``sequence_parallelism_gb300/``.

Everything here is plain NumPy in float64: slow, and written so that each
function can be checked against the pages by eye.

Sources (web pages, cited by title and section):

* "Ring Attention" (Ultralytics glossary), section "Cómo funciona la atención
  en anillo": the sequence is cut into N blocks; device i keeps query block i
  and at step s works on the key/value block j = (i - s) mod N; the partial
  results are combined by a cumulative softmax (running sum of exponentiated
  scores and running weighted-value sum, divided at the end); production
  kernels also subtract a running maximum; striped attention spreads each
  device's tokens uniformly over the sequence.
* "Ulysses SP: entrenar modelos con millones de tokens" (Keryc), section
  "Cómo funciona Ulysses Sequence Parallelism (SP)": all-to-all from
  sequence shards to "all positions, subset of heads" and back.
* "DeepSpeed-Ulysses" (orangingq blog), section "Method": the redistribution
  (N/P, d) -> (N, d/P) and its inverse.
* "Ulysses SPで100万トークン学習" (aitoolresearcher review), section 3
  ("6ステップ"): causal mask carried by position_ids in O(n) memory instead
  of a 4D mask.

Readings of points the pages leave open:

* causal semantics of position_ids: a document restarts wherever
  position_ids does not continue by +1 (and at token 0); token i may attend
  token j iff both lie in the same document and j <= i;
* GQA: query head h uses key/value head h // (Hq / Hkv);
* striped block p = the tokens t with t mod P == p (stripe width 1);
* head group r of the Ulysses layout = heads r*H/P ... (r+1)*H/P - 1, and the
  head-sharded tensor is laid out [P][B][S][H/P][d];
* a query row with no allowed key has out = 0 and lse = -inf.

attention_backward adds the gradients of that definition (the pages print no
backward formulas; they are the derivatives of the forward);
attention_backward_rows and attention_backward_keys give the same gradients
for sampled query rows (dq) and sampled key rows (dk, dv) at full sequence
lengths.

Parity status: every function here is pinned by ``tests/test_oracle.py`` and
``tests/test_oracle_backward.py`` (worked example of the Ring Attention page,
closed forms, a library routine, float64 autograd, finite differences, brute
force and invariants); none is "parity unpinned".
"""

from .attention import (  # noqa: F401
    allowed_mask,
    attention_backward,
    attention_backward_keys,
    attention_backward_rows,
    attention_rows,
    blockwise_ring_attention,
    block_tokens,
    doc_starts,
    full_attention,
    merge_partials,
    ring_partial,
    ring_partial_backward,
    ring_unstabilised_f32,
    segment_ids,
)
from .permute import head_to_seq, seq_to_head  # noqa: F401
