"""Writes ring_tiny_seed0.json: the Ring Attention page's worked example.

Source: "Ring Attention" (Ultralytics glossary), section "Cómo funciona la
atención en anillo".  The page seeds torch with 0, draws q, k, v together as
one standard-normal tensor of shape (3, 32, 16) (4 devices x block 8, d 16)
and reports that the blockwise result matches full softmax attention within
atol 1e-5 ("True"), each device only ever holding an 8 x 8 score block of the
32 x 32 matrix.

The inputs are frozen here because torch's CPU generator is the only source of
those exact numbers; the expected output is computed by the oracle (float64)
and by nothing else.  Run from the repository root:

    python tests/golden/make_ring_tiny.py
"""

import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def main():
    torch.manual_seed(0)
    qkv = torch.randn(3, 32, 16)  # the page's draw: n_devices * block = 32, dim = 16
    q, k, v = (qkv[i].numpy().astype(np.float32) for i in range(3))
    as4 = lambda a: a.astype(np.float64)[None, :, None, :]  # [B=1][S][H=1][d]
    out, lse = oracle.full_attention(as4(q), as4(k), as4(v))
    doc = {
        "source": "Ring Attention (Ultralytics glossary), section 'Cómo funciona la atención en anillo'",
        "recipe": "torch.manual_seed(0); q, k, v = torch.randn(3, 32, 16)",
        "page_facts": {
            "n_devices": 4, "block": 8, "dim": 16,
            "score_block": [8, 8], "full_matrix": [32, 32],
            "allclose_atol": 1e-5, "matches_full_attention": True,
        },
        "q": [[float(x) for x in row] for row in q],
        "k": [[float(x) for x in row] for row in k],
        "v": [[float(x) for x in row] for row in v],
        "expected_out_oracle_f64": [[repr(float(x)) for x in row] for row in out[0, :, 0, :]],
        "expected_lse_oracle_f64": [repr(float(x)) for x in lse[0, 0, :]],
    }
    # one matrix row per line keeps the fixture diff-able
    lines = ["{"]
    items = list(doc.items())
    for n, (key, val) in enumerate(items):
        sep = "," if n + 1 < len(items) else ""
        if isinstance(val, list) and val and isinstance(val[0], list):
            rows = ",\n  ".join(json.dumps(r) for r in val)
            lines.append(f"{json.dumps(key)}: [\n  {rows}]{sep}")
        else:
            lines.append(f"{json.dumps(key)}: {json.dumps(val, ensure_ascii=False)}{sep}")
    lines.append("}")
    with open(os.path.join(HERE, "ring_tiny_seed0.json"), "w", encoding="utf-8") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
