"""Write tests/golden/smallhead_ctx16.json: a small regression fixture for the oracle.

Shape: 4 query heads / 2 KV heads, head_dim 8 -- the hidden=32 / headDim=8
fixture of dotLLM issue #199 ("perf(cuda): tensor-core (mma.sync FP16) decode
attention kernel", §0), here with 16 cached rows. The inputs are stored in the
file (f32 q as decimal strings, f16 K/V as bit patterns) and the expected
output comes from the oracle alone; no value here comes from the CUDA path.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def main():
    rng = np.random.Generator(np.random.PCG64([5, 16]))
    n_head, n_kv, hd, cap = 4, 2, 8, 16
    q = rng.standard_normal((1, n_head, hd), dtype=np.float32)
    k = rng.standard_normal((1, cap, n_kv, hd), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((1, cap, n_kv, hd), dtype=np.float32).astype(np.float16)
    positions = np.array([cap - 1], np.int32)
    scale = 1.0 / math.sqrt(hd)
    o = oracle.attn_decode(q, k, v, positions, n_head, n_kv, hd, cap, scale)
    doc = {
        "what": "oracle output for a 4/2-head, head_dim 8, 16-row decode (regression pin)",
        "shape": {"n_seq": 1, "n_head": n_head, "n_kv_head": n_kv, "head_dim": hd, "cap": cap},
        "scale": scale,
        "positions": positions.tolist(),
        "q_f32": [repr(float(x)) for x in q.ravel()],
        "k_f16_bits": k.view(np.uint16).ravel().tolist(),
        "v_f16_bits": v.view(np.uint16).ravel().tolist(),
        "o_f64": [repr(float(x)) for x in o.ravel()],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "smallhead_ctx16.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
