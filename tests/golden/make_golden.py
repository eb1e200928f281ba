"""Write the oracle regression fixtures in this folder.

Calls only ``oracle/`` (and the seeded input generator); run from the
repository root with ``python tests/golden/make_golden.py``.
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads import synthetic as syn  # noqa: E402


def fixture(content_bits):
    lay = oracle.Layout(content_bits, 4)
    w = syn.custom(f"golden_c{content_bits}", [150], heads=2, content_bits=content_bits, seed=11)
    table, npages = syn.make_paging(w)
    ckv, kr = syn.sequence_tokens(w, 0)
    L = int(syn.sequence_lengths(w)[0])
    model = oracle.PagedCacheModel(lay, npages, table)
    model.write(np.zeros(L, int), np.arange(L), ckv, kr, [L])
    q = syn.queries(w, 0)[0]
    out, lse = oracle.mla_decode_fp64(q, model.effective_keys(0, L), w.softmax_scale)
    return {
        "workload": {"lengths": [L], "heads": 2, "content_bits": content_bits, "seed": 11},
        "token_bytes_hex": {str(t): model.token_bytes(0, t).hex() for t in (0, 4, 17, 21, 149)},
        "out_first_channels": out[:, :8].tolist(),
        "out_checksum": float(out.sum()),
        "lse": lse.tolist(),
    }


if __name__ == "__main__":
    for bits in (4, 2):
        with open(os.path.join(HERE, f"oracle_c{bits}r4_L150.json"), "w") as f:
            json.dump(fixture(bits), f, indent=1)
