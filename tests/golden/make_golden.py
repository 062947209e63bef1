"""Write the oracle regression fixture for the tiny decode workload.

Calls only ``oracle/`` (and the seeded input generator). The pages print no
worked example with numbers, so the stored values are the oracle's own on the
seeded tiny workload (1 sequence, 4 query heads over 1 kv head, depth 64, 256
keys in four 64-row pages, scale 1/8, seed 0); the fixture guards the oracle
against unnoticed drift. Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from split_paged_decode_gb300.workloads import WORKLOADS, bf16_bits, generate  # noqa: E402


def main():
    inp = generate(WORKLOADS["tiny"])
    out, lse = oracle.decode(bf16_bits(inp.q), bf16_bits(inp.k_pages), bf16_bits(inp.v_pages),
                             inp.page_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    doc = {
        "what": "fp64 oracle output on the seeded tiny decode workload (regression fixture)",
        "workload": "tiny: B1 T1 Hq4 Hkv1 D64 L256 PS64 identity pages, scale 1/8, seed 0",
        "written_by": "tests/golden/make_golden.py (oracle only)",
        "out": out.reshape(4, 64).tolist(),
        "lse": lse.reshape(4).tolist(),
    }
    path = os.path.join(ROOT, "tests", "golden", "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
