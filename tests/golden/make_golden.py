"""Writes the oracle regression fixtures in this folder.

Calls only ``oracle/`` and the seeded input generators; run it from the
repository root (``python tests/golden/make_golden.py``) after a change to
the oracle's arithmetic that a cited reading justifies.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import moe_inputs as mi  # noqa: E402
from oracle import moe as om  # noqa: E402
from oracle import mx_formats as mx  # noqa: E402


def tiny_case(a16):
    shp = mi.small_shape(H=128, I=48, Ip=64, E=5, topk=3, a16=a16)
    case = mi.make_case("small", 6, shape=shp)
    res = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                       case.w2, case.w2_scale, shp.E, a16=a16, block_m=4)
    return dict(
        seed=case.seed, M=6, H=128, I=48, Ip=64, E=5, topk=3, block_m=4, a16=a16,
        sorted_route=res.sort.sorted_route.tolist(),
        block_expert=res.sort.block_expert.tolist(),
        out_bf16_bits=mx.bf16_bits(res.out_bf16).reshape(-1).tolist(),
    )


def main():
    for a16 in (False, True):
        name = "tiny_a16w4.json" if a16 else "tiny_a8w4.json"
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(tiny_case(a16), f)


if __name__ == "__main__":
    main()
