"""Golden fixtures: the pages' own numbers and oracle regression values.

* ``ep_local_routes.txt`` is the pages' table of local routes per token
  count (AITER #5904 "Add tuned a8w4 fused-MoE configs for DeepSeek
  V4.1-Flash (TP4 + EP, gfx950)", Fused-MoE kernel expert-parallel
  benchmark). Our seeded expert-parallel routing must give the same local
  route density (about 1.5 per token) within sampling noise.
* ``tiny_*.json`` are written by ``tests/golden/make_golden.py`` from the
  oracle alone; they freeze the oracle's arithmetic so any change to it is
  deliberate.
"""
import json
import os

import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe as om
from oracle import mx_formats as mx

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _page_table():
    rows = []
    for line in open(os.path.join(HERE, "ep_local_routes.txt")):
        if line.strip() and not line.startswith("#"):
            t, r = line.split()
            rows.append((int(t), int(r)))
    return rows


@pytest.mark.parametrize("tokens", [1024, 4096, 16384])
def test_ep_routing_local_density_matches_page(tokens):
    page = dict(_page_table())[tokens]
    case_ids, _ = mi.make_routing(mi.SHAPES["ep"], tokens,
                                  mi._gen(mi.call_seed(2, tokens)), "uniform")
    ours = int((case_ids < mi.SHAPES["ep"].E).sum())
    # both counts are random: a route is local with p = 96/384, so each has
    # variance ~ n p (1 - p) with n = 6 * tokens; allow 4 sigma of the difference
    n, p = 6 * tokens, 96 / 384
    sigma_diff = (2 * n * p * (1 - p)) ** 0.5
    assert abs(ours - page) <= 4 * sigma_diff, (ours, page)


@pytest.mark.parametrize("name", ["tiny_a8w4.json", "tiny_a16w4.json"])
def test_oracle_regression_fixture(name):
    ref = json.load(open(os.path.join(HERE, name)))
    shp = mi.small_shape(H=ref["H"], I=ref["I"], Ip=ref["Ip"], E=ref["E"],
                         topk=ref["topk"], a16=ref["a16"])
    case = mi.make_case("small", ref["M"], shape=shp)
    assert case.seed == ref["seed"]
    res = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                       case.w2, case.w2_scale, shp.E, a16=ref["a16"], block_m=ref["block_m"])
    assert res.sort.sorted_route.tolist() == ref["sorted_route"]
    assert res.sort.block_expert.tolist() == ref["block_expert"]
    assert mx.bf16_bits(res.out_bf16).reshape(-1).tolist() == ref["out_bf16_bits"]
