"""Changed-input CUDA-graph replay and input preservation.

The validation of AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE
tuning" (Validation and limits) runs eager and changed-input graph checks:
original, changed-input, concentrated-routing and restored-input cases, and
checks that the inputs are preserved. The library reads everything
data-dependent (expert counts, the padded route count, the tile schedule)
on the device, and its launch shapes depend only on M, H, Ip, E and topk, so
one captured call must give the right answer for any routing of the same
shape. Here one call is captured once; x, topk_ids and topk_weights are
overwritten in place with other inputs (other tokens and uniform routing,
then 80 % of the routes on a few hot experts, then every token on the same
experts), the graph is replayed and each result is compared with a fresh
oracle run; finally the original inputs are restored and replayed. Every
input buffer (activations, routing, prepacked weights and scales) must be
bit-identical before and after the calls. The graph is destroyed before the
buffers it uses are freed.
"""
import numpy as np
import pytest
import torch

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from moe_check import check_outputs, layer_for, sample_tokens, weights_for

pytestmark = pytest.mark.gpu


def _same_experts(case, experts):
    """Every token routed to the same `experts` (k of them), with the case's
    routing weights."""
    ids = torch.tensor(experts, dtype=torch.int32).expand(case.M, len(experts)).contiguous()
    return mi.MoeCase(case.shape, case.M, case.x, ids, case.topk_weights, case.w1,
                      case.w1_scale, case.w2, case.w2_scale, case.seed)


def _concentrated(case, E):
    """Every token's k routes drawn from the same k + 1 experts (seeded)."""
    k = case.topk_ids.shape[1]
    g = torch.Generator().manual_seed(case.seed + 5)
    hot = torch.randperm(E, generator=g)[:k + 1].to(torch.int32)
    pick = torch.rand(case.M, k + 1, generator=g).argsort(dim=1)[:, :k]
    ids = hot[pick].contiguous()
    return mi.MoeCase(case.shape, case.M, case.x, ids, case.topk_weights, case.w1,
                      case.w1_scale, case.w2, case.w2_scale, case.seed)


def _cases(shape_name, M, shp=None, weights=None):
    """Original, changed-input, concentrated-routing and same-experts cases
    of one shape and token count."""
    a = mi.make_case(shape_name, M, shape=shp, weights=weights)
    b = mi.make_case(shape_name, M, variant=2, shape=shp, weights=weights)
    k, E = a.topk_ids.shape[1], a.shape.E
    if a.shape.E_route >= 16 + k and not a.shape.shared_expert:
        c = mi.make_case(shape_name, M, variant=3, routing="hot", shape=shp, weights=weights)
    else:
        c = _concentrated(b, E)
    d = _same_experts(a, [(E - 1 - 3 * j) % E for j in range(k)])
    return [("original", a), ("changed", b), ("concentrated", c), ("same_experts", d),
            ("restored", a)]


def _snapshot(*tensors):
    return [t.detach().clone() for t in tensors]


def _run_graph_sequence(layer, cases, a16, tokens=None):
    first = cases[0][1]
    M, H, k = first.M, layer.H, first.topk_ids.shape[1]
    x = first.x.cuda()
    ids = first.topk_ids.cuda()
    w = first.topk_weights.cuda()
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(layer.workspace_bytes(M, k), dtype=torch.uint8, device="cuda")
    weights_before = _snapshot(layer.w1, layer.w1_scale, layer.w2, layer.w2_scale)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        layer(x, ids, w, out=out, ws=ws)                  # eager call (loads, attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer(x, ids, w, out=out, ws=ws)
    torch.cuda.synchronize()
    stats = []
    for label, case in cases:
        x.copy_(case.x)
        ids.copy_(case.topk_ids)
        w.copy_(case.topk_weights)
        ws.fill_(0xFF)
        out.view(torch.int16).fill_(-1)
        inputs_before = _snapshot(x, ids, w)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for before, now in zip(inputs_before, (x, ids, w)):
            assert torch.equal(before, now), f"{label}: an input was written"
        st = check_outputs(case, layer, a16, out, ws, tokens=tokens)
        st["graph_case"] = label
        stats.append(st)
    del g                                                # graph before its buffers
    torch.cuda.synchronize()
    for before, now in zip(weights_before, (layer.w1, layer.w1_scale, layer.w2, layer.w2_scale)):
        assert torch.equal(before, now), "weights were written"
    return stats


@pytest.mark.parametrize("a16", [False, True])
@pytest.mark.parametrize("M", [9, 130])
def test_changed_input_graph_replay_small(cuda_lib, a16, M):
    # M=9: the one-launch decode front (<= 256 routes); M=130: sort + gather
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=8, a16=a16)
    w = mi.make_weights(shp, 13)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=a16)
    for st in _run_graph_sequence(layer, _cases("small", M, shp=shp, weights=w), a16):
        print(st)


@pytest.mark.parametrize("name,M", [("backbone", 12), ("backbone", 96), ("a16w4_385", 12)])
def test_changed_input_graph_replay_model_shapes(cuda_lib, name, M):
    layer = layer_for(name)
    a16 = mi.SHAPES[name].a16
    cases = _cases(name, M, weights=weights_for(name))
    tok = None if M <= 12 else sample_tokens(M, 8, 17)
    for st in _run_graph_sequence(layer, cases, a16, tokens=tok):
        print(st)


@pytest.mark.parametrize("a16", [False, True])
def test_eager_call_preserves_inputs(cuda_lib, a16):
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=10, a16=a16)
    w = mi.make_weights(shp, 19)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=a16)
    case = mi.make_case("small", 300, shape=shp, weights=w)
    x, ids, wt = case.x.cuda(), case.topk_ids.cuda(), case.topk_weights.cuda()
    before = _snapshot(x, ids, wt, layer.w1, layer.w1_scale, layer.w2, layer.w2_scale)
    out = layer(x, ids, wt)
    torch.cuda.synchronize()
    after = (x, ids, wt, layer.w1, layer.w1_scale, layer.w2, layer.w2_scale)
    assert all(torch.equal(b, a) for b, a in zip(before, after))
    assert np.isfinite(out.float().cpu().numpy()).all()
