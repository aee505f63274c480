"""GPU parity of the gating kernel (moe_router_topk) against the oracle.

Bars: expert ids bit-exact (the selection compares FP32 logits on both
sides, ties to the lower expert); routing weights within rtol 1e-5 (the GPU
forms the softmax of at most 16 logits in FP32: expf within 2 ulp, a sum of
<= 16 terms and one division keep the relative error below ~2e-6; the
oracle works in FP64). The last test feeds the kernel's output to the fused
call and compares that with the oracle."""
import numpy as np
import pytest
import torch

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from moe_check import check_outputs, compare, sample_tokens, weights_for, layer_for
from oracle import router as orr

pytestmark = pytest.mark.gpu

RTOL = 1e-5


def _logits(M, E, seed, ties=False):
    g = torch.Generator().manual_seed(seed)
    L = torch.randn(M, E, generator=g, dtype=torch.float32)
    if ties:
        L = torch.round(L * 2) / 2            # many exact ties, +0.0 and -0.0
    return L


@pytest.mark.parametrize("M,E,k,shared,ties", [
    (1, 384, 6, None, False),
    (7, 128, 3, None, False),
    (64, 33, 8, None, False),          # E not a multiple of 32
    (333, 96, 1, None, False),
    (50, 512, 16, None, False),        # largest E and topk
    (40, 384, 6, 384, False),          # shared expert column (385 / top-7)
    (257, 384, 6, None, True),
    (200, 16, 16, None, True),         # topk = E
    (768, 384, 6, None, False),        # decode bucket of the backbone
    (16384, 384, 6, None, False),      # prefill bucket
])
def test_router_parity(cuda_lib, M, E, k, shared, ties):
    L = _logits(M, E, 1000 + M + E + k, ties)
    ids, w = m.moe_router_topk(L.cuda(), k, shared_id=shared)
    torch.cuda.synchronize()
    ref_ids, ref_w = orr.router_topk(L.numpy(), k, shared_id=shared)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), ref_w, rtol=RTOL, atol=0)


def test_router_zero_tokens(cuda_lib):
    ids, w = m.moe_router_topk(torch.empty(0, 384, dtype=torch.float32, device="cuda"), 6)
    assert ids.shape == (0, 6) and w.shape == (0, 6)


def test_router_feeds_the_fused_call(cuda_lib):
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=8)
    w = mi.make_weights(shp, 21)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=False)
    case = mi.make_case("small", 96, shape=shp, weights=w)
    L = _logits(96, 8, 77)
    ids, wt = m.moe_router_topk(L.cuda(), 3)
    ref_ids, _ = orr.router_topk(L.numpy(), 3)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    # the same ids and FP32 weights go to the GPU call and to the oracle
    case.topk_ids = ids.cpu()
    case.topk_weights = wt.cpu()
    print(compare(case, layer, False))


@pytest.mark.parametrize("a16", [False, True])
def test_separate_shared_expert(cuda_lib, a16):
    # 8 routed experts plus one separate shared expert (weight 1 for every
    # token), routed by the gating kernel; the oracle sees all 9 experts
    shp = mi.small_shape(H=512, I=192, Ip=256, E=9, topk=4, E_route=8, a16=a16)
    w = mi.make_weights(shp, 31)
    routed = [w[k][:8] for k in ("w1", "w1_scale", "w2", "w2_scale")]
    shared = [w[k][8] for k in ("w1", "w1_scale", "w2", "w2_scale")]
    layer = m.MoeLayer(*routed, a16=a16, shared_expert=shared)
    assert layer.E == 9 and layer.shared_id == 8
    L = _logits(70, 8, 91)
    ids, wt = layer.route(L.cuda(), 3)
    ids_c, wt_c = ids.cpu(), wt.cpu()
    assert (ids_c[:, 3] == 8).all() and (wt_c[:, 3] == 1.0).all()
    ref_ids, _ = orr.router_topk(L.numpy(), 3, shared_id=8)
    assert np.array_equal(ids_c.numpy(), ref_ids)
    case = mi.make_case("small", 70, shape=shp, weights=w)
    case.topk_ids = ids_c
    case.topk_weights = wt_c
    print(compare(case, layer, a16))


# ------------------------------------------------------------ gated calls
# fused_moe_*_gated: the gating (the same selection and softmax as
# moe_router_topk) in front of the fused call; up to 256 routes it runs
# inside the decode front kernel, beyond that as its own launch.

def _gated_check(layer, case, logits, topk, a16, shared=None, tokens=None):
    M = case.M
    x = case.x.cuda()
    lg = logits.cuda()
    kout = topk + (1 if shared is not None else 0)
    ws = torch.empty(layer.workspace_bytes(M, kout), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    out = torch.empty(M, layer.H, dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    out, ids, w = m.fused_moe_gated(x, lg, topk, layer.w1, layer.w1_scale, layer.w2,
                                    layer.w2_scale, layer.E, layer.Ip, a16=a16, shared_id=shared,
                                    out=out, ws=ws)
    torch.cuda.synchronize()
    ref_ids, ref_w = orr.router_topk(logits.numpy(), topk, shared_id=shared)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), ref_w, rtol=RTOL, atol=0)
    # the layer's result on the routing it produced, against the oracle
    case.topk_ids = ids.cpu()
    case.topk_weights = w.cpu()
    return check_outputs(case, layer, a16, out, ws, tokens=tokens)


@pytest.mark.parametrize("name,M", [("backbone", 6), ("backbone", 24), ("draft", 5),
                                    ("ep", 16), ("a16w4_384", 12)])
def test_gated_call_decode(cuda_lib, name, M):
    # at most 256 routes: gating, sort and gather in the call's first kernel
    shp = mi.SHAPES[name]
    layer = layer_for(name)
    case = mi.make_case(name, M, weights=weights_for(name))
    logits = _logits(M, shp.E_route, 4000 + M)
    print(_gated_check(layer, case, logits, shp.topk, shp.a16))


def test_gated_call_shared_expert_decode(cuda_lib):
    # 384 routed experts top-6 plus the shared expert 384 (7 columns)
    layer = layer_for("a16w4_385")
    case = mi.make_case("a16w4_385", 12, weights=weights_for("a16w4_385"))
    logits = _logits(12, 384, 4100)
    print(_gated_check(layer, case, logits, 6, True, shared=384))


@pytest.mark.parametrize("a16", [False, True])
def test_gated_call_separate_launch(cuda_lib, a16):
    # more than 256 routes: the gating kernel runs as its own launch
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=8, a16=a16)
    w = mi.make_weights(shp, 23)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=a16)
    case = mi.make_case("small", 130, shape=shp, weights=w)
    print(_gated_check(layer, case, _logits(130, 8, 4200), 3, a16))


def test_gated_call_prefill_sample(cuda_lib):
    layer = layer_for("backbone")
    case = mi.make_case("backbone", 4096, weights=weights_for("backbone"))
    logits = _logits(4096, 384, 4300)
    print(_gated_check(layer, case, logits, 6, False, tokens=sample_tokens(4096, 8, 5)))


def test_gated_call_graph_replay_changed_logits(cuda_lib):
    # one captured gated call, replayed on new logits written in place
    layer = layer_for("backbone")
    M = 12
    x = mi.make_case("backbone", M, weights=weights_for("backbone")).x.cuda()
    lg = _logits(M, 384, 4400).cuda()
    out = torch.empty(M, layer.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(M, 6, dtype=torch.int32, device="cuda")
    w = torch.empty(M, 6, dtype=torch.float32, device="cuda")
    ws = torch.empty(layer.workspace_bytes(M, 6), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward_gated(x, lg, 6, out=out, ws=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.fused_moe_gated(x, lg, 6, layer.w1, layer.w1_scale, layer.w2, layer.w2_scale, layer.E,
                          layer.Ip, out=out, ws=ws, topk_ids=ids, topk_weights=w, stream=s)
    for seed in (4401, 4402):
        new = _logits(M, 384, seed)
        lg.copy_(new)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref_ids, _ = orr.router_topk(new.numpy(), 6)
        assert np.array_equal(ids.cpu().numpy(), ref_ids)
        case = mi.make_case("backbone", M, weights=weights_for("backbone"))
        case.topk_ids = ids.cpu()
        case.topk_weights = w.cpu()
        print(check_outputs(case, layer, False, out, ws))
    del g
