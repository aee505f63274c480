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
from moe_check import compare
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
