"""GPU parity of the separate shared expert of its own intermediate size.

The pages run DeepSeek's shared expert alongside the routed ones (AITER
#5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning", Performance on the
measured runtime: shared-first MoE including the shared expert; the 385
top-7 layout of AITER #6286). Here the shared expert has an intermediate
size Is of its own; the layer stores it as ceil(Is / Ip) pieces appended
after the routed experts, and the gating gives every token those columns
with weight 1. Two comparisons per case:

* against the oracle of the layer as it stores the experts (routed experts
  plus the pieces, cut by the oracle's own shared_expert_pieces): every bar
  of the fused-call parity (sort lists bit-exact, intermediate codes,
  output with the rounding-decision budget);
* against the oracle with the shared MLP computed separately (its full
  intermediate, one dense pass over every token) and added to the routed
  experts' FP64 sum before the one BF16 rounding, with the same tolerance.
"""
import numpy as np
import pytest
import torch

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from moe_check import ATOL, RTOL, check_outputs, run_case, sample_tokens
from oracle import moe as om
from oracle import router as orr

pytestmark = pytest.mark.gpu


def _shared(H, Is, seed):
    shp = mi.small_shape(H=H, I=Is, Ip=Is, E=1, topk=1)
    w = mi.make_weights(shp, seed)
    return tuple(w[k][0] for k in ("w1", "w1_scale", "w2", "w2_scale"))


def _run(routed_shape, routed_w, shared, M, topk, a16, seed, tokens=None):
    E_r = routed_shape.E
    layer = m.MoeLayer(routed_w["w1"], routed_w["w1_scale"], routed_w["w2"],
                       routed_w["w2_scale"], a16=a16, shared_expert=shared)
    Ip = routed_shape.Ip
    n = -(-(shared[2].shape[1] * 2) // Ip)
    assert layer.n_shared == n and layer.E == E_r + n and layer.shared_id == E_r
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(M, E_r, generator=g, dtype=torch.float32)
    ids, wt = layer.route(logits.cuda(), topk)
    ids_c, wt_c = ids.cpu(), wt.cpu()
    ref_ids, _ = orr.router_topk(logits.numpy(), topk, shared_id=E_r, n_shared=n)
    assert np.array_equal(ids_c.numpy(), ref_ids)
    # the layer's own expert layout: routed experts plus the oracle's pieces
    pieces = om.shared_expert_pieces(*shared, Ip)
    wcat = {k: torch.cat([routed_w[k], torch.from_numpy(p)])
            for k, p in zip(("w1", "w1_scale", "w2", "w2_scale"), pieces)}
    x = mi.make_x(M, routed_shape.H, mi._gen(seed + 1))
    case = mi.MoeCase(routed_shape, M, x, ids_c, wt_c, wcat["w1"], wcat["w1_scale"],
                      wcat["w2"], wcat["w2_scale"], seed)
    out, ws = run_case(layer, case)
    st = check_outputs(case, layer, a16, out, ws, tokens=tokens)
    # the shared MLP computed separately and added in
    sel = np.arange(M) if tokens is None else np.asarray(tokens)
    k_r = topk
    want = om.fused_moe_with_shared(x[sel], ids_c[sel, :k_r], wt_c[sel, :k_r], routed_w["w1"],
                                    routed_w["w1_scale"], routed_w["w2"], routed_w["w2_scale"],
                                    E_r, shared, a16=a16)
    # the two oracle forms are the same sum in FP64 (up to summation order)
    pieces_f64 = om.fused_moe(x, ids_c, wt_c, wcat["w1"], wcat["w1_scale"], wcat["w2"],
                              wcat["w2_scale"], layer.E, a16=a16, tokens=sel).out_f64
    sep_f64 = om.fused_moe(x[sel], ids_c[sel, :topk], wt_c[sel, :topk], routed_w["w1"],
                           routed_w["w1_scale"], routed_w["w2"], routed_w["w2_scale"], E_r,
                           a16=a16).out_f64 + om.shared_mlp(x[sel], *shared, a16=a16)
    np.testing.assert_allclose(pieces_f64, sep_f64, rtol=1e-9, atol=1e-9 * np.abs(sep_f64).max())
    got = out.cpu()[torch.from_numpy(sel)].to(torch.float64).numpy()
    err = np.abs(got - want)
    over = err > ATOL + RTOL * np.abs(want)
    st["separate_max_abs_err"] = float(err.max())
    st["separate_over_plain"] = int(over.sum())
    # elements beyond the plain bar are the ones check_outputs covered with
    # the rounding-decision budget (same GPU output, the same sum)
    assert over.sum() <= st["n_needing_budget"] + 2, st
    return st


@pytest.mark.parametrize("a16", [False, True])
@pytest.mark.parametrize("Is", [256, 384, 128])
def test_separate_shared_expert_own_size_small(cuda_lib, a16, Is):
    shp = mi.small_shape(H=512, I=256, Ip=256, E=8, topk=3, E_route=8, a16=a16)
    w = mi.make_weights(shp, 51)
    print(_run(shp, w, _shared(512, Is, 53 + Is), 70, 3, a16, 55))


@pytest.mark.parametrize("M", [12, 300])
def test_separate_shared_expert_backbone(cuda_lib, M):
    # backbone routed experts (Ip = 640) with a shared expert of intermediate
    # 1280: two pieces, scheduled first in both GEMM stages
    shp = mi.SHAPES["backbone"]
    w = mi.make_weights(shp, mi.weight_seed(1))
    tok = None if M <= 12 else sample_tokens(M, 8, 9)
    print(_run(shp, w, _shared(shp.H, 1280, 61), M, 6, False, 63 + M, tokens=tok))
