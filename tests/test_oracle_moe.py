"""Pins of the oracle's sort and two-stage MoE arithmetic.

Each test checks the oracle against something other than itself:
* the sort against Python's ``sorted`` on tiny inputs and permutation
  invariants (stable grouping by expert, padding to block_m, dropped ids);
* the layer against a scalar brute force written here from the step list
  (own nibble decoding, E4M3 decode taken from torch, math.fsum sums);
* special cases: one expert with k=1 and weight 1 is a dense SwiGLU MLP,
  zero-weight routes contribute nothing, the output is linear in the
  routing weights, a fused shared expert equals a dense MLP added in.

Steps follow AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning"
(Configuration) and AITER #5904 "Add tuned a8w4 fused-MoE configs for
DeepSeek V4.1-Flash (TP4 + EP, gfx950)" (Fused-MoE kernel expert-parallel
benchmark: sorting, both stages and the intermediate quantization).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe as om
from oracle import mx_formats as mx


# ------------------------------------------------------------------ sort

def _brute_sort(ids, E, bm):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    R = len(flat)
    pairs = sorted((e, r) for r, e in enumerate(flat) if 0 <= e < E)
    layout, block_expert = [], []
    for e in range(E):
        seg = [r for (ee, r) in pairs if ee == e]
        if not seg:
            continue
        nb = -(-len(seg) // bm)
        layout += seg + [R] * (nb * bm - len(seg))
        block_expert += [e] * nb
    return layout, block_expert


@pytest.mark.parametrize("bm", [1, 4, 16])
@pytest.mark.parametrize("seed", range(6))
def test_sort_matches_brute_force(bm, seed):
    g = torch.Generator().manual_seed(seed)
    M, k, E = 7 + seed, 3, 5 + seed
    ids = torch.randint(-1, E + 2, (M, k), generator=g).to(torch.int32)
    w = torch.rand(M, k, generator=g)
    res = om.moe_sort(ids, w, E, bm)
    layout, be = _brute_sort(ids, E, bm)
    assert res.sorted_route.tolist() == layout
    assert res.block_expert.tolist() == be
    assert res.num_padded == len(layout) and res.num_padded % bm == 0
    wf = w.reshape(-1).numpy()
    R = M * k
    for p, r in enumerate(layout):
        if r == R:
            assert res.sorted_w[p] == 0
        else:
            assert res.sorted_w[p] == wf[r] and res.route_pos[r] == p
    dropped = [r for r, e in enumerate(ids.reshape(-1).tolist()) if not 0 <= e < E]
    assert all(res.route_pos[r] == -1 for r in dropped)


def test_sort_permutation_invariants_large():
    shp = mi.SHAPES["backbone"]
    g = torch.Generator().manual_seed(11)
    ids, w = mi.make_routing(shp, 4096, g, "zipf")
    res = om.moe_sort(ids, w, shp.E, 64)
    R = ids.numel()
    valid = res.sorted_route[res.sorted_route != R]
    assert np.array_equal(np.sort(valid), np.arange(R))      # every route once
    flat = ids.reshape(-1).numpy()
    for e in range(shp.E):
        lo, hi = res.expert_off[e], res.expert_off[e + 1]
        seg = res.sorted_route[lo:hi]
        real = seg[seg != R]
        assert (flat[real] == e).all()
        assert (np.diff(real) > 0).all()                       # stable: ascending r
        assert (seg[len(real):] == R).all()                    # pads at the end
        assert (hi - lo) % 64 == 0 and (hi - lo) < len(real) + 64
        if len(real) == 0:
            assert hi == lo                                    # empty expert: no block
    assert np.array_equal(res.route_pos[res.sorted_route[res.sorted_route != R]],
                          np.nonzero(res.sorted_route != R)[0])


def test_sort_drops_non_local_experts():
    ids = torch.tensor([[0, 5], [7, 1]], dtype=torch.int32)
    res = om.moe_sort(ids, torch.ones(2, 2), 4, 2)
    assert res.sorted_route.tolist() == [0, 4, 3, 4]
    assert res.route_pos.tolist() == [0, -1, -1, 2]


# ---------------------------------------------------- brute-force layer

def _e2m1(code):
    s = -1.0 if code & 8 else 1.0
    return s * {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}[code & 7]


_E4M3_TORCH = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
    torch.float8_e4m3fn).to(torch.float64).tolist()


def _w_elem(packed, scale, n, kk):
    byte = int(packed[n, kk // 2])
    code = byte & 15 if kk % 2 == 0 else byte >> 4
    return _e2m1(code) * 2.0 ** (int(scale[n, kk // 32]) - 127)


def _quant_row_brute(vals):
    """Per-1x32 FP8: scale 2^(floor(log2 amax) - 8); nearest E4M3, ties to
    even code, saturate at 448 (written independently of the oracle)."""
    codes, sc = [], []
    finite = [(c, v) for c, v in enumerate(_E4M3_TORCH[:127])]
    for b in range(0, len(vals), 32):
        blk = vals[b:b + 32]
        amax = max(abs(v) for v in blk)
        if amax == 0:
            codes += [0] * 32
            sc.append(0)
            continue
        m, ex = math.frexp(amax)
        e = min(max(ex - 1 - 8, -127), 127)
        sc.append(e + 127)
        for v in blk:
            a = min(abs(v) / 2.0 ** e, 448.0)
            best = min(finite, key=lambda cv: (abs(cv[1] - a), cv[0] % 2))
            c = best[0]
            if v < 0 or (v == 0 and math.copysign(1, v) < 0):
                c |= 0x80
            codes.append(c)
    return codes, sc


def _bf16_exact(v):
    """Nearest bfloat16 value (ties to even), by exact rational arithmetic."""
    if v == 0:
        return v
    q = Fraction(abs(v))
    e = math.floor(math.log2(abs(v)))
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    quantum = Fraction(2) ** max(e - 7, -133)
    r = round(q / quantum) * quantum          # Fraction round: half to even
    return math.copysign(float(r), v)


def _brute_layer(case, a16=False):
    x = case.x.to(torch.float64).numpy()
    ids = case.topk_ids.numpy()
    wts = case.topk_weights.numpy()
    W1, W1s, W2, W2s = (t.numpy() for t in (case.w1, case.w1_scale, case.w2, case.w2_scale))
    M, H = x.shape
    k = ids.shape[1]
    E = case.shape.E
    Ip = W2.shape[2] * 2
    out = np.zeros((M, H))
    inter = {}
    for t in range(M):
        if a16:
            xv = [float(v) for v in x[t]]
        else:
            codes, sc = _quant_row_brute([float(v) for v in x[t]])
            xv = [_E4M3_TORCH[c] * 2.0 ** (sc[i // 32] - 127) for i, c in enumerate(codes)]
        for j in range(k):
            e = int(ids[t, j])
            if not 0 <= e < E:
                continue
            act = []
            for i in range(Ip):
                gate = math.fsum(xv[kk] * _w_elem(W1[e], W1s[e], 2 * i, kk) for kk in range(H))
                up = math.fsum(xv[kk] * _w_elem(W1[e], W1s[e], 2 * i + 1, kk) for kk in range(H))
                act.append(gate / (1.0 + math.exp(-gate)) * up)
            if a16:
                av = [_bf16_exact(v) for v in act]
                inter[t * k + j] = av
            else:
                ac, asc = _quant_row_brute(act)
                av = [_E4M3_TORCH[c] * 2.0 ** (asc[i // 32] - 127) for i, c in enumerate(ac)]
                inter[t * k + j] = (ac, asc)
            for n in range(H):
                y = math.fsum(av[i] * _w_elem(W2[e], W2s[e], n, i) for i in range(Ip))
                out[t, n] += float(wts[t, j]) * y
    return out, inter


TINY = mi.small_shape(H=64, I=48, Ip=64, E=3, topk=2)


@pytest.mark.parametrize("a16", [False, True])
def test_layer_matches_scalar_brute_force(a16):
    shp = mi.small_shape(H=64, I=48, Ip=64, E=3, topk=2, a16=a16)
    case = mi.make_case("small", 4, shape=shp)
    case.topk_ids[3, 1] = 7          # a dropped (non-local) route
    res = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                       case.w2, case.w2_scale, shp.E, a16=a16, block_m=4)
    ref, inter = _brute_layer(case, a16=a16)
    assert np.allclose(res.out_f64, ref, rtol=1e-12, atol=1e-12)
    R = case.topk_ids.numel()
    for i, p in enumerate(res.inter_rows):
        r = int(res.sort.sorted_route[p])
        if a16:
            assert res.aq[i].tolist() == inter[r]
        else:
            assert res.aq[i].tolist() == inter[r][0]
            assert res.as_[i].tolist() == inter[r][1]
    assert len(res.inter_rows) == R - 1
    # padded intermediate columns (48..63) quantise to zero codes
    if not a16:
        assert (res.aq[:, 48:] == 0).all()


def test_single_expert_top1_is_dense_swiglu_mlp():
    shp = mi.small_shape(H=128, I=64, Ip=64, E=1, topk=1)
    case = mi.make_case("small", 9, shape=shp)
    case.topk_weights[:] = 1.0
    res = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                       case.w2, case.w2_scale, 1, block_m=4)
    x = case.x.to(torch.float64).numpy()
    xq, xs = mx.quant_mxfp8(x)
    xd = torch.from_numpy(mx.dequant_mxfp8(xq, xs))
    w1 = torch.from_numpy(mx.dequant_mxfp4(case.w1[0].numpy(), case.w1_scale[0].numpy()))
    w2 = torch.from_numpy(mx.dequant_mxfp4(case.w2[0].numpy(), case.w2_scale[0].numpy()))
    gate = xd @ w1[0::2].T
    up = xd @ w1[1::2].T
    act = torch.nn.functional.silu(gate) * up
    aq, as_ = mx.quant_mxfp8(act.numpy())
    y = torch.from_numpy(mx.dequant_mxfp8(aq, as_)) @ w2.T
    assert np.allclose(res.out_f64, y.numpy(), rtol=1e-12, atol=1e-10)


def test_zero_weight_routes_contribute_nothing():
    shp = mi.small_shape(H=128, I=64, Ip=64, E=6, topk=3)
    case = mi.make_case("small", 12, shape=shp)
    w = case.topk_weights.clone()
    w[::2, 1] = 0.0
    a = om.fused_moe(case.x, case.topk_ids, w, case.w1, case.w1_scale, case.w2,
                     case.w2_scale, shp.E, block_m=4)
    ids = case.topk_ids.clone()
    ids[::2, 1] = -1
    b = om.fused_moe(case.x, ids, w, case.w1, case.w1_scale, case.w2, case.w2_scale,
                     shp.E, block_m=4)
    assert np.array_equal(a.out_bf16, b.out_bf16)
    assert np.array_equal(a.out_f64, b.out_f64)


def test_output_is_linear_in_routing_weights():
    shp = mi.small_shape(H=128, I=64, Ip=64, E=6, topk=3)
    case = mi.make_case("small", 10, shape=shp)
    args = (case.x, case.topk_ids)
    wargs = (case.w1, case.w1_scale, case.w2, case.w2_scale, shp.E)
    g = torch.Generator().manual_seed(5)
    wa = torch.rand(10, 3, generator=g)
    wb = torch.rand(10, 3, generator=g)
    fa = om.fused_moe(*args, wa, *wargs).out_f64
    fb = om.fused_moe(*args, wb, *wargs).out_f64
    fab = om.fused_moe(*args, (wa.double() + wb.double()).float(), *wargs).out_f64
    f2 = om.fused_moe(*args, wa * 4, *wargs).out_f64
    scale = np.abs(fa).max() + np.abs(fb).max()
    # (wa+wb) is rounded to float32 once; allow that rounding
    assert np.abs(fab - (fa + fb)).max() <= 1e-6 * scale
    assert np.array_equal(f2, 4 * fa)                       # power-of-two scaling is exact


def test_fused_shared_expert_is_a_dense_mlp_added_in():
    shp = mi.small_shape(H=128, I=64, Ip=64, E=5, topk=3, shared_expert=True)
    case = mi.make_case("small", 8, shape=shp)
    assert (case.topk_ids[:, -1] == 4).all() and (case.topk_weights[:, -1] == 1).all()
    full = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                        case.w2, case.w2_scale, shp.E).out_f64
    routed_ids = case.topk_ids.clone()
    routed_ids[:, -1] = -1
    routed = om.fused_moe(case.x, routed_ids, case.topk_weights, case.w1, case.w1_scale,
                          case.w2, case.w2_scale, shp.E).out_f64
    sh_ids = torch.full((8, 1), 0, dtype=torch.int32)
    dense = om.fused_moe(case.x, sh_ids, torch.ones(8, 1), case.w1[4:5], case.w1_scale[4:5],
                         case.w2[4:5], case.w2_scale[4:5], 1).out_f64
    assert np.allclose(full, routed + dense, rtol=0, atol=1e-9 * np.abs(full).max())


def test_token_sampling_matches_full_run():
    shp = mi.small_shape(H=128, I=64, Ip=64, E=6, topk=3)
    case = mi.make_case("small", 20, shape=shp)
    full = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                        case.w2, case.w2_scale, shp.E)
    sel = [0, 7, 19]
    part = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                        case.w2, case.w2_scale, shp.E, tokens=sel)
    assert np.array_equal(part.out_bf16, full.out_bf16[sel])


def test_token_with_no_local_route_is_zero():
    shp = mi.small_shape(H=128, I=64, Ip=64, E=4, topk=2, E_route=16)
    case = mi.make_case("small", 30, shape=shp)
    res = om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                       case.w2, case.w2_scale, shp.E)
    none_local = (case.topk_ids >= 4).all(dim=1).numpy()
    assert none_local.any()
    assert (res.out_bf16[none_local] == 0).all()


# ------------------------------------------------- separate shared expert

def _shared_case(Is, seed):
    shp = mi.small_shape(H=256, I=Is, Ip=Is, E=1, topk=1)
    w = mi.make_weights(shp, seed)
    return w["w1"][0], w["w1_scale"][0], w["w2"][0], w["w2_scale"][0]


@pytest.mark.parametrize("Is,Ip", [(256, 128), (384, 128), (96, 128), (128, 128)])
def test_shared_mlp_is_the_sum_of_its_pieces(Is, Ip):
    # SiLU(gate)*up acts on each intermediate index alone and the down
    # projection sums over them: the shared MLP equals the sum of its
    # Ip-sized pieces run as experts of weight 1 (zero-padded at the end)
    sh = _shared_case(Is, 31 + Is)
    x = mi.make_x(11, 256, mi._gen(3))
    full = om.shared_mlp(x, *sh)
    pieces = om.shared_expert_pieces(*sh, Ip)
    n = pieces[0].shape[0]
    assert n == -(-Is // Ip)
    ids = torch.arange(n, dtype=torch.int32).expand(11, n).contiguous()
    res = om.fused_moe(x, ids, torch.ones(11, n), *pieces, n).out_f64
    np.testing.assert_allclose(res, full, rtol=1e-12, atol=1e-12 * np.abs(full).max())


def test_shared_mlp_is_a_dense_swiglu_mlp():
    # brute force from the step list on a tiny shape: every token, weight 1
    sh = _shared_case(64, 77)
    x = mi.make_x(3, 256, mi._gen(5))
    got = om.shared_mlp(x, *sh)
    xq, xs = mx.quant_mxfp8(x.to(torch.float64).numpy())
    xd = mx.dequant_mxfp8(xq, xs)
    h = xd @ mx.dequant_mxfp4(sh[0].numpy(), sh[1].numpy()).T
    a = h[:, 0::2] / (1 + np.exp(-h[:, 0::2])) * h[:, 1::2]
    aq, as_ = mx.quant_mxfp8(a)
    y = mx.dequant_mxfp8(aq, as_) @ mx.dequant_mxfp4(sh[2].numpy(), sh[3].numpy()).T
    np.testing.assert_allclose(got, y, rtol=1e-12, atol=1e-12)


def test_routed_plus_shared_matches_the_fused_shared_layout():
    # with the routed size the separate shared expert equals the 385/top-7
    # style layout: the shared expert appended as expert E with a weight-1
    # column (both FP64 sums, one BF16 rounding)
    shp = mi.small_shape(H=256, I=128, Ip=128, E=5, topk=2)
    w = mi.make_weights(shp, 41)
    case = mi.make_case("small", 9, shape=shp, weights=w)
    sh = _shared_case(128, 43)
    sep = om.fused_moe_with_shared(case.x, case.topk_ids, case.topk_weights, case.w1,
                                   case.w1_scale, case.w2, case.w2_scale, 5, sh)
    cat = [torch.cat([a, b[None]]) for a, b in zip((case.w1, case.w1_scale, case.w2,
                                                    case.w2_scale), sh)]
    ids = torch.cat([case.topk_ids, torch.full((9, 1), 5, dtype=torch.int32)], 1)
    wts = torch.cat([case.topk_weights, torch.ones(9, 1)], 1)
    fused = om.fused_moe(case.x, ids, wts, *cat, 6)
    np.testing.assert_allclose(sep, fused.out_bf16, rtol=2 ** -7, atol=0)
    assert (sep == fused.out_bf16).mean() > 0.99

