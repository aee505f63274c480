"""GPU parity of the whole fused MoE call against the oracle.

Small geometries are compared in full (every token, every intermediate row);
the pages' geometries (draft, backbone incl. the M31/32/33/255/256/257
boundary checks and concentrated routing, expert-parallel shard, a16w4
384-top6 and 385-top7 with the fused shared expert at decode and prefill
sizes, Zipf prefill stress) are
compared on every route of a seeded sample of tokens, at the sizes and in the
launch configuration the benchmark uses. At M=16384 the stage-one
intermediate of every route of three whole experts is compared as well: the
most loaded expert, the one whose route blocks open the last wave of
stage-one tiles, and the last non-empty expert; the sampled tokens include
tokens of each of them. Workspace and output are poisoned (0xFF) before each
call, so anything left unwritten shows up.
"""
import numpy as np
import pytest
import torch

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from moe_check import compare, layer_for, sample_tokens, tokens_of_expert
from oracle import moe as om

pytestmark = pytest.mark.gpu


def _small_layer(shp, seed):
    w = mi.make_weights(shp, seed)
    return w, m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=shp.a16)


@pytest.mark.parametrize("a16", [False, True])
@pytest.mark.parametrize("M", [1, 5, 37, 130, 600])
def test_small_geometry_full(cuda_lib, a16, M):
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=10, a16=a16)
    w, layer = _small_layer(shp, 5)
    case = mi.make_case("small", M, shape=shp, weights=w)
    st = compare(case, layer, a16)
    print(st)


@pytest.mark.parametrize("a16", [False, True])
@pytest.mark.parametrize("bm", [16, 32, 64, 128, 256])
def test_explicit_block_m(cuda_lib, a16, bm):
    # the route block a tuning table sets (the *_bm entry points): every
    # supported block on both variants, several tiles and a ragged tail
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=10, a16=a16)
    w = mi.make_weights(shp, 5)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=a16,
                       block_m_table=[(1 << 30, bm)])
    case = mi.make_case("small", 130, shape=shp, weights=w)
    st = compare(case, layer, a16)
    assert st["block_m"] == bm


@pytest.mark.parametrize("a16", [False, True])
@pytest.mark.parametrize("pf", [(1, 1), (64, 64), (4, 16)])
def test_explicit_prefetch(cuda_lib, a16, pf):
    # the second tuning knob (fused_moe_*_cfg): weight L2 prefetch leads at
    # their extremes; they move weights into L2 earlier or later and must
    # not change the result
    shp = mi.small_shape(H=512, I=192, Ip=256, E=8, topk=3, E_route=10, a16=a16)
    w = mi.make_weights(shp, 5)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"], a16=a16,
                       block_m_table=[(1 << 30, 16, pf[0], pf[1])])
    assert layer.prefetch_for(130, 3) == pf
    case = mi.make_case("small", 130, shape=shp, weights=w)
    compare(case, layer, a16)


def test_explicit_prefetch_backbone(cuda_lib):
    # the pages' backbone geometry at a decode bucket, sampled tokens
    wts = __import__("moe_check").weights_for("backbone", 0)
    layer = m.MoeLayer(wts["w1"], wts["w1_scale"], wts["w2"], wts["w2_scale"],
                       block_m_table=[(1 << 30, 16, 32, 4)])
    case = mi.make_case("backbone", 384, weights=wts)
    print(compare(case, layer, False, tokens=sample_tokens(384, 8, 11)))


@pytest.mark.parametrize("name,M,split", [("ep", 64, 1), ("backbone", 6, 2), ("draft", 40, 1),
                                          ("a16w4_384", 12, 2), ("a16w4_385", 300, 2),
                                          ("a16w4_385", 300, 1)])
def test_explicit_split_walk(cuda_lib, name, M, split):
    # the third tuning knob: the GEMMs' split walk asked for explicitly (the
    # expert-parallel shard, whose routes are mostly dropped; the draft at 40
    # tokens) and switched off (the plain kernels, whole tiles in both
    # stages, where the library would split), on both variants
    a16 = mi.SHAPES[name].a16
    wts = __import__("moe_check").weights_for(name, 0)
    layer = m.MoeLayer(wts["w1"], wts["w1_scale"], wts["w2"], wts["w2_scale"], a16=a16,
                       block_m_table=[(1 << 30, 16, 0, 0, split)])
    assert layer.split_for(M, 6) == split
    case = mi.make_case(name, M, weights=wts)
    print(compare(case, layer, a16, tokens=None if M <= 12 else sample_tokens(M, 8, M)))


def test_empty_experts_and_all_dropped_tokens(cuda_lib):
    shp = mi.small_shape(H=256, I=128, Ip=128, E=16, topk=2, E_route=64)
    w, layer = _small_layer(shp, 9)
    case = mi.make_case("small", 20, shape=shp, weights=w)
    assert ((case.topk_ids >= 16).all(dim=1)).any()   # some tokens have no local route
    compare(case, layer, False)


def test_zero_tokens(cuda_lib):
    shp = mi.small_shape(H=256, I=128, Ip=128, E=4, topk=2)
    w, layer = _small_layer(shp, 3)
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    wt = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    out = layer(x, ids, wt)
    assert out.shape == (0, 256)


def _config_case(name, M, routing="uniform", variant=0, n_tok=8):
    layer = layer_for(name, variant)
    case = mi.make_case(name, M, variant=variant, routing=routing,
                        weights=__import__("moe_check").weights_for(name, variant))
    return layer, case, sample_tokens(M, n_tok, M + variant)


@pytest.mark.parametrize("M", [5])
def test_draft(cuda_lib, M):
    layer, case, tok = _config_case("draft", M)
    print(compare(case, layer, False, tokens=None))


@pytest.mark.parametrize("M", [6, 96, 768, 31, 32, 33, 255, 256, 257])
def test_backbone(cuda_lib, M):
    layer, case, tok = _config_case("backbone", M)
    print(compare(case, layer, False, tokens=None if M <= 6 else tok))


def test_backbone_concentrated_routing(cuda_lib):
    layer, case, tok = _config_case("backbone", 384, routing="hot", variant=1)
    print(compare(case, layer, False, tokens=tok))


def _prefill_experts(case, layer):
    """(experts to check whole, tokens to compare) for a prefill case: the
    most loaded expert, the expert of the route block that opens the last
    wave of stage-one tiles (CTA slots = SMs x 2 at route blocks <= 128),
    and the last non-empty expert; 24 tokens of each of the latter two, 16
    of the first and 16 drawn from all tokens."""
    M, k = case.M, case.topk_ids.shape[1]
    bm = layer.workspace_layout(M, k)["block_m"]
    srt = om.moe_sort(case.topk_ids, case.topk_weights, layer.E, bm)
    cnt = srt.expert_cnt
    hot = int(np.argmax(cnt))
    last = int(np.nonzero(cnt)[0][-1])
    n_tiles = 2 * layer.Ip // 128
    slots = torch.cuda.get_device_properties(0).multi_processor_count * 2
    tiles = srt.num_padded // bm * n_tiles
    first_last_wave = (tiles // slots) * slots
    if first_last_wave >= tiles:
        first_last_wave = max(tiles - slots, 0)
    wave = int(srt.block_expert[first_last_wave // n_tiles])
    experts = sorted({hot, last, wave})
    tok = np.unique(np.concatenate([
        tokens_of_expert(case, hot, 16, 1), tokens_of_expert(case, wave, 24, 2),
        tokens_of_expert(case, last, 24, 3), sample_tokens(M, 16, 4)]))
    return experts, tok


@pytest.mark.parametrize("M", [1, 16, 1024])
def test_expert_parallel_shard(cuda_lib, M):
    layer, case, tok = _config_case("ep", M)
    print(compare(case, layer, False, tokens=None if M <= 16 else tok))


def test_expert_parallel_shard_prefill_whole_experts(cuda_lib):
    layer, case, _ = _config_case("ep", 16384)
    experts, tok = _prefill_experts(case, layer)
    print(compare(case, layer, False, tokens=tok, whole_experts=experts))


@pytest.mark.parametrize("name", ["a16w4_384", "a16w4_385"])
@pytest.mark.parametrize("M", [12, 1024])
def test_a16w4(cuda_lib, name, M):
    layer, case, tok = _config_case(name, M)
    print(compare(case, layer, True, tokens=None if M <= 12 else tok))


def test_a16w4_prefill_4096(cuda_lib):
    # route blocks of 64 rows and the grouped stage-2 tile walk (the BF16
    # intermediate is larger than 32 MB) on the 384-expert a16w4 geometry
    layer, case, tok = _config_case("a16w4_384", 4096, n_tok=32)
    print(compare(case, layer, True, tokens=tok))


def test_a16w4_shared_expert_prefill_whole_experts(cuda_lib):
    # 385 experts top-7 at M=16384: the shared expert (id 384) holds 16384
    # routes, the most loaded segment, and is the last expert in the list
    layer, case, _ = _config_case("a16w4_385", 16384)
    experts, tok = _prefill_experts(case, layer)
    assert 384 in experts
    experts = sorted(set(experts) | {383})
    print(compare(case, layer, True, tokens=tok, whole_experts=experts))


def test_zipf_prefill_stress(cuda_lib):
    layer = layer_for("backbone")
    w = __import__("moe_check").weights_for("backbone")
    case = mi.make_case("backbone", 16384, routing="zipf", weights=w)
    counts = np.bincount(case.topk_ids.reshape(-1).numpy(), minlength=384)
    assert counts.max() > 20 * np.median(counts)
    experts, tok = _prefill_experts(case, layer)
    print(compare(case, layer, False, tokens=tok, whole_experts=experts))
