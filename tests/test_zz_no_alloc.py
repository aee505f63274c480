"""fused_moe_a8w4_noalloc: the fused call for callers that cannot allocate.

Some callers of this library cannot hand it a workspace - for instance a
plugin living inside an engine that owns all device memory and gives its
plugins no allocator, or a path that may not call a device allocator at
all. For them the library keeps one static device scratch array of
NOALLOC_WORKSPACE_BYTES. These tests call that entry point through the C ABI
twice in a row (the array keeps the previous call's contents, so the second
call also checks that nothing depends on it starting clean) and compare its
output with the ordinary fused_moe_a8w4 on the same inputs, within the
parity tolerance the other tests use. They also check that a shape whose
scratch would not fit is refused before any launch.

The file name makes pytest collect it last; it passes on its own in a fresh
process as well as after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from moe_check import ATOL, RTOL, layer_for, weights_for

pytestmark = pytest.mark.gpu


def _inputs(name, M, variant=0):
    case = mi.make_case(name, M, variant=variant, weights=weights_for(name))
    return case.x.cuda(), case.topk_ids.cuda(), case.topk_weights.cuda()


def _check_close(got, want):
    g = got.float().cpu().numpy()
    w = want.float().cpu().numpy()
    err = np.abs(g - w)
    assert (err <= ATOL + RTOL * np.abs(w)).all(), float(err.max())
    assert np.isfinite(g).all()


@pytest.mark.parametrize("name,Ms", [("draft", (5, 3)), ("backbone", (6, 12))])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, name, Ms):
    layer = layer_for(name)
    for M in Ms:                                   # two calls in a row on the shared scratch
        assert layer.workspace_bytes(M, mi.SHAPES[name].topk) <= m.NOALLOC_WORKSPACE_BYTES
        x, ids, w = _inputs(name, M)
        want = m.fused_moe_a8w4(x, ids, w, layer.w1, layer.w1_scale, layer.w2, layer.w2_scale,
                                layer.E, layer.Ip)
        out = torch.full((M, layer.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        got = m.fused_moe_a8w4_noalloc(x, ids, w, layer.w1, layer.w1_scale, layer.w2,
                                       layer.w2_scale, layer.E, layer.Ip, out=out)
        torch.cuda.synchronize()
        _check_close(got, want)
        # the device status of the call just made, read from the library's
        # scratch: no wait gave up, and the padded route count is the one
        # the workspace entry point computed
        code, padded = m.moe_noalloc_status()
        assert code == 0
        lay = layer.workspace_layout(M, mi.SHAPES[name].topk)
        assert 0 < padded <= lay["p_max"] and padded % lay["block_m"] == 0


def test_noalloc_refuses_shapes_that_do_not_fit(cuda_lib):
    layer = layer_for("backbone")
    M = 768
    assert layer.workspace_bytes(M, 6) > m.NOALLOC_WORKSPACE_BYTES
    x, ids, w = _inputs("backbone", M)
    out = torch.zeros(M, layer.H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoeError) as exc:
        m.fused_moe_a8w4_noalloc(x, ids, w, layer.w1, layer.w1_scale, layer.w2, layer.w2_scale,
                                 layer.E, layer.Ip, out=out)
    assert exc.value.code == 3                     # MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out.float() == 0).all()                # nothing was launched
