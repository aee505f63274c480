"""Device-side failure reporting, tested without a GPU fault: a bounded wait
on a barrier that nothing completes gives up after ~1 ms, sets the timeout
bit of the status word, the kernel returns, and the context stays usable
(a fused call right after it matches the oracle)."""
import pytest

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from moe_check import compare

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 6


def test_bounded_wait_gives_up_and_reports(cuda_lib):
    code, returned = m.moe_debug_wait_selftest(timeout_us=1000)
    assert returned == 1
    assert code == MOE_ERR_TIMEOUT


def test_context_usable_after_a_reported_timeout(cuda_lib):
    assert m.moe_debug_wait_selftest(timeout_us=1000) == (MOE_ERR_TIMEOUT, 1)
    shp = mi.small_shape(H=256, I=128, Ip=128, E=4, topk=2)
    w = mi.make_weights(shp, 3)
    layer = m.MoeLayer(w["w1"], w["w1_scale"], w["w2"], w["w2_scale"])
    case = mi.make_case("small", 9, shape=shp, weights=w)
    compare(case, layer, False)
