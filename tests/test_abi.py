"""The C-ABI library loads without a GPU, exports every function the header
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes

import pytest

import block_scaled_moe_sort_gb300 as m
from block_scaled_moe_sort_gb300 import build as b


@pytest.fixture(scope="module")
def L():
    b.build()
    return m.lib()


def test_header_declares_the_entry_points():
    names = m.declared_functions()
    for want in ["moe_sort", "moe_quant_act_mx", "fused_moe_a8w4", "fused_moe_a16w4", "moe_router_topk",
                 "moe_prepack_scales_mx", "fused_moe_workspace_bytes", "moe_status_string",
                 "moe_prepack_weights_a16w4", "moe_dequant_a16w4"]:
        assert want in names


def test_library_exports_every_declared_symbol(L):
    raw = ctypes.CDLL(b.LIB)
    missing = [n for n in m.declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_status_strings(L):
    for code in range(8):
        assert L.moe_status_string(code) != b"unknown status"
    assert L.moe_status_string(3) == b"workspace too small"


FAKE = 0x10000  # an aligned host-side address; never dereferenced on error paths


def _call(L, fn, M=4, H=256, topk=2, E=8, Ip=128, ws=FAKE, ws_bytes=1 << 40, x=FAKE, ids=FAKE,
          w=FAKE, w1=FAKE, w1s=FAKE, w2=FAKE, w2s=FAKE, out=FAKE):
    return getattr(L, fn)(x, ids, w, M, H, topk, w1, w1s, w2, w2s, E, Ip, out, ws, ws_bytes, None)


@pytest.mark.parametrize("fn", ["fused_moe_a8w4", "fused_moe_a16w4"])
def test_fused_rejects_bad_arguments_on_host(L, fn):
    assert _call(L, fn, ws=None) == 1                 # null workspace
    assert _call(L, fn, x=None) == 1                  # null input with M > 0
    assert _call(L, fn, M=-1) == 1
    assert _call(L, fn, H=200) == 2                   # H % 128
    assert _call(L, fn, Ip=96) == 2                   # Ip % 128
    assert _call(L, fn, E=513) == 2
    assert _call(L, fn, topk=17) == 2
    assert _call(L, fn, out=FAKE + 16) == 4           # misaligned
    assert _call(L, fn, ws_bytes=16) == 3             # workspace too small
    assert _call(L, fn, M=0, x=None, ids=None, w=None, out=None) == 0  # empty call, no launch


def test_workspace_size_and_layout(L):
    for a16 in (0, 1):
        n = L.fused_moe_workspace_bytes(96, 5120, 640, 384, 6, a16)
        lay = m.fused_moe_workspace_layout(96, 5120, 640, 384, 6, bool(a16))
        assert n == lay["total_bytes"] > 0
        offs = [lay[k] for k in ("status_off", "expert_off_off", "sorted_route_off",
                                 "sorted_w_off", "block_expert_off", "route_pos_off",
                                 "sort_scratch_off", "act_off",
                                 "inter_off", "acc_off", "split_part_off", "split_cnt_off")]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
        assert lay["block_m"] in (16, 32, 64, 128, 256)
        assert lay["p_max"] % lay["block_m"] == 0
        assert lay["acc_off"] + 96 * 5120 * 4 <= n
    assert L.fused_moe_workspace_bytes(4, 200, 128, 8, 2, 0) == 0


def test_sort_capacity_bound(L):
    # every route plus block_m - 1 pads per possibly non-empty expert
    assert L.moe_sort_max_padded(5, 3, 128, 16) == 15 + 15 * 15
    assert L.moe_sort_max_padded(1000, 6, 384, 64) == -(-(6000 + 384 * 63) // 64) * 64
    assert L.moe_sort_max_padded(0, 6, 384, 64) == 0
    assert L.moe_sort_max_padded(4, 2, 8, 24) == -1   # unsupported block


def test_sort_and_quant_reject_bad_arguments(L):
    args = [FAKE, FAKE, 4, 2, 8, 16, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0, None]
    bad = list(args); bad[5] = 48
    assert L.moe_sort(*bad) == 2
    bad = list(args); bad[4] = 600
    assert L.moe_sort(*bad) == 2
    bad = list(args); bad[6] = None
    assert L.moe_sort(*bad) == 1
    big = list(args); big[2] = 5000                    # 10000 routes need histogram scratch
    assert L.moe_sort_workspace_bytes(5000, 2, 8, 16) == 2 * 8 * 4
    assert L.moe_sort(*big) == 3                       # no workspace given
    assert L.moe_quant_act_mx(FAKE, 4, 100, 100, FAKE, FAKE, None) == 2   # K % 32
    assert L.moe_quant_act_mx(FAKE, 4, 128, 64, FAKE, FAKE, None) == 1    # ldx < K
    assert L.moe_quant_act_mx(FAKE + 8, 4, 128, 128, FAKE, FAKE, None) == 4
    assert L.moe_prepack_scales_mx(FAKE, 2, 100, 256, FAKE, None) == 2
    assert L.moe_prepacked_scale_bytes(2, 256, 512) == 2 * 256 * 16
    for fn in ("moe_prepack_weights_mx", "moe_prepack_weights_a16w4"):
        f = getattr(L, fn)
        assert f(FAKE, 2, 100, 256, FAKE + 0x1000, None) == 2          # N % 128
        assert f(FAKE, 2, 128, 256, FAKE, None) == 1                   # out aliases w
        assert f(FAKE + 8, 2, 128, 256, FAKE + 0x1000, None) == 4
        assert f(None, 2, 128, 256, FAKE, None) == 1
    assert L.moe_dequant_a16w4(FAKE, FAKE, 1, 128, 200, FAKE, None) == 2     # K % 128
    assert L.moe_dequant_a16w4(FAKE, None, 1, 128, 256, FAKE, None) == 1
    assert L.moe_dequant_a16w4(FAKE, FAKE, 1, 128, 256, FAKE + 4, None) == 4


def test_call_config_checks(L):
    import block_scaled_moe_sort_gb300 as mm
    args = [FAKE, FAKE, FAKE, 4, 256, 2, FAKE, FAKE, FAKE, FAKE, 8, 128, FAKE, FAKE, 1 << 40]
    for fn in ("fused_moe_a8w4_cfg", "fused_moe_a16w4_cfg"):
        f = getattr(L, fn)
        for sp in (-1, 3):                                  # split walk: 0, 1 or 2
            bad = mm.MoeCallConfig(0, 0, 0, sp)
            assert f(*args, ctypes.byref(bad), None) == 2
        far = mm.MoeCallConfig(0, 65, 0, 0)                 # lead past 64 tiles
        assert f(*args, ctypes.byref(far), None) == 2
        neg = mm.MoeCallConfig(0, 0, -1, 0)
        assert f(*args, ctypes.byref(neg), None) == 2
        odd = mm.MoeCallConfig(48, 0, 0, 0)                 # not a route block
        assert f(*args, ctypes.byref(odd), None) == 2


def test_device_status_decoding(L):
    assert L.moe_decode_device_status(0) == 0
    assert L.moe_decode_device_status(1) == 6
    assert L.moe_decode_device_status(2) == 7
    assert L.moe_decode_device_status(3) == 6     # a timeout is reported first
    assert L.moe_status_string(7).startswith(b"device-side check")


def test_router_rejects_bad_arguments_on_host(L):
    def call(M=4, E=384, ld=384, k=6, shared=-1, lg=FAKE, ids=FAKE, w=FAKE, n_shared=1):
        return L.moe_router_topk(lg, M, E, ld, k, shared, n_shared, ids, w, None)
    assert call(M=-1) == 1
    assert call(ld=100) == 1                   # ld < E
    assert call(k=0) == 1 and call(E=4, ld=4, k=5) == 1
    assert call(lg=None) == 1
    assert call(E=600, ld=600) == 2            # > 512 experts
    assert call(k=16, shared=384) == 2         # 17 output columns
    assert call(shared=0) == 1                 # a routed expert as the shared one
    assert call(shared=383) == 1
    assert call(shared=512) == 1               # beyond the sort's expert range
    assert call(shared=384, n_shared=0) == 1
    assert call(shared=510, n_shared=3) == 1   # the last id beyond 511
    assert call(k=6, shared=384, n_shared=11) == 2   # 17 columns
    assert call(w=FAKE + 4) == 4               # misaligned
    assert call(M=0, lg=None, ids=None, w=None) == 0   # empty call, no launch


def test_explicit_block_m_validation(L):
    assert L.fused_moe_workspace_bytes_bm(96, 5120, 640, 384, 6, 0, 48) == 0
    for bm in (16, 32, 64, 128, 256):
        n = L.fused_moe_workspace_bytes_bm(96, 5120, 640, 384, 6, 0, bm)
        lay = m.fused_moe_workspace_layout(96, 5120, 640, 384, 6, False, bm)
        assert n == lay["total_bytes"] > 0 and lay["block_m"] == bm
    assert (L.fused_moe_workspace_bytes_bm(96, 5120, 640, 384, 6, 1, 0)
            == L.fused_moe_workspace_bytes(96, 5120, 640, 384, 6, 1))
    args = [FAKE, FAKE, FAKE, 4, 256, 2, FAKE, FAKE, FAKE, FAKE, 8, 128, FAKE, FAKE, 1 << 40]
    assert L.fused_moe_a8w4_bm(*args, 24, None) == 2
    assert L.fused_moe_a16w4_bm(*args, 512, None) == 2


@pytest.mark.parametrize("fn", ["fused_moe_a8w4_gated", "fused_moe_a16w4_gated"])
def test_gated_rejects_bad_arguments_on_host(L, fn):
    def call(M=4, ld=384, E_route=384, topk=6, shared=-1, lg=FAKE, ids=FAKE, w=FAKE, E=384,
             H=256, Ip=128, ws=FAKE, ws_bytes=1 << 40, n_shared=1):
        return getattr(L, fn)(FAKE, lg, ld, E_route, topk, shared, n_shared, M, H, FAKE, FAKE,
                              FAKE, FAKE, E, Ip, FAKE, ids, w, ws, ws_bytes, None)
    assert call(ld=100) == 1                   # ld < E_route
    assert call(topk=0) == 1 and call(topk=385) == 1
    assert call(shared=10) == 1                # a routed expert as the shared one
    assert call(shared=512) == 1
    assert call(shared=384, n_shared=0) == 1 and call(shared=500, n_shared=13) == 1
    assert call(lg=None) == 1 and call(ids=None) == 1 and call(w=None) == 1
    assert call(E_route=600, ld=600) == 2      # > 512 routed experts
    assert call(topk=16, shared=384) == 2      # 17 columns
    assert call(ids=FAKE + 8) == 4             # misaligned
    assert call(ws_bytes=16) == 3              # workspace too small
    assert call(H=200) == 2                    # the fused call's own checks
    assert call(M=0, lg=None, ids=None, w=None) == 0   # empty call, no launch


def test_noalloc_status_rejects_bad_arguments_on_host(L):
    assert L.moe_noalloc_status(None, None) == 1
    assert L.moe_noalloc_status(FAKE + 4, None) == 4


def test_wait_selftest_rejects_bad_arguments_on_host(L):
    assert L.moe_debug_wait_selftest(None, 1000, None) == 1
    assert L.moe_debug_wait_selftest(FAKE, 0, None) == 1
    assert L.moe_debug_wait_selftest(FAKE, 2000000, None) == 1
    assert L.moe_debug_wait_selftest(FAKE + 4, 1000, None) == 4
