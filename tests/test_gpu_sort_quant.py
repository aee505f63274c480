"""GPU parity of the route sort, the activation quantisation and the weight
scale prepack against the oracle / the documented layout (bit-exact)."""
import numpy as np
import pytest
import torch

import block_scaled_moe_sort_gb300 as m
import moe_inputs as mi
from oracle import moe as om
from oracle import mx_formats as mx

pytestmark = pytest.mark.gpu


def _sort_case(M, k, E, E_route, mode, seed):
    g = mi._gen(seed)
    shp = mi.small_shape(E=E, topk=k, E_route=E_route)
    return mi.make_routing(shp, M, g, mode)


CASES = [
    # M, topk, E, E_route, routing
    (0, 6, 384, 384, "uniform"),
    (1, 6, 96, 384, "uniform"),     # expert-parallel: most routes dropped
    (5, 3, 128, 128, "uniform"),
    (31, 6, 384, 384, "uniform"),
    (257, 6, 384, 384, "uniform"),
    (768, 6, 384, 384, "hot"),
    (4096, 6, 96, 384, "uniform"),
    (16384, 6, 384, 384, "zipf"),
    (16384, 7, 385, 385, "uniform"),
    (3000, 16, 512, 512, "uniform"),
]


@pytest.mark.parametrize("bm", [16, 64, 128, 256])
@pytest.mark.parametrize("M,k,E,E_route,mode", CASES)
def test_sort_bit_exact(cuda_lib, M, k, E, E_route, mode, bm):
    ids, w = _sort_case(M, k, E, E_route, mode, seed=M * 7 + k + bm)
    if M >= 3:
        ids[2, 0] = -5  # an invalid id is dropped, not faulted
    res = m.moe_sort(ids.cuda(), w.cuda(), E, bm)
    torch.cuda.synchronize()
    ref = om.moe_sort(ids, w, E, bm)
    P = ref.num_padded
    assert int(res["num_padded"].item()) == P
    sr = res["sorted_route"].cpu().numpy()
    assert np.array_equal(sr[:P], ref.sorted_route)
    assert (sr[P:] == M * k).all()
    sw = res["sorted_w"].cpu().numpy()
    assert np.array_equal(sw[:P].view(np.uint32), ref.sorted_w.view(np.uint32))
    assert (sw[P:] == 0).all()
    be = res["block_expert"].cpu().numpy()
    assert np.array_equal(be[:P // bm], ref.block_expert)
    assert (be[P // bm:] == -1).all()
    assert np.array_equal(res["expert_off"].cpu().numpy(), ref.expert_off)
    assert np.array_equal(res["route_pos"].cpu().numpy(), ref.route_pos)


def _quant_inputs():
    g = mi._gen(77)
    x = torch.randn(300, 5120, generator=g)
    x[0] = 0.0                                           # all-zero blocks
    x[1, :32] = 448.0                                    # amax exactly on the limit
    x[2] *= 1e-38                                        # bfloat16 subnormals
    x[3] *= 3e38 / 6                                     # near the top of the range
    x[4, 5] = -0.0
    x[5] = torch.randn(5120, generator=g) * torch.exp(torch.randn(5120, generator=g) * 8)
    x[6, 0:32] = torch.tensor([1.0] + [2.0 ** -20] * 31)  # tiny values under a big amax
    return x.to(torch.bfloat16)


def test_quant_act_bit_exact(cuda_lib):
    x = _quant_inputs()
    q, s = m.moe_quant_act_mx(x.cuda())
    torch.cuda.synchronize()
    rq, rs = mx.quant_mxfp8(x.to(torch.float64).numpy())
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("M,K", [(1, 32), (7, 640), (33, 2304), (1025, 5120)])
def test_quant_act_shapes(cuda_lib, M, K):
    g = mi._gen(M + K)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    q, s = m.moe_quant_act_mx(x.cuda())
    rq, rs = mx.quant_mxfp8(x.to(torch.float64).numpy())
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 256, 640), (2, 1280, 5120)])
def test_prepack_scale_layout(cuda_lib, E, N, K):
    g = np.random.default_rng(E * N + K)
    s = g.integers(0, 256, size=(E, N, K // 32), dtype=np.uint8)
    got = m.moe_prepack_scales_mx(torch.from_numpy(s).cuda()).cpu().numpy()
    e, n, i = np.meshgrid(np.arange(E), np.arange(N), np.arange(K // 32), indexing="ij")
    atom = (e * (N // 128) + n // 128) * (K // 128) + i // 4
    r = n % 128
    off = atom * 512 + (r % 32) * 16 + (r // 32) * 4 + i % 4
    want = np.zeros(E * N * K // 32, dtype=np.uint8)
    want[off.reshape(-1)] = s.reshape(-1)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("E,N,K", [(2, 256, 256), (1, 128, 5120)])
def test_a16w4_dequant_exact(cuda_lib, E, N, K):
    # The a16w4 GEMMs' weight dequantisation (a16w4 prepack + the converter's
    # rotations, masks and scale multiplication, run by the same device
    # routine) against the OCP MXFP4 definition: every byte of codes and
    # every finite E8M0 scale 0..254, exact wherever the product is a BF16
    # number and infinite past the BF16 range; the NaN scale 255 gives no
    # finite value for a nonzero code.
    g = np.random.default_rng(E * N + K)
    w = g.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    w.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)
    s = (np.arange(E * N * (K // 32)) % 256).astype(np.uint8).reshape(E, N, K // 32)
    s = np.ascontiguousarray(s[:, g.permutation(N), :])
    wp = m.moe_prepack_weights_a16w4(torch.from_numpy(w).cuda())
    sp = m.moe_prepack_scales_mx(torch.from_numpy(s).cuda())
    got = m.moe_dequant_a16w4(wp, sp, E, N, K).cpu().to(torch.float64).numpy()
    finite_scale = np.repeat(s != 255, 32, axis=-1)
    want = mx.bf16_round(np.where(finite_scale, mx.dequant_mxfp4(w, np.where(s == 255, 0, s)), 0))
    assert np.array_equal(got[finite_scale], want[finite_scale])
    # the sign of zero as well (code 8 is -0)
    assert np.array_equal(np.signbit(got[finite_scale]), np.signbit(want[finite_scale]))
    codes = mx.unpack_e2m1(w)
    nan_scale = ~finite_scale & ((codes & 7) != 0)
    assert not np.isfinite(got[nan_scale]).any()
    # the a8w4 prepack is the plain tile copy; the a16w4 one moves bits only
    # inside each 32-bit word (same bytes per tile row, same popcount per word)
    plain = m.moe_prepack_weights_mx(torch.from_numpy(w).cuda()).cpu().numpy().view(np.uint32)
    a16 = wp.cpu().numpy().view(np.uint32)
    pc = lambda a: np.unpackbits(a.view(np.uint8)).reshape(-1, 32).sum(axis=1)
    assert np.array_equal(pc(plain), pc(a16)) and not np.array_equal(plain, a16)
