"""The expert products in the q8-and-descriptor form (smoe_experts_gateup_q8 / smoe_experts_down_q8, GPU, through the
C ABI): per-token q8 activations with the routed rows' token indices, and each expert's 2-bit weights behind its own
pointer pair (here: separately allocated tensors, so that nothing relies on the experts being contiguous).  Checked
against the oracle per element (the same bound as the other product tests) and bit-for-bit against the operand-form
calls on the same inputs; a null descriptor is reported in the tile list's kernel status and zeroes that expert."""
import numpy as np
import pytest

import oracle
from quantized_routed_expert_smoe_gb300 import synth

from helpers import deq_a, deq_w, tile_list, to_operand

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_smoe_gb300 import build, binding
    build.build()
    binding.load_library()
    binding.device_check()
    return binding


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def tiles_dev(B, offsets, n, E):
    tl = tile_list(offsets, B.TILE_ROWS)
    raw = np.zeros(B.tiles_bytes(n, E) // 4, np.int32)
    raw[0], raw[2] = tl.shape[0], n
    raw[4:4 + tl.size] = tl.ravel()
    return dev(raw)


def per_expert(B, codes, scales):
    """each expert's matrix in its own allocation (with a gap between them), and the descriptor array"""
    keep = []
    for e in range(codes.shape[0]):
        pad = torch.empty(4096, dtype=torch.uint8, device="cuda")  # keeps the experts apart in memory
        keep.append((dev(codes[e]), dev(np.ascontiguousarray(scales[e]).view(np.int16)), pad))
    return B.q2_descriptors([(c, s) for c, s, _ in keep]), keep


@pytest.mark.parametrize("shape", [(200, 256, 6, 3, 128), (150, 384, 5, 2, 192)])
def test_q8_entry_matches_oracle_and_operand_form(B, shape):
    T, H, E, K, F = shape
    inp = synth.make_custom(T, H, E, K, F, seed=31 + T)
    ids, _ = oracle.route(inp["logits"], K)
    g = oracle.group(ids, E)
    n = T * K
    xc, xs = oracle.quantize_q8(inp["x"])
    wgu, keep_gu = per_expert(B, inp["wgu_c"], inp["wgu_s"])
    wd, keep_d = per_expert(B, inp["wd_c"], inp["wd_s"])
    work = torch.empty(B.experts_q8_work_bytes(n, E, H, F), dtype=torch.uint8, device="cuda")
    # gate/up
    tiles = tiles_dev(B, g["offsets"], n, E)
    gu = torch.full((n, 2 * F), float("nan"), dtype=torch.float32, device="cuda")
    B.smoe_experts_gateup_q8(dev(xc), dev(xs.view(np.int16)), dev(g["src"]), tiles, n, E, wgu, H, F, work, gu)
    assert host(tiles)[3] == 0
    got = host(gu)
    want = oracle.gateup(xc, xs, g["src"], g["offsets"], inp["wgu_c"], inp["wgu_s"], H, F)
    A = deq_a(xc, xs)[g["src"]]
    for e in range(E):
        r0, r1 = int(g["offsets"][e]), int(g["offsets"][e + 1])
        mag = np.abs(A[r0:r1]) @ np.abs(deq_w(inp["wgu_c"][e], inp["wgu_s"][e], H)).T
        assert np.all(np.abs(got[r0:r1] - want[r0:r1]) <= 2e-6 * mag + 1e-30), e
    # the operand-form call on the same inputs gives the same bits
    gu2 = torch.full((n, 2 * F), float("nan"), dtype=torch.float32, device="cuda")
    src = g["src"].astype(np.int64)
    B.smoe_experts_gateup(dev(to_operand(xc[src], xs[src])), tiles_dev(B, g["offsets"], n, E), n, E,
                          B.pack_weights(inp["wgu_c"], inp["wgu_s"]), H, F, gu2)
    assert np.array_equal(host(gu2), got)
    # down, from the oracle's H
    hc, hs = oracle.swiglu_requant(want, F)
    tiles = tiles_dev(B, g["offsets"], n, E)
    dm = torch.full((n, H), float("nan"), dtype=torch.float32, device="cuda")
    B.smoe_experts_down_q8(dev(hc), dev(hs.view(np.int16)), tiles, n, E, wd, H, F, work, dm)
    assert host(tiles)[3] == 0
    got_d = host(dm)
    want_d = oracle.down(hc, hs, g["offsets"], inp["wd_c"], inp["wd_s"], H, F)
    Hd = deq_a(hc, hs)
    for e in range(E):
        r0, r1 = int(g["offsets"][e]), int(g["offsets"][e + 1])
        mag = np.abs(Hd[r0:r1]) @ np.abs(deq_w(inp["wd_c"][e], inp["wd_s"][e], F)).T
        assert np.all(np.abs(got_d[r0:r1] - want_d[r0:r1]) <= 2e-6 * mag + 1e-30), e
    dm2 = torch.full((n, H), float("nan"), dtype=torch.float32, device="cuda")
    B.smoe_experts_down(dev(to_operand(hc, hs)), tiles_dev(B, g["offsets"], n, E), n, E,
                        B.pack_weights(inp["wd_c"], inp["wd_s"]), H, F, dm2)
    assert np.array_equal(host(dm2), got_d)


def test_q8_entry_null_descriptor(B):
    T, H, E, K, F = 64, 256, 4, 2, 128
    inp = synth.make_custom(T, H, E, K, F, seed=77)
    ids, _ = oracle.route(inp["logits"], K)
    g = oracle.group(ids, E)
    n = T * K
    xc, xs = oracle.quantize_q8(inp["x"])
    wgu, keep = per_expert(B, inp["wgu_c"], inp["wgu_s"])
    ptrs = wgu.clone()
    ptrs[2 * 2] = 0  # expert 2's codes pointer
    work = torch.empty(B.experts_q8_work_bytes(n, E, H, F), dtype=torch.uint8, device="cuda")
    tiles = tiles_dev(B, g["offsets"], n, E)
    gu = torch.full((n, 2 * F), float("nan"), dtype=torch.float32, device="cuda")
    B.smoe_experts_gateup_q8(dev(xc), dev(xs.view(np.int16)), dev(g["src"]), tiles, n, E, ptrs, H, F, work, gu)
    assert host(tiles)[3] == B.SMOE_ERR_ARG
    got = host(gu)
    r0, r1 = int(g["offsets"][2]), int(g["offsets"][3])
    assert r1 > r0 and np.all(got[r0:r1] == 0.0)
    want = oracle.gateup(xc, xs, g["src"], g["offsets"], inp["wgu_c"], inp["wgu_s"], H, F)
    other = np.r_[0:r0, r1:n]
    assert np.allclose(got[other], want[other], rtol=0, atol=1e-3 * np.abs(want).max())
