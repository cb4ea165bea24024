"""Pins of the oracle's router projection (page "src/prefill/prefill.cpp", Prefill::run, MoE half: the router's BF16
projection of the hidden state with its low part; reading: xh = bf16_rne(x), xl = bf16_rne(x - xh), logits =
W_r . (xh + xl) in double), against exact rational arithmetic, bounds from the format, one-hot weights and numpy."""
from fractions import Fraction

import numpy as np

import oracle
from quantized_routed_expert_smoe_gb300 import synth


def as_f(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_bf16_split_worked_ties_and_exact_values():
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1.5, -0.375, 2 ** -130, 65504.0], np.float32)
    xh, xl = oracle.bf16_split(x)
    h, l = as_f(xh), as_f(xl)
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: to the even neighbour 1, remainder 2^-8
    assert h[1] == 1.0 and l[1] == 2 ** -8
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even): up, remainder -2^-8
    assert h[2] == 1 + 2 ** -6 and l[2] == -(2 ** -8)
    # values with at most 8 significant bits are their own high part (the subnormal 2^-130 too)
    for i in (0, 3, 4, 5):
        assert h[i] == x[i] and l[i] == 0.0


def test_bf16_split_reconstructs_within_the_format_bound():
    x = synth.make_rows(64, 256, seed=21).ravel()
    xh, xl = oracle.bf16_split(x)
    h, l = as_f(xh).astype(np.float64), as_f(xl).astype(np.float64)
    xd = x.astype(np.float64)
    # |x - xh| <= half an ulp of 8 significant bits, and xl rounds that remainder again to 8 bits
    assert np.all(np.abs(xd - h) <= 2.0 ** -8 * np.abs(xd))
    assert np.all(np.abs(xd - h - l) <= 2.0 ** -16 * np.abs(xd) + 1e-45)
    # exact check on a few values with rational arithmetic
    for i in range(0, x.size, 997):
        err = Fraction(float(x[i])) - Fraction(float(h[i])) - Fraction(float(l[i]))
        assert abs(err) <= Fraction(1, 2 ** 16) * abs(Fraction(float(x[i])))


def test_router_logits_match_numpy_and_one_hot_rows():
    cfg = synth.CONFIGS["tiny"]
    x = synth.make_layer(cfg)["x"]
    wr = synth.make_router(cfg)
    lg = oracle.router_logits(x, wr)
    xh, xl = oracle.bf16_split(x)
    a = as_f(xh).astype(np.float64) + as_f(xl).astype(np.float64)
    assert np.allclose(lg, a @ as_f(wr).astype(np.float64).T, rtol=1e-12, atol=1e-13)
    # router row e = 1 at column c(e): logit e = xh + xl at that column (an index mix-up picks another one)
    E, H = wr.shape
    cols = (np.arange(E) * 7) % H
    one = np.zeros((E, H), np.uint16)
    one[np.arange(E), cols] = 0x3F80  # bf16 1.0
    assert np.array_equal(oracle.router_logits(x, one), a[:, cols])


def test_router_route_orders_by_the_projection():
    # router rows c_e * e_0 (c_e exact in bf16): every logit is c_e * a[t] with a = xh + xl of x[t][0], so the top-K
    # follow c_e's order (its reverse for a negative a[t]), and the two equal c_e tie to the lower id
    T, H, E, K = 6, 64, 32, 4
    x = synth.make_rows(T, H, seed=22)
    c = (np.arange(E, dtype=np.float32) - 16.0) / 8.0  # multiples of 1/8: exact in bf16
    c[9] = c[7]
    wr = np.zeros((E, H), np.uint16)
    wr[:, 0] = (c.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(as_f(wr[:, 0]), c)
    xh, xl = oracle.bf16_split(x[:, :1])
    a = as_f(xh)[:, 0].astype(np.float64) + as_f(xl)[:, 0].astype(np.float64)
    ids, w, _ = oracle.router_route(x, wr, K)
    for t in range(T):
        logit = (c.astype(np.float64) * a[t]).astype(np.float32)
        want = sorted(range(E), key=lambda e: (-logit[e], e))[:K]
        assert list(ids[t]) == want
        assert abs(w[t].sum() - 1.0) < 1e-12
