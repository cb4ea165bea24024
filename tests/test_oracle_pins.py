"""Pins of the CPU oracle against facts that do not come from the oracle itself (CPU only).

Each test checks one oracle function against something fixed independently of its code: a library routine
(numpy's IEEE half conversion, numpy's stable sort, numpy matmul, scipy's logistic function), a closed form, an
invariant of the definition, or a hand-worked case.  Together they are chosen so that a plausible slip anywhere in
the oracle (a dropped term, a wrong sign or offset, a swapped gate/up, a transposed operand, round-half-even in
place of half-away, an unstable sort, a wrong tie rule) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from quantized_routed_expert_smoe_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ------------------------------------------------------------------------------------------------ fp16 conversion
def test_f2h_matches_numpy_ieee_half():
    rng = np.random.default_rng(123)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, 6.1035156e-05, 5.9604645e-08, 2.9802322e-08,
                  2.9802326e-08, 8.940697e-08, 1e-9, 0.5, 1.0 / 3.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11],
                 np.float32),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f2h(v) for v in vals], np.uint16)
    assert np.array_equal(got, want)
    back = np.array([oracle.h2f(h) for h in want], np.float32)
    assert np.array_equal(back, want.view(np.float16).astype(np.float32))


# ------------------------------------------------------------------------------------------------ route
def _numpy_topk(logits, K):
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        ids[t] = order[:K]
    return ids


def test_route_ids_match_library_sort_and_weights_match_full_softmax():
    inp = synth.make_layer(synth.CONFIGS["tiny"], with_weights=False)
    K = 2
    ids, w = oracle.route(inp["logits"], K)
    assert np.array_equal(ids, _numpy_topk(inp["logits"], K))
    p = scipy.special.softmax(inp["logits"].astype(np.float64), axis=1)  # full softmax first
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_full_size_shape_against_library_sort():
    inp = synth.make_layer(synth.CONFIGS["t1024"], with_weights=False)
    lg = inp["logits"][:200]
    ids, w = oracle.route(lg, 10)
    assert np.array_equal(ids, _numpy_topk(lg, 10))
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 1e-12)


def test_route_ties_go_to_lower_expert_id():
    lg = np.zeros((3, 8), np.float32)
    lg[0] = [1, 3, 3, 0, 3, 2, 2, 0]      # three-way tie at the top
    lg[1] = [5, 5, 5, 5, 5, 5, 5, 5]      # everything tied
    lg[2] = [0, 0, 0, 0, 0, 0, 7, 0]
    ids, w = oracle.route(lg, 4)
    assert ids[0].tolist() == [1, 2, 4, 5]
    assert ids[1].tolist() == [0, 1, 2, 3]
    assert ids[2].tolist() == [6, 0, 1, 2]
    np.testing.assert_allclose(w[1], [0.25] * 4, rtol=0, atol=1e-15)
    e3 = np.exp(-1.0)
    np.testing.assert_allclose(w[0], np.array([1, 1, 1, e3]) / (3 + e3), rtol=1e-14)


def test_route_k_equals_e_and_k_one():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((7, 6)).astype(np.float32)
    ids, w = oracle.route(lg, 6)
    np.testing.assert_allclose(w, np.sort(scipy.special.softmax(lg.astype(np.float64), 1), 1)[:, ::-1], rtol=1e-12)
    ids1, w1 = oracle.route(lg, 1)
    assert np.array_equal(ids1[:, 0], np.argmax(lg, 1)) and np.all(w1 == 1.0)


# ------------------------------------------------------------------------------------------------ group
def _check_group(ids, E, g):
    T, K = ids.shape
    flat = ids.ravel()
    n = flat.size
    order = np.argsort(flat, kind="stable")          # the library's stable sort
    assert np.array_equal(g["counts"], np.bincount(flat, minlength=E))
    assert g["offsets"][0] == 0 and np.array_equal(np.diff(g["offsets"]), g["counts"])
    assert np.array_equal(g["src"], (order // K).astype(np.int32))
    slot = np.empty(n, np.int32)
    slot[order] = np.arange(n)
    assert np.array_equal(g["slot"], slot)
    # every row of expert e holds a pair routed to e, in ascending pair order
    for e in range(E):
        r0, r1 = int(g["offsets"][e]), int(g["offsets"][e + 1])
        pairs = order[r0:r1]
        assert np.all(flat[pairs] == e) and np.all(np.diff(pairs) > 0)


@pytest.mark.parametrize("cfg", ["tiny", "t1024", "skew8192"])
def test_group_matches_stable_library_sort(cfg):
    c = synth.CONFIGS[cfg]
    inp = synth.make_layer(c, with_weights=False)
    ids, _ = oracle.route(inp["logits"], c.K)
    _check_group(ids, c.E, oracle.group(ids, c.E))


def test_group_edge_cases():
    # one expert takes everything (several tiles), unrouted experts, ragged tails
    ids = np.zeros((300, 2), np.int32)
    ids[:, 1] = 3
    ids[7, 0] = 5
    g = oracle.group(ids, 8)
    _check_group(ids, 8, g)
    assert g["counts"].tolist() == [299, 0, 0, 300, 0, 1, 0, 0]
    assert g["offsets"].tolist() == [0, 299, 299, 299, 599, 599, 600, 600, 600]
    # the pair of token 7 routed to expert 5 is the only row of expert 5, and its k is 0
    assert g["src"][599] == 7 and g["slot"][14] == 599
    with pytest.raises(ValueError):
        oracle.group(np.array([[0, 8]], np.int32), 8)
    with pytest.raises(ValueError):
        oracle.group(np.array([[-1, 0]], np.int32), 8)


# ------------------------------------------------------------------------------------------------ q8
def test_q8_hand_worked_blocks():
    # block A: amax 127 -> d = 127/127 = 1.0 exactly; codes are roundf(x): halves go AWAY from zero (2.5 -> 3)
    a = np.zeros(32, np.float32)
    a[:10] = [127, -127, 2.5, -2.5, 0.5, -0.5, 1.5, 126.5, 63.49, -0.49]
    # block B: amax 1 -> d = fp16(1/127) = 129/16384 (0x2008); x = 2.5 d is exact, x/d = 2.5 -> 3
    d_b = 129.0 / 16384.0
    b = np.zeros(32, np.float32)
    b[:6] = [1.0, -1.0, 0.5, np.float32(2.5 * d_b), np.float32(-3.5 * d_b), np.float32(0.5 * d_b)]
    # block C: all zero -> d = 0, codes 0;  block D: amax 1e-9 -> amax/127 rounds to fp16 zero -> codes 0
    c = np.zeros(32, np.float32)
    dd = np.zeros(32, np.float32)
    dd[3] = 1e-9
    # block E: amax 1e-5 -> d = one fp16 subnormal unit (2^-24); 1e-5 / 2^-24 = 167.8 clamps to 127
    e = np.zeros(32, np.float32)
    e[0], e[1] = 1e-5, -3e-7
    x = np.stack([a, b, c, dd, e]).astype(np.float32)
    codes, scales = oracle.quantize_q8(x)
    assert scales[:, 0].tolist() == [0x3C00, 0x2008, 0, 0, 0x0001]
    assert codes[0, :10].tolist() == [127, -127, 3, -3, 1, -1, 2, 127, 63, 0]
    assert codes[1, :6].tolist() == [127, -127, 64, 3, -4, 1]
    assert not codes[2].any() and not codes[3].any()
    assert codes[4, :2].tolist() == [127, -5]


def test_q8_bounds_and_full_range_on_random_rows():
    x = synth.make_rows(64, 2560, seed=9, scale=3.0)
    codes, scales = oracle.quantize_q8(x)
    d = scales.view(np.float16).astype(np.float64)
    blocks = x.reshape(64, 80, 32).astype(np.float64)
    q = codes.reshape(64, 80, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    # the scale is amax/127 rounded to fp16 (numpy's IEEE half as the library routine)
    assert np.array_equal(scales, (amax.astype(np.float32) / np.float32(127)).astype(np.float16).view(np.uint16))
    assert np.all(np.abs(q).max(axis=2) == 127)
    err = np.abs(blocks - d[..., None] * q)
    assert np.all(err <= d[..., None] * (0.5 + 1e-6))


# ------------------------------------------------------------------------------------------------ expert products
def _deq_w(codes, scales, cols):
    """Dequantise 2-bit rows with numpy bit operations: w = d * (q - 2)."""
    rows = codes.shape[0]
    q = np.stack([(codes >> (2 * i)) & 3 for i in range(4)], axis=-1).reshape(rows, cols).astype(np.float64)
    d = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)
    return d * (q - 2.0)


def _deq_a(codes, scales):
    return codes.astype(np.float64) * np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)


def test_gateup_and_down_match_numpy_matmul_on_dequantised_values():
    inp = synth.make_custom(T=40, H=128, E=5, K=3, F=96, seed=11)
    ids, w = oracle.route(inp["logits"], 3)
    g = oracle.group(ids, 5)
    xc, xs = oracle.quantize_q8(inp["x"])
    gu = oracle.gateup(xc, xs, g["src"], g["offsets"], inp["wgu_c"], inp["wgu_s"], 128, 96)
    A = _deq_a(xc, xs)
    for e in range(5):
        r0, r1 = g["offsets"][e], g["offsets"][e + 1]
        W = _deq_w(inp["wgu_c"][e], inp["wgu_s"][e], 128)
        np.testing.assert_allclose(gu[r0:r1], A[g["src"][r0:r1]] @ W.T, rtol=1e-12, atol=1e-12)
    hc, hs = oracle.swiglu_requant(gu, 96)
    dm = oracle.down(hc, hs, g["offsets"], inp["wd_c"], inp["wd_s"], 128, 96)
    Hd = _deq_a(hc, hs)
    for e in range(5):
        r0, r1 = g["offsets"][e], g["offsets"][e + 1]
        W = _deq_w(inp["wd_c"][e], inp["wd_s"][e], 96)
        np.testing.assert_allclose(dm[r0:r1], Hd[r0:r1] @ W.T, rtol=1e-12, atol=1e-12)


def test_all_codes_two_give_exact_zero():
    inp = synth.make_custom(T=16, H=64, E=3, K=2, F=64, seed=3)
    inp["wgu_c"][:] = 0b10101010
    y = oracle.layer(inp)
    assert np.all(y == 0.0)
    inp = synth.make_custom(T=16, H=64, E=3, K=2, F=64, seed=3)
    inp["wd_c"][:] = 0b10101010
    assert np.all(oracle.layer(inp) == 0.0)


def test_constant_row_closed_form():
    # x = v everywhere: every block has amax v, d_a = fp16(v/127) and every code is 127; weight codes all 3
    # (q - 2 = 1) with one common d_w: g_j = u_j = (H/32) * d_w * d_a * 32 * 127 for every j.
    H, F, v = 256, 64, 0.75
    xc, xs = oracle.quantize_q8(np.full((1, H), v, np.float32))
    assert np.all(xc == 127)
    d_a = float(np.float16(np.float32(v) / np.float32(127)))
    d_w = float(np.float16(0.0125))
    wc = np.full((1, 2 * F, H // 4), 0xFF, np.uint8)
    ws = np.full((1, 2 * F, H // 32), np.float16(0.0125).view(np.uint16), np.uint16)
    gu = oracle.gateup(xc, xs, np.zeros(1, np.int32), np.array([0, 1], np.int32), wc, ws, H, F)
    want = H * d_w * d_a * 127.0
    assert np.all(gu == want)
    # SwiGLU of the closed form: h = silu(want) * want (scipy's logistic function as the library routine)
    hc, hs = oracle.swiglu_requant(gu, F)
    h = np.float32(want * scipy.special.expit(want) * want)
    assert np.all(hc == 127) and np.all(hs == (h / np.float32(127)).astype(np.float16).view(np.uint16))


def test_swiglu_matches_library_logistic_and_gate_up_order():
    gu = synth.make_gu(64, 128, seed=4, scale=2.0)
    hc, hs = oracle.swiglu_requant(gu, 128)
    g = gu[:, :128].astype(np.float64)
    u = gu[:, 128:].astype(np.float64)
    h = (g * scipy.special.expit(g) * u).astype(np.float32)
    d = hs.view(np.float16).astype(np.float64)
    blocks = h.reshape(64, 4, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    assert np.array_equal(hs, (amax.astype(np.float32) / np.float32(127)).astype(np.float16).view(np.uint16))
    err = np.abs(blocks - d[..., None] * hc.reshape(64, 4, 32))
    assert np.all(err <= d[..., None] * (0.5 + 1e-6))
    # the double and fp32 entry points agree on the same values
    hc2, hs2 = oracle.swiglu_requant(gu.astype(np.float64), 128)
    assert np.array_equal(hc, hc2) and np.array_equal(hs, hs2)


def test_combine_matches_numpy_gather():
    rng = np.random.default_rng(2)
    T, K, H = 30, 3, 64
    n = T * K
    dm = rng.standard_normal((n, H))
    slot = rng.permutation(n).astype(np.int32)
    w = rng.random((T, K))
    y = oracle.combine(dm, slot, w, T, K, H)
    want = np.einsum("tk,tkh->th", w, dm[slot.reshape(T, K)])
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)
    # renormalised weights on equal rows give the row back
    dm2 = np.tile(rng.standard_normal(H), (n, 1))
    w2 = w / w.sum(1, keepdims=True)
    np.testing.assert_allclose(oracle.combine(dm2, slot, w2, T, K, H), np.tile(dm2[0], (T, 1)), rtol=1e-13)


# ------------------------------------------------------------------------------------------------ whole block
def test_layer_equals_bruteforce_and_per_token_path_tiny():
    inp = synth.make_layer(synth.CONFIGS["tiny"])
    y = oracle.layer(inp)
    yb = oracle.layer_bruteforce(inp)
    rms = np.sqrt((y ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(y - yb) <= 1e-9 * rms)
    toks = np.array([0, 5, 17, 63])
    yt, ids, w = oracle.layer_tokens(inp, toks)
    assert np.array_equal(yt, y[toks])


def test_layer_matches_numpy_pipeline_with_ragged_shape():
    # an independent numpy restatement at a ragged shape: numpy sort for the top-K, scipy softmax, numpy matmuls
    T, H, E, K, F = 37, 96, 7, 3, 64
    inp = synth.make_custom(T, H, E, K, F, seed=21)
    y = oracle.layer(inp)
    lg = inp["logits"]
    ids = _numpy_topk(lg, K)
    p = scipy.special.softmax(lg.astype(np.float64), 1)
    sel = np.take_along_axis(p, ids.astype(np.int64), 1)
    w = sel / sel.sum(1, keepdims=True)
    xc, xs = oracle.quantize_q8(inp["x"])
    A = _deq_a(xc, xs)
    want = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            e = ids[t, k]
            g = _deq_w(inp["wgu_c"][e], inp["wgu_s"][e], H) @ A[t]
            h = (g[:F] * scipy.special.expit(g[:F]) * g[F:]).astype(np.float32)[None, :]
            hc, hs = oracle.quantize_q8(h)
            want[t] += w[t, k] * (_deq_w(inp["wd_c"][e], inp["wd_s"][e], F) @ _deq_a(hc, hs)[0])
    rms = np.sqrt((want ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(y - want) <= 1e-9 * rms)


def test_zipf_alpha_constant_matches_golden_file():
    with open(os.path.join(HERE, "golden", "zipf_alpha.json")) as f:
        gold = json.load(f)
    assert synth.ZIPF_ALPHA == gold["alpha"]
    assert abs(gold["top32_share"] - 0.5) <= 0.01
