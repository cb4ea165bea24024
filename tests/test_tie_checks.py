"""The helpers the GPU block test uses where floating point decides an H code, checked on CPU: the per-token oracle
hands out the same H as its grouped path; check_h_decisions accepts the oracle's own decisions and a flip made at a
genuine near tie, and rejects a flip away from a tie, a flip by 2 and a scale moved by two fp16 steps;
tie_correction accounts a changed code exactly (the oracle's own down and combine on the changed H agree with the
oracle's output plus the correction)."""
import numpy as np
import pytest

import oracle
from quantized_routed_expert_smoe_gb300 import synth

from helpers import check_h_decisions, tie_correction


@pytest.fixture(scope="module")
def tiny():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_layer(cfg)
    return cfg, inp, oracle.layer_tokens_h(inp, np.arange(cfg.T))


def test_per_token_h_equals_grouped_h(tiny):
    cfg, inp, (y, ids, w, h, hc, hs) = tiny
    g = oracle.group(ids, cfg.E)
    xc, xs = oracle.quantize_q8(inp["x"])
    gu = oracle.gateup(xc, xs, g["src"], g["offsets"], inp["wgu_c"], inp["wgu_s"], cfg.H, cfg.F)
    c, s = oracle.swiglu_requant(gu, cfg.F)
    assert np.array_equal(c[g["slot"]].reshape(hc.shape), hc)
    assert np.array_equal(s[g["slot"]].reshape(hs.shape), hs)
    # the codes are the q8 rule applied to the handed-out h
    c2, s2 = oracle.quantize_q8(h.reshape(-1, cfg.F))
    assert np.array_equal(c2.reshape(hc.shape), hc) and np.array_equal(s2.reshape(hs.shape), hs)
    assert np.allclose(y, oracle.layer(inp), rtol=0, atol=1e-12 * np.abs(y).max())


def _flip_at(h, hc, hs, t, k, j, towards_tie):
    """A copy of (h, hc) in which code (t, k, j) moved by one towards a .5 tie that h is placed next to (or, with
    towards_tie False, by one while h stays where it is)."""
    h, hc = h.copy(), hc.copy()
    d = float(hs[t, k, j // 32].view(np.float16))
    q = int(hc[t, k, j])
    q = q if abs(q) < 126 else q - np.sign(q) * 2
    hc[t, k, j] = q
    if towards_tie:
        h[t, k, j] = np.float32((q + 0.5 - 1e-6) * d)   # the oracle's h just below the tie between q and q + 1
    else:
        h[t, k, j] = np.float32(q * d)                  # right on q: no tie anywhere near
    g = hc.copy()
    g[t, k, j] = q + 1
    return h, hc, g


def test_check_h_decisions(tiny):
    cfg, inp, (y, ids, w, h, hc, hs) = tiny
    sf, cf = check_h_decisions(hc, hs, h, hc, hs)
    assert not sf.any() and not cf.any()
    h2, hc2, g = _flip_at(h, hc, hs, 3, 1, 70, towards_tie=True)
    sf, cf = check_h_decisions(g, hs, h2, hc2, hs)
    assert cf.sum() == 1 and cf[3, 1, 70]
    h2, hc2, g = _flip_at(h, hc, hs, 3, 1, 70, towards_tie=False)
    with pytest.raises(AssertionError, match="away from a .5 tie"):
        check_h_decisions(g, hs, h2, hc2, hs)
    g = hc.copy()
    g[5, 0, 9] = np.int8(int(hc[5, 0, 9]) + (2 if hc[5, 0, 9] < 100 else -2))
    with pytest.raises(AssertionError, match="more than 1"):
        check_h_decisions(g, hs, h, hc, hs)
    s2 = hs.copy()
    s2[2, 1, 1] = (s2[2, 1, 1].view(np.float16) * np.float16(1.01)).view(np.uint16)
    with pytest.raises(AssertionError, match="fp16 step|midpoint"):
        check_h_decisions(hc, s2, h, hc, hs)


def test_tie_correction_is_exact(tiny):
    cfg, inp, (y, ids, w, h, hc, hs) = tiny
    assert not tie_correction(hc, hs, hc, hs, ids, w, inp["wd_c"], inp["wd_s"]).any()
    g = hc.copy()
    g[7, 0, 33] += 1 if g[7, 0, 33] < 127 else -1
    g[40, 1, 127] += 1 if g[40, 1, 127] < 127 else -1
    s2 = hs.copy()
    s2[40, 1, 2] = np.nextafter(hs[40, 1, 2].view(np.float16), np.float16(np.inf)).view(np.uint16)
    corr = tie_correction(g, s2, hc, hs, ids, w, inp["wd_c"], inp["wd_s"])
    # the oracle's own down and combine, fed the changed H in routed-row order
    grp = oracle.group(ids, cfg.E)
    T, K, F = hc.shape
    hc_rows = np.empty((T * K, F), np.int8)
    hs_rows = np.empty((T * K, F // 32), np.uint16)
    hc_rows[grp["slot"]] = g.reshape(T * K, F)
    hs_rows[grp["slot"]] = s2.reshape(T * K, F // 32)
    dm = oracle.down(hc_rows, hs_rows, grp["offsets"], inp["wd_c"], inp["wd_s"], cfg.H, cfg.F)
    y2 = oracle.combine(dm, grp["slot"], w, T, K, cfg.H)
    assert np.abs(corr).max() > 0
    assert np.allclose(y2, y + corr, rtol=0, atol=1e-12 * np.abs(y).max())
    assert np.array_equal(np.nonzero(np.abs(corr).max(axis=1))[0], [7, 40])
