"""Property checks of the oracle over random ragged shapes (hypothesis, CPU): the grouped block equals the brute-force
route (every weight and q8 value dequantised to double, plain dot products, no grouping), the per-token sampled
path equals the whole chunk, and the routing weights sum to one and never increase with k."""
import numpy as np
import pytest

import oracle
from quantized_routed_expert_smoe_gb300 import synth

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


shapes = st.tuples(
    st.integers(1, 24),                    # T
    st.sampled_from([32, 64, 96]),         # H
    st.integers(1, 9),                     # E
    st.integers(1, 4),                     # K (clipped to E)
    st.sampled_from([32, 64]),             # F
    st.integers(0, 2 ** 31 - 1),           # seed
)


@settings(max_examples=25, deadline=None)
@given(shapes)
def test_grouped_block_equals_bruteforce(shape):
    T, H, E, K, F, seed = shape
    K = min(K, E)
    inp = synth.make_custom(T, H, E, K, F, seed)
    y = oracle.layer(inp)
    yb = oracle.layer_bruteforce(inp)
    scale = max(np.abs(yb).max(), 1e-300)
    assert np.abs(y - yb).max() <= 1e-9 * scale
    toks = np.arange(0, T, 3)
    yt, ids, w = oracle.layer_tokens(inp, toks)
    assert np.abs(yt - y[toks]).max() <= 1e-12 * scale
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 1e-15)
    assert all(len(set(r.tolist())) == K for r in ids)


@settings(max_examples=25, deadline=None)
@given(st.integers(1, 40), st.sampled_from([32, 64, 256]), st.integers(0, 2 ** 31 - 1), st.floats(1e-3, 1e3))
def test_q8_bound_and_range(rows, cols, seed, scale):
    x = synth.make_rows(rows, cols, seed, scale=scale)
    c, s = oracle.quantize_q8(x)
    d = s.view(np.float16).astype(np.float64).repeat(32, axis=1)
    err = np.abs(x.astype(np.float64) - d * c)
    # half a step of the block's scale, plus the scale's own fp16 rounding carried by up to 127 steps
    assert np.all(err <= d / 2 + np.abs(x) * 2.0 ** -10 + 1e-30)
    assert np.abs(c.astype(np.int32)).max() <= 127
