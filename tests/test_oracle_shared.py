"""Pins of the oracle's shared expert (the "shared expert and its scalar gate" of page "src/prefill/prefill.cpp",
Prefill::run, MoE half; read as one more expert in the routed experts' form that every token takes, plus
sg = sigmoid(x . w_sg)), each against something other than the oracle's own formula: special values, a reflection
invariant, one-hot inputs, the brute-force (dequantise-everything) route, exact zeros."""
import numpy as np

import oracle
from quantized_routed_expert_smoe_gb300 import synth


def tiny_shared():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_layer(cfg)
    inp.update(synth.make_shared(cfg))
    return inp


def test_shared_gate_special_values_and_reflection():
    x = synth.make_rows(8, 64, seed=3)
    # w_sg = 0: every gate is exactly one half
    assert np.all(oracle.shared_gate(x, np.zeros(64, np.float32)) == 0.5)
    # sigmoid(-z) = 1 - sigmoid(z): negating w_sg reflects every gate
    w = (synth.make_rows(1, 64, seed=4)[0] * 0.1).astype(np.float32)
    a, b = oracle.shared_gate(x, w), oracle.shared_gate(x, -w)
    assert np.allclose(a + b, 1.0, rtol=0, atol=1e-15)
    assert np.all((a > 0) & (a < 1))


def test_shared_gate_one_hot_rows_pick_one_weight():
    # x row i = c e_i: the gate's logit is c * w_sg[i] (a transposed or shifted index would pick another weight)
    H, c = 64, 2.0
    w = (synth.make_rows(1, H, seed=6)[0] * 0.3).astype(np.float32)
    xo = np.zeros((H, H), np.float32)
    xo[np.arange(H), np.arange(H)] = c
    sg = oracle.shared_gate(xo, w)
    assert np.allclose(np.log(sg / (1.0 - sg)), c * w.astype(np.float64), rtol=1e-9, atol=1e-12)


def test_shared_expert_equals_the_bruteforce_one_expert_block():
    # A block with one expert and top-1 routing sends every token to that expert with weight exactly 1, so its output
    # is the shared expert's row.  The brute-force route dequantises every weight and q8 value to double and takes
    # plain dot products (no block structure, no grouping): a different computation of the same numbers.
    inp = tiny_shared()
    T, F = inp["T"], inp["F"]
    s = oracle.shared_expert(inp["x"], inp["sgu_c"], inp["sgu_s"], inp["sd_c"], inp["sd_s"], F)
    one = dict(inp, E=1, K=1, logits=np.zeros((T, 1), np.float32), wgu_c=inp["sgu_c"][None],
               wgu_s=inp["sgu_s"][None], wd_c=inp["sd_c"][None], wd_s=inp["sd_s"][None])
    y1 = oracle.layer_bruteforce(one)
    assert np.abs(s).max() > 0
    assert np.allclose(s, y1, rtol=1e-12, atol=1e-12 * np.abs(y1).max())


def test_zero_shared_weights_leave_the_block_unchanged():
    inp = tiny_shared()
    inp["sgu_c"] = np.full_like(inp["sgu_c"], 0xAA)  # every 2-bit code 2: every gate/up weight 0
    assert np.array_equal(oracle.layer_shared(inp), oracle.layer(inp))


def test_combine_shared_closed_forms():
    rng = np.random.default_rng(5)
    T, K, H = 6, 3, 32
    n = T * K
    dm = rng.standard_normal((n, H))
    slot = rng.permutation(n).astype(np.int32)
    w = rng.random((T, K))
    S = rng.standard_normal((T, H))
    sg = rng.random(T)
    # no routed rows: exactly the gated shared rows
    assert np.array_equal(oracle.combine_shared(np.zeros_like(dm), slot, w, S, sg, T, K, H), sg[:, None] * S)
    # a closed gate: exactly the routed combine
    assert np.array_equal(oracle.combine_shared(dm, slot, w, S, np.zeros(T), T, K, H),
                          oracle.combine(dm, slot, w, T, K, H))


def test_sampled_tokens_match_the_whole_chunk():
    inp = tiny_shared()
    y = oracle.layer_shared(inp)
    toks = np.array([0, 7, 31, 63])
    yt, ids, _ = oracle.layer_tokens_shared(inp, toks)
    assert np.allclose(yt, y[toks], rtol=0, atol=1e-12 * np.abs(y).max())
    assert np.array_equal(ids, oracle.route(inp["logits"], inp["K"])[0][toks])
