"""Parity of the router projection fused into the top-K (smoe_router_topk) with the oracle (GPU: sm_103a).

Bars: the bf16 split of the activations is bit-exact; the ids equal the oracle's, except that where the oracle's
double logits of two experts lie within DELTA of each other (the tensor cores accumulate in fp32, the oracle in
double: a near-tie may resolve either way) the set and order may differ there, and at least 99 % of the tokens match
exactly; every weight is within 2e-5 of exp(l_k - l_1) / sum over the returned ids of the oracle's double logits.
"""
import numpy as np
import pytest

import oracle
from quantized_routed_expert_smoe_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DELTA = 2e-4  # logits are O(1) here; fp32 accumulation of 2 x H exact products errs by ~1e-5


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


def run_router(B, x, wr, K):
    T, H = x.shape
    E = wr.shape[0]
    ids = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    work = torch.empty(max(B.router_work_bytes(T, H), 16), dtype=torch.uint8, device="cuda")
    B.smoe_router_topk(dev(x), dev(wr.view(np.int16)), ids, w, work)
    return host(ids), host(w), host(work)[:4 * T * H].view(np.uint16).reshape(2, T, H)


def check_route(ids_g, w_g, ids_o, lg, K):
    T = ids_g.shape[0]
    exact = 0
    for t in range(T):
        g, o = ids_g[t], ids_o[t]
        assert len(set(g.tolist())) == K and g.min() >= 0 and g.max() < lg.shape[1]
        v = lg[t][g]
        # returned best first, up to near-ties
        assert np.all(np.diff(v) <= DELTA), (t, v)
        if np.array_equal(g, o):
            exact += 1
        else:
            kth = np.sort(lg[t])[::-1][K - 1]
            for e in set(g.tolist()) ^ set(o.tolist()):
                assert abs(lg[t][e] - kth) <= DELTA, (t, e, lg[t][e], kth)
        ex = np.exp(v - v.max())
        assert np.abs(w_g[t] - ex / ex.sum()).max() <= 2e-5
    assert exact >= 0.99 * T, f"{exact} of {T} tokens exact"


@pytest.mark.parametrize("T,H,E,K", [(1, 64, 32, 1), (129, 2560, 512, 10), (300, 256, 64, 4), (1000, 512, 96, 16),
                                     (77, 256, 16, 2), (200, 128, 288, 3)])
def test_router_parity_shapes(B, T, H, E, K):
    x = synth.make_rows(T, H, seed=T + H)
    wr = synth.make_router(dict(E=E, H=H, seed=E + K), sigma=1.0 / np.sqrt(H))
    ids, w, split = run_router(B, x, wr, K)
    xh, xl = oracle.bf16_split(x)
    assert np.array_equal(split[0], xh) and np.array_equal(split[1], xl)
    ids_o, _, lg = oracle.router_route(x, wr, K)
    check_route(ids, w, ids_o, lg, K)


def test_router_parity_t8192(B):
    cfg = synth.CONFIGS["t8192"]
    x = synth.make_layer(cfg, with_weights=False)["x"]
    wr = synth.make_router(cfg)
    ids, w, _ = run_router(B, x, wr, cfg.K)
    ids_o, _, lg = oracle.router_route(x, wr, cfg.K)
    check_route(ids, w, ids_o, lg, cfg.K)


def test_router_exact_logits_tie_to_the_lower_id(B):
    # Small-integer activations and weights: every product and partial sum is an integer below 2^24, so the tensor
    # cores' fp32 logits are exact and equal the oracle's -- many exact ties (duplicated router rows in one half and
    # across the two halves of E among them), which must go to the lower id: ids bit for bit.
    T, H, E, K = 300, 512, 512, 10
    rng = np.random.default_rng(33)
    x = rng.integers(-2, 3, size=(T, H)).astype(np.float32)
    wv = rng.integers(-2, 3, size=(E, H)).astype(np.float32)
    wv[6] = wv[5]
    wv[300] = wv[100]
    wr = (wv.view(np.uint32) >> 16).astype(np.uint16)  # small integers are exact in bf16
    ids, w, split = run_router(B, x, wr, K)
    assert not split[1].any()  # no low part
    ids_o, w_o, lg = oracle.router_route(x, wr, K)
    assert np.array_equal(lg, np.round(lg))
    assert np.array_equal(ids, ids_o)
    assert np.abs(w - w_o).max() <= 2e-6
    ties = sum(len(np.unique(lg[t][ids_o[t]])) < K for t in range(T))
    assert ties > T // 10  # the case really exercises ties


@pytest.mark.parametrize("name", ["tiny", "t1024"])
def test_block_with_router(B, name):
    cfg = synth.CONFIGS[name]
    inp = synth.make_layer(cfg)
    wr = synth.make_router(cfg)
    blk = B.SmoeBlock(cfg.T, cfg.H, cfg.E, cfg.K, cfg.F, inp["wgu_c"], inp["wgu_s"], inp["wd_c"], inp["wd_s"],
                      router=wr)
    y = host(blk.run(None, dev(inp["x"]))).astype(np.float64)
    assert blk.device_status() == (0, 0)
    ids_g = host(blk.ids)
    ids_o, _, lg = oracle.router_route(inp["x"], wr, cfg.K)
    # the rest of the block on the oracle's own (fp32-rounded) router logits, for the tokens routed alike
    ref = dict(inp, logits=lg.astype(np.float32))
    same = np.nonzero((ids_g == ids_o).all(axis=1))[0]
    assert same.size >= 0.99 * cfg.T
    toks = same if name == "tiny" else same[np.random.default_rng(cfg.seed).choice(same.size, 24, replace=False)]
    y_o, _, _ = oracle.layer_tokens(ref, np.sort(toks))
    y_s = y[np.sort(toks)]
    rms = np.sqrt((y_o ** 2).mean(axis=1))
    assert np.all(np.abs(y_s - y_o).max(axis=1) <= 2e-3 * rms)
