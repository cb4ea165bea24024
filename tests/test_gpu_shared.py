"""Parity of the shared expert through the C ABI (GPU: sm_103a) with the CPU oracle.

Bars: the scalar gate |sg_gpu - sg_oracle| <= 4e-6 (an fp32 dot product of H terms against double); the combine
with the shared row per element <= 1e-6 of the sum of the magnitudes it adds; the block's output per token row
max |y_gpu - y_oracle| <= 2e-3 * RMS(y_oracle row), as for the routed block.
"""
import numpy as np
import pytest

import oracle
from quantized_routed_expert_smoe_gb300 import synth

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


@pytest.mark.parametrize("T,H", [(1, 64), (333, 2560), (4099, 256)])
def test_shared_gate_parity(B, T, H):
    x = synth.make_rows(T, H, seed=11)
    wsg = (synth.make_rows(1, H, seed=12)[0] * 0.02).astype(np.float32)
    sg = torch.empty(max(T, 4), dtype=torch.float32, device="cuda")
    B.smoe_shared_gate(dev(x), dev(wsg), sg[:T])
    got = host(sg)[:T].astype(np.float64)
    want = oracle.shared_gate(x, wsg)
    assert np.abs(got - want).max() <= 4e-6


def test_combine_shared_parity(B):
    rng = np.random.default_rng(14)
    T, K, H = 513, 10, 2560
    n = T * K
    dm = synth.make_dm(n, H, seed=15)
    ds = synth.make_dm(T, H, seed=16)
    slot = rng.permutation(n).astype(np.int32)
    w = rng.random((T, K)).astype(np.float32)
    sg = rng.random(T).astype(np.float32)
    y = torch.empty(T, H, dtype=torch.float32, device="cuda")
    B.smoe_combine_shared(dev(dm), dev(slot), dev(w), dev(ds), dev(sg), y)
    got = host(y)
    want = oracle.combine_shared(dm.astype(np.float64), slot, w.astype(np.float64), ds.astype(np.float64),
                                 sg.astype(np.float64), T, K, H)
    mag = np.einsum("tk,tkh->th", np.abs(w.astype(np.float64)), np.abs(dm[slot.reshape(T, K)].astype(np.float64)))
    mag += np.abs(sg.astype(np.float64))[:, None] * np.abs(ds.astype(np.float64))
    assert np.all(np.abs(got - want) <= 1e-6 * mag + 1e-30)


@pytest.mark.parametrize("name", ["tiny", "t1024", "t8192"])
def test_block_with_shared_expert(B, name):
    cfg = synth.CONFIGS[name]
    inp = synth.make_layer(cfg)
    inp.update(synth.make_shared(cfg))
    shared = {k: inp[k] for k in ("sgu_c", "sgu_s", "sd_c", "sd_s", "wsg")}
    blk = B.SmoeBlock(cfg.T, cfg.H, cfg.E, cfg.K, cfg.F, inp["wgu_c"], inp["wgu_s"], inp["wd_c"], inp["wd_s"],
                      shared=shared)
    y = host(blk.run(dev(inp["logits"]), dev(inp["x"]))).astype(np.float64)
    assert blk.device_status() == (0, 0)
    # the shared expert's grouping: one expert, row r = token r
    assert np.array_equal(host(blk.s_src)[:cfg.T], np.arange(cfg.T))
    assert int(host(blk.s_tiles)[1]) == 0 and int(host(blk.s_tiles)[3]) == 0
    if name == "tiny":
        toks = np.arange(cfg.T)
        y_o = oracle.layer_shared(inp)
    else:
        rng = np.random.default_rng(cfg.seed + 100)
        toks = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, 24, replace=False)]))
        y_o, _, _ = oracle.layer_tokens_shared(inp, toks)
    y_s = y[toks]
    rms = np.sqrt((y_o ** 2).mean(axis=1))
    err = np.abs(y_s - y_o).max(axis=1)
    assert np.all(err <= 2e-3 * rms), f"worst err/rms {float((err / rms).max()):.3e}"
    assert np.isfinite(y).all()
    # the shared term is really there: the routed-only block differs by far more than the bar
    y_r = oracle.layer_tokens(inp, toks)[0] if name != "tiny" else oracle.layer(inp)
    assert np.abs(y_r - y_o).max() > 0.1 * np.sqrt((y_o ** 2).mean())
    del blk
    torch.cuda.empty_cache()


@pytest.mark.parametrize("with_shared,with_router,graphs", [(False, False, False), (True, False, False),
                                                             (True, True, False), (False, False, True),
                                                             (True, True, True)])
def test_pipeline_matches_run(B, with_shared, with_router, graphs):
    # SmoePipeline (host in, host out, copies overlapped with the neighbouring steps' compute) gives every step's
    # output bit for bit as the plain run on device inputs, over more steps than it has buffers
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_layer(cfg)
    shared = None
    if with_shared:
        inp.update(synth.make_shared(cfg))
        shared = {k: inp[k] for k in ("sgu_c", "sgu_s", "sd_c", "sd_s", "wsg")}
    blk = B.SmoeBlock(cfg.T, cfg.H, cfg.E, cfg.K, cfg.F, inp["wgu_c"], inp["wgu_s"], inp["wd_c"], inp["wd_s"],
                      shared=shared, router=synth.make_router(cfg) if with_router else None)
    steps = 5
    xs = [synth.make_rows(cfg.T, cfg.H, seed=40 + s) for s in range(steps)]
    lgs = [synth.make_rows(cfg.T, cfg.E, seed=50 + s, scale=0.5) for s in range(steps)]
    want = [host(blk.run(dev(lgs[s]), dev(xs[s]))).copy() for s in range(steps)]
    pipe = B.SmoePipeline(blk, graphs=graphs)  # (graphs: each buffer set's run() captured, then replayed)
    # a block with its own router projection takes no logits: the pipeline copies none
    h_in = [(None if with_router else torch.from_numpy(lgs[s]).pin_memory(), torch.from_numpy(xs[s]).pin_memory())
            for s in range(steps)]
    h_out = [torch.empty(cfg.T, cfg.H, dtype=torch.float32).pin_memory() for _ in range(steps)]
    for s in range(steps):
        pipe.submit(h_in[s][0], h_in[s][1], h_out[s])
    pipe.synchronize()
    for s in range(steps):
        assert np.array_equal(h_out[s].numpy(), want[s]), f"step {s}"
    assert blk.device_status() == (0, 0)


@pytest.mark.parametrize("name", ["tiny", "t1024"])
def test_native_block_matches_run(B, name):
    # the block as libsmoe's own object (smoe_block_*): chunks from and into pinned host memory through its copy
    # streams and graphs, and device to device, give every chunk's output bit for bit as SmoeBlock.run; more chunks
    # than device sets, and a second round after a sync
    cfg = synth.CONFIGS[name]
    inp = synth.make_layer(cfg)
    blk = B.SmoeBlock(cfg.T, cfg.H, cfg.E, cfg.K, cfg.F, inp["wgu_c"], inp["wgu_s"], inp["wd_c"], inp["wd_s"])
    nb = B.NativeBlock(cfg.T, cfg.H, cfg.E, cfg.K, cfg.F, inp["wgu_c"], inp["wgu_s"], inp["wd_c"], inp["wd_s"])
    steps = 5
    xs = [synth.make_rows(cfg.T, cfg.H, seed=60 + s) for s in range(steps)]
    lgs = [synth.make_rows(cfg.T, cfg.E, seed=70 + s, scale=0.5) for s in range(steps)]
    want = [host(blk.run(dev(lgs[s]), dev(xs[s]))).copy() for s in range(steps)]
    h_lg = [torch.from_numpy(lgs[s]).pin_memory() for s in range(steps)]
    h_x = [torch.from_numpy(xs[s]).pin_memory() for s in range(steps)]
    for rnd in range(2):
        h_out = [torch.full((cfg.T, cfg.H), float("nan")).pin_memory() for _ in range(steps)]
        for s in range(steps):
            nb.submit_host(h_lg[s], h_x[s], h_out[s])
        nb.sync()
        for s in range(steps):
            assert np.array_equal(h_out[s].numpy(), want[s]), f"round {rnd} chunk {s}"
        assert nb.device_status() == (0, 0)
    y = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device="cuda")
    nb.run(dev(lgs[2]), dev(xs[2]), y)
    assert np.array_equal(host(y), want[2])
    # pageable host memory is correct too (its copies do not overlap the compute)
    h_page = torch.empty(cfg.T, cfg.H, dtype=torch.float32)
    nb.submit_host(torch.from_numpy(lgs[1]), torch.from_numpy(xs[1]), h_page)
    nb.sync()
    assert np.array_equal(h_page.numpy(), want[1])
    nb.close()
    del blk
    torch.cuda.empty_cache()
