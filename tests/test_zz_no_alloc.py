"""smoe_group_noalloc -- the grouping call that allocates nothing -- against smoe_group (GPU, through the C ABI).

Some callers cannot hand the library a scratch buffer: their device memory is planned once up front, or they may
not call cudaMalloc between requests because it can synchronise the device.  smoe_group_noalloc keeps the scratch
in a device array inside the library instead.  This test checks that its tables are identical to smoe_group's on two
calls in a row (the second call reuses the array the first one left behind), on two different routings.  The file
is named to be collected last, so that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _tables(binding, fn, ids, E):
    T, K = ids.shape
    n = T * K
    dev = torch.device("cuda")
    counts = torch.full((E,), -1, dtype=torch.int32, device=dev)
    offsets = torch.full((E + 4,), -1, dtype=torch.int32, device=dev)
    src = torch.full((n,), -1, dtype=torch.int32, device=dev)
    slot = torch.full((n,), -1, dtype=torch.int32, device=dev)
    tiles = torch.full((binding.tiles_bytes(n, E) // 4,), -1, dtype=torch.int32, device=dev)
    ids_d = torch.from_numpy(np.ascontiguousarray(ids)).to(dev)
    if fn == "alloc":
        work = torch.empty(max(binding.group_work_bytes(n, E), 16), dtype=torch.uint8, device=dev)
        binding.smoe_group(ids_d, E, counts, offsets, src, slot, tiles, work)
    else:
        binding.smoe_group_noalloc(ids_d, E, counts, offsets, src, slot, tiles)
    torch.cuda.synchronize()
    nt = int(tiles[0].item())
    return [t.cpu().numpy() for t in (counts, offsets[:E + 1], src, slot, tiles[:4 + 4 * nt])]


def test_noalloc_group_matches_group_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_smoe_gb300 import build, binding
    build.build()
    binding.load_library()
    binding.device_check()
    rng = np.random.default_rng(2024)
    # a full-size routing (81,920 pairs over 512 experts), then a skewed smaller one (most pairs on a few experts)
    first = rng.integers(0, 512, size=(8192, 10)).astype(np.int32)
    second = np.minimum(rng.zipf(1.3, size=(3001, 7)) - 1, 299).astype(np.int32)
    for ids, E in ((first, 512), (second, 300)):
        want = _tables(binding, "alloc", ids, E)
        got = _tables(binding, "noalloc", ids, E)
        for w, g in zip(want, got):
            assert np.array_equal(w, g)


def test_noalloc_group_empty_chunk_and_bad_ids():
    """An empty chunk (T = 0: no pairs, no chunks of the counting pass) gives an empty tile list and all-zero
    offsets, as smoe_group does; a routed id outside [0, E) is reported in the tile-list header exactly as
    smoe_group reports it, and the call after it (a good routing) is unaffected."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_smoe_gb300 import build, binding
    build.build()
    binding.load_library()
    binding.device_check()
    empty = np.zeros((0, 4), np.int32)
    for fn in ("alloc", "noalloc"):
        counts, offsets, _, _, tiles = _tables(binding, fn, empty, 8)
        assert np.all(counts == 0) and np.all(offsets == 0)
        assert tiles[0] == 0 and tiles[1] == 0 and tiles[2] == 0
    bad = np.array([[0, 1], [9, 2], [3, -1]], np.int32)
    want = _tables(binding, "alloc", bad, 4)
    got = _tables(binding, "noalloc", bad, 4)
    assert want[4][1] == 4 and got[4][1] == 4  # SMOE_ERR_RANGE in header[1]
    for w, g in zip(want, got):
        assert np.array_equal(w, g)
    good = np.random.default_rng(9).integers(0, 64, size=(500, 6)).astype(np.int32)
    for w, g in zip(_tables(binding, "alloc", good, 64), _tables(binding, "noalloc", good, 64)):
        assert np.array_equal(w, g)
