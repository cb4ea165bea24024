"""The C-ABI library builds for sm_103a, loads without a GPU, exports every symbol include/smoe.h declares, and
rejects bad arguments on the host before it touches a device (CPU only: no compute call runs here)."""
import ctypes
import os
import re

import pytest

from quantized_routed_expert_smoe_gb300 import build as smoe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smoe.h")


@pytest.fixture(scope="module")
def lib():
    smoe_build.build()
    from quantized_routed_expert_smoe_gb300 import binding
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(smoe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_seven_steps():
    names = declared_functions()
    for step in ["smoe_route_topk", "smoe_group", "smoe_quantize_q8", "smoe_gather_q8", "smoe_experts_gateup",
                 "smoe_swiglu_requant", "smoe_experts_down", "smoe_combine"]:
        assert step in names


def test_library_exports_every_declared_symbol(lib):
    from quantized_routed_expert_smoe_gb300 import binding
    names = declared_functions()
    assert set(names) == set(binding.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name


def test_sizing_helpers(lib):
    from quantized_routed_expert_smoe_gb300 import binding
    assert binding.max_tiles(81920, 512) == (81920 + 191) // 192 + 512
    assert binding.max_tiles(128, 16) == 1 + 16
    assert binding.max_tiles(0, 16) == 0
    assert binding.tiles_bytes(128, 16) == 16 * 18
    assert binding.group_work_bytes(81920, 512) >= 512 * 4
    assert binding.pack_q2_bytes(2, 128, 64) == 2 * 128 * (16 + 4)
    # the router's scratch: the bf16 hi and lo planes of the activations, then two halves' top-16 candidates
    assert binding.router_work_bytes(8192, 2560) == 2 * 2 * 8192 * 2560 + 8192 * 2 * 16 * 8
    assert binding.router_work_bytes(0, 2560) == 0


def test_host_side_rejections_need_no_gpu(lib):
    fake = ctypes.c_void_p(1 << 20)          # 16-byte aligned, never dereferenced on these paths
    odd = ctypes.c_void_p((1 << 20) + 4)     # misaligned
    null = ctypes.c_void_p(0)
    ARG, UNSUP = 1, 3
    # route: K > E, E too large, null / misaligned pointers
    assert lib.smoe_route_topk(fake, 4, 8, 9, fake, fake, null) == ARG
    assert lib.smoe_route_topk(fake, 4, 2048, 2, fake, fake, null) == ARG
    assert lib.smoe_route_topk(null, 4, 16, 2, fake, fake, null) == ARG
    assert lib.smoe_route_topk(odd, 4, 16, 2, fake, fake, null) == ARG
    assert lib.smoe_route_topk(fake, 0, 16, 2, fake, fake, null) == 0  # empty chunk: nothing to do
    # q8: cols not a multiple of 32
    assert lib.smoe_quantize_q8(fake, 4, 48, fake, fake, null) == ARG
    # gemm shapes the kernels do not cover
    assert lib.smoe_experts_gateup(fake, fake, 10, 4, fake, 96, 64, fake, null) == UNSUP
    assert lib.smoe_experts_down(odd, fake, 10, 4, fake, 256, 64, fake, null) == ARG  # misaligned rows
    # gather: cols not a multiple of 32, misaligned scales or output
    assert lib.smoe_gather_q8(fake, fake, 4, 48, fake, 8, fake, null) == ARG
    assert lib.smoe_gather_q8(fake, odd, 4, 128, fake, 8, fake, null) == ARG
    assert lib.smoe_gather_q8(fake, fake, 4, 128, fake, 8, odd, null) == ARG
    assert lib.smoe_gather_q8(fake, fake, 4, 128, fake, 0, fake, null) == 0  # nothing routed: nothing to do
    # SwiGLU: the operand form needs F % 64 == 0
    assert lib.smoe_swiglu_requant(fake, 4, 96, fake, fake, fake, null) == ARG
    assert lib.smoe_experts_down(fake, fake, 10, 4, fake, 256, 48, fake, null) == UNSUP
    assert lib.smoe_pack_q2(fake, fake, 2, 100, 64, fake, null) == ARG  # rows % 128
    # shared expert: H % 4, misaligned gate output, misaligned shared rows in the combine
    assert lib.smoe_shared_gate(fake, fake, 4, 30, fake, null) == ARG
    assert lib.smoe_shared_gate(fake, fake, 4, 32, odd, null) == ARG
    assert lib.smoe_shared_gate(fake, fake, 0, 32, fake, null) == 0  # empty chunk: nothing to do
    assert lib.smoe_combine_shared(fake, fake, fake, 4, 2, 32, odd, fake, fake, null) == ARG
    assert lib.smoe_combine_shared(fake, fake, fake, 4, 2, 32, fake, null, fake, null) == ARG
    # the narrow Dm: fp16 rows need H % 8 for the combine; misaligned rows; the down product's shape rules
    assert lib.smoe_combine_h(fake, fake, fake, 4, 2, 36, fake, null) == ARG
    assert lib.smoe_combine_h(odd, fake, fake, 4, 2, 32, fake, null) == ARG
    assert lib.smoe_combine_h(fake, fake, fake, 4, 0, 32, fake, null) == ARG
    assert lib.smoe_combine_h(fake, fake, fake, 0, 2, 32, fake, null) == 0  # empty chunk: nothing to do
    assert lib.smoe_experts_down_h(fake, fake, 10, 4, fake, 256, 64, odd, null) == ARG
    assert lib.smoe_experts_down_h(fake, fake, 10, 4, fake, 256, 48, fake, null) == UNSUP
    # router: H % 64, E out of range or not a multiple of 16 (of 32 above 256), K > 16
    assert lib.smoe_router_topk(fake, fake, 4, 96, 64, 2, fake, fake, fake, null) == ARG
    assert lib.smoe_router_topk(fake, fake, 4, 128, 8, 2, fake, fake, fake, null) == ARG
    assert lib.smoe_router_topk(fake, fake, 4, 128, 528, 2, fake, fake, fake, null) == ARG
    assert lib.smoe_router_topk(fake, fake, 4, 128, 272, 2, fake, fake, fake, null) == ARG
    assert lib.smoe_router_topk(fake, fake, 4, 128, 64, 17, fake, fake, fake, null) == ARG
    assert lib.smoe_router_topk(fake, fake, 0, 128, 64, 2, fake, fake, fake, null) == 0  # empty chunk
    # group: tiles buffer too small; a T whose T * K would overflow is refused before the product is formed
    assert lib.smoe_group(fake, 8, 2, 4, fake, fake, fake, fake, fake, 16, fake, 1 << 20, null) == ARG
    assert lib.smoe_group(fake, 1 << 62, 32, 4, fake, fake, fake, fake, fake, 1 << 40, fake, 1 << 40, null) == ARG
    # the allocation-free grouping: the same host-side checks (tiles buffer too small, E above the maximum, a huge
    # T, misaligned outputs) before it looks at the device or its scratch array
    assert lib.smoe_group_noalloc(fake, 8, 2, 4, fake, fake, fake, fake, fake, 16, null) == ARG
    assert lib.smoe_group_noalloc(fake, 8, 2, 2048, fake, fake, fake, fake, fake, 1 << 20, null) == ARG
    assert lib.smoe_group_noalloc(fake, 1 << 62, 32, 4, fake, fake, fake, fake, fake, 1 << 40, null) == ARG
    assert lib.smoe_group_noalloc(fake, 1 << 40, 4, 4, fake, fake, fake, fake, fake, 1 << 40, null) == ARG
    assert lib.smoe_group_noalloc(fake, 8, 2, 4, odd, fake, fake, fake, fake, 1 << 20, null) == ARG
    assert lib.smoe_group_noalloc(fake, 8, 2, 4, fake, fake, fake, odd, fake, 1 << 20, null) == ARG
    assert lib.smoe_group_noalloc(fake, 8, 0, 4, fake, fake, fake, fake, fake, 1 << 20, null) == ARG
    # the block object: bad sizes, null or misaligned weights, a null block -- refused before any device work
    h = ctypes.c_void_p(123)
    assert lib.smoe_block_create(0, 256, 16, 2, 128, fake, fake, ctypes.byref(h)) == ARG and h.value is None
    assert lib.smoe_block_create(64, 200, 16, 2, 128, fake, fake, ctypes.byref(h)) == ARG
    assert lib.smoe_block_create(64, 256, 16, 17, 128, fake, fake, ctypes.byref(h)) == ARG
    assert lib.smoe_block_create(64, 256, 16, 2, 96, fake, fake, ctypes.byref(h)) == ARG
    assert lib.smoe_block_create(64, 256, 16, 2, 128, null, fake, ctypes.byref(h)) == ARG
    assert lib.smoe_block_create(64, 256, 16, 2, 128, fake, odd, ctypes.byref(h)) == ARG
    assert lib.smoe_block_create(64, 256, 16, 2, 128, fake, fake, None) == ARG
    assert lib.smoe_block_run(null, fake, fake, fake, null) == ARG
    assert lib.smoe_block_submit_host(null, fake, fake, fake, null) == ARG
    assert lib.smoe_block_sync(null, null) == ARG
    g, k = ctypes.c_int(), ctypes.c_int()
    assert lib.smoe_block_status(null, ctypes.byref(g), ctypes.byref(k)) == ARG
    lib.smoe_block_destroy(null)  # a no-op
    if not _has_gpu():
        assert lib.smoe_block_create(64, 256, 16, 2, 128, fake, fake, ctypes.byref(h)) == UNSUP and h.value is None
    # well-formed arguments on a machine without an sm_103 device: a clean error, never a fallback
    st = lib.smoe_route_topk(fake, 4, 16, 2, fake, fake, null)
    if not _has_gpu():
        assert st == UNSUP
    assert lib.smoe_status_string(UNSUP).decode().startswith("unsupported")


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def test_binding_fails_loudly_without_library(tmp_path):
    from quantized_routed_expert_smoe_gb300 import binding
    saved = binding._lib
    try:
        binding._lib = None
        with pytest.raises(RuntimeError, match="no fallback"):
            binding.load_library(str(tmp_path / "libsmoe.so"))
    finally:
        binding._lib = saved


def test_build_targets_sm103a_only():
    assert smoe_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_header_is_plain_c(tmp_path):
    # the boundary is a C ABI: the header compiles as C99 (no C++ types or overloads leak into it)
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "smoe.h"\nint main(void) { return smoe_max_tiles(0, 1) == 0 ? 0 : 1; }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I" + os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
