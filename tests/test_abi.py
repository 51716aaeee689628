"""The C-ABI library builds, loads and exports every symbol the header
declares; host-only entry points (sizes, defaults, status strings, argument
validation that returns before any CUDA call) work without a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bakron.h")


@pytest.fixture(scope="module")
def L():
    from kronecker_factored_gptq_gb300 import bakron as kb
    if not os.path.exists(kb.LIB_PATH):
        from kronecker_factored_gptq_gb300 import build
        build.build()
    return kb.lib()


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(bakron_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("bakron_prepare", "bakron_quantize", "bakron_quantize_antidiag",
                 "bakron_rowscale", "bakron_workspace_size", "bakron_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), "libbakron.so does not export %s" % name


def test_binding_lists_every_export():
    from kronecker_factored_gptq_gb300 import bakron as kb
    assert set(declared_functions()) == set(kb.EXPORTS)


def test_status_strings_and_version(L):
    from kronecker_factored_gptq_gb300 import bakron as kb
    for code in range(8):
        assert L.bakron_status_string(code)
    assert L.bakron_status_string(99) == b"unknown status"
    assert L.bakron_version() >= 10000
    o = kb.default_opts()
    assert o.tile == 128 and o.leaf_width == 1 and o.spin_budget_cycles > 0


def test_workspace_sizes(L):
    from kronecker_factored_gptq_gb300 import bakron as kb
    s1 = kb.workspace_size(64, 64)
    s2 = kb.workspace_size(8192, 8192)
    assert 0 < s1 < s2
    # W~, E (hi, lo), Y (hi, lo) and four factor halves, fp32, padded to 128
    assert s2 >= 4 * 8192 * 8192 * 9
    assert kb.prepare_workspace_size(8192, 8192) >= 3 * 4 * 8192 * 8192
    b = ctypes.c_size_t(0)
    assert L.bakron_workspace_size(0, 5, None, ctypes.byref(b)) == 1
    assert L.bakron_workspace_size(5, 5, None, None) == 1
    assert L.bakron_prepare_workspace_size(0, 0, ctypes.byref(b)) == 1


def test_invalid_arguments_return_before_any_cuda_call(L):
    from kronecker_factored_gptq_gb300 import bakron as kb
    vp = ctypes.c_void_p
    fake = vp(0x1000)
    o = kb.default_opts()
    # null pointers
    assert L.bakron_quantize(None, 4, 4, fake, fake, fake, -8, 7, fake, fake, None, None,
                             fake, 1 << 20, None) == 1
    # qmin > qmax
    assert L.bakron_quantize(fake, 4, 4, fake, fake, fake, 7, -8, fake, fake, None, None,
                             fake, 1 << 20, None) == 1
    # workspace too small
    assert L.bakron_quantize(fake, 4, 4, fake, fake, fake, -8, 7, fake, fake, None, None,
                             fake, 16, None) == 1
    # bad options
    bad = kb.default_opts(tile=64)
    assert L.bakron_quantize(fake, 4, 4, fake, fake, fake, -8, 7, fake, fake, None,
                             ctypes.byref(bad), fake, 1 << 20, None) == 1
    assert L.bakron_quantize_antidiag(fake, 0, 4, fake, fake, fake, -8, 7, fake, fake, None, None,
                                      0.0, None, ctypes.byref(o), fake, 1 << 20, None) == 1
    assert L.bakron_prepare(None, 4, 0.0, None, 0, 0.0, fake, None, None, None, None, fake,
                            1 << 20, None) == 1
    assert L.bakron_prepare(fake, 4, -1.0, None, 0, 0.0, fake, None, None, None, None, fake,
                            1 << 20, None) == 1
    assert L.bakron_rowscale(fake, 4, 4, 0, fake, None) == 1


def test_size_limits(L):
    """Documented caps: at most 2^20 tiles of W, factor orders up to 65536
    (the host work lists stay small; no GPU could hold larger workspaces)."""
    b = ctypes.c_size_t(0)
    n = ctypes.c_int64(0)
    assert L.bakron_workspace_size(1 << 20, 128, None, ctypes.byref(b)) == 0   # 8192 x 1 tiles
    assert L.bakron_workspace_size((1 << 17) + 1, 1 << 17, None, ctypes.byref(b)) == 1   # 1025 x 1024
    assert L.bakron_workspace_size(1 << 20, 1 << 20, None, ctypes.byref(b)) == 1
    assert L.bakron_prepare_workspace_size(1 << 12, 0, ctypes.byref(b)) == 0
    assert L.bakron_prepare_workspace_size((1 << 16) + 1, 0, ctypes.byref(b)) == 1
    assert L.bakron_prepare_workspace_size(1 << 20, 1 << 20, ctypes.byref(b)) == 1
    assert L.bakron_factors_workspace_size(100, (1 << 16) + 1, 0, ctypes.byref(b)) == 1
    assert L.bakron_schedule_export(0, 2048, 1024, None, 0, ctypes.byref(n)) == 1
    assert L.bakron_schedule_export(2, 513, 1, None, 0, ctypes.byref(n)) == 1
    assert L.bakron_schedule_export(2, 16, 1, None, 0, ctypes.byref(n)) == 0 and n.value > 0


def test_plan_size_and_invalid_plan_arguments(L):
    """The plan holds a header and both solves' work lists (16 bytes per
    128-tile product) of the shape's tile grid; shapes with the same grid
    share it.  Bad arguments return before any CUDA call."""
    from kronecker_factored_gptq_gb300 import bakron as kb
    b = ctypes.c_size_t(0)
    assert L.bakron_plan_size(8192, 8192, ctypes.byref(b)) == 0
    n = (len(kb.schedule_export(kb.SCHEDULE_SOLVE, 64, 64)) and
         int(kb.schedule_export(kb.SCHEDULE_SOLVE, 64, 64)[2]) +
         int(kb.schedule_export(kb.SCHEDULE_ROWS, 64, 64)[2]))
    assert b.value == 256 + 16 * n
    assert kb.plan_size(8100, 8192) == kb.plan_size(8192, 8192)
    assert L.bakron_plan_size(0, 8, ctypes.byref(b)) == 1
    assert L.bakron_plan_size(8, 8, None) == 1
    fake = ctypes.c_void_p(0x1000)
    assert L.bakron_plan_init(8, 8, None, 1 << 20, None) == 1
    assert L.bakron_plan_init(8, 8, ctypes.c_void_p(0x1004), 1 << 20, None) == 1   # unaligned
    assert L.bakron_plan_init(8, 8, fake, 16, None) == 1                           # too small


ALLOC_CALLS = ("cudaMalloc", "cudaMallocAsync", "cudaMallocManaged", "cudaHostAlloc",
               "cudaMallocHost", "cudaFree", "cudaFreeHost", "cudaFreeAsync",
               "cudaDeviceSynchronize")


def test_library_source_allocates_no_device_or_pinned_memory():
    """The ownership rule of the header: the library allocates no device or
    pinned host memory, keeps none between calls and never synchronises the
    whole device; every buffer is the caller's (workspace, plan, outputs)."""
    csrc = os.path.join(ROOT, "kronecker_factored_gptq_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h", ".cpp")):
            continue
        txt = re.sub(r"//[^\n]*|/\*.*?\*/", "", open(os.path.join(csrc, f)).read(), flags=re.S)
        for call in ALLOC_CALLS:
            assert not re.search(r"\b%s\s*\(" % call, txt), "%s calls %s" % (f, call)
