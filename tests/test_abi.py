"""Host-only checks of the C ABI: the library builds for sm_103a, loads without a GPU, exports every
symbol the headers declare, and rejects bad configurations before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include"))) if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from routed_expert_ffn_07_b300 import build
    build.build()
    from routed_expert_ffn_07_b300 import capi
    return capi


def _declared():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_boundary():
    names = _declared()
    for required in ("moe_create", "moe_set_layer", "moe_route", "moe_layer_forward", "moe_stack_forward",
                     "moe_destroy", "moe_layer_forward_host", "moe_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(so, n)]
    assert not missing, missing


def test_status_strings(lib):
    for s in range(8):
        assert lib.moe_status_str(s) and lib.moe_status_str(s) != "unknown status"
    assert lib.moe_version() >= 1


@pytest.mark.parametrize("kw", [
    dict(d=0), dict(f=-1), dict(n_experts=0), dict(top_k=0), dict(top_k=33), dict(n_layers=0), dict(max_tokens=0),
    dict(act=7), dict(wfmt=9), dict(has_shared=2), dict(top_k=20, n_experts=16),
])
def test_create_rejects_bad_config(lib, kw):
    base = dict(d=1024, f=256, n_experts=64, top_k=8, n_layers=2, max_tokens=16, has_shared=True)
    base.update(kw)
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_create(**base)
    assert ei.value.status == 1


@pytest.mark.parametrize("kw", [dict(d=1000), dict(f=200), dict(n_experts=2048), dict(wfmt=0, max_tokens=64)])
def test_create_unsupported_shapes(lib, kw):
    base = dict(d=1024, f=256, n_experts=64, top_k=8, n_layers=2, max_tokens=16, has_shared=True)
    base.update(kw)
    with pytest.raises(lib.MoeError) as ei:
        lib.moe_create(**base)
    assert ei.value.status == 2


def test_null_handles_rejected(lib):
    L = lib.lib
    assert L.moe_destroy(None) == 1
    assert L.moe_layer_forward(None, 0, None, 1, None, None) == 1
    assert L.moe_stack_forward(None, None, 1, None, None) == 1
    assert L.moe_route(None, 0, None, 1, None, None, None, None, None) == 1
    assert L.moe_create(None, None) == 1


def test_generator_rejects_bad_args(lib):
    assert lib.lib.moe_gen_int4_planes(None, 1, 0, 0, 0, 1, 16, None) == 1
    assert lib.lib.moe_gen_int4_planes(ctypes.c_void_p(16), 1, 0, 0, 0, 1, 12, None) == 1


def test_noalloc_route_validates_before_touching_the_device(lib):
    L = lib.lib
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) & ~15
    # T beyond the fixed scratch, E beyond it, K beyond it: unsupported; bad pointers / sizes: invalid
    assert L.moe_route_noalloc(p, None, p, 1, 17, 256, 8, 2, None, None, None, None, None) == 2
    assert L.moe_route_noalloc(p, None, p, 1, 4, 256, 2048, 2, None, None, None, None, None) == 2
    assert L.moe_route_noalloc(p, None, p, 1, 4, 256, 64, 33, None, None, None, None, None) == 2
    assert L.moe_route_noalloc(None, None, p, 1, 4, 256, 8, 2, None, None, None, None, None) == 1
    assert L.moe_route_noalloc(p + 2, None, p, 1, 4, 256, 8, 2, None, None, None, None, None) == 1
    assert L.moe_route_noalloc(p, None, p, 1, 4, 250, 8, 2, None, None, None, None, None) == 1
    assert L.moe_route_noalloc(p, None, p, 7, 4, 256, 8, 2, None, None, None, None, None) == 1


def test_selftest_rejects_bad_budget_before_the_device(lib):
    assert lib.lib.moe_selftest_bounded_waits(10, None) == 1
    assert lib.lib.moe_selftest_bounded_waits(10 ** 12, None) == 1


def test_device_memory_is_allocated_and_synchronised_only_in_create_and_destroy():
    """The boundary stores pointers: cudaMalloc / cudaFree / cudaDeviceSynchronize appear only in the
    bodies of moe_create and moe_destroy (a scan of the library's sources)."""
    import re
    csrc = os.path.join(ROOT, "routed_expert_ffn_07_b300", "csrc")
    calls = re.compile(r"\b(cudaMalloc|cudaMallocAsync|cudaFree|cudaFreeAsync|cudaDeviceSynchronize)\s*\(")
    opener = re.compile(r"^[A-Za-z_][\w:<>\*& ]*\b(\w+)\s*\([^;]*$")
    found = []
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh")):
            continue
        func = None
        for line in open(os.path.join(csrc, name)):
            m = opener.match(line)
            if m and not line.startswith((" ", "\t", "#", "//")):
                func = m.group(1)
            code = line.split("//")[0]
            if calls.search(code):
                found.append((name, func))
    assert found, "the scan found no allocation at all"
    assert {f for _, f in found} <= {"moe_create", "moe_destroy"}, found
