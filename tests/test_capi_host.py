"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/tsdf.h declares, rejects
invalid arguments before touching CUDA, and never reaches the oracle."""
import ctypes
import os
import re

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(REPO, "include", "tsdf.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsdf_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from hash_blocked_tsdf_gb300 import _build, binding
    _build.build_tsdf_library()
    return binding.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tsdf_create", "tsdf_integrate", "tsdf_block_count", "tsdf_export_blocks",
              "tsdf_allocate", "tsdf_update", "tsdf_get_stats", "tsdf_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_binding_covers_every_declared_symbol():
    from hash_blocked_tsdf_gb300 import binding
    assert sorted(binding.SIGNATURES) == declared_functions()


def _err(lib):
    return lib.tsdf_last_error().decode()


def test_create_rejects_bad_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.tsdf_create(0, 0.01, 0.04, ctypes.byref(h)) == -1 and not h.value
    assert "pool_capacity" in _err(lib)
    assert lib.tsdf_create((1 << 23) + 1, 0.01, 0.04, ctypes.byref(h)) == -1
    assert lib.tsdf_create(16, -0.01, 0.04, ctypes.byref(h)) == -1
    assert lib.tsdf_create(16, float("nan"), 0.04, ctypes.byref(h)) == -1
    assert lib.tsdf_create(16, 0.01, float("inf"), ctypes.byref(h)) == -1
    assert lib.tsdf_create(16, 0.0001, 1.0, ctypes.byref(h)) == -1      # 20001 band samples
    assert "too large" in _err(lib)
    assert lib.tsdf_create_ex(16, 48, 0.01, 0.04, ctypes.byref(h)) == -1  # not a power of two
    assert lib.tsdf_create_ex(16, 16, 0.01, 0.04, ctypes.byref(h)) == -1  # below 2 * pool
    assert lib.tsdf_create(16, 0.01, 0.04, None) == -1


def test_calls_on_a_null_volume_are_rejected(lib):
    K = (ctypes.c_float * 4)(500, 500, 320, 240)
    pose = (ctypes.c_float * 16)(1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1)
    assert lib.tsdf_integrate(None, 1, 1, 640, 480, K, pose, None) == -1
    assert lib.tsdf_allocate(None, 1, 640, 480, K, pose, None) == -1
    assert lib.tsdf_update(None, 1, 1, 640, 480, K, pose, None) == -1
    assert lib.tsdf_reset(None, None) == -1
    assert lib.tsdf_destroy(None) == -1
    out = ctypes.c_uint32()
    assert lib.tsdf_block_count(None, None, ctypes.byref(out)) == -1
    assert lib.tsdf_integrate_batch(None, 2, 1, 1, 640, 480, K, pose, None) == -1
    assert lib.tsdf_allocate_blocks(None, 1, 4, None) == -1
    assert lib.tsdf_set_occlusion(None, 1) == -1
    assert lib.tsdf_set_pool_layout(None, 1) == -1
    assert "null" in _err(lib)


def test_create_fails_loudly_without_a_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = lib.tsdf_create(16, 0.01, 0.04, ctypes.byref(h))
    assert rc in (-2, -3) and not h.value
    assert _err(lib)


def test_missing_library_raises(monkeypatch, tmp_path):
    from hash_blocked_tsdf_gb300 import binding
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not found"):
        binding.load_library()


def test_product_path_never_touches_the_oracle(lib):
    pkg = os.path.join(REPO, "hash_blocked_tsdf_gb300")
    imports = re.compile(r"^\s*(import\s+oracle|from\s+oracle\b|from\s+\.\.\s*import\s+oracle)",
                         re.M)
    for root, _, files in os.walk(pkg):
        for f in files:
            text = open(os.path.join(root, f), errors="ignore").read()
            if f.endswith(".py"):
                assert not imports.search(text), f"{f} imports the oracle"
            if f.endswith((".cu", ".cuh", ".h", ".c", ".py")):
                assert "oracle_" not in text and "liboracle" not in text, f"{f} calls the oracle"
    assert not hasattr(lib, "oracle_integrate")


def _header_struct_fields(name):
    """Field names of `typedef struct <name> { ... } <name>;` in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct " + name + r" \{(.*?)\} " + name + ";", text, re.S).group(1)
    fields = []
    for decl in body.split(";"):
        m = re.search(r"(\w+)\s*(\[[^\]]*\])?\s*$", decl.strip())
        if m:
            fields.append(m.group(1))
    return fields


@pytest.mark.parametrize("name", ["tsdf_info", "tsdf_pool_view", "tsdf_stats"])
def test_binding_structs_follow_the_header(name):
    # the ctypes mirrors must list the header's fields in the header's order
    from hash_blocked_tsdf_gb300 import binding
    mirror = [f for f, _ in getattr(binding, name)._fields_]
    assert mirror == _header_struct_fields(name)


def test_binding_constants_follow_the_header():
    from hash_blocked_tsdf_gb300 import binding
    defs = dict(re.findall(r"#define (TSDF_[A-Z_]+) \(?(-?\d+)", open(HEADER).read()))
    pairs = {
        "TSDF_UPDATE_ADAPTIVE": binding.UPDATE_KERNELS["adaptive"],
        "TSDF_UPDATE_PER_SAMPLE": binding.UPDATE_KERNELS["per_sample"],
        "TSDF_UPDATE_PRE_REDUCED": binding.UPDATE_KERNELS["pre_reduced"],
        "TSDF_UPDATE_FUSED": binding.UPDATE_KERNELS["fused"],
        "TSDF_UPDATE_AUTO": binding.UPDATE_KERNELS["auto"],
        "TSDF_OCCLUSION_RAY": binding.OCCLUSION_TESTS["ray"],
        "TSDF_OCCLUSION_REPROJECT": binding.OCCLUSION_TESTS["reproject"],
        "TSDF_LAYOUT_INTERLEAVED": binding.POOL_LAYOUTS["interleaved"],
        "TSDF_LAYOUT_PLANAR": binding.POOL_LAYOUTS["planar"],
        "TSDF_PROBE_HIST_BINS": binding.PROBE_HIST_BINS,
    }
    for k, v in pairs.items():
        assert int(defs[k]) == v, k
