"""The C-ABI library builds, loads and exports every symbol include/pagedkv.h
declares; host-side argument validation rejects bad calls before any launch.
No compute call is made (no GPU needed)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "pagedkv.h"


def _declared():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?[\s\*]+([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_303_gb300 import build, ops
    build.build()
    return ops.lib()


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ("kv_build_slot_mapping", "kv_build_decode_slots", "kv_store", "paged_attn_prefill",
              "paged_attn_decode", "paged_attn_prefill_workspace_size",
              "paged_attn_decode_workspace_size", "pkv_last_error", "pkv_device_status"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), f"libpagedkv.so does not export {n}"


def test_binding_covers_every_declared_symbol():
    from paged_kv_cache_303_gb300 import ops
    assert set(_declared()) <= set(ops.SIGNATURES), set(_declared()) - set(ops.SIGNATURES)


def test_library_is_built_for_sm103a_only():
    from paged_kv_cache_303_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_version(lib):
    assert lib.pkv_version() == 1


def _err(lib):
    return lib.pkv_last_error().decode()


def test_kv_store_validation_before_launch(lib):
    # negative sizes and null pointers are rejected on the host
    assert lib.kv_store(None, 0, None, 0, None, None, None, -1, 8, 128, 0, None) == 1
    assert lib.kv_store(None, 1024, None, 1024, None, None, None, 3, 8, 128, 10, None) == 1
    assert "null" in _err(lib)
    p = ctypes.c_void_p(16)   # never dereferenced: the stride check fails first
    assert lib.kv_store(p, 512, p, 1024, p, p, p, 3, 8, 128, 10, None) == 1
    assert "row strides" in _err(lib)
    # zero tokens is a valid no-op
    assert lib.kv_store(None, 0, None, 0, None, None, None, 0, 8, 128, 0, None) == 0


def test_attention_validation_before_launch(lib):
    p = ctypes.c_void_p(256)
    # head_dim 96 is not supported
    rc = lib.paged_attn_decode(p, 96 * 4, p, p, 1, p, 1, 1, p, 1, 4, 2, 96, 16, 16, 0.1, p, 96 * 4,
                               None, None, 0, None)
    assert rc == 2 and "head_dim" in _err(lib)
    # num_heads not a multiple of num_kv_heads
    rc = lib.paged_attn_decode(p, 640, p, p, 1, p, 1, 1, p, 1, 5, 2, 128, 16, 16, 0.1, p, 640,
                               None, None, 0, None)
    assert rc == 1
    # block table too small for max_context_len
    rc = lib.paged_attn_decode(p, 512, p, p, 4, p, 1, 1, p, 1, 4, 2, 128, 16, 17, 0.1, p, 512,
                               None, None, 0, None)
    assert rc == 1 and "capacity" in _err(lib)
    # prefill: packed mode without k
    rc = lib.paged_attn_prefill(p, 512, None, 0, None, 0, None, None, 0, None, 0, 0, p, p, 4, 4,
                                1, 4, 4, 4, 2, 128, 0, 0.1, p, 512, None, p, 1024, None)
    assert rc == 1 and "packed" in _err(lib)
    # prefill: misaligned q row stride
    rc = lib.paged_attn_prefill(p, 516, p, 256, p, 256, None, None, 0, None, 0, 0, p, p, 4, 4,
                                1, 4, 4, 4, 2, 128, 0, 0.1, p, 512, None, p, 1024, None)
    assert rc == 1 or rc == 2


def test_workspace_sizes_are_monotone(lib):
    a = lib.paged_attn_prefill_workspace_size(8, 1000, 500, 16)
    b = lib.paged_attn_prefill_workspace_size(8, 20000, 4096, 16)
    assert 0 < a < b
    assert lib.paged_attn_decode_workspace_size(0, 16, 8, 128, 100) == 0


def test_product_never_imports_the_oracle():
    pkg = ROOT / "paged_kv_cache_303_gb300"
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")) + \
            list(pkg.rglob("*.h")):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f
        assert "oracle.c" not in text and "liboracle" not in text, f
    for f in (ROOT / "oracle").glob("*"):
        if f.suffix in (".py", ".c"):
            text = f.read_text()
            assert "import paged_kv_cache_303_gb300" not in text, f
            assert "from paged_kv_cache_303_gb300" not in text, f
            assert "libpagedkv" not in text and "pagedkv.h" not in text, f


def test_fused_entry_points_validate_before_launch(lib):
    p = ctypes.c_void_p(256)
    # paged_attn_decode_store: key/value are required
    rc = lib.paged_attn_decode_store(p, 256, None, 0, None, 0, p, p, 4, p, 1, 1, p, 1, 2, 1, 128,
                                     16, 16, 0.1, p, 256, None, None, 0, None)
    assert rc == 1 and "key" in _err(lib)
    # ... with row strides that are not multiples of 8 elements
    rc = lib.paged_attn_decode_store(p, 256, p, 132, p, 128, p, p, 4, p, 1, 1, p, 1, 2, 1, 128,
                                     16, 16, 0.1, p, 256, None, None, 0, None)
    assert rc == 2
    # qk_norm_rope_store: head_dim 96 unsupported, theta must be positive
    rc = lib.qk_norm_rope_store(p, 384, p, 96, p, 96, p, p, p, 1e-6, 1e6, p, 384, None, 0, p, p, p,
                                4, 4, 1, 96, 64, None)
    assert rc == 2 and "head_dim" in _err(lib)
    rc = lib.qk_norm_rope_store(p, 512, p, 128, p, 128, p, p, p, 1e-6, 0.0, p, 512, None, 0, p, p, p,
                                4, 4, 1, 128, 64, None)
    assert rc == 1 and "theta" in _err(lib)
    rc = lib.qk_norm_rope_store(p, 512, p, 128, p, 128, None, p, p, 1e-6, 1e6, p, 512, None, 0, p, p,
                                p, 4, 4, 1, 128, 64, None)
    assert rc == 1 and "null" in _err(lib)
    # an in-place q_out must keep q's row stride
    rc = lib.qk_norm_rope_store(p, 1024, p, 128, p, 128, p, p, p, 1e-6, 1e6, p, 512, None, 0, p, p,
                                p, 4, 4, 1, 128, 64, None)
    assert rc == 1 and "in-place" in _err(lib)
    # zero tokens is a valid no-op
    assert lib.qk_norm_rope_store(None, 0, None, 0, None, 0, None, None, None, 1e-6, 1e6, None, 0,
                                  None, 0, None, None, None, 0, 4, 1, 128, 0, None) == 0


def test_decode_chunk_tiles_setter_sizes_the_workspace(lib):
    auto = lib.paged_attn_decode_workspace_size(4, 16, 8, 128, 4096)
    try:
        assert lib.pkv_set_decode_chunk_tiles(1) == 0
        # 32-key chunks: 128 splits of a 4096-key context, each with a
        # head_dim row and an (m, l) pair per (row, head)
        forced = lib.paged_attn_decode_workspace_size(4, 16, 8, 128, 4096)
        assert forced >= 256 + 4 * 16 * 128 * (128 + 2) * 4
        assert lib.pkv_set_decode_chunk_tiles(-1) == 1
        assert lib.pkv_set_decode_chunk_tiles(4097) == 1
    finally:
        assert lib.pkv_set_decode_chunk_tiles(0) == 0
    assert lib.paged_attn_decode_workspace_size(4, 16, 8, 128, 4096) == auto < forced
