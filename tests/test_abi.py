"""CPU checks of the C ABI: the library builds, loads and exports every entry
point include/cf.h declares; the Python binding mirrors them by name."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cf.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(cf_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from co_prefill_decode_gb300 import build, load_library
    build.build()
    return load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("cf_create", "cf_layer_step", "cf_decode_attn", "cf_prefill_attn", "cf_gemm",
                     "cf_kv_append", "cf_destroy", "cf_get_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    import co_prefill_decode_gb300 as cf
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(cf.EXPORTS) == declared_functions()


def test_binding_methods_use_c_names():
    import co_prefill_decode_gb300 as cf
    for name in ("cf_layer_step", "cf_decode_attn", "cf_prefill_attn", "cf_gemm", "cf_kv_append",
                 "cf_get_error"):
        assert callable(getattr(cf.Engine, name))


def test_struct_layouts_match_header():
    import ctypes
    import co_prefill_decode_gb300 as cf
    # field order of the structs in cf.h
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for struct, cls in (("cf_config", cf.cf_config), ("cf_weights", cf.cf_weights),
                        ("cf_kv_pool", cf.cf_kv_pool), ("cf_batch", cf.cf_batch),
                        ("cf_latency_model", cf.cf_latency_model), ("cf_rank_load", cf.cf_rank_load),
                        ("cf_latency_parts", cf.cf_latency_parts), ("cf_dispatch_state", cf.cf_dispatch_state),
                        ("cf_dispatch_result", cf.cf_dispatch_result)):
        body = re.search(r"typedef struct \{([^{}]*?)\}\s*" + struct + ";", src).group(1)
        fields = re.findall(r"\**\s*(\w+)\s*(?:,|;)", body)
        assert [f[0] for f in cls._fields_] == fields, struct
    assert ctypes.sizeof(cf.cf_config) == 12 * 4


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "co_prefill_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
