"""The C-ABI library builds, loads and exports every symbol include/hs.h
declares; host-side argument and configuration checks (no GPU needed)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from tiered_kv_cache_int8_gb300.build import build
    build()
    from tiered_kv_cache_int8_gb300 import hs
    return hs.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/hs.h but not exported"
    from tiered_kv_cache_int8_gb300 import hs
    assert sorted(hs.EXPORTED) == names


def cfg(**over):
    from tiered_kv_cache_int8_gb300.hs import HsConfig
    base = dict(n_layers=1, max_requests=2, max_context=4096, h_q=32, h_kv=8, d_qk=128, d_v=128,
                shared_kv=0, d_idx=128, top_k=256, hot_slots=512, softmax_scale=0.0, device=0)
    base.update(over)
    return HsConfig(**base)


@pytest.mark.parametrize("over", [
    dict(top_k=600),                 # k > B
    dict(hot_slots=20000, top_k=16),  # B too large
    dict(d_idx=48),                  # not a power of two
    dict(d_idx=512),
    dict(d_qk=64, d_v=64),           # GQA head dim
    dict(h_q=24, h_kv=8),            # group of 3
    dict(h_kv=16, h_q=32),
    dict(n_layers=0),
    dict(max_context=0),
    dict(max_context=(1 << 20) + 1),
    dict(top_k=0),
    dict(shared_kv=2),
    dict(softmax_scale=-1.0),
    dict(fetch_mode=3),
    dict(replacement=3),             # none of LRU, FIFO, random
    dict(page_size=3),               # pages: a power of two up to 64
    dict(page_size=128),
    dict(page_size=16, top_k=264, hot_slots=512),   # k not a whole number of pages
    dict(page_size=16, hot_slots=528),              # page slots not a multiple of 4
    dict(page_size=16, d_idx=32),                   # bounds rows of 64 or 128 keys only
    dict(page_size=16, idx_heads=4),
    dict(page_size=16, write_allocate=1),
    dict(page_size=16, shared_kv=1, h_kv=1, h_q=16, d_qk=576, d_v=512),
])
def test_unsupported_configs_are_rejected_before_touching_the_gpu(L, over):
    from tiered_kv_cache_int8_gb300 import hs
    h = ctypes.c_void_p()
    rc = L.hs_create(ctypes.byref(cfg(**over)), ctypes.byref(h))
    assert rc == hs.HS_ERR_CONFIG and not h
    assert L.hs_last_error(None).decode().startswith("hs_create:")


def test_row_elems_and_status_strings(L):
    assert L.hs_row_elems(ctypes.byref(cfg())) == 8 * 256
    assert L.hs_row_elems(ctypes.byref(cfg(h_kv=1, h_q=8))) == 256
    assert L.hs_row_elems(ctypes.byref(cfg(top_k=9999))) == 0
    assert L.hs_status_string(0) == b"HS_OK"
    assert L.hs_status_string(-4) == b"HS_ERR_CAPACITY"
    assert L.hs_status_string(-99) == b"HS_ERR_UNKNOWN"


def test_null_arguments(L):
    from tiered_kv_cache_int8_gb300 import hs
    h = ctypes.c_void_p()
    assert L.hs_create(None, ctypes.byref(h)) == hs.HS_ERR_INVALID
    assert L.hs_append(None, 0, 1, None, 1, None, None, None) == hs.HS_ERR_INVALID
    assert L.hs_decode_layer(None, 0, 1, None, None, None, None, None, None, None, None) == hs.HS_ERR_INVALID
    assert L.hs_stats(None, None) == hs.HS_ERR_INVALID
    assert L.hs_snapshot(None, 0, 0, None, 0, None, None, None, None) == hs.HS_ERR_INVALID
    L.hs_destroy(None)


def test_no_gpu_means_a_cuda_error_not_a_fallback(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from tiered_kv_cache_int8_gb300 import hs
    h = ctypes.c_void_p()
    rc = L.hs_create(ctypes.byref(cfg()), ctypes.byref(h))
    assert rc == hs.HS_ERR_CUDA and not h
    with pytest.raises(hs.HsError):
        hs.HiSparseCache(n_layers=1, max_requests=1, max_context=64, h_q=8, h_kv=1, d_qk=128, d_v=128,
                         d_idx=16, top_k=8, hot_slots=8)


def test_plain_c_caller(L, tmp_path):
    # the boundary is plain C: a C99 program compiled against include/hs.h and
    # linked to libhs.so runs its host-side checks (tests/c/abi_from_c.c)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib_dir = os.path.join(ROOT, "tiered_kv_cache_int8_gb300")
    exe = str(tmp_path / "abi_from_c")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-L", lib_dir, "-lhs",
                    f"-Wl,-rpath,{lib_dir}", "-o", exe], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi_from_c: ok" in r.stdout


def header_struct_fields(name):
    """(type, field) pairs of `typedef struct <name> { ... }` in include/hs.h."""
    text = open(os.path.join(ROOT, "include", "hs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef struct " + name + r"\s*\{(.*?)\}\s*" + name + r"_t;", text, flags=re.S).group(1)
    return re.findall(r"\b(int32_t|uint32_t|uint64_t|float)\s+(\w+)\s*;", body)


@pytest.mark.parametrize("struct, cls", [("hs_config", "HsConfig"), ("hs_stats", "HsStats")])
def test_binding_structs_follow_the_header(struct, cls):
    # the ctypes mirrors must list the header's fields in order, with the same types
    from tiered_kv_cache_int8_gb300 import hs
    ctype = {"int32_t": ctypes.c_int32, "uint32_t": ctypes.c_uint32, "uint64_t": ctypes.c_uint64,
             "float": ctypes.c_float}
    want = [(f, ctype[t]) for t, f in header_struct_fields(struct)]
    got = list(getattr(hs, cls)._fields_)
    assert [f for f, _ in got] == [f for f, _ in want]
    assert [t for _, t in got] == [t for _, t in want]
