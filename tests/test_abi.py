"""The C ABI library loads and exports every function include/csa2.h declares
(no GPU needed: nothing is computed)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "csa2.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(csa2_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libpath():
    from sparse_attention_decode_csa2_gb300 import build
    return build.build()


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("csa2_quantize_kv_fp4", "csa2_index_scores", "csa2_topk", "csa2_hier_pool_index",
              "csa2_sparse_attn_fp4", "csa2_layer_group", "csa2_workspace_size"):
        assert n in names


def test_library_exports_every_declared_function(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_function(libpath):
    from sparse_attention_decode_csa2_gb300 import csa2
    assert set(declared_functions()) <= set(csa2.EXPORTED)


def test_host_side_calls_without_gpu_work(libpath):
    lib = ctypes.CDLL(libpath)
    lib.csa2_status_string.restype = ctypes.c_char_p
    assert lib.csa2_status_string(0) == b"CSA2_OK"
    assert lib.csa2_status_string(5) == b"CSA2_ERR_BAD_INDEX"
    assert lib.csa2_version() >= 100
    # argument validation happens before any device work
    lib.csa2_quantize_kv_fp4.restype = ctypes.c_int
    lib.csa2_quantize_kv_fp4.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p]
    assert lib.csa2_quantize_kv_fp4(None, 4, 512, None, None) == 1      # null pointers
    assert lib.csa2_quantize_kv_fp4(16, 4, 256, 16, None) == 2          # unsupported d
    lib.csa2_layer_group.restype = ctypes.c_int
    lib.csa2_layer_group.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert lib.csa2_layer_group(None, 0, None, None, 0, None) == 1


def test_binding_refuses_cpu_tensors(libpath):
    import torch
    from sparse_attention_decode_csa2_gb300 import csa2
    with pytest.raises(ValueError):
        csa2.quantize_kv_fp4(torch.zeros(4, 512))
