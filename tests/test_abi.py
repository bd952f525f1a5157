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


def test_binding_refuses_outputs_of_the_wrong_shape(libpath):
    # the library writes exactly the documented layout through an output pointer: a
    # caller's tensor of another shape is refused before its device is even looked at
    import torch
    from sparse_attention_decode_csa2_gb300 import csa2
    with pytest.raises(ValueError, match="shape"):
        csa2._out(torch.zeros(4, 287, dtype=torch.uint8), (4, 288), torch.uint8, "out")
    with pytest.raises(ValueError, match="shape"):
        csa2._out(torch.zeros(2, 64, 511), (2, 64, 512), torch.float32, "out")
    with pytest.raises(ValueError, match="CUDA"):   # right shape, but host memory
        csa2._out(torch.zeros(2, 64), (2, 64), torch.float32, "lse")


def test_mxfp4_argument_validation_before_any_device_work(libpath):
    from sparse_attention_decode_csa2_gb300 import csa2
    lib = csa2.lib
    # quantiser: null pointers, d not a multiple of 32, d too wide
    assert lib.csa2_quantize_mxfp4(None, 4, 128, None, None) == 1
    assert lib.csa2_quantize_mxfp4(16, 4, 48, 16, None) == 1
    assert lib.csa2_quantize_mxfp4(16, 4, 8192, 16, None) == 1
    assert lib.csa2_quantize_mxfp4(8, 4, 128, 16, None) == 1          # x not 16-byte aligned
    # scorer: (q, k, B, H_I, D_I, N, stride, q_per_seq, q_pos, ratio, scores, stream)
    args = lambda **kw: [kw.get("q", 64), kw.get("k", 64), kw.get("B", 4), kw.get("H_I", 32),
                         kw.get("D_I", 128), kw.get("N", 100), kw.get("stride", 100),
                         kw.get("qps", 1), None, kw.get("ratio", 1), kw.get("scores", 64), None]
    assert lib.csa2_index_scores_mxfp4(*args(q=None)) == 1             # null query
    assert lib.csa2_index_scores_mxfp4(*args(D_I=64)) == 2             # only D_I = 128
    assert lib.csa2_index_scores_mxfp4(*args(H_I=65)) == 2             # H_I <= 64
    assert lib.csa2_index_scores_mxfp4(*args(stride=102)) == 2         # 68 * stride % 16 != 0
    assert lib.csa2_index_scores_mxfp4(*args(k=72)) == 1               # K not 16-byte aligned
    assert lib.csa2_index_scores_mxfp4(*args(stride=50)) == 1          # stride < N
    assert lib.csa2_index_scores_mxfp4(*args(ratio=0)) == 1
    assert lib.csa2_index_scores_mxfp4(*args(scores=None)) == 1
    # pool re-index: P < 1, k < 1
    pargs = [64, 64, 4, 32, 128, 100, 100, 1, 64, 0, 8, 64, 64, 1 << 20, None]
    assert lib.csa2_hier_pool_index_mxfp4(*pargs) == 1


def _group(csa2, modes, B=32, N=16384, k=2048, pool=0, pool_block=0, fmt=0):
    L = len(modes)
    layers = (csa2.Csa2Layer * L)()
    for l, m in enumerate(modes):
        layers[l] = csa2.Csa2Layer(m, 64, None if m == 2 else 64, 64, 64, 64, None)
    g = csa2.Csa2GroupArgs(64, 64, B, 64, 8, 512, 64, N, N, 1, None, 4, k, pool, 64 if pool else None,
                           1.0 / 512 ** 0.5, pool_block, 0, 0, fmt)
    return layers, g


def test_index_scan_rejects_rows_beyond_32_bit_coordinates(libpath):
    import ctypes
    # the full E4M3 scan addresses indexer-K rows with 32-bit tensor coordinates: a call
    # whose sequences span 2^31 rows or more is refused before any device work
    from sparse_attention_decode_csa2_gb300 import csa2
    lib = csa2.lib
    fake = 1 << 20                     # aligned, never dereferenced: validation fails first
    half = 1 << 30
    code = lib.csa2_index_scores(fake, fake, 2, 8, 64, half, half, 1, None, 4, fake, None)
    assert code == 2                   # CSA2_ERR_UNSUPPORTED: rows = 2^30 + 2^30
    layers, g = _group(csa2, [0], B=2, N=half)
    assert lib.csa2_layer_group(layers, 1, ctypes.byref(g), fake, 1 << 40, None) == 2


def test_layer_group_launch_counts(libpath):
    import ctypes
    from sparse_attention_decode_csa2_gb300 import csa2
    count = lambda layers, g: csa2.lib.csa2_layer_group_launches(layers, len(layers),
                                                                  ctypes.byref(g))
    # without a device the SM count defaults to 148: 4 splits of 512 slots for 32 queries,
    # merged inside the attention kernel (one cluster per query)
    layers, g = _group(csa2, [0])
    assert count(layers, g) == 1 + 1 + 1                  # indexer, top-k, attention
    layers, g = _group(csa2, [0, 2, 1, 2])
    assert count(layers, g) == 3 + 1 + (2 + 1) + 1        # Reindex: scores + top-k
    layers, g = _group(csa2, [0, 1], pool=8192)
    assert count(layers, g) == (1 + 1 + 1 + 1) + (2 + 1)  # Full also selects the pool
    layers, g = _group(csa2, [0, 1], pool=16384, pool_block=8)
    assert count(layers, g) == (1 + 3 + 1 + 1) + (2 + 1)  # blockwise pool: three kernels
    # 160 queries: one CTA per query
    layers, g = _group(csa2, [0, 2], B=160, k=2048)
    assert count(layers, g) == (1 + 1 + 1) + 1
    layers, g = _group(csa2, [2, 0])                      # no Full layer first
    assert count(layers, g) == -1
    layers, g = _group(csa2, [0], B=0)
    assert count(layers, g) == 0


def test_workspace_sizes_grow_with_the_problem(libpath):
    from sparse_attention_decode_csa2_gb300 import csa2
    ws = csa2.lib.csa2_workspace_size
    base = ws(32, 16384, 2048, 64, 0)
    assert base >= 256 + 32 * 16384 * 4                    # status word + scores
    assert ws(32, 16384, 2048, 64, 16384) > base           # pool scores and pool scratch
    assert ws(64, 16384, 2048, 64, 0) > base
    assert ws(0, 0, 0, 0, 0) == 256                        # the status word alone
    assert csa2.lib.csa2_block_pool_workspace_size(16, 262144, 8, 2048) > 0


def test_empty_batches_and_contexts_return_ok_without_device_work(libpath):
    from sparse_attention_decode_csa2_gb300 import csa2
    lib = csa2.lib
    # B = 0: nothing to score, no pointer needed
    assert lib.csa2_index_scores_mxfp4(None, None, 0, 32, 128, 100, 100, 1, None, 1, None,
                                       None) == 0
    assert lib.csa2_index_scores(None, None, 0, 8, 64, 100, 100, 1, None, 1, None, None) == 0
    # N = 0: an empty context
    assert lib.csa2_index_scores_mxfp4(64, 64, 4, 32, 128, 0, 0, 1, None, 1, 64, None) == 0
    # top-k of an empty batch still needs the status word
    assert lib.csa2_topk(None, 0, 100, 8, None, 1, None, None, 0, None) == 3
    assert lib.csa2_topk(None, 0, 100, 8, None, 1, None, 64, 256, None) == 0
    assert lib.csa2_quantize_mxfp4(None, 0, 128, None, None) == 0   # empty: a no-op
    assert lib.csa2_quantize_kv_fp4(None, 0, 512, None, None) == 0
