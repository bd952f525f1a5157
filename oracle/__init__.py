"""CSA2 oracle (test infrastructure only).

A plain single-threaded CPU definition of the CSA2 sparse-attention hot path
in fp64 (``csa2_oracle.c``), bound with ctypes.  Only the test suite, the
package's smoke check and the benchmark's CPU-baseline leg may import it.  It
imports nothing from the CUDA package and shares no code with it.

Every function cites the passage of the DeepSeek-V4.1-Flash pages it follows;
the readings taken where the pages are silent are listed in the header of
``csa2_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
# CSA2_ORACLE_LIB names a prebuilt copy to load instead (the mutation tests
# compile copies of csa2_oracle.c with one planted mistake each)
_VARIANT = os.environ.get("CSA2_ORACLE_LIB")
_LIB_PATH = _VARIANT or os.path.join(_HERE, "_libcsa2_oracle.so")
_lock = threading.Lock()
_lib = None

FULL, REINDEX, REUSE = 0, 1, 2


def compile_command(src: str, out: str):
    """gcc command that builds the oracle library `out` from `src`."""
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", out, src,
            "-lm"]


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, no fast-math, no FMA contraction)."""
    if _VARIANT:
        return _LIB_PATH
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(compile_command(_SRC, tmp), check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            sig = {
                "orc_e2m1_value": (dbl, [i32]),
                "orc_e4m3_value": (dbl, [i32]),
                "orc_e4m3_encode": (i32, [dbl]),
                "orc_e2m1_encode_magnitude": (i32, [dbl]),
                "orc_fp4_row_bytes": (i64, [i32]),
                "orc_quantize_kv_fp4": (None, [vp, i64, i32, vp]),
                "orc_dequantize_kv_fp4": (None, [vp, i64, i32, vp]),
                "orc_n_visible": (i64, [vp, i32, i32, i64]),
                "orc_index_scores": (None, [vp, vp, i32, i32, i32, i64, i64, i32, vp, i32, vp]),
                "orc_topk": (None, [vp, i32, i64, i32, vp, i32, vp]),
                "orc_hier_pool_index": (None, [vp, vp, i32, i32, i32, i64, i64, i32, vp, i32, i32,
                                               vp]),
                "orc_sparse_attn": (None, [vp, vp, i32, i32, i32, i64, i64, i32, vp, i32, dbl,
                                           vp, vp]),
                "orc_block_pool": (None, [vp, i32, i64, vp, i32, i32, i32, vp]),
                "orc_e8m0_value": (dbl, [i32]),
                "orc_mxfp4_row_bytes": (i64, [i32]),
                "orc_quantize_mxfp4": (None, [vp, i64, i32, vp]),
                "orc_index_scores_fmt": (None, [vp, vp, i32, i32, i32, i64, i64, i32, vp, i32, i32,
                                                vp]),
                "orc_hier_pool_index_fmt": (None, [vp, vp, i32, i32, i32, i64, i64, i32, vp, i32,
                                                   i32, i32, vp]),
                "orc_sparse_attn_swa": (None, [vp, vp, i32, i32, i32, i64, i64, i32, vp, i32, vp,
                                               i64, i32, vp, dbl, vp, vp]),
                "orc_layer_group": (i32, [i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                          i32, i64, i64, i32, vp, i32, i32, i32, i32, vp, vp,
                                          i64, i32, i32, dbl]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# --- formats (DeepSeek-V4.1-Flash pages: release summary "CSA2"; walkthrough 1.(5).4) ---

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(code)


def e4m3_value(byte: int) -> float:
    return _load().orc_e4m3_value(byte)


def e4m3_encode(v: float) -> int:
    return _load().orc_e4m3_encode(float(v))


def e2m1_encode_magnitude(q: float) -> int:
    return _load().orc_e2m1_encode_magnitude(float(q))


def fp4_row_bytes(d: int) -> int:
    return int(_load().orc_fp4_row_bytes(d))


def quantize_kv_fp4(x: np.ndarray) -> np.ndarray:
    """fp32 [n][d] -> uint8 [n][d/2 + d/16] (walkthrough 1.(5).4 "FP4 Main KV Cache")."""
    x = _c(x, np.float32)
    n, d = x.shape
    out = np.empty((n, fp4_row_bytes(d)), dtype=np.uint8)
    _load().orc_quantize_kv_fp4(_ptr(x), n, d, _ptr(out))
    return out


def dequantize_kv_fp4(rows: np.ndarray, d: int) -> np.ndarray:
    rows = _c(rows, np.uint8)
    n = rows.shape[0]
    out = np.empty((n, d), dtype=np.float64)
    _load().orc_dequantize_kv_fp4(_ptr(rows), n, d, _ptr(out))
    return out


def n_visible(q_pos: Optional[np.ndarray], q: int, ratio: int, N: int) -> int:
    qp = None if q_pos is None else _c(q_pos, np.int32)
    return int(_load().orc_n_visible(_ptr(qp), q, ratio, N))


# --- indexer, top-k, pool (walkthrough 1.(4), 1.(4).1, 1.(4).2) ---

def index_scores(q_fp8, k_fp8, N: int, kv_seq_stride: int, q_per_seq: int, q_pos, ratio: int):
    """q_fp8 [B][H_I][D_I], k_fp8 [S*stride][D_I] -> fp64 scores [B][N] (-inf if invisible)."""
    q_fp8 = _c(q_fp8, np.uint8)
    k_fp8 = _c(k_fp8, np.uint8)
    B, H_I, D_I = q_fp8.shape
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.empty((B, N), dtype=np.float64)
    _load().orc_index_scores(_ptr(q_fp8), _ptr(k_fp8), B, H_I, D_I, N, kv_seq_stride, q_per_seq,
                             _ptr(qp), ratio, _ptr(out))
    return out


def topk(scores, k: int, q_pos=None, ratio: int = 1) -> np.ndarray:
    """scores [B][N] (any float type, compared as fp64) -> int32 idx [B][k]."""
    scores = _c(scores, np.float64)
    B, N = scores.shape
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.empty((B, k), dtype=np.int32)
    _load().orc_topk(_ptr(scores), B, N, k, _ptr(qp), ratio, _ptr(out))
    return out


# --- MXFP4 indexer rows (walkthrough 1.(5).4: OCP MXFP4 indexer q and K) ---

def e8m0_value(byte: int) -> float:
    return _load().orc_e8m0_value(int(byte))


def mxfp4_row_bytes(d: int) -> int:
    return int(_load().orc_mxfp4_row_bytes(d))


def quantize_mxfp4(x: np.ndarray) -> np.ndarray:
    """fp32 [..., d] (d % 32 == 0) -> uint8 [..., d/2 + d/32] OCP MXFP4 rows."""
    x = _c(x, np.float32)
    d = x.shape[-1]
    rows = x.reshape(-1, d)
    out = np.empty((rows.shape[0], mxfp4_row_bytes(d)), dtype=np.uint8)
    _load().orc_quantize_mxfp4(_ptr(rows), rows.shape[0], d, _ptr(out))
    return out.reshape(x.shape[:-1] + (out.shape[-1],))


def index_scores_mxfp4(q_mx, k_mx, D_I: int, N: int, kv_seq_stride: int, q_per_seq: int, q_pos,
                       ratio: int):
    """MXFP4 q [B][H_I][row], K [S*stride][row] -> fp64 scores [B][N] (R3 with R11)."""
    q_mx = _c(q_mx, np.uint8)
    k_mx = _c(k_mx, np.uint8)
    B, H_I = q_mx.shape[0], q_mx.shape[1]
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.empty((B, N), dtype=np.float64)
    _load().orc_index_scores_fmt(_ptr(q_mx), _ptr(k_mx), B, H_I, D_I, N, kv_seq_stride, q_per_seq,
                                 _ptr(qp), ratio, 1, _ptr(out))
    return out


def hier_pool_index_mxfp4(q_mx, k_mx, D_I: int, N: int, kv_seq_stride: int, q_per_seq: int,
                          pool, k: int):
    q_mx = _c(q_mx, np.uint8)
    k_mx = _c(k_mx, np.uint8)
    pool = _c(pool, np.int32)
    B, H_I = q_mx.shape[0], q_mx.shape[1]
    P = pool.shape[1]
    out = np.empty((B, k), dtype=np.int32)
    _load().orc_hier_pool_index_fmt(_ptr(q_mx), _ptr(k_mx), B, H_I, D_I, N, kv_seq_stride,
                                    q_per_seq, _ptr(pool), P, k, 1, _ptr(out))
    return out


def block_pool(scores, block: int, n_blocks: int, q_pos=None, ratio: int = 1) -> np.ndarray:
    """Blockwise candidate pool of the Hierarchical Sparse Indexer (walkthrough
    1.(4).2): scores [B][N] -> int32 pool [B][n_blocks * block]."""
    scores = _c(scores, np.float64)
    B, N = scores.shape
    qp = None if q_pos is None else _c(q_pos, np.int32)
    out = np.empty((B, n_blocks * block), dtype=np.int32)
    _load().orc_block_pool(_ptr(scores), B, N, _ptr(qp), ratio, block, n_blocks, _ptr(out))
    return out


def hier_pool_index(q_fp8, k_fp8, N: int, kv_seq_stride: int, q_per_seq: int, pool, k: int):
    q_fp8 = _c(q_fp8, np.uint8)
    k_fp8 = _c(k_fp8, np.uint8)
    pool = _c(pool, np.int32)
    B, H_I, D_I = q_fp8.shape
    P = pool.shape[1]
    out = np.empty((B, k), dtype=np.int32)
    _load().orc_hier_pool_index(_ptr(q_fp8), _ptr(k_fp8), B, H_I, D_I, N, kv_seq_stride,
                                q_per_seq, _ptr(pool), P, k, _ptr(out))
    return out


# --- attention (walkthrough 1.(4), 1.(5).4, 3.(2).1) ---

def sparse_attn(q_bf16, kv_fp4, N: int, kv_seq_stride: int, q_per_seq: int, idx, scale: float):
    """q_bf16 [B][H][D] (uint16 bits), kv_fp4 [S*stride][9D/16], idx [B][k] -> (out, lse) fp64."""
    q_bf16 = _c(q_bf16, np.uint16)
    kv_fp4 = _c(kv_fp4, np.uint8)
    idx = _c(idx, np.int32)
    B, H, D = q_bf16.shape
    k = idx.shape[1]
    out = np.empty((B, H, D), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    _load().orc_sparse_attn(_ptr(q_bf16), _ptr(kv_fp4), B, H, D, N, kv_seq_stride, q_per_seq,
                            _ptr(idx), k, float(scale), _ptr(out), _ptr(lse))
    return out, lse


def sparse_attn_swa(q_bf16, kv_fp4, N: int, kv_seq_stride: int, q_per_seq: int, idx,
                    swa_kv, swa_ring: int, n_win: int, q_pos, scale: float):
    """Sparse attention with the query's sliding window of the layer's SWA KV in the
    same softmax (reading R10).  swa_kv E4M3 [S][swa_ring][D] -> (out, lse) fp64."""
    q_bf16 = _c(q_bf16, np.uint16)
    kv_fp4 = _c(kv_fp4, np.uint8)
    idx = _c(idx, np.int32)
    swa = None if swa_kv is None else _c(swa_kv, np.uint8)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    B, H, D = q_bf16.shape
    k = idx.shape[1]
    out = np.empty((B, H, D), dtype=np.float64)
    lse = np.empty((B, H), dtype=np.float64)
    _load().orc_sparse_attn_swa(_ptr(q_bf16), _ptr(kv_fp4), B, H, D, N, kv_seq_stride, q_per_seq,
                                _ptr(idx), k, _ptr(swa), swa_ring, n_win, _ptr(qp), float(scale),
                                _ptr(out), _ptr(lse))
    return out, lse


def layer_group(modes: Sequence[int], q_bf16: Sequence[np.ndarray], qi_fp8: Sequence[np.ndarray],
                kv_fp4, ki_fp8, N: int, kv_seq_stride: int, q_per_seq: int, q_pos, ratio: int,
                k: int, pool_size: int, scale: float, pool_block: int = 0,
                swa_kv: Optional[Sequence[np.ndarray]] = None, swa_ring: int = 0, n_win: int = 0,
                indexer_fmt: int = 0, D_I: Optional[int] = None):
    """Runs the layer schedule (walkthrough 1.(4).1 and 1.(4).2).  pool_block > 0
    builds the blockwise pool (pool_size / pool_block blocks of pool_block entries).

    Returns (outs, lses, idxs, pool) with one array per layer."""
    L = len(modes)
    q_bf16 = [_c(q, np.uint16) for q in q_bf16]
    B, H, D = q_bf16[0].shape
    H_I = None
    qis = []
    for l in range(L):
        qi = qi_fp8[l]
        if qi is None:
            qis.append(None)
        else:
            qi = _c(qi, np.uint8)
            H_I = qi.shape[1]
            if D_I is None:
                D_I = qi.shape[2]
            qis.append(qi)
    kv_fp4 = _c(kv_fp4, np.uint8)
    ki_fp8 = _c(ki_fp8, np.uint8)
    qp = None if q_pos is None else _c(q_pos, np.int32)
    outs = [np.empty((B, H, D), np.float64) for _ in range(L)]
    lses = [np.empty((B, H), np.float64) for _ in range(L)]
    idxs = [np.empty((B, k), np.int32) for _ in range(L)]
    pool = np.empty((B, max(pool_size, 1)), np.int32)
    P = ctypes.c_void_p
    arr = lambda xs: (P * L)(*[_ptr(x) for x in xs])
    modes_c = (ctypes.c_int * L)(*modes)
    swas = None if swa_kv is None else [_c(x, np.uint8) for x in swa_kv]
    rc = _load().orc_layer_group(L, modes_c, arr(q_bf16), arr(qis), arr(outs), arr(lses),
                                 arr(idxs), _ptr(kv_fp4), _ptr(ki_fp8), B, H, H_I, D, D_I, N,
                                 kv_seq_stride, q_per_seq, _ptr(qp), ratio, k, pool_size,
                                 pool_block, _ptr(pool), None if swas is None else arr(swas),
                                 swa_ring, n_win, indexer_fmt, float(scale))
    if rc != 0:
        raise ValueError("invalid layer schedule")
    return outs, lses, idxs, (pool if pool_size > 0 else None)
