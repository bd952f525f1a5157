"""Thin Python binding of libcsa2.so (declared in include/csa2.h).

Argument marshalling only: every function checks tensor devices, dtypes and
shapes, passes raw device pointers and the current CUDA stream to the C ABI,
and raises ``Csa2Error`` on a non-OK status.  There is no CPU path: importing
this module loads the shared library and raises if it has not been built
(``python -m sparse_attention_decode_csa2_gb300.build``), and every call
requires CUDA tensors.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa2.so")

FULL, REINDEX, REUSE = 0, 1, 2
D_LATENT = 512
ROW_BYTES = D_LATENT // 2 + D_LATENT // 16

STATUS_NAMES = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED",
                3: "CSA2_ERR_WORKSPACE", 4: "CSA2_ERR_CUDA", 5: "CSA2_ERR_BAD_INDEX",
                6: "CSA2_ERR_TIMEOUT"}


class Csa2Error(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        msg = f"{where}: {STATUS_NAMES.get(code, code)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.code = code


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -m sparse_attention_decode_csa2_gb300.build` (needs nvcc)")

lib = ctypes.CDLL(LIB_PATH)

_vp, _i32, _i64, _sz, _f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                              ctypes.c_float)


class Csa2Layer(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("q_bf16", _vp), ("qi_fp8", _vp), ("out", _vp),
                ("lse", _vp), ("idx_out", _vp), ("swa_kv", _vp)]


class Csa2GroupArgs(ctypes.Structure):
    _fields_ = [("kv_fp4", _vp), ("ki_fp8", _vp), ("B", ctypes.c_int), ("H", ctypes.c_int),
                ("H_I", ctypes.c_int), ("D", ctypes.c_int), ("D_I", ctypes.c_int),
                ("N", ctypes.c_int64), ("kv_seq_stride", ctypes.c_int64),
                ("q_per_seq", ctypes.c_int), ("q_pos", _vp), ("ratio", ctypes.c_int),
                ("k", ctypes.c_int), ("pool_size", ctypes.c_int), ("pool_out", _vp),
                ("softmax_scale", ctypes.c_float), ("pool_block", ctypes.c_int),
                ("swa_ring", ctypes.c_int64), ("n_win", ctypes.c_int),
                ("indexer_fmt", ctypes.c_int), ("q_ready", _vp)]


INDEXER_E4M3, INDEXER_MXFP4 = 0, 1
UPLOAD_RAW, UPLOAD_KV_FP4 = 0, 1


class Csa2UploadSeg(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_uint64), ("src_off", ctypes.c_uint64), ("rows", ctypes.c_uint64),
                ("row_bytes", ctypes.c_uint64), ("dst_stride", ctypes.c_uint64),
                ("kind", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


def mxfp4_row_bytes(d: int) -> int:
    return d // 2 + d // 32


def _mx_dim(row_bytes: int) -> int:
    # an MXFP4 row of d elements has 17 d / 32 bytes
    if row_bytes % 17:
        raise ValueError(f"{row_bytes} bytes is not an MXFP4 row")
    return row_bytes * 32 // 17


_SIGS = {
    "csa2_status_string": (ctypes.c_char_p, [_i32]),
    "csa2_version": (_i32, []),
    "csa2_last_cuda_error": (ctypes.c_char_p, []),
    "csa2_quantize_kv_fp4": (_i32, [_vp, _i64, _i32, _vp, _vp]),
    "csa2_upload": (_i32, [_vp, _sz, _i32, _vp, _sz, _vp]),
    "csa2_index_scores": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp, _i32, _vp,
                                 _vp]),
    "csa2_quantize_mxfp4": (_i32, [_vp, _i64, _i32, _vp, _vp]),
    "csa2_index_scores_mxfp4": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp, _i32,
                                       _vp, _vp]),
    "csa2_hier_pool_index_mxfp4": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp,
                                          _i32, _i32, _vp, _vp, _sz, _vp]),
    "csa2_topk": (_i32, [_vp, _i32, _i64, _i32, _vp, _i32, _vp, _vp, _sz, _vp]),
    "csa2_block_pool": (_i32, [_vp, _i32, _i64, _vp, _i32, _i32, _i32, _vp, _vp, _sz, _vp]),
    "csa2_block_pool_workspace_size": (_sz, [_i32, _i64, _i32, _i32]),
    "csa2_hier_pool_index": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp, _i32,
                                    _i32, _vp, _vp, _sz, _vp]),
    "csa2_sparse_attn_fp4": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp, _i32,
                                    _f32, _vp, _vp, _vp, _sz, _vp]),
    "csa2_sparse_attn_fp4_swa": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp, _i32,
                                        _vp, _i64, _i32, _vp, _f32, _vp, _vp, _vp, _sz, _vp]),
    "csa2_sparse_attn_fp4_noalloc": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i64, _i32, _vp,
                                            _i32, _f32, _vp, _vp, _vp]),
    "csa2_layer_group": (_i32, [ctypes.POINTER(Csa2Layer), _i32, ctypes.POINTER(Csa2GroupArgs),
                                _vp, _sz, _vp]),
    "csa2_layer_group_launches": (_i32, [ctypes.POINTER(Csa2Layer), _i32,
                                         ctypes.POINTER(Csa2GroupArgs)]),
    "csa2_workspace_size": (_sz, [_i32, _i64, _i32, _i32, _i32]),
    "csa2_workspace_init": (_i32, [_vp, _sz, _vp]),
    "csa2_read_status": (_i32, [_vp, _vp, ctypes.POINTER(ctypes.c_int32)]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def _check(code: int, where: str) -> None:
    if code != 0:
        detail = lib.csa2_last_cuda_error().decode() if code == 4 else ""
        raise Csa2Error(code, where, detail)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _out(t: torch.Tensor, shape, dtype, name: str) -> torch.Tensor:
    """A caller-supplied output: the library writes exactly `shape` elements
    through its pointer, so a tensor of another shape is refused before any
    launch (it would be written out of bounds or only in part)."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return _dev(t, dtype, name)


def _bits16(t: torch.Tensor, name: str) -> torch.Tensor:
    """bf16 tensor (or its int16/uint16 bit view) -> same storage as int16."""
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    elif t.dtype == torch.uint16:
        t = t.view(torch.int16)
    return _dev(t, torch.int16, name)


def _opt_pos(q_pos: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    return None if q_pos is None else _dev(q_pos, torch.int32, "q_pos")


# ---------------------------------------------------------------------------
# workspace
# ---------------------------------------------------------------------------

def workspace_size(B: int, N: int = 0, k: int = 0, H: int = 0, P: int = 0) -> int:
    return int(lib.csa2_workspace_size(B, N, k, H, P))


def make_workspace(B: int, N: int = 0, k: int = 0, H: int = 0, P: int = 0,
                   device=None) -> torch.Tensor:
    n = workspace_size(B, N, k, H, P)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    _check(lib.csa2_workspace_init(ws.data_ptr(), n, _stream()), "csa2_workspace_init")
    return ws


def read_status(ws: torch.Tensor):
    """Synchronises the current stream; returns (status_code, raw_bits) and clears the word."""
    bits = ctypes.c_int32(0)
    code = lib.csa2_read_status(ws.data_ptr(), _stream(), ctypes.byref(bits))
    return int(code), int(bits.value)


# ---------------------------------------------------------------------------
# operations (same names as the C ABI without the csa2_ prefix)
# ---------------------------------------------------------------------------

def quantize_kv_fp4(x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """fp32 [n][512] -> uint8 [n][288] FP4 rows."""
    x = _dev(x, torch.float32, "x")
    n, d = x.reshape(-1, x.shape[-1]).shape
    if out is None:
        out = torch.empty((n, d // 2 + d // 16), dtype=torch.uint8, device=x.device)
    _out(out, (n, d // 2 + d // 16), torch.uint8, "out")
    _check(lib.csa2_quantize_kv_fp4(_ptr(x), n, d, _ptr(out), _stream()), "csa2_quantize_kv_fp4")
    return out


class StepUpload:
    """One packed host-to-device transfer per decode step (csa2_upload).

    ``segments`` lists the step's inputs as ``(kind, dst)`` pairs: ``dst`` is a
    2-D device tensor view whose rows receive the segment (rows may be strided,
    each row contiguous).  UPLOAD_RAW copies the row bytes as they are;
    UPLOAD_KV_FP4 takes fp32 latent rows of 512 channels and writes them into
    ``dst``'s 288-byte FP4 rows (as csa2_quantize_kv_fp4 packs them).  The
    pinned host buffer (table + payloads) and the device staging area are
    allocated once; ``payloads[i]`` is the host view the caller fills with
    segment i's rows before each call."""

    def __init__(self, segments, device=None):
        specs = []
        for kind, dst in segments:
            if dst.dim() != 2 or dst.stride(1) != 1 or not dst.is_cuda:
                raise ValueError("a segment destination is a 2-D CUDA view with contiguous rows")
            esz = dst.element_size()
            if kind == UPLOAD_KV_FP4:
                if dst.dtype != torch.uint8 or dst.shape[1] != ROW_BYTES:
                    raise ValueError("an FP4 segment writes uint8 rows of 288 bytes")
                row_bytes, pshape, pdtype = D_LATENT * 4, (dst.shape[0], D_LATENT), torch.float32
            elif kind == UPLOAD_RAW:
                row_bytes, pshape, pdtype = dst.shape[1] * esz, tuple(dst.shape), dst.dtype
            else:
                raise ValueError(f"unknown segment kind {kind}")
            specs.append((kind, dst, row_bytes, pshape, pdtype, dst.stride(0) * esz))
        self.n = len(specs)
        off = (self.n * ctypes.sizeof(Csa2UploadSeg) + 15) // 16 * 16
        table = (Csa2UploadSeg * max(1, self.n))()
        offs = []
        for i, (kind, dst, row_bytes, pshape, pdtype, stride) in enumerate(specs):
            table[i] = Csa2UploadSeg(dst.data_ptr(), off, dst.shape[0], row_bytes, stride, kind, 0)
            offs.append(off)
            off += (dst.shape[0] * row_bytes + 15) // 16 * 16
        self.bytes = max(off, 16)
        self.host = torch.zeros(self.bytes, dtype=torch.uint8).pin_memory()
        nt = self.n * ctypes.sizeof(Csa2UploadSeg)
        if nt:
            ctypes.memmove(self.host.data_ptr(), ctypes.addressof(table), nt)
        self.stage = torch.empty(self.bytes, dtype=torch.uint8,
                                 device=device if device is not None else specs[0][1].device)
        self.payloads = [self.host[o:o + pshape[0] * rb].view(pdtype).view(pshape)
                         for o, (_, _, rb, pshape, pdtype, _) in zip(offs, specs)]
        self._keep = [sp[1] for sp in specs]   # the destinations outlive the table

    def __call__(self) -> None:
        _check(lib.csa2_upload(self.host.data_ptr(), self.bytes, self.n, self.stage.data_ptr(),
                               self.bytes, _stream()), "csa2_upload")


def index_scores(q_fp8: torch.Tensor, k_fp8: torch.Tensor, N: int, kv_seq_stride: int,
                 q_per_seq: int, q_pos: Optional[torch.Tensor], ratio: int,
                 out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """E4M3 q [B][H_I][D_I], E4M3 K [S*stride][D_I] -> fp32 scores [B][N]."""
    q_fp8 = _dev(q_fp8, torch.uint8, "q_fp8")
    k_fp8 = _dev(k_fp8, torch.uint8, "k_fp8")
    B, H_I, D_I = q_fp8.shape
    if out is None:
        out = torch.empty((B, N), dtype=torch.float32, device=q_fp8.device)
    _out(out, (B, N), torch.float32, "scores")
    qp = _opt_pos(q_pos)
    _check(lib.csa2_index_scores(_ptr(q_fp8), _ptr(k_fp8), B, H_I, D_I, N, kv_seq_stride,
                                 q_per_seq, _ptr(qp), ratio, _ptr(out), _stream()),
           "csa2_index_scores")
    return out


def quantize_mxfp4(x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """fp32 [..., d] -> uint8 [..., d/2 + d/32] MXFP4 rows."""
    x = _dev(x, torch.float32, "x")
    d = x.shape[-1]
    n = x.numel() // d
    if out is None:
        out = torch.empty(x.shape[:-1] + (mxfp4_row_bytes(d),), dtype=torch.uint8,
                          device=x.device)
    _out(out, x.shape[:-1] + (mxfp4_row_bytes(d),), torch.uint8, "out")
    _check(lib.csa2_quantize_mxfp4(_ptr(x), n, d, _ptr(out), _stream()), "csa2_quantize_mxfp4")
    return out


def index_scores_mxfp4(q_mx: torch.Tensor, k_mx: torch.Tensor, N: int, kv_seq_stride: int,
                       q_per_seq: int, q_pos: Optional[torch.Tensor], ratio: int,
                       out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """MXFP4 q [B][H_I][68], MXFP4 K [S*stride][68] -> fp32 scores [B][N]."""
    q_mx = _dev(q_mx, torch.uint8, "q_mx")
    k_mx = _dev(k_mx, torch.uint8, "k_mx")
    B, H_I, rb = q_mx.shape
    if out is None:
        out = torch.empty((B, N), dtype=torch.float32, device=q_mx.device)
    _out(out, (B, N), torch.float32, "scores")
    qp = _opt_pos(q_pos)
    _check(lib.csa2_index_scores_mxfp4(_ptr(q_mx), _ptr(k_mx), B, H_I, _mx_dim(rb), N,
                                       kv_seq_stride, q_per_seq, _ptr(qp), ratio, _ptr(out),
                                       _stream()), "csa2_index_scores_mxfp4")
    return out


def hier_pool_index_mxfp4(q_mx: torch.Tensor, k_mx: torch.Tensor, N: int, kv_seq_stride: int,
                          q_per_seq: int, pool: torch.Tensor, k: int,
                          ws: Optional[torch.Tensor] = None,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    q_mx = _dev(q_mx, torch.uint8, "q_mx")
    k_mx = _dev(k_mx, torch.uint8, "k_mx")
    pool = _dev(pool, torch.int32, "pool")
    B, H_I, rb = q_mx.shape
    P = pool.shape[1]
    if ws is None:
        ws = make_workspace(B, 0, k, 0, P, q_mx.device)
    if out is None:
        out = torch.empty((B, k), dtype=torch.int32, device=q_mx.device)
    _out(out, (B, k), torch.int32, "idx")
    _check(lib.csa2_hier_pool_index_mxfp4(_ptr(q_mx), _ptr(k_mx), B, H_I, _mx_dim(rb), N,
                                          kv_seq_stride, q_per_seq, _ptr(pool), P, k, _ptr(out),
                                          _ptr(ws), ws.numel(), _stream()),
           "csa2_hier_pool_index_mxfp4")
    return out


def topk(scores: torch.Tensor, k: int, q_pos: Optional[torch.Tensor] = None, ratio: int = 1,
         ws: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    scores = _dev(scores, torch.float32, "scores")
    B, N = scores.shape
    if ws is None:
        ws = make_workspace(B, N, k, 0, 0, scores.device)
    if out is None:
        out = torch.empty((B, k), dtype=torch.int32, device=scores.device)
    _out(out, (B, k), torch.int32, "idx")
    qp = _opt_pos(q_pos)
    _check(lib.csa2_topk(_ptr(scores), B, N, k, _ptr(qp), ratio, _ptr(out), _ptr(ws),
                         ws.numel(), _stream()), "csa2_topk")
    return out


def hier_pool_index(q_fp8: torch.Tensor, k_fp8: torch.Tensor, N: int, kv_seq_stride: int,
                    q_per_seq: int, pool: torch.Tensor, k: int, ws: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    q_fp8 = _dev(q_fp8, torch.uint8, "q_fp8")
    k_fp8 = _dev(k_fp8, torch.uint8, "k_fp8")
    pool = _dev(pool, torch.int32, "pool")
    B, H_I, D_I = q_fp8.shape
    P = pool.shape[1]
    if ws is None:
        ws = make_workspace(B, 0, k, 0, P, q_fp8.device)
    if out is None:
        out = torch.empty((B, k), dtype=torch.int32, device=q_fp8.device)
    _out(out, (B, k), torch.int32, "idx")
    _check(lib.csa2_hier_pool_index(_ptr(q_fp8), _ptr(k_fp8), B, H_I, D_I, N, kv_seq_stride,
                                    q_per_seq, _ptr(pool), P, k, _ptr(out), _ptr(ws), ws.numel(),
                                    _stream()), "csa2_hier_pool_index")
    return out


def block_pool(scores: torch.Tensor, block: int, n_blocks: int,
               q_pos: Optional[torch.Tensor] = None, ratio: int = 1,
               ws: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Blockwise candidate pool: fp32 scores [B][N] -> int32 pool [B][n_blocks * block]."""
    scores = _dev(scores, torch.float32, "scores")
    B, N = scores.shape
    qp = _opt_pos(q_pos)
    if ws is None:
        n = max(int(lib.csa2_block_pool_workspace_size(B, N, block, n_blocks)), 256)
        ws = torch.empty(n, dtype=torch.uint8, device=scores.device)
    if out is None:
        out = torch.empty((B, n_blocks * block), dtype=torch.int32, device=scores.device)
    _out(out, (B, n_blocks * block), torch.int32, "pool")
    _check(lib.csa2_block_pool(_ptr(scores), B, N, _ptr(qp), ratio, block, n_blocks, _ptr(out),
                               _ptr(ws), ws.numel(), _stream()), "csa2_block_pool")
    return out


def sparse_attn_fp4(q_bf16: torch.Tensor, kv_fp4: torch.Tensor, N: int, kv_seq_stride: int,
                    q_per_seq: int, idx: torch.Tensor, softmax_scale: Optional[float] = None,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    ws: Optional[torch.Tensor] = None, want_lse: bool = True):
    """bf16 q [B][H][512], FP4 rows [S*stride][288], idx [B][k] -> (out fp32 [B][H][512], lse)."""
    q = _bits16(q_bf16, "q_bf16")
    kv_fp4 = _dev(kv_fp4, torch.uint8, "kv_fp4")
    idx = _dev(idx, torch.int32, "idx")
    B, H, D = q.shape
    k = idx.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if ws is None:
        ws = make_workspace(B, 0, k, H, 0, q.device)
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float32, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _out(out, (B, H, D), torch.float32, "out")
    if lse is not None:
        _out(lse, (B, H), torch.float32, "lse")
    _check(lib.csa2_sparse_attn_fp4(_ptr(q), _ptr(kv_fp4), B, H, D, N, kv_seq_stride, q_per_seq,
                                    _ptr(idx), k, softmax_scale, _ptr(out), _ptr(lse), _ptr(ws),
                                    ws.numel(), _stream()), "csa2_sparse_attn_fp4")
    return out, lse


def sparse_attn_fp4_swa(q_bf16: torch.Tensor, kv_fp4: torch.Tensor, N: int, kv_seq_stride: int,
                        q_per_seq: int, idx: torch.Tensor, swa_kv: torch.Tensor, n_win: int,
                        q_pos: torch.Tensor, softmax_scale: Optional[float] = None,
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        ws: Optional[torch.Tensor] = None, want_lse: bool = True):
    """sparse_attn_fp4 plus each query's window of the layer's SWA KV (E4M3
    [S][ring][512], token t at row t mod ring) in the same softmax."""
    q = _bits16(q_bf16, "q_bf16")
    kv_fp4 = _dev(kv_fp4, torch.uint8, "kv_fp4")
    idx = _dev(idx, torch.int32, "idx")
    swa_kv = _dev(swa_kv, torch.uint8, "swa_kv")
    qp = _dev(q_pos, torch.int32, "q_pos")
    B, H, D = q.shape
    k = idx.shape[1]
    ring = swa_kv.shape[-2]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if ws is None:
        ws = make_workspace(B, 0, k, H, 0, q.device)
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.float32, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _out(out, (B, H, D), torch.float32, "out")
    if lse is not None:
        _out(lse, (B, H), torch.float32, "lse")
    _check(lib.csa2_sparse_attn_fp4_swa(_ptr(q), _ptr(kv_fp4), B, H, D, N, kv_seq_stride,
                                        q_per_seq, _ptr(idx), k, _ptr(swa_kv), ring, n_win,
                                        _ptr(qp), softmax_scale, _ptr(out), _ptr(lse), _ptr(ws),
                                        ws.numel(), _stream()), "csa2_sparse_attn_fp4_swa")
    return out, lse


class LayerGroup:
    """Prepared arguments of csa2_layer_group: tensors are kept alive and the
    ctypes structs are built once, so repeated calls (and CUDA-graph capture)
    only cross the C ABI."""

    def __init__(self, modes: Sequence[int], q_bf16: Sequence[torch.Tensor],
                 qi_fp8: Sequence[Optional[torch.Tensor]], kv_fp4: torch.Tensor,
                 ki_fp8: torch.Tensor, N: int, kv_seq_stride: int, q_per_seq: int,
                 q_pos: Optional[torch.Tensor], ratio: int, k: int, pool_size: int = 0,
                 softmax_scale: Optional[float] = None, want_lse: bool = True,
                 reuse_idx_copy: bool = True, pool_block: int = 0,
                 swa_kv: Optional[Sequence[Optional[torch.Tensor]]] = None, n_win: int = 0,
                 indexer_fmt: int = INDEXER_E4M3, q_ready: Optional[torch.cuda.Event] = None):
        L = len(modes)
        self.modes = list(modes)
        self.q = [_bits16(q, f"q_bf16[{l}]") for l, q in enumerate(q_bf16)]
        self.qi = [None if qi is None else _dev(qi, torch.uint8, f"qi_fp8[{l}]")
                   for l, qi in enumerate(qi_fp8)]
        self.kv = _dev(kv_fp4, torch.uint8, "kv_fp4")
        self.ki = _dev(ki_fp8, torch.uint8, "ki_fp8")
        self.q_pos = _opt_pos(q_pos)
        dev = self.kv.device
        B, H, D = self.q[0].shape
        H_I = D_I = 0
        for qi in self.qi:
            if qi is not None:
                _, H_I, D_I = qi.shape
                if indexer_fmt == INDEXER_MXFP4:
                    D_I = _mx_dim(D_I)
        if softmax_scale is None:
            softmax_scale = 1.0 / math.sqrt(D)
        self.B, self.H, self.D, self.k, self.N = B, H, D, k, N
        self.out = [torch.empty((B, H, D), dtype=torch.float32, device=dev) for _ in range(L)]
        self.lse = [torch.empty((B, H), dtype=torch.float32, device=dev) if want_lse else None
                    for _ in range(L)]
        self.idx = [torch.empty((B, k), dtype=torch.int32, device=dev)
                    if (m != REUSE or reuse_idx_copy) else None for m in self.modes]
        self.pool = (torch.empty((B, pool_size), dtype=torch.int32, device=dev)
                     if pool_size > 0 else None)
        self.ws = make_workspace(B, N, k, H, pool_size, dev)
        self.swa = ([None] * L if swa_kv is None else
                    [None if x is None else _dev(x, torch.uint8, f"swa_kv[{l}]")
                     for l, x in enumerate(swa_kv)])
        ring = next((x.shape[-2] for x in self.swa if x is not None), 0)
        self._layers = (Csa2Layer * L)()
        for l in range(L):
            self._layers[l] = Csa2Layer(self.modes[l], _ptr(self.q[l]), _ptr(self.qi[l]),
                                        _ptr(self.out[l]), _ptr(self.lse[l]), _ptr(self.idx[l]),
                                        _ptr(self.swa[l]))
        self._args = Csa2GroupArgs(_ptr(self.kv), _ptr(self.ki), B, H, H_I, D, D_I, N,
                                   kv_seq_stride, q_per_seq, _ptr(self.q_pos), ratio, k,
                                   pool_size, _ptr(self.pool), softmax_scale, pool_block, ring,
                                   n_win, indexer_fmt,
                                   q_ready.cuda_event if q_ready is not None else None)
        self._q_ready = q_ready   # kept alive with the struct that names it

    def __call__(self):
        _check(lib.csa2_layer_group(self._layers, len(self.modes), ctypes.byref(self._args),
                                    _ptr(self.ws), self.ws.numel(), _stream()),
               "csa2_layer_group")
        return self.out, self.lse, self.idx, self.pool


def group_launches(group: LayerGroup) -> int:
    """Kernel launches one call of `group` enqueues."""
    return int(lib.csa2_layer_group_launches(group._layers, len(group.modes),
                                             ctypes.byref(group._args)))


def layer_group(modes, q_bf16, qi_fp8, kv_fp4, ki_fp8, N, kv_seq_stride, q_per_seq, q_pos, ratio,
                k, pool_size=0, softmax_scale=None, pool_block=0, swa_kv=None, n_win=0,
                indexer_fmt=INDEXER_E4M3):
    """One-shot csa2_layer_group; returns (outs, lses, idxs, pool)."""
    return LayerGroup(modes, q_bf16, qi_fp8, kv_fp4, ki_fp8, N, kv_seq_stride, q_per_seq, q_pos,
                      ratio, k, pool_size, softmax_scale, pool_block=pool_block, swa_kv=swa_kv,
                      n_win=n_win, indexer_fmt=indexer_fmt)()
