"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle's tests.

This module draws random numbers and packs them into the input byte formats;
it performs none of the attention method's arithmetic (no quantisation of the
main KV, no scoring, no selection, no attention).

Recipe (one counter-based SplitMix64 stream per (workload, seed, tensor, layer),
defined in ``gen.c``):

* main-KV latent  : fp32 N(0,1) (Box-Muller in fp64, rounded to fp32), [N][512] per sequence
* indexer K       : integers U{-8..8} (or N(0,1) rounded to bf16 for the float workload),
                    stored as FP8 E4M3 with unit scale, [N][D_I] per sequence
* indexer q       : same distribution as indexer K, [H_I][D_I] per query and layer
* MXFP4 indexer   : (workloads with the MXFP4 indexer format) rows of D_I / 2 code bytes
                    and D_I / 32 E8M0 scale bytes drawn directly in that format: every
                    4-bit E2M1 code uniform over its 16 values (counter = element), every
                    scale byte uniform over {126, 127} (counter = 2^40 + block), for K and q
                    alike.  Values are then multiples of 1/4 and every score is a multiple
                    of 1/16 below 2^20, which fp32 holds exactly.
* main query      : bf16 N(0,1) (fp64 -> fp32 -> bf16, round-to-nearest-even), [H][512]
                    per query and layer
* query positions : the last token of each decode context, or consecutive tokens
                    at the end of the context for the prefill-shaped workload

The E4M3 bytes of the indexer inputs come from PyTorch's float8_e4m3fn cast
(round-to-nearest-even) after clamping to +-448; for integers in [-8, 8] the
cast is exact.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_libcsa2gen.so")
_lock = threading.Lock()
_lib = None

NTHREADS = max(1, min(32, os.cpu_count() or 1))

TENSOR_KV = 1
TENSOR_KI = 2
TENSOR_QI = 3
TENSOR_Q = 4
TENSOR_SWA = 5


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i32, vp = ctypes.c_uint64, ctypes.c_int32, ctypes.c_void_p
            lib.csa2gen_stream_key.restype = u64
            lib.csa2gen_stream_key.argtypes = [u64, u64, u64]
            lib.csa2gen_draw.restype = u64
            lib.csa2gen_draw.argtypes = [u64, u64]
            for name in ("csa2gen_normal_f64", "csa2gen_normal_f32", "csa2gen_normal_bf16"):
                getattr(lib, name).restype = None
                getattr(lib, name).argtypes = [u64, u64, u64, vp, ctypes.c_int]
            for name in ("csa2gen_uniform_i8", "csa2gen_uniform_i32"):
                getattr(lib, name).restype = None
                getattr(lib, name).argtypes = [u64, u64, u64, i32, i32, vp, ctypes.c_int]
            _lib = lib
    return _lib


def stream_key(workload_id: int, seed: int, tensor: int, layer: int = 0) -> int:
    return int(_load().csa2gen_stream_key(workload_id, seed, tensor * 256 + layer))


def draw(key: int, i: int) -> int:
    return int(_load().csa2gen_draw(key, i))


def normal_f64(key: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    _load().csa2gen_normal_f64(key, start, count, out.ctypes.data, NTHREADS)
    return out


def normal_f32(key: int, start: int, count: int, out: Optional[np.ndarray] = None) -> np.ndarray:
    if out is None:
        out = np.empty(count, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == count
    _load().csa2gen_normal_f32(key, start, count, out.ctypes.data, NTHREADS)
    return out


def normal_bf16(key: int, start: int, count: int) -> np.ndarray:
    """bf16 bit patterns (uint16)."""
    out = np.empty(count, dtype=np.uint16)
    _load().csa2gen_normal_bf16(key, start, count, out.ctypes.data, NTHREADS)
    return out


def uniform_int8(key: int, start: int, count: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(count, dtype=np.int8)
    _load().csa2gen_uniform_i8(key, start, count, lo, hi, out.ctypes.data, NTHREADS)
    return out


def float_to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Encode float values as FP8 E4M3 bytes (RNE, saturating at +-448) with PyTorch's cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

FULL, REINDEX, REUSE = 0, 1, 2
MODE_NAMES = {FULL: "FULL", REINDEX: "REINDEX", REUSE: "REUSE"}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape, seeds and layer schedule of one synthetic CSA2 workload."""
    name: str
    workload_id: int
    B: int                 # queries
    N: int                 # compressed entries per sequence
    H: int                 # main query heads
    H_I: int               # indexer heads
    k: int                 # top-k
    ratio: int = 4         # compression ratio (tokens per entry)
    D: int = 512           # latent channels
    D_I: int = 64          # indexer head dim
    q_per_seq: int = 1     # queries sharing one context (sequence index = q // q_per_seq)
    seeds: Sequence[int] = (0,)          # one seed per sequence
    first_pos: Optional[int] = None      # position of query 0 of each sequence (None: last token)
    modes: Sequence[int] = (FULL,)
    pool: int = 0          # hierarchical candidate pool size (0 = flat indexer)
    pool_block: int = 0    # > 1: blockwise pool of pool / pool_block blocks (else top-pool)
    float_indexer: bool = False          # bf16 N(0,1) indexer inputs instead of integers
    n_win: int = 0         # SWA window of every layer (0: no SWA branch)
    swa_ring: int = 0      # rows of each sequence's SWA KV ring
    indexer_fmt: int = 0   # 0: E4M3 indexer rows of D_I bytes; 1: MXFP4 rows

    @property
    def n_seq(self) -> int:
        return self.B // self.q_per_seq

    @property
    def row_bytes(self) -> int:
        return self.D // 2 + self.D // 16

    @property
    def kv_seq_stride(self) -> int:
        return self.N

    @property
    def idx_row_bytes(self) -> int:
        """Bytes of one indexer q or K row in the workload's indexer format."""
        return self.D_I // 2 + self.D_I // 32 if self.indexer_fmt else self.D_I

    def seed_of_seq(self, s: int) -> int:
        return int(self.seeds[s])

    def q_pos(self) -> np.ndarray:
        ctx = self.N * self.ratio
        pos = np.empty(self.B, dtype=np.int32)
        for q in range(self.B):
            j = q % self.q_per_seq
            if self.first_pos is None:
                pos[q] = ctx - 1
            else:
                pos[q] = self.first_pos + j
        return pos

    # --- per-sequence tensors ----------------------------------------------
    def kv_latent(self, s: int, row_start: int = 0, n_rows: Optional[int] = None,
                  out: Optional[np.ndarray] = None) -> np.ndarray:
        """fp32 [n_rows][D] main-KV latent rows of sequence s."""
        if n_rows is None:
            n_rows = self.N - row_start
        key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_KV)
        flat = None if out is None else out.reshape(-1)
        return normal_f32(key, row_start * self.D, n_rows * self.D, flat).reshape(n_rows, self.D)

    def kv_latent_rows(self, s: int, rows: np.ndarray) -> np.ndarray:
        """fp32 [len(rows)][D] latent for an arbitrary set of row indices of sequence s."""
        rows = np.asarray(rows, dtype=np.int64)
        out = np.empty((rows.size, self.D), dtype=np.float32)
        for i, r in enumerate(rows):
            out[i] = self.kv_latent(s, int(r), 1)[0]
        return out

    def _indexer_values(self, key: int, start: int, count: int) -> np.ndarray:
        if self.float_indexer:
            return bf16_bits_to_float(normal_bf16(key, start, count))
        return uniform_int8(key, start, count, -8, 8).astype(np.float32)

    def ki_fp8(self, s: int) -> np.ndarray:
        """E4M3 bytes [N][D_I] of sequence s's indexer K."""
        key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_KI)
        vals = self._indexer_values(key, 0, self.N * self.D_I)
        return float_to_e4m3_bytes(vals).reshape(self.N, self.D_I)

    def _mx_rows(self, key: int, row0: int, n_rows: int) -> np.ndarray:
        """MXFP4 rows [n_rows][D_I/2 + D_I/32] drawn in the format (see the recipe)."""
        d = self.D_I
        nib = uniform_int8(key, row0 * d, n_rows * d, 0, 15).astype(np.uint8).reshape(n_rows, d)
        sc = uniform_int8(key, (1 << 40) + row0 * (d // 32), n_rows * (d // 32), 126, 127)
        out = np.empty((n_rows, d // 2 + d // 32), dtype=np.uint8)
        out[:, :d // 2] = nib[:, 0::2] | (nib[:, 1::2] << 4)
        out[:, d // 2:] = sc.astype(np.uint8).reshape(n_rows, d // 32)
        return out

    def ki_rows(self, s: int) -> np.ndarray:
        """Indexer K [N][idx_row_bytes] of sequence s in the workload's indexer format."""
        if not self.indexer_fmt:
            return self.ki_fp8(s)
        key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_KI)
        return self._mx_rows(key, 0, self.N)

    def qi_rows(self, layer: int, qs: Optional[Sequence[int]] = None) -> np.ndarray:
        """Indexer queries [len(qs)][H_I][idx_row_bytes] of one layer in the indexer format."""
        if not self.indexer_fmt:
            return self.qi_fp8(layer, qs)
        qs = range(self.B) if qs is None else qs
        out = []
        for q in qs:
            s, j = divmod(q, self.q_per_seq)
            key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_QI, layer)
            out.append(self._mx_rows(key, j * self.H_I, self.H_I))
        if not out:
            return np.zeros((0, self.H_I, self.idx_row_bytes), np.uint8)
        return np.stack(out)

    def swa_kv(self, layer: int, s: int) -> np.ndarray:
        """E4M3 bytes [swa_ring][D] of layer `layer`'s SWA KV ring of sequence s
        (token t at row t mod swa_ring): N(0,1) latents cast to E4M3."""
        key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_SWA, layer)
        vals = normal_f32(key, 0, self.swa_ring * self.D)
        return float_to_e4m3_bytes(vals).reshape(self.swa_ring, self.D)

    # --- per-query, per-layer tensors --------------------------------------
    def qi_fp8(self, layer: int, qs: Optional[Sequence[int]] = None) -> np.ndarray:
        """E4M3 bytes [len(qs)][H_I][D_I] of the indexer queries of one layer."""
        qs = range(self.B) if qs is None else qs
        sz = self.H_I * self.D_I
        out = []
        for q in qs:
            s, j = divmod(q, self.q_per_seq)
            key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_QI, layer)
            out.append(self._indexer_values(key, j * sz, sz))
        vals = np.stack(out) if out else np.zeros((0, sz), np.float32)
        return float_to_e4m3_bytes(vals).reshape(len(out), self.H_I, self.D_I)

    def q_bf16(self, layer: int, qs: Optional[Sequence[int]] = None) -> np.ndarray:
        """bf16 bits [len(qs)][H][D] of the main queries of one layer."""
        qs = range(self.B) if qs is None else qs
        sz = self.H * self.D
        if self.q_per_seq > 1 and qs is not None and len(qs) > 0 and list(qs) == list(range(self.B)):
            # contiguous query runs per sequence: generate in bulk
            out = np.empty((self.B, sz), dtype=np.uint16)
            for s in range(self.n_seq):
                key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_Q, layer)
                out[s * self.q_per_seq:(s + 1) * self.q_per_seq] = normal_bf16(
                    key, 0, self.q_per_seq * sz).reshape(self.q_per_seq, sz)
            return out.reshape(self.B, self.H, self.D)
        rows = []
        for q in qs:
            s, j = divmod(q, self.q_per_seq)
            key = stream_key(self.workload_id, self.seed_of_seq(s), TENSOR_Q, layer)
            rows.append(normal_bf16(key, j * sz, sz))
        return np.stack(rows).reshape(len(rows), self.H, self.D)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _seeds(first: int, n: int) -> List[int]:
    return list(range(first, first + n))


# The five workloads.  Sizes follow the CSA2 configuration of the
# DeepSeek-V4.1-Flash pages (64 x 512 MQA heads, FP4 E2M1 + E4M3/16 main KV,
# ratio-4 compression); the remaining parameters are fixed here.
TINY_FULL = Workload("tiny_full_1q_ctx4k", 1, B=1, N=1024, H=16, H_I=4, k=128, seeds=(0,))
DECODE_64K = Workload("decode_b32_ctx64k", 2, B=32, N=16384, H=64, H_I=8, k=2048,
                      seeds=tuple(_seeds(1, 32)))
GROUP_128K = Workload("group_full_reindex_reuse_b64_ctx128k", 3, B=64, N=32768, H=64, H_I=8,
                      k=2048, seeds=tuple(_seeds(3000, 64)), modes=(FULL, REINDEX, REUSE))
HIER_1M = Workload("hier_pool8192_b16_ctx1m", 4, B=16, N=262144, H=64, H_I=8, k=2048,
                   seeds=tuple(_seeds(4000, 16)), modes=(FULL, REINDEX, REINDEX, REINDEX),
                   pool=8192)
# The pages' own candidate pool: at most 2048 blocks of 8 positions (16384
# candidates), block score = max index score in the block.
HIER_BLOCK_1M = Workload("hier_block2048x8_b16_ctx1m", 6, B=16, N=262144, H=64, H_I=8, k=2048,
                         seeds=tuple(_seeds(6000, 16)), modes=(FULL, REINDEX, REINDEX, REINDEX),
                         pool=16384, pool_block=8)
# Decode with every query's own 128-token SWA window in the same softmax.
DECODE_64K_SWA = Workload("decode_swa128_b32_ctx64k", 7, B=32, N=16384, H=64, H_I=8, k=2048,
                          seeds=tuple(_seeds(7000, 32)), n_win=128, swa_ring=128)
# The pages' production decoder: 20 CSA2 layers at m = 1 in five groups of four
# (Full + 3 Reuse, then Reindex + 3 Reuse four times), indexer 32 heads x 128,
# top-k 512, blockwise pool of at most 2048 blocks x 8, SWA window 128.
DECODER20 = Workload("decoder20_prod_b32_ctx64k", 8, B=32, N=65536, H=64, H_I=32, D_I=128, k=512,
                     ratio=1, seeds=tuple(_seeds(8000, 32)),
                     modes=(FULL, REUSE, REUSE, REUSE) + (REINDEX, REUSE, REUSE, REUSE) * 4,
                     pool=16384, pool_block=8, n_win=128, swa_ring=128)
# The production decoder with the indexer query and key in MXFP4 (68-byte rows).
DECODER20_MX = Workload("decoder20_mxfp4_b32_ctx64k", 9, B=32, N=65536, H=64, H_I=32, D_I=128,
                        k=512, ratio=1, seeds=tuple(_seeds(9000, 32)),
                        modes=(FULL, REUSE, REUSE, REUSE) + (REINDEX, REUSE, REUSE, REUSE) * 4,
                        pool=16384, pool_block=8, n_win=128, swa_ring=128, indexer_fmt=1)
# The pages' production encoder: 18 CSA2 layers at m = 2 in three groups of six
# (Full + 5 Reuse), indexer 32 heads x 128, top-k 512, SWA window 128; a chunk of
# the last 512 prompt tokens of a 64K-token prompt (ring of 1024 SWA rows holds
# every window the chunk reads).
ENCODER18 = Workload("encoder18_chunk512_ctx64k", 10, B=512, N=32768, H=64, H_I=32, D_I=128,
                     k=512, ratio=2, q_per_seq=512, seeds=(10000,), first_pos=65536 - 512,
                     modes=(FULL,) + (REUSE,) * 5 + (FULL,) + (REUSE,) * 5 + (FULL,) + (REUSE,) * 5,
                     n_win=128, swa_ring=1024)
PREFILL_128K = Workload("prefill_4096q_ctx128k", 5, B=4096, N=32768, H=64, H_I=8, k=2048,
                        q_per_seq=4096, seeds=(5000,), first_pos=126976, float_indexer=True)

WORKLOADS = {w.name: w for w in (TINY_FULL, DECODE_64K, GROUP_128K, HIER_1M, PREFILL_128K,
                                  HIER_BLOCK_1M, DECODE_64K_SWA, DECODER20, DECODER20_MX,
                                  ENCODER18)}
