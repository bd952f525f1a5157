"""Device-resident inputs of a synthetic CSA2 workload.

Draws the seeded inputs (``synthetic``), uploads them and writes the FP4
main-KV cache with the library's own packer (``csa2_quantize_kv_fp4``), one
sequence at a time so host memory stays bounded.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

from . import csa2
from .synthetic import FULL, REINDEX, REUSE, Workload


@dataclasses.dataclass
class DeviceInputs:
    w: Workload
    kv_fp4: torch.Tensor            # uint8 [S*N][288]
    ki_fp8: torch.Tensor            # uint8 [S*N][idx_row_bytes] indexer K (E4M3 or MXFP4)
    q: List[torch.Tensor]           # int16 (bf16 bits) [B][H][D] per layer
    qi: List[Optional[torch.Tensor]]  # uint8 [B][H_I][idx_row_bytes] per layer (None: REUSE)
    q_pos: torch.Tensor             # int32 [B]
    swa: Optional[List[torch.Tensor]] = None  # uint8 E4M3 [S][ring][D] per layer (n_win > 0)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.w.D))

    def layer_group(self, **kw) -> "csa2.LayerGroup":
        w = self.w
        return csa2.LayerGroup(w.modes, self.q, self.qi, self.kv_fp4, self.ki_fp8, w.N,
                               w.kv_seq_stride, w.q_per_seq, self.q_pos, w.ratio, w.k, w.pool,
                               self.scale, pool_block=w.pool_block, swa_kv=self.swa,
                               n_win=w.n_win, indexer_fmt=w.indexer_fmt, **kw)


def _to_dev(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False)


def prepare(w: Workload, device="cuda", layers: Optional[int] = None) -> DeviceInputs:
    S, N = w.n_seq, w.N
    kv = torch.empty((S * N, w.row_bytes), dtype=torch.uint8, device=device)
    ki = torch.empty((S * N, w.idx_row_bytes), dtype=torch.uint8, device=device)
    rows_per_chunk = max(1, min(N, (256 << 20) // (w.D * 4)))
    host = torch.empty((rows_per_chunk, w.D), dtype=torch.float32).pin_memory()
    dev_chunk = torch.empty((rows_per_chunk, w.D), dtype=torch.float32, device=device)
    for s in range(S):
        for r0 in range(0, N, rows_per_chunk):
            n = min(rows_per_chunk, N - r0)
            w.kv_latent(s, r0, n, out=host.numpy()[:n])
            dev_chunk[:n].copy_(host[:n], non_blocking=False)
            csa2.quantize_kv_fp4(dev_chunk[:n], out=kv[s * N + r0:s * N + r0 + n])
        ki[s * N:(s + 1) * N].copy_(torch.from_numpy(w.ki_rows(s)))
    torch.cuda.synchronize()
    L = len(w.modes) if layers is None else layers
    q = [_to_dev(w.q_bf16(l).view(np.int16), device) for l in range(L)]
    qi = [None if w.modes[l] == REUSE else _to_dev(w.qi_rows(l), device) for l in range(L)]
    q_pos = _to_dev(w.q_pos(), device)
    swa = None
    if w.n_win > 0:
        swa = [_to_dev(np.stack([w.swa_kv(l, s) for s in range(S)]), device) for l in range(L)]
    return DeviceInputs(w, kv, ki, q, qi, q_pos, swa)
