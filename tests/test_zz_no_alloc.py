"""csa2_sparse_attn_fp4_noalloc: the attention entry point for callers that
cannot allocate device memory (stream capture in progress, hosts that own all
allocations, loops that must not touch the allocator).  It must give the same
results as csa2_sparse_attn_fp4, which takes a caller workspace, on two calls
in a row (the second call reuses the library's fixed scratch array that the
first one filled).  Collected last on purpose; needs a GPU."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import ATTN_MAX_ABS, ATTN_REL_L2, assert_lse_close, attn_errors, bf16_bits

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512.0)


def _case(seed, B, H, N, k):
    rng = np.random.default_rng(seed)
    kv = oracle.quantize_kv_fp4(rng.standard_normal((B * N, 512)).astype(np.float32))
    q = bf16_bits(rng.standard_normal((B, H, 512)))
    idx = np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(B)]).astype(np.int32)
    idx[0, -7:] = -1
    return (torch.from_numpy(q.view(np.int16)).cuda(), torch.from_numpy(kv).cuda(),
            torch.from_numpy(idx).cuda())


def _noalloc(lib, q, kv, idx, N, out, lse):
    B, H, D = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.csa2_sparse_attn_fp4_noalloc(q.data_ptr(), kv.data_ptr(), B, H, D, N, N, 1,
                                           idx.data_ptr(), idx.shape[1], SCALE, out.data_ptr(),
                                           lse.data_ptr(), stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2
    lib = csa2.lib
    B, H, N, k = 4, 64, 5000, 4096       # 8 split chunks per query, their lse through scratch
    assert csa2.workspace_size(B, 0, k, H, 0) > 256
    for seed in (1, 2):                  # two calls in a row, different inputs
        q, kv, idx = _case(seed, B, H, N, k)
        ref_out, ref_lse = csa2.sparse_attn_fp4(q, kv, N, N, 1, idx, SCALE)
        out = torch.full((B, H, 512), float("nan"), device="cuda")
        lse = torch.full((B, H), float("nan"), device="cuda")
        assert _noalloc(lib, q, kv, idx, N, out, lse) == 0
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit-identical results
        assert torch.equal(out, ref_out), seed
        assert torch.equal(lse, ref_lse), seed
        if seed == 1:      # and within the attention tolerance of the fp64 oracle
            qn = q.cpu().numpy().view(np.uint16)
            o_ref, l_ref = oracle.sparse_attn(qn, kv.cpu().numpy(), N, N, 1, idx.cpu().numpy(),
                                              SCALE)
            max_abs, rel = attn_errors(out.cpu().numpy(), o_ref)
            assert max_abs <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (seed, max_abs, rel)
            assert_lse_close(lse.cpu().numpy(), l_ref)


def test_noalloc_rejects_requests_beyond_its_scratch():
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2
    B, H, k = 40, 64, 16384              # split partials of this request vs the fixed array
    q = torch.zeros((B, H, 512), dtype=torch.int16, device="cuda")
    kv = torch.zeros((100, 288), dtype=torch.uint8, device="cuda")
    idx = torch.full((B, k), -1, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, H, 512), device="cuda")
    lse = torch.zeros((B, H), device="cuda")
    if csa2.workspace_size(B, 0, k, H, 0) - 256 <= (256 << 10):
        pytest.skip("this device's split policy keeps the request small")
    assert _noalloc(csa2.lib, q, kv, idx, 100, out, lse) == 3      # CSA2_ERR_WORKSPACE
