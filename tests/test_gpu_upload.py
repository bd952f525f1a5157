"""csa2_upload on the GPU: one packed host buffer places raw rows (16-byte and
byte-granular paths, strided destinations) and packs fp32 latent rows into
FP4 cache rows bit-identical to the oracle's packer; bytes outside the
segments stay untouched."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def test_packed_upload_places_raw_rows_and_packs_fp4_rows():
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2
    rng = np.random.default_rng(11)
    big = torch.zeros((20, 256), dtype=torch.uint8, device="cuda")
    odd = torch.zeros((8, 64), dtype=torch.uint8, device="cuda")
    cache = torch.zeros((40, 288), dtype=torch.uint8, device="cuda")
    d_fast = big[3:13, 16:80]           # 10 rows of 64 bytes, 256 apart: 16-byte path
    d_odd = odd[1:6, 5:42]              # 5 rows of 37 bytes at an odd address: byte path
    d_fp4 = cache[2::3][:8]             # 8 FP4 rows, 864 bytes apart
    up = csa2.StepUpload([(csa2.UPLOAD_RAW, d_fast), (csa2.UPLOAD_RAW, d_odd),
                          (csa2.UPLOAD_KV_FP4, d_fp4)])
    raw1 = rng.integers(0, 256, (10, 64), dtype=np.uint8)
    raw2 = rng.integers(0, 256, (5, 37), dtype=np.uint8)
    lat = rng.standard_normal((8, 512)).astype(np.float32)
    lat[0] = 0.0                        # an all-zero row: zero scales
    lat[1, :16] = [448.0 * 6] + [0.1] * 15
    up.payloads[0].copy_(torch.from_numpy(raw1))
    up.payloads[1].copy_(torch.from_numpy(raw2))
    up.payloads[2].copy_(torch.from_numpy(lat))
    for _ in range(2):                  # the same buffers serve every call
        up()
        torch.cuda.synchronize()
        exp_big = np.zeros((20, 256), np.uint8)
        exp_big[3:13, 16:80] = raw1
        assert (big.cpu().numpy() == exp_big).all()
        exp_odd = np.zeros((8, 64), np.uint8)
        exp_odd[1:6, 5:42] = raw2
        assert (odd.cpu().numpy() == exp_odd).all()
        exp_cache = np.zeros((40, 288), np.uint8)
        exp_cache[2:26:3] = oracle.quantize_kv_fp4(lat)
        assert (cache.cpu().numpy() == exp_cache).all()
