"""Host-side validation of csa2_upload's segment table: every malformed table
is refused with CSA2_ERR_INVALID_ARG before anything is enqueued (no GPU
needed)."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def csa2():
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2 as c
    return c


def _buf(csa2, segs, payload_bytes=4096):
    n = len(segs)
    table = (csa2.Csa2UploadSeg * max(1, n))(*segs)
    size = n * ctypes.sizeof(csa2.Csa2UploadSeg) + payload_bytes
    buf = (ctypes.c_uint8 * size)()
    ctypes.memmove(buf, ctypes.addressof(table), n * ctypes.sizeof(csa2.Csa2UploadSeg))
    return buf, size


def _call(csa2, segs, payload_bytes=4096, stage=0x10000, stage_bytes=None):
    buf, size = _buf(csa2, segs, payload_bytes)
    return csa2.lib.csa2_upload(ctypes.addressof(buf), size, len(segs), stage,
                                size if stage_bytes is None else stage_bytes, None)


def test_table_entry_is_48_bytes(csa2):
    assert ctypes.sizeof(csa2.Csa2UploadSeg) == 48


@pytest.mark.parametrize("bad", [
    dict(kind=7),                                   # unknown kind
    dict(src_off=48 + 8),                           # payload not 16-byte aligned
    dict(src_off=16),                               # payload overlaps the table
    dict(rows=1000, row_bytes=1024),                # payload past the buffer
    dict(kind=1, row_bytes=1024),                   # FP4 rows take 2048-byte latent rows
    dict(kind=1, row_bytes=2048, rows=2, dst_stride=100),   # FP4 rows closer than 288 bytes
    dict(kind=1, row_bytes=2048, rows=1, dst=0x1008),       # FP4 destination not 16-byte aligned
    dict(rows=2, row_bytes=64, dst_stride=32),      # RAW rows overlapping
    dict(reserved=1),
    dict(dst=0),                                    # no destination
])
def test_malformed_segments_are_refused(csa2, bad):
    f = dict(dst=0x1000, src_off=48, rows=1, row_bytes=64, dst_stride=64, kind=0, reserved=0)
    f.update(bad)
    seg = csa2.Csa2UploadSeg(f["dst"], f["src_off"], f["rows"], f["row_bytes"], f["dst_stride"],
                             f["kind"], f["reserved"])
    assert _call(csa2, [seg]) == 1     # CSA2_ERR_INVALID_ARG


def test_malformed_calls_are_refused(csa2):
    seg = csa2.Csa2UploadSeg(0x1000, 48, 1, 64, 64, 0, 0)
    buf, size = _buf(csa2, [seg])
    up = csa2.lib.csa2_upload
    assert up(ctypes.addressof(buf), size, -1, 0x10000, size, None) == 1   # negative count
    assert up(ctypes.addressof(buf), 40, 1, 0x10000, size, None) == 1     # shorter than the table
    assert up(ctypes.addressof(buf), size, 1, 0x10000, size - 16, None) == 1  # staging too small
    assert up(ctypes.addressof(buf), size, 1, 0x10008, size, None) == 1    # staging misaligned
    assert up(None, size, 1, 0x10000, size, None) == 1
