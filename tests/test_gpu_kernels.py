"""Per-kernel parity of the CUDA path (through the C ABI) against the oracle at
small, ragged sizes that still span several tiles.  Needs a GPU."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines, parse_float
from helpers import (assert_attn_close, assert_float_selection_ok, assert_lse_close, bf16_bits,
                     cuda, e4m3_bytes, int_e4m3)

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512.0)


@pytest.fixture(scope="module")
def C():
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2
    return csa2


# ---------------------------------------------------------------- FP4 packer

def _golden_rows():
    blocks = []
    for line in golden_lines("fp4_blocks.txt"):
        vals = line.split("|")[0].split()
        blocks.append(np.array([parse_float(t) for t in vals], np.float32))
    rows = np.zeros((len(blocks), 512), np.float32)
    for i, b in enumerate(blocks):
        for p in range(32):
            rows[i, 16 * p:16 * p + 16] = blocks[(i + p) % len(blocks)]
    return rows


def test_quantize_bit_exact(C):
    rng = np.random.default_rng(0)
    n = 20000 + 7
    x = rng.standard_normal((n, 512)).astype(np.float32)
    x *= rng.choice([1e-4, 1e-2, 0.3, 1.0, 17.0, 900.0], (n, 1)).astype(np.float32)
    x[::97, 5:40] = 0.0
    x[::89, 100] = -0.0
    x = np.concatenate([x, _golden_rows()])
    got = C.quantize_kv_fp4(cuda(x)).cpu().numpy()
    ref = oracle.quantize_kv_fp4(x)
    assert got.shape == (x.shape[0], 288)
    assert (got == ref).all(), np.argwhere(got != ref)[:5]


def test_quantize_midpoints_and_neighbours_bit_exact(C):
    # blocks whose scale is each E4M3 value s (absmax = 6 s), elements at every E2M1
    # midpoint t*s and the fp32 numbers next to it
    svals = [oracle.e4m3_value(b) for b in range(1, 0x7F)]
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for s in svals:
        blk = [np.float32(6 * s)]
        for t in mids:
            m = np.float32(t * s)
            blk += [m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(1e9))]
        blk = np.array(blk[:16], np.float32)
        blk2 = -np.array([np.float32(6 * s)] + [np.float32(t * s) for t in mids] * 2 + [0.0],
                         np.float32)
        assert blk.size == 16 and blk2.size == 16
        row = np.zeros(512, np.float32)
        for p in range(16):
            row[32 * p:32 * p + 16] = blk
            row[32 * p + 16:32 * p + 32] = blk2
        rows.append(row)
    x = np.stack(rows)
    got = C.quantize_kv_fp4(cuda(x)).cpu().numpy()
    assert (got == oracle.quantize_kv_fp4(x)).all()


def test_quantize_empty_is_a_no_op(C):
    out = C.quantize_kv_fp4(torch.zeros((0, 512), device="cuda"))
    assert out.shape == (0, 288)


# ---------------------------------------------------------------- indexer scores

@pytest.mark.parametrize("B,N,H_I,D_I,q_per_seq", [
    (3, 1000, 4, 64, 1), (4, 777, 8, 32, 2), (2, 513, 32, 128, 1), (48, 700, 8, 64, 16),
    (32, 3000, 8, 64, 32), (1, 1024, 4, 64, 1)])
def test_index_scores_exact_for_integer_inputs(C, B, N, H_I, D_I, q_per_seq):
    rng = np.random.default_rng(B * 1000 + N)
    S = B // q_per_seq
    qi = int_e4m3(rng, (B, H_I, D_I))
    ki = int_e4m3(rng, (S * N, D_I))
    pos = rng.integers(-2, 4 * N + 9, B).astype(np.int32)
    pos[0] = 4 * N - 1
    got = C.index_scores(cuda(qi), cuda(ki), N, N, q_per_seq, cuda(pos), 4).cpu().numpy()
    ref = oracle.index_scores(qi, ki, N, N, q_per_seq, pos, 4)
    assert (got.astype(np.float64) == ref).all()
    got = C.index_scores(cuda(qi), cuda(ki), N, N, q_per_seq, None, 4).cpu().numpy()
    assert np.isfinite(got).all()


@pytest.mark.parametrize("q_per_seq", [1, 16])
def test_index_scores_float_inputs_within_fp32_rounding(C, q_per_seq):
    rng = np.random.default_rng(5)
    B, N, H_I, D_I = 32, 1500, 8, 64
    qi = e4m3_bytes(rng.standard_normal((B, H_I, D_I)))
    ki = e4m3_bytes(rng.standard_normal(((B // q_per_seq) * N, D_I)))
    got = C.index_scores(cuda(qi), cuda(ki), N, N, q_per_seq, None, 4).cpu().numpy()
    ref = oracle.index_scores(qi, ki, N, N, q_per_seq, None, 4)
    # bound: 64-term fp32 sum of exactly representable products (head sum is exact)
    qf = torch.from_numpy(qi).view(torch.float8_e4m3fn).double().sum(1).numpy()      # [B][D_I]
    kf = torch.from_numpy(ki).view(torch.float8_e4m3fn).double().numpy()
    for q in range(B):
        s = q // q_per_seq
        mag = np.abs(kf[s * N:(s + 1) * N]) @ np.abs(qf[q])
        assert (np.abs(got[q] - ref[q]) <= 64 * 2.0 ** -24 * mag + 1e-30).all()


# ---------------------------------------------------------------- top-k

@pytest.mark.parametrize("B,N,k,kind", [
    (5, 1000, 7, "ties"), (3, 16384 + 37, 2048, "ties"), (2, 50000, 2048, "ties"),
    (2, 50000, 4096, "normal"), (4, 3000, 1, "normal"), (3, 700, 2048, "ties"),
    (2, 2048, 2048, "normal"), (2, 1000, 128, "equal"), (2, 70000, 100, "signed_zero"),
    (16, 8192, 2048, "ties"), (2, 262144, 8192, "ties"), (3, 300001, 2048, "normal"),
    (2, 262144, 16384, "ties"), (2, 1 << 21, 2048, "ties"),
    # dispatch boundaries: clusters of 8 (B <= 19, N >= 16384), 4 (B <= 38, N >= 8192) and
    # 2 (B <= 76, N >= 4096) CTAs per row, one CTA per row beyond or for shorter rows; a row
    # length that is no multiple of 4
    (19, 32768, 2048, "ties"), (38, 20001, 1000, "normal"), (40, 5000, 300, "ties"),
    (2, 32768, 16384, "ties"), (7, 32767, 4095, "equal"), (4, 8192, 700, "normal"),
    (4, 16383, 2048, "ties"),
    # clusters of 2 (39 <= B <= 76), and the last level of a long row on a cluster
    (64, 32768, 2048, "ties"), (76, 4096, 100, "normal"), (50, 20001, 3000, "normal"),
    (16, 262144, 2048, "ties")])
def test_topk_bit_exact(C, B, N, k, kind):
    rng = np.random.default_rng(N + k)
    if kind == "ties":
        s = rng.integers(-40, 40, (B, N)).astype(np.float32) * 64
    elif kind == "normal":
        s = rng.standard_normal((B, N)).astype(np.float32)
    elif kind == "equal":
        s = np.full((B, N), 3.5, np.float32)
    else:
        s = np.where(rng.random((B, N)) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        s[:, ::7] = -1.0
    pos = rng.integers(-1, 4 * N + 4, B).astype(np.int32)
    pos[0] = 4 * N + 100
    ws = C.make_workspace(B, N, k)
    got = C.topk(cuda(s), k, cuda(pos), 4, ws).cpu().numpy()
    ref = oracle.topk(s.astype(np.float64), k, pos, 4)
    assert (got == ref).all()
    got = C.topk(cuda(s), k, None, 1, ws).cpu().numpy()
    assert (got == oracle.topk(s.astype(np.float64), k)).all()


@pytest.mark.parametrize("B,N,k,kind", [
    (2, 40000, 2048, "ties"), (2, 40000, 8192, "normal"), (2, 262144, 2048, "normal"),
    (2, 262144, 8192, "ties"), (3, 50000, 20000, "ties"), (1, 2200000, 2048, "normal"),
    (2, 40000, 3000, "equal")])
def test_topk_one_kernel_long_rows_bit_exact(C, B, N, k, kind):
    # Rows longer than 32768 candidates take the one-kernel selection when the
    # workspace holds only the 256-byte status word, when k > 16384, or when a
    # row needs more than 64 chunks of 32768 (N > 2^21); ties still go to the
    # lower index and the output is ascending, -1 padded.
    rng = np.random.default_rng(3 * N + k)
    if kind == "ties":
        s = rng.integers(-40, 40, (B, N)).astype(np.float32) * 64
    elif kind == "normal":
        s = rng.standard_normal((B, N)).astype(np.float32)
    else:
        s = np.full((B, N), -2.25, np.float32)
    pos = rng.integers(4 * 30000, 4 * N + 4, B).astype(np.int32)
    pos[0] = 4 * N + 100
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert C.workspace_size(B, N, k) > 256 or N > (1 << 21) or k > 16384
    got = C.topk(cuda(s), k, cuda(pos), 4, small).cpu().numpy()
    ref = oracle.topk(s.astype(np.float64), k, pos, 4)
    assert (got == ref).all()
    got = C.topk(cuda(s), k, None, 1, small).cpu().numpy()
    assert (got == oracle.topk(s.astype(np.float64), k)).all()
    assert C.read_status(small) == (0, 0)


def test_topk_with_infinities(C):
    rng = np.random.default_rng(9)
    s = rng.integers(-3, 3, (3, 5000)).astype(np.float32)
    s[:, ::3] = -np.inf
    s[1, ::11] = np.inf
    got = C.topk(cuda(s), 1700).cpu().numpy()
    assert (got == oracle.topk(s.astype(np.float64), 1700)).all()


# ---------------------------------------------------------------- hierarchical pool

@pytest.mark.parametrize("N,P,k", [(5000, 1024, 128), (262144 // 8, 8192, 2048), (3000, 700, 800)])
def test_hier_pool_bit_exact(C, N, P, k):
    rng = np.random.default_rng(P)
    B, H_I, D_I = 4, 8, 64
    qi0 = int_e4m3(rng, (B, H_I, D_I))
    qi1 = int_e4m3(rng, (B, H_I, D_I))
    ki = int_e4m3(rng, (B * N, D_I))
    pos = np.array([4 * N - 1, 4 * (P // 2) - 1, 4 * N - 1, 4 * (N // 3)], np.int32)
    pool = oracle.topk(oracle.index_scores(qi0, ki, N, N, 1, pos, 4), P, pos, 4)
    got = C.hier_pool_index(cuda(qi1), cuda(ki), N, N, 1, cuda(pool), k).cpu().numpy()
    ref = oracle.hier_pool_index(qi1, ki, N, N, 1, pool, k)
    assert (got == ref).all()


@pytest.mark.parametrize("P,k", [(40000, 2048), (40000, 8192)])
def test_hier_pool_longer_than_one_cta_bit_exact(C, P, k):
    # a pool of more than 32768 candidates: selected through the position map
    # by the one-kernel long-row selection
    rng = np.random.default_rng(P + k)
    B, N, H_I, D_I = 2, 50000, 8, 64
    qi0 = int_e4m3(rng, (B, H_I, D_I))
    qi1 = int_e4m3(rng, (B, H_I, D_I))
    ki = int_e4m3(rng, (B * N, D_I))
    pos = np.array([4 * N - 1, 4 * (N - 3000)], np.int32)
    pool = oracle.topk(oracle.index_scores(qi0, ki, N, N, 1, pos, 4), P, pos, 4)
    got = C.hier_pool_index(cuda(qi1), cuda(ki), N, N, 1, cuda(pool), k).cpu().numpy()
    assert (got == oracle.hier_pool_index(qi1, ki, N, N, 1, pool, k)).all()


def test_hier_pool_flags_unsorted_pool(C):
    rng = np.random.default_rng(1)
    B, N, P = 2, 500, 64
    qi = int_e4m3(rng, (B, 4, 64))
    ki = int_e4m3(rng, (B * N, 64))
    pool = np.stack([np.sort(rng.choice(N, P, replace=False)) for _ in range(B)]).astype(np.int32)
    ws = C.make_workspace(B, 0, 8, 0, P)
    C.hier_pool_index(cuda(qi), cuda(ki), N, N, 1, cuda(pool), 8, ws)
    assert C.read_status(ws) == (0, 0)
    bad = pool.copy()
    bad[1, 10], bad[1, 11] = bad[1, 11], bad[1, 10]
    C.hier_pool_index(cuda(qi), cuda(ki), N, N, 1, cuda(bad), 8, ws)
    code, bits = C.read_status(ws)
    assert code == 5 and bits & 1


# ---------------------------------------------------------------- attention

def _attn_case(rng, B, H, N, k, pad=0, dup=False, q_per_seq=1):
    S = B // q_per_seq
    x = rng.standard_normal((S * N, 512)).astype(np.float32)
    kv = oracle.quantize_kv_fp4(x)
    q = bf16_bits(rng.standard_normal((B, H, 512)))
    idx = np.stack([rng.choice(N, k, replace=False) for _ in range(B)]).astype(np.int32)
    idx.sort(1)
    if pad:
        idx[:, k - pad:] = -1
        idx[0, ::5] = -1
    if dup:
        idx[-1, 1::2] = idx[-1, 0::2][: len(idx[-1, 1::2])]
    return kv, q, idx


@pytest.mark.parametrize("B,H,N,k,pad,dup", [
    (2, 64, 3000, 2048, 0, False), (3, 64, 900, 333, 40, True), (1, 16, 1024, 128, 0, False),
    (5, 32, 600, 257, 3, False), (4, 64, 70, 1, 0, False), (2, 16, 5000, 4096, 100, False),
    (40, 64, 2200, 2048, 0, False),
    # a query's slots split over 4, 8 and 2 CTAs, then merged
    (32, 64, 3000, 2048, 0, False), (16, 16, 3000, 2048, 7, False),
    (64, 32, 1500, 1024, 0, False),
    # one CTA per query (B above the SM count) over more slots than the kernel keeps in
    # shared memory: slots past the first 2048 are read from global memory
    (153, 16, 3000, 2500, 3, False)])
def test_attention_matches_oracle(C, B, H, N, k, pad, dup):
    rng = np.random.default_rng(B * 7 + H + k)
    kv, q, idx = _attn_case(rng, B, H, N, k, pad, dup)
    out, lse = C.sparse_attn_fp4(cuda(q, torch.int16), cuda(kv), N, N, 1, cuda(idx), SCALE)
    ref_o, ref_l = oracle.sparse_attn(q, kv, N, N, 1, idx, SCALE)
    assert_attn_close(out.cpu().numpy(), ref_o, (B, H, N, k))
    assert_lse_close(lse.cpu().numpy(), ref_l)


def test_attention_shared_context_and_empty_rows(C):
    rng = np.random.default_rng(11)
    B, H, N, k = 6, 64, 800, 300
    kv, q, idx = _attn_case(rng, B, H, N, k, q_per_seq=6)
    idx[2] = -1                      # no valid entry: out 0, lse -inf
    out, lse = C.sparse_attn_fp4(cuda(q, torch.int16), cuda(kv), N, 0, 6, cuda(idx), SCALE)
    ref_o, ref_l = oracle.sparse_attn(q, kv, N, 0, 6, idx, SCALE)
    assert_attn_close(out.cpu().numpy(), ref_o)
    assert_lse_close(lse.cpu().numpy(), ref_l)
    assert (out[2] == 0).all() and torch.isneginf(lse[2]).all()


def test_attention_out_of_range_index_sets_status_and_is_skipped(C):
    rng = np.random.default_rng(12)
    B, H, N, k = 2, 64, 500, 100
    kv, q, idx = _attn_case(rng, B, H, N, k)
    ws = C.make_workspace(B, N, k, H)
    C.sparse_attn_fp4(cuda(q, torch.int16), cuda(kv), N, N, 1, cuda(idx), SCALE, ws=ws)
    assert C.read_status(ws) == (0, 0)
    bad = idx.copy()
    bad[1, 3] = N + 5
    bad[0, 7] = -9
    out, _ = C.sparse_attn_fp4(cuda(q, torch.int16), cuda(kv), N, N, 1, cuda(bad), SCALE, ws=ws)
    code, bits = C.read_status(ws)
    assert code == 5 and (bits & 1)
    skip = bad.copy()
    skip[1, 3] = -1
    skip[0, 7] = -1
    ref_o, _ = oracle.sparse_attn(q, kv, N, N, 1, skip, SCALE)
    assert_attn_close(out.cpu().numpy(), ref_o)


# ---------------------------------------------------------------- blockwise pool

@pytest.mark.parametrize("B,N,block,nblk,ties", [(3, 1000, 8, 20, False), (4, 4096, 8, 64, True),
                                                (2, 777, 3, 300, True), (5, 70000, 8, 2048, False),
                                                (2, 262144, 8, 2048, True), (3, 129, 1, 40, True)])
def test_block_pool_bit_exact(C, B, N, block, nblk, ties):
    # walkthrough 1.(4).2: block score = max over its visible entries, top
    # blocks by (score desc, block asc), pool = their visible entries, -1 padded
    rng = np.random.default_rng(B * 1000 + block + nblk)
    if ties:
        scores = rng.integers(-40, 41, (B, N)).astype(np.float32)
    else:
        scores = rng.standard_normal((B, N)).astype(np.float32)
    ratio = 4
    pos = rng.integers(-2, ratio * N + 5, B).astype(np.int32)
    pos[0] = ratio * N - 1            # everything visible
    if B > 2:
        pos[1] = ratio * 5 + 2        # 5 visible entries: fewer blocks than asked
    got = C.block_pool(cuda(scores), block, nblk, cuda(pos), ratio).cpu().numpy()
    want = oracle.block_pool(scores.astype(np.float64), block, nblk, pos, ratio)
    assert np.array_equal(got, want)


def test_layer_group_with_blockwise_pool_matches_oracle(C):
    rng = np.random.default_rng(77)
    modes = (0, 1, 2, 1)
    B, N, H, H_I, k = 3, 6000, 64, 8, 256
    kv, ki, qs, qis, pos = _group(rng, B, N, H, H_I, k, modes, 0)
    outs, lses, idxs, gpool = C.layer_group(modes, [cuda(q, torch.int16) for q in qs],
                                            [None if qi is None else cuda(qi) for qi in qis],
                                            cuda(kv), cuda(ki), N, N, 1, cuda(pos), 4, k, 1024,
                                            SCALE, pool_block=8)
    r_outs, r_lses, r_idxs, r_pool = oracle.layer_group(modes, qs, qis, kv, ki, N, N, 1, pos, 4,
                                                        k, 1024, SCALE, pool_block=8)
    assert (gpool.cpu().numpy() == r_pool).all()
    for l in range(len(modes)):
        assert (idxs[l].cpu().numpy() == r_idxs[l]).all(), l
        assert_attn_close(outs[l].cpu().numpy(), r_outs[l], l)
        assert_lse_close(lses[l].cpu().numpy(), r_lses[l])


# ---------------------------------------------------------------- SWA branch

def _swa_rows(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("B,H,k,n_win,ring,want_lse", [
    (4, 64, 2048, 128, 128, True), (3, 16, 300, 128, 200, True), (2, 32, 777, 7, 16, False),
    (5, 64, 64, 300, 512, True), (40, 64, 1024, 128, 130, True), (2, 64, 2048, 1, 1, True)])
def test_sparse_attn_swa_matches_oracle(C, B, H, k, n_win, ring, want_lse):
    # walkthrough 1.(4): each query attends its selected entries and its layer's
    # own SWA KV window in one softmax; reading R10 fixes the ring layout
    rng = np.random.default_rng(B * 131 + n_win + ring)
    N = 3000
    kv = oracle.quantize_kv_fp4(rng.standard_normal((B * N, 512)).astype(np.float32))
    q = bf16_bits(rng.standard_normal((B, H, 512)))
    idx = np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(B)]).astype(np.int32)
    idx[0, -9:] = -1
    if B > 2:
        idx[2, :] = -1                                  # the window alone
    swa = _swa_rows(rng, (B, ring, 512))
    pos = rng.integers(0, 5000, B).astype(np.int32)
    pos[-1] = min(3, n_win - 1) if n_win > 1 else 0     # a window cut by the sequence start
    if B > 3:
        pos[3] = -1                                     # no window
    ref_o, ref_l = oracle.sparse_attn_swa(q, kv, N, N, 1, idx, swa, ring, n_win, pos, SCALE)
    out, lse = C.sparse_attn_fp4_swa(cuda(q, torch.int16), cuda(kv), N, N, 1, cuda(idx),
                                     cuda(swa), n_win, cuda(pos), SCALE, want_lse=want_lse)
    assert_attn_close(out.cpu().numpy(), ref_o)
    if want_lse:
        assert_lse_close(lse.cpu().numpy(), ref_l)


def test_layer_group_with_swa_matches_oracle(C):
    rng = np.random.default_rng(91)
    modes = (0, 1, 2)
    B, N, H, H_I, k, ring, n_win = 3, 5000, 64, 8, 512, 160, 128
    kv, ki, qs, qis, pos = _group(rng, B, N, H, H_I, k, modes, 0)
    swas = [_swa_rows(rng, (B, ring, 512)), None, _swa_rows(rng, (B, ring, 512))]
    outs, lses, idxs, _ = C.layer_group(modes, [cuda(q, torch.int16) for q in qs],
                                        [None if qi is None else cuda(qi) for qi in qis],
                                        cuda(kv), cuda(ki), N, N, 1, cuda(pos), 4, k, 0, SCALE,
                                        swa_kv=[None if x is None else cuda(x) for x in swas],
                                        n_win=n_win)
    r_outs, r_lses, r_idxs, _ = oracle.layer_group(
        modes, qs, qis, kv, ki, N, N, 1, pos, 4, k, 0, SCALE,
        swa_kv=[x if x is not None else np.zeros((B, ring, 512), np.uint8) for x in swas],
        swa_ring=ring, n_win=n_win)
    # the oracle attends a zero window where the GPU layer has none: compare
    # layer 1 with the plain sparse attention instead
    o1, l1 = oracle.sparse_attn(qs[1], kv, N, N, 1, r_idxs[1], SCALE)
    r_outs[1], r_lses[1] = o1, l1
    for l in range(len(modes)):
        assert (idxs[l].cpu().numpy() == r_idxs[l]).all(), l
        assert_attn_close(outs[l].cpu().numpy(), r_outs[l], l)
        assert_lse_close(lses[l].cpu().numpy(), r_lses[l])


# ---------------------------------------------------------------- layer group

def _group(rng, B, N, H, H_I, k, layers, pool, ratio=4):
    x = rng.standard_normal((B * N, 512)).astype(np.float32)
    kv = oracle.quantize_kv_fp4(x)
    ki = int_e4m3(rng, (B * N, 64))
    qs = [bf16_bits(rng.standard_normal((B, H, 512))) for _ in layers]
    qis = [None if m == 2 else int_e4m3(rng, (B, H_I, 64)) for m in layers]
    pos = rng.integers(4 * k, ratio * N + 3, B).astype(np.int32)
    return kv, ki, qs, qis, pos


@pytest.mark.parametrize("modes,pool", [((0,), 0), ((0, 1, 2), 0), ((0, 2, 1, 2, 2), 0),
                                        ((0, 1, 1, 1), 1024), ((0, 2, 1), 512)])
def test_layer_group_matches_oracle(C, modes, pool):
    rng = np.random.default_rng(len(modes) * 10 + pool)
    B, N, H, H_I, k = 3, 4000, 64, 8, 256
    kv, ki, qs, qis, pos = _group(rng, B, N, H, H_I, k, modes, pool)
    outs, lses, idxs, gpool = C.layer_group(modes, [cuda(q, torch.int16) for q in qs],
                                            [None if qi is None else cuda(qi) for qi in qis],
                                            cuda(kv), cuda(ki), N, N, 1, cuda(pos), 4, k, pool,
                                            SCALE)
    r_outs, r_lses, r_idxs, r_pool = oracle.layer_group(modes, qs, qis, kv, ki, N, N, 1, pos, 4,
                                                        k, pool, SCALE)
    for l in range(len(modes)):
        assert (idxs[l].cpu().numpy() == r_idxs[l]).all(), l
        assert_attn_close(outs[l].cpu().numpy(), r_outs[l], l)
        assert_lse_close(lses[l].cpu().numpy(), r_lses[l])
    if pool:
        assert (gpool.cpu().numpy() == r_pool).all()


def test_layer_group_with_one_split_per_query_matches_oracle(C):
    # B >= the SM count: every query's attention is one CTA (no merge kernel), so a Reuse
    # layer follows another attention directly and writes its index copy itself
    rng = np.random.default_rng(160)
    B, N, H, H_I, k = 160, 600, 16, 8, 64
    modes = (0, 2, 2, 1, 2)
    kv, ki, qs, qis, pos = _group(rng, B, N, H, H_I, k, modes, 0)
    outs, lses, idxs, _ = C.layer_group(modes, [cuda(q, torch.int16) for q in qs],
                                        [None if qi is None else cuda(qi) for qi in qis],
                                        cuda(kv), cuda(ki), N, N, 1, cuda(pos), 4, k, 0, SCALE)
    r_outs, r_lses, r_idxs, _ = oracle.layer_group(modes, qs, qis, kv, ki, N, N, 1, pos, 4, k,
                                                   0, SCALE)
    for l in range(len(modes)):
        assert (idxs[l].cpu().numpy() == r_idxs[l]).all(), l
        assert_attn_close(outs[l].cpu().numpy(), r_outs[l], l)
        assert_lse_close(lses[l].cpu().numpy(), r_lses[l])


def test_layer_group_rejects_bad_schedules(C):
    rng = np.random.default_rng(0)
    B, N, H, k = 2, 500, 64, 64
    kv, ki, qs, qis, pos = _group(rng, B, N, H, 4, k, (1, 2), 0)
    from sparse_attention_decode_csa2_gb300.csa2 import Csa2Error
    with pytest.raises(Csa2Error) as e:
        C.layer_group((1, 2), [cuda(q, torch.int16) for q in qs], [cuda(qis[0]), None], cuda(kv),
                      cuda(ki), N, N, 1, cuda(pos), 4, k)
    assert e.value.code == 1
    with pytest.raises(Csa2Error) as e:   # pool smaller than k
        C.layer_group((0, 2), [cuda(q, torch.int16) for q in qs], [cuda(qis[0]), None], cuda(kv),
                      cuda(ki), N, N, 1, cuda(pos), 4, k, pool_size=k - 1)
    assert e.value.code == 1


def test_invalid_arguments_launch_nothing(C):
    from sparse_attention_decode_csa2_gb300.csa2 import Csa2Error
    q = torch.zeros((2, 48, 512), dtype=torch.int16, device="cuda")
    kv = torch.zeros((10, 288), dtype=torch.uint8, device="cuda")
    idx = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(Csa2Error) as e:
        C.sparse_attn_fp4(q, kv, 10, 10, 1, idx, SCALE)
    assert e.value.code == 2          # H = 48 unsupported
    q = torch.zeros((2, 64, 512), dtype=torch.int16, device="cuda")
    with pytest.raises(Csa2Error) as e:
        C.sparse_attn_fp4(q, kv, 10, 10, 1, idx, -1.0)
    assert e.value.code == 1
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(Csa2Error) as e:
        C.sparse_attn_fp4(q, kv, 10, 10, 1, idx, SCALE, ws=ws)
    assert e.value.code == 3
