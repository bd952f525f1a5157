"""GPU parity of the MXFP4 indexer (DeepSeek-V4.1-Flash walkthrough 1.(5).4:
indexer query and key in OCP MXFP4) against the oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import golden_lines, parse_float
from helpers import (assert_attn_close, assert_float_selection_ok, assert_lse_close, bf16_bits,
                     cuda)

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(512.0)
D_I = 128


@pytest.fixture(scope="module")
def C():
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2
    return csa2


def _mx_float(rng, shape, spread=6):
    # normal values with a per-row power-of-two spread of magnitudes
    x = rng.standard_normal(shape) * np.exp2(rng.integers(-spread, spread + 1, shape[:-1] + (1,)))
    return x.astype(np.float32)


def _mx_int(rng, shape):
    """Rows whose every 32-block has scale byte 127: integer values in
    {0, +-1, +-2, +-3, +-4, +-6} with a 4 or 6 in each block, so scores are
    integers that fp32 holds exactly."""
    v = rng.choice([0, 1, 2, 3, 4, 6], shape) * rng.choice([-1, 1], shape)
    v[..., ::32] = rng.choice([-6, -4, 4, 6], v[..., ::32].shape)
    return oracle.quantize_mxfp4(v.astype(np.float32))


# ---------------------------------------------------------------- quantiser

@pytest.mark.parametrize("n,d", [(1000, 128), (37, 32), (5, 64), (9, 96), (300, 256), (3, 4096)])
def test_quantize_mxfp4_bit_exact(C, n, d):
    rng = np.random.default_rng(n * 7 + d)
    x = _mx_float(rng, (n, d), spread=40)
    x[0, :32] = 0.0
    if n > 2:
        x[1, :] = np.float32(2.0 ** -140) * rng.standard_normal(d).astype(np.float32)  # subnormal
        x[2, ::3] = -0.0
    got = C.quantize_mxfp4(cuda(x)).cpu().numpy()
    assert (got == oracle.quantize_mxfp4(x)).all()


def test_quantize_mxfp4_golden_rows_and_ties(C):
    n = 0
    for line in golden_lines("mxfp4_rows.txt"):
        d, vals, want = (t.strip() for t in line.split("|"))
        x = np.zeros(int(d), np.float32)
        for tok in vals.split():
            ch, v = tok.split(":")
            x[int(ch)] = np.float32(parse_float(v))
        got = C.quantize_mxfp4(cuda(x[None])).cpu().numpy()[0].tobytes()
        assert got == bytes.fromhex(want.replace(" ", "")), line
        n += 1
    assert n == 3
    # every E2M1 midpoint and its fp32 neighbours, at several block scales
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 7.9], np.float32)
    pts = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 10)])
    rows = []
    for e in (-130, -20, 0, 17, 100):
        blk = np.zeros(32, np.float32)
        blk[:pts.size] = (pts.astype(np.float64) * 2.0 ** e).astype(np.float32)
        blk[31] = np.float32(8.0 * 2.0 ** e)  # absmax above every point: shared exponent e + 1
        rows.append(blk)
    x = np.stack(rows)
    assert (C.quantize_mxfp4(cuda(x)).cpu().numpy() == oracle.quantize_mxfp4(x)).all()


def test_quantize_mxfp4_empty_is_a_no_op(C):
    out = torch.full((0, 68), 7, dtype=torch.uint8, device="cuda")
    C.quantize_mxfp4(torch.empty((0, 128), device="cuda"), out)


# ---------------------------------------------------------------- scores

@pytest.mark.parametrize("B,N,H_I,q_per_seq,ratio", [
    (32, 1501, 32, 1, 4), (32, 1501, 64, 16, 1), (3, 128, 1, 1, 1), (4, 130, 8, 2, 2),
    (18, 4000, 32, 9, 4)])
def test_index_scores_mxfp4_exact_for_integer_rows(C, B, N, H_I, q_per_seq, ratio):
    rng = np.random.default_rng(B * N + H_I)
    stride = (N + 3) // 4 * 4
    S = B // q_per_seq
    q = _mx_int(rng, (B, H_I, D_I))
    k = _mx_int(rng, (S * stride, D_I))
    pos = rng.integers(-2, ratio * N + 5, B).astype(np.int32)
    pos[0] = ratio * N + 100
    got = C.index_scores_mxfp4(cuda(q), cuda(k), N, stride, q_per_seq, cuda(pos),
                               ratio).cpu().numpy()
    ref = oracle.index_scores_mxfp4(q, k, D_I, N, stride, q_per_seq, pos, ratio)
    assert (got == ref).all()


@pytest.mark.parametrize("B,N,H_I,q_per_seq", [(32, 3001, 32, 1), (16, 1000, 64, 16)])
def test_index_scores_mxfp4_float_rows_within_fp32_rounding(C, B, N, H_I, q_per_seq):
    rng = np.random.default_rng(N + H_I)
    stride = (N + 3) // 4 * 4
    S = B // q_per_seq
    q = oracle.quantize_mxfp4(_mx_float(rng, (B, H_I, D_I)))
    k = oracle.quantize_mxfp4(_mx_float(rng, (S * stride, D_I)))
    got = C.index_scores_mxfp4(cuda(q), cuda(k), N, stride, q_per_seq, None, 1).cpu().numpy()
    ref = oracle.index_scores_mxfp4(q, k, D_I, N, stride, q_per_seq, None, 1)
    # bound from the arithmetic: the head sum is compensated (<= 2 ulp of qsum)
    # and each 32-term block sum of exact products is an fp32 pairwise-split
    # sum: |err| <= 40 * 2^-24 * sum_d |qsum_d k_d|
    qa = np.abs(_dequant(q)).sum(axis=1)           # [B][D_I] >= |qsum|
    ka = np.abs(_dequant(k))                        # [S*stride][D_I]
    for b in range(B):
        s = b // q_per_seq
        mag = ka[s * stride:s * stride + N] @ qa[b]
        assert (np.abs(got[b] - ref[b]) <= 40 * 2.0 ** -24 * mag + 1e-30).all(), b
    # and the selections follow the float-indexer rule
    k_sel = 256
    gi = C.topk(cuda(got.astype(np.float32)), k_sel).cpu().numpy()
    ri = oracle.topk(ref, k_sel)
    for b in range(B):
        assert_float_selection_ok(gi[b], ri[b], ref[b], b)


def _dequant(rows):
    rows = np.asarray(rows, np.uint8)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0, -0.5, -1, -1.5, -2, -3, -4, -6])
    codes = rows[..., :64]
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(rows.shape[:-1] + (128,))
    sc = np.exp2(rows[..., 64:].astype(np.float64) - 127.0)
    return e2m1[nib] * np.repeat(sc, 32, axis=-1)


def test_index_scores_mxfp4_rejects_unsupported_shapes(C):
    q = torch.zeros((4, 8, 68), dtype=torch.uint8, device="cuda")
    k = torch.zeros((4 * 102, 68), dtype=torch.uint8, device="cuda")
    with pytest.raises(C.Csa2Error):  # stride not a multiple of 4 with several sequences
        C.index_scores_mxfp4(q, k, 100, 102, 1, None, 1)
    with pytest.raises(C.Csa2Error):  # D_I = 64
        C.index_scores_mxfp4(q[..., :34].contiguous(), k[:, :34].contiguous(), 100, 100, 1,
                             None, 1)
    C.index_scores_mxfp4(q[:1], k, 100, 0, 1, None, 1)  # one sequence: any stride


# ---------------------------------------------------------------- pool and group

@pytest.mark.parametrize("N,P,k", [(5000, 1024, 128), (32768, 8192, 512), (3000, 700, 800)])
def test_hier_pool_index_mxfp4_bit_exact_for_integer_rows(C, N, P, k):
    rng = np.random.default_rng(P + k)
    B, H_I = 4, 32
    q0, q1 = _mx_int(rng, (B, H_I, D_I)), _mx_int(rng, (B, H_I, D_I))
    ki = _mx_int(rng, (B * N, D_I))
    pos = np.array([N - 1, P // 2, N - 1, N // 3], np.int32)
    pool = oracle.topk(oracle.index_scores_mxfp4(q0, ki, D_I, N, N, 1, pos, 1), P, pos, 1)
    got = C.hier_pool_index_mxfp4(cuda(q1), cuda(ki), N, N, 1, cuda(pool), k).cpu().numpy()
    assert (got == oracle.hier_pool_index_mxfp4(q1, ki, D_I, N, N, 1, pool, k)).all()


def test_hier_pool_index_mxfp4_float_rows_follow_the_selection_rule(C):
    rng = np.random.default_rng(77)
    B, H_I, N, P, k = 8, 32, 20000, 4096, 512
    q0 = oracle.quantize_mxfp4(_mx_float(rng, (B, H_I, D_I)))
    q1 = oracle.quantize_mxfp4(_mx_float(rng, (B, H_I, D_I)))
    ki = oracle.quantize_mxfp4(_mx_float(rng, (B * N, D_I)))
    pool = oracle.topk(oracle.index_scores_mxfp4(q0, ki, D_I, N, N, 1, None, 1), P)
    got = C.hier_pool_index_mxfp4(cuda(q1), cuda(ki), N, N, 1, cuda(pool), k).cpu().numpy()
    s1 = oracle.index_scores_mxfp4(q1, ki, D_I, N, N, 1, None, 1)
    ref = oracle.hier_pool_index_mxfp4(q1, ki, D_I, N, N, 1, pool, k)
    for b in range(B):
        assert_float_selection_ok(got[b], ref[b], s1[b], b)


@pytest.mark.parametrize("modes,pool,pool_block,n_win", [((0, 2, 1, 2), 0, 0, 0),
                                                         ((0, 1, 2, 1), 1024, 0, 0),
                                                         ((0, 2, 1, 1), 1024, 8, 0),
                                                         ((0, 2, 1, 2), 512, 8, 128)])
def test_layer_group_with_mxfp4_indexer_matches_oracle(C, modes, pool, pool_block, n_win):
    rng = np.random.default_rng(len(modes) + pool + pool_block + n_win)
    B, N, H, H_I, k = 3, 4000, 64, 32, 256
    kv = oracle.quantize_kv_fp4(rng.standard_normal((B * N, 512)).astype(np.float32))
    ki = _mx_int(rng, (B * N, D_I))
    qs = [bf16_bits(rng.standard_normal((B, H, 512))) for _ in modes]
    qis = [None if m == 2 else _mx_int(rng, (B, H_I, D_I)) for m in modes]
    pos = rng.integers(4 * k, N + 3, B).astype(np.int32)
    ring = 256
    swa = None
    if n_win:  # each layer's SWA ring: E4M3 rows of N(0,1) latents
        swa = [torch.from_numpy(rng.standard_normal((B, ring, 512)).astype(np.float32))
               .to(torch.float8_e4m3fn).view(torch.uint8).numpy() for _ in modes]
    outs, lses, idxs, gpool = C.layer_group(
        modes, [cuda(q, torch.int16) for q in qs], [None if qi is None else cuda(qi) for qi in qis],
        cuda(kv), cuda(ki), N, N, 1, cuda(pos), 1, k, pool, SCALE, pool_block=pool_block,
        swa_kv=None if swa is None else [cuda(x) for x in swa], n_win=n_win,
        indexer_fmt=C.INDEXER_MXFP4)
    r_outs, r_lses, r_idxs, r_pool = oracle.layer_group(
        modes, qs, qis, kv, ki, N, N, 1, pos, 1, k, pool, SCALE, pool_block=pool_block,
        swa_kv=swa, swa_ring=ring if n_win else 0, n_win=n_win, indexer_fmt=1, D_I=D_I)
    for l in range(len(modes)):
        assert (idxs[l].cpu().numpy() == r_idxs[l]).all(), l
        assert_attn_close(outs[l].cpu().numpy(), r_outs[l], l)
        assert_lse_close(lses[l].cpu().numpy(), r_lses[l])
    if pool:
        assert (gpool.cpu().numpy() == r_pool).all()
