"""Pins of the oracle's MXFP4 indexer (DeepSeek-V4.1-Flash walkthrough 1.(5).4:
indexer query and key in the OCP MXFP4 format; 1.(4) "CSA2" for the scores).
CPU only."""
import math

import numpy as np

import oracle
from helpers import bf16_bits
from conftest import golden_lines, parse_float

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])


def _decode(rows, d):
    """Independent decoder: table lookup of nibbles times 2^(scale byte - 127)."""
    rows = np.asarray(rows, np.uint8)
    codes = rows[..., : d // 2]
    lo = (codes & 15).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    nib = np.stack([lo, hi], axis=-1).reshape(rows.shape[:-1] + (d,))
    scale = np.exp2(rows[..., d // 2:].astype(np.float64) - 127.0)
    return E2M1[nib] * np.repeat(scale, 32, axis=-1)


def test_e8m0_is_a_power_of_two_over_the_full_range():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(134) == 128.0
    assert oracle.e8m0_value(254) == 2.0 ** 127


def test_row_is_68_bytes_for_128_dims():
    assert oracle.mxfp4_row_bytes(128) == 68
    assert oracle.mxfp4_row_bytes(32) == 17


def test_quantise_golden_rows():
    n = 0
    for line in golden_lines("mxfp4_rows.txt"):
        d, vals, want = (t.strip() for t in line.split("|"))
        d = int(d)
        x = np.zeros(d, np.float32)
        for tok in vals.split():
            ch, v = tok.split(":")
            x[int(ch)] = np.float32(parse_float(v))
        want = bytes.fromhex(want.replace(" ", ""))
        got = oracle.quantize_mxfp4(x[None])[0].tobytes()
        assert got == want, (line, got.hex())
        n += 1
    assert n == 3


def test_each_element_is_the_nearest_grid_point_with_the_ocp_shared_exponent():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((40, 128)) * np.exp2(rng.integers(-20, 20, (40, 1)))).astype(
        np.float32)
    x[3, 32:64] = 0.0
    rows = oracle.quantize_mxfp4(x)
    dq = _decode(rows, 128)
    grid = E2M1[:8]
    for r in range(40):
        for b in range(4):
            blk = x[r, 32 * b: 32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            sbyte = int(rows[r, 64 + b])
            if amax == 0:
                assert sbyte == 0
                assert (dq[r, 32 * b: 32 * b + 32] == 0).all()
                continue
            assert sbyte - 127 == math.floor(math.log2(amax)) - 2
            X = 2.0 ** (int(sbyte) - 127)
            q = np.abs(blk) / X
            # the block maximum lands in [4, 8): the largest element never underflows
            assert 4 <= q.max() < 8
            got = np.abs(dq[r, 32 * b: 32 * b + 32]) / X
            for qi, gi in zip(q, got):
                dist = np.abs(grid - qi)
                assert dist[grid == gi][0] == dist.min()
            # sign follows the input (zero elements keep the sign bit of the input)
            nz = blk != 0
            assert (np.sign(dq[r, 32 * b: 32 * b + 32][nz & (got > 0)]) ==
                    np.sign(blk[nz & (got > 0)])).all()


def test_quantise_is_exponent_equivariant_and_sign_symmetric():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((8, 64)).astype(np.float32)
    base = oracle.quantize_mxfp4(x)
    for m in (-9, -1, 3, 17):
        sc = oracle.quantize_mxfp4((x * np.float32(2.0 ** m)).astype(np.float32))
        assert (sc[:, :32] == base[:, :32]).all()
        assert (sc[:, 32:].astype(int) == base[:, 32:].astype(int) + m).all()
    neg = oracle.quantize_mxfp4(-x)
    assert (neg[:, :32] == (base[:, :32] ^ 0x88)).all()
    assert (neg[:, 32:] == base[:, 32:]).all()


def test_quantise_of_representable_rows_is_identity():
    # rows whose every block has a largest magnitude code of 4 or 6 are fixed points
    rng = np.random.default_rng(13)
    rows = np.zeros((16, 68), np.uint8)
    nib = rng.integers(0, 16, (16, 128))
    nib[:, ::32] = rng.choice([6, 7, 14, 15], (16, 4))
    rows[:, :64] = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    rows[:, 64:] = rng.integers(100, 160, (16, 4))
    x = _decode(rows, 128).astype(np.float32)
    assert (oracle.quantize_mxfp4(x) == rows).all()


def test_scores_equal_decoded_matrix_products_and_respect_visibility():
    rng = np.random.default_rng(14)
    B, H_I, D_I, S, N = 4, 3, 64, 2, 37
    q = oracle.quantize_mxfp4(rng.standard_normal((B, H_I, D_I)).astype(np.float32))
    k = oracle.quantize_mxfp4(rng.standard_normal((S * N, D_I)).astype(np.float32))
    q_pos = np.array([5, 100, 17, 0], np.int32)
    ratio = 4
    s = oracle.index_scores_mxfp4(q, k, D_I, N, N, 2, q_pos, ratio)
    qd, kd = _decode(q, D_I), _decode(k, D_I).reshape(S, N, D_I)
    for b in range(B):
        want = (qd[b] @ kd[b // 2].T).sum(axis=0)
        nv = min(N, (int(q_pos[b]) + 1) // ratio)
        np.testing.assert_allclose(s[b, :nv], want[:nv], rtol=1e-12, atol=1e-9)
        assert np.isneginf(s[b, nv:]).all()


def test_integer_valued_rows_give_exact_integer_scores():
    # scale byte 127 and codes of integer magnitude: products and sums are integers
    rng = np.random.default_rng(15)
    ints = np.array([0, 1, 2, 3, 4, 6])
    qv = rng.choice(ints, (2, 2, 32)) * rng.choice([-1, 1], (2, 2, 32))
    kv = rng.choice(ints, (9, 32)) * rng.choice([-1, 1], (9, 32))
    qv[..., 0] = 6
    kv[..., 0] = 6
    q = oracle.quantize_mxfp4(qv.astype(np.float32))
    k = oracle.quantize_mxfp4(kv.astype(np.float32))
    assert (q[..., 16] == 127).all() and (k[..., 16] == 127).all()
    s = oracle.index_scores_mxfp4(q, k, 32, 9, 0, 2, None, 1)
    want = np.einsum("bhd,nd->bn", qv, kv)
    assert (s == want).all()


def _brute_pool_topk(scores, pool, k):
    out = []
    for b in range(scores.shape[0]):
        cand = sorted({int(j) for j in pool[b] if 0 <= j < scores.shape[1]},
                      key=lambda j: (-scores[b, j], j))[:k]
        out.append(sorted(cand) + [-1] * (k - len(cand)))
    return np.array(out, np.int32)


def test_pool_reindex_ranks_the_pooled_entries_by_the_mxfp4_score():
    rng = np.random.default_rng(16)
    B, H_I, D_I, N, P, k = 3, 2, 64, 60, 20, 7
    q = oracle.quantize_mxfp4(rng.standard_normal((B, H_I, D_I)).astype(np.float32))
    kk = oracle.quantize_mxfp4(rng.standard_normal((B * N, D_I)).astype(np.float32))
    pool = np.stack([rng.permutation(N)[:P] for _ in range(B)]).astype(np.int32)
    pool[1, 15:] = -1
    pool[2, :] = -1
    pool[2, :4] = [3, 9, 1, 50]
    got = oracle.hier_pool_index_mxfp4(q, kk, D_I, N, N, 1, pool, k)
    s = oracle.index_scores_mxfp4(q, kk, D_I, N, N, 1, None, 1)
    assert (got == _brute_pool_topk(s, pool, k)).all()


def test_layer_group_with_mxfp4_indexer_selects_by_the_mxfp4_scores():
    rng = np.random.default_rng(17)
    B, H, D, H_I, D_I, N, k, P = 2, 2, 512, 2, 64, 48, 6, 16
    modes = [0, 1, 2]  # Full, Reindex, Reuse
    qs = [bf16_bits(rng.standard_normal((B, H, D)))
          for _ in modes]
    qis = [oracle.quantize_mxfp4(rng.standard_normal((B, H_I, D_I)).astype(np.float32))
           for _ in modes]
    qis[2] = None
    kv = oracle.quantize_kv_fp4(rng.standard_normal((B * N, D)).astype(np.float32))
    ki = oracle.quantize_mxfp4(rng.standard_normal((B * N, D_I)).astype(np.float32))
    q_pos = np.array([N - 1, 30], np.int32)
    outs, lses, idxs, pool = oracle.layer_group(
        modes, qs, qis, kv, ki, N, N, 1, q_pos, 1, k, P, 1 / math.sqrt(D), indexer_fmt=1,
        D_I=D_I)
    s0 = oracle.index_scores_mxfp4(qis[0], ki, D_I, N, N, 1, q_pos, 1)
    assert (idxs[0] == oracle.topk(s0, k, q_pos, 1)).all()
    assert (pool == oracle.topk(s0, P, q_pos, 1)).all()
    s1 = oracle.index_scores_mxfp4(qis[1], ki, D_I, N, N, 1, q_pos, 1)
    assert (idxs[1] == _brute_pool_topk(s1, pool, k)).all()
    assert (idxs[2] == idxs[1]).all()
