"""Pins of the oracle's sparse MQA attention and layer modes (DeepSeek-V4.1-Flash
walkthrough 1.(4) "CSA2", 1.(4).1 "Cross-Layer KV and Index Reuse",
1.(4).2 "Hierarchical Sparse Indexer", 1.(5).4 "FP4 Main KV Cache").  CPU only."""
import math

import numpy as np
import torch

import oracle

D = 512
SCALE = 1.0 / math.sqrt(512.0)


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _kv(rng, n):
    return oracle.quantize_kv_fp4(rng.standard_normal((n, D)).astype(np.float32))


def test_all_entries_selected_equals_dense_softmax_attention():
    rng = np.random.default_rng(0)
    N, H = 96, 8
    kv = _kv(rng, N)
    q = _bf16(rng.standard_normal((1, H, D)))
    idx = np.arange(N, dtype=np.int32)[None]
    out, lse = oracle.sparse_attn(q, kv, N, N, 1, idx, SCALE)
    v = torch.from_numpy(oracle.dequantize_kv_fp4(kv, D))               # [N][D]
    qt = torch.from_numpy(_bf16_to_f64(q)[0])                             # [H][D]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt[None], v[None].expand(H, N, D)[None], v[None].expand(H, N, D)[None], scale=SCALE)[0]
    np.testing.assert_allclose(out[0], ref.numpy()[0], rtol=1e-12, atol=1e-13)
    ref_lse = torch.logsumexp(SCALE * qt @ v.T, dim=-1).numpy()
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-13)


def test_zero_query_gives_mean_of_selected_values():
    rng = np.random.default_rng(1)
    N = 50
    kv = _kv(rng, N)
    q = np.zeros((1, 4, D), np.uint16)
    idx = np.array([[3, 7, 11, 40, -1, -1]], np.int32)
    out, lse = oracle.sparse_attn(q, kv, N, N, 1, idx, SCALE)
    v = oracle.dequantize_kv_fp4(kv, D)
    want = v[[3, 7, 11, 40]].mean(0)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], want, rtol=1e-13, atol=1e-15)
        assert abs(lse[0, h] - math.log(4)) < 1e-14


def test_single_entry_returns_that_entry():
    rng = np.random.default_rng(2)
    kv = _kv(rng, 10)
    q = _bf16(rng.standard_normal((1, 3, D)))
    out, lse = oracle.sparse_attn(q, kv, 10, 10, 1, np.array([[-1, 6, -1]], np.int32), SCALE)
    v = oracle.dequantize_kv_fp4(kv, D)[6]
    for h in range(3):
        assert (out[0, h] == v).all()
        np.testing.assert_allclose(lse[0, h], SCALE * _bf16_to_f64(q)[0, h] @ v, rtol=1e-13)


def test_two_entries_weights_are_a_sigmoid():
    rng = np.random.default_rng(3)
    kv = _kv(rng, 2)
    q = _bf16(rng.standard_normal((1, 1, D)))
    out, _ = oracle.sparse_attn(q, kv, 2, 2, 1, np.array([[0, 1]], np.int32), SCALE)
    v = oracle.dequantize_kv_fp4(kv, D)
    l = SCALE * (v @ _bf16_to_f64(q)[0, 0])
    p0 = 1.0 / (1.0 + math.exp(l[1] - l[0]))
    np.testing.assert_allclose(out[0, 0], p0 * v[0] + (1 - p0) * v[1], rtol=1e-12, atol=1e-14)


def test_permuting_indices_does_not_change_the_result():
    rng = np.random.default_rng(4)
    N = 64
    kv = _kv(rng, N)
    q = _bf16(rng.standard_normal((1, 4, D)))
    idx = rng.choice(N, 20, replace=False).astype(np.int32)[None]
    o1, l1 = oracle.sparse_attn(q, kv, N, N, 1, idx, SCALE)
    o2, l2 = oracle.sparse_attn(q, kv, N, N, 1, idx[:, ::-1].copy(), SCALE)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_no_valid_entry_gives_zero_and_minus_inf():
    rng = np.random.default_rng(5)
    kv = _kv(rng, 4)
    q = _bf16(rng.standard_normal((2, 2, D)))
    out, lse = oracle.sparse_attn(q, kv, 4, 4, 1, np.full((2, 5), -1, np.int32), SCALE)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_sequences_are_addressed_by_query():
    rng = np.random.default_rng(6)
    N = 30
    kv = _kv(rng, 2 * N)
    q = _bf16(rng.standard_normal((4, 2, D)))
    idx = rng.integers(0, N, (4, 7)).astype(np.int32)
    out, _ = oracle.sparse_attn(q, kv, N, N, 2, idx, SCALE)
    o_seq1, _ = oracle.sparse_attn(q[2:], kv[N:], N, N, 2, idx[2:], SCALE)
    assert (out[2:] == o_seq1).all()


# ---------------------------------------------------------------- modes

def _group_inputs(rng, B=2, N=200, H=4, H_I=2, D_I=64, layers=3):
    kv = _kv(rng, B * N)
    ki = torch.tensor(rng.integers(-8, 9, (B * N, D_I)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    qs = [_bf16(rng.standard_normal((B, H, D))) for _ in range(layers)]
    qis = [torch.tensor(rng.integers(-8, 9, (B, H_I, D_I)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy() for _ in range(layers)]
    return kv, ki, qs, qis


def test_reuse_equals_recomputation_with_previous_indices():
    rng = np.random.default_rng(7)
    B, N, k = 2, 200, 16
    kv, ki, qs, qis = _group_inputs(rng, B, N)
    pos = np.array([4 * N - 1, 4 * 150 - 1], np.int32)
    outs, lses, idxs, _ = oracle.layer_group([0, 1, 2], qs, [qis[0], qis[1], None], kv, ki, N, N,
                                             1, pos, 4, k, 0, SCALE)
    # Reuse: same indices as the Reindex layer, attention recomputed with its own q
    assert (idxs[2] == idxs[1]).all()
    o, l = oracle.sparse_attn(qs[2], kv, N, N, 1, idxs[1], SCALE)
    assert (o == outs[2]).all() and (l == lses[2]).all()
    # Full: flat indexer with its own q
    want = oracle.topk(oracle.index_scores(qis[0], ki, N, N, 1, pos, 4), k, pos, 4)
    assert (idxs[0] == want).all()
    # Reindex: same shared K, its own q
    want = oracle.topk(oracle.index_scores(qis[1], ki, N, N, 1, pos, 4), k, pos, 4)
    assert (idxs[1] == want).all()


def test_reindex_with_the_full_layers_query_selects_the_same_entries():
    rng = np.random.default_rng(8)
    kv, ki, qs, qis = _group_inputs(rng, layers=2)
    _, _, idxs, _ = oracle.layer_group([0, 1], qs, [qis[0], qis[0]], kv, ki, 200, 200, 1, None, 4,
                                       16, 0, SCALE)
    assert (idxs[0] == idxs[1]).all()


def test_pool_of_every_entry_equals_flat_schedule():
    rng = np.random.default_rng(9)
    B, N, k = 2, 200, 16
    kv, ki, qs, qis = _group_inputs(rng, B, N)
    flat = oracle.layer_group([0, 1, 2], qs, [qis[0], qis[1], None], kv, ki, N, N, 1, None, 4, k,
                              0, SCALE)
    hier = oracle.layer_group([0, 1, 2], qs, [qis[0], qis[1], None], kv, ki, N, N, 1, None, 4, k,
                              N, SCALE)
    for a, b in zip(flat[2], hier[2]):
        assert (a == b).all()
    assert (hier[3] == np.arange(N)).all()


def test_full_layer_selection_lies_inside_its_pool():
    rng = np.random.default_rng(10)
    B, N, k = 2, 200, 16
    kv, ki, qs, qis = _group_inputs(rng, B, N)
    _, _, idxs, pool = oracle.layer_group([0, 1, 1], qs, [qis[0], qis[1], qis[2]], kv, ki, N, N,
                                          1, None, 4, k, 48, SCALE)
    for b in range(B):
        assert set(idxs[0][b]) <= set(pool[b])
        assert set(idxs[1][b]) <= set(pool[b]) and set(idxs[2][b]) <= set(pool[b])
        # top-k of the full scores equals top-k within the pool
    hier = oracle.hier_pool_index(qis[0], ki, N, N, 1, pool, k)
    assert (hier == idxs[0]).all()


def test_schedule_must_start_with_full():
    rng = np.random.default_rng(11)
    kv, ki, qs, qis = _group_inputs(rng)
    import pytest
    with pytest.raises(ValueError):
        oracle.layer_group([1, 2], qs[:2], [qis[0], None], kv, ki, 200, 200, 1, None, 4, 16, 0,
                           SCALE)


def test_blockwise_pool_schedule_selects_inside_the_pool():
    # Full builds the blockwise pool (walkthrough 1.(4).2); Reindex layers pick
    # their top-k among pool entries only; Reuse repeats the latest indices.
    rng = np.random.default_rng(21)
    B, N, k = 2, 96, 8
    kv, ki, qs, qis = _group_inputs(rng, B, N)
    pos = np.array([4 * N - 1, 4 * 70 + 1], np.int32)
    outs, lses, idxs, pool = oracle.layer_group([0, 1, 2], qs, [qis[0], qis[1], None], kv, ki, N,
                                                N, 1, pos, 4, k, 24, SCALE, pool_block=8)
    scores = oracle.index_scores(qis[0], ki, N, N, 1, pos, 4)
    assert np.array_equal(pool, oracle.block_pool(scores, 8, 3, pos, 4))
    for q in range(B):
        members = set(pool[q][pool[q] >= 0].tolist())
        assert set(idxs[1][q][idxs[1][q] >= 0].tolist()) <= members
    assert np.array_equal(idxs[2], idxs[1])


# ---------------------------------------------------------------- SWA branch

def _e4m3_rows(rng, n, scale=1.0):
    x = (rng.standard_normal((n, D)) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_decode(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


def _sdpa(q_bits, v):
    """fp64 softmax attention of every head of one query over rows v [n][D]."""
    qt = torch.from_numpy(_bf16_to_f64(q_bits))                            # [H][D]
    vt = torch.from_numpy(v)
    H, n = qt.shape[0], vt.shape[0]
    o = torch.nn.functional.scaled_dot_product_attention(
        qt[:, None], vt[None].expand(H, n, D), vt[None].expand(H, n, D), scale=SCALE)[:, 0]
    return o.numpy(), torch.logsumexp(SCALE * qt @ vt.T, dim=-1).numpy()


def test_swa_window_alone_equals_dense_attention_over_the_window():
    # R10: the query at position pos attends tokens max(0, pos - n_win + 1) .. pos,
    # token t at ring row t mod ring.  Rows outside the window hold 448s that
    # would dominate any softmax they entered.
    rng = np.random.default_rng(30)
    H, ring, n_win = 4, 40, 16
    q = _bf16(rng.standard_normal((3, H, D)))
    kv = _kv(rng, 8)
    idx = np.full((3, 4), -1, np.int32)
    for pos in (0, 9, 15, 16, 57, 1000):
        swa = np.full((3, ring, D), 0x7E, np.uint8)       # E4M3 448 everywhere
        toks = list(range(max(0, pos - n_win + 1), pos + 1))
        rows = _e4m3_rows(rng, len(toks))
        for s in range(3):
            for i, t in enumerate(toks):
                swa[s, t % ring] = rows[i]
        out, lse = oracle.sparse_attn_swa(q, kv, 8, 0, 3, idx, swa, ring, n_win,
                                          np.full(3, pos, np.int32), SCALE)
        for b in range(3):
            ref_o, ref_l = _sdpa(q[b], _e4m3_decode(rows))
            np.testing.assert_allclose(out[b], ref_o, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lse[b], ref_l, rtol=1e-12)


def test_joint_softmax_is_the_lse_merge_of_its_two_parts():
    rng = np.random.default_rng(31)
    B, H, N, k, ring, n_win = 3, 8, 200, 24, 160, 128
    kv = _kv(rng, B * N)
    q = _bf16(rng.standard_normal((B, H, D)))
    idx = np.stack([np.sort(rng.choice(N, k, replace=False)) for _ in range(B)]).astype(np.int32)
    idx[1, -5:] = -1
    swa = np.stack([_e4m3_rows(rng, ring, 0.7) for _ in range(B)])
    pos = np.array([4000, 70, 127], np.int32)
    o, l = oracle.sparse_attn_swa(q, kv, N, N, 1, idx, swa, ring, n_win, pos, SCALE)
    o1, l1 = oracle.sparse_attn(q, kv, N, N, 1, idx, SCALE)
    none = np.full((B, 1), -1, np.int32)
    o2, l2 = oracle.sparse_attn_swa(q, kv, N, N, 1, none, swa, ring, n_win, pos, SCALE)
    L = np.logaddexp(l1, l2)
    merged = np.exp(l1 - L)[..., None] * o1 + np.exp(l2 - L)[..., None] * o2
    np.testing.assert_allclose(o, merged, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(l, L, rtol=1e-12)


def test_without_a_window_the_swa_attention_is_the_sparse_attention():
    rng = np.random.default_rng(32)
    B, H, N, k = 2, 4, 64, 10
    kv = _kv(rng, B * N)
    q = _bf16(rng.standard_normal((B, H, D)))
    idx = rng.integers(-1, N, (B, k)).astype(np.int32)
    o1, l1 = oracle.sparse_attn(q, kv, N, N, 1, idx, SCALE)
    swa = np.stack([_e4m3_rows(rng, 8) for _ in range(B)])
    for args in ((None, 0, 0), (swa, 8, 0)):
        o2, l2 = oracle.sparse_attn_swa(q, kv, N, N, 1, idx, *args, np.array([50, 60], np.int32),
                                        SCALE)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_layer_group_with_swa_matches_per_layer_attention():
    rng = np.random.default_rng(33)
    B, N, k, ring, n_win = 2, 150, 12, 128, 128
    kv, ki, qs, qis = _group_inputs(rng, B, N)
    swas = [np.stack([_e4m3_rows(rng, ring) for _ in range(B)]) for _ in range(3)]
    pos = np.array([4 * N - 1, 300], np.int32)
    outs, lses, idxs, _ = oracle.layer_group([0, 1, 2], qs, [qis[0], qis[1], None], kv, ki, N, N,
                                             1, pos, 4, k, 0, SCALE, swa_kv=swas, swa_ring=ring,
                                             n_win=n_win)
    for l in range(3):
        o, lse = oracle.sparse_attn_swa(qs[l], kv, N, N, 1, idxs[l], swas[l], ring, n_win, pos,
                                        SCALE)
        assert np.array_equal(outs[l], o) and np.array_equal(lses[l], lse)
