"""Pins of the oracle's indexer scores, top-k and hierarchical pool
(DeepSeek-V4.1-Flash walkthrough 1.(4) "CSA2", 1.(4).1, 1.(4).2).  CPU only."""
import itertools
from fractions import Fraction

import numpy as np
import torch

import oracle


def _e4m3(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _e4m3_to_float(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).float().numpy()


# ---------------------------------------------------------------- visibility

def test_visible_count_matches_closed_form():
    # entry j is visible iff ratio*j + ratio - 1 <= pos  <=>  j < floor((pos+1)/ratio)
    N = 50
    for ratio in (1, 2, 4, 7):
        for pos in range(-3, ratio * N + 10):
            want = min(N, max(0, (pos + 1) // ratio))
            assert oracle.n_visible(np.array([pos], np.int32), 0, ratio, N) == want
    assert oracle.n_visible(None, 0, 4, N) == N


# ---------------------------------------------------------------- scores

def test_scores_of_integer_inputs_equal_integer_arithmetic():
    rng = np.random.default_rng(0)
    B, H_I, D_I, N = 3, 4, 64, 40
    qi = rng.integers(-8, 9, (B, H_I, D_I))
    ki = rng.integers(-8, 9, (B, N, D_I))
    s = oracle.index_scores(_e4m3(qi), _e4m3(ki).reshape(B * N, D_I), N, N, 1, None, 4)
    want = np.einsum("bhd,bnd->bn", qi.astype(np.int64), ki.astype(np.int64))
    assert (s == want).all()


def test_single_head_score_is_a_matrix_vector_product():
    rng = np.random.default_rng(1)
    N, D_I = 33, 64
    q = _e4m3(rng.standard_normal((1, 1, D_I)))
    k = _e4m3(rng.standard_normal((N, D_I)))
    s = oracle.index_scores(q, k, N, 0, 1, None, 1)[0]
    want = _e4m3_to_float(k).astype(np.float64) @ _e4m3_to_float(q)[0, 0].astype(np.float64)
    np.testing.assert_allclose(s, want, rtol=1e-14, atol=1e-12)


def test_float_scores_are_exact_rationals():
    # products of two E4M3 values have <= 8 significant bits; the fp64 sum of
    # 2 heads x 64 of them is exact, so it must equal exact rational arithmetic
    rng = np.random.default_rng(2)
    q = _e4m3(rng.standard_normal((1, 2, 64)) * 3)
    k = _e4m3(rng.standard_normal((5, 64)) * 3)
    s = oracle.index_scores(q, k, 5, 0, 1, None, 1)[0]
    qf, kf = _e4m3_to_float(q)[0], _e4m3_to_float(k)
    for j in range(5):
        exact = sum(Fraction(float(qf[h, d])) * Fraction(float(kf[j, d]))
                    for h in range(2) for d in range(64))
        assert Fraction(s[j]) == exact


def test_invisible_entries_score_minus_inf_and_sequences_are_separate():
    rng = np.random.default_rng(3)
    N, D_I = 16, 64
    qi = _e4m3(rng.integers(-8, 9, (4, 2, D_I)))
    ki = _e4m3(rng.integers(-8, 9, (2 * N, D_I)))
    pos = np.array([3, 17, 63, -1], np.int32)
    s = oracle.index_scores(qi, ki, N, N, 2, pos, 4)  # queries 0,1 -> seq 0; 2,3 -> seq 1
    for q in range(4):
        nv = min(N, max(0, (pos[q] + 1) // 4))
        assert np.isneginf(s[q, nv:]).all() and np.isfinite(s[q, :nv]).all()
    # query 2 reads sequence 1's keys
    s2 = oracle.index_scores(qi[2:3], ki[N:], N, N, 1, pos[2:3], 4)
    assert (s2 == s[2:3]).all()


# ---------------------------------------------------------------- top-k

def _brute_topk(row, k, n_vis):
    """Entry j is selected iff fewer than k visible entries outrank it, where i
    outranks j when s_i > s_j, or s_i == s_j and i < j."""
    sel = []
    for j in range(n_vis):
        better = sum(1 for i in range(n_vis)
                     if row[i] > row[j] or (row[i] == row[j] and i < j))
        if better < k:
            sel.append(j)
    return sel + [-1] * (k - len(sel))


def test_topk_matches_brute_force_rank_definition_on_tiny_rows():
    rng = np.random.default_rng(4)
    for trial in range(300):
        N = int(rng.integers(1, 14))
        k = int(rng.integers(1, N + 3))
        vals = rng.integers(-3, 4, N).astype(np.float64)          # heavy ties
        if trial % 3 == 0:
            vals = rng.standard_normal(N)
        pos = int(rng.integers(-1, 4 * N + 2))
        got = oracle.topk(vals[None], k, np.array([pos], np.int32), 4)[0]
        n_vis = min(N, max(0, (pos + 1) // 4))
        assert list(got) == _brute_topk(vals, k, n_vis), (vals, k, pos)


def test_topk_all_equal_takes_lowest_indices():
    s = np.zeros((2, 100))
    got = oracle.topk(s, 10)
    assert (got == np.arange(10)).all()


def test_topk_k_equal_visible_returns_every_visible_entry():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((3, 64))
    got = oracle.topk(s, 64)
    assert (got == np.arange(64)).all()
    pos = np.array([4 * 20 - 1, 4 * 64 + 100, 2], np.int32)
    got = oracle.topk(s, 64, pos, 4)
    assert (got[0, :20] == np.arange(20)).all() and (got[0, 20:] == -1).all()
    assert (got[1] == np.arange(64)).all()
    assert (got[2] == -1).all()


def test_topk_output_is_ascending_and_selects_the_largest():
    rng = np.random.default_rng(6)
    s = rng.integers(-100, 100, (4, 500)).astype(np.float64)
    got = oracle.topk(s, 37)
    for r in range(4):
        g = got[r]
        assert (np.diff(g) > 0).all()
        kth = np.sort(s[r])[::-1][36]
        assert (s[r, g] >= kth).all()
        assert (s[r, np.setdiff1d(np.arange(500), g)] <= kth).all()


def test_topk_permutation_exhaustive_small():
    # all orderings of a small multiset of scores
    base = [2.0, 2.0, 1.0, 5.0, 1.0]
    for perm in set(itertools.permutations(base)):
        row = np.array(perm)
        for k in range(1, 6):
            assert list(oracle.topk(row[None], k)[0]) == _brute_topk(row, k, 5)


# ---------------------------------------------------------------- hierarchical pool

def test_pool_of_all_visible_entries_reproduces_flat_indexer():
    rng = np.random.default_rng(7)
    B, H_I, D_I, N, k = 3, 8, 64, 300, 20
    qi = _e4m3(rng.integers(-8, 9, (B, H_I, D_I)))
    ki = _e4m3(rng.integers(-8, 9, (B * N, D_I)))
    flat = oracle.topk(oracle.index_scores(qi, ki, N, N, 1, None, 4), k)
    pool = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    hier = oracle.hier_pool_index(qi, ki, N, N, 1, pool, k)
    assert (hier == flat).all()


def test_pool_restricts_selection_and_skips_padding():
    rng = np.random.default_rng(8)
    B, H_I, D_I, N, k = 2, 2, 64, 200, 8
    qi = _e4m3(rng.integers(-8, 9, (B, H_I, D_I)))
    ki = _e4m3(rng.integers(-8, 9, (B * N, D_I)))
    scores = oracle.index_scores(qi, ki, N, N, 1, None, 4)
    pool = np.full((B, 40), -1, np.int32)
    pool[:, :30] = np.stack([np.sort(rng.choice(N, 30, replace=False)) for _ in range(B)])
    got = oracle.hier_pool_index(qi, ki, N, N, 1, pool, k)
    for b in range(B):
        cand = pool[b, :30]
        order = sorted(cand, key=lambda j: (-scores[b, j], j))[:k]
        assert list(got[b]) == sorted(order)
    # fewer pool entries than k: padded with -1
    got = oracle.hier_pool_index(qi, ki, N, N, 1, pool[:, :5], k)
    assert (got[:, 5:] == -1).all() and (got[:, :5] >= 0).all()


# ---------------------------------------------------------------- blockwise pool

def _golden_block_pool():
    from conftest import golden_lines
    scores, cases = None, []
    for line in golden_lines("block_pool.txt"):
        tok = line.split()
        if tok[0] == "scores":
            scores = np.array([float(t) for t in tok[1:]])
        elif tok[0] == "case":
            colon = tok.index(":")
            cases.append((int(tok[1]), int(tok[2]), [int(t) for t in tok[colon + 1:]]))
    return scores, cases


def test_block_pool_matches_hand_derived_cases():
    scores, cases = _golden_block_pool()
    assert scores is not None and len(cases) == 4
    for pos, nblk, want in cases:
        got = oracle.block_pool(scores[None, :], 4, nblk, np.array([pos], np.int32), 1)
        assert got[0].tolist() == want, (pos, nblk)


def _check_block_pool(scores, q_pos, ratio, block, nblk, pool):
    """Properties that fix the blockwise pool: ascending visible entries of
    whole kept blocks, -1 only at the tail, and no unkept block beats a kept
    one (ties: the lower block index is kept)."""
    B, N = scores.shape
    for q in range(B):
        nv = oracle.n_visible(q_pos, q, ratio, N)
        nb = -(-nv // block)
        row = pool[q]
        valid = row[row >= 0]
        assert np.all(row[len(valid):] == -1), "padding only at the tail"
        assert np.all(np.diff(valid) > 0) and (len(valid) == 0 or valid[-1] < nv)
        kept = sorted(set((valid // block).tolist()))
        assert len(kept) == min(nblk, nb)
        want = [j for b in kept for j in range(b * block, min((b + 1) * block, nv))]
        assert valid.tolist() == want, "the pool is every visible entry of the kept blocks"
        bmax = [scores[q, b * block:min((b + 1) * block, nv)].max() for b in range(nb)]
        for s in kept:
            for u in set(range(nb)) - set(kept):
                assert bmax[s] > bmax[u] or (bmax[s] == bmax[u] and s < u), (q, s, u)
        if nv > 0:
            assert int(np.argmax(scores[q, :nv])) // block in kept


def test_block_pool_properties_on_random_rows_with_ties():
    rng = np.random.default_rng(11)
    for trial in range(60):
        B, N = 4, int(rng.integers(1, 90))
        block = int(rng.choice([1, 2, 3, 8]))
        nblk = int(rng.integers(1, 12))
        ratio = int(rng.choice([1, 4]))
        scores = rng.integers(-3, 4, (B, N)).astype(np.float64)  # heavy ties
        q_pos = rng.integers(-2, ratio * N + 3, B).astype(np.int32)
        pool = oracle.block_pool(scores, block, nblk, q_pos, ratio)
        assert pool.shape == (B, nblk * block)
        _check_block_pool(scores, q_pos, ratio, block, nblk, pool)


def test_block_pool_of_one_entry_blocks_is_the_flat_top_p():
    rng = np.random.default_rng(12)
    scores = rng.standard_normal((5, 300))
    q_pos = np.array([1199, 800, 3, -1, 500], np.int32)
    for P in (1, 17, 300, 400):
        assert np.array_equal(oracle.block_pool(scores, 1, P, q_pos, 4),
                              oracle.topk(scores, P, q_pos, 4))


def test_block_pool_with_every_block_kept_is_every_visible_entry():
    rng = np.random.default_rng(13)
    scores = rng.standard_normal((3, 64))
    pool = oracle.block_pool(scores, 8, 8, np.array([63, 40, 0], np.int32), 1)
    for q, nv in enumerate((64, 41, 1)):
        assert pool[q].tolist() == list(range(nv)) + [-1] * (64 - nv)
