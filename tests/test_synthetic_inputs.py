"""The seeded input generator (``synthetic``) against its own recipe: the
SplitMix64 stream against published reference outputs, the normal and integer
draws against their definitions and their distributions, the bf16/E4M3 packing
against PyTorch's casts, and the workload shapes against the stated
configurations.  CPU only."""
import math

import numpy as np
import pytest
import torch

from conftest import golden_lines
from sparse_attention_decode_csa2_gb300 import synthetic as syn

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def test_stream_outputs_match_published_splitmix64_vectors():
    # draw(key, i) is output i of a SplitMix64 generator whose state starts at key
    n = 0
    for line in golden_lines("splitmix64.txt"):
        seed, outs = (t.strip() for t in line.split("|"))
        for i, want in enumerate(outs.split()):
            assert syn.draw(int(seed), i) == int(want), (seed, i)
            n += 1
    assert n == 9


def _u1_u2(key, i):
    u1 = ((syn.draw(key, 2 * i) >> 11) + 1) * 2.0 ** -53
    u2 = (syn.draw(key, 2 * i + 1) >> 11) * 2.0 ** -53
    return u1, u2


def test_normal_draws_follow_the_box_muller_definition():
    key = syn.stream_key(2, 7, syn.TENSOR_KV)
    got = syn.normal_f64(key, 100, 64)
    for t in range(64):
        u1, u2 = _u1_u2(key, 100 + t)
        assert 0.0 < u1 <= 1.0 and 0.0 <= u2 < 1.0
        want = math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
        assert got[t] == pytest.approx(want, rel=1e-14, abs=1e-300)


def test_normal_draws_are_standard_normal():
    scipy_stats = pytest.importorskip("scipy.stats")
    x = syn.normal_f64(syn.stream_key(3, 11, syn.TENSOR_Q), 0, 200_000)
    n = x.size
    assert abs(x.mean()) < 5 / math.sqrt(n)
    assert abs(x.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    p1 = np.mean(np.abs(x) < 1.0)
    assert abs(p1 - 0.682689) < 5 * math.sqrt(0.68 * 0.32 / n)
    assert scipy_stats.kstest(x, "norm").pvalue > 1e-4


def test_fp32_and_bf16_draws_are_the_rounded_fp64_draws():
    key = syn.stream_key(4, 5, syn.TENSOR_Q, 3)
    f64 = syn.normal_f64(key, 0, 4096)
    f32 = syn.normal_f32(key, 0, 4096)
    assert (f32 == f64.astype(np.float32)).all()
    bf = syn.normal_bf16(key, 0, 4096)
    want = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (bf == want).all()


def test_any_sub_range_and_any_thread_split_give_the_same_elements():
    key = syn.stream_key(5, 1, syn.TENSOR_KV)
    whole = syn.normal_f32(key, 0, 140_000)          # split over threads
    part = syn.normal_f32(key, 70_001, 69_999)
    assert (whole[70_001:] == part).all()
    ints = syn.uniform_int8(key, 0, 140_000, -8, 8)
    assert (ints[123_456:123_556] == syn.uniform_int8(key, 123_456, 100, -8, 8)).all()


def test_uniform_integers_follow_the_rejection_definition_and_are_uniform():
    scipy_stats = pytest.importorskip("scipy.stats")
    key = syn.stream_key(1, 0, syn.TENSOR_KI)
    got = syn.uniform_int8(key, 0, 2000, -8, 8)
    m = 17
    lim = m * ((1 << 32) // m)
    for i in range(2000):
        r = 0
        while True:
            x = syn.draw(key, i + (r << 40)) >> 32
            if x < lim:
                break
            r += 1
        assert got[i] == -8 + x % m
    big = syn.uniform_int8(key, 0, 340_000, -8, 8)
    assert big.min() == -8 and big.max() == 8
    counts = np.bincount(big.astype(np.int64) + 8, minlength=17)
    assert scipy_stats.chisquare(counts).pvalue > 1e-4
    nib = syn.uniform_int8(key, 0, 160_000, 0, 15)
    assert scipy_stats.chisquare(np.bincount(nib.astype(np.int64), minlength=16)).pvalue > 1e-4


def test_stream_keys_of_distinct_tensors_are_distinct():
    keys = {syn.stream_key(w, s, t, l) for w in range(1, 11) for s in range(40)
            for t in range(1, 6) for l in range(4)}
    assert len(keys) == 10 * 40 * 5 * 4


def test_integer_indexer_values_are_exact_in_e4m3():
    w = syn.WORKLOADS["tiny_full_1q_ctx4k"]
    ki = w.ki_fp8(0)
    assert ki.shape == (w.N, w.D_I) and ki.dtype == np.uint8
    vals = torch.from_numpy(ki.copy()).view(torch.float8_e4m3fn).float().numpy()
    key = syn.stream_key(w.workload_id, w.seed_of_seq(0), syn.TENSOR_KI)
    ints = syn.uniform_int8(key, 0, w.N * w.D_I, -8, 8).reshape(w.N, w.D_I)
    assert (vals == ints).all()


def test_mxfp4_rows_are_drawn_in_the_format():
    w = syn.WORKLOADS["decoder20_mxfp4_b32_ctx64k"]
    key = syn.stream_key(w.workload_id, w.seed_of_seq(0), syn.TENSOR_KI)
    rows = w._mx_rows(key, 5, 64)
    assert rows.shape == (64, 68)
    assert set(np.unique(rows[:, 64:])) <= {126, 127}
    # code nibbles follow the element counter: element e of row r is draw r * 128 + e
    nib = syn.uniform_int8(key, 5 * 128, 64 * 128, 0, 15).astype(np.uint8).reshape(64, 128)
    assert (rows[:, :64] & 15 == nib[:, 0::2]).all() and (rows[:, :64] >> 4 == nib[:, 1::2]).all()
    q = w.qi_rows(0, [0, 1])
    assert q.shape == (2, w.H_I, 68)


# the stated configurations: (name, queries, entries per sequence, ratio, heads, indexer
# heads x dim, top-k, schedule, pool, query positions)
CONFIGS = [
    ("tiny_full_1q_ctx4k", 1, 1024, 4, 16, (4, 64), 128, ("FULL",), 0, [4095]),
    ("decode_b32_ctx64k", 32, 16384, 4, 64, (8, 64), 2048, ("FULL",), 0, [65535] * 32),
    ("group_full_reindex_reuse_b64_ctx128k", 64, 32768, 4, 64, (8, 64), 2048,
     ("FULL", "REINDEX", "REUSE"), 0, [131071] * 64),
    ("hier_pool8192_b16_ctx1m", 16, 262144, 4, 64, (8, 64), 2048,
     ("FULL", "REINDEX", "REINDEX", "REINDEX"), 8192, [1048575] * 16),
    ("prefill_4096q_ctx128k", 4096, 32768, 4, 64, (8, 64), 2048, ("FULL",), 0,
     list(range(126976, 131072))),
]


@pytest.mark.parametrize("name,B,N,ratio,H,idx,k,modes,pool,pos", CONFIGS)
def test_workloads_have_the_stated_shapes(name, B, N, ratio, H, idx, k, modes, pool, pos):
    w = syn.WORKLOADS[name]
    assert (w.B, w.N, w.ratio, w.H, (w.H_I, w.D_I), w.k, w.pool) == (B, N, ratio, H, idx, k, pool)
    assert tuple(syn.MODE_NAMES[m] for m in w.modes) == modes
    assert w.q_pos().tolist() == pos
    assert w.D == 512 and w.row_bytes == 288
    # one seed per sequence, distinct across sequences
    assert len(set(w.seeds)) == w.n_seq
    # every query of the decode configurations sees its whole context
    assert all((p + 1) // ratio <= N for p in pos)


def test_decode_seeds_and_the_tiny_seed_are_the_stated_ones():
    assert list(syn.WORKLOADS["decode_b32_ctx64k"].seeds) == list(range(1, 33))
    assert list(syn.WORKLOADS["tiny_full_1q_ctx4k"].seeds) == [0]
    assert syn.WORKLOADS["prefill_4096q_ctx128k"].float_indexer
