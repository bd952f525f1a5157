"""Shared helpers of the GPU parity tests."""
import math

import numpy as np
import torch

ATTN_MAX_ABS = 2e-3   # attention tolerance against the fp64 oracle
ATTN_REL_L2 = 1e-3
FLOAT_SCORE_REL = 1e-5  # float indexer inputs: selections may differ only this close to s_k


def e4m3_bytes(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, np.float32)).clamp(-448, 448).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def int_e4m3(rng, shape) -> np.ndarray:
    return e4m3_bytes(rng.integers(-8, 9, shape))


def bf16_bits(x) -> np.ndarray:
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def cuda(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def attn_errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.abs(got - ref).max()) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))
    return max_abs, rel


def assert_attn_close(got, ref, what=""):
    max_abs, rel = attn_errors(got, ref)
    assert max_abs <= ATTN_MAX_ABS and rel <= ATTN_REL_L2, (what, max_abs, rel)
    return max_abs, rel


def assert_lse_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    assert (np.isneginf(got) == np.isneginf(ref)).all(), what
    d = np.abs(np.where(both_inf, 0, got - ref))
    assert d.max(initial=0) <= 1e-4 * max(1.0, float(np.abs(np.where(both_inf, 0, ref)).max(initial=0))), (what, d.max())


def assert_float_selection_ok(got_idx, ref_idx, ref_scores, what=""):
    """Float indexer inputs: the GPU set may differ from the oracle's only by
    entries whose oracle score lies within FLOAT_SCORE_REL * |s_k| of the oracle
    k-th score s_k; both sets have the same size."""
    g = set(int(j) for j in got_idx if j >= 0)
    r = set(int(j) for j in ref_idx if j >= 0)
    assert len(g) == len(r), what
    diff = g ^ r
    if not diff:
        return 0
    s_k = min(ref_scores[j] for j in r)
    tol = FLOAT_SCORE_REL * abs(s_k)
    bad = [j for j in diff if abs(ref_scores[j] - s_k) > tol]
    assert not bad, (what, bad[:5], s_k)
    # the result is still ascending
    gl = [int(j) for j in got_idx if j >= 0]
    assert gl == sorted(gl)
    return len(diff)
