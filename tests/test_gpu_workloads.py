"""Parity of the whole CSA2 path at the ten workloads' full sizes, in the
launch configuration the benchmark times (csa2_layer_group over the
device-resident cache).  The oracle recomputes sampled queries one by one:
their FP4 rows (from the same seeded latent), indexer scores, top-k / pool
selections and attention outputs.  Needs a GPU."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_attn_close, assert_float_selection_ok, assert_lse_close

pytestmark = pytest.mark.gpu

NAMES = ["tiny_full_1q_ctx4k", "decode_b32_ctx64k", "group_full_reindex_reuse_b64_ctx128k",
         "hier_pool8192_b16_ctx1m", "prefill_4096q_ctx128k", "hier_block2048x8_b16_ctx1m",
         "decode_swa128_b32_ctx64k", "decoder20_prod_b32_ctx64k", "decoder20_mxfp4_b32_ctx64k",
         "encoder18_chunk512_ctx64k"]


def _sample(B, n):
    if B <= n:
        return list(range(B))
    rng = np.random.default_rng(B)
    mid = sorted(rng.choice(np.arange(1, B - 1), n - 2, replace=False).tolist())
    return [0] + mid + [B - 1]


@pytest.mark.parametrize("name", NAMES)
def test_workload_parity(name):
    from sparse_attention_decode_csa2_gb300 import build
    build.build()
    from sparse_attention_decode_csa2_gb300 import csa2, workload
    from sparse_attention_decode_csa2_gb300.synthetic import REINDEX, REUSE, WORKLOADS
    w = WORKLOADS[name]
    inp = workload.prepare(w)
    lg = inp.layer_group()
    outs, lses, idxs, pool = lg()
    code, bits = csa2.read_status(lg.ws)
    assert code == 0, bits
    pos = w.q_pos()
    n_samples = {1: 1, 2: 4, 3: 3, 4: 3, 5: 6, 6: 3, 7: 4, 8: 2, 9: 2, 10: 3}[w.workload_id]
    if w.indexer_fmt:
        def scores_of(qi, ki, qpos):
            return oracle.index_scores_mxfp4(qi, ki, w.D_I, w.N, 0, 1, qpos, w.ratio)

        def pool_index(qi, ki, opool):
            return oracle.hier_pool_index_mxfp4(qi, ki, w.D_I, w.N, 0, 1, opool, w.k)
    else:
        def scores_of(qi, ki, qpos):
            return oracle.index_scores(qi, ki, w.N, 0, 1, qpos, w.ratio)

        def pool_index(qi, ki, opool):
            return oracle.hier_pool_index(qi, ki, w.N, 0, 1, opool, w.k)
    for q in _sample(w.B, n_samples):
        s = q // w.q_per_seq
        ki = w.ki_rows(s)
        qpos = pos[q:q + 1]
        latest = None
        opool = None
        attended = []
        for l, mode in enumerate(w.modes):
            got_idx = idxs[l][q].cpu().numpy() if idxs[l] is not None else None
            if mode == REUSE:
                ref_idx = latest
            else:
                qi = w.qi_rows(l, [q])
                if mode == REINDEX and w.pool:
                    ref_idx = pool_index(qi, ki, opool)[0]
                    assert (got_idx == ref_idx).all(), (name, q, l)
                else:
                    sc = scores_of(qi, ki, qpos)
                    ref_idx = oracle.topk(sc, w.k, qpos, w.ratio)[0]
                    if w.pool and l == 0:
                        if w.pool_block > 1:
                            opool = oracle.block_pool(sc, w.pool_block, w.pool // w.pool_block,
                                                      qpos, w.ratio)
                        else:
                            opool = oracle.topk(sc, w.pool, qpos, w.ratio)
                        assert (pool[q].cpu().numpy() == opool[0]).all(), (name, q)
                    if w.float_indexer:
                        assert_float_selection_ok(got_idx, ref_idx, sc[0], (name, q, l))
                    else:
                        assert (got_idx == ref_idx).all(), (name, q, l)
            if got_idx is not None and mode == REUSE:
                assert (got_idx == latest).all(), (name, q, l)   # copy of the reused indices
            latest = got_idx if got_idx is not None else ref_idx
            attended.append(latest)
        # FP4 rows of every attended entry: oracle-quantised from the same latent,
        # byte-identical to the GPU cache
        rows = np.unique(np.concatenate([a[a >= 0] for a in attended]))
        ref_rows = oracle.quantize_kv_fp4(w.kv_latent_rows(s, rows))
        got_rows = inp.kv_fp4[s * w.N + torch.from_numpy(rows).cuda()].cpu().numpy()
        assert (got_rows == ref_rows).all(), (name, q)
        kv_sparse = np.zeros((w.N, w.row_bytes), np.uint8)
        kv_sparse[rows] = ref_rows
        for l in range(len(w.modes)):
            ql = w.q_bf16(l, [q])
            if w.n_win:
                ref_o, ref_l = oracle.sparse_attn_swa(ql, kv_sparse, w.N, 0, 1, attended[l][None],
                                                      w.swa_kv(l, s)[None], w.swa_ring, w.n_win,
                                                      qpos, inp.scale)
            else:
                ref_o, ref_l = oracle.sparse_attn(ql, kv_sparse, w.N, 0, 1, attended[l][None],
                                                  inp.scale)
            assert_attn_close(outs[l][q].cpu().numpy(), ref_o[0], (name, q, l))
            assert_lse_close(lses[l][q].cpu().numpy(), ref_l[0], (name, q, l))
