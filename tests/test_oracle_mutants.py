"""The oracle's pins catch plausible mistakes.  Each case plants one mistake in
a copy of ``oracle/csa2_oracle.c`` (a wrong constant, index, tie rule, sign,
bound or schedule step), builds that copy on the CPU and runs the oracle pin
tests against it in a subprocess; at least one pin must fail.  An unchanged
copy built the same way must pass them all.  CPU only."""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "csa2_oracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_select.py",
        "tests/test_oracle_attention.py", "tests/test_oracle_mxfp4.py"]

# (name, text in csa2_oracle.c, replacement): each text occurs exactly once
MUTANTS = [
    ("fp4 scale divisor 4 instead of 6",
     "orc_e4m3_encode(amax / 6.0)", "orc_e4m3_encode(amax / 4.0)"),
    ("e2m1 ties to the larger code",
     """    double d = fabs(orc_e2m1_value(c) - q);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {""",
     """    double d = fabs(orc_e2m1_value(c) - q);
    if (d <= best_d) {"""),
    ("e4m3 ties to the larger code",
     """    double d = fabs(orc_e4m3_value(c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {""",
     """    double d = fabs(orc_e4m3_value(c) - a);
    if (d <= best_d) {"""),
    ("e4m3 exponent bias 8",
     "else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 7);",
     "else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 8);"),
    ("fp4 nibbles swapped",
     """        int mag = (s == 0.0) ? 0 : orc_e2m1_encode_magnitude(fabs(xv) / s);
        int code = (signbit(xv) ? 8 : 0) | mag;
        codes[ch / 2] |= (uint8_t)((ch & 1) ? (code << 4) : code);""",
     """        int mag = (s == 0.0) ? 0 : orc_e2m1_encode_magnitude(fabs(xv) / s);
        int code = (signbit(xv) ? 8 : 0) | mag;
        codes[ch / 2] |= (uint8_t)((ch & 1) ? code : (code << 4));"""),
    ("fp4 sign of negative zero dropped",
     """        int mag = (s == 0.0) ? 0 : orc_e2m1_encode_magnitude(fabs(xv) / s);
        int code = (signbit(xv) ? 8 : 0) | mag;""",
     """        int mag = (s == 0.0) ? 0 : orc_e2m1_encode_magnitude(fabs(xv) / s);
        int code = (xv < 0.0 ? 8 : 0) | mag;"""),
    ("fp4 dequantise with the scale of the wrong block",
     "out[ch] = orc_e2m1_value(code) * orc_e4m3_value(scales[ch / 16]);",
     "out[ch] = orc_e2m1_value(code) * orc_e4m3_value(scales[ch / 32]);"),
    ("mxfp4 shared exponent off by one",
     "shared = (e - 1) - 2;", "shared = (e - 1) - 1;"),
    ("visibility from the entry's first token",
     "(int64_t)ratio * n + ratio - 1 <= pos", "(int64_t)ratio * n <= pos"),
    ("indexer score drops the last head",
     """      idx_row_values(kseq + j * rb, D_I, fmt, kj);
      double s = 0.0;
      for (int h = 0; h < H_I; ++h) {""",
     """      idx_row_values(kseq + j * rb, D_I, fmt, kj);
      double s = 0.0;
      for (int h = 0; h < H_I - 1; ++h) {"""),
    ("top-k ties to the higher index",
     "return (x->j < y->j) ? -1 : (x->j > y->j);",
     "return (x->j > y->j) ? -1 : (x->j < y->j);"),
    ("top-k output in rank order",
     "  qsort(out, (size_t)take, sizeof(int32_t), cmp_i32);\n", ""),
    ("block score = its first entry's score",
     "if (scores[(int64_t)q * N + j] > m) m = scores[(int64_t)q * N + j];",
     "if (j == b * block) m = scores[(int64_t)q * N + j];"),
    ("attention logits without the softmax scale",
     "logit[t] = scale * dot;", "logit[t] = dot;"),
    ("lse without the max shift",
     "if (lse) lse[h] = m + log(l);", "if (lse) lse[h] = log(l);"),
    ("swa window one token longer",
     "int64_t t0 = pos - n_win + 1 > 0 ? pos - n_win + 1 : 0;",
     "int64_t t0 = pos - n_win > 0 ? pos - n_win : 0;"),
    ("pool re-index returns pool slots instead of entry ids",
     "      c[n].j = j;", "      c[n].j = p;"),
    ("mxfp4 scale byte biased by 126",
     "scales[b] = (uint8_t)(shared + 127);", "scales[b] = (uint8_t)(shared + 126);"),
    ("e2m1 normal values halved",
     "(1.0 + 0.5 * m) * ldexp(1.0, e - 1)", "(1.0 + 0.5 * m) * ldexp(1.0, e - 2)"),
    ("softmax weights not normalised",
     "double p = logit[t] / l;", "double p = logit[t];"),
    ("top-k ranks invisible entries too",
     """    for (int64_t j = 0; j < nv; ++j) {
      c[j].s = scores[(int64_t)q * N + j];
      c[j].j = j;
    }
    select_topk(c, nv, k, idx + (int64_t)q * k);""",
     """    for (int64_t j = 0; j < N; ++j) {
      c[j].s = scores[(int64_t)q * N + j];
      c[j].j = j;
    }
    select_topk(c, N, k, idx + (int64_t)q * k);"""),
    ("blockwise pool drops the partial last block",
     "int64_t nb = (nv + block - 1) / block;", "int64_t nb = nv / block;"),
    ("reindex in the pool scores with the first layer's query",
     "orc_hier_pool_index_fmt(qi_fp8[l], ki_fp8", "orc_hier_pool_index_fmt(qi_fp8[0], ki_fp8"),
    ("swa ring row off by one",
     "(s * swa_ring + t % swa_ring) * D", "(s * swa_ring + (t + 1) % swa_ring) * D"),
    # (swapping the nibbles in the MXFP4 decode is no mistake the oracle can show: q and K
    # are permuted alike inside one scale block, so every score is unchanged; the byte
    # order itself is pinned by the quantiser's golden rows)
    ("e8m0 bias 128",
     "double orc_e8m0_value(int byte) { return ldexp(1.0, byte - 127); }",
     "double orc_e8m0_value(int byte) { return ldexp(1.0, byte - 128); }"),
    ("reuse takes the full layer's indices past a reindex",
     """      latest = idx;
    } else if (modes[l] == ORC_REUSE) {""",
     """    } else if (modes[l] == ORC_REUSE) {"""),
]


def _build_and_run(text: str, workdir: str):
    """Build one copy of the oracle from `text` and run the pins against it."""
    os.makedirs(workdir, exist_ok=True)
    src = os.path.join(workdir, "csa2_oracle.c")
    with open(src, "w") as f:
        f.write(text)
    lib = os.path.join(workdir, "libcsa2_oracle_variant.so")
    subprocess.run(oracle.compile_command(src, lib), check=True)
    env = dict(os.environ, CSA2_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-3000:]


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    """Every copy (the unchanged one under the key None) built and run, several at a time."""
    text = open(SRC).read()
    jobs = {None: text}
    for name, old, new in MUTANTS:
        assert text.count(old) == 1, name
        jobs[name] = text.replace(old, new)
    base = tmp_path_factory.mktemp("oracle_mutants")
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        futs = {key: ex.submit(_build_and_run, body, str(base / f"m{i}"))
                for i, (key, body) in enumerate(jobs.items())}
        return {key: f.result() for key, f in futs.items()}


def test_an_unchanged_copy_passes_every_pin(runs):
    rc, out = runs[None]
    assert rc == 0, out


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(runs, name):
    rc, out = runs[name]
    # exit code 1: the run completed and some pin failed (not a crash or a usage error)
    assert rc == 1, f"{name} survived the pins:\n{out}"
