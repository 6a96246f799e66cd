"""Mutation check of the oracle's pins: each case plants one plausible mistake
in a copy of oracle/ep_oracle.c, builds it, and runs tests/test_oracle.py
against it (EP_ORACLE_LIB); at least one pin must fail.  An unmodified copy
built the same way must pass.  CPU only."""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ep_oracle.c")

# (name, text in ep_oracle.c, replacement)
MUTANTS = [
    ("topk tie to higher id",
     "    if (a->v < b->v) return 1;\n    return (a->e < b->e) ? -1 : (a->e > b->e ? 1 : 0);",
     "    if (a->v < b->v) return 1;\n    return (a->e > b->e) ? -1 : (a->e < b->e ? 1 : 0);"),
    ("weight sum drops the first pick", "sum += ex[k];", "sum += k ? ex[k] : 0.0;"),
    ("weight exponent sign", "ex[k] = exp((double)row[k].v - top);",
     "ex[k] = exp(top - (double)row[k].v);"),
    ("expert map ignored", "int32_t id = expert_map ? expert_map[e] : e;",
     "int32_t id = e;"),
    ("out-of-range map entries kept", "topk_idx[t * K + k] = (id >= 0 && id < E) ? id : -1;",
     "topk_idx[t * K + k] = id;"),
    ("greedy ties to the higher set", "if (best < 0 || load[s] < load[best]) best = s;",
     "if (best < 0 || load[s] <= load[best]) best = s;"),
    ("layout: tokens in reverse within an expert",
     "        for (int64_t t = 0; t < N; ++t) {\n            for (int32_t k = 0; k < K; ++k) {\n"
     "                if (topk_idx[t * K + k] == e) {",
     "        for (int64_t t = N - 1; t >= 0; --t) {\n            for (int32_t k = 0; k < K; ++k) {\n"
     "                if (topk_idx[t * K + k] == e) {"),
    ("rank offsets inclusive",
     "            rank_expert_offsets[(int64_t)r * E + e] = run;\n"
     "            run += counts[(int64_t)r * E + e];",
     "            run += counts[(int64_t)r * E + e];\n"
     "            rank_expert_offsets[(int64_t)r * E + e] = run;"),
    ("masked_m ignores the capacity", "masked_m[e] = total < cap ? total : cap;",
     "masked_m[e] = total;"),
    ("masked capacity off by one", "if (slot >= cap) return -1;", "if (slot > cap) return -1;"),
    ("fp8 truncates instead of rounding", "double m = nearbyint(n);", "double m = floor(n);"),
    ("fp8 without saturation", "if (code > 0x7E) code = 0x7E;", ""),
    ("fp8 scale constant", "amax / 448.0f", "amax / 447.0f"),
    ("fp8 zero block scale", "(amax == 0.0f) ? 1.0f :", "(amax == 0.0f) ? 0.5f :"),
    ("bf16 rounds half up", "u += 0x7FFFu + lsb;", "u += 0x8000u;"),
    ("combine in reverse pick order",
     "            for (int32_t k = 0; k < K; ++k) {\n                if (rows[k] < 0) continue;",
     "            for (int32_t k = K - 1; k >= 0; --k) {\n                if (rows[k] < 0) continue;"),
    ("combine uses the first weight for every pick",
     "acc = fmaf(topk_w[t * K + k],", "acc = fmaf(topk_w[t * K],"),
    ("combine skips the last pick", "            for (int32_t k = 0; k < K; ++k) {\n"
     "                if (rows[k] < 0) continue;",
     "            for (int32_t k = 0; k < K - 1; ++k) {\n                if (rows[k] < 0) continue;"),
]


def _build_and_test(src_text, tmp):
    c = os.path.join(tmp, "m.c")
    so = os.path.join(tmp, "m.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", so, c, "-lm"], check=True)
    env = dict(os.environ, EP_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests",
                        "test_oracle.py"), "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_every_planted_mistake_fails_a_pin():
    base = open(SRC).read()
    jobs = [("control", base)]
    for name, old, new in MUTANTS:
        assert base.count(old) >= 1, f"mutation target not found: {name}"
        jobs.append((name, base.replace(old, new)))
    with tempfile.TemporaryDirectory() as td:
        dirs = []
        for i in range(len(jobs)):
            d = os.path.join(td, str(i))
            os.makedirs(d)
            dirs.append(d)
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            codes = list(ex.map(lambda j: _build_and_test(j[1][1], dirs[j[0]]),
                                enumerate(jobs)))
    results = dict(zip([n for n, _ in jobs], codes))
    assert results.pop("control") == 0, "the unmodified oracle must pass its pins"
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, f"mistakes no pin caught: {survivors}"
