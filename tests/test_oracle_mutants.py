"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle/ep_oracle.c (on the CPU),
compiles it, and runs the oracle pin tests against it (EP_ORACLE_LIB); at least
one pin must fail.  The oracle itself is untouched."""
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ep_oracle.c")
PIN_TESTS = ["tests/test_oracle_worked.py", "tests/test_oracle_order.py", "tests/test_oracle_invariants.py",
             "tests/test_oracle_fp8.py", "tests/test_oracle_bruteforce.py", "tests/test_oracle_ll_hier.py"]

# (name, original text, mutated text)
MUTANTS = [
    ("channel prefix exclusive",
     "for (int t = lo; t < hi; ++t) acc += itir[((int64_t)s * T + t) * R + d];\n                cpm[((int64_t)s * R + d) * C + c] = acc;",
     "cpm[((int64_t)s * R + d) * C + c] = acc;\n                for (int t = lo; t < hi; ++t) acc += itir[((int64_t)s * T + t) * R + d];"),
    ("send position off by one",
     "send_pos[i] = recv_offsets[d * R + s] + running++;",
     "send_pos[i] = recv_offsets[d * R + s] + ++running;"),
    ("receive offsets inclusive",
     "recv_offsets[d * R + s] = acc;\n            acc += recv_count[d * R + s];",
     "acc += recv_count[d * R + s];\n            recv_offsets[d * R + s] = acc;"),
    ("experts dealt round-robin to ranks",
     "in_rank[e / L] = 1;", "in_rank[e % R] = 1;"),
    ("permute orders local expert before rank",
     "if (p->d != q->d) return p->d < q->d ? -1 : 1;\n    if (p->l != q->l) return p->l < q->l ? -1 : 1;",
     "if (p->l != q->l) return p->l < q->l ? -1 : 1;\n    if (p->d != q->d) return p->d < q->d ? -1 : 1;"),
    ("received top-k index global instead of local",
     "recv_topk_idx[row * K + k] = (int32_t)(e - (int64_t)d * L);",
     "recv_topk_idx[row * K + k] = (int32_t)e;"),
    ("combine ranks in descending order",
     "float final_sum = 0.0f;\n                for (int d = 0; d < R; ++d) {",
     "float final_sum = 0.0f;\n                for (int d = R - 1; d >= 0; --d) {"),
    ("combine multiply and add rounded separately",
     "partial = fmaf(w[tok * K + k], yv, partial);\n                        has = 1;\n                    }\n                    if (has) {\n                        volatile float acc",
     "{ volatile float pr = w[tok * K + k] * yv; partial = pr + partial; }\n                        has = 1;\n                    }\n                    if (has) {\n                        volatile float acc"),
    ("ties rounded away from zero",
     "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    ("scale by reciprocal multiply",
     "volatile float scale = amax / 448.0f;", "volatile float scale = amax * (1.0f / 448.0f);"),
    ("bf16 truncation",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;", "(void)lower;"),
    ("zero counts left at the sentinel",
     "for (int e = 0; e < E; ++e) counts[(int64_t)e * R + s] = running[e];",
     "for (int e = 0; e < E; ++e) if (running[e]) counts[(int64_t)e * R + s] = running[e];"),
    ("slots not restarted per source",
     "memset(running, 0, sizeof(int32_t) * (size_t)E);", ";"),
    ("hierarchical combine without the node level",
     "volatile float a = node_sum + partial;\n                        node_sum = a;",
     "volatile float a = final_sum + partial;\n                        final_sum = a;"),
    ("home rank by node of the source",
     "if (s % G != h % G) continue;", "if (s / G != h % G) continue;"),
    ("expert blocks not rounded to the alignment",
     "acc += round_up(n, align);", "acc += n;"),
    ("aligned permute places a block at its unpadded start",
     "row += padded;\n        i = j;", "row += cnt;\n        i = j;"),
    ("low-latency combine multiply and add rounded separately",
     "acc = fmaf(w[tok * K + k], orc_bf16_to_f32(y_ll[row * H + j]), acc);",
     "{ volatile float pr = w[tok * K + k] * orc_bf16_to_f32(y_ll[row * H + j]); acc = pr + acc; }"),
    ("low-latency combine in descending k order",
     "for (int k = 0; k < K; ++k) {\n                    int64_t e = topk_idx[tok * K + k];\n"
     "                    if (e < 0 || e >= E) continue;\n                    int d = (int)(e / L), l = (int)(e % L);",
     "for (int k = K - 1; k >= 0; --k) {\n                    int64_t e = topk_idx[tok * K + k];\n"
     "                    if (e < 0 || e >= E) continue;\n                    int d = (int)(e / L), l = (int)(e % L);"),
    ("low-latency combine ignores the source's begin in the packed block",
     "int64_t row = ((int64_t)d * L + l) * per_expert + begin + slot[tok * K + k];",
     "int64_t row = ((int64_t)d * L + l) * per_expert + slot[tok * K + k]; (void)begin;"),
    ("dequantisation with the first block's scale for every block",
     "scales[r * S + j / 128]", "scales[r * S]"),
    ("stage B forwards the row at its offset inside the home rank's block",
     "staging + (int64_t)i * H,", "staging + (int64_t)(i - stage_base[h]) * H,"),
    ("stage A reads the source token with transposed indices",
     "memcpy(staging + (int64_t)p * H, x + ((int64_t)s * T + t) * H,",
     "memcpy(staging + (int64_t)p * H, x + ((int64_t)t * R + s) * H,"),
]


def _build(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: pattern must occur once"
    mut = src.replace(old, new)
    shutil.copy(os.path.join(ROOT, "oracle", "ep_oracle.h"), tmp)
    c = os.path.join(tmp, "ep_oracle.c")
    open(c, "w").write(mut)
    so = os.path.join(tmp, "libmutant.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c, "-lm"],
                   check=True)
    return so


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new):
    with tempfile.TemporaryDirectory() as tmp:
        so = _build(tmp, name, old, new)
        env = dict(os.environ, EP_ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"]
                           + PIN_TESTS, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, f"no pin caught the mutant '{name}':\n{r.stdout[-2000:]}"


def test_unmutated_copy_passes():
    """Control: the same procedure with no mistake planted passes every pin."""
    with tempfile.TemporaryDirectory() as tmp:
        so = _build(tmp, "none", "#include <math.h>", "#include <math.h>")
        env = dict(os.environ, EP_ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"]
                           + PIN_TESTS, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-2000:]
