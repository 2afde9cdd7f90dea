"""The FP8 codec divides each channel by its block scale through a correctly
rounded reciprocal and one Markstein correction step instead of an IEEE
division per channel.  tests/c/e4m3_division.c restates that arithmetic in C
and compares its e4m3 codes with those of the IEEE quotient (the oracle's
encoder) for every bf16 x under every finite bf16 block maximum (about
1.05e9 pairs, ~50 s of CPU time spread over the cores), and for every block
maximum around the scale below which the codec falls back to the division.
EP_E4M3_DIVISION_SAMPLE=1 walks every 13th block maximum instead."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = tmp_path_factory.mktemp("e4m3") / "e4m3_division"
    r = subprocess.run([gcc, "-std=c11", "-O2", "-ffp-contract=off", "-Wall", "-Werror",
                        "-I", os.path.join(ROOT, "oracle"), os.path.join(ROOT, "tests", "c", "e4m3_division.c"),
                        os.path.join(ROOT, "oracle", "ep_oracle.c"), "-lm", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def _run(exe, jobs):
    procs = [subprocess.Popen([exe] + [str(a) for a in args], stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for args in jobs]
    pairs = bad_code = bad_quot = 0
    for p in procs:
        out, err = p.communicate(timeout=1800)
        assert p.returncode == 0, err
        n, c, q = map(int, out.split())
        pairs, bad_code, bad_quot = pairs + n, bad_code + c, bad_quot + q
    return pairs, bad_code, bad_quot


def test_reciprocal_division_gives_the_ieee_codes(checker):
    full = os.environ.get("EP_E4M3_DIVISION_SAMPLE") != "1"
    step = 1 if full else 13
    shards = max(1, min(os.cpu_count() or 1, 16))
    jobs = [(1 + j * step, shards * step) for j in range(shards)]
    pairs, bad_code, bad_quot = _run(checker, jobs)
    assert pairs > (1_000_000_000 if full else 70_000_000)
    assert bad_code == 0 and bad_quot == 0


def test_around_the_fallback_scale(checker):
    # scale = amax / 448 crosses 2^-100 at amax = 1.75 * 2^-92 (bf16 0x11E0)
    pairs, bad_code, bad_quot = _run(checker, [(0x11C0, 1, 0x1200)])
    assert pairs > 100_000
    assert bad_code == 0 and bad_quot == 0
