"""The kernel's unit schedule, walked on the CPU.

tests/schedule_harness.cu compiles the library's own scheduling code as
host code and runs, for every CTA of the persistent grid, the walk the
kernel runs. Every (sequence, token block, head group) unit must come up
exactly once and the visited key tiles must add up to the plan. Covers the
tile shapes of every group size (powers of two, G = 1, G not dividing 128,
G > 128), head shards, varlen mixes and grids smaller than the unit count.
"""
import os
import subprocess

import numpy as np
import pytest

from long_causal_gqa_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HARNESS = os.path.join(ROOT, "tests", "schedule_harness.cu")


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_harness")
    subprocess.run([build.nvcc_path(), *build.ARCH_FLAGS, "-O1", "-std=c++17", "-I",
                    os.path.join(ROOT, "include"), "-o", exe, HARNESS], check=True)
    return exe


def run(exe, cases):
    text = "".join("%d %d %d %d %d %d %d %s\n" % (int(c), hq, hkv, kb, kc, sms, len(lens),
                                                  " ".join(map(str, lens)))
                   for c, hq, hkv, kb, kc, sms, lens in cases)
    out = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout
    lines = out.strip().splitlines()
    assert len(lines) == len(cases)
    return lines


HEADLINE = [
    (True, 64, 8, 0, 0, 152, (10231,)),
    (True, 64, 8, 0, 0, 152, (7700,)),
    (True, 64, 8, 0, 0, 152, (8184, 8199, 8510, 10231)),
    (True, 64, 8, 0, 0, 152, (32768,)),
    (False, 64, 8, 0, 0, 152, (19316,)),
    (False, 64, 8, 0, 0, 152, (34121,)),
    (True, 64, 8, 0, 0, 148, (10231,)),
]


def test_workload_schedules(harness):
    for case, line in zip(HEADLINE, run(harness, HEADLINE)):
        assert line.startswith("ok"), (case, line)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (64, 64), (24, 8), (40, 8), (48, 8), (56, 8),
                                    (16, 8), (32, 2), (128, 1), (96, 1), (256, 1), (262, 2),
                                    (384, 3), (12, 1)])
def test_group_sizes(harness, hq, hkv):
    cases = []
    for causal in (True, False):
        for sms in (152, 7, 1):
            for lens in ((1,), (255,), (256,), (257,), (1000,), (5, 0, 129, 1, 300, 0, 64),
                         (3000, 2999, 1)):
                cases.append((causal, hq, hkv, 0, 0, sms, lens))
    for case, line in zip(cases, run(harness, cases)):
        assert line.startswith("ok"), (case, line)


def test_head_shards(harness):
    cases = []
    for hq, hkv in ((64, 8), (64, 64), (40, 8), (256, 1)):
        for kb in range(0, hkv, max(1, hkv // 4)):
            for kc in (0, 1, hkv - kb):
                for causal in (True, False):
                    cases.append((causal, hq, hkv, kb, kc, 152, (10231,)))
                    cases.append((causal, hq, hkv, kb, kc, 13, (700, 0, 33, 1024)))
    for case, line in zip(cases, run(harness, cases)):
        assert line.startswith("ok"), (case, line)


def test_random_mixes(harness):
    rng = np.random.default_rng(77)
    cases = []
    for _ in range(60):
        hkv = int(rng.choice([1, 2, 3, 8]))
        g = int(rng.choice([1, 2, 3, 5, 6, 7, 8, 16, 24, 64, 128, 130]))
        n = int(rng.integers(1, 40))
        lens = tuple(int(x) for x in rng.integers(0, 3000, n))
        if sum(lens) == 0:
            lens = lens + (17,)
        cases.append((bool(rng.integers(2)), g * hkv, hkv, 0, 0, int(rng.choice([152, 9, 2])),
                      lens))
    for case, line in zip(cases, run(harness, cases)):
        assert line.startswith("ok"), (case, line)
