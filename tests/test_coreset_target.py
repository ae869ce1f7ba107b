"""The coreset target in integer arithmetic (the kernels' header, built for the
host with g++) equals ceil(fp32(top_p) * double(total)) taken with IEEE double
rounding, clamped to [1, total], on random and boundary inputs: totals around
2^53 where the double conversion rounds, ties of the product's rounding, tiny
and subnormal top_p, and top_p one ulp below 1."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "moe_expert_step_gb300", "csrc")


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("target") / "target_harness")
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", CSRC, os.path.join(HERE, "target_harness.cpp"), "-o", exe],
                   check=True)
    return exe


def expected(bits: int, total: int) -> int:
    tp = float(np.array([bits], np.uint32).view(np.float32)[0])
    return min(max(math.ceil(tp * float(total)), 1), total)


def cases():
    rng = np.random.default_rng(7)
    out = []
    f32 = lambda x: int(np.array([x], np.float32).view(np.uint32)[0])
    tps = [f32(x) for x in (0.9, 0.7, 0.5, 0.3, 1e-6, 0.1, 0.99999994)] + [1, 2, 0x00400000, f32(np.float32(2.0 ** -30))]
    tps += [int(b) for b in rng.integers(0x00000001, f32(0.99999994) + 1, 400)]
    totals = [1, 2, 3, 7, 2 ** 53 - 1, 2 ** 53, 2 ** 53 + 1, 2 ** 53 + 2, 2 ** 53 + 3, 2 ** 54 + 2, 2 ** 54 + 6,
              2 ** 59 - 1, 2 ** 59 + 12345, 2 ** 62 + 2 ** 9 + 2 ** 8, 2 ** 63 - 1]
    totals += [int(t) for t in rng.integers(1, 2 ** 62, 300)]
    totals += [int(t) for t in rng.integers(2 ** 52, 2 ** 60, 300)]
    for tp in tps[:11]:
        out += [(tp, t) for t in totals]
    for i, tp in enumerate(tps[11:]):
        out += [(tp, totals[(7 * i + j) % len(totals)]) for j in range(8)]
    return out


def test_target_matches_ieee_double(harness):
    cs = cases()
    inp = "".join(f"{b} {t}\n" for b, t in cs)
    res = subprocess.run([harness], input=inp, capture_output=True, text=True, check=True).stdout.split()
    assert len(res) == len(cs)
    bad = [(b, t, int(r), expected(b, t)) for (b, t), r in zip(cs, res) if int(r) != expected(b, t)]
    assert not bad, bad[:5]
