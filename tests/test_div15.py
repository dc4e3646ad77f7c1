"""The 4-bit format's step of a normal group is fp16_down(fp32_down(x / 15)),
x = fp32_down(max - min).  The kernels form fl(x / 15) as q = fl(x * c),
c = fl(1/15), corrected once with fused multiply-adds (q + fl(x - 15 q) * c,
the FMA method for division by a constant), then round it down with the sign
of the exact remainder x - 15 q.  This checks, for every binary32 x in
[0, 2^18) -- which holds the range of any two finite fp16 values -- that the
corrected quotient is the IEEE quotient and the rounded-down one the largest
binary32 q with 15 q <= x, on the host with C's fmaf (split over processes)."""

import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_fma_division_by_15_is_correctly_rounded(tmp_path):
    exe = str(tmp_path / "div15")
    r = subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-o", exe,
                        os.path.join(HERE, "native", "div15_exhaustive.c"), "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    end = 0x48800000
    parts = max(1, min(16, os.cpu_count() or 1))
    bounds = [end * i // parts for i in range(parts + 1)]
    procs = [subprocess.Popen([exe, str(bounds[i]), str(bounds[i + 1])], stdout=subprocess.PIPE,
                              text=True) for i in range(parts)]
    outs = [p.communicate()[0] for p in procs]
    for p, out in zip(procs, outs):
        assert p.returncode == 0, out
    assert sum(int(o.split()[1]) for o in outs) == end
