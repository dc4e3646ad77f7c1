"""The 8-bit metadata kernel finds each code without a search: from the
guesses fm = floor(fl(fl(m - lo) * fl(1 / step))) and gM = ceil(same for M) it
takes
    code_min = fm - 1 + [dec(fm) <= m] + [dec(fm + 1) <= m],
    code_max = gM - 1 + [dec(gM) < M] + [dec(gM - 1) < M],
which is the definition (the largest c with dec(c) <= m, the smallest with
dec(c) >= M, dec(c) = fma(c, step, lo)) whenever the defining code is within
one of the guess -- true for a 16-bit page with a step in [2^-100, inf), whose
step is at least 16 fp32 ulps of every value in it.  Each comparison is the
sign bit of a difference (rounded down for <=, where an exact zero is -0).
This checks the rule
against the definition (all 256 codes tried) on the host with C's fmaf, over
every page of two 16-bit values up to 16 apart with every value between,
whole random pages, every exact grid hit of random pages (where the rounded
guess lands one past the code) and random wide pages near grid points, for
bf16 and fp16."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))


def test_branch_free_codes_equal_definition(tmp_path):
    exe = str(tmp_path / "meta8_codes")
    r = subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-frounding-math", "-o", exe,
                        os.path.join(HERE, "native", "meta8_codes_check.c"), "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    runs = []
    for fmt, n in (("0", 65280), ("1", 63487)):  # finite bf16 / fp16 values (one zero)
        for i in range(4):
            runs.append([fmt, "tight", "16", str(n * i // 4), str(n * (i + 1) // 4)])
        runs.append([fmt, "pages", "1500", "0x51" + fmt, "4096"])
        runs.append([fmt, "exact", "300000", "0x52" + fmt, "2000"])
        runs.append([fmt, "exact", "60000", "0x53" + fmt, "60000"])
        runs.append([fmt, "random", "1000000", "0x54" + fmt])
    procs = [subprocess.Popen([exe] + a, stdout=subprocess.PIPE, text=True) for a in runs]
    outs = [p.communicate()[0] for p in procs]
    for a, p, out in zip(runs, procs, outs):
        assert p.returncode == 0, (a, out)
        assert out.startswith("ok "), (a, out)
    assert sum(int(o.split()[1]) for o in outs) > 5 * 10 ** 7
