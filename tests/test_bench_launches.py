"""The bench's gpu_launches claim: the library's kernels in one step, by its
dispatch rules, against the launch lists taken on the GPU (ncu, one pass,
duration only) for three workloads:
  32K GQA:     meta_kernel; attn (exact) + merge; unit_select_kernel, attn
               (sparse) + merge                                    -> 6
  1.3B MHA:    the same kernels at d = 64                          -> 6
  OPT-30B 4-bit: meta_q4_kernel; attn + merge; score_kernel, topk_warp_kernel
               (writing the unions), attn (writing out)            -> 6
"""

import bench
from workloads import by_name


def test_step_launches_match_the_launch_lists():
    assert bench.step_launches(by_name("llama3-8b-gqa-b16-n32k")) == 6
    assert bench.step_launches(by_name("mha-1.3b-b8-h32-d64-n8k")) == 6
    assert bench.step_launches(by_name("opt-30b-q4-b64-h56-n2k")) == 6


def test_step_launches_short_contexts():
    # below 256 selection pages the score / top-K kernels select; with one
    # query head per kv head the top-K writes the unions (no union kernel)
    w = by_name("tiny-mha-b1-h16-d64-n1k")
    assert bench.step_launches(w) == 7
    assert bench.step_launches(w.replace(Hkv=4)) == 8
