"""Host-side pins of the reduction workload against the figures the pages
print ("03 CUDA Shared Memory: Tiling, Bank Conflicts, and Reduction",
section "Reduction"):

* 2^24 inputs folded by 256-thread blocks take three launches,
  65,536 -> 256 -> 1 values (checked on the library's own plan);
* over the eight folding steps of a 256-value block, version 0
  (`tid % (2*s) == 0`) keeps min(8, a_j) warps busy per step, 47 in all;
  version 1 (`tid < s`) keeps ceil(a_j / 32), 12 in all, a_j = 256 / 2^(j+1)
  (checked on a model of the kernels' branch conditions).
"""
import math

import shared_memory_tiled_fp32_gb300 as tg

BLOCK = 256


def active_warps_per_step(cond, steps):
    """Warps with at least one thread for which cond(tid, s) holds, per step."""
    out = []
    for s in steps:
        warps = {tid // 32 for tid in range(BLOCK) if cond(tid, s)}
        out.append(len(warps))
    return out


def test_pass_counts_match_the_pages():
    for v in ("interleaved", "sequential", "shuffle"):
        p = tg.reduce_plan(v, 2 ** 24, num_sms=152)
        assert p["passes"] == 3 and p["counts"] == [65536, 256, 1]
        assert p["workspace_bytes"] == 4 * (65536 + 256)
    assert tg.reduce_plan("atomic", 2 ** 24, num_sms=152)["passes"] == 2
    f = tg.reduce_plan("fast", 2 ** 24, num_sms=152)
    assert f["passes"] == 2 and f["counts"] == [4 * 152, 1] and f["workspace_bytes"] == 4 * 4 * 152


def test_active_warps_47_and_12():
    # version 0: s = 1, 2, 4, ..., 128, thread tid works when tid % (2s) == 0
    v0 = active_warps_per_step(lambda tid, s: tid % (2 * s) == 0, [2 ** j for j in range(8)])
    # version 1: s = 128, 64, ..., 1, thread tid works when tid < s
    v1 = active_warps_per_step(lambda tid, s: tid < s, [128 >> j for j in range(8)])
    a = [BLOCK // 2 ** (j + 1) for j in range(8)]
    assert v0 == [min(8, aj) for aj in a] and sum(v0) == 47
    assert v1 == [math.ceil(aj / 32) for aj in a] and sum(v1) == 12
    # both versions add the same number of values per step
    assert [sum(1 for t in range(BLOCK) if t % (2 * s) == 0) for s in [2 ** j for j in range(8)]] == a
    assert [sum(1 for t in range(BLOCK) if t < s) for s in [128 >> j for j in range(8)]] == a
