"""Host logic of the benchmark on CPU: the per-expert roof, the per-workload
record's entries, and the one-core leg of the oracle timing (BLAS threads and
the calling thread's affinity are restored afterwards)."""
import os

import numpy as np

import bench

CFG = dict(world=8, tokens_per_slot=1024, hidden=7168, num_experts=256, topk=8, inter=2048)


def test_per_expert_roof_single_expert_is_its_own_roof():
    H, I = CFG["hidden"], CFG["inter"]
    for c in (1, 256, 100000):
        counts = np.zeros(256, dtype=np.int64)
        counts[3] = c
        flops = 6.0 * c * H * I
        bts = 3.0 * H * I * 2 + 4.0 * c * H + 4.0 * c * I
        want = max(flops / 2e15, bts / 8e12)
        assert np.isclose(bench.per_expert_roof_s(CFG, counts, 2000.0, 8000.0), want, rtol=1e-12)


def test_per_expert_roof_bounds():
    """The sum of per-expert roofs is never below the plain roof (max of the
    sums) and never above the sum of both times; empty experts cost nothing."""
    rng = np.random.default_rng(1)
    H, I = CFG["hidden"], CFG["inter"]
    for _ in range(5):
        counts = rng.zipf(1.5, size=256).clip(max=8192) * (rng.random(256) < 0.7)
        t = bench.per_expert_roof_s(CFG, counts, 1900.0, 6700.0)
        flops = sum(6.0 * c * H * I for c in counts)
        bts = sum(3.0 * H * I * 2 + 4.0 * c * H + 4.0 * c * I for c in counts if c > 0)
        tf, tb = flops / 1.9e15, bts / 6.7e12
        assert max(tf, tb) * (1 - 1e-12) <= t <= (tf + tb) * (1 + 1e-12)
    assert bench.per_expert_roof_s(CFG, np.zeros(256, dtype=np.int64), 1900.0, 6700.0) == 0.0


def test_workload_summary_entry():
    counts = np.full(256, 256, dtype=np.int64)
    stages = {"route": 0.01, "dispatch": 0.2, "expert_ffn": 4.5, "combine": 0.17}
    e = bench.workload_summary("deepseek", CFG, 0, 20, 20 * 4.9, stages, None, counts)
    assert e["fused"] is False and e["ms_per_step"] == 4.9
    assert np.isclose(e["tokens_per_s"], 8192 / 4.9e-3)
    assert e["ffn_roof"]["bound"] in ("hbm", "tensor") and 0 < e["ffn_roof"]["frac"] < 2
    assert e["stage_bandwidth"]["dispatch_frac"] > 0 and e["experts_hit"] == 256
    f = bench.workload_summary("decode", CFG, 1, 20, 20 * 3.5, {"fused": 3.5}, None, counts)
    assert "dispatch_frac" not in f["stage_bandwidth"] and f["fused"] is True


def test_one_core_leg_restores_threads_and_affinity():
    before_threads = bench.blas_threads()
    before_aff = os.sched_getaffinity(0)
    with bench.OneCore() as one:
        if one.getf is not None:
            assert one.threads == 1
        assert len(os.sched_getaffinity(0)) == 1
        a = np.ones((64, 64))
        assert (a @ a)[0, 0] == 64.0
    assert bench.blas_threads() == before_threads
    assert os.sched_getaffinity(0) == before_aff


def test_clock_summary_keeps_only_the_timed_window():
    c = bench.ClockSampler(0)
    c.lines = ["2026/12/03 06:13:02.100, 2070, 2070, 500.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "2026/12/03 06:13:02.300, 1600, 2070, 580.2, 0x4, Not Active, Not Active, Not Active, Active",
               "2026/12/03 06:13:03.300, 1500, 2070, 590.0, 0x4, Not Active, Not Active, Active, Active"]
    c.mark(c._when("2026/12/03 06:13:02.050"), c._when("2026/12/03 06:13:02.350"))
    s = c.summary()
    assert s["samples"] == 2 and s["sm_min_mhz"] == 1600.0 and s["reasons"] == ["sw_power_cap"]
    c.window = None                                  # no window: every sample counts
    s = c.summary()
    assert s["samples"] == 3 and "sw_thermal_slowdown" in s["reasons"] and s["sm_min_mhz"] == 1500.0


def test_code_hash_ignores_comments_only():
    """The traffic record is keyed to the kernels' code: a comment edit or
    re-indentation keeps the key, any code edit changes it, and comment
    markers inside string or character literals are code."""
    src = ('// header\n#include "x.cuh"\n/* block\n comment */ int f(int a) {\n'
           '  return a + 1;  // trailing\n}\nconst char *s = "a // b /* c */";\nchar q = \'/\';\n')
    base = bench.code_of(src)
    assert "header" not in base and "trailing" not in base and "block" not in base
    assert '"a // b /* c */"' in base and "'/'" in base
    assert bench.code_of(src.replace("// trailing", "// other words")) == base
    assert bench.code_of(src.replace("  return", "\n\n      return")) == base
    assert bench.code_of(src.replace("a + 1", "a + 2")) != base
    assert bench.code_of(src.replace('"a // b /* c */"', '"a // b"')) != base


def _profile_commands():
    """Every `python bench.py ...` and `python -m pytest ...` command written
    in the committed ncu summaries (continuation lines joined)."""
    import glob
    import re
    cmds = []
    for path in sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md"))):
        text = re.sub(r"\\\n\s*", " ", open(path, encoding="utf-8").read())
        for line in text.splitlines():
            for m in re.finditer(r"python (bench\.py|-m pytest)([^`\n]*)", line):
                cmds.append((os.path.basename(path), m.group(1), m.group(2).strip()))
    return cmds


def test_profile_commands_run_committed_files_with_valid_flags():
    """The commands the profile summaries give still parse: bench.py accepts
    every flag they pass and knows every workload they name, and the test
    files they run exist."""
    import shlex
    import moe_synth as ms
    cmds = _profile_commands()
    assert len(cmds) >= 10
    for src, what, rest in cmds:
        argv = shlex.split(rest)
        if what == "bench.py":
            argv = ["deepseek" if a == "NAME" else a for a in argv]
            args = bench.parse(argv)
            assert args.config in ms.CONFIGS, (src, rest)
        else:
            tests = [a for a in argv if a.startswith("tests/")]
            assert tests and all(os.path.exists(os.path.join(bench.ROOT, t)) for t in tests), (src, rest)
            if "-k" in argv:  # every word of the selection names something in the file
                text = "".join(open(os.path.join(bench.ROOT, t), encoding="utf-8").read() for t in tests)
                words = [w for w in argv[argv.index("-k") + 1].split() if w not in ("and", "or", "not")]
                assert all(w in text for w in words), (src, rest)
