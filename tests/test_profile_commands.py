"""Every ncu summary under profiles/ names the command that made it; those
commands must run committed files with arguments the benchmark accepts, and
ncu must be told not to touch the clocks."""
import glob
import os
import re
import shlex

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def commands(path):
    for line in open(path).read().splitlines():
        line = line.strip()
        if line.startswith("ncu ") and "python bench.py" in line:
            yield line


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_commands_are_runnable(path):
    import bench
    cmds = list(commands(path))
    assert cmds, "a summary names the command that made it"
    for cmd in cmds:
        assert "--clock-control none" in cmd
        args = shlex.split(cmd.split("python bench.py", 1)[1])
        parsed = bench.build_parser().parse_args(args)
        assert parsed.warmup >= 3
        # the launch list takes the duration metric alone; other metrics only
        # on one kernel and at most three launches
        ncu_part = cmd.split("python bench.py", 1)[0]
        metrics = re.search(r"--metrics (\S+)", ncu_part)
        full_set = re.search(r"--set \w+", ncu_part)
        if (metrics and metrics.group(1) != "gpu__time_duration.sum") or full_set:
            assert re.search(r"-k \S+", cmd) and re.search(r"-c [123]\b", cmd), cmd
