"""Runs a pytest suite again in a child process with environment switches set.

Several library switches (kernel choices) are read once per process, so the suites that
exercise the non-default kernels re-run an existing test file in a child pytest. A child
whose tests were all skipped or deselected would still exit 0, so the result is read from
the child's summary: it must report at least one passed test and none skipped.
"""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_child_pytest(test_file, env_extra, k=None, timeout=900):
    env = dict(os.environ, **env_extra)
    cmd = [sys.executable, "-m", "pytest", "-q", "-rs", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", test_file)]
    if k:
        cmd += ["-k", k]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    tail = r.stdout[-3000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    lines = [l for l in r.stdout.splitlines() if re.search(r"\d+ passed", l)]
    assert lines, "child pytest printed no pass count:\n" + tail
    summary = lines[-1]
    passed = int(re.search(r"(\d+) passed", summary).group(1))
    assert passed > 0, summary
    assert "skipped" not in summary and "SKIPPED" not in r.stdout, "child skipped tests:\n" + tail
    return passed
