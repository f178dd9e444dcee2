"""The ncu and timing summaries under profiles/ name the commands that made
them; every concrete `python bench.py ...` line there must still parse with
the committed bench.py, and every ncu capture must keep its clocks
unlocked."""
import glob
import os
import re
import shlex

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _command_lines():
    """(file, command) for every command in the summaries' code blocks, with
    backslash continuations joined and trailing comments dropped."""
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        in_block, buf = False, ""
        for raw in open(path):
            line = raw.rstrip("\n")
            if line.startswith("```"):
                in_block, buf = not in_block, ""
                continue
            if not in_block:
                continue
            line = re.sub(r"\s+#.*$", "", line)
            buf += line.strip() + " "
            if line.endswith("\\"):
                buf = buf.replace("\\ ", "")
                continue
            if buf.strip():
                out.append((os.path.basename(path), buf.strip()))
            buf = ""
    return out


def test_profiles_hold_commands():
    cmds = _command_lines()
    assert any("ncu" in c for _, c in cmds)
    assert any(c.startswith("python bench.py") for _, c in cmds)


@pytest.mark.parametrize("where,cmd", [(f, c) for f, c in _command_lines() if "python bench.py" in c])
def test_bench_commands_parse(where, cmd):
    import bench
    args = cmd[cmd.index("python bench.py") + len("python bench.py"):]
    if re.search(r"[<\[]|\.\.\.", args):  # a template line (placeholders, optional flags)
        args = re.sub(r"<[^>]*>", "1", args)
        while "[" in args:  # optional flags, innermost first
            args = re.sub(r"\[[^\[\]]*\]", "", args)
        args = re.sub(r"\d+,\.\.\.,\d+", "4096,8192", args)
    bench.parse_args(shlex.split(args))


@pytest.mark.parametrize("where,cmd", [(f, c) for f, c in _command_lines() if c.startswith("ncu ")])
def test_ncu_captures_leave_clocks_alone(where, cmd):
    if cmd.startswith("ncu -i"):  # reading a report back, no GPU
        return
    assert "--clock-control none" in cmd, (where, cmd)
