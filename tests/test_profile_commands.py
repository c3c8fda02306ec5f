"""The commands quoted in profiles/*.md run committed code: every
`python bench.py ...` there parses with bench.py's own argument parser
(known flags, a known --kernel, at least 3 warm-up steps), and every file
quotes at least one command."""
import pathlib
import re
import shlex

import pytest

import bench

ROOT = pathlib.Path(__file__).resolve().parent.parent
PROFILES = sorted((ROOT / "profiles").glob("*.md"))


def bench_commands(text):
    # join continued lines, then take each `python bench.py` up to the end
    # of the shell word list (a redirection, a pipe, a command separator, a
    # comment or closing markdown quote)
    text = re.sub(r"\\\n\s*", " ", text)
    for m in re.finditer(r"python bench\.py([^\n`#>|&;]*)", text):
        yield m.group(1)


def test_profiles_exist():
    assert PROFILES, "profiles/ holds the ncu summaries"


@pytest.mark.parametrize("path", PROFILES, ids=lambda p: p.name)
def test_profile_commands_parse(path):
    text = path.read_text()
    cmds = list(bench_commands(text))
    assert cmds, f"{path.name} quotes no bench.py command"
    # a quoted shell loop (`for k in a b c; do`) runs its command once per value
    loops = {m.group(1): m.group(2).split() for m in re.finditer(r"for (\w+) in ([^;\n]*);", text)}
    ap = bench.build_parser()
    for c in cmds:
        variants = [c]
        for var, values in loops.items():
            if "$" + var in c:
                variants = [v.replace("$" + var, val) for v in variants for val in values]
        for v in variants:
            assert "$" not in v, (path.name, v)
            args = ap.parse_args(shlex.split(v))
            assert args.warmup >= 3, (path.name, v)
