"""Every name a function of the benchmark, the entry points or the Python binding reads is
defined somewhere: a local, an enclosing function's variable, a module-level binding or a
builtin. The GPU legs of these files cannot run on a CPU machine, so a misspelt or stale name
on them would otherwise only show up on the GPU."""
import builtins
import pathlib
import symtable

import pytest

ROOT = pathlib.Path(__file__).resolve().parent.parent
FILES = ["bench.py", "__graft_entry__.py", "scaled_quantize_fp8_gb300/binding.py",
         "scaled_quantize_fp8_gb300/_lib.py", "scaled_quantize_fp8_gb300/build.py",
         "scaled_quantize_fp8_gb300/__init__.py", "workloads/generators.py"]


def undefined_globals(path):
    src = path.read_text()
    top = symtable.symtable(src, str(path), "exec")
    defined = {s.get_name() for s in top.get_symbols()
               if s.is_assigned() or s.is_imported() or s.is_namespace()}
    bad = []

    def walk(t):
        for s in t.get_symbols():
            n = s.get_name()
            if s.is_referenced() and s.is_global() and n not in defined \
                    and not hasattr(builtins, n) and n != "__file__":
                bad.append(f"{t.get_name()}: {n}")
        for c in t.get_children():
            walk(c)

    for c in top.get_children():
        walk(c)
    return bad


@pytest.mark.parametrize("name", FILES)
def test_no_undefined_names(name):
    assert undefined_globals(ROOT / name) == []


def test_checker_finds_a_stale_name(tmp_path):
    """The checker itself: a function reading a name bound nowhere is reported."""
    f = tmp_path / "m.py"
    f.write_text("import os\n\ndef run():\n    x = os.sep\n    step()\n    return x\n")
    assert undefined_globals(f) == ["run: step"]
