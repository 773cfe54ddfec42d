"""Every name a function of the committed Python sources reads is bound somewhere: in the
function, an enclosing function, the module, or the builtins.

Paths that only run on a GPU (the benchmark's workloads, the GPU tests) are not executed
by the CPU suite, so a name left undefined by an edit there would only show on the GPU
box; this check reads the sources' symbol tables instead."""

import builtins
import glob
import os
import symtable

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = sorted(
    [os.path.join(ROOT, f) for f in ("bench.py", "synth.py", "__graft_entry__.py")]
    + glob.glob(os.path.join(ROOT, "compressed_attention_gb300", "*.py"))
    + glob.glob(os.path.join(ROOT, "oracle", "*.py"))
    + glob.glob(os.path.join(ROOT, "tests", "*.py"))
)
# set at run time by the interpreter or by pytest, not by an assignment in the file
IMPLICIT = {"__file__", "__name__", "__builtins__", "__doc__", "__spec__", "__path__"}


def _unbound(path):
    top = symtable.symtable(open(path).read(), path, "exec")
    module_names = {s.get_name() for s in top.get_symbols()
                    if s.is_assigned() or s.is_imported() or s.is_namespace()}
    defined = module_names | set(dir(builtins)) | IMPLICIT
    missing = []

    def walk(table):
        for child in table.get_children():
            if child.get_type() in ("function", "lambda") or child.get_type().endswith("function"):
                for s in child.get_symbols():
                    if s.is_referenced() and s.is_global() and not s.is_declared_global() \
                            and s.get_name() not in defined:
                        missing.append(f"{child.get_name()}:{s.get_name()}")
            walk(child)

    walk(top)
    return missing


@pytest.mark.parametrize("path", SOURCES, ids=[os.path.relpath(p, ROOT) for p in SOURCES])
def test_every_name_is_bound(path):
    assert _unbound(path) == []


def test_the_check_sees_an_unbound_name(tmp_path):
    """The check itself: a function reading a name nobody binds is reported."""
    f = tmp_path / "m.py"
    f.write_text("import os\n\ndef run():\n    def write():\n        pass\n    return (step,), os.sep, write\n")
    assert _unbound(str(f)) == ["run:step"]
