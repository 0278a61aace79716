"""Static checks of bench.py on CPU: its GPU legs cannot run here, so every
name they load must at least resolve (a local, a parameter, a name of an
enclosing function, a module-level name or a builtin). This catches the
class of mistake that would otherwise surface only as a NameError on the GPU
box."""
import builtins
import os
import symtable

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _unresolved(path):
    src = open(path).read()
    top = symtable.symtable(src, path, "exec")
    module_names = {s.get_name() for s in top.get_symbols() if s.is_assigned() or s.is_imported()}
    known = module_names | set(dir(builtins))
    bad = []

    def walk(table, enclosing):
        names = {s.get_name() for s in table.get_symbols()
                 if s.is_assigned() or s.is_parameter() or s.is_imported()}
        scope = enclosing | names
        for s in table.get_symbols():
            if not s.is_referenced() or s.get_name() in scope:
                continue
            if s.is_global() or s.is_free():
                if s.get_name() not in known and s.get_name() not in enclosing:
                    bad.append(f"{table.get_name()}:{s.get_name()}")
        for child in table.get_children():
            walk(child, scope if table.get_type() == "function" else enclosing)

    for child in top.get_children():
        walk(child, set())
    return bad


def test_every_name_in_bench_resolves():
    assert _unresolved(os.path.join(ROOT, "bench.py")) == []


def test_the_check_catches_an_undefined_name(tmp_path):
    p = tmp_path / "planted.py"
    p.write_text("import json\n\ndef f(x):\n    y = x + 1\n    return json.dumps({'a': r['gbs'] / y})\n")
    assert _unresolved(str(p)) == ["f:r"]
