"""bench.py's code hash, the key under which profiles/dram_traffic.txt keeps
ncu's DRAM counters: it ignores comments and blank lines, and nothing else;
and the counter lines are well formed."""
import importlib.util
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _sha(tmp_path, text, name="k.cu"):
    p = tmp_path / name
    p.write_text(text)
    return _bench().code_sha(str(p))


def test_comments_and_blank_lines_do_not_change_the_hash(tmp_path):
    base = "int f(int a) {\n  return a + 1;\n}\n"
    commented = "// header\n\nint f(int a) {  /* the\n argument */\n  return a + 1;  // one more\n}\n\n"
    assert _sha(tmp_path, base, "a.cu") == _sha(tmp_path, commented, "b.cu")


def test_code_and_literals_change_the_hash(tmp_path):
    base = "int f(int a) {\n  return a + 1;\n}\n"
    assert _sha(tmp_path, base, "a.cu") != _sha(tmp_path, base.replace("+ 1", "+ 2"), "b.cu")
    lit = 'const char* s = "a // b";\n'
    assert _sha(tmp_path, lit, "c.cu") != _sha(tmp_path, 'const char* s = "a ";\n', "d.cu")
    assert _sha(tmp_path, 'const char* s = "/* x */";\n', "e.cu") != _sha(tmp_path, 'const char* s = "";\n', "f.cu")


def test_traffic_lines_are_well_formed():
    """Every counter line names a known kernel, its code hash and its bytes;
    bench.py reports the counters only while the hash matches the source."""
    known = {"decode_fused", "routed_gateup", "routed_down", "router_shared_gateup", "combine", "lm_gemv"}
    lines = open(os.path.join(ROOT, "profiles", "dram_traffic.txt")).read().split("\n")
    for ln in filter(None, lines):
        f = dict(kv.split("=", 1) for kv in ln.split() if "=" in kv)
        assert f["kernel"] in known, ln
        assert re.fullmatch(r"[0-9a-f]{16}", f["code_sha"]), ln
        assert int(f["bytes_per_launch"]) == int(f["read"]) + int(f["write"]), ln
