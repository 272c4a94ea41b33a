"""bench.py's kernel-source hash, which decides whether the DRAM traffic
recorded by ncu (profiles/dram_traffic.json) still describes the kernels:
comments and whitespace do not count, code and string literals do."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_for_hash", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_strip_keeps_code_and_literals():
    strip = _bench().strip_c_comments
    assert strip("int a = 1; // note\n/* block\n comment */ int b;") == "int a = 1; int b;"
    assert strip('asm("st.v8 [%0]; // not a comment");') == 'asm("st.v8 [%0]; // not a comment");'
    assert strip("char c = '/'; char d = '\\''; int e; // x") == "char c = '/'; char d = '\\''; int e;"
    assert strip("a  =\n\tb;") == "a = b;"


def _sha_of(bench, tmp_path, sources):
    csrc = tmp_path / "speculative_decoding_verify_split_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    for f in csrc.iterdir():
        f.unlink()
    for name, text in sources.items():
        (csrc / name).write_text(text)
    bench.ROOT = str(tmp_path)
    return bench.kernel_source_sha()


def test_hash_ignores_comments_not_code(tmp_path):
    bench = _bench()
    base = _sha_of(bench, tmp_path, {"k.cu": "__global__ void k() { int x = 1; }\n"})
    reworded = _sha_of(bench, tmp_path, {"k.cu": "// a kernel\n__global__ void k() {\n  int x = 1;  // one\n}\n"})
    changed = _sha_of(bench, tmp_path, {"k.cu": "__global__ void k() { int x = 2; }\n"})
    renamed = _sha_of(bench, tmp_path, {"j.cu": "__global__ void k() { int x = 1; }\n"})
    assert base == reworded
    assert base != changed and base != renamed
