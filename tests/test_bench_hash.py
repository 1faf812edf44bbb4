"""The source hash that keys profiled figures to the kernel code they were measured on (bench.py)."""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_code_only_drops_comments_and_layout():
    b = _bench()
    a = b.code_only("int a = 1; // note\n/* block\n comment */ int  b =\n 2;")
    assert a == "int a = 1; int b = 2;"
    # comment markers inside string literals are code
    assert b.code_only('asm("x // y /* z */");  // c') == 'asm("x // y /* z */");'
    assert b.code_only('const char* s = "a\\"//b"; // c') == 'const char* s = "a\\"//b";'


def test_code_changes_change_the_hash_and_comments_do_not():
    b = _bench()
    base = "__global__ void k(float* p) { p[0] = 1.f; }\n"
    assert b.code_only(base) == b.code_only("// header\n" + base.replace("{", "{ /* body */"))
    assert b.code_only(base) != b.code_only(base.replace("1.f", "2.f"))


def test_hash_is_stable_and_short():
    b = _bench()
    h = b.kernel_source_hash()
    assert h == b.kernel_source_hash() and len(h) == 16


def test_hash_covers_existing_sources_of_the_kernel():
    b = _bench()
    for f in b.KERNEL_SOURCES["k_verify"]:
        assert os.path.exists(os.path.join(ROOT, f)), f
    assert any(f.endswith("sv_kernels.cu") for f in b.KERNEL_SOURCES["k_verify"])
