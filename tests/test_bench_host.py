"""Host logic of bench.py that needs no GPU: the kernel-source digest that
decides whether the committed ncu traffic figure still describes the kernel
(it ignores comments and blank space, and nothing else)."""
import bench


def test_code_only_drops_comments_and_blank_space():
    src = "int a; // one\n/* two\n lines */ int  b;\n\tint c; /*x*/int d;"
    assert bench.code_only(src) == "int a; int b; int c; int d;"


def test_code_only_keeps_literals():
    src = 'asm("add.u32 %0, 1; // not a comment" ::"r"(v)); char c = \'/\'; const char* s = "/* kept */";'
    assert bench.code_only(src) == src


def test_code_only_sees_code_changes():
    assert bench.code_only("x = a + b; // sum") != bench.code_only("x = a - b; // sum")
    assert bench.code_only("f(1);\n// note\n") == bench.code_only("f(1); /* other note */")


def test_digest_is_sixteen_hex_digits():
    d = bench.kernel_source_digest()
    assert len(d) == 16 and int(d, 16) >= 0
