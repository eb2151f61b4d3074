"""The key that ties a profile capture to the kernels it measured
(bench.source_sha) follows the code and ignores comments and blank space."""
import bench

SRC = '''// leading comment
#include "x.h"
/* block
   comment */ int f(int a)   // trailing
{
    asm volatile("ld.global.cg.s32 %0, [%1]; // not a comment" : "=r"(a));
    const char c = '/';   /* inline */ return a + c;
}
'''


def test_comments_and_blank_space_do_not_count():
    edited = (SRC.replace("// leading comment", "// another comment\n\n")
                 .replace("/* inline */", "/* longer\n inline comment */")
                 .replace("int f(int a)", "int   f(int a)"))
    assert bench.code_only(edited) == bench.code_only(SRC)
    assert "leading" not in bench.code_only(SRC) and "inline" not in bench.code_only(SRC)


def test_code_and_string_literals_count():
    for old, new in (("a + c", "a - c"), ("ld.global.cg", "ld.global.ca"),
                     ("// not a comment", "// still not a comment"), ("'/'", "'*'")):
        assert bench.code_only(SRC.replace(old, new)) != bench.code_only(SRC), old


def test_current_sources_hash():
    h = bench.source_sha()
    assert len(h) == 16 and int(h, 16) >= 0
