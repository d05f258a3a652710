"""bench.py's guard on the recorded DRAM traffic: it hashes the kernel sources'
code without comments, so a comment-only edit keeps a capture valid while any
change to the code (including inside string literals, e.g. inline PTX) makes it
stale."""
import bench

SRC = ('int a = 1;  // remark one\n'
       '/* remark two\n   continued */\n'
       'asm("ex2.approx.f32 %0, %1; // kept");\n'
       "char q = '\"'; const char* s = \"x /* y */ z\";\n")


def test_comments_are_dropped_and_literals_kept():
    code = bench._code_only(SRC)
    assert "remark" not in code and "continued" not in code
    assert "// kept" in code
    assert "\"x /* y */ z\"" in code
    assert "'\"'" in code


def test_comment_edits_keep_the_code_and_code_edits_change_it():
    edited_comment = SRC.replace("remark one", "a longer remark").replace("remark two", "remark 2")
    assert bench._code_only(edited_comment) == bench._code_only(SRC)
    assert bench._code_only(SRC.replace("int a = 1", "int a = 2")) != bench._code_only(SRC)
    assert bench._code_only(SRC.replace("ex2.approx", "ex2.approx.ftz")) != bench._code_only(SRC)

