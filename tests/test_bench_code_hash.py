"""bench.py keys its ncu traffic figures to a hash of each kernel file's code:
comments and blank lines do not count, everything else does."""

import bench


def test_comments_and_blank_lines_do_not_count():
    a = "int x = 1;  // one\n\n/* block\n comment */ float y;\n"
    b = "   int x = 1;\nfloat y;   // other words\n"
    assert bench.code_text(a) == bench.code_text(b) == "int x = 1;\nfloat y;"


def test_comment_markers_inside_literals_are_code():
    src = 'const char *p = "a // b /* c */";\nchar q = \'/\';  // d\n'
    assert bench.code_text(src) == 'const char *p = "a // b /* c */";\nchar q = \'/\';'


def test_code_changes_change_the_hash():
    assert bench.code_text("x = 1;") != bench.code_text("x = 2;")
