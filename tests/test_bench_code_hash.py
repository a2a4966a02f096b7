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


def _profile_hashes():
    """(kernel file, code hash) pairs the committed ncu summaries name."""
    import os
    import re
    root = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
    pairs = set()
    for name in os.listdir(root):
        if name.endswith(".md"):
            text = open(os.path.join(root, name), encoding="utf-8").read()
            pairs |= set(re.findall(r"([a-z_0-9]+\.cu) code sha256\s+([0-9a-f]{12})", text))
    return pairs


def test_traffic_figures_and_profiles_name_the_same_captures():
    """Every traffic figure the bench reports comes from a capture that a
    committed summary describes, and the summaries agree on each file's code."""
    pairs = _profile_hashes()
    by_file = {}
    for f, h in pairs:
        by_file.setdefault(f, set()).add(h)
    assert all(len(hs) == 1 for hs in by_file.values()), by_file
    named = {h for _, h in pairs}
    for workload, t in bench.TRAFFIC.items():
        assert t["source"] in named, workload


def test_every_default_workload_has_current_traffic():
    """The committed traffic figures match the kernel files as they stand, so
    that the default run reports a traffic figure for every workload it
    measures (a kernel edit without a new capture would show up as null)."""
    for workload in [bench.DEFAULT_WORKLOAD] + list(bench.DEFAULT_PATHS):
        t = bench.TRAFFIC.get(workload)
        assert t is not None, workload
        current = {bench.file_hash(f) for f in set(bench.KERNEL_SOURCE.values())}
        if "file" in t:
            current = {bench.file_hash(t["file"])}
        assert t["source"] in current, workload
