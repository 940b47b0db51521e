"""The source hash that ties a committed ncu summary to the kernel sources:
comments and blank lines do not change it, code does."""
import bench


def _sources():
    import os
    out = {}
    for name in bench.KERNEL_SOURCES:
        with open(os.path.join(bench.ROOT, "smem_swizzle_layouts_gb300", "csrc", name)) as f:
            out[name] = f.read()
    return out


def test_comments_and_blank_lines_leave_the_hash_alone():
    src = _sources()
    base = bench._source_hash(lambda n: src[n])
    assert base == bench._source_hash()
    name = bench.KERNEL_SOURCES[0]
    edited = dict(src)
    edited[name] = "// a new comment line\n\n" + src[name].replace("\n", "   // trailing note\n", 3)
    assert bench._source_hash(lambda n: edited[n]) == base


def test_a_code_change_changes_the_hash():
    src = _sources()
    base = bench._source_hash(lambda n: src[n])
    name = bench.KERNEL_SOURCES[1]
    edited = dict(src)
    edited[name] = src[name] + "\nstatic_assert(true, \"\");\n"
    assert bench._source_hash(lambda n: edited[n]) != base


def test_code_lines_strip_only_comments():
    text = "int a = 1; // one\n\n   // whole-line comment\nint b = 2;\n"
    assert bench._code_lines(text) == "int a = 1;\nint b = 2;"
