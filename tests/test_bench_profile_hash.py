"""The bench reports ncu's DRAM traffic only while the committed profile was
taken on the current kernel code: the hash over the kernel sources ignores
comments and white space, and changes with any code token."""
import os
import shutil

import bench


def _hash_of(tmp_path, edit=None):
    d = tmp_path / "csrc"
    if not d.exists():
        d.mkdir()
        for f in bench.KERNEL_SOURCES:
            shutil.copy(os.path.join(bench.CSRC, f), d / f)
    if edit:
        f, old, new = edit
        text = (d / f).read_text()
        assert old in text
        (d / f).write_text(text.replace(old, new, 1))
    saved = bench.CSRC
    bench.CSRC = str(d)
    try:
        return bench.kernel_source_hash()
    finally:
        bench.CSRC = saved


def test_comment_and_whitespace_edits_keep_the_hash(tmp_path):
    h0 = _hash_of(tmp_path)
    assert h0 == bench.kernel_source_hash()
    h1 = _hash_of(tmp_path, ("dflash_sweep.cu", "// ---- the kernel", "// ---- the  kernel, reworded"))
    h2 = _hash_of(tmp_path, ("dflash_internal.h", "constexpr int kStages = 12;", "constexpr int   kStages = 12; /* ring */"))
    assert h0 == h1 == h2


def test_code_edits_change_the_hash(tmp_path):
    h0 = _hash_of(tmp_path)
    h1 = _hash_of(tmp_path, ("dflash_internal.h", "constexpr int kStages = 12;", "constexpr int kStages = 16;"))
    assert h0 != h1
