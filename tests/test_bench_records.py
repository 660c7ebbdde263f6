"""The bench's use of the committed ncu traffic record (CPU only): the record is
keyed to the code of the round's sources, comments and blank space left out."""
import json
import os

import bench


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1;  // count\n/* a block\n   comment */ const char* s = "// kept";\n'
           "char q = '\"'; int b = a / 2; /**/ int c = 3;\n")
    assert bench._code_only(src) == ('int a = 1; const char* s = "// kept"; '
                                     "char q = '\"'; int b = a / 2; int c = 3;")


def test_a_comment_edit_keeps_the_hash_and_a_code_edit_changes_it():
    base = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    comment = "int f(int x) {\n  // the next integer\n  return x + 1;\n}\n"
    code = "int f(int x) {\n  return x + 2;  // one more\n}\n"
    assert bench._code_only(base) == bench._code_only(comment)
    assert bench._code_only(base) != bench._code_only(code)


def test_committed_record_names_its_sources_and_command():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    ent = rec["w4_v262144_bf16"]
    assert ent["source_files"] == list(bench.ROUND_SOURCES)
    assert ent["command"].startswith("ncu ") and "--clock-control none" in ent["command"]
    assert ent["dram_bytes_per_launch"] > 0
