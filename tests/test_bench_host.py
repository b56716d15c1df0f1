"""Host logic of bench.py that needs no GPU: the code-only source hash that
ties a committed ncu traffic figure to the kernel it was measured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_keeps_strings():
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "x // y /* z */";\n  int   b;\n'
    assert bench.code_only(src) == 'int a = 1; const char* s = "x // y /* z */"; int b;'


def test_comment_edits_keep_the_hash_and_code_edits_change_it():
    base = "__global__ void k(int* p) {\n  // one\n  p[0] = 1;  /* two */\n}\n"
    recommented = "__global__ void k(int* p) {\n  // a different note\n  p[0] = 1;\n}\n"
    changed = "__global__ void k(int* p) {\n  // one\n  p[0] = 2;  /* two */\n}\n"
    assert bench.code_only(base) == bench.code_only(recommented)
    assert bench.code_only(base) != bench.code_only(changed)

