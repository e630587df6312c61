"""The source hash that ties a committed ncu summary to the kernel it was
taken from: comments may change, code may not."""
from tiled_mma_atom_gb300 import build


def test_code_only_strips_comments_and_blank_lines():
    src = ("// header\n"
           "int a = 1;   // trailing\n"
           "\n"
           "/* block\n comment */ int b = 2;\n"
           "asm(\"mov.u32 %0, 1;\");  // after a string\n")
    assert build._code_only(src) == 'int a = 1;\n int b = 2;\nasm("mov.u32 %0, 1;");'


def test_comment_edits_keep_the_hash_code_edits_change_it(tmp_path, monkeypatch):
    monkeypatch.setattr(build, "CSRC", str(tmp_path))
    (tmp_path / "device.cuh").write_text("// shared\nint shared_helper();\n")
    k = tmp_path / "k.cu"
    k.write_text("// kernel\n__global__ void k() { int x = 1; }\n")
    h0 = build.source_hash("k.cu")
    k.write_text("// kernel, reworded comment\n__global__ void k() { int x = 1; }  // note\n")
    assert build.source_hash("k.cu") == h0
    k.write_text("// kernel\n__global__ void k() { int x = 2; }\n")
    assert build.source_hash("k.cu") != h0
    (tmp_path / "device.cuh").write_text("// shared\nint shared_helper(int);\n")
    k.write_text("// kernel\n__global__ void k() { int x = 1; }\n")
    assert build.source_hash("k.cu") != h0
