"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import exact_bf16_top_gb300 as tk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "topk_bf16.h")


@pytest.fixture(scope="module")
def lib():
    tk._build.build()
    return tk.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(topk_bf16_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("topk_bf16_select", "topk_bf16_status_string", "topk_bf16_select_ex",
              "topk_bf16_plan", "topk_bf16_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", tk.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(topk_bf16_\w+)\b", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "topk_bf16.h"\nint main(void){return (int)TOPK_OK;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                    "-c", str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_options_struct_layout_matches_the_header(tmp_path):
    # The binding's ctypes mirror of topk_bf16_options_t must agree with the C
    # compiler on its size and on every field's offset.
    fields = [f for f, _ in tk._Options._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "topk_bf16.h"\n'
                   'int main(void){printf("%zu", sizeof(topk_bf16_options_t));'
                   + "".join('printf(" %%zu", offsetof(topk_bf16_options_t, %s));' % f for f in fields)
                   + 'return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                    "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(tk._Options)
    assert got[1:] == [getattr(tk._Options, f).offset for f in fields]
    assert "hold" in fields


def test_status_strings(lib):
    for s in range(7):
        assert tk.status_string(s)


def _call(lib, logits=16, stride=8, rows=1, width=8, valid=16, k=1, mode=0, table=None,
          table_stride=0, page=64, out=16):
    return lib.topk_bf16_select(logits, stride, rows, width, valid, k, mode, table, table_stride,
                                page, out, None)


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), 3), (dict(k=2049), 3), (dict(rows=-1), 1), (dict(mode=2), 1),
    (dict(width=(1 << 20) + 8, stride=(1 << 20) + 8), 4), (dict(width=16, stride=8), 4),
    (dict(width=-1), 4), (dict(logits=None), 1), (dict(valid=None), 1), (dict(out=None), 1),
    (dict(logits=18), 2), (dict(stride=12, width=8), 2), (dict(out=18), 2),
    (dict(table=16, page=48, table_stride=1), 1), (dict(table=16, page=0, table_stride=1), 1),
    (dict(table=16, page=4, table_stride=1), 1),
])
def test_bad_arguments_rejected_on_host(lib, kw, status):
    assert _call(lib, **kw) == status


def test_zero_rows_is_a_no_op(lib):
    assert _call(lib, rows=0, logits=None, valid=None, out=None) == 0


def _ordered(lib, logits=16, stride=8, rows=1, width=8, valid_len=16, k=1, tops=16, tops_stride=8,
             table=None, table_stride=0, page=64, block_rows=64, q=1, out=16, valid=16, ids=None):
    return lib.topk_bf16_select_ordered(logits, stride, rows, width, valid_len, k, tops, tops_stride,
                                        table, table_stride, page, block_rows, q, out, valid, ids,
                                        None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), 3), (dict(valid=None), 1), (dict(valid=18), 2), (dict(ids=18), 2),
    (dict(tops=24), 2), (dict(tops_stride=12), 2), (dict(tops_stride=0), 1), (dict(q=0), 1),
    (dict(table=16, table_stride=1, block_rows=32), 1), (dict(table=16, table_stride=1, block_rows=96), 1),
    (dict(width=(1 << 20) + 8, stride=(1 << 20) + 8, tops_stride=1 << 17), 4),
])
def test_ordered_bad_arguments_rejected_on_host(lib, kw, status):
    assert _ordered(lib, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(n=33), 1), (dict(n=0), 3), (dict(n=4096), 3), (dict(width=(1 << 17) + 8, stride=(1 << 17) + 8,
                                                              tops_stride=(1 << 14) + 8), 1),
    (dict(valid=None), 1), (dict(tops=20), 2),
])
def test_words_bad_arguments_rejected_on_host(lib, kw, status):
    a = dict(logits=16, stride=8, rows=1, width=8, valid_len=16, n=32, tops=16, tops_stride=8, out=16,
             valid=16)
    a.update(kw)
    assert lib.topk_bf16_select_words(a["logits"], a["stride"], a["rows"], a["width"], a["valid_len"],
                                      a["n"], a["tops"], a["tops_stride"], a["out"], a["valid"],
                                      None, None) == status


def test_tops_bad_arguments_rejected_on_host(lib):
    assert lib.topk_bf16_tops(16, 8, 1, 8, 16, 24, 8, None) == 2    # misaligned tops
    assert lib.topk_bf16_tops(16, 8, 1, 8, 16, 16, 4, None) == 2    # stride not a multiple of 8
    assert lib.topk_bf16_tops(16, 8, 1, 80, 16, 16, 8, None) == 4   # width above the row stride
    assert lib.topk_bf16_tops(16, 8, 0, 8, 16, 16, 8, None) == 0    # no rows: nothing to do
