"""The ctypes mirrors of the C ABI's argument structs (speculative_decoding_draft_04_gb300/_lib.py)
have the layout of the structs in include/spec.h: every field at the C compiler's
offset and every struct of the C size.  A small C program built with the host
compiler prints offsetof / sizeof for each field the binding names (a name the
header does not have fails the build)."""
import ctypes
import os
import shutil
import subprocess

import pytest

from speculative_decoding_draft_04_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MIRRORS = {
    "spec_draft_args": _lib.DraftArgs,
    "spec_verify_args": _lib.VerifyArgs,
    "spec_cycle_host_args": _lib.CycleHostArgs,
    "spec_rnn_draft_args": _lib.RnnDraftArgs,
    "spec_confidence_args": _lib.ConfidenceArgs,
    "spec_schedule_args": _lib.ScheduleArgs,
    "spec_tree_draft_args": _lib.TreeDraftArgs,
    "spec_tree_verify_args": _lib.TreeVerifyArgs,
    "spec_op_args": _lib.OpArgs,
    "spec_op_result": _lib.OpResult,
}


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "spec.h"', "int main(void) {"]
    for cname, py in MIRRORS.items():
        lines.append(f'  printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'  printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    d = tmp_path_factory.mktemp("abi_layout")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        struct, field, value = line.split()
        table[(struct, field)] = int(value)
    return table


@pytest.mark.parametrize("cname", list(MIRRORS))
def test_struct_layout_matches_the_header(c_layout, cname):
    py = MIRRORS[cname]
    assert ctypes.sizeof(py) == c_layout[(cname, "sizeof")], cname
    for f, _ in py._fields_:
        assert getattr(py, f).offset == c_layout[(cname, f)], (cname, f)
