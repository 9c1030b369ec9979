"""The binding's ctypes structures match include/attn.h field by field (no GPU): a small C
program compiled against the header prints each field's offset and each struct's size."""
import ctypes
import os
import shutil
import subprocess

import pytest

import online_softmax_fa2_gb300 as ofa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def c_layout(tmp_path, struct, fields):
    src = tmp_path / "layout.c"
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "attn.h"', "int main(void) {",
             f'    printf("size %zu\\n", sizeof({struct}));']
    for f in fields:
        lines.append(f'    printf("{f} %zu\\n", offsetof({struct}, {f}));')
    lines += ["    return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([shutil.which("gcc") or "gcc", "-std=c11", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.strip().splitlines())}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("struct,cls", [("attn_fwd_params_t", ofa.Params), ("attn_bwd_params_t", ofa.BwdParams)])
def test_ctypes_mirror_matches_the_header(tmp_path, struct, cls):
    fields = [name for name, _ in cls._fields_]
    got = c_layout(tmp_path, struct, fields)
    assert got["size"] == ctypes.sizeof(cls), (struct, got["size"], ctypes.sizeof(cls))
    for name in fields:
        assert got[name] == getattr(cls, name).offset, (struct, name, got[name], getattr(cls, name).offset)
