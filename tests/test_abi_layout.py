"""The ctypes mirrors in the binding match the C structs of include/cf.h
(size and every field offset), checked by compiling a small C program with
the host compiler against the header (CPU only)."""
import ctypes
import json
import os
import shutil
import subprocess

import pytest

from back_gemm_fusion_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = {
    "cf_matrix": B.cf_matrix,
    "cf_op": B.cf_op,
    "cf_epi_desc": B.cf_epi_desc,
    "cf_b2b_desc": B.cf_b2b_desc,
    "cf_device_model": B.cf_device_model,
    "cf_cost": B.cf_cost,
}


def test_struct_layouts_match(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "cf.h"', "int main(void) {", 'printf("{");']
    first = True
    for name, cls in STRUCTS.items():
        for field, _ in cls._fields_:
            sep = "" if first else ","
            first = False
            lines.append(f'printf("{sep}\\"{name}.{field}\\": %zu", offsetof({name}, {field}));')
        lines.append(f'printf(",\\"{name}\\": %zu", sizeof({name}));')
    lines += ['printf("}\\n");', "return 0; }"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    c = json.loads(subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout)
    for name, cls in STRUCTS.items():
        assert c[name] == ctypes.sizeof(cls), (name, c[name], ctypes.sizeof(cls))
        for field, _ in cls._fields_:
            assert c[f"{name}.{field}"] == getattr(cls, field).offset, (name, field)
