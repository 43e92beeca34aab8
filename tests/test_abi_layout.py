"""The Python binding's ctypes structures have the C header's layout (CPU
only): a small C program compiled against include/lf.h prints every field's
offset and every struct's size, which must equal ctypes' view."""
import os
import shutil
import subprocess
import tempfile

import pytest

from conftest import ROOT

STRUCTS = ("lf_config", "lf_weights", "lf_sampling", "lf_info")


@pytest.fixture(scope="module")
def pm():
    import persistent_monokernel_gb300 as pm
    return pm


def _c_layout(pm):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include "lf.h"', "int main(void) {"]
    for st in STRUCTS:
        lines.append(f'printf("{st} size %zu\\n", sizeof({st}));')
        for name, _ in getattr(pm, st)._fields_:
            lines.append(f'printf("{st} {name} %zu\\n", offsetof({st}, {name}));')
    lines += ["return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(src, "w") as f:
            f.write("\n".join(lines))
        subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True,
                       capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    layout = {}
    for line in out.splitlines():
        st, name, val = line.split()
        layout[(st, name)] = int(val)
    return layout


def test_ctypes_structures_match_the_c_header(pm):
    layout = _c_layout(pm)
    for st in STRUCTS:
        cls = getattr(pm, st)
        assert layout[(st, "size")] == __import__("ctypes").sizeof(cls), st
        for name, _ in cls._fields_:
            assert layout[(st, name)] == getattr(cls, name).offset, (st, name)
