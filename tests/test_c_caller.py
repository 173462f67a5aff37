"""The C ABI from C: a small program compiled by gcc against include/tgemm.h
and linked to libtgemm.so.  The compiler's own offsets and sizes of the three
public structs must equal the Python binding's ctypes layouts, and a plan made
from C must equal the same plan made through the binding.  No GPU: tgemm_plan
and tgemm_version never touch the device."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = (("Options", "tgemm_options"), ("PlanInfo", "tgemm_plan_info"), ("Epilogue", "tgemm_epilogue"),
           ("Counters", "tgemm_counters"))


@pytest.fixture(scope="module")
def tg():
    from tests.conftest import build_library
    build_library()
    import tiled_dense_gemm_02_gb300 as lib
    return lib


def program(tg) -> str:
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "tgemm.h"', "int main(void) {"]
    for cls_name, c_name in STRUCTS:
        cls = getattr(tg, cls_name)
        lines.append(f'  printf("size {cls_name} %zu\\n", sizeof({c_name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("offset {cls_name} {field} %zu\\n", offsetof({c_name}, {field}));')
    lines += [
        "  tgemm_options o = {0};",
        "  o.simt_split = 0;",
        "  tgemm_plan_info p;",
        "  int st = tgemm_plan(4096, 4096, 4096, (const void*)0x10000000, 4096, (const void*)0x20000000, 4096,",
        "                      (const void*)0x40000000, 4096, TGEMM_F32, &o, 0, 152, &p);",
        '  printf("plan %d %d %d %d %d %d\\n", st, p.kernel, p.tiles_m, p.tiles_n, p.ctas, p.dp_tiles);',
        "  st = tgemm_plan(4096, 4096, 4096, (const void*)0x10000000, 4096, (const void*)0x20000000, 4096,",
        "                  (const void*)0x40000000, 4096, TGEMM_BF16_F32OUT, NULL, 0, 152, &p);",
        '  printf("plan %d %d %d %d %d %d\\n", st, p.kernel, p.tile_m, p.tile_n, p.ctas, p.swap_ab);',
        '  printf("version %d\\n", tgemm_version());',
        "  return 0;",
        "}",
    ]
    return "\n".join(lines) + "\n"


@pytest.fixture(scope="module")
def c_output(tg, tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    d = tmp_path_factory.mktemp("c_caller")
    src, exe = d / "caller.c", d / "caller"
    src.write_text(program(tg))
    libdir = os.path.join(ROOT, "tiled_dense_gemm_02_gb300")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-ltgemm", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return out.splitlines()


def test_struct_layouts_from_the_compiler(tg, c_output):
    for cls_name, _ in STRUCTS:
        cls = getattr(tg, cls_name)
        assert f"size {cls_name} {ctypes.sizeof(cls)}" in c_output, cls_name
        for field, _ in cls._fields_:
            assert f"offset {cls_name} {field} {getattr(cls, field).offset}" in c_output, (cls_name, field)


def test_plans_from_c_equal_plans_from_python(tg, c_output):
    plans = [line.split()[1:] for line in c_output if line.startswith("plan ")]
    st, p = tg.plan(4096, 4096, 4096, 0x10000000, 4096, 0x20000000, 4096, 0x40000000, 4096, tg.F32,
                    {"simt_split": 0}, sm_count=152)
    assert [int(v) for v in plans[0]] == [st, p.kernel, p.tiles_m, p.tiles_n, p.ctas, p.dp_tiles]
    st, p = tg.plan(4096, 4096, 4096, 0x10000000, 4096, 0x20000000, 4096, 0x40000000, 4096, tg.BF16_F32OUT, None,
                    sm_count=152)
    assert [int(v) for v in plans[1]] == [st, p.kernel, p.tile_m, p.tile_n, p.ctas, p.swap_ab]
    assert f"version {tg.version()}" in c_output
