"""include/ar.h is a plain C header: it compiles as C11, and a C program that
calls every entry point links against libar_gb300.so (compile and link only;
nothing is run, so no GPU is needed)."""
import os
import shutil
import subprocess

import pytest

from all_reduce_reduction_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

C_PROGRAM = r"""
#include "ar.h"
#include <stdio.h>

int main(void) {
    ar_handle_t h = NULL;
    ar_info info;
    ar_plan_t plan = NULL;
    ar_op op = {0};
    const void *in[AR_MAX_RANKS] = {0};
    void *out[AR_MAX_RANKS] = {0};
    float us[4];
    int a = 0, p = 0, t = 0, w = 0, s = 0;
    if (ar_create(8, 4096, AR_BF16, &h) != AR_OK)
        return 1;
    ar_allreduce(h, in, out, AR_ONE_SHOT, AR_LL, 0);
    ar_allreduce_n(h, in, out, 128, AR_ALGO_AUTO, AR_PROTO_AUTO, 0);
    ar_reduce_scatter(h, in, out, 0);
    ar_all_gather(h, out, 0);
    ar_ll_pack(h, in[0], (uint64_t *)out[0], 16, 7u, 0);
    ar_ll_unpack(h, (const uint64_t *)in[0], out[0], 16, 7u, 0);
    ar_combine(h, in, (const float *)in[0], out[0], 1, 16, 0);
    ar_tune(h, 0);
    ar_get_tuning(h, 4096, &a, &p, us);
    ar_set_timeout(h, 0);
    ar_set_pdl(h, 1);
    ar_set_ll_transport(h, AR_LL_AUTO);
    ar_set_hb_staging(h, AR_HB_STAGING_AUTO);
    ar_get_hb_staging(h, 4096, &a);
    ar_set_grid_divisor(h, 0);
    ar_get_grid_divisor(h, 4096, AR_TWO_SHOT, AR_HB, &a);
    ar_debug_drop_rank(h, -1);
    ar_round(AR_FP16, (const float *)in[0], out[0], 1, 0);
    ar_get_info(h, &info);
    ar_plan_compile(h, &op, 1, 1, 0, &plan);
    ar_plan_builtin(h, AR_TWO_SHOT, 0, 0, &plan);
    ar_plan_execute(plan, in, out, 0);
    ar_plan_stats(plan, &t, &w, &s);
    ar_plan_destroy(plan);
    ar_allreduce_ll_static(8, 4096, AR_BF16, in, out, 0);
    printf("%s %d\n", ar_strerror(ar_status(h, 0)), info.R);
    return ar_destroy(h);
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_is_c11_and_every_entry_point_links(tmp_path):
    lib = cuda_build.build()
    src = tmp_path / "use_ar.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_ar"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I" + os.path.join(ROOT, "include"), "-I" + CUDA_INC, str(src), "-o", str(exe),
           "-L" + os.path.dirname(lib), "-lar_gb300", "-Wl,-rpath," + os.path.dirname(lib)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


@pytest.mark.skipif(shutil.which("g++") is None, reason="no C++ compiler")
def test_header_is_usable_from_cpp17(tmp_path):
    """The same header from C++ (its extern "C" block): a C++17 program
    calling a few entry points compiles and links without name mangling."""
    lib = cuda_build.build()
    src = tmp_path / "use_ar.cpp"
    src.write_text(r'''
#include "ar.h"
#include <cstdio>
int main() {
    ar_handle_t h = nullptr;
    if (ar_create(8, 4096, AR_BF16, &h) != AR_OK)
        return 1;
    ar_info info{};
    ar_get_info(h, &info);
    std::printf("%s %d\n", ar_strerror(ar_status(h, nullptr)), info.R);
    return ar_destroy(h);
}
''')
    exe = tmp_path / "use_ar_cpp"
    cmd = ["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I" + os.path.join(ROOT, "include"), "-I" + CUDA_INC, str(src), "-o", str(exe),
           "-L" + os.path.dirname(lib), "-lar_gb300", "-Wl,-rpath," + os.path.dirname(lib)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def _layout_program():
    from all_reduce_reduction_gb300 import ar_info, ar_op
    lines = ['#include "ar.h"', "#include <stddef.h>", "#include <stdio.h>", "int main(void) {"]
    for cls in (ar_info, ar_op):
        name = cls.__name__
        lines.append('    printf("%s size %%zu\\n", sizeof(%s));' % (name, name))
        for field, _ in cls._fields_:
            lines.append('    printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (name, field, name, field))
    lines += ["    return 0;", "}"]
    return "\n".join(lines) + "\n"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_binding_structs_match_the_header_layout(tmp_path):
    """Every field of the ctypes ar_info and ar_op sits at the offset the C
    compiler gives it from include/ar.h, and the sizes agree (a field added
    to one side only, or declared with another width, fails here)."""
    import ctypes
    from all_reduce_reduction_gb300 import ar_info, ar_op
    src = tmp_path / "layout.c"
    src.write_text(_layout_program())
    exe = tmp_path / "layout"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
           "-I" + CUDA_INC, str(src), "-o", str(exe)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(line.rsplit(" ", 1) for line in out if line)
    for cls in (ar_info, ar_op):
        name = cls.__name__
        assert int(got.pop("%s size" % name)) == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert int(got.pop("%s.%s" % (name, field))) == getattr(cls, field).offset, (name, field)
    assert not got
    # and the header declares exactly the binding's fields, in order
    import re
    header = open(os.path.join(ROOT, "include", "ar.h")).read()
    header = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    for cls in (ar_info, ar_op):
        body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (cls.__name__, cls.__name__),
                         header, re.S).group(1)
        names = []
        for decl in body.split(";"):
            decl = re.sub(r"\[[^\]]*\]", "", decl).strip()
            if decl:
                names += [part.split()[-1] for part in decl.split(",")]
        assert names == [f for f, _ in cls._fields_], cls.__name__
