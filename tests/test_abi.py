"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, sizes workspaces, and rejects invalid calls on the host before any
launch (only argument combinations that fail validation are passed here)."""
import ctypes
import os
import re

import pytest

from sparse_mixture_experts_71_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    lib = B.load()
    declared = _declared()
    assert {"moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(B.EXPORTED) == declared


def test_status_strings():
    lib = B.load()
    for code, text in B.STATUS.items():
        assert lib.moe_status_string(code).decode() == text


def test_workspace_size():
    c = B.config(4096, 1024, 4096, 8, 2)
    n = B.workspace_size(c)
    # at least the permuted rows, the hidden activations and the fp32 expert outputs
    assert n >= 8192 * (1024 * 2 + 4096 * 2 + 1024 * 4)
    assert n % 256 == 0
    capped = B.workspace_size(B.config(4096, 1024, 4096, 8, 2, capacity=100))
    assert capped < n
    assert B.workspace_size(B.config(4096, 1024, 4096, 8, 9)) == 0  # k > E
    assert B.workspace_size(B.config(0, 64, 64, 4, 2)) > 0
    # shared experts: K = k + n_shared assignments per token
    assert B.workspace_size(B.config(4096, 1024, 4096, 9, 2, n_shared=1)) > \
        B.workspace_size(B.config(4096, 1024, 4096, 9, 2))


FAKE = 1 << 20  # a 256-aligned address that is never dereferenced (calls fail first)


@pytest.mark.parametrize("cfg,status", [
    (None, 1),
    (B.config(16, 64, 64, 4, 5), 1),            # k > E
    (B.config(16, 64, 64, 300, 2), 4),          # E > 256
    (B.config(16, 64, 64, 16, 9), 4),           # k > 8
    (B.config(16, 60, 64, 4, 2), 2),            # d not a multiple of 8
    (B.config(16, 64, 68, 4, 2), 2),            # d_ff not a multiple of 8
    (B.config(-1, 64, 64, 4, 2), 1),            # T < 0
    (B.config(16, 64, 64, 4, 1, n_shared=4), 1),   # every expert shared
    (B.config(16, 64, 64, 4, 2, n_shared=3), 1),   # k > routed experts
    (B.config(16, 64, 64, 16, 6, n_shared=3), 4),  # k + n_shared > 8
    (B.config(16, 64, 64, 4, 1, n_shared=-1), 1),  # n_shared < 0
])
def test_forward_rejects_bad_config(cfg, status):
    lib = B.load()
    ref = ctypes.byref(cfg) if cfg is not None else None
    st = lib.moe_forward(ref, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                         None, FAKE, 1 << 40, None)
    assert st == status


def test_calls_reject_null_misaligned_and_small_workspace():
    lib = B.load()
    c = B.config(16, 64, 64, 4, 2)
    cr = ctypes.byref(c)
    need = B.workspace_size(c)
    # null required pointer
    assert lib.moe_forward(cr, None, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                           None, FAKE, need, None) == 1
    # misaligned x
    assert lib.moe_forward(cr, FAKE + 8, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                           None, None, FAKE, need, None) == 2
    # workspace too small / misaligned
    assert lib.moe_forward(cr, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                           None, FAKE, need - 1, None) == 3
    assert lib.moe_forward(cr, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                           None, FAKE + 16, need, None) == 3
    assert lib.moe_route(cr, FAKE, FAKE, None, None, None, None, None, FAKE, None, None, None, FAKE,
                         need, None) == 1
    assert lib.moe_dispatch(cr, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need,
                            None) == 1  # perm_w without topk_w
    assert lib.moe_expert_ffn(cr, FAKE, FAKE, FAKE, FAKE, FAKE + 4, FAKE, None, FAKE, FAKE, need,
                              None) == 2
    assert lib.moe_combine(cr, FAKE, None, FAKE, None) == 1
    assert lib.moe_get_device_error(None, None, None, None) == 1
    assert lib.moe_check_wait_timeout(None, ctypes.c_uint64(1000), None) == 1
    assert lib.moe_update_balance_bias(cr, None, FAKE, ctypes.c_float(0.1), None) == 1
    assert lib.moe_check_wait_timeout(FAKE + 16, ctypes.c_uint64(1000), None) == 3
    # the segment-map check: no workspace, a misaligned one, one below 3 MiB
    assert lib.moe_check_segment_maps(None, 3 << 20, None) == 3
    assert lib.moe_check_segment_maps(FAKE + 16, 3 << 20, None) == 3
    assert lib.moe_check_segment_maps(FAKE, (3 << 20) - 1, None) == 3


def test_pipeline_workspace_and_host_rejections():
    lib = B.load()
    c = B.config(64, 64, 128, 4, 2)
    one, two = B.pipeline_workspace_size(c, 1), B.pipeline_workspace_size(c, 2)
    tile = 64 * 64 * 2
    # the forward workspace plus per slot x, y (bf16 [T][d]) and the loss
    assert one >= B.workspace_size(c) + 2 * tile and one % 256 == 0
    assert two - one >= 2 * tile
    assert B.pipeline_workspace_size(c, 0) == 0 and B.pipeline_workspace_size(c, 5) == 0
    assert B.pipeline_workspace_size(B.config(0, 64, 128, 4, 2), 2) == 0  # T = 0
    assert B.pipeline_workspace_size(B.config(64, 64, 128, 4, 5), 2) == 0  # k > E
    cr = ctypes.byref(c)
    h = ctypes.c_void_p()
    out = ctypes.byref(h)
    args = (FAKE, None, FAKE, FAKE, FAKE, FAKE)  # W_r, logit_bias, W1, b1, W2, b2
    assert lib.moe_pipeline_create(cr, 2, *args, FAKE, two, None, None) == 1  # no out
    assert lib.moe_pipeline_create(None, 2, *args, FAKE, two, None, out) == 1
    assert lib.moe_pipeline_create(ctypes.byref(B.config(64, 64, 128, 300, 2)), 2, *args, FAKE,
                                   1 << 40, None, out) == 4
    assert lib.moe_pipeline_create(cr, 0, *args, FAKE, two, None, out) == 1  # depth
    assert lib.moe_pipeline_create(cr, 2, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, two, None,
                                   out) == 1  # W1 missing
    assert lib.moe_pipeline_create(cr, 2, FAKE, None, FAKE + 8, FAKE, FAKE, FAKE, FAKE, two,
                                   None, out) == 2
    assert lib.moe_pipeline_create(cr, 2, *args, FAKE, two - 1, None, out) == 3
    assert lib.moe_pipeline_create(cr, 2, *args, FAKE + 16, two, None, out) == 3
    assert h.value is None
    assert lib.moe_pipeline_submit(None, FAKE, FAKE, None) == 1
    assert lib.moe_pipeline_join(None) == 1
    assert lib.moe_pipeline_destroy(None) == 0


def test_expert_choice_host_side():
    lib = B.load()
    ec = B.config(4096, 1024, 4096, 8, 2, routing="expert")
    assert B.expert_choice_capacity(ec) == 1024                                   # ceil(T k / E)
    assert B.expert_choice_capacity(B.config(10, 64, 64, 3, 1, routing="expert")) == 4
    assert B.expert_choice_capacity(B.config(10, 64, 64, 3, 1, capacity=50, routing="expert")) == 10
    assert B.expert_choice_capacity(B.config(10, 64, 64, 3, 1, capacity=0, routing="expert")) == 0
    assert B.expert_choice_capacity(B.config(10, 64, 64, 3, 9, routing="expert")) == -1
    # E*C permuted rows, a [T][E] slot map and the [E][T] probabilities
    assert B.workspace_size(ec) >= 8 * 1024 * (1024 * 2 + 4096 * 2 + 1024 * 4) + 2 * 4096 * 8 * 4
    bad = B.config(16, 64, 64, 4, 2)
    bad.routing = 2
    assert B.workspace_size(bad) == 0
    cr = ctypes.byref(B.config(16, 64, 64, 4, 2, routing="expert"))
    need = B.workspace_size(B.config(16, 64, 64, 4, 2, routing="expert"))
    # the token-choice steps refuse an expert-choice layer, and the reverse
    assert lib.moe_route(cr, FAKE, FAKE, None, None, None, None, FAKE, FAKE, None, None, None, FAKE,
                         need, None) == 4
    assert lib.moe_dispatch(cr, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, FAKE, need,
                            None) == 4
    assert lib.moe_dispatch_noalloc(cr, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, None) == 4
    tc = ctypes.byref(B.config(16, 64, 64, 4, 2))
    args = (FAKE, FAKE, None, None, None, None, FAKE, FAKE, FAKE, FAKE, None, None, None)
    assert lib.moe_route_expert_choice(tc, *args, FAKE, need, None) == 1
    assert lib.moe_route_expert_choice(cr, *args, FAKE, need - 1, None) == 3
    assert lib.moe_route_expert_choice(cr, FAKE, FAKE, None, None, None, None, FAKE, None, FAKE,
                                       FAKE, None, None, None, FAKE, need, None) == 1
    # shared experts are not combined with expert choice
    sh = ctypes.byref(B.config(16, 64, 64, 4, 1, n_shared=1, routing="expert"))
    assert lib.moe_forward(sh, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                           None, None, FAKE, 1 << 40, None) == 4


def test_backward_host_side():
    lib = B.load()
    c = B.config(64, 64, 128, 4, 2)
    n = lib.moe_backward_workspace_size(ctypes.byref(c))
    assert n >= B.workspace_size(c) and n % 256 == 0
    # every variant of both dtypes has a backward pass
    for ok in (B.config(64, 64, 128, 4, 2, routing="expert"), B.config(64, 64, 128, 4, 1, n_shared=1),
               B.config(64, 64, 128, 4, 2, capacity=5, overflow="reroute"),
               B.config(64, 64, 128, 4, 2, dtype="f32"),
               B.config(64, 64, 128, 4, 2, dtype="f32", routing="expert")):
        assert lib.moe_backward_workspace_size(ctypes.byref(ok)) >= B.workspace_size(ok)
    # fp32 token rows take twice the bytes of bf16 ones (the bf16 layout adds
    # only the tensor maps and the slot-score partials)
    f32 = B.config(64, 64, 128, 4, 2, dtype="f32")
    assert lib.moe_backward_workspace_size(ctypes.byref(f32)) - B.workspace_size(f32) < \
        n - B.workspace_size(c) + 3 * 128 * 128 * 2
    bad = B.config(64, 64, 128, 300, 2)  # E > 256: unsupported configuration
    assert lib.moe_backward_workspace_size(ctypes.byref(bad)) == 0
    assert lib.moe_backward(ctypes.byref(bad), *([FAKE] * 8), ctypes.c_float(0),
                            ctypes.c_float(0), *([FAKE] * 6), FAKE, 1 << 40, None) == 4
    cr = ctypes.byref(c)
    args = [FAKE] * 8
    outs = [FAKE] * 6  # dx, dW_r, dW1, db1, dW2, db2
    assert lib.moe_backward(cr, *args, ctypes.c_float(0), ctypes.c_float(0), *outs, FAKE, n - 1,
                            None) == 3
    assert lib.moe_backward(cr, *args[:7], None, ctypes.c_float(0), ctypes.c_float(0), *outs, FAKE,
                            n, None) == 1  # no dy
    assert lib.moe_backward(cr, FAKE + 8, *args[1:], ctypes.c_float(0), ctypes.c_float(0), *outs,
                            FAKE, n, None) == 2


@pytest.mark.parametrize("header", sorted(h for h in os.listdir(os.path.join(ROOT, "include"))
                                          if h.endswith(".h")))
def test_header_is_plain_c(header, tmp_path):
    """Each public header compiles on its own as C99 (a C ABI, no C++ or torch
    types), warnings as errors."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "t.c"
    src.write_text(f'#include "{header}"\nint main(void) {{ return 0; }}\n')
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-fsyntax-only", "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_product_path_never_imports_the_oracle():
    """The oracle is test infrastructure: nothing in the package imports it."""
    pkg = os.path.join(ROOT, "sparse_mixture_experts_71_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith(".py"):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, re.M), fn


C_PROGRAM = r"""
#include <stdio.h>
#include "moe.h"
#include "moe_pipeline.h"
#include "moe_backward.h"
int main(void) {
    moe_config c = {4096, 1024, 4096, 8, 2, MOE_BF16, -1, 1, 0, MOE_TOKEN_CHOICE, MOE_DROP};
    size_t ws = moe_workspace_size(&c);
    size_t wb = moe_backward_workspace_size(&c);
    size_t wp = moe_pipeline_workspace_size(&c, 2);
    c.routing = MOE_EXPERT_CHOICE;
    int C = moe_expert_choice_capacity(&c);
    moe_status bad = moe_forward(&c, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);
    printf("%zu %zu %zu %d %d %s\n", ws, wb, wp, C, (int)bad, moe_status_string(bad));
    return (ws > 0 && wb > ws && wp > ws && C == 1024 && bad == MOE_ERR_INVALID_ARG) ? 0 : 1;
}
"""


def test_c_program_links_and_calls_the_library(tmp_path):
    """A plain C99 program builds against the headers, links libmoe.so and
    calls its host-side entry points (no GPU needed for these)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    B.load()  # the library is built
    libdir = os.path.join(ROOT, "sparse_mixture_experts_71_b300")
    src, exe = tmp_path / "t.c", tmp_path / "t"
    src.write_text(C_PROGRAM)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lmoe", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split()[3] == "1024"
