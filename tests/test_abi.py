"""The C-ABI library loads and exports every entry point include/lcgemm.h declares (CPU only)."""
import ctypes
import os
import re

import pytest

import complexity_matmul_gb300 as lcg
from complexity_matmul_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"LCGEMM_API\s+[\w\s\*]*?\b(lcgemm_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def library():
    _build.build()
    return lcg.lib()


def test_library_exports_all_declared_symbols(library):
    declared = _declared()
    assert {"lcgemm_create", "lcgemm_run", "lcgemm_destroy"} <= declared
    missing = [n for n in sorted(declared) if not hasattr(library, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(lcg.EXPORTS) <= declared


def test_strerror_is_static_and_total(library):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 12345):
        s = library.lcgemm_strerror(code)
        assert isinstance(s, bytes) and s
    assert b"aligned" in library.lcgemm_strerror(-2)


def test_null_handle_rejected_without_gpu(library):
    assert library.lcgemm_run(None, 8, 8, 8, None, 8, None, 8, None, 8, 1, 0, None) == lcg.ERR_ARG
    assert library.lcgemm_set_option(None, 1, 5) == lcg.ERR_ARG
    assert library.lcgemm_last_algo(None) == lcg.ERR_ARG
    assert library.lcgemm_destroy(None) == lcg.OK
    assert library.lcgemm_create(None, 0) == lcg.ERR_ARG


def test_create_fails_cleanly_without_device(library):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    assert library.lcgemm_create(ctypes.byref(h), 0) == lcg.ERR_ARG
    assert not h.value


def test_product_path_does_not_touch_the_oracle():
    """The package never imports, links or executes anything under oracle/."""
    pkg = os.path.join(ROOT, "complexity_matmul_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.lower(), fn


def test_epilogue_struct_layout_matches_header(tmp_path):
    """The binding's ctypes mirror of lcgemm_epilogue has the C compiler's size and offsets."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "lcgemm.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu\\n", sizeof(lcgemm_epilogue),'
                   ' offsetof(lcgemm_epilogue, bias), offsetof(lcgemm_epilogue, residual),'
                   ' offsetof(lcgemm_epilogue, ldr), offsetof(lcgemm_epilogue, act)); return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    E = lcg.Epilogue
    assert got == [ctypes.sizeof(E), E.bias.offset, E.residual.offset, E.ldr.offset, E.act.offset]


def test_epilogue_entry_rejects_planning_and_null_handles(library):
    ep = lcg.Epilogue(None, None, 0, lcg.ACT_RELU)
    assert library.lcgemm_run_epilogue(None, 8, 8, 8, None, 8, None, 8, None, 8, 1, 0, ctypes.byref(ep),
                                       None) == lcg.ERR_ARG
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    assert h.run_epilogue_raw(8, 8, 8, None, 8, None, 8, None, 8, lcg.BF16, lcg.PLAIN, act="relu") == lcg.ERR_ARG
    h.close()


@pytest.mark.parametrize("option,bad", [(lcg.OPT_WAIT_TIMEOUT_US, 0), (lcg.OPT_WAIT_TIMEOUT_US, 61_000_000),
                                        (lcg.OPT_GROUP_ORDER, 2), (lcg.OPT_SPLIT, -1), (lcg.OPT_MAX_CTAS, -1),
                                        (lcg.OPT_PEAK_GFLOPS, 0), (lcg.OPT_HBM_GBPS, -5),
                                        (lcg.OPT_DEBUG_DROP_SIGNAL, 3), (lcg.OPT_PLAIN_KERNEL, 6),
                                        (lcg.OPT_LCMA_KERNEL, 3), (lcg.OPT_PDL, 2), (999, 1)])
def test_set_option_rejects_bad_values(option, bad):
    """Every option checks its range (and unknown keys are refused) with LCGEMM_ERR_ARG, on a
    planning handle, without a GPU."""
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    try:
        rc = h._lib.lcgemm_set_option(h._h, option, bad)
        assert rc == lcg.ERR_ARG
    finally:
        h.close()


def test_set_option_accepts_valid_values():
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    try:
        for option, good in [(lcg.OPT_WAIT_TIMEOUT_US, 1000), (lcg.OPT_GROUP_ORDER, 0), (lcg.OPT_SPLIT, 1),
                             (lcg.OPT_MAX_CTAS, 76), (lcg.OPT_PEAK_GFLOPS, 1951800), (lcg.OPT_HBM_GBPS, 6700),
                             (lcg.OPT_PLAIN_KERNEL, 4), (lcg.OPT_LCMA_KERNEL, 2), (lcg.OPT_PDL, 0)]:
            assert h._lib.lcgemm_set_option(h._h, option, good) == lcg.OK
    finally:
        h.close()
