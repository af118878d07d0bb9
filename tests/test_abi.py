"""The C-ABI library loads on the host, exports every entry point include/bsp.h
declares, and its structs have the layout the Python binding assumes. No
device calls."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "bsp.h")


@pytest.fixture(scope="module")
def native():
    from block_sparse_paged_gb300 import build
    build.build()
    from block_sparse_paged_gb300 import _native
    return _native


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsp_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(native):
    lib = native.load()
    names = declared_functions()
    assert "bsp_plan" in names and "bsp_decode_run" in names and "bsp_prefill_run" in names
    assert "bsp_merge_state" in names
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(native.EXPORTED) == names


def test_struct_layout_matches_header(native, tmp_path):
    prog = tmp_path / "sizes.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "bsp.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(bsp_problem), sizeof(bsp_capacity), sizeof(bsp_plan_info),
         sizeof(bsp_work_item), sizeof(bsp_merge_entry));
  printf("%zu %zu %zu %zu %zu %zu\n", offsetof(bsp_plan_info, total_work), offsetof(bsp_plan_info, off_header),
         offsetof(bsp_plan_info, off_partial_o), offsetof(bsp_plan_info, valid),
         offsetof(bsp_plan_info, off_gather), offsetof(bsp_capacity, max_gather_pages));
  return 0;
}''')
    exe = tmp_path / "sizes"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    sizes, offs = subprocess.check_output([str(exe)], text=True).strip().split("\n")
    want = [ctypes.sizeof(native.Problem), ctypes.sizeof(native.Capacity), ctypes.sizeof(native.PlanInfo),
            native.WORK_ITEM_DTYPE.itemsize, native.MERGE_ENTRY_DTYPE.itemsize]
    assert [int(x) for x in sizes.split()] == want
    PI = native.PlanInfo
    assert [int(x) for x in offs.split()] == [PI.total_work.offset, PI.off_header.offset, PI.off_partial_o.offset,
                                              PI.valid.offset, PI.off_gather.offset,
                                              native.Capacity.max_gather_pages.offset]


def test_version_and_error_strings(native):
    lib = native.load()
    assert lib.bsp_version().decode().startswith("bsp")
    assert isinstance(lib.bsp_last_error(), bytes)


def test_workspace_size_rejects_bad_problem(native):
    lib = native.load()
    bad = native.Problem(0, 6, 4, 128, 16, 0, 0)   # 6 % 4 != 0
    cap = native.Capacity(8, 16, 8)
    assert lib.bsp_workspace_size(ctypes.byref(bad), ctypes.byref(cap)) == 0
    assert b"multiple" in lib.bsp_last_error()
    good = native.Problem(0, 32, 8, 128, 16, 0, 0)
    ws = lib.bsp_workspace_size(ctypes.byref(good), ctypes.byref(cap))
    st = lib.bsp_host_staging_size(ctypes.byref(good), ctypes.byref(cap))
    assert 0 < st < ws and ws % 256 == 0


def test_product_package_has_no_oracle_imports():
    """The product package never imports the oracle (no CPU fallback)."""
    pkg = os.path.join(ROOT, "block_sparse_paged_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
                assert "attention.c" not in text and "liboracle" not in text, f


def test_bounded_wait_self_test_rejects_bad_arguments(native):
    """Argument checks of bsp_check_bounded_wait happen on the host, before any
    launch (no device needed)."""
    lib = native.load()
    assert lib.bsp_check_bounded_wait(1000, None, None) == native.BSP_ERR_INVALID_ARG
    assert lib.bsp_check_bounded_wait(0, ctypes.c_void_p(16), None) == native.BSP_ERR_INVALID_ARG
    assert lib.bsp_check_bounded_wait(1 << 34, ctypes.c_void_p(16), None) == native.BSP_ERR_INVALID_ARG


def test_gather_region_in_the_workspace(native):
    """capacity.max_gather_pages (prefill) adds a K and a V region of that many
    pages to the workspace, after the partial states; the plan reports where,
    and how many pages its table has. Decode rejects a region."""
    import numpy as np
    lib = native.load()
    pre = native.Problem(1, 32, 8, 128, 1, 1, 0)
    base = lib.bsp_workspace_size(ctypes.byref(pre), ctypes.byref(native.Capacity(2, 16, 4096, 1, 0)))
    pages = 5000
    ws = lib.bsp_workspace_size(ctypes.byref(pre), ctypes.byref(native.Capacity(2, 16, 4096, 1, pages)))
    pool = -(-pages * 1 * 8 * 128 * 2 // 256) * 256
    assert ws == base + 2 * pool
    cap = native.Capacity(2, 16, 4096, 1, pages)
    staging = np.zeros(lib.bsp_host_staging_size(ctypes.byref(pre), ctypes.byref(cap)), np.uint8)
    qo = np.array([0, 100, 300], np.int32)
    kv = np.array([0, 700, 2000], np.int32)
    lp = np.ones(2, np.int32)
    info = native.PlanInfo()
    native.check(lib.bsp_plan(ctypes.byref(pre), ctypes.byref(cap), 2, qo.ctypes.data_as(ctypes.c_void_p),
                              kv.ctypes.data_as(ctypes.c_void_p), lp.ctypes.data_as(ctypes.c_void_p), 2, 1,
                              staging.ctypes.data_as(ctypes.c_void_p), None, 0, None, ctypes.byref(info)))
    assert info.num_table_pages == 2000 and info.gather_pool_bytes == pool
    assert info.off_gather == info.workspace_bytes - 2 * pool and info.off_gather % 256 == 0
    dec = native.Problem(0, 32, 8, 128, 1, 0, 0)
    assert lib.bsp_workspace_size(ctypes.byref(dec), ctypes.byref(native.Capacity(2, 16, 2, 1, 10))) == 0
    assert b"max_gather_pages" in lib.bsp_last_error()
