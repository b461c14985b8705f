"""The C-ABI library loads and exports every function include/fmm.h declares.

No compute call is made here (this tier runs without a GPU)."""
import ctypes as C
import os
import subprocess

import pytest

from body_forces_morton_b300 import native


@pytest.fixture(scope="module")
def built():
    from body_forces_morton_b300 import build
    return build.build()


def test_header_declares_the_boundary():
    names = native.declared_functions()
    for required in ("fmm_plan_create", "fmm_eval", "fmm_kdk_step", "fmm_destroy", "fmm_last_error",
                     "fmm_plan_stats", "fmm_eval_host", "fmm_plan_export"):
        assert required in names


def test_library_exports_every_declared_symbol(built):
    out = subprocess.run(["nm", "-D", "--defined-only", built], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [f for f in native.declared_functions() if f not in exported]
    assert not missing, missing
    lib = C.CDLL(built)
    for f in native.declared_functions():
        assert hasattr(lib, f)


def test_build_targets_sm_103a():
    from body_forces_morton_b300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(native, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(native, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        native.lib()


def test_destroy_accepts_null_and_last_error_is_a_string(built):
    lib = native.lib()
    lib.fmm_destroy(None)
    assert isinstance(native.fmm_last_error(), str)
