"""The C-ABI library builds for sm_103a, loads without a GPU, and exports
every entry point that the headers under include/ declare (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for f in sorted(os.listdir(INCLUDE)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(dflash_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("dflash_select_init", "dflash_select_run", "dflash_verify_prefix", "dflash_select_destroy",
                     "dflash_last_error", "dflash_select_sync_status", "dflash_select_step_host",
                     "dflash_select_run_sampled", "dflash_verify_rejection", "dflash_conv2_init", "dflash_conv2_run",
                     "dflash_conv2_sync_status", "dflash_conv2_destroy"):
        assert required in names


def test_library_builds_and_exports_every_declared_symbol():
    from speculative_decoding_draft_tcgen05_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    import speculative_decoding_draft_tcgen05_gb300 as pkg
    assert pkg.lib() is not None
    # a pure host call that needs no GPU
    assert pkg.dflash_last_error() == ""


def test_no_cpu_fallback_in_product_package():
    """The product package never imports the oracle."""
    pkg_dir = os.path.join(ROOT, "speculative_decoding_draft_tcgen05_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import oracle|from oracle)", src, flags=re.M), f
                assert "liboracle" not in src, f


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library the binding raises; it never falls back to
    anything else."""
    import speculative_decoding_draft_tcgen05_gb300 as pkg
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "libdflash_select.so"))
    monkeypatch.setattr(pkg, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        pkg.lib()
