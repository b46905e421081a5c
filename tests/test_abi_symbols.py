"""The C-ABI library builds, loads without a GPU and exports every entry
point that include/dflash.h declares (no compute calls here)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "dflash.h"), encoding="utf-8").read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_02_gb300 import dflash
    lib = ctypes.CDLL(dflash.LIB_PATH)
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dflash.EXPORTED)


def test_host_only_calls_work_without_a_gpu():
    import __graft_entry__
    __graft_entry__.build()
    from block_diffusion_speculative_02_gb300 import dflash
    assert dflash.dflash_version() >= 100
    assert dflash.status_string(0) == "ok"
    assert "workspace" in dflash.status_string(-4)
