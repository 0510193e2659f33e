"""The C ABI library loads and exports every entry point its header declares (no GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "purlin.h")


@pytest.fixture(scope="session")
def libpath():
    from copy_reduce_datapath_gb300 import build
    return build.build()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PL_API\s+[^;(]*?\b(pl_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pl_collective", "pl_allreduce", "pl_ctx_create", "pl_ctx_destroy", "pl_ctx_status",
                 "pl_layout_create", "pl_layout_destroy", "pl_status_str", "pl_abi_version"):
        assert must in names


def test_every_declared_symbol_is_exported(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_exports_are_only_the_abi(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True, check=True)
    exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
    assert exported == set(declared_functions())


def test_abi_version_and_status_strings(libpath):
    from copy_reduce_datapath_gb300 import purlin as P
    assert P.pl_abi_version() == 2
    for st in range(8):
        assert P.pl_status_str(st) and P.pl_status_str(st) != "unknown status"
    assert P.pl_status_str(99) == "unknown status"


def test_no_gpu_is_a_clean_error(libpath):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from copy_reduce_datapath_gb300 import purlin as P
    with pytest.raises(P.PurlinError) as e:
        P.pl_ctx_create(0, 0)
    assert e.value.status == P.PL_ERR_CUDA
