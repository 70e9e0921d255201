"""The C-ABI library builds, loads without a GPU and exports every entry
point that include/moe_expert.h declares; host-side checks answer without
touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_expert.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from moe_expert_dispatch_gb300 import LIB_PATH
    return ctypes.CDLL(LIB_PATH)


def test_header_declares_the_block():
    names = declared_functions()
    for n in ("moe_counts", "moe_permute", "moe_unpermute", "moe_expert_forward",
              "moe_expert_backward", "moe_quantize_mxfp8", "moe_expert_forward_mxfp8"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_queries(lib):
    import moe_expert_dispatch_gb300 as m
    assert m.moe_padded_rows(8192, 8, 128) == 9216
    assert m.moe_padded_rows(5, 3, 1) == 5
    ws = m.moe_workspace_size(4096, 4096, 14336, 8, 2)
    # Xp, O: cap x H bf16; h: cap x F bf16 (cap = 9216 padded rows)
    assert ws >= 9216 * (4096 * 2 * 2 + 14336 * 2)
    assert m.moe_workspace_size(16, 100, 128, 4, 2) == 0     # H % 128 != 0 is unsupported
    assert m.moe_workspace_size(16, 128, 128, 4, 5) == 0     # k > E
    s = m._lib.moe_status_string(3)
    assert b"expert id" in s


def test_invalid_arguments_rejected_before_any_launch(lib):
    import moe_expert_dispatch_gb300 as m
    c = m.config()
    st = m._lib.moe_expert_forward(None, None, None, None, None, None, 4, 128, 128, 4, 2, None,
                                   None, 0, ctypes.byref(c), None)
    assert st == 1
    st = m._lib.moe_expert_forward(None, None, None, None, None, None, 4, 100, 128, 4, 2, None,
                                   None, 0, ctypes.byref(c), None)
    assert st == 2
    assert m._lib.moe_counts(None, 10, 0, None, None, None, 0, None) == 1
    assert m._lib.moe_quantize_mxfp8(None, 4, 33, None, None, None) == 1
    assert m._lib.moe_permute_quantize_mxfp8(None, 4, 48, None, 2, None, None, None) == 1
    assert m._lib.moe_permute_quantize_mxfp8(None, 4, 64, None, 33, None, None, None) == 1
    assert m._lib.moe_permute_quantize_mxfp8(None, 0, 64, None, 2, None, None, None) == 0


def test_binding_rejects_host_tensors_before_the_library(lib):
    # the binding checks device, dtype and layout itself, so no call reaches
    # the library with a host pointer
    import torch
    import moe_expert_dispatch_gb300 as m
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    rows = torch.zeros((4, 2), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_permute_quantize_mxfp8(x, rows)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_quantize_mxfp8(x)
    with pytest.raises(ValueError, match="CUDA"):
        m.moe_unpermute(x, rows, torch.zeros((4, 2)))



def test_package_refuses_to_import_without_the_library(tmp_path):
    # a copy of the package without libmoe_gb300.so: the import fails loudly
    # instead of falling back to anything else
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "moe_expert_dispatch_gb300", "__init__.py")
    pkg = tmp_path / "moe_expert_dispatch_gb300"
    pkg.mkdir()
    shutil.copy(src, pkg / "__init__.py")
    out = subprocess.run([sys.executable, "-c", "import moe_expert_dispatch_gb300"],
                         capture_output=True, text=True, cwd=tmp_path, timeout=300)
    assert out.returncode != 0
    assert "ImportError" in out.stderr and "no CPU or eager fallback" in out.stderr


def test_product_and_oracle_share_nothing():
    # the library and its binding never name the oracle, and the oracle
    # never names the library: parity compares two independent programs
    import glob
    product = [p for ext in ("py", "cu", "cuh", "h")
               for p in glob.glob(os.path.join(ROOT, "moe_expert_dispatch_gb300", "**", "*." + ext),
                                  recursive=True)]
    product += glob.glob(os.path.join(ROOT, "include", "*.h"))
    assert product
    for p in product:
        assert "oracle" not in open(p, encoding="utf-8").read(), p
    for p in glob.glob(os.path.join(ROOT, "oracle", "**", "*.py"), recursive=True):
        text = open(p, encoding="utf-8").read()
        assert "moe_expert_dispatch_gb300" not in text and "libmoe" not in text, p
