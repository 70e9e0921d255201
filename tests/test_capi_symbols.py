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


def test_debug_build_exports_the_same_symbols(lib):
    """The MOE_DEBUG library (device-side bounds checks) is built beside the
    release one and offers the same entry points; it maps its own error bit
    to a status of its own."""
    path = os.path.join(ROOT, "moe_expert_dispatch_gb300", "libmoe_gb300_debug.so")
    dbg = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(dbg, n)]
    assert not missing, missing
    dbg.moe_status_string.restype = ctypes.c_char_p
    assert b"debug build" in dbg.moe_status_string(7)


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
    # T * k past the int32 row space is refused, also where the product
    # itself would overflow 64 bits
    assert m._lib.moe_route_topk_workspace_size(1 << 62, 32, 64) == 0
    assert m._lib.moe_permute_workspace_size(1 << 62, 32, 64) == 0
    assert m.moe_workspace_size(1 << 62, 4096, 14336, 8, 2) == 0
    assert m.moe_workspace_size(1 << 30, 4096, 14336, 8, 2) == 0     # 2^31 routed rows
    assert m._lib.moe_route_topk_workspace_size(4096, 2, 8) > 0


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



class _FakeCuda:
    """Stands in for a contiguous CUDA tensor on device `index`: enough of
    the tensor interface for the binding's checks, and a data_ptr that fails
    the test if a call ever gets as far as the library."""

    def __init__(self, shape, dtype, index=0):
        import torch
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.device = torch.device("cuda", index)
        self.is_cuda = True

    def is_contiguous(self):
        return True

    def numel(self):
        n = 1
        for d in self.shape:
            n *= d
        return n

    def data_ptr(self):
        raise AssertionError("the call reached the library")


def test_binding_refuses_tensors_on_two_devices(lib):
    # every kernel of a call runs on the device of its tensors: a call whose
    # tensors (inputs, outputs or workspace) span two devices is refused on
    # the host, and so are outputs of the wrong type or size
    import torch
    import moe_expert_dispatch_gb300 as m
    bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
    ids0 = _FakeCuda((4, 2), i32, 0)
    with pytest.raises(ValueError, match="one device"):
        m.moe_counts(ids0, 8, counts=_FakeCuda((8,), i32, 1))
    with pytest.raises(ValueError, match="one device"):
        m.moe_counts_static(ids0, 8, offsets=_FakeCuda((9,), i32, 1))
    with pytest.raises(ValueError, match="at least 9"):
        m.moe_counts_static(ids0, 8, offsets=_FakeCuda((8,), i32, 0))
    with pytest.raises(ValueError, match="int32"):
        m.moe_counts(ids0, 8, counts=_FakeCuda((8,), f32, 0))
    x, wg, wu, wd = (_FakeCuda((4, 128), bf), _FakeCuda((8, 128, 256), bf),
                     _FakeCuda((8, 128, 256), bf), _FakeCuda((8, 256, 128), bf))
    probs = _FakeCuda((4, 2), f32, 0)
    with pytest.raises(ValueError, match="one device"):
        m.moe_expert_forward(x, wg, wu, _FakeCuda((8, 256, 128), bf, 1), ids0, probs)
    with pytest.raises(ValueError, match="one device"):
        m.moe_expert_forward(x, wg, wu, wd, ids0, probs, y=_FakeCuda((4, 128), bf, 1))
    with pytest.raises(ValueError, match="one device"):
        m.moe_expert_backward(x, x, wg, wu, wd, ids0, probs, _FakeCuda((1024,), torch.uint8, 0),
                              dprobs=_FakeCuda((4, 2), f32, 1))
    with pytest.raises(ValueError, match="one device"):
        m.moe_unpermute(_FakeCuda((8, 128), bf, 1), ids0, probs)


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


def test_host_checks_under_address_and_undefined_behaviour_sanitizers(lib):
    """The host-side argument and size checks (including the overflow guards
    of the workspace sizes) run against the library built with
    AddressSanitizer and UndefinedBehaviorSanitizer on its host code: every
    check answers as in the release build, and neither sanitizer reports."""
    import importlib.util
    import shutil
    import subprocess
    import sys
    import torch
    if torch.cuda.is_available() or os.environ.get("MOE_GB300_SANITIZE"):
        pytest.skip("host-only: the cases carry fake device addresses")
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("no gcc to locate the sanitizer runtimes")
    rts = [subprocess.run([gcc, f"-print-file-name={n}"], capture_output=True,
                          text=True).stdout.strip() for n in ("libasan.so", "libubsan.so")]
    if not all(os.path.isabs(r) and os.path.exists(r) for r in rts):
        pytest.skip("sanitizer runtimes not installed")
    spec = importlib.util.spec_from_file_location(
        "_moe_build", os.path.join(ROOT, "moe_expert_dispatch_gb300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build(variants=("sanitize",))
    env = dict(os.environ, LD_PRELOAD=":".join(rts), MOE_GB300_SANITIZE="1",
               ASAN_OPTIONS="detect_leaks=0:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    probe = subprocess.run(
        [sys.executable, "-c", "import moe_expert_dispatch_gb300 as m; "
         "print(m.LIB_PATH); print('loaded' if 'libmoe_gb300_sanitize.so' in "
         "open('/proc/self/maps').read() else 'missing')"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr[-3000:]
    assert probe.stdout.split() == [os.path.join(ROOT, "moe_expert_dispatch_gb300",
                                                 "libmoe_gb300_sanitize.so"), "loaded"]
    out = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", __file__, "-k",
         "host_side or invalid_arguments or refuses_tensors or rejects_host"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    log = out.stdout + out.stderr
    assert out.returncode == 0, log[-4000:]
    assert "5 passed" in out.stdout, log[-4000:]
    assert "runtime error" not in log and "AddressSanitizer" not in log, log[-4000:]


def test_no_cluster_multicast_copies():
    # every CTA loads its own operands: no bulk copy in the kernels carries
    # .multicast::cluster. The one multicast form allowed is the MMA commit
    # that signals both CTAs of a pair (tcgen05.commit ... multicast::cluster),
    # which moves no data.
    import glob
    import re
    srcs = glob.glob(os.path.join(ROOT, "moe_expert_dispatch_gb300", "csrc", "*.cu*"))
    srcs += glob.glob(os.path.join(ROOT, "moe_expert_dispatch_gb300", "csrc", "*.h"))
    assert srcs
    seen = 0
    for p in srcs:
        text = open(p, encoding="utf-8").read()
        # each inline-asm string: the instruction text between quotes
        for instr in re.findall(r'"([^"\n]*)"', text):
            if "multicast" not in instr:
                continue
            seen += 1
            assert not re.search(r"cp\.async|cp\.reduce|\.bulk", instr), (p, instr)
            assert instr.lstrip().startswith("tcgen05.commit"), (p, instr)
    assert seen >= 1        # the scan does see the pair commit


def test_host_side_argument_errors_of_every_entry_point(lib):
    # each call is wrong in one way the host can see; it must answer with
    # that status at once, before any device work (this machine has no GPU,
    # so a call that reached the device would answer MOE_ERR_CUDA instead).
    # P is a fake, aligned device address that no check dereferences; with a
    # GPU present the test does not run, so a missing check could never hand
    # such an address to a kernel.
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only: the cases carry fake device addresses")
    import moe_expert_dispatch_gb300 as m
    L = m._lib
    P = ctypes.c_void_p(1 << 20)
    U = ctypes.c_void_p((1 << 20) + 8)      # not 16-byte aligned
    c = m.config()
    cs = m.config(save_for_backward=True)
    INV, UNS, WS = 1, 2, 4
    cases = [
        ("counts: E = 0", INV, lambda: L.moe_counts(P, 10, 0, P, P, P, 1 << 20, None)),
        ("counts: no workspace", WS, lambda: L.moe_counts(P, 10, 4, P, P, None, 0, None)),
        ("route_topk: k = 0", INV, lambda: L.moe_route_topk(P, 4, 8, 0, P, P, P, P, P, 1 << 20, None)),
        ("route_topk: k > E", INV, lambda: L.moe_route_topk(P, 4, 4, 5, P, P, P, P, P, 1 << 20, None)),
        ("route_topk: workspace too small", WS,
         lambda: L.moe_route_topk(P, 4, 8, 2, P, P, P, P, P, 16, None)),
        ("permute: unaligned x", INV,
         lambda: L.moe_permute(U, 4, 64, P, P, 2, 4, 1, P, P, P, P, P, P, P, 1 << 20, None)),
        ("permute: no workspace", WS,
         lambda: L.moe_permute(P, 4, 64, P, P, 2, 4, 1, P, P, P, P, P, P, None, 0, None)),
        ("unpermute: H % 8 != 0", INV, lambda: L.moe_unpermute(P, P, P, 4, 2, 12, P, None)),
        ("unpermute: k > 32", INV, lambda: L.moe_unpermute(P, P, P, 4, 33, 64, P, None)),
        ("quantize: unaligned input", INV, lambda: L.moe_quantize_mxfp8(U, 4, 64, P, P, None)),
        ("quantize_t: rows % 32 != 0", INV, lambda: L.moe_quantize_mxfp8_t(P, 1, 48, 64, P, P, None)),
        ("quantize_dual: cols % 128 != 0", INV,
         lambda: L.moe_quantize_mxfp8_dual(P, 1, 64, 96, P, P, P, P, None)),
        ("permute_quantize: H % 32 != 0", INV,
         lambda: L.moe_permute_quantize_mxfp8(P, 4, 48, P, 2, P, P, None)),
        ("forward: F % 128 != 0", UNS,
         lambda: L.moe_expert_forward(P, P, P, P, P, P, 4, 128, 100, 4, 2, P, P, 1 << 30,
                                      ctypes.byref(c), None)),
        ("forward: k > E", INV,
         lambda: L.moe_expert_forward(P, P, P, P, P, P, 4, 128, 128, 2, 3, P, P, 1 << 30,
                                      ctypes.byref(c), None)),
        ("forward: workspace too small", WS,
         lambda: L.moe_expert_forward(P, P, P, P, P, P, 4, 128, 128, 4, 2, P, P, 256,
                                      ctypes.byref(c), None)),
        ("forward_from_logits: no logits", INV,
         lambda: L.moe_expert_forward_from_logits(P, P, P, P, None, 4, 128, 128, 4, 2, P, P, P,
                                                  P, 1 << 30, ctypes.byref(c), None)),
        ("pipelined: zero chunks", INV,
         lambda: L.moe_expert_forward_pipelined(P, P, P, P, P, P, 4, 128, 128, 4, 2, P, 0, P,
                                                1 << 30, ctypes.byref(c), P, U)),
        ("pipelined: aux stream = stream", INV,
         lambda: L.moe_expert_forward_pipelined(P, P, P, P, P, P, 4, 128, 128, 4, 2, P, 2, P,
                                                1 << 30, ctypes.byref(c), P, P)),
        ("backward: no weight gradients", INV,
         lambda: L.moe_expert_backward(P, P, P, P, P, P, P, 4, 128, 128, 4, 2, P, 1 << 30, P,
                                       None, None, None, P, 0, P, 1 << 30, ctypes.byref(cs), None)),
        ("forward_mxfp8: no weights", INV,
         lambda: L.moe_expert_forward_mxfp8(P, None, None, None, None, None, None, P, P, 4, 128,
                                            128, 4, 2, P, P, 1 << 30, ctypes.byref(c), None)),
    ]
    for name, want, call in cases:
        assert call() == want, name
