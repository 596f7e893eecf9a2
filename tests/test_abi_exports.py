"""The C-ABI library builds, loads without a GPU and exports every function
that include/*.h declares (no compute calls here)."""
import ctypes
import glob
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text):
            name = m.group(1)
            # a declaration: "<type> name(" at statement start
            pre = text[:m.start()].rstrip()
            if pre.endswith(("*", "qsm_status", "size_t", "int32_t", "char")) \
                    and name not in ("sizeof",):
                names.append(name)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("moe_route", "moe_group_tokens", "moe_ffn_forward",
                     "q8_gemv", "moe_route_workspace_bytes",
                     "moe_ffn_workspace_bytes", "qsm_status_str"):
        assert required in names


@pytest.mark.skipif(shutil.which("nvcc") is None and
                    not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc missing")
def test_library_builds_loads_and_exports_everything():
    from quantized_sparse_moe_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)          # loads without touching a GPU
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"
    lib.qsm_abi_version.restype = ctypes.c_int32
    assert lib.qsm_abi_version() == 4
    lib.qsm_status_str.restype = ctypes.c_char_p
    assert lib.qsm_status_str(0) == b"ok"
    # host-only helpers need no device
    lib.moe_group_max_tiles.restype = ctypes.c_int32
    assert lib.moe_group_max_tiles(1, 8, 256, 8) == 8
    assert lib.moe_group_max_tiles(4096, 8, 256, 128) == 256 + (32768 - 256) // 128
    # exported dynamic symbols are exactly the declared ones (plus none else)
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", path],
                             capture_output=True, text=True).stdout
        exported = {l.split()[-1] for l in out.splitlines()
                    if " T " in l}
        assert set(declared_functions()) <= exported


@pytest.mark.skipif(shutil.which("nvcc") is None and
                    not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc missing")
def test_decode_layer_coresidency_check():
    """qsm_decode_layer_fits: the one-launch decode layer runs only when its
    whole grid can be resident (host logic, no GPU)."""
    import quantized_sparse_moe_gb300 as qsm
    from quantized_sparse_moe_gb300 import build
    lib = ctypes.CDLL(build.build())
    f = lib.qsm_decode_layer_fits
    f.argtypes = [ctypes.POINTER(qsm.MoELayerC), ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32]
    f.restype = ctypes.c_int32

    def layer(qtype, H=2048, I=512, E=256, k=8):
        def qw(experts, rows, cols):
            return qsm.QWeightsC(qtype, experts, rows, cols, None, None, None)
        return qsm.MoELayerC(H, I, E, k, qw(E, 2 * I, H), qw(E, H, I), qw(1, 2 * I, H),
                             qw(1, H, I), None)

    q8 = layer(qsm.Q8_0)
    assert f(ctypes.byref(q8), 1, 152, 1) == 1      # GB300: 152 SMs, one CTA each
    assert f(ctypes.byref(q8), 8, 152, 1) == 1
    assert f(ctypes.byref(q8), 1, 152, 0) == 0      # no CTA fits an SM
    assert f(ctypes.byref(q8), 1, 120, 1) == 0      # fewer SMs than 16-row blocks of y
    assert f(ctypes.byref(q8), 9, 152, 1) == 0      # more than 8 tokens
    assert f(ctypes.byref(q8), 0, 152, 1) == 0
    a4 = layer(qsm.AFFINE4_G64)
    assert f(ctypes.byref(a4), 4, 152, 1) == 1
    assert f(ctypes.byref(layer(qsm.Q8_0, E=512)), 2, 152, 1) == 1
