"""The C-ABI library on a host without a GPU: it loads, exports every
function include/mxq.h declares with the signature the binding uses, and
rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import fp4_quantization_gb300 as mxq
from fp4_quantization_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"MXQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for required in ("mx_quantize_rowcol", "mx_quantize_gated", "nvfp4_quantize_transpose",
                     "bf16_amax"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = _lib.lib()
    names = declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(L, name), name
    # The binding's signature table covers exactly the declared functions.
    assert set(_lib.SIGNATURES) == set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_status_strings():
    L = _lib.lib()
    for code, name in mxq.STATUS_NAMES.items():
        assert L.mxq_status_string(code).decode().startswith(name)
    assert L.mxq_status_string(99) == b"unknown mxq status"


def _rowcol(**kw):
    args = dict(x=None, M=64, K=64, ldx=64, flags=3, q_row=None, s_row=None, q_col=None,
                s_col=None, dbias=None, ws=None, ws_bytes=0, err=None, stream=None)
    args.update(kw)
    return _lib.lib().mx_quantize_rowcol(*args.values())


@pytest.mark.parametrize("kw,status", [
    (dict(flags=0), 1),                    # no direction
    (dict(flags=16 | 1), 1),               # unknown flag bit
    (dict(flags=1 | 4 | 8), 1),            # dbias with gelu
    (dict(M=-32), 2),
    (dict(M=48), 2),                       # not a multiple of 32
    (dict(K=40, ldx=40), 2),
    (dict(ldx=32), 2),                     # ldx < K
])
def test_rowcol_host_validation(kw, status):
    assert _rowcol(**kw) == status


def test_gated_and_nvfp4_host_validation():
    L = _lib.lib()
    assert L.mx_quantize_gated(None, 64, 64, 100, 3, None, None, None, None, None, None) == 2
    assert L.mx_quantize_gated(None, 64, 48, 96, 3, None, None, None, None, None, None) == 2
    assert L.mx_quantize_gated(None, 64, 64, 128, 4, None, None, None, None, None, None) == 1
    nv = L.nvfp4_quantize_transpose
    assert nv(None, 24, 32, 32, 3, None, None, None, None, None, None, None, 0, None, None) == 2
    assert nv(None, 48, 64, 64, 3, None, None, None, None, None, None, None, 0, None, None) == 2
    assert nv(None, 32, 32, 32, 0, None, None, None, None, None, None, None, 0, None, None) == 1
    assert nv(None, 32, 32, 32, 3, None, None, None, None, None, None, None, 0, None, None) == 1
    assert L.bf16_amax(None, 16, 12, 12, None, None) == 1
    assert L.bf16_amax(None, 16, 12, 12, ctypes.c_void_p(16), None) == 2
    assert L.mxq_selftest_bounded_wait(10, None, None) == 1


def test_backward_and_geglu_host_validation():
    L = _lib.lib()
    GELU, SILU = mxq.ACT_GELU_TANH, mxq.ACT_SILU

    def dact(M=64, K=64, ldg=64, ldx=64, flags=3 | GELU):
        return L.mx_quantize_dact(None, None, M, K, ldg, ldx, flags, None, None, None, None, None,
                                  None, 0, None, None)

    assert dact(flags=3) == 1                      # no activation
    assert dact(flags=3 | GELU | SILU) == 1        # two activations
    assert dact(flags=GELU) == 1                   # no direction
    assert dact(flags=3 | GELU | 16) == 1          # unknown bit
    assert dact(M=48) == 2 and dact(K=40, ldg=40, ldx=40) == 2
    assert dact(ldg=32) == 2 and dact(ldx=32) == 2

    def dgated(M=64, N=64, ldg=64, ldx=128, flags=3):
        return L.mx_quantize_dgated(None, None, M, N, ldg, ldx, flags, None, None, None, None,
                                    None, None)

    assert dgated(flags=3 | GELU | SILU) == 1 and dgated(flags=0) == 1
    assert dgated(ldx=100) == 2 and dgated(ldg=32) == 2 and dgated(N=48, ldg=48, ldx=96) == 2
    assert L.mx_quantize_gated(None, 64, 64, 128, 3 | GELU | SILU, None, None, None, None, None,
                               None) == 1
    assert L.mxq_workspace_bytes(mxq.OP_DACT, 256, 64, mxq.DBIAS) == 2 * 64 * 4
    assert L.mxq_workspace_bytes(mxq.OP_DACT, 256, 64, 0) == 0


def test_host_path_host_validation():
    L = _lib.lib()

    def call(M=64, K=64, ldx=64, flags=3, ws=None, ws_bytes=0):
        return L.mx_quantize_rowcol_host(ctypes.c_void_p(16), M, K, ldx, flags,
                                         ctypes.c_void_p(16), ctypes.c_void_p(16),
                                         ctypes.c_void_p(16), ctypes.c_void_p(16), ws, ws_bytes,
                                         None)

    assert call(flags=0) == 1 and call(flags=3 | mxq.DBIAS) == 1
    assert call(M=48) == 2 and call(ldx=32) == 2
    assert call() == 5                                     # no workspace
    need = L.mxq_workspace_bytes(mxq.OP_ROWCOL_HOST, 64, 64, 3)
    assert need > 0
    assert call(ws=ctypes.c_void_p(256), ws_bytes=need - 1) == 5
    assert call(ws=ctypes.c_void_p(128), ws_bytes=need) == 3   # not 256-byte aligned
    assert call(M=0) == 0
