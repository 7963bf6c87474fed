"""The C-ABI library builds, loads and exports every symbol include/mao.h declares.

CPU only: these calls validate arguments or report sizes and never launch a kernel.
"""

import ctypes
import os
import re

from matrix_aware_optimizers_gb300 import _abi


def _declared_symbols(root):
    with open(os.path.join(root, "include", "mao.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?([a-z_0-9]+)\(", text, flags=re.M))


def test_header_and_binding_agree():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    declared = _declared_symbols(root)
    assert declared == set(_abi.EXPORTS), declared ^ set(_abi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _abi.EXPORTS:
        assert hasattr(lib, name), name
    assert lib.mao_abi_version() == 1


def test_status_strings(lib):
    assert lib.mao_status_string(0) == b"MAO_OK"
    assert lib.mao_status_string(4) == b"MAO_ERR_WORKSPACE"
    assert lib.mao_status_string(99) == b"MAO_ERR_UNKNOWN"


def _mats(*shapes, dtype=_abi.MAO_BF16, data=None):
    arr = (_abi.MaoMat * len(shapes))()
    for i, (r, c) in enumerate(shapes):
        arr[i] = _abi.MaoMat(data, r, c, c, dtype, 0)
    return arr


def test_workspace_bytes_host_only(lib):
    one = lib.ns_workspace_bytes(_mats((768, 768)), 1, _abi.MAO_BF16)
    two = lib.ns_workspace_bytes(_mats((768, 768), (768, 768)), 2, _abi.MAO_BF16)
    f32 = lib.ns_workspace_bytes(_mats((768, 768)), 1, _abi.MAO_F32)
    # two ping-pong X buffers plus A and B, bf16: at least 4 * 768^2 * 2 bytes per matrix
    assert one >= 4 * 768 * 768 * 2
    assert two >= 2 * 4 * 768 * 768 * 2
    assert f32 >= 2 * (one - 4096)
    # invalid arguments report 0
    assert lib.ns_workspace_bytes(_mats((0, 5)), 1, _abi.MAO_BF16) == 0
    assert lib.ns_workspace_bytes(_mats((5, 5)), 1, 7) == 0
    assert lib.ns_workspace_bytes(None, 1, _abi.MAO_BF16) == 0


def test_invalid_arguments_rejected_before_any_launch(lib):
    fake = 0x10000  # never dereferenced: every call below fails validation first
    m = _mats((4, 4), data=fake)
    assert lib.muon_momentum_update(None, m, 1, 0.9, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.muon_momentum_update(m, m, 0, 0.9, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.muon_momentum_update(m, m, 1, float("nan"), None) == _abi.MAO_ERR_INVALID_ARG
    other = _mats((4, 5), data=fake)
    assert lib.muon_momentum_update(m, other, 1, 0.9, None) == _abi.MAO_ERR_INVALID_ARG
    odd = _mats((4, 4), data=fake + 1)
    assert lib.muon_momentum_update(odd, m, 1, 0.9, None) == _abi.MAO_ERR_MISALIGNED
    bad_ld = (_abi.MaoMat * 1)(_abi.MaoMat(fake, 4, 4, 3, _abi.MAO_BF16, 0))
    assert lib.muon_momentum_update(bad_ld, m, 1, 0.9, None) == _abi.MAO_ERR_INVALID_ARG

    co = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    ws = ctypes.c_void_p(fake)
    assert lib.ns_orthogonalize(m, m, 1, 0, co, 0, 1e-7, 1, None, ws, 1 << 20, None) == 1
    assert lib.ns_orthogonalize(m, m, 1, 5, co, 2, 1e-7, 1, None, ws, 1 << 20, None) == 1
    assert lib.ns_orthogonalize(m, m, 1, 5, None, 0, 1e-7, 1, None, ws, 1 << 20, None) == 1
    assert lib.ns_orthogonalize(m, m, 1, 5, co, 0, -1.0, 1, None, ws, 1 << 20, None) == 1
    assert lib.ns_orthogonalize(m, m, 1, 5, co, 0, 1e-7, 1, None, None, 1 << 20, None) == 1
    assert lib.ns_orthogonalize(m, m, 1, 5, co, 0, 1e-7, 1, None, ctypes.c_void_p(fake + 16),
                                1 << 20, None) == _abi.MAO_ERR_MISALIGNED
    nul = _mats((4, 4), data=None)
    assert lib.ns_orthogonalize(m, nul, 1, 5, co, 0, 1e-7, 1, None, ws, 1 << 20, None) == 1

    assert lib.sign_pack_bits(m, None, None) == 1
    assert lib.majority_vote_packed(ctypes.c_void_p(fake), 0, 4, 100, ctypes.c_void_p(fake), None) == 1
    assert lib.majority_vote_packed(ctypes.c_void_p(fake), 3, 2, 100, ctypes.c_void_p(fake), None) == 1
    assert lib.apply_update(m, None, None, 1, 0.01, None) == 1
    votes = (ctypes.c_void_p * 1)(fake)
    assert lib.apply_update(m, votes, m, 1, 0.01, None) == 1
