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


def test_int8_variant_arguments_rejected_before_any_launch(lib):
    fake = 0x10000
    p = ctypes.c_void_p(fake)
    m = _mats((4, 4), data=fake)
    assert lib.sign_int8(m, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.sign_int8(None, p, None) == _abi.MAO_ERR_INVALID_ARG
    i8 = _mats((4, 4), dtype=_abi.MAO_I8, data=fake)
    assert lib.sign_int8(i8, p, None) == _abi.MAO_ERR_INVALID_ARG  # input must be f32/bf16
    # workers 1..127, stride >= n, at least one output, word-aligned vote
    assert lib.majority_vote_int8(p, 0, 64, 64, p, None, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.majority_vote_int8(p, 128, 64, 64, p, None, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.majority_vote_int8(p, 3, 63, 64, p, None, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.majority_vote_int8(p, 3, 64, 0, p, None, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.majority_vote_int8(None, 3, 64, 64, p, None, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.majority_vote_int8(p, 3, 64, 64, None, None, None, None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.majority_vote_int8(p, 3, 64, 64, None, None, ctypes.c_void_p(fake + 2),
                                  None) == _abi.MAO_ERR_MISALIGNED


def test_sign_matrix_inputs_only_where_declared(lib):
    fake = 0x10000
    co = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    ws = ctypes.c_void_p(fake)
    out = _mats((4, 40), dtype=_abi.MAO_F32, data=fake)
    # packed signs need ld == cols
    bad = (_abi.MaoMat * 1)(_abi.MaoMat(fake, 4, 40, 48, _abi.MAO_SIGN1, 0))
    assert lib.ns_orthogonalize(bad, out, 1, 5, co, 0, 1e-7, 1, None, ws, 1 << 30, None) == 1
    assert lib.ns_orthogonalize_noalloc(bad, out, 1, 5, co, 0, 1e-7, 1, None, None) == 1
    # packed words are 4-byte aligned
    odd = (_abi.MaoMat * 1)(_abi.MaoMat(fake + 2, 4, 40, 40, _abi.MAO_SIGN1, 0))
    assert lib.ns_orthogonalize(odd, out, 1, 5, co, 0, 1e-7, 1, None, ws, 1 << 30,
                                None) == _abi.MAO_ERR_MISALIGNED
    # int8 and packed signs are inputs only: not outputs, not momentum or update operands
    i8 = _mats((4, 40), dtype=_abi.MAO_I8, data=fake)
    s1 = _mats((4, 40), dtype=_abi.MAO_SIGN1, data=fake)
    f32 = _mats((4, 40), dtype=_abi.MAO_F32, data=fake)
    assert lib.ns_orthogonalize(f32, i8, 1, 5, co, 0, 1e-7, 1, None, ws, 1 << 30, None) == 1
    assert lib.muon_momentum_update(i8, f32, 1, 0.9, None) == 1
    assert lib.muon_momentum_update(f32, s1, 1, 0.9, None) == 1
    assert lib.apply_update(f32, None, i8, 1, 0.01, None) == 1
    # workspace sizes do not depend on the input encoding
    assert lib.ns_workspace_bytes(i8, 1, 1) == lib.ns_workspace_bytes(f32, 1, 1) > 0


def test_blockwise_arguments_and_sizes(lib):
    fake = 0x10000
    co = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    ws = ctypes.c_void_p(fake)
    X = _mats((300, 1000), dtype=_abi.MAO_BF16, data=fake)
    # the workspace of a blockwise call is that of its blocks as one batch
    blocks = _mats(*([(128, 256)] * 6 + [(128, 232)] * 2 + [(44, 256)] * 3 + [(44, 232)]))
    assert lib.ns_blockwise_workspace_bytes(X, 1, 128, 256, 1) == lib.ns_workspace_bytes(blocks, 12, 1)
    assert lib.ns_blockwise_workspace_bytes(X, 1, 300, 1000, 1) == lib.ns_workspace_bytes(X, 1, 1)
    assert lib.ns_blockwise_workspace_bytes(X, 1, 0, 256, 1) == 0
    big = _mats((2048, 1024), dtype=_abi.MAO_BF16, data=fake)
    assert lib.ns_blockwise_workspace_bytes(big, 1, 1, 1, 1) == 0  # 2^21 blocks > 2^20
    out = _mats((300, 1000), dtype=_abi.MAO_F32, data=fake)
    s1 = (_abi.MaoMat * 1)(_abi.MaoMat(fake, 300, 1000, 1000, _abi.MAO_SIGN1, 0))
    args = (1, 128, 256, 5, co, 0, 1e-7, 1, ws, 1 << 40, None)
    assert lib.ns_orthogonalize_blockwise(s1, out, *args) == _abi.MAO_ERR_INVALID_ARG
    assert lib.ns_orthogonalize_blockwise(X, out, 1, 0, 256, 5, co, 0, 1e-7, 1, ws, 1 << 40,
                                          None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.ns_orthogonalize_blockwise(X, out, 1, 128, 256, 5, co, 0, 1e-7, 1, None, 1 << 40,
                                          None) == _abi.MAO_ERR_INVALID_ARG
    assert lib.ns_orthogonalize_blockwise(X, X, 1, 128, 256, 5, co, 1, 1e-7, 1, ws, 1 << 40,
                                          None) == _abi.MAO_ERR_INVALID_ARG


def test_muon_step_arguments_rejected_before_any_launch(lib):
    fake = 0x10000
    co = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    ws = ctypes.c_void_p(fake)
    W = _mats((64, 96), data=fake)
    M = _mats((64, 96), data=fake + 4096)
    G = _mats((64, 96), data=fake + 8192)

    def call(W=W, M=M, G=G, W_out=None, batch=1, mu=0.95, lr=0.02, steps=5, coeffs=co,
             stride=0, eps=1e-7, compute=_abi.MAO_BF16, ws=ws, nbytes=1 << 30):
        return lib.muon_step(W, M, G, W_out, batch, mu, lr, steps, coeffs, stride, eps, compute,
                             ws, nbytes, None)

    assert call(W=None) == _abi.MAO_ERR_INVALID_ARG
    assert call(batch=0) == _abi.MAO_ERR_INVALID_ARG
    assert call(steps=0) == _abi.MAO_ERR_INVALID_ARG
    assert call(stride=2) == _abi.MAO_ERR_INVALID_ARG
    assert call(mu=float("nan")) == _abi.MAO_ERR_INVALID_ARG
    assert call(lr=float("inf")) == _abi.MAO_ERR_INVALID_ARG
    assert call(eps=-1.0) == _abi.MAO_ERR_INVALID_ARG
    assert call(compute=_abi.MAO_F32) == _abi.MAO_ERR_UNSUPPORTED  # tensor-core path only
    assert call(G=_mats((64, 95), data=fake)) == _abi.MAO_ERR_INVALID_ARG
    assert call(W_out=_mats((64, 96), dtype=_abi.MAO_F32, data=fake)) == _abi.MAO_ERR_INVALID_ARG
    assert call(W_out=_mats((64, 95), data=fake)) == _abi.MAO_ERR_INVALID_ARG
    assert call(ws=None) == _abi.MAO_ERR_INVALID_ARG
    assert call(ws=ctypes.c_void_p(fake + 16)) == _abi.MAO_ERR_MISALIGNED


def test_sign_muon_step_argument_checks(lib):
    fake = 0x10000
    co = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    ws = ctypes.c_void_p(fake)
    W = _mats((6, 40), dtype=_abi.MAO_F32, data=fake)
    M = (_abi.MaoMat * 2)(*[_abi.MaoMat(fake, 6, 40, 40, _abi.MAO_F32, 0) for _ in range(2)])
    p = ctypes.c_void_p(fake)
    nw = (6 * 40 + 31) // 32

    def call(W=W, M=M, n=2, words=p, stride=nw, vote=p, ws=ws, wsb=1 << 30):
        return lib.sign_muon_step(W, M, M, n, words, stride, vote, 0.95, 0.02, 5, co, 0, 1e-7,
                                  0, ws, wsb, None)

    assert call(words=None) == _abi.MAO_ERR_INVALID_ARG
    assert call(vote=None) == _abi.MAO_ERR_INVALID_ARG
    assert call(n=0) == _abi.MAO_ERR_INVALID_ARG
    assert call(stride=nw - 1) == _abi.MAO_ERR_INVALID_ARG          # rows would overlap
    assert call(words=ctypes.c_void_p(fake + 2)) == _abi.MAO_ERR_MISALIGNED
    assert call(ws=None) == _abi.MAO_ERR_INVALID_ARG
    assert call(wsb=16) == _abi.MAO_ERR_WORKSPACE
    other = (_abi.MaoMat * 2)(*[_abi.MaoMat(fake, 6, 41, 41, _abi.MAO_F32, 0) for _ in range(2)])
    assert call(M=other) == _abi.MAO_ERR_INVALID_ARG                 # worker shape != W
