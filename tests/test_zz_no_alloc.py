"""ns_orthogonalize_noalloc: the Newton–Schulz entry point that allocates nothing.

It is for callers that cannot call cudaMalloc (a host framework that owns every device
allocation through its own pool, or a latency-critical loop that must not pay
cudaMalloc's implicit device synchronisation): they pass only inputs and outputs, and the
scratch is a fixed device array inside libmao. These tests call it through the C ABI and
compare it with ns_orthogonalize, which takes a caller-provided workspace: both run the
same deterministic kernels on the same plan, so their outputs must be equal bit for bit.
They are also compared with the fp64 oracle at the Newton–Schulz tolerances.

This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from matrix_aware_optimizers_gb300 import _abi

QUINTIC = (3.4445, -4.7750, 2.0315)
TOL = {_abi.MAO_F32: 1e-4, _abi.MAO_BF16: 2e-2}  # the tolerances of the other NS tests


def _mats(ts):
    arr = (_abi.MaoMat * len(ts))()
    for i, t in enumerate(ts):
        dt = _abi.MAO_BF16 if t.dtype == torch.bfloat16 else _abi.MAO_F32
        arr[i] = _abi.MaoMat(t.data_ptr(), t.shape[0], t.shape[1], t.stride(0), dt, 0)
    return arr


def _coeffs():
    return (ctypes.c_float * 3)(*QUINTIC)


def _words(x):
    return torch.zeros((x.shape[0] * x.shape[1] + 31) // 32, dtype=torch.int32, device=x.device)


def _bits_arg(bits):
    if bits is None:
        return None
    return (ctypes.c_void_p * len(bits))(*[b.data_ptr() for b in bits])


def _existing(lib, ins, compute, stream, with_bits=False):
    outs = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for x in ins]
    bits = [_words(x) for x in ins] if with_bits else None
    m = _mats(ins)
    n = lib.ns_workspace_bytes(m, len(ins), compute)
    ws = torch.empty(n, dtype=torch.uint8, device=ins[0].device)
    st = lib.ns_orthogonalize(m, _mats(outs), len(ins), 5, _coeffs(), 0, 1e-7, compute,
                              _bits_arg(bits), ctypes.c_void_p(ws.data_ptr()), n, stream)
    assert st == _abi.MAO_OK, lib.mao_status_string(st)
    return outs, bits


def _noalloc(lib, ins, compute, stream, with_bits=False):
    outs = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for x in ins]
    bits = [_words(x) for x in ins] if with_bits else None
    st = lib.ns_orthogonalize_noalloc(_mats(ins), _mats(outs), len(ins), 5, _coeffs(), 0, 1e-7,
                                      compute, _bits_arg(bits), stream)
    assert st == _abi.MAO_OK, lib.mao_status_string(st)
    return outs, bits


def _rel_to_oracle(x, u):
    want = oracle.newton_schulz(x.float().cpu().numpy(), 5, QUINTIC, 1e-7)
    got = u.double().cpu().numpy()
    return float(np.linalg.norm(got - want) / np.linalg.norm(want))


@pytest.mark.gpu
@pytest.mark.parametrize("compute", [_abi.MAO_BF16, _abi.MAO_F32])
def test_noalloc_matches_workspace_entry_point_twice(lib, cuda, compute):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = torch.bfloat16 if compute == _abi.MAO_BF16 else torch.float32
    g = torch.Generator(device=cuda)
    g.manual_seed(99)
    # Three calls in a row on the shared scratch. The first leaves large values behind
    # (inputs scaled by 1e4); the next ones use other shapes, one of them with row lengths
    # that are not multiples of 64 (the zero-padded columns of the scratch layout), and
    # the last also writes the packed signs. Stale scratch contents would show up as a
    # difference from the call with a fresh workspace.
    calls = [
        ([torch.randn((256, 640), generator=g, device=cuda).mul(1e4).to(dt),
          torch.randn((640, 256), generator=g, device=cuda).mul(1e4).to(dt)], False),
        ([torch.randn((300, 500), generator=g, device=cuda).to(dt)], False),
        ([torch.randn((384, 512), generator=g, device=cuda).to(dt),
          torch.randn((500, 300), generator=g, device=cuda).to(dt)], True),
    ]
    for ins, with_bits in calls:
        got, got_bits = _noalloc(lib, ins, compute, stream, with_bits)
        want, want_bits = _existing(lib, ins, compute, stream, with_bits)
        assert lib.mao_sync_status(stream) == _abi.MAO_OK
        for x, a, b in zip(ins, got, want):
            assert torch.equal(a, b), tuple(x.shape)
            assert _rel_to_oracle(x, a) <= TOL[compute], tuple(x.shape)
        if with_bits:
            for a, b in zip(got_bits, want_bits):
                assert torch.equal(a, b)


def test_noalloc_rejects_batches_beyond_the_scratch_size(lib):
    limit = lib.ns_noalloc_workspace_bytes()
    assert limit == 16 * 1024 * 1024
    # 2048 x 2048 needs ~32 MiB of scratch in bf16: refused before any device work
    big = (_abi.MaoMat * 1)(_abi.MaoMat(0x10000, 2048, 2048, 2048, _abi.MAO_BF16, 0))
    out = (_abi.MaoMat * 1)(_abi.MaoMat(0x10000, 2048, 2048, 2048, _abi.MAO_F32, 0))
    assert lib.ns_workspace_bytes(big, 1, _abi.MAO_BF16) > limit
    st = lib.ns_orthogonalize_noalloc(big, out, 1, 5, _coeffs(), 0, 1e-7, _abi.MAO_BF16,
                                      None, None)
    assert st == _abi.MAO_ERR_WORKSPACE
