"""ns_orthogonalize_noalloc: the Newton–Schulz entry point that allocates nothing.

It is for callers that cannot call cudaMalloc (a host framework that owns every device
allocation through its own pool, or a latency-critical loop that must not pay
cudaMalloc's implicit device synchronisation): they pass only inputs and outputs, and the
scratch is a fixed 16 MiB device array inside libmao. These tests call it through the C
ABI and compare it with ns_orthogonalize, which takes a caller-provided workspace.

This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

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


def _existing(lib, ins, compute, stream):
    outs = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for x in ins]
    m = _mats(ins)
    n = lib.ns_workspace_bytes(m, len(ins), compute)
    ws = torch.empty(n, dtype=torch.uint8, device=ins[0].device)
    st = lib.ns_orthogonalize(m, _mats(outs), len(ins), 5, _coeffs(), 0, 1e-7, compute, None,
                              ctypes.c_void_p(ws.data_ptr()), n, stream)
    assert st == _abi.MAO_OK, lib.mao_status_string(st)
    return outs


def _noalloc(lib, ins, compute, stream):
    outs = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for x in ins]
    st = lib.ns_orthogonalize_noalloc(_mats(ins), _mats(outs), len(ins), 5, _coeffs(), 0, 1e-7,
                                      compute, None, stream)
    assert st == _abi.MAO_OK, lib.mao_status_string(st)
    return outs


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.gpu
@pytest.mark.parametrize("compute", [_abi.MAO_BF16, _abi.MAO_F32])
def test_noalloc_matches_workspace_entry_point_twice(lib, cuda, compute):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = torch.bfloat16 if compute == _abi.MAO_BF16 else torch.float32
    g = torch.Generator(device=cuda)
    g.manual_seed(99)
    # first call: two matrices of different shapes; second call: new inputs and another
    # shape, so stale scratch contents from the first call would show up as a mismatch
    calls = [
        [torch.randn((256, 640), generator=g, device=cuda).to(dt),
         torch.randn((640, 256), generator=g, device=cuda).to(dt)],
        [torch.randn((384, 512), generator=g, device=cuda).to(dt)],
    ]
    for ins in calls:
        got = _noalloc(lib, ins, compute, stream)
        want = _existing(lib, ins, compute, stream)
        assert lib.mao_sync_status(stream) == _abi.MAO_OK
        for a, b in zip(got, want):
            assert _rel(a, b) <= TOL[compute]


def test_noalloc_rejects_batches_beyond_the_scratch_size(lib):
    # 2048 x 2048 needs ~32 MiB of scratch in bf16: refused before any device work
    big = (_abi.MaoMat * 1)(_abi.MaoMat(0x10000, 2048, 2048, 2048, _abi.MAO_BF16, 0))
    out = (_abi.MaoMat * 1)(_abi.MaoMat(0x10000, 2048, 2048, 2048, _abi.MAO_F32, 0))
    assert lib.ns_workspace_bytes(big, 1, _abi.MAO_BF16) > _abi.NOALLOC_WORKSPACE_BYTES
    st = lib.ns_orthogonalize_noalloc(big, out, 1, 5, _coeffs(), 0, 1e-7, _abi.MAO_BF16,
                                      None, None)
    assert st == _abi.MAO_ERR_WORKSPACE
