"""The library's calls can be captured in a CUDA graph and replayed.

A whole optimizer step (momentum, Newton–Schulz with its staging and tensor-core launches,
vote, update; or one Dion call) is captured once, replayed, and compared bit for bit with
the same step launched eagerly on identical inputs. Capture-safe means: no host
synchronisation, no allocation and no per-call host state inside a call.
"""

import pytest
import torch

import bench
import matrix_aware_optimizers_gb300 as mao
from matrix_aware_optimizers_gb300 import workloads

pytestmark = pytest.mark.gpu


def _clone_inputs(inp):
    return {k: [t.clone() for t in v] for k, v in inp.items()}


@pytest.mark.parametrize("cfg,shapes", [(2, [(768, 2304), (768, 768), (3072, 768)]),
                                        (1, None), (6, [(768, 2304), (768, 768)])])
def test_graph_replay_equals_eager(cuda, cfg, shapes):
    wl = workloads.workload(cfg)
    base = workloads.generate(wl, cuda, shapes=shapes)
    eager = bench.Step(wl, _clone_inputs(base), cuda)
    graphed = bench.Step(wl, _clone_inputs(base), cuda)
    # the first call of each kind runs outside the capture (one-time device attributes)
    warm = bench.Step(wl, _clone_inputs(base), cuda)
    warm()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        graphed()
    torch.cuda.synchronize()
    for _ in range(3):
        eager()
        g.replay()
    torch.cuda.synchronize()
    mao.sync_status()
    for a, b in zip(eager.W, graphed.W):
        assert torch.equal(a, b)
    for a, b in zip(eager.M, graphed.M):
        assert torch.equal(a, b)
    if cfg == 6:
        for a, b in zip(eager.Q, graphed.Q):
            assert torch.equal(a, b)
