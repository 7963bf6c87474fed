"""GPU checks of the fused Muon step (muon_step: momentum, Newton–Schulz, update in one call).

* Against the composed calls (muon_momentum_update, ns_orthogonalize into an fp32 U,
  apply_update): M and W bit-identical. The fused path feeds the same fp32 accumulator values
  into the same fmaf(-lr, u, w) that apply_update computes from the stored fp32 U.
* Against the fp64 oracle ([SignMuon] §2 "Fluxo Algorítmico"; momentum form from [Dion]):
  M bit-exact; the change of W within the bf16 Newton–Schulz tolerance (relative Frobenius
  2e-2 of lr*U) plus one rounding of W to its storage type.
"""

import numpy as np
import pytest
import torch

import matrix_aware_optimizers_gb300 as mao
import oracle
from helpers import rel_fro, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-2
DT = {"f32": torch.float32, "bf16": torch.bfloat16}
EPS = {"f32": 2.0 ** -24, "bf16": 2.0 ** -8}  # unit roundoff of the storage type


def _inputs(gen, shapes, wdt, mdt, gdt, dev):
    W = [(torch.randn(s, generator=gen) * 0.02).to(DT[wdt]).to(dev) for s in shapes]
    M = [(torch.randn(s, generator=gen) * 0.01).to(DT[mdt]).to(dev) for s in shapes]
    G = [(torch.randn(s, generator=gen) * 0.02).to(DT[gdt]).to(dev) for s in shapes]
    return W, M, G


SHAPES = [(256, 640), (640, 256), (384, 384), (300, 700), (256, 640), (130, 520)]


@pytest.mark.parametrize("wdt,mdt,gdt", [("bf16", "bf16", "bf16"), ("bf16", "f32", "bf16"),
                                         ("f32", "f32", "f32")])
@pytest.mark.parametrize("steps", [5, 1])
def test_muon_step_matches_composed_calls(cuda, wdt, mdt, gdt, steps):
    gen = torch.Generator().manual_seed(60 + steps)
    W, M, G = _inputs(gen, SHAPES, wdt, mdt, gdt, cuda)
    W2, M2 = [w.clone() for w in W], [m.clone() for m in M]
    mu, lr = 0.95, 0.02
    mao.muon_step(W, M, G, mu, lr, steps, mao.QUINTIC, 1e-7)
    mao.sync_status()
    # composed: momentum, Newton-Schulz into fp32 U, update from U
    mao.muon_momentum_update(M2, G, mu)
    U = [torch.empty(m.shape, dtype=torch.float32, device=cuda) for m in M2]
    mao.ns_orthogonalize(M2, U, steps, mao.QUINTIC, 1e-7, "bf16")
    mao.apply_update(W2, lr, U=U)
    mao.sync_status()
    for a, b in zip(M, M2):
        assert torch.equal(a, b)
    for a, b in zip(W, W2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("wdt,mdt", [("bf16", "bf16"), ("bf16", "f32")])
def test_muon_step_oracle_parity(cuda, wdt, mdt):
    gen = torch.Generator().manual_seed(70)
    shapes = [(256, 640), (640, 256), (384, 384), (300, 700)]
    W, M, G = _inputs(gen, shapes, wdt, mdt, "bf16", cuda)
    host = [[to_np(t) for t in ts] for ts in (W, M, G)]
    mu, lr = 0.95, 0.5  # a large lr makes the update dominate W's rounding
    coeffs = [mao.QUINTIC] * 4 + [(1.5, -0.5, 0.0)]  # per-step coefficients
    mao.muon_step(W, M, G, mu, lr, 5, coeffs, 1e-7)
    mao.sync_status()
    out = oracle.muon_step(host[0], host[1], host[2], mu, lr, steps=5, coeffs=coeffs,
                           m_store="bf16" if mdt == "bf16" else "f32")
    for k in range(len(shapes)):
        assert np.array_equal(to_np(M[k]), out["M"][k])
        w0, w_new, w_ref = host[0][k].astype(np.float64), to_np(W[k]).astype(np.float64), out["W"][k]
        err = np.linalg.norm(w_new - w_ref)
        assert err <= TOL * np.linalg.norm(w0 - w_ref) + EPS[wdt] * np.linalg.norm(w_ref)


def test_muon_step_rejects_bad_arguments(cuda):
    W = torch.zeros((64, 96), dtype=torch.bfloat16, device=cuda)
    M, G = W.clone(), W.clone()
    with pytest.raises(mao.MaoError):  # fp32 compute: not fused
        mao.muon_step(W, M, G, 0.9, 0.1, compute="f32",
                      ws=torch.empty(1 << 20, dtype=torch.uint8, device=cuda))
    with pytest.raises(mao.MaoError):  # shapes differ
        mao.muon_step(W, M, torch.zeros((64, 95), dtype=torch.bfloat16, device=cuda), 0.9, 0.1)
    with pytest.raises(mao.MaoError):  # workspace too small
        mao.muon_step(W, M, G, 0.9, 0.1, ws=torch.empty(256, dtype=torch.uint8, device=cuda))


def test_muon_step_out_of_place(cuda):
    gen = torch.Generator().manual_seed(75)
    W, M, G = _inputs(gen, SHAPES, "bf16", "bf16", "bf16", cuda)
    W0 = [w.clone() for w in W]
    M2 = [m.clone() for m in M]
    W_out = [torch.full_like(w, float("nan")) for w in W]
    mao.muon_step(W, M, G, 0.95, 0.02, W_out=W_out)
    W_in_place = [w.clone() for w in W0]
    mao.muon_step(W_in_place, M2, G, 0.95, 0.02)
    W_alias = [w.clone() for w in W0]
    mao.sync_status()
    for a, b in zip(W, W0):
        assert torch.equal(a, b)  # W only read
    for a, b in zip(W_out, W_in_place):
        assert torch.equal(a, b)
    for a, b in zip(M, M2):
        assert torch.equal(a, b)
    # W_out aliasing W is the in-place update
    gen = torch.Generator().manual_seed(75)
    _, Ma, Ga = _inputs(gen, SHAPES, "bf16", "bf16", "bf16", cuda)
    mao.muon_step(W_alias, Ma, Ga, 0.95, 0.02, W_out=W_alias)
    mao.sync_status()
    for a, b in zip(W_alias, W_in_place):
        assert torch.equal(a, b)


@pytest.mark.parametrize("shape,dt,compute", [((64, 128), "f32", "f32"),
                                              ((128, 64), "f32", "f32"),
                                              ((96, 160), "bf16", "f32"),
                                              ((300, 500), "bf16", "bf16"),
                                              ((500, 300), "bf16", "bf16")])
def test_sign_muon_step_equals_composed_calls(cuda, shape, dt, compute):
    """sign_muon_step (one call) against muon_momentum_update, ns_orthogonalize with packed
    signs, majority_vote_packed and apply_update: M, every worker's words, the vote and W bit
    for bit ([SignMuon] §2 "Fluxo Algorítmico", steps 1-4)."""
    g = torch.Generator()
    g.manual_seed(21)
    Wn = 4
    R, C = shape
    W0 = (torch.randn(shape, generator=g) * 0.02).to(DT[dt]).to(cuda)
    M0 = torch.randn(shape, generator=g).to(DT[dt]).to(cuda)
    Gs = [torch.randn(shape, generator=g).to(DT[dt]).to(cuda) for _ in range(Wn)]
    nw = mao.packed_words(R, C)
    stride = (nw + 3) // 4 * 4
    # one call
    W1, M1 = W0.clone(), [M0.clone() for _ in range(Wn)]
    words1 = torch.zeros((Wn, stride), dtype=torch.int32, device=cuda)
    vote1 = torch.zeros(stride, dtype=torch.int32, device=cuda)
    mao.sign_muon_step(W1, M1, Gs, words1, vote1, 0.95, 1e-3, 5, mao.QUINTIC, 1e-7, compute)
    # the composed calls
    W2, M2 = W0.clone(), [M0.clone() for _ in range(Wn)]
    words2 = torch.zeros((Wn, stride), dtype=torch.int32, device=cuda)
    mao.muon_momentum_update(M2, Gs, 0.95)
    mao.ns_orthogonalize(M2, None, 5, mao.QUINTIC, 1e-7, compute,
                         sign_bits=[words2[m, :nw] for m in range(Wn)])
    vote2 = mao.majority_vote_packed(words2, R * C)
    mao.apply_update(W2, 1e-3, vote=vote2)
    mao.sync_status()
    for a, b in zip(M1, M2):
        assert torch.equal(a, b)
    assert torch.equal(words1[:, :nw], words2[:, :nw])
    assert torch.equal(vote1[:nw], vote2[:nw])
    assert torch.equal(W1, W2)
    # and the vote against the oracle's vote of these words
    w = words2[:, :nw].cpu().numpy().view(np.uint32)
    assert np.array_equal(vote1[:nw].cpu().numpy().view(np.uint32), oracle.majority_vote(w, R * C))


@pytest.mark.parametrize("shape,workers,compute", [((520, 264), 4, "bf16"), ((37, 104), 9, "f32"),
                                                   ((1024, 512), 17, "bf16")])
def test_sign_muon_step_vote_update_blocks(cuda, shape, workers, compute):
    """The vote-and-update pass over several blocks of vote words, a partial last block, a
    last word with padding bits, and more than 8 workers (wider counters): vote and W bit for
    bit against majority_vote_packed and apply_update of the same words."""
    g = torch.Generator()
    g.manual_seed(24 + workers)
    R, C = shape
    W0 = (torch.randn(shape, generator=g) * 0.02).to(torch.bfloat16).to(cuda)
    M0 = torch.randn(shape, generator=g).to(torch.bfloat16).to(cuda)
    Gs = [torch.randn(shape, generator=g).to(torch.bfloat16).to(cuda) for _ in range(workers)]
    nw = mao.packed_words(R, C)
    stride = (nw + 3) // 4 * 4
    W1, M1 = W0.clone(), [M0.clone() for _ in range(workers)]
    words = torch.zeros((workers, stride), dtype=torch.int32, device=cuda)
    vote1 = torch.zeros(stride, dtype=torch.int32, device=cuda)
    mao.sign_muon_step(W1, M1, Gs, words, vote1, 0.95, 1e-3, 5, mao.QUINTIC, 1e-7, compute)
    vote2 = mao.majority_vote_packed(words, R * C)
    W2 = W0.clone()
    mao.apply_update(W2, 1e-3, vote=vote2)
    mao.sync_status()
    assert torch.equal(vote1[:nw], vote2[:nw])
    assert torch.equal(W1, W2)
    w = words[:, :nw].cpu().numpy().view(np.uint32)
    assert np.array_equal(vote1[:nw].cpu().numpy().view(np.uint32), oracle.majority_vote(w, R * C))


def test_sign_muon_step_prepared_call(cuda):
    """A prepared sign_muon_step (arguments marshalled once) called twice gives what two
    direct calls give, bit for bit."""
    g = torch.Generator()
    g.manual_seed(23)
    Wn, R, C = 4, 64, 128
    W0 = (torch.randn((R, C), generator=g) * 0.02).to(cuda)
    M0 = torch.randn((R, C), generator=g).to(cuda)
    G1 = [torch.randn((R, C), generator=g).to(cuda) for _ in range(Wn)]
    nw = mao.packed_words(R, C)
    stride = (nw + 3) // 4 * 4
    res = []
    for prepared in (False, True):
        W, M = W0.clone(), [M0.clone() for _ in range(Wn)]
        words = torch.zeros((Wn, stride), dtype=torch.int32, device=cuda)
        vote = torch.zeros(stride, dtype=torch.int32, device=cuda)
        args = (W, M, G1, words, vote, 0.95, 1e-3, 5, mao.QUINTIC, 1e-7, "f32")
        if prepared:
            call = mao.sign_muon_step(*args, prepare=True)
            call()
            call()
        else:
            mao.sign_muon_step(*args)
            mao.sign_muon_step(*args)
        mao.sync_status()
        res.append((W, M, words, vote))
    for a, b in zip(res[0], res[1]):
        for x, y in zip(a if isinstance(a, list) else [a], b if isinstance(b, list) else [b]):
            assert torch.equal(x, y)


def test_sign_muon_step_strided_weights(cuda):
    """The vote-and-update pass on W rows with padding (ld > cols, 20 columns: words span
    rows) gives the same W and words as on a contiguous W."""
    g = torch.Generator()
    g.manual_seed(22)
    Wn, R, C = 3, 48, 20
    base = (torch.randn((R, C), generator=g) * 0.02).to(cuda)
    Wpad = torch.zeros((R, C + 12), device=cuda)
    Wpad[:, :C] = base
    Wv = Wpad[:, :C]
    Wc = base.clone()
    M0 = torch.randn((R, C), generator=g).to(cuda)
    Gs = [torch.randn((R, C), generator=g).to(cuda) for _ in range(Wn)]
    nw = mao.packed_words(R, C)
    stride = (nw + 3) // 4 * 4
    out = []
    for W in (Wv, Wc):
        M = [M0.clone() for _ in range(Wn)]
        words = torch.zeros((Wn, stride), dtype=torch.int32, device=cuda)
        vote = torch.zeros(stride, dtype=torch.int32, device=cuda)
        mao.sign_muon_step(W, M, Gs, words, vote, 0.9, 1e-2, 5, mao.QUINTIC, 1e-7, "f32")
        out.append((words.clone(), vote.clone()))
    mao.sync_status()
    assert torch.equal(Wv, Wc)
    assert torch.equal(Wpad[:, C:], torch.zeros((R, 12), device=cuda))  # padding untouched
    assert torch.equal(out[0][0][:, :nw], out[1][0][:, :nw])
    assert torch.equal(out[0][1][:nw], out[1][1][:nw])


def test_muon_step_host_equals_muon_step(cuda):
    """muon_step_host (host gradients in, host weights out, through the C ABI) against
    muon_step on device data: M and W bit for bit, and the host copy of W' equal to the
    device result; two calls on two streams ordered by the events."""
    g = torch.Generator()
    g.manual_seed(31)
    shapes = [(256, 640), (640, 256), (384, 384)]
    W, M, G = _inputs(g, shapes, "bf16", "bf16", "bf16", cuda)
    # gradients in one device slab and one pinned host slab
    sizes = [r * c for r, c in shapes]
    g_dev = torch.empty(sum(sizes), dtype=torch.bfloat16, device=cuda)
    G_views, o = [], 0
    for (r, c), n in zip(shapes, sizes):
        G_views.append(g_dev[o:o + n].view(r, c))
        o += n
    g_host = torch.cat([x.reshape(-1).cpu() for x in G]).pin_memory()
    w_dev = torch.empty(sum(sizes), dtype=torch.bfloat16, device=cuda)
    W_out, o = [], 0
    for (r, c), n in zip(shapes, sizes):
        W_out.append(w_dev[o:o + n].view(r, c))
        o += n
    w_host = torch.empty(sum(sizes), dtype=torch.bfloat16).pin_memory()
    M1 = [m.clone() for m in M]
    s0, s1 = torch.cuda.Stream(), torch.cuda.Stream()
    ev0, ev1 = torch.cuda.Event(), torch.cuda.Event()
    ev0.record(s0)
    ev1.record(s1)
    s0.wait_stream(torch.cuda.current_stream())
    s1.wait_stream(torch.cuda.current_stream())
    # step 1 on s0 (W -> W_out), step 2 on s1 (W_out -> W) after step 1's compute
    W1 = [w.clone() for w in W]
    mao.muon_step_host(W1, M1, G_views, 0.95, 0.02, g_host, g_dev, w_host, w_dev, W_out=W_out,
                       stream=s0, record_event=ev0)
    mao.muon_step_host(W_out, M1, G_views, 0.95, 0.02, g_host, g_dev, w_host, w_dev, W_out=W1,
                       stream=s1, wait_event=ev0, record_event=ev1)
    torch.cuda.synchronize()
    mao.sync_status()
    # the same two steps on device data
    W2 = [w.clone() for w in W]
    M2 = [m.clone() for m in M]
    mao.muon_step(W2, M2, G, 0.95, 0.02)
    first = [w.clone() for w in W2]
    mao.muon_step(W2, M2, G, 0.95, 0.02)
    mao.sync_status()
    for a, b in zip(M1, M2):
        assert torch.equal(a, b)
    for a, b in zip(W1, W2):
        assert torch.equal(a, b)
    # the host copy holds the first call's W' (the second call's copy reads w_dev, which
    # still holds step 1's output: step 2 wrote W1)
    assert torch.equal(w_host, torch.cat([x.reshape(-1).cpu() for x in first]))
