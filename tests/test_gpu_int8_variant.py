"""GPU parity of the Sign-Muon variants beside the 1-bit path ([SignMuon] §2 steps 3 and 5).

  * int8 signs (sign_int8) and the integer SUM + threshold vote (majority_vote_int8) have
    unique results: bit-exact against the oracle, on every output (sums, S_bar, packed vote);
  * the packed vote of the int8 variant equals majority_vote_packed on the same signs;
  * the post-vote polar step is ns_orthogonalize on an int8 or packed-sign input: the staged
    values are exact, so the three encodings of one S_bar (int8, packed words, bf16 +-1) give
    identical outputs, and the result matches the oracle within the Newton–Schulz tolerances
    (relative Frobenius 1e-4 fp32 / 2e-2 bf16);
  * whole int8-variant steps (with and without the polar step) through bench.Step, the
    launch sequence the benchmark times, at a small size and at the 4096 x 4096, 8-worker size.
"""

import numpy as np
import pytest
import torch

import bench
import oracle
from helpers import bits_of, check_sign_agreement, rel_fro, to_np, words_np
from matrix_aware_optimizers_gb300 import workloads
import matrix_aware_optimizers_gb300 as mao

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
TOL = {"f32": 1e-4, "bf16": 2e-2}


def _special_values(gen, shape, dtype, device):
    U = torch.randn(shape, generator=gen)
    flat = U.view(-1)
    n = flat.numel()
    idx = torch.randperm(n, generator=gen)
    flat[idx[: n // 10]] = 0.0
    flat[idx[n // 10: n // 5]] = -0.0
    if n >= 20:
        flat[idx[n // 5]] = float("nan")
        flat[idx[n // 5 + 1]] = -float("inf")
        flat[idx[n // 5 + 2]] = 1e-40
        flat[idx[n // 5 + 3]] = -1e-40
    return U.to(dtype).to(device)


def _i8(t):
    return t.detach().cpu().numpy().astype(np.int8)


def _rand_signs(gen, Wn, stride, n):
    s = torch.randint(0, 2, (Wn, stride), generator=gen, dtype=torch.int8) * 2 - 1
    return s.to(torch.int8)


# ------------------------------------------------------------------ sign_int8

@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 8), (7, 13), (64, 128), (33, 96), (4096, 64), (5, 1000),
                                   (3, 16)])
def test_sign_int8_bit_exact(cuda, dt, shape):
    gen = torch.Generator().manual_seed(41)
    U = _special_values(gen, shape, DT[dt], cuda)
    s = mao.sign_int8(U)
    torch.cuda.synchronize()
    assert np.array_equal(_i8(s), oracle.sign_of(to_np(U)))


@pytest.mark.parametrize("ld", [72, 70, 65])
def test_sign_int8_strided(cuda, ld):
    gen = torch.Generator().manual_seed(42)
    big = torch.randn((40, ld), generator=gen).to(torch.bfloat16).to(cuda)
    U = big[:, :64]
    s = mao.sign_int8(U)
    torch.cuda.synchronize()
    assert np.array_equal(_i8(s), oracle.sign_of(to_np(U)))


def test_sign_int8_matches_packed_signs(cuda):
    gen = torch.Generator().manual_seed(43)
    U = _special_values(gen, (96, 320), torch.float32, cuda)
    s = mao.sign_int8(U)
    bits = mao.sign_pack_bits(U)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(words_np(bits), U.numel()), (_i8(s).reshape(-1) > 0).astype(np.uint8))


# ------------------------------------------------------------- majority_vote_int8

def _check_vote(s, n, sums, sbar, vote):
    Wn = s.shape[0]
    S = [_i8(s[m, :n]) for m in range(Wn)]
    want_sum, want_sbar = oracle.int8_sum_vote(S)
    if sums is not None:
        assert np.array_equal(_i8(sums).astype(np.int64), want_sum)
    if sbar is not None:
        assert np.array_equal(_i8(sbar), want_sbar)
    if vote is not None:
        assert np.array_equal(words_np(vote)[: (n + 31) // 32], oracle.pack_signs(want_sbar))


@pytest.mark.parametrize("Wn", [1, 2, 3, 8, 33, 127])
@pytest.mark.parametrize("n", [1, 31, 32, 33, 4096, 100003])
def test_vote_int8_bit_exact(cuda, Wn, n):
    gen = torch.Generator().manual_seed(1000 * Wn + n % 997)
    stride = (n + 15) // 16 * 16
    s = _rand_signs(gen, Wn, stride, n).to(cuda)
    sums, sbar, vote = mao.majority_vote_int8(s, n, sum=True, s_bar=True, vote=True)
    torch.cuda.synchronize()
    _check_vote(s, n, sums, sbar, vote)


@pytest.mark.parametrize("Wn", [2, 7])
def test_vote_int8_equals_packed_vote(cuda, Wn):
    # the two aggregation variants decide identically on the same worker signs
    gen = torch.Generator().manual_seed(44)
    n = 5000
    s = _rand_signs(gen, Wn, n, n).to(cuda)
    _, _, vote8 = mao.majority_vote_int8(s, n, vote=True)
    nw = mao.packed_words(1, n)
    words = torch.zeros((Wn, nw), dtype=torch.int32, device=cuda)
    for m in range(Wn):
        mao.sign_pack_bits(s[m].float().view(1, n), words[m])
    vote1 = mao.majority_vote_packed(words, n)
    torch.cuda.synchronize()
    assert torch.equal(vote8[:nw], vote1[:nw])


@pytest.mark.parametrize("offset,extra", [(1, 3), (0, 5), (3, 0)])
def test_vote_int8_unaligned_and_subsets(cuda, offset, extra):
    # byte-path launches: buffers off the 16-byte grid, strides not multiples of 16
    gen = torch.Generator().manual_seed(45)
    Wn, n = 5, 777
    stride = n + extra
    raw = _rand_signs(gen, 1, Wn * stride + offset + 16, 0).to(cuda)
    s = raw[0, offset: offset + Wn * stride].view(Wn, stride)
    out = torch.zeros(n + 16, dtype=torch.int8, device=cuda)
    sums_only = out[offset: offset + n]
    r = mao.majority_vote_int8(s, n, sum=sums_only)
    assert r[1] is None and r[2] is None
    _, _, vote = mao.majority_vote_int8(s, n, vote=True)
    _, sbar, _ = mao.majority_vote_int8(s, n, s_bar=True)
    torch.cuda.synchronize()
    _check_vote(s, n, sums_only, sbar, vote)


def test_vote_int8_general_integers(cuda):
    # entries other than +-1 are summed as integers (here |sum| <= 3 * 40 < 128)
    gen = torch.Generator().manual_seed(46)
    Wn, n = 40, 4099
    s = (torch.randint(-3, 4, (Wn, n + 13), generator=gen)).to(torch.int8).to(cuda)
    sums, sbar, vote = mao.majority_vote_int8(s, n, sum=True, s_bar=True, vote=True)
    torch.cuda.synchronize()
    _check_vote(s, n, sums, sbar, vote)
    assert np.any(_i8(sums) == 0)  # ties occur and give +1 (checked through the oracle)


def test_vote_int8_rejects_bad_arguments(cuda):
    s = torch.ones((128, 64), dtype=torch.int8, device=cuda)
    with pytest.raises(mao.MaoError):
        mao.majority_vote_int8(s, 64, vote=True)          # 128 workers
    with pytest.raises(mao.MaoError):
        mao.majority_vote_int8(s[:2], 64)                 # no output requested
    with pytest.raises(mao.MaoError):
        mao.majority_vote_int8(s.view(256, 32)[:2], 64, vote=True)  # stride 32 < n


# ------------------------------------------------- post-vote polar: int8 / packed inputs

@pytest.mark.parametrize("compute", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(64, 128), (256, 640), (300, 1000), (200, 72), (33, 96)])
def test_polar_of_sign_matrix_all_encodings(cuda, compute, shape):
    gen = torch.Generator().manual_seed(47)
    R, C = shape
    sbar = (torch.randint(0, 2, shape, generator=gen) * 2 - 1).to(torch.int8).to(cuda)
    words = mao.sign_pack_bits(sbar.float())
    outs = [torch.empty(shape, dtype=torch.float32, device=cuda) for _ in range(3)]
    mao.ns_orthogonalize(sbar, outs[0], 5, mao.QUINTIC, 1e-7, compute)
    mao.ns_orthogonalize(mao.PackedSigns(words, R, C), outs[1], 5, mao.QUINTIC, 1e-7, compute)
    mao.ns_orthogonalize(sbar.to(torch.bfloat16), outs[2], 5, mao.QUINTIC, 1e-7, compute)
    mao.sync_status()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    want = oracle.post_vote_polar(_i8(sbar), 5, oracle.QUINTIC, 1e-7)
    assert rel_fro(to_np(outs[0]), want) <= TOL[compute]


def test_polar_of_int8_strided_input(cuda):
    gen = torch.Generator().manual_seed(48)
    big = (torch.randint(0, 2, (128, 200), generator=gen) * 2 - 1).to(torch.int8).to(cuda)
    for cols in (192, 190):  # 8-byte loads, then the element path
        x = big[:, :cols]
        out = torch.empty((128, cols), dtype=torch.float32, device=cuda)
        mao.ns_orthogonalize(x, out, 5, mao.QUINTIC, 1e-7, "bf16")
        mao.sync_status()
        want = oracle.post_vote_polar(_i8(x), 5, oracle.QUINTIC, 1e-7)
        assert rel_fro(to_np(out), want) <= TOL["bf16"]


# ------------------------------------------------------------ whole int8-variant steps

def _run_variant_step(wl, dev, post_polar):
    inp = workloads.generate(wl, dev)
    step = bench.Step(wl, inp, dev, "int8", post_polar)
    step.momentum()
    step.ns()
    M_after = [m.clone() for m in step.M]
    W_before = [w.clone() for w in step.W]
    step.update()
    mao.sync_status()
    return step, M_after, W_before


@pytest.mark.parametrize("post_polar", [False, True])
def test_int8_variant_step_small(cuda, post_polar):
    wl = workloads.workload(1)
    step, M_after, W_before = _run_variant_step(wl, cuda, post_polar)
    R, C = wl.shapes[0]
    n = R * C
    S = []
    for m in range(wl.workers):
        u_ref = oracle.newton_schulz(to_np(M_after[m]), wl.steps, wl.coeffs, wl.eps)
        u = to_np(step.U[m])
        assert rel_fro(u, u_ref) <= TOL[wl.compute]
        s = _i8(step.s8[m, :n])
        assert np.array_equal(s, oracle.sign_of(u).reshape(-1))  # signs of the stored U
        check_sign_agreement(u, u_ref, (s > 0).astype(np.uint8), strict_rms=1e-3)
        S.append(s)
    _, S_bar = oracle.int8_sum_vote(S)
    S_bar = S_bar.reshape(R, C)
    wstore = "bf16" if wl.w_dtype == torch.bfloat16 else "f32"
    if post_polar:
        assert np.array_equal(_i8(step.sbar).reshape(R, C), S_bar)
        ub = to_np(step.U_bar)
        assert rel_fro(ub, oracle.post_vote_polar(S_bar, wl.steps, wl.coeffs, wl.eps)) <= TOL[wl.compute]
        assert np.array_equal(to_np(step.W[0]), oracle.apply_update(to_np(W_before[0]), ub, wl.lr, wstore))
    else:
        assert np.array_equal(words_np(step.vote)[: (n + 31) // 32], oracle.pack_signs(S_bar))
        assert np.array_equal(to_np(step.W[0]), oracle.apply_update(to_np(W_before[0]), S_bar, wl.lr, wstore))


@pytest.mark.parametrize("post_polar", [False, True])
def test_int8_variant_step_4096_w8_full(cuda, post_polar):
    wl = workloads.workload(3)
    step, M_after, W_before = _run_variant_step(wl, cuda, post_polar)
    R, C = wl.shapes[0]
    n = R * C
    S = [_i8(step.s8[m, :n]) for m in range(wl.workers)]
    # sampled worker: int8 signs equal the signs of its stored U, U within tolerance
    u = to_np(step.U[0])
    assert np.array_equal(S[0], oracle.sign_of(u).reshape(-1))
    u_ref = oracle.newton_schulz(to_np(M_after[0]), wl.steps, wl.coeffs, wl.eps)
    assert rel_fro(u, u_ref) <= TOL["bf16"]
    sums, S_bar = oracle.int8_sum_vote(S)
    assert np.all(np.abs(sums) <= wl.workers)
    S_bar = S_bar.reshape(R, C)
    if post_polar:
        assert np.array_equal(_i8(step.sbar).reshape(R, C), S_bar)
        # the 4096 x 4096 polar step is checked through its properties: S_bar's singular
        # vectors are kept, singular values land in the quintic's output band
        ub = step.U_bar.float()
        gram = (ub @ ub.t()).double()
        ev = torch.linalg.eigvalsh(gram).clamp_min(0).sqrt().cpu().numpy()
        assert ev.max() <= 1.2024 * 1.02
        assert np.mean(ev >= 0.6798 * 0.98) >= 0.95
        # the update is bit-exact on the stored direction (sampled rows)
        rows = [0, 1, 2047, 4095]
        want = oracle.apply_update(to_np(W_before[0][rows]), to_np(step.U_bar[rows]), wl.lr, "bf16")
        assert np.array_equal(to_np(step.W[0][rows]), want)
    else:
        assert np.array_equal(words_np(step.vote)[: n // 32], oracle.pack_signs(S_bar))
        assert np.array_equal(to_np(step.W[0]), oracle.apply_update(to_np(W_before[0]), S_bar, wl.lr, "bf16"))
