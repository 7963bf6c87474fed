"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names what fixes the expected value: a hand-computed table under
tests/golden/, a closed form, a library routine, an invariant or brute force.
"""

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import rounding

QUINTIC = (3.4445, -4.7750, 2.0315)


# ----------------------------------------------------------------- rounding

def _read_table(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_bf16_rne_hand_table(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "bf16_rne.txt"))
    src = np.array([int(r[0], 16) for r in rows], dtype=np.uint32).view(np.float32)
    want = np.array([int(r[1], 16) for r in rows], dtype=np.uint32)
    got = oracle.bf16_rne(src).view(np.uint32) >> 16
    assert got.tolist() == want.tolist()


def test_bf16_rne_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),
        rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = oracle.bf16_rne(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def _round_fraction_to_f32(q):
    """Independent nearest-even rounding of an exact rational to fp32 (normal range)."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = math.floor(math.log2(q))
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    n = q / ulp
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(lo * ulp)


def test_fma_f32_matches_exact_rational():
    rng = np.random.default_rng(2)
    a = rng.standard_normal(3000).astype(np.float32)
    b = (rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000)).astype(np.float32)
    c = (rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000)).astype(np.float32)
    got = rounding.fma_f32(a, b, c)
    for i in range(a.size):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        assert float(got[i]) == _round_fraction_to_f32(exact), i


def test_fma_f32_double_rounding_traps():
    # a*b = 2^-24 (1 - 2^-46) exactly. With c = 1 + 2^-23 (odd last bit) the exact
    # sum lies just below the fp32 midpoint 1 + 3*2^-24; fp64 rounds it onto the
    # midpoint, and a naive second rounding would pick the even neighbour above.
    a = np.float32(2.0 ** -24 * (1 + 2.0 ** -23))
    b = np.float32(1 - 2.0 ** -23)
    c_odd = np.float32(1 + 2.0 ** -23)
    c_even = np.float32(1 + 2.0 ** -22)
    got = rounding.fma_f32(np.array([a, a]), np.array([b, b]), np.array([c_odd, c_even]))
    assert got[0] == np.float32(1 + 2.0 ** -23)          # stays below the midpoint
    assert got[1] == np.float32(1 + 2.0 ** -22)
    # exact ties go to even
    t = rounding.fma_f32(np.float32(2.0 ** -24), np.float32(1.0), np.float32(1 + 2.0 ** -23))
    assert t == np.float32(1 + 2.0 ** -22)


def test_momentum_hand_table(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "momentum_rounding.txt"))
    M = np.array([float(r[0]) for r in rows], np.float32)
    G = np.array([float(r[1]) for r in rows], np.float32)
    want = np.array([float(r[2]) for r in rows], np.float32)
    got = oracle.momentum(M, G, 0.95, "bf16")
    assert got.tolist() == want.tolist()
    assert oracle.momentum(np.float32(1.0), np.float32(0.0), 0.95, "f32") == np.float32(0.95)


def test_update_hand_table(golden_dir):
    rows = _read_table(os.path.join(golden_dir, "update_rounding.txt"))
    W = np.array([float(r[0]) for r in rows], np.float32)
    D = np.array([float(r[1]) for r in rows], np.float32)
    want = np.array([float(r[2]) for r in rows], np.float32)
    got = oracle.apply_update(W, D, 1e-3, "bf16")
    assert got.tolist() == want.tolist()


# ------------------------------------------------------------ Newton–Schulz

def _p(s, a, b, c):
    return a * s + b * s ** 3 + c * s ** 5


def _ns_by_svd(M, steps, coeffs, eps=1e-7):
    """Closed form: an odd matrix polynomial keeps singular vectors and maps sigma."""
    M = np.asarray(M, np.float64)
    Uv, s, Vt = np.linalg.svd(M, full_matrices=False)
    s = s / (np.linalg.norm(M, "fro") + eps)
    for _ in range(steps):
        s = _p(s, *coeffs)
    return (Uv * s) @ Vt


@pytest.mark.parametrize("shape", [(8, 8), (16, 40), (40, 16), (64, 128), (128, 64), (1, 9), (9, 1)])
@pytest.mark.parametrize("steps", [1, 5])
def test_ns_matches_svd_closed_form(shape, steps):
    rng = np.random.default_rng(sum(shape) * 7 + steps)
    M = rng.standard_normal(shape)
    got = oracle.newton_schulz(M, steps, QUINTIC)
    want = _ns_by_svd(M, steps, QUINTIC)
    assert np.linalg.norm(got - want) <= 1e-10 * np.linalg.norm(want)


def test_ns_per_step_coefficients():
    rng = np.random.default_rng(3)
    M = rng.standard_normal((12, 20))
    co = [(3.0, -3.2, 1.2), (2.0, -1.5, 0.5), QUINTIC]
    got = oracle.newton_schulz(M, 3, co)
    Uv, s, Vt = np.linalg.svd(M, full_matrices=False)
    s = s / (np.linalg.norm(M) + 1e-7)
    for t in co:
        s = _p(s, *t)
    assert np.allclose(got, (Uv * s) @ Vt, rtol=0, atol=1e-12)


@pytest.mark.parametrize("shape", [(6, 6), (5, 11), (11, 5)])
def test_cubic_ns_converges_to_polar_factor(shape):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(4)
    # well-conditioned input: normalised singular values >= 0.05
    Q1, _ = np.linalg.qr(rng.standard_normal((shape[0], shape[0])))
    Q2, _ = np.linalg.qr(rng.standard_normal((shape[1], shape[1])))
    k = min(shape)
    sig = np.linspace(1.0, 0.3, k)
    M = (Q1[:, :k] * sig) @ Q2[:, :k].T
    got = oracle.newton_schulz(M, 40, oracle.CUBIC)
    if shape[0] >= shape[1]:
        polar, _ = scipy_linalg.polar(M, side="right")
    else:
        polar = scipy_linalg.polar(M.T, side="right")[0].T
    assert np.abs(got - polar).max() <= 1e-12


def test_quintic_singular_value_band():
    rng = np.random.default_rng(5)
    M = rng.standard_normal((48, 96))
    U = oracle.newton_schulz(M, 5, QUINTIC)
    s_in = np.linalg.svd(M / (np.linalg.norm(M) + 1e-7), compute_uv=False)
    s_out = np.linalg.svd(U, compute_uv=False)
    assert s_in.min() >= 1.5e-3
    # p^5 maps [1.5e-3, 1] into [0.6798, 1.2024] (fixed points 0.8680, 1.2637)
    assert s_out.min() >= 0.6798 - 1e-9 and s_out.max() <= 1.2024 + 1e-9


def test_ns_invariants():
    rng = np.random.default_rng(6)
    M = rng.standard_normal((24, 40))
    U = oracle.newton_schulz(M, 5, QUINTIC)
    # transpose
    assert np.allclose(oracle.newton_schulz(M.T, 5, QUINTIC), U.T, atol=1e-12)
    # positive scale (up to eps)
    assert np.allclose(oracle.newton_schulz(37.5 * M, 5, QUINTIC), U, atol=1e-8)
    # signed permutations on both sides
    P = np.eye(24)[rng.permutation(24)] * rng.choice([-1, 1], 24)[:, None]
    Q = np.eye(40)[rng.permutation(40)] * rng.choice([-1, 1], 40)[:, None]
    assert np.allclose(oracle.newton_schulz(P @ M @ Q, 5, QUINTIC), P @ U @ Q, atol=1e-12)


def test_ns_zero_matrix_is_zero():
    Z = np.zeros((4, 7))
    assert np.array_equal(oracle.newton_schulz(Z, 5, QUINTIC), Z)


# ------------------------------------------------------------ sign and pack

def _read_pack_cases(path):
    cases, cur = [], {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            cur[key] = vals
            if key == "words":
                cases.append(cur)
                cur = {}
    return cases


def test_pack_hand_cases(golden_dir):
    for case in _read_pack_cases(os.path.join(golden_dir, "pack_signs.txt")):
        R, C = map(int, case["shape"])
        U = np.array([float(v) for v in case["values"]], np.float32).reshape(R, C)
        want = [int(w, 16) for w in case["words"]]
        S = oracle.sign_of(U)
        assert oracle.pack_signs(S).tolist() == want
        assert oracle.pack_signs_loop(S).tolist() == want


def test_pack_size_is_one_bit_per_entry():
    # 1 bit per entry: a 4096 x 4096 matrix packs into 2 MiB of words
    S = np.ones((4096, 4096), np.int8)
    words = oracle.pack_signs(S)
    assert words.nbytes == 4096 * 4096 // 8 == 2 * 1024 * 1024
    assert oracle.pack_signs(np.ones(33, np.int8)).tolist() == [0xFFFFFFFF, 1]


def test_pack_unpack_roundtrip_and_popcount():
    rng = np.random.default_rng(7)
    S = rng.choice(np.array([-1, 1], np.int8), 1000)
    w = oracle.pack_signs(S)
    assert np.array_equal(oracle.unpack_signs(w, 1000), S)
    assert sum(bin(int(x)).count("1") for x in w) == int((S > 0).sum())


# ------------------------------------------------------------------- vote

@pytest.mark.parametrize("Wn", range(1, 9))
def test_vote_exhaustive_brute_force(Wn):
    # every pattern of Wn signs at one entry; entries = all 2^Wn patterns
    patterns = list(itertools.product([-1, 1], repeat=Wn))
    n = len(patterns)
    words = np.stack([oracle.pack_signs(np.array([p[m] for p in patterns], np.int8))
                      for m in range(Wn)])
    vote = oracle.unpack_signs(oracle.majority_vote(words, n), n)
    for i, p in enumerate(patterns):
        plus, minus = p.count(1), p.count(-1)
        assert vote[i] == (1 if plus >= minus else -1)


def test_vote_single_worker_is_identity():
    rng = np.random.default_rng(8)
    S = rng.choice(np.array([-1, 1], np.int8), 777)
    w = oracle.pack_signs(S)[None, :]
    assert np.array_equal(oracle.majority_vote(w, 777), w[0])


def test_vote_random_up_to_16_workers():
    rng = np.random.default_rng(9)
    for Wn in (9, 12, 15, 16):
        S = rng.choice(np.array([-1, 1], np.int8), (Wn, 500))
        words = np.stack([oracle.pack_signs(s) for s in S])
        vote = oracle.unpack_signs(oracle.majority_vote(words, 500), 500)
        cnt = (S > 0).sum(0)
        assert np.array_equal(vote, np.where(2 * cnt >= Wn, 1, -1))


# ------------------------------------------------------------- composition

def test_sign_muon_step_composition():
    rng = np.random.default_rng(10)
    R, C, Wn = 6, 10, 3
    W = oracle.bf16_rne(rng.standard_normal((R, C)).astype(np.float32) * 0.02)
    Ms = [oracle.bf16_rne(rng.standard_normal((R, C)).astype(np.float32)) for _ in range(Wn)]
    Gs = [oracle.bf16_rne(rng.standard_normal((R, C)).astype(np.float32)) for _ in range(Wn)]
    out = oracle.sign_muon_step(W, Ms, Gs, 0.95, 1e-3, 5, QUINTIC, m_store="bf16", w_store="bf16")
    # independent route: momentum in fp64 (bf16 rounding tolerance), NS by SVD,
    # vote by counting, update by direct arithmetic
    tot = np.zeros((R, C), np.int64)
    for m in range(Wn):
        Mm = 0.95 * Ms[m].astype(np.float64) + Gs[m]
        assert np.allclose(out["M"][m], Mm, rtol=2 ** -8, atol=0)
        U = _ns_by_svd(out["M"][m], 5, QUINTIC)
        assert np.allclose(out["U"][m], U, atol=1e-10)
        tot += np.where(U < 0, -1, 1)
    S_bar = np.where(tot >= 0, 1, -1)
    assert np.array_equal(out["S_bar"], S_bar)
    W_ref = W.astype(np.float64) - 1e-3 * S_bar
    assert np.allclose(out["W"], W_ref, rtol=2 ** -8, atol=0)


def _read_sections(path):
    """Sections [name] of 'key values...' lines; matrix rows separated by ';'."""
    cases, cur = {}, None
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("["):
                cur = cases.setdefault(line.strip("[]"), {})
                continue
            key, rest = line.split(None, 1)
            if ";" in rest or key in ("M", "G", "M_new", "U", "W", "W_new"):
                cur[key] = np.array([[float(v) for v in row.split()] for row in rest.split(";")])
            else:
                vals = [float(v) for v in rest.split()]
                cur[key] = vals if len(vals) > 1 else vals[0]
    return cases


def test_muon_step_hand_table(golden_dir):
    """oracle.muon_step against hand-worked steps (tests/golden/muon_step_hand.txt): dyadic
    momentum with known singular values, the polynomial applied to them by hand, and the
    update W - eta U entry by entry (wide and tall orientations, cubic and quintic, eta as
    the fp32 value of lr)."""
    cases = _read_sections(os.path.join(golden_dir, "muon_step_hand.txt"))
    assert len(cases) == 5
    for name, c in cases.items():
        out = oracle.muon_step([c["W"]], [c["M"]], [c["G"]], c["mu"], c["lr"], int(c["steps"]),
                               tuple(c["coeffs"]), eps=0.0, m_store="f32")
        assert np.array_equal(out["M"][0], c["M_new"]), name
        assert np.allclose(out["U"][0], c["U"], rtol=0, atol=1e-15), name
        assert np.allclose(out["W"][0], c["W_new"], rtol=0, atol=1e-15), name
        # the same update through apply_update_f64 on the hand-worked U
        assert np.allclose(oracle.apply_update_f64(c["W"], c["U"], c["lr"]), c["W_new"],
                           rtol=0, atol=1e-15), name


def test_apply_update_f64_lr_is_fp32_value():
    # W - float32(lr) * D: lr = 0.02 is 10737418 * 2^-29 in fp32; with D = 1 and W = 0 the
    # fp64 result is exactly that value, negated
    got = oracle.apply_update_f64(np.zeros((1, 2)), np.array([[1.0, -2.0]]), 0.02)
    eta = 10737418 * 2.0 ** -29
    assert got.tolist() == [[-eta, 2 * eta]]
    assert eta != 0.02


@pytest.mark.parametrize("shape", [(24, 40), (40, 24), (32, 32)])
@pytest.mark.parametrize("m_store", ["f32", "bf16"])
def test_muon_step_matches_svd_route(shape, m_store):
    """oracle.muon_step against an independent route: the momentum built from bf16-exact
    dyadic inputs with mu = 1/2 (so mu M + G is exact in every precision and needs no
    rounding), the polar direction by the SVD closed form U diag(p^5(s/(||M||+eps))) V^T,
    and the update W - float32(lr) U by plain subtraction."""
    rng = np.random.default_rng(shape[0] * 100 + shape[1] + len(m_store))
    n = 3
    Ws = [rng.integers(-64, 65, shape) / 256.0 for _ in range(n)]
    Ms = [rng.integers(-32, 33, shape) / 64.0 for _ in range(n)]
    Gs = [rng.integers(-32, 33, shape) / 128.0 for _ in range(n)]
    lr = 0.02
    out = oracle.muon_step(Ws, Ms, Gs, 0.5, lr, 5, QUINTIC, m_store=m_store)
    eta = float(np.float32(lr))
    for i in range(n):
        M_new = 0.5 * Ms[i] + Gs[i]
        assert np.array_equal(out["M"][i], M_new)
        U = _ns_by_svd(M_new, 5, QUINTIC)
        assert np.linalg.norm(out["U"][i] - U) <= 1e-10 * np.linalg.norm(U)
        W_new = Ws[i] - eta * U
        assert np.linalg.norm(out["W"][i] - W_new) <= 1e-12 * np.linalg.norm(Ws[i] - W_new)
        # a sign slip (W + eta U) or a transposed direction would be far off
        assert np.linalg.norm(out["W"][i] - (Ws[i] + eta * U)) > 1.0 * eta * np.linalg.norm(U)


def test_dense_flop_count():
    # (4 m^2 n + 2 m^3) per iteration: 64 x 128, 5 steps
    assert oracle.ns_dense_flops(64, 128, 5) == 5 * (4 * 64 * 64 * 128 + 2 * 64 ** 3) == 13_107_200


# --------------------------------------------- int8 all-reduce variant, post-vote polar

@pytest.mark.parametrize("Wn", [1, 2, 3, 4, 7, 8])
def test_int8_sum_vote_brute_force_and_bit_vote(Wn):
    patterns = np.array(list(itertools.product([-1, 1], repeat=Wn)), np.int8)  # [2^Wn][Wn]
    S = [patterns[:, m] for m in range(Wn)]
    sums, vote = oracle.int8_sum_vote(S)
    for i, p in enumerate(patterns):
        assert sums[i] == int(sum(int(x) for x in p))
        assert vote[i] == (1 if list(p).count(1) >= list(p).count(-1) else -1)
    # the int8 all-reduce variant and the 1-bit all-gather variant decide identically
    words = np.stack([oracle.pack_signs(s) for s in S])
    bits_vote = oracle.unpack_signs(oracle.majority_vote(words, len(patterns)), len(patterns))
    assert np.array_equal(vote, bits_vote)


def test_post_vote_polar_is_ns_of_sign_matrix():
    rng = np.random.default_rng(11)
    S_bar = rng.choice(np.array([-1, 1], np.int8), (12, 20))
    got = oracle.post_vote_polar(S_bar, 5, QUINTIC)
    assert np.linalg.norm(got - _ns_by_svd(S_bar.astype(np.float64), 5, QUINTIC)) <= 1e-10 * np.linalg.norm(got)


@pytest.mark.parametrize("Wn", [2, 3, 5])
def test_sign_muon_step_variants_agree(Wn):
    # the all-reduce (int8) and all-gather (1-bit) variants are two encodings of one vote
    rng = np.random.default_rng(20 + Wn)
    R, C = 7, 9
    W = rng.standard_normal((R, C)).astype(np.float32) * 0.02
    Ms = [rng.standard_normal((R, C)).astype(np.float32) for _ in range(Wn)]
    Gs = [rng.standard_normal((R, C)).astype(np.float32) for _ in range(Wn)]
    a = oracle.sign_muon_step(W, Ms, Gs, 0.9, 1e-3, 3, QUINTIC, variant="bits")
    b = oracle.sign_muon_step(W, Ms, Gs, 0.9, 1e-3, 3, QUINTIC, variant="int8")
    assert np.array_equal(a["S_bar"], b["S_bar"]) and np.array_equal(a["W"], b["W"])
    # the int8 sums are the counts: (#plus - #minus), odd worker counts never tie
    tot = sum(np.where(u < 0, -1, 1) for u in a["U"])
    assert np.array_equal(b["sums"], tot)
    if Wn % 2:
        assert np.all(b["sums"] != 0)


def test_sign_muon_step_post_polar_reaches_polar_of_vote():
    # with the cubic iteration run long enough, the post-vote direction is the polar factor
    # of S_bar (scipy), and the update moves W by exactly -eta times it
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(31)
    R, C, Wn = 6, 11, 3
    W = rng.standard_normal((R, C)).astype(np.float32)
    Ms = [rng.standard_normal((R, C)).astype(np.float32) for _ in range(Wn)]
    Gs = [rng.standard_normal((R, C)).astype(np.float32) for _ in range(Wn)]
    out = oracle.sign_muon_step(W, Ms, Gs, 0.9, 0.5, 60, (1.5, -0.5, 0.0), variant="int8",
                                post_polar=True)
    Q, _ = scipy_linalg.polar(out["S_bar"].astype(np.float64).T)  # C x R, orthonormal columns
    assert np.allclose(out["U_bar"], Q.T, atol=1e-9)
    assert np.allclose(out["W"], W.astype(np.float64) - 0.5 * Q.T, atol=1e-9)
    # rows of the polar factor of a full-row-rank matrix are orthonormal
    assert np.allclose(out["U_bar"] @ out["U_bar"].T, np.eye(R), atol=1e-9)


# ----------------------------------------------------------------- blockwise NS

def test_blockwise_single_block_is_full_ns():
    rng = np.random.default_rng(50)
    M = rng.standard_normal((24, 40))
    assert np.array_equal(oracle.blockwise_newton_schulz(M, 24, 40, 5, QUINTIC),
                          oracle.newton_schulz(M, 5, QUINTIC))
    assert np.array_equal(oracle.blockwise_newton_schulz(M, 100, 100, 5, QUINTIC),
                          oracle.newton_schulz(M, 5, QUINTIC))


def test_blockwise_blocks_are_independent():
    rng = np.random.default_rng(51)
    M = rng.standard_normal((30, 50))
    base = oracle.blockwise_newton_schulz(M, 16, 24, 5, QUINTIC)
    M2 = M.copy()
    M2[16:, 24:48] *= -3.0  # change one block (rows 16..29, columns 24..47)
    other = oracle.blockwise_newton_schulz(M2, 16, 24, 5, QUINTIC)
    changed = np.zeros(M.shape, bool)
    changed[16:, 24:48] = True
    assert np.array_equal(base[~changed], other[~changed])
    # scaling a block by -3: the odd polynomial of the normalised block flips its sign only
    assert np.allclose(other[changed], -base[changed], atol=1e-12)


def test_blockwise_cubic_on_block_diagonal_reaches_full_polar():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(52)
    A, B = rng.standard_normal((8, 12)), rng.standard_normal((6, 9))
    M = np.zeros((14, 21))
    M[:8, :12], M[8:, 12:] = A, B
    got = oracle.blockwise_newton_schulz(M, 8, 12, 60, (1.5, -0.5, 0.0))
    Q, _ = scipy_linalg.polar(M.T)
    assert np.allclose(got, Q.T, atol=1e-9)
    # the whole-matrix quintic result is not blockwise: on a generic input they differ
    G = rng.standard_normal((14, 21))
    assert np.linalg.norm(oracle.blockwise_newton_schulz(G, 8, 12, 5, QUINTIC)
                          - oracle.newton_schulz(G, 5, QUINTIC)) > 0.1
