"""Pins for the fp64 oracle, against things other than itself.

* exact rational brute force (fractions.Fraction) on tiny sizes, all layouts;
* hand-worked FC examples and split/rounding tables in tests/golden/;
* closed forms: identity and rank-1 operands;
* S == C for non-negative operands, S >= |C| always;
* the block-sum invariant of the 3D grid for all three ops;
* torch's float32 -> bf16 cast as a library special case of ``bf16_rne``;
* a planted mistake in the oracle is caught by these pins.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import fc_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fc_hand_examples.json")


def _bits(a):
    return fc_inputs.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _frac(bits):
    return [[Fraction(float(v)) for v in row] for row in fc_inputs.bf16_bits_to_f32(bits)]


def _store(logical_bits, t):
    """Stored array for a logical matrix (transposed copy if t)."""
    return np.ascontiguousarray(logical_bits.T) if t else logical_bits


@pytest.mark.parametrize("M,N,R", [(1, 1, 1), (2, 3, 7), (3, 2, 1), (7, 16, 17),
                                   (16, 17, 3), (17, 7, 16)])
@pytest.mark.parametrize("a_t", [False, True])
@pytest.mark.parametrize("b_t", [False, True])
def test_gemm_vs_exact_rationals(M, N, R, a_t, b_t):
    A = fc_inputs.normal_bf16((M, R), seed=11, tid=M * 100 + R)
    B = fc_inputs.normal_bf16((R, N), seed=12, tid=N * 100 + R)
    C, S = oracle.gemm(_store(A, a_t), a_t, _store(B, b_t), b_t)
    Af, Bf = _frac(A), _frac(B)
    for i in range(M):
        for j in range(N):
            exact = sum(Af[i][r] * Bf[r][j] for r in range(R))
            sabs = sum(abs(Af[i][r]) * abs(Bf[r][j]) for r in range(R))
            # fp64 accumulation of exact products: error <= R * 2^-52 * S
            tol = float(sabs) * R * 2.0 ** -52
            assert abs(Fraction(C[i, j]) - exact) <= Fraction(tol)
            assert abs(Fraction(S[i, j]) - sabs) <= Fraction(tol)


def test_hand_examples():
    g = json.load(open(GOLDEN))
    X, W, dY = _bits(g["X"]), _bits(g["W"]), _bits(g["dY"])
    Y, _ = oracle.fc_fwd(X, W)
    dX, _ = oracle.fc_dgrad(dY, W)
    dW, _ = oracle.fc_wgrad(X, dY)
    assert np.array_equal(Y, np.array(g["Y"], float))
    assert np.array_equal(dX, np.array(g["dX"], float))
    assert np.array_equal(dW, np.array(g["dW"], float))
    # the same products with every operand stored transposed
    Xt, Wt, dYt = (np.ascontiguousarray(m.T) for m in (X, W, dY))
    assert np.array_equal(oracle.fc_fwd(Xt, Wt, True, True)[0], Y)
    assert np.array_equal(oracle.fc_dgrad(dYt, Wt, True, True)[0], dX)
    assert np.array_equal(oracle.fc_wgrad(Xt, dYt, True, True)[0], dW)


def test_split_rule_table():
    g = json.load(open(GOLDEN))["split_rule"]
    for case in g["cases"]:
        got = [list(oracle.split_range(case["D"], case["G"], b)) for b in range(case["G"])]
        assert got == case["ranges"], case


@pytest.mark.parametrize("D", [0, 1, 7, 8, 9, 63, 1000, 5000, 6144, 24577])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
def test_split_rule_properties(D, G):
    ranges = [oracle.split_range(D, G, b) for b in range(G)]
    assert ranges[0][0] == 0 and ranges[-1][1] == D
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    for a, b in ranges:
        assert a % 8 == 0 or a == D
    # balanced: whole-unit counts differ by at most one
    units = [(s + 7) // 8 for s in sizes]
    assert max(units) - min(units) <= 1 or D == 0


def test_bf16_rne_table():
    g = json.load(open(GOLDEN))["bf16_rne"]
    vals = np.array([c[0] for c in g["cases"]], dtype=np.float64)
    want = np.array([int(c[1], 16) for c in g["cases"]], dtype=np.uint16)
    assert np.array_equal(oracle.bf16_rne(vals), want)


def test_bf16_rne_matches_torch_cast_on_floats():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    f = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0,
        rng.standard_normal(2000).astype(np.float32) * 1e-39,   # subnormals
        np.float32(1.0) + np.arange(512, dtype=np.float32) * np.float32(2.0 ** -9),
    ])
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_roundtrip():
    b = fc_inputs.normal_bf16((4096,), seed=3, tid=1)
    assert np.array_equal(oracle.bf16_rne(oracle.bf16_to_f64(b)), b)


@pytest.mark.parametrize("op", oracle.OPS)
def test_identity_closed_form(op):
    n = 24
    I = _bits(np.eye(n))
    P = fc_inputs.normal_bf16((n, n), seed=4, tid=7)
    if op == "fwd":       # X . I == X
        C, _ = oracle.fc_fwd(P, I)
    elif op == "dgrad":   # dY . I^T == dY
        C, _ = oracle.fc_dgrad(P, I)
    else:                 # I^T . dY == dY
        C, _ = oracle.fc_wgrad(I, P)
    assert np.array_equal(C, oracle.bf16_to_f64(P))


def test_rank1_closed_form():
    a = np.array([1, -2, 3, 0, 2], float)       # T
    b = np.array([2, 1, -1], float)             # K
    c = np.array([1, 3, -2], float)             # K
    d = np.array([-1, 2, 1, 4], float)          # N
    X, W = _bits(np.outer(a, b)), _bits(np.outer(c, d))
    Y, _ = oracle.fc_fwd(X, W)
    assert np.array_equal(Y, float(b @ c) * np.outer(a, d))


def test_nonnegative_S_equals_C_and_S_bounds():
    A = fc_inputs.normal_bf16((33, 65), seed=8, tid=1)
    B = fc_inputs.normal_bf16((65, 40), seed=8, tid=2)
    C, S = oracle.gemm(A, False, B, False)
    assert np.all(S >= np.abs(C))
    Aa, Ba = A & np.uint16(0x7FFF), B & np.uint16(0x7FFF)
    C2, S2 = oracle.gemm(Aa, False, Ba, False)
    assert np.array_equal(C2, S2)
    assert np.allclose(S2, S, rtol=1e-14, atol=0)


@pytest.mark.parametrize("op", oracle.OPS)
@pytest.mark.parametrize("grid", [(2, 2, 2), (1, 4, 4), (3, 1, 2), (2, 3, 1)])
def test_block_sum_invariant(op, grid):
    T, K, N = 41, 50, 36   # ragged against the 8-element units
    X = fc_inputs.small_int_bf16((T, K), seed=9, tid=1, h=2)
    W = fc_inputs.small_int_bf16((K, N), seed=9, tid=2, h=2)
    dY = fc_inputs.small_int_bf16((T, N), seed=9, tid=3, h=2)
    P, Q = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (X, dY)}[op]
    full, Sfull = oracle.fc(op, P, Q)
    vg, Svg = oracle.fc_vgrid(op, P, Q, False, False, T, K, N, grid)
    assert np.array_equal(vg, full)          # integers: exact
    assert np.array_equal(Svg, Sfull)
    # every block equals the full product restricted to that block when the
    # reduced axis has one block
    gx, gy, gz = grid
    for x in range(gx):
        for y in range(gy):
            for z in range(gz):
                Cb, _, rows, cols = oracle.fc_block(op, P, Q, False, False, T, K, N,
                                                    grid, (x, y, z))
                assert Cb.shape == (rows[1] - rows[0], cols[1] - cols[0])


def test_block_partials_random_fp():
    T, K, N = 64, 96, 80
    X = fc_inputs.normal_bf16((T, K), seed=10, tid=1)
    W = fc_inputs.normal_bf16((K, N), seed=10, tid=2, sigma=0.02)
    full, S = oracle.fc_fwd(X, W)
    vg, _ = oracle.fc_vgrid("fwd", X, W, False, False, T, K, N, (2, 2, 2))
    assert np.all(np.abs(vg - full) <= 1e-13 * S)


def test_entries_match_full():
    X = fc_inputs.normal_bf16((50, 70), seed=12, tid=1)
    dY = fc_inputs.normal_bf16((50, 30), seed=12, tid=2)
    C, S = oracle.fc_wgrad(X, dY)
    I = np.array([0, 69, 13, 5]); J = np.array([0, 29, 7, 22])
    Ce, Se = oracle.fc_entries("wgrad", X, dY, False, False, I, J)
    assert np.array_equal(Ce, C[I, J]) and np.array_equal(Se, S[I, J])


def test_planted_mistake_is_caught(monkeypatch):
    """A dgrad that forgets the transpose of W must fail the hand pin."""
    g = json.load(open(GOLDEN))
    real = oracle.operands

    def wrong(op, P, Q, p_t, q_t):
        if op == "dgrad":
            return P, p_t, Q, q_t     # W instead of W^T
        return real(op, P, Q, p_t, q_t)

    monkeypatch.setattr(oracle, "operands", wrong)
    with pytest.raises(AssertionError):
        dX, _ = oracle.fc_dgrad(_bits(g["dY"]), _bits(g["W"]))
        assert np.array_equal(dX, np.array(g["dX"], float))


@pytest.mark.parametrize("G", [1, 2, 3, 4])
def test_shards_gather_back_to_the_block(G):
    Wb = fc_inputs.normal_bf16((45, 24), seed=14, tid=1)
    shards = oracle.shard_rows(Wb, G)
    assert [s.shape[0] for s in shards] == [b - a for a, b in
                                           (oracle.split_range(45, G, z) for z in range(G))]
    assert np.array_equal(oracle.gather_shards(shards), Wb)


@pytest.mark.parametrize("grid,xy", [((2, 2, 2), (1, 0)), ((1, 4, 4), (0, 3)), ((3, 1, 2), (2, 0))])
def test_wgrad_zsharded_is_the_vgrid_block_cut_in_shards(grid, xy):
    T, K, N = 41, 50, 36
    X = fc_inputs.small_int_bf16((T, K), seed=15, tid=1, h=2)
    dY = fc_inputs.small_int_bf16((T, N), seed=15, tid=3, h=2)
    Cs, Ss = oracle.wgrad_zsharded(X, dY, False, False, T, K, N, grid, xy)
    full, Sfull = oracle.fc_vgrid("wgrad", X, dY, False, False, T, K, N, grid)
    Kx = oracle.split_range(K, grid[0], xy[0])
    Ny = oracle.split_range(N, grid[1], xy[1])
    assert np.array_equal(oracle.gather_shards(Cs), full[Kx[0]:Kx[1], Ny[0]:Ny[1]])
    assert np.array_equal(oracle.gather_shards(Ss), Sfull[Kx[0]:Kx[1], Ny[0]:Ny[1]])
    assert len(Cs) == grid[2]


def test_thread_count_setter_keeps_results():
    """The oracle's thread count is a setting, not arithmetic: one thread and
    all threads give the same bits."""
    A = fc_inputs.normal_bf16((37, 29), 5, 1)
    B = fc_inputs.normal_bf16((29, 41), 5, 2)
    before = oracle.max_threads()
    try:
        assert oracle.set_threads(1) == 1
        C1, S1 = oracle.gemm(A, False, B, False)
        n = os.cpu_count() or 1
        assert oracle.set_threads(n) == n
        Cn, Sn = oracle.gemm(A, False, B, False)
    finally:
        oracle.set_threads(before)
    assert np.array_equal(C1, Cn) and np.array_equal(S1, Sn)


@pytest.mark.parametrize("T,K,N", [(1, 1, 1), (5, 7, 3), (16, 9, 12)])
def test_op_equivalences_through_transposed_copies(T, K, N):
    """dgrad(dY, W) = fwd(dY, W^T) and wgrad(X, dY) = fwd(X^T, dY), with the
    transposes made as explicit copies (the other addressing path); and
    each op with its operands stored transposed (flags) equals the op on the
    plain layout."""
    X = fc_inputs.normal_bf16((T, K), 21, 1)
    W = fc_inputs.normal_bf16((K, N), 21, 2)
    dY = fc_inputs.normal_bf16((T, N), 21, 3)
    Wt = np.ascontiguousarray(W.T)
    Xt = np.ascontiguousarray(X.T)
    dYt = np.ascontiguousarray(dY.T)
    dx, sdx = oracle.fc("dgrad", dY, W)
    dx2, sdx2 = oracle.fc("fwd", dY, Wt)
    assert np.array_equal(dx, dx2) and np.array_equal(sdx, sdx2)
    dw, sdw = oracle.fc("wgrad", X, dY)
    dw2, sdw2 = oracle.fc("fwd", Xt, dY)
    assert np.array_equal(dw, dw2) and np.array_equal(sdw, sdw2)
    for op, P, Q, Pt, Qt in (("fwd", X, W, Xt, Wt), ("dgrad", dY, W, dYt, Wt),
                             ("wgrad", X, dY, Xt, dYt)):
        ref, _ = oracle.fc(op, P, Q)
        for p_t, q_t in ((True, False), (False, True), (True, True)):
            got, _ = oracle.fc(op, Pt if p_t else P, Qt if q_t else Q, p_t, q_t)
            assert np.array_equal(got, ref), (op, p_t, q_t)


def _block_pin_mismatches(block_extents):
    """Cases of the hand-worked block-extent table that `block_extents`
    gets wrong (empty when every op of every case matches)."""
    g = json.load(open(GOLDEN))["block_extents"]
    bad = []
    for case in g["cases"]:
        T, K, N = case["TKN"]
        for op in oracle.OPS:
            want = tuple(tuple(r) for r in case[op])
            try:
                got = tuple(tuple(r) for r in block_extents(op, T, K, N, tuple(case["grid"]),
                                                            tuple(case["coords"])))
            except AssertionError:
                got = None
            if got != want:
                bad.append((case["TKN"], case["grid"], case["coords"], op, got, want))
    return bad


def test_block_extents_hand_table():
    """Which grid axis cuts which dimension (T by G_z, K by G_x, N by G_y) and
    each op's (output rows, reduced range, output cols), pinned by hand on
    asymmetric grids: any permutation of the axes fails here, where the
    block-sum invariant (which holds for every permutation) cannot tell."""
    assert _block_pin_mismatches(oracle.block_extents) == []


def _swap_axes(which):
    real = oracle.block_extents

    def wrong(op, T, K, N, grid, coords):
        gx, gy, gz = grid
        x, y, z = coords
        if which == "xy":
            return real(op, T, K, N, (gy, gx, gz), (y, x, z))
        if which == "xz":
            return real(op, T, K, N, (gz, gy, gx), (z, y, x))
        # dgrad reducing over the output columns' axis instead of N's
        rows, red, cols = real(op, T, K, N, grid, coords)
        return (rows, cols, red) if op == "dgrad" else (rows, red, cols)
    return wrong


@pytest.mark.parametrize("which", ["xy", "xz", "dgrad_roles"])
def test_planted_block_axis_mistake_is_caught(which):
    """A grid whose G_x and G_y (or G_x and G_z) trade places, or a data
    gradient with its reduced and output ranges exchanged, fails the hand
    table; the block-sum invariant alone would pass all three."""
    wrong = _swap_axes(which)
    assert _block_pin_mismatches(wrong)
    if which != "dgrad_roles":
        T, K, N, grid = 41, 50, 36, (3, 1, 2)
        X = fc_inputs.small_int_bf16((T, K), seed=9, tid=1, h=2)
        W = fc_inputs.small_int_bf16((K, N), seed=9, tid=2, h=2)
        real = oracle.block_extents
        try:
            oracle.block_extents = wrong
            vg, _ = oracle.fc_vgrid("fwd", X, W, False, False, T, K, N, (2, 2, 2))
        finally:
            oracle.block_extents = real
        assert np.array_equal(vg, oracle.fc_fwd(X, W)[0])   # the invariant cannot tell
