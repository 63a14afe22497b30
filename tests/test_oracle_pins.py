"""Pins of the fp64 oracle against things other than itself.

Each test ties one oracle function to something the page or the mathematics
fixes: hand-worked bytes, an exhaustive brute-force search, an independent
library routine (numpy packbits / matmul, torch fp64 linear), a closed form,
or a figure the page prints.  Method source: "BitDelta : servir 14 modèles Zen
depuis un seul cluster GPU" (Hanzo blog), sections "Le fondement
mathématique", "Architecture de service", "Détails d'infrastructure".
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_to_f64(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _read_cases(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split(";")]


# ---------------------------------------------------------------- sign packing

@pytest.mark.parametrize("case", list(_read_cases("sign_bytes.txt")), ids=lambda c: c[0])
def test_sign_bits_hand_worked_bytes(case):
    """Hand-worked bytes ("Détails d'infrastructure": 8 signs per byte; LSB-first, >=0 -> 1)."""
    _, rows, cols, wb, wf, expect = case
    rows, cols = int(rows), int(cols)
    wb = np.array([int(h, 16) for h in wb.split(",")], np.uint16).reshape(rows, cols)
    wf = np.array([int(h, 16) for h in wf.split(",")], np.uint16).reshape(rows, cols)
    expect = np.array([int(h, 16) for h in expect.split(",")], np.uint8).reshape(rows, cols // 8)
    assert np.array_equal(oracle.sign_bits(wb, wf), expect)


@pytest.mark.parametrize("shape", [(1, 8), (3, 24), (7, 136), (33, 512)])
def test_sign_bits_match_numpy_packbits(shape):
    """Layout pin: numpy's own little-endian packbits over the row gives the same bytes."""
    wb, wf = synth.matrix_pair(*shape, 0.02, 1e-3, seed=11)
    wb, wf = synth.as_u16(wb), synth.as_u16(wf)
    d = _bf16_to_f64(wf) - _bf16_to_f64(wb)
    ref = np.packbits(d >= 0.0, axis=1, bitorder="little")
    assert np.array_equal(oracle.sign_bits(wb, wf), ref)


def test_unpack_inverts_pack():
    """unpack(pack(s)) = s for an arbitrary +-1 pattern (the listing's {-1, +1})."""
    rng = np.random.default_rng(5)
    s = rng.choice(np.array([-1, 1], np.int8), size=(9, 64))
    wb = np.full(s.shape, 0x3F80, np.uint16)                     # 1.0
    wf = np.where(s > 0, 0x4000, 0x0000).astype(np.uint16)       # 2.0 or 0.0
    bits = oracle.sign_bits(wb, wf)
    assert np.array_equal(oracle.unpack_signs(bits, 64), s)
    assert np.array_equal(np.unpackbits(bits, axis=1, bitorder="little").astype(np.int8) * 2 - 1, s)


# ---------------------------------------------------------------- alpha

def _objective(delta, signs, alphas):
    # ||Delta - alpha * s||^2 for every alpha in the grid
    return ((delta[None, :] - alphas[:, None] * signs[None, :]) ** 2).sum(axis=1)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_brute_force_signs_and_scale_on_1x8(seed):
    """Exhaustive search over all 256 sign patterns and a fine alpha grid.

    The L2-optimal 1-bit code of a row is s = sign(Delta) with alpha = mean|Delta|
    ("Le fondement mathématique").  Deltas here are nonzero so the optimum is unique.
    """
    rng = np.random.default_rng(100 + seed)
    wb = synth.as_u16(synth.bf16_normal((1, 8), 0.02, synth.generator(seed, "cpu"), "cpu"))
    d_target = rng.laplace(0.0, 1e-3, size=8)
    d_target[np.abs(d_target) < 1e-4] = 1e-4
    wf = synth.as_u16(torch.from_numpy(_bf16_to_f64(wb) + d_target[None]).to(torch.bfloat16))
    delta = (_bf16_to_f64(wf) - _bf16_to_f64(wb))[0]
    assert np.all(delta != 0.0)
    grid = np.linspace(0.0, 4e-3, 40001)
    best = (math.inf, None, None)
    for pattern in itertools.product((-1.0, 1.0), repeat=8):
        s = np.array(pattern)
        obj = _objective(delta, s, grid)
        i = int(np.argmin(obj))
        if obj[i] < best[0]:
            best = (obj[i], s, grid[i])
    _, s_best, a_best = best
    bits = oracle.sign_bits(wb, wf)
    assert np.array_equal(oracle.unpack_signs(bits, 8)[0].astype(np.float64), s_best)
    a = oracle.alpha(wb, wf, oracle.ALPHA_SCALAR)[0]
    assert abs(a - a_best) <= grid[1] - grid[0]


@pytest.mark.parametrize("shape,mode", [((4, 8), 0), ((8, 16), 0), ((4, 8), 1), ((8, 16), 1)])
def test_alpha_is_least_squares_scale(shape, mode):
    """For the fixed packed signs, scanning alpha on a 1e4-point grid finds the oracle's alpha."""
    wb, wf = synth.matrix_pair(*shape, 0.02, 1e-3, seed=21)
    wb, wf = synth.as_u16(wb), synth.as_u16(wf)
    delta = _bf16_to_f64(wf) - _bf16_to_f64(wb)
    s = oracle.unpack_signs(oracle.sign_bits(wb, wf), shape[1]).astype(np.float64)
    a = oracle.alpha(wb, wf, mode)
    rows = [delta.reshape(-1)] if mode == 0 else list(delta)
    srows = [s.reshape(-1)] if mode == 0 else list(s)
    for r, (dr, sr) in enumerate(zip(rows, srows)):
        grid = np.linspace(0.0, 3.0 * np.abs(dr).max() + 1e-12, 10001)
        i = int(np.argmin(_objective(dr, sr, grid)))
        assert abs(a[r] - grid[i]) <= grid[1] - grid[0]


def test_alpha_of_laplace_deltas_is_b():
    """E|Delta| = b for Laplace(0, b) ("Le fondement mathématique"), n = 2^22.

    W_base = 0 so Delta is the bf16-rounded draw itself; rounding is unbiased to
    far below the sampling error, and the SD of |Delta| is b, so
    |alpha/b - 1| <= 5/sqrt(n).
    """
    n_out, n_in = 1024, 4096
    g = synth.generator(7, "cpu")
    d = synth.laplace_f32((n_out, n_in), 1e-3, g, "cpu").to(torch.bfloat16)
    wb = np.zeros((n_out, n_in), np.uint16)
    wf = synth.as_u16(d)
    a = oracle.alpha(wb, wf, oracle.ALPHA_SCALAR)[0]
    assert abs(a / 1e-3 - 1.0) <= 5.0 / math.sqrt(n_out * n_in)


def test_alpha_on_realistic_base_is_close_to_b():
    """With a N(0, 0.02) base, bf16 rounding of W_ft moves alpha/b by well under 1%."""
    wb, wf = synth.matrix_pair(512, 2048, 0.02, 1e-3, seed=3)
    a = oracle.alpha(synth.as_u16(wb), synth.as_u16(wf), oracle.ALPHA_SCALAR)[0]
    assert abs(a / 1e-3 - 1.0) < 0.01


def test_per_row_alpha_tracks_per_row_b():
    """Per-row alpha (one per output dimension, "Détails d'infrastructure") follows b_j."""
    n_out, n_in = 64, 16384
    g = synth.generator(9, "cpu")
    b = torch.linspace(5e-4, 2e-3, n_out)
    d = synth.laplace_f32((n_out, n_in), b, g, "cpu").to(torch.bfloat16)
    a = oracle.alpha(np.zeros((n_out, n_in), np.uint16), synth.as_u16(d), oracle.ALPHA_PER_ROW)
    assert np.all(np.abs(a / b.numpy().astype(np.float64) - 1.0) <= 5.0 / math.sqrt(n_in))


def test_reconstruction_residual_closed_form():
    """||W_ft - W_eff||_F / ||Delta||_F = sqrt(1 - (E|D|)^2 / E[D^2]) = sqrt(1/2) for Laplace."""
    n_out, n_in = 1024, 2048
    g = synth.generator(13, "cpu")
    d = synth.laplace_f32((n_out, n_in), 1e-3, g, "cpu").to(torch.bfloat16)
    wb = np.zeros((n_out, n_in), np.uint16)
    wf = synth.as_u16(d)
    bits, a32, _ = oracle.compress(wb, wf, oracle.ALPHA_SCALAR)
    weff = oracle.w_eff(wb, bits, a32, oracle.ALPHA_SCALAR)
    delta = oracle.delta(wb, wf)
    ratio = np.linalg.norm(_bf16_to_f64(wf) - weff) / np.linalg.norm(delta)
    assert abs(ratio - math.sqrt(0.5)) < 0.01


def test_delta_is_exact_difference():
    wb = np.array([[0x3F80, 0x0001, 0x8000, 0xC000]], np.uint16)
    wf = np.array([[0x4000, 0x3F80, 0x0000, 0x3F80]], np.uint16)
    d = oracle.delta(wb, wf)
    assert d.tolist() == [[1.0, 1.0 - 2.0 ** -133, 0.0, 3.0]]


# ---------------------------------------------------------------- fused linear

def _case(n_out, n_in, m, mode, seed):
    b = "row:5e-4:2e-3" if mode == 1 else 1e-3
    wb, wf = synth.matrix_pair(n_out, n_in, 0.02, b, seed=seed)
    x = synth.activations(m, n_in, seed=seed + 1)
    wb, wf, x = synth.as_u16(wb), synth.as_u16(wf), synth.as_u16(x)
    bits, a32, _ = oracle.compress(wb, wf, mode)
    return x, wb, bits, a32


@pytest.mark.parametrize("n_out,n_in,m,mode", [(24, 40, 5, 0), (17, 64, 3, 1), (1, 8, 1, 0)])
def test_linear_equals_unpack_then_dense_matmul(n_out, n_in, m, mode):
    """The listing's reference: unpack -> W_eff -> F.linear, via numpy unpackbits and matmul."""
    x, wb, bits, a32 = _case(n_out, n_in, m, mode, seed=31)
    s = np.unpackbits(bits, axis=1, bitorder="little").astype(np.float64) * 2.0 - 1.0
    a = a32.astype(np.float64)
    w = _bf16_to_f64(wb) + (a[:, None] if mode == 1 else a[0]) * s
    ref = _bf16_to_f64(x) @ w.T
    y, mag = oracle.linear(x, wb, bits, a32, mode)
    assert y.shape == (m, n_out)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(mag, np.abs(_bf16_to_f64(x)) @ np.abs(w).T, rtol=1e-12, atol=1e-15)


def test_linear_equals_torch_fp64_linear():
    x, wb, bits, a32 = _case(33, 96, 7, 0, seed=41)
    w = torch.from_numpy(oracle.w_eff(wb, bits, a32, 0))
    ref = torch.nn.functional.linear(torch.from_numpy(_bf16_to_f64(x)), w).numpy()
    y, _ = oracle.linear(x, wb, bits, a32, 0)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-15)


def test_alpha_zero_reduces_to_base_linear():
    x, wb, bits, _ = _case(20, 48, 4, 0, seed=51)
    y, _ = oracle.linear(x, wb, bits, np.zeros(1, np.float32), 0)
    np.testing.assert_allclose(y, _bf16_to_f64(x) @ _bf16_to_f64(wb).T, rtol=1e-12, atol=1e-15)


def test_zero_base_unit_alpha_is_exact_sign_product():
    """W_base = 0, alpha = 1: y = x . S^T; with integer x this is exact integer arithmetic."""
    rng = np.random.default_rng(8)
    n_out, n_in, m = 13, 72, 6
    s = rng.choice(np.array([-1, 1], np.int64), size=(n_out, n_in))
    xi = rng.integers(-8, 9, size=(m, n_in))
    x = synth.as_u16(torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16))
    wb = np.zeros((n_out, n_in), np.uint16)
    wf = np.where(s > 0, 0x3F80, 0xBF80).astype(np.uint16)
    bits = oracle.sign_bits(wb, wf)
    y, _ = oracle.linear(x, wb, bits, np.ones(1, np.float32), 0)
    assert np.array_equal(y, (xi @ s.T).astype(np.float64))


def test_sampled_outputs_match_full():
    x, wb, bits, a32 = _case(40, 64, 9, 1, seed=61)
    y, mag = oracle.linear(x, wb, bits, a32, 1)
    ts = np.array([0, 8, 3, 5, 8])
    js = np.array([0, 39, 17, 1, 0])
    ys, ms = oracle.linear_sampled(x, wb, bits, a32, 1, ts, js)
    assert np.array_equal(ys, y[ts, js]) and np.array_equal(ms, mag[ts, js])


# ---------------------------------------------------------------- multi-tenant form

def _variants(n_var, n_out, n_in, seed):
    g = synth.generator(seed, "cpu")
    wb = synth.bf16_normal((n_out, n_in), 0.015, g, "cpu")
    bits, alphas, modes = [], [], []
    for v in range(n_var):
        d = synth.laplace_f32((n_out, n_in), 5e-4 + 1e-4 * v, g, "cpu")
        wf = (wb.float() + d).to(torch.bfloat16)
        mode = v % 2
        b, a, _ = oracle.compress(synth.as_u16(wb), synth.as_u16(wf), mode)
        bits.append(b), alphas.append(a), modes.append(mode)
    return synth.as_u16(wb), bits, alphas, np.array(modes, np.int32)


def test_grouped_single_variant_equals_linear():
    wb, bits, alphas, modes = _variants(1, 24, 64, seed=71)
    x = synth.as_u16(synth.activations(6, 64, seed=72))
    ids = np.zeros(6, np.int32)
    y, mag = oracle.linear_grouped(x, ids, wb, bits, alphas, modes)
    y1, mag1 = oracle.linear(x, wb, bits[0], alphas[0], int(modes[0]))
    assert np.array_equal(y, y1) and np.array_equal(mag, mag1)


def test_grouped_rows_equal_per_variant_linear_and_permutation_invariance():
    wb, bits, alphas, modes = _variants(4, 16, 48, seed=81)
    m = 11
    x = synth.as_u16(synth.activations(m, 48, seed=82))
    ids = np.array([3, 0, 0, 2, 1, 3, 3, 0, 2, 2, 3], np.int32)
    y, _ = oracle.linear_grouped(x, ids, wb, bits, alphas, modes)
    for t in range(m):
        v = ids[t]
        yt, _ = oracle.linear(x[t:t + 1], wb, bits[v], alphas[v], int(modes[v]))
        assert np.array_equal(y[t], yt[0])
    perm = np.random.default_rng(0).permutation(m)
    yp, _ = oracle.linear_grouped(x[perm], ids[perm], wb, bits, alphas, modes)
    assert np.array_equal(yp, y[perm])
    ts, js = np.array([0, 10, 4]), np.array([15, 0, 7])
    ys, _ = oracle.linear_grouped_sampled(x, ids, wb, bits, alphas, modes, ts, js)
    assert np.array_equal(ys, y[ts, js])


def test_grouped_rejects_bad_variant_id():
    wb, bits, alphas, modes = _variants(2, 8, 16, seed=91)
    x = synth.as_u16(synth.activations(2, 16, seed=92))
    with pytest.raises(ValueError):
        oracle.linear_grouped(x, np.array([0, 2], np.int32), wb, bits, alphas, modes)


# ---------------------------------------------------------------- storage arithmetic

def test_storage_arithmetic_matches_printed_figures():
    printed = {k: float(v) for k, v, _ in _read_cases("storage_arithmetic.txt")}
    params_70b = 70_000_000_000
    base_gb = params_70b * 2 / 1e9
    delta_gb = oracle.packed_bytes(1, params_70b) / 1e9
    assert base_gb == printed["base_70b_bf16_gb"]
    assert delta_gb == printed["delta_70b_gb"]
    assert 14 * base_gb / 1000 == printed["naive_14_variants_tb"]
    total = base_gb + 14 * delta_gb                     # 262.5, printed as "approximately 262"
    assert abs(total - printed["bitdelta_14_variants_gb"]) < 1.0
    assert round(100 * (1 - total / (14 * base_gb))) == printed["reduction_percent"]
    assert oracle.packed_bytes(4096, 4096) == 4096 * int(printed["packed_4096x4096_cols"])
    for n_out, n_in in [(4096, 4096), (11008, 4096), (3, 24)]:
        assert oracle.packed_bytes(n_out, n_in) / (n_out * n_in * 4) == printed["fraction_of_fp32_delta"]
        assert oracle.packed_bytes(n_out, n_in) * 16 == n_out * n_in * 2   # 1/16 of a bf16 delta


def _weff_cases():
    out = []
    with open(os.path.join(GOLDEN, "weff_bf16.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, wb, a, sbit, exp = [p.strip() for p in line.split(";")]
            out.append((name, int(wb, 16), float(a), int(sbit), int(exp, 16)))
    return out


@pytest.mark.parametrize("case", _weff_cases(), ids=lambda c: c[0])
def test_weff_bf16_hand_worked_rounding(case):
    name, wb, a, sbit, exp = case
    w = np.array([[wb] * 8], np.uint16)
    bits = np.array([[0xFF if sbit else 0x00]], np.uint8)
    got = oracle.w_eff_bf16(w, bits, np.array([a], np.float32), 0)
    assert np.all(got == exp), (name, [hex(v) for v in got[0]], hex(exp))


def test_weff_bf16_special_cases_and_half_ulp_bound():
    wb, wf = synth.matrix_pair(64, 256, 0.02, 1e-3, seed=11)
    wb_h, wf_h = synth.as_u16(wb), synth.as_u16(wf)
    bits, a32, _ = oracle.compress(wb_h, wf_h, 0)
    # alpha = 0: W_eff is W_base itself (the base has no -0.0 entries, which +0.0 would turn into +0.0)
    assert not np.any(wb_h == 0x8000)
    assert np.array_equal(oracle.w_eff_bf16(wb_h, bits, np.zeros(1, np.float32), 0), wb_h)
    # W_base = 0, alpha exact in bf16: W_eff = +-alpha exactly
    z = np.zeros_like(wb_h)
    alpha_exact = np.array([0.0078125], np.float32)
    s = oracle.unpack_signs(bits, 256).astype(np.float64)
    got = _bf16_to_f64(oracle.w_eff_bf16(z, bits, alpha_exact, 0))
    assert np.array_equal(got, 0.0078125 * s)
    # general case, per-row alpha: within half a bf16 ulp of the exact fp64 W_eff
    bits1, a1, _ = oracle.compress(wb_h, wf_h, 1)
    exact = oracle.w_eff(wb_h, bits1, a1, 1)
    got = _bf16_to_f64(oracle.w_eff_bf16(wb_h, bits1, a1, 1))
    ulp = 2.0 ** (np.floor(np.log2(np.abs(exact))) - 7)
    assert np.all(np.abs(got - exact) <= 0.5 * ulp * (1 + 2.0 ** -16))
