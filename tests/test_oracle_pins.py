"""Pins for the CPU oracle: library routines in float64, hand-derived format
tables, finite differences, closed forms and invariants.

None of these re-types the oracle's own formula: each compares it with
something fixed independently (torch's float64 layer_norm / rms_norm and
autograd, torch's dtype conversions, the OCP format definitions worked out by
hand, or a property that holds whatever the implementation).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import parse_float, read_golden

LN, RMS = 0, 1


def _bits8(t):
    return t.view(torch.uint8).numpy()


# ---------------------------------------------------------------- E4M3 format

def test_e4m3_golden_table(orc):
    for code_s, val_s in read_golden("e4m3_codes.txt"):
        code, val = int(code_s, 16), parse_float(val_s)
        assert orc.e4m3_decode(code) == val, hex(code)
        assert orc.e4m3_encode(val) == code, hex(code)


def test_e4m3_roundtrip_all_codes(orc):
    for c in range(256):
        v = orc.e4m3_decode(c)
        if (c & 0x7F) == 0x7F:
            assert math.isnan(v)
            assert orc.e4m3_encode(v) == 0x7F
            continue
        assert orc.e4m3_encode(v) == c, hex(c)


def test_e4m3_midpoints_round_to_even(orc):
    finite = [c for c in range(0x00, 0x7F)]  # positive codes 0 .. 0x7E
    for c in finite[:-1]:
        lo, hi = orc.e4m3_decode(c), orc.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == even, hex(c)
        assert orc.e4m3_encode(-mid) == even | 0x80, hex(c)
        eps = (hi - lo) * 1e-6
        assert orc.e4m3_encode(mid - eps) == c
        assert orc.e4m3_encode(mid + eps) == c + 1


def test_e4m3_saturation_and_specials(orc):
    for v in [448.0, 449.0, 463.999, 464.0, 480.0, 1e6, float("inf")]:
        assert orc.e4m3_encode(v) == 0x7E, v
        assert orc.e4m3_encode(-v) == 0xFE, v
    assert orc.e4m3_encode(float("nan")) == 0x7F
    assert orc.e4m3_encode(2.0 ** -10) == 0x00      # tie between 0 and 2^-9 -> even (0)
    assert orc.e4m3_encode(1.5 * 2.0 ** -10) == 0x01
    assert orc.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 (x 2^-9) -> even
    assert orc.e4m3_encode(-0.0) == 0x80


def test_e4m3_matches_torch_conversion_in_range(orc):
    # torch's float32 -> float8_e4m3fn conversion (round to nearest even) is an
    # independent implementation; it does not saturate, so stay below 464.
    g = torch.Generator().manual_seed(1)
    v = torch.cat([
        torch.randn(3000, generator=g) * 40,
        torch.randn(2000, generator=g) * 0.01,
        (torch.rand(500, generator=g) * 2 - 1) * 463.0,
        torch.tensor([0.0, -0.0, 2.0 ** -9, 2.0 ** -10, 448.0, -448.0, 300.0, 3 * 2.0 ** -10]),
    ]).to(torch.float32)
    v = v[v.abs() < 464.0]
    ref = _bits8(v.to(torch.float8_e4m3fn))
    got = np.array([orc.e4m3_encode(float(a)) for a in v.tolist()], dtype=np.uint8)
    assert np.array_equal(ref, got)


# ---------------------------------------------------------------- E8M0 scales

def test_e8m0_golden(orc):
    for a_s, c_s in read_golden("e8m0_codes.txt"):
        a = float(np.float32(parse_float(a_s)))
        assert orc.e8m0_code(a) == int(c_s), a_s


def test_e8m0_powers_of_two(orc):
    for k in range(-119, 128):
        a = float(np.float32(2.0 ** k))
        assert orc.e8m0_code(a) == min(254, max(0, k - 8 + 127))


def test_mxfp8_golden_block(orc):
    rows = read_golden("mxfp8_block.txt")
    assert rows[0][0] == "scale"
    scale = int(rows[0][1])
    vals = [parse_float(r[0]) for r in rows[1:]]
    codes = [int(r[1], 16) for r in rows[1:]]
    z = np.zeros((1, 32))
    z[0, :len(vals)] = vals
    q, s = orc.mxfp8_rowwise(z)
    assert s[0, 0] == scale
    assert list(q[0, :len(vals)]) == codes
    assert all(q[0, len(vals):] == 0)


def test_mxfp8_saturating_floor_rule(orc):
    # amax 500 lies in [2^8, 2^9): scale code 127 (x1) and 500 saturates to 448.
    z = np.zeros((1, 32))
    z[0, 0], z[0, 1] = 500.0, -460.0
    q, s = orc.mxfp8_rowwise(z)
    assert s[0, 0] == 127 and q[0, 0] == 0x7E and q[0, 1] == 0xFE


def test_mxfp8_power_of_two_equivariance(orc):
    g = np.random.default_rng(3)
    z = g.standard_normal((4, 64)) * 3
    q0, s0 = orc.mxfp8_rowwise(z)
    for k in (-20, -3, 5, 40):
        q1, s1 = orc.mxfp8_rowwise(z * 2.0 ** k)
        assert np.array_equal(q0, q1)
        assert np.array_equal(s1.astype(int), s0.astype(int) + k)


def test_mxfp8_colwise_is_rowwise_of_transpose(orc):
    g = np.random.default_rng(4)
    # Rows with very different magnitudes: a transposed block would change scales.
    z = g.standard_normal((64, 96)) * (10.0 ** g.uniform(-2, 2, size=(64, 1)))
    qc, sc = orc.mxfp8_colwise(z)
    qr, sr = orc.mxfp8_rowwise(np.ascontiguousarray(z.T))
    assert np.array_equal(qc, qr.T)
    assert np.array_equal(sc, sr.T)
    qrow, _ = orc.mxfp8_rowwise(z)
    assert not np.array_equal(qc, qrow)


def test_mxfp8_nan_block(orc):
    z = np.ones((1, 64))
    z[0, 3] = np.nan
    q, s = orc.mxfp8_rowwise(z)
    assert s[0, 0] == 255 and all(q[0, :32] == 0x7F)
    assert s[0, 1] == 119 and all(q[0, 32:] == 0x78)


# ---------------------------------------------------------------- delayed scaling

def test_delayed_golden(orc):
    rows = read_golden("delayed_e4m3.txt")
    z = np.array([parse_float(r[0]) for r in rows])
    q, amax, sinv = orc.quant_delayed(z, 448.0 / 30.0)
    assert list(q) == [int(r[1], 16) for r in rows]
    assert amax == np.float32(40.0)
    assert sinv == np.float32(1.0 / np.float64(np.float32(448.0 / 30.0)))


def test_delayed_amax_nan_propagates(orc):
    q, amax, _ = orc.quant_delayed(np.array([1.0, np.nan, 3.0]), 1.0)
    assert math.isnan(amax) and q[1] == 0x7F


# ---------------------------------------------------------------- stored-dtype rounding

def _special_f32():
    g = torch.Generator().manual_seed(5)
    v = torch.cat([
        torch.randn(4000, generator=g) * 100,
        torch.randn(1000, generator=g) * 1e-30,
        torch.randn(1000, generator=g) * 1e-40,  # fp32 subnormals
        torch.randn(500, generator=g) * 1e37,
        torch.tensor([0.0, -0.0, 65504.0, 65520.0, 65536.0, 3.3895e38, 3.4e38, 6e-8, 3e-8]),
    ]).to(torch.float32)
    # exact ties for bf16: low 16 bits = 0x8000
    bits = torch.randint(0, 2 ** 31 - 2 ** 24, (500,), generator=g, dtype=torch.int64)
    ties = ((bits & ~0xFFFF) | 0x8000).to(torch.int32).view(torch.float32)
    return torch.cat([v, ties[torch.isfinite(ties)]])


def test_bf16_rounding_matches_torch(orc):
    v = _special_f32()
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([orc.bf16_bits(float(a)) for a in v.tolist()], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_f16_rounding_matches_torch(orc):
    v = _special_f32()
    ref = v.to(torch.float16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([orc.f16_bits(float(a)) for a in v.tolist()], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_bf16_rounding_is_single_rounding_from_double(orc):
    # 1 + 2^-8 + 2^-40: rounding through fp32 first would give the tie 1 + 2^-8
    # and then 1.0; one rounding from double gives 1 + 2^-7.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    one_plus = np.array([1.0 + 2.0 ** -7], dtype=np.float32).view(np.uint32)[0] >> 16
    assert orc.bf16_bits(v) == one_plus


def test_widen_is_exact(orc):
    g = torch.Generator().manual_seed(6)
    v = torch.randn(257, generator=g) * 7
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        t = v.to(dt)
        assert np.array_equal(orc.widen(t), t.to(torch.float64).numpy())


# ---------------------------------------------------------------- forward

def _rand_case(seed, rows, hidden, in_dt, w_dt, beta=True):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, hidden, generator=g) * 2 + 0.5).to(in_dt)
    gamma = (1 + 0.1 * torch.randn(hidden, generator=g)).to(w_dt)
    b = (0.1 * torch.randn(hidden, generator=g)).to(w_dt) if beta else None
    return x, gamma, b


@pytest.mark.parametrize("in_dt,w_dt", [(torch.float32, torch.float32),
                                        (torch.bfloat16, torch.float32),
                                        (torch.float16, torch.bfloat16)])
@pytest.mark.parametrize("zcg", [False, True])
def test_layernorm_fwd_matches_torch_float64(orc, in_dt, w_dt, zcg):
    x, gamma, beta = _rand_case(10, 33, 200, in_dt, w_dt)
    z, mu, rs = orc.norm_fwd(x, gamma, beta, LN, zcg, 1e-5)
    w = gamma.double() + (1.0 if zcg else 0.0)
    ref = F.layer_norm(x.double(), (200,), w, beta.double(), 1e-5)
    np.testing.assert_allclose(z, ref.numpy(), rtol=1e-12, atol=1e-12)
    xd = x.double()
    np.testing.assert_allclose(mu, xd.mean(1).numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(rs, (1 / torch.sqrt(xd.var(1, unbiased=False) + 1e-5)).numpy(),
                               rtol=1e-12)


@pytest.mark.parametrize("in_dt,w_dt", [(torch.float32, torch.float32),
                                        (torch.bfloat16, torch.bfloat16)])
@pytest.mark.parametrize("zcg", [False, True])
def test_rmsnorm_fwd_matches_torch_float64(orc, in_dt, w_dt, zcg):
    x, gamma, _ = _rand_case(11, 31, 96, in_dt, w_dt, beta=False)
    z, _, rs = orc.norm_fwd(x, gamma, None, RMS, zcg, 1e-6)
    w = gamma.double() + (1.0 if zcg else 0.0)
    ref = F.rms_norm(x.double(), (96,), w, 1e-6)
    np.testing.assert_allclose(z, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_fwd_invariants_eps0(orc):
    g = torch.Generator().manual_seed(12)
    x = torch.randn(8, 64, generator=g) * 3 + 1
    one = torch.ones(64)
    zero = torch.zeros(64)
    z, _, _ = orc.norm_fwd(x, one, zero, LN, False, 0.0)
    np.testing.assert_allclose(z.mean(1), 0, atol=1e-13)
    np.testing.assert_allclose((z ** 2).mean(1), 1, rtol=1e-13)
    z, _, _ = orc.norm_fwd(x, one, None, RMS, False, 0.0)
    np.testing.assert_allclose((z ** 2).mean(1), 1, rtol=1e-13)


def test_fwd_shift_scale_invariance(orc):
    g = torch.Generator().manual_seed(13)
    x = torch.randint(-512, 513, (4, 48), generator=g).float() / 256  # 2^-8 grid
    gamma = torch.randn(48, generator=g)
    beta = torch.randn(48, generator=g)
    z0, _, _ = orc.norm_fwd(x, gamma, beta, LN, False, 0.0)
    z1, _, _ = orc.norm_fwd(x * 4 + 3, gamma, beta, LN, False, 0.0)  # exact in fp32
    np.testing.assert_allclose(z0, z1, rtol=1e-12, atol=1e-12)
    r0, _, _ = orc.norm_fwd(x, gamma, None, RMS, False, 0.0)
    r1, _, _ = orc.norm_fwd(x * 0.25, gamma, None, RMS, False, 0.0)
    np.testing.assert_allclose(r0, r1, rtol=1e-12, atol=1e-12)


def test_fwd_constant_and_zero_rows(orc):
    H, eps, c = 16, 1e-5, 0.75
    x = torch.full((1, H), c)
    gamma = torch.linspace(0.5, 2.0, H)
    beta = torch.linspace(-1, 1, H)
    z, mu, rs = orc.norm_fwd(x, gamma, beta, LN, False, eps)
    assert np.array_equal(z[0], beta.double().numpy())      # (x - mu) = 0 exactly
    assert mu[0] == c and rs[0] == 1 / math.sqrt(eps)
    z, _, rs = orc.norm_fwd(x, gamma, None, RMS, False, eps)
    np.testing.assert_allclose(z[0], c * gamma.double().numpy() / math.sqrt(c * c + eps),
                               rtol=1e-14)
    z, _, rs = orc.norm_fwd(torch.zeros(1, H), gamma, None, RMS, False, eps)
    assert np.all(z == 0) and rs[0] == 1 / math.sqrt(eps)


def test_fwd_two_element_closed_form(orc):
    a, b, eps = 1.25, -0.5, 1e-3
    z, _, _ = orc.norm_fwd(torch.tensor([[a, b]]), torch.ones(2), torch.zeros(2), LN, False, eps)
    h = (a - b) / 2
    ref = h / math.sqrt(h * h + eps)
    np.testing.assert_allclose(z[0], [ref, -ref], rtol=1e-14)


def test_fwd_zero_centered_gamma_is_one_plus_gamma(orc):
    x, gamma, beta = _rand_case(14, 5, 40, torch.float32, torch.float32)
    z0, _, _ = orc.norm_fwd(x, gamma, beta, LN, True, 1e-5)
    z1, _, _ = orc.norm_fwd(x, (gamma.double() + 1).float(), beta, LN, False, 1e-5)
    np.testing.assert_allclose(z0, z1, rtol=1e-6, atol=1e-6)  # 1+gamma rounded to fp32 in z1


# ---------------------------------------------------------------- backward

def _grid_case(seed, rows, hidden):
    """Inputs on a 2^-8 grid so that +-2^-12 perturbations are exact in fp32."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(-512, 513, (rows, hidden), generator=g).float() / 256
    gamma = torch.randint(64, 448, (hidden,), generator=g).float() / 256
    beta = torch.randint(-128, 129, (hidden,), generator=g).float() / 256
    dz = torch.randint(-512, 513, (rows, hidden), generator=g).float() / 256
    return x, gamma, beta, dz


@pytest.mark.parametrize("norm", [LN, RMS])
@pytest.mark.parametrize("zcg", [False, True])
def test_bwd_finite_differences(orc, norm, zcg):
    x, gamma, beta, dz = _grid_case(20 + norm + 2 * zcg, 4, 8)
    b = beta if norm == LN else None
    eps, h = 1e-3, 2.0 ** -12
    dzd = dz.double().numpy()

    def loss(xx, gg, bb):
        z, _, _ = orc.norm_fwd(xx, gg, bb, norm, zcg, eps)
        return float((dzd * z).sum())

    _, mu, rs = orc.norm_fwd(x, gamma, b, norm, zcg, eps)
    mu32 = mu.astype(np.float32) if norm == LN else None
    dx, dg, db = orc.norm_bwd(dz, x, mu32, rs.astype(np.float32), gamma, None, norm, zcg)
    for i in range(4):
        for j in range(8):
            xp, xm = x.clone(), x.clone()
            xp[i, j] += h
            xm[i, j] -= h
            fd = (loss(xp, gamma, b) - loss(xm, gamma, b)) / (2 * h)
            assert abs(fd - dx[i, j]) <= 2e-5 * max(1.0, abs(fd)), (i, j, fd, dx[i, j])
    for j in range(8):
        gp, gm = gamma.clone(), gamma.clone()
        gp[j] += h
        gm[j] -= h
        fd = (loss(x, gp, b) - loss(x, gm, b)) / (2 * h)
        assert abs(fd - dg[j]) <= 2e-5 * max(1.0, abs(fd)), (j, fd, dg[j])
        if norm == LN:
            bp, bm = beta.clone(), beta.clone()
            bp[j] += h
            bm[j] -= h
            fd = (loss(x, gamma, bp) - loss(x, gamma, bm)) / (2 * h)
            assert abs(fd - db[j]) <= 2e-5 * max(1.0, abs(fd))


@pytest.mark.parametrize("norm", [LN, RMS])
def test_bwd_matches_torch_autograd_float64(orc, norm):
    g = torch.Generator().manual_seed(30 + norm)
    R, H, eps = 6, 72, 1e-5
    x = (torch.randn(R, H, generator=g) * 2 + 0.3).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=g))
    beta = 0.1 * torch.randn(H, generator=g)
    dz = torch.randn(R, H, generator=g).to(torch.bfloat16)
    dres = torch.randn(R, H, generator=g).to(torch.bfloat16)
    xd = x.double().requires_grad_(True)
    wd = gamma.double().requires_grad_(True)
    bd = beta.double().requires_grad_(True)
    if norm == LN:
        zt = F.layer_norm(xd, (H,), wd, bd, eps)
    else:
        zt = F.rms_norm(xd, (H,), wd, eps)
    zt.backward(dz.double())
    # Statistics as stored by the forward (fp32), as the backward receives them.
    _, mu, rs = orc.norm_fwd(x, gamma, beta if norm == LN else None, norm, False, eps)
    dx, dg, db = orc.norm_bwd(dz, x, mu.astype(np.float32) if norm == LN else None,
                              rs.astype(np.float32), gamma, dres, norm, False)
    ref_dx = xd.grad.numpy() + dres.double().numpy()
    np.testing.assert_allclose(dx, ref_dx, rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(dg, wd.grad.numpy(), rtol=2e-6, atol=2e-6)
    if norm == LN:
        np.testing.assert_allclose(db, bd.grad.numpy(), rtol=1e-12, atol=1e-12)
    else:
        assert db is None


def test_bwd_invariants(orc):
    # Rows of +-1 with equal counts: mean 0 and variance 1 exactly, so with
    # eps = 0 the stored fp32 statistics are exact and the invariants hold to
    # double rounding.  LayerNorm: sum_j dx = 0 and sum_j dx * xhat = 0;
    # RMSNorm: sum_j dx * x = 0.
    g = torch.Generator().manual_seed(40)
    H = 64
    signs = torch.stack([torch.randperm(H, generator=g) % 2 for _ in range(5)]).float() * 2 - 1
    gamma = 1 + 0.1 * torch.randn(H, generator=g)
    dz = torch.randn(5, H, generator=g)
    _, mu, rs = orc.norm_fwd(signs, gamma, torch.zeros(H), LN, False, 0.0)
    assert np.all(mu == 0) and np.all(rs == 1)
    dx, _, _ = orc.norm_bwd(dz, signs, mu.astype(np.float32), rs.astype(np.float32), gamma,
                            None, LN, False)
    xs = signs.double().numpy()
    np.testing.assert_allclose(dx.sum(1), 0, atol=1e-13)
    np.testing.assert_allclose((dx * xs).sum(1), 0, atol=1e-13)
    _, _, rs = orc.norm_fwd(signs, gamma, None, RMS, False, 0.0)
    dx, _, _ = orc.norm_bwd(dz, signs, None, rs.astype(np.float32), gamma, None, RMS, False)
    np.testing.assert_allclose((dx * xs).sum(1), 0, atol=1e-13)
    # General rows: the same sums vanish up to the fp32 rounding of the stats.
    x = torch.randn(5, H, generator=g) * 3 + 1
    _, mu, rs = orc.norm_fwd(x, gamma, torch.zeros(H), LN, False, 0.0)
    dx, _, _ = orc.norm_bwd(dz, x, mu.astype(np.float32), rs.astype(np.float32), gamma, None,
                            LN, False)
    xh = (x.double().numpy() - mu[:, None]) * rs[:, None]
    scale = np.abs(dx).sum(1)
    assert np.all(np.abs(dx.sum(1)) <= 1e-6 * scale)
    assert np.all(np.abs((dx * xh).sum(1)) <= 1e-6 * scale)


def test_bwd_add_adds_dresidual(orc):
    g = torch.Generator().manual_seed(41)
    x = torch.randn(3, 40, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(40, generator=g)).to(torch.bfloat16)
    dz = torch.randn(3, 40, generator=g).to(torch.bfloat16)
    dres = torch.randn(3, 40, generator=g).to(torch.bfloat16)
    _, _, rs = orc.norm_fwd(x, gamma, None, RMS, False, 1e-6)
    rs32 = rs.astype(np.float32)
    a, ga, _ = orc.norm_bwd(dz, x, None, rs32, gamma, None, RMS, False)
    b, gb, _ = orc.norm_bwd(dz, x, None, rs32, gamma, dres, RMS, False)
    np.testing.assert_allclose(b - a, dres.double().numpy(), rtol=0, atol=1e-14)
    assert np.array_equal(ga, gb)


def test_bwd_zero_centered_gamma_uses_one_plus_gamma(orc):
    x, gamma, _, dz = _grid_case(42, 3, 16)
    _, _, rs = orc.norm_fwd(x, gamma, None, RMS, True, 1e-5)
    rs32 = rs.astype(np.float32)
    a, ga, _ = orc.norm_bwd(dz, x, None, rs32, gamma, None, RMS, True)
    b, gb, _ = orc.norm_bwd(dz, x, None, rs32, gamma + 1, None, RMS, False)  # exact on grid
    np.testing.assert_allclose(a, b, rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(ga, gb, rtol=1e-15, atol=1e-15)


# ---------------------------------------------------------------- GEMM-ready scale order

def test_mxfp8_swizzle_golden_offsets(orc):
    """Offsets worked by hand from the tile description (tests/golden)."""
    R, B = 130, 5
    s = (np.arange(R * B, dtype=np.int64).reshape(R, B) * 7 % 251 + 1).astype(np.uint8)
    out, held = orc.mxfp8_swizzle(s)
    assert out.size == 256 * 8 and held.sum() == R * B
    for r, c, off in read_golden("mxfp8_swizzle.txt"):
        r, c, off = int(r), int(c), int(off)
        assert held[off] and out[off] == s[r, c], (r, c, off)


def test_mxfp8_swizzle_is_a_padded_permutation(orc):
    g = np.random.default_rng(3)
    for R, B in [(128, 4), (1, 1), (300, 9), (256, 160)]:
        s = g.integers(1, 255, size=(R, B)).astype(np.uint8)
        out, held = orc.mxfp8_swizzle(s)
        Rp, Bp = -(-R // 128) * 128, -(-B // 4) * 4
        assert out.size == Rp * Bp
        assert held.sum() == R * B and np.all(out[~held] == 0)
        assert sorted(out[held].tolist()) == sorted(s.ravel().tolist())
        # an exactly tiled matrix: every 512-byte tile holds one 128 x 4 block
        if R % 128 == 0 and B % 4 == 0:
            tiles = out.reshape(R // 128, B // 4, 512)
            for tr in range(R // 128):
                for tc in range(B // 4):
                    blk = s[tr * 128:(tr + 1) * 128, tc * 4:(tc + 1) * 4]
                    assert sorted(tiles[tr, tc].tolist()) == sorted(blk.ravel().tolist())
