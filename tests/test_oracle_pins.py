"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks one oracle function against a value printed on the pages, a published
table, a closed form, an independent library routine or brute force, chosen so that a
plausible slip (a dropped term, a sign, a transposed operand, a wrong bit position) fails.
"""
import math
import os

import numpy as np
import pytest
import torch
from scipy import integrate, stats

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------------------------------
# fp16 rounding: against numpy's correctly rounded double -> half conversion
# ---------------------------------------------------------------------------------------
def test_fp16_round_trip_against_numpy():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
         2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11), 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0],
    ])
    for x in xs:
        with np.errstate(over="ignore"):
            want = np.array([x], np.float64).astype(np.float16).view(np.uint16)[0]
        got = O.double_to_half(float(x))
        assert got == want, (x, hex(got), hex(want))
    for h in range(0, 0x7C00, 7):
        for s in (0, 0x8000):
            want = float(np.array([h | s], np.uint16).view(np.float16)[0])
            assert O.half_to_double(h | s) == want


# ---------------------------------------------------------------------------------------
# Lloyd-Max for N(0,1)
# ---------------------------------------------------------------------------------------
def test_lloyd_max_two_levels_closed_form():
    c, t, mse, _ = O.lloyd_max_normal(2)
    assert np.allclose(c, [-math.sqrt(2 / math.pi), math.sqrt(2 / math.pi)], atol=1e-14)
    assert abs(t[0]) < 1e-15
    assert abs(mse - (1 - 2 / math.pi)) < 1e-13


def test_lloyd_max_against_max_1960_table():
    table, printed = {}, {}
    for row in _rows("max1960_gaussian.txt"):
        table.setdefault(int(row[0]), {})[row[1]] = [float(v) for v in row[2:]]
        printed[(int(row[0]), row[1])] = row[2:]
    for levels, entries in table.items():
        c, t, mse, _ = O.lloyd_max_normal(levels)
        pos = c[levels // 2:]
        assert np.allclose(pos, entries["output"], atol=1.5e-3), (levels, pos)
        if "threshold" in entries:
            assert np.allclose(t[levels // 2:], entries["threshold"], atol=1.5e-3), (levels, t)
        # half a unit of the last printed digit, plus the table's own hand-computation slack
        txt = printed[(levels, "mse")][0]
        tol = 0.5 * 10.0 ** -len(txt.split(".")[1]) + 5e-6
        assert abs(mse - entries["mse"][0]) < tol, (levels, mse)


@pytest.mark.parametrize("levels", [4, 8, 16])
def test_lloyd_max_conditions_by_quadrature(levels):
    """Centroid and midpoint conditions and the MSE, re-derived with numerical quadrature."""
    c, t, mse, _ = O.lloyd_max_normal(levels)
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    total = 0.0
    for j in range(levels):
        a, b = edges[j], edges[j + 1]
        mass = stats.norm.cdf(b) - stats.norm.cdf(a)
        first = integrate.quad(lambda x: x * stats.norm.pdf(x), a, b, epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(first / mass - c[j]) < 1e-9
        total += integrate.quad(lambda x: (x - c[j]) ** 2 * stats.norm.pdf(x), a, b, epsabs=1e-14,
                                epsrel=1e-13)[0]
    assert np.allclose(t, 0.5 * (c[:-1] + c[1:]), atol=1e-15)
    assert abs(total - mse) < 1e-10
    assert np.allclose(c, -c[::-1], atol=1e-14)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_scaling_and_boundaries(bits):
    c64, _, _, _ = O.lloyd_max_normal(1 << bits)
    cents, bnds = O.codebook(bits, 128)
    assert cents.dtype == np.float32 and bnds.dtype == np.float32
    assert np.array_equal(cents, (c64 / math.sqrt(128)).astype(np.float32))
    mids = (0.5 * (cents[:-1].astype(np.float64) + cents[1:].astype(np.float64))).astype(np.float32)
    assert np.array_equal(bnds, mids)
    assert np.all(np.diff(cents) > 0) and np.all(np.diff(bnds) > 0)
    assert bnds[(1 << bits) // 2 - 1] == 0.0


# ---------------------------------------------------------------------------------------
# Rotations
# ---------------------------------------------------------------------------------------
def _planar_params(rng, d=128):
    th = rng.uniform(0, 2 * math.pi, d // 2)
    return np.stack([np.cos(th), np.sin(th)], -1).astype(np.float32).reshape(-1)


def _iso_params(rng, d=128):
    g = rng.standard_normal((d // 4, 4))
    return (g / np.linalg.norm(g, axis=1, keepdims=True)).astype(np.float32).reshape(-1)


def test_fma_counts_printed_on_the_pages():
    rng = np.random.default_rng(1)
    counts = {r[0]: (int(r[1]), int(r[2])) for r in _rows("fma_counts.txt")}
    x = rng.standard_normal(128)
    _, n_planar = O.rotate(O.PLANAR, _planar_params(rng), x)
    _, n_iso = O.rotate(O.ISO, _iso_params(rng), x)
    _, n_dense = O.matvec(np.eye(128), x)
    assert n_planar == counts["planar"][1]
    assert n_iso == counts["iso"][1]
    assert n_dense == counts["dense"][1]
    assert n_dense // n_planar == 64 and n_dense // n_iso == 32


def _dense_params(rng, d=128):
    q, r = np.linalg.qr(rng.standard_normal((d, d)))
    return (q * np.sign(np.diag(r))[None, :]).astype(np.float32)


def test_dense_rotation_cost_matrix_and_inverse():
    """TurboQuant's dense rotation: 16,384 multiply-adds, equal to its matrix, inverse = transpose."""
    rng = np.random.default_rng(70)
    R = _dense_params(rng)
    x = rng.standard_normal(128)
    y, n = O.rotate(O.DENSE, R, x)
    assert n == 16384
    assert np.allclose(y, R.astype(np.float64) @ x, atol=1e-12)
    assert np.array_equal(O.rotation_matrix(O.DENSE, R, 128), R.astype(np.float64))
    back, _ = O.rotate(O.DENSE, R, y, inverse=True)
    assert np.allclose(back, R.astype(np.float64).T @ y, atol=1e-12)
    assert np.allclose(back, x, atol=1e-5)


def test_planar_is_complex_multiplication():
    """(x_2i + i x_2i+1) * exp(i t): an independent statement of the Givens rotation."""
    rng = np.random.default_rng(2)
    p = _planar_params(rng)
    x = rng.standard_normal(128)
    y, _ = O.rotate(O.PLANAR, p, x)
    z = (x[0::2] + 1j * x[1::2]) * (p[0::2].astype(np.float64) + 1j * p[1::2].astype(np.float64))
    assert np.allclose(y[0::2], z.real, atol=1e-13) and np.allclose(y[1::2], z.imag, atol=1e-13)


def _quat_as_complex(q):
    a, b, c, d = q
    return np.array([[a + 1j * b, c + 1j * d], [-c + 1j * d, a - 1j * b]])


def test_iso_is_hamilton_left_product():
    """q (x) x through the 2x2 complex-matrix representation of quaternions."""
    rng = np.random.default_rng(3)
    p = _iso_params(rng)
    x = rng.standard_normal(128)
    y, _ = O.rotate(O.ISO, p, x)
    for blk in range(32):
        q = p[4 * blk:4 * blk + 4].astype(np.float64)
        prod = _quat_as_complex(q) @ _quat_as_complex(x[4 * blk:4 * blk + 4])
        want = np.array([prod[0, 0].real, prod[0, 0].imag, prod[0, 1].real, prod[0, 1].imag])
        assert np.allclose(y[4 * blk:4 * blk + 4], want, atol=1e-13)
    # special case: q = i maps (x0, x1, x2, x3) -> (-x1, x0, -x3, x2)
    qi = np.tile(np.array([0, 1, 0, 0], np.float32), 32)
    y, _ = O.rotate(O.ISO, qi, x)
    assert np.array_equal(y[0:4], [-x[1], x[0], -x[3], x[2]])


def test_right_product_is_a_different_rotation():
    """Negative control: the complex-matrix pin tells the left product from the right one."""
    rng = np.random.default_rng(4)
    q = _iso_params(rng)[:4].astype(np.float64)
    x = rng.standard_normal(4)
    right = _quat_as_complex(x) @ _quat_as_complex(q)
    left, _ = O.rotate(O.ISO, np.tile(q.astype(np.float32), 32), np.tile(x, 32))
    assert not np.allclose(left[:4], [right[0, 0].real, right[0, 0].imag, right[0, 1].real, right[0, 1].imag])


@pytest.mark.parametrize("mode", [O.PLANAR, O.ISO])
def test_rotation_is_orthogonal_and_matches_its_matrix(mode):
    rng = np.random.default_rng(5 + mode)
    p = _planar_params(rng) if mode == O.PLANAR else _iso_params(rng)
    R = O.rotation_matrix(mode, p, 128)
    assert np.abs(R @ R.T - np.eye(128)).max() < 1e-6     # float32 parameters
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    rq, _ = O.rotate(mode, p, q)
    rk, _ = O.rotate(mode, p, k)
    assert np.allclose(rq, R @ q, atol=1e-13)
    assert abs(rq @ rk - q @ k) < 1e-5 * np.linalg.norm(q) * np.linalg.norm(k)
    assert abs(np.linalg.norm(rq) - np.linalg.norm(q)) < 1e-6 * np.linalg.norm(q)
    back, _ = O.rotate(mode, p, rq, inverse=True)
    assert np.allclose(back, R.T @ rq, atol=1e-13)
    assert np.allclose(back, q, atol=1e-5)


# ---------------------------------------------------------------------------------------
# Coding
# ---------------------------------------------------------------------------------------
def _identity_planar():
    return np.tile(np.array([1.0, 0.0], np.float32), 64)


@pytest.mark.parametrize("bits", [3, 4])
def test_codes_are_nearest_centroid_brute_force(bits):
    """With the identity rotation u = x / |x|; boundary counting must equal argmin |u - c|."""
    rng = np.random.default_rng(10 + bits)
    cents, bnds = O.codebook(bits, 128)
    for _ in range(200):
        x = (rng.standard_normal(128) * rng.uniform(0.1, 30)).astype(np.float16)
        codes, n16, margin = O.encode(O.PLANAR, bits, _identity_planar(), bnds, x)
        xd = x.astype(np.float64)
        n = np.linalg.norm(xd)
        u = (xd / n).astype(np.float32).astype(np.float64)
        brute = np.argmin(np.abs(u[:, None] - cents.astype(np.float64)[None, :]), axis=1)
        ok = margin > 1e-6
        assert np.array_equal(codes[ok], brute[ok])
        assert n16 == np.array([n]).astype(np.float16).view(np.uint16)[0]


@pytest.mark.parametrize("bits", [3, 4])
def test_zero_vector_and_ties_take_the_lower_bin(bits):
    _, bnds = O.codebook(bits, 128)
    L = 1 << bits
    codes, n16, _ = O.encode(O.PLANAR, bits, _identity_planar(), bnds, np.zeros(128, np.float16))
    assert n16 == 0 and np.all(codes == L // 2 - 1)
    x = np.zeros(128, np.float16)
    x[7] = 3.0                      # u = e_7: coordinates that are exactly 0 sit on the middle boundary
    codes, _, _ = O.encode(O.PLANAR, bits, _identity_planar(), bnds, x)
    assert codes[0] == L // 2 - 1 and codes[7] == L - 1


@pytest.mark.parametrize("bits,mode", [(3, O.PLANAR), (4, O.ISO)])
def test_codec_distortion_matches_lloyd_max_mse(bits, mode):
    """For Gaussian vectors the relative reconstruction error approaches the Lloyd-Max MSE."""
    rng = np.random.default_rng(20 + bits)
    p = _planar_params(rng) if mode == O.PLANAR else _iso_params(rng)
    cents, bnds = O.codebook(bits, 128)
    _, _, mse, _ = O.lloyd_max_normal(1 << bits)
    errs = []
    for _ in range(300):
        x = rng.standard_normal(128).astype(np.float16)
        codes, n16, _ = O.encode(mode, bits, p, bnds, x)
        xh = O.dequant(mode, bits, p, cents, codes, n16)
        xd = x.astype(np.float64)
        errs.append(np.sum((xd - xh) ** 2) / np.sum(xd ** 2))
    assert abs(np.mean(errs) - mse) < 0.08 * mse, (np.mean(errs), mse)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_dense_rotation_spreads_outliers(bits):
    """The distortion of a dense random rotation (TurboQuant) is an expectation over the draw of
    the rotation: averaged over fresh rotations, keys with x10 outlier channels code to the
    Lloyd-Max MSE of N(0,1).  A block-local rotation (iso) cannot move an outlier out of its
    4-dim block, so the same keys land far above it."""
    rng = np.random.default_rng(80 + bits)
    cents, bnds = O.codebook(bits, 128)
    _, _, mse, _ = O.lloyd_max_normal(1 << bits)
    dense, local = [], []
    for _ in range(200):
        R = _dense_params(rng)
        p = _iso_params(rng)
        x = rng.standard_normal(128)
        x[[3, 40, 77, 101]] *= 10
        x = x.astype(np.float16)
        xd = x.astype(np.float64)
        for mode, rot, errs in ((O.DENSE, R, dense), (O.ISO, p, local)):
            codes, n16, _ = O.encode(mode, bits, rot, bnds, x)
            xh = O.dequant(mode, bits, rot, cents, codes, n16)
            errs.append(np.sum((xd - xh) ** 2) / np.sum(xd ** 2))
    assert abs(np.mean(dense) - mse) < 0.1 * mse, (np.mean(dense), mse)
    assert np.mean(local) > 2.5 * mse, (np.mean(local), mse)


# ---------------------------------------------------------------------------------------
# Packing
# ---------------------------------------------------------------------------------------
def test_pack_4bit_fixture():
    rows = _rows("pack_4bit.txt")
    want = np.array([int(h, 16) for h in rows[1][1:]], np.uint8)
    codes = (np.arange(128) % 16).astype(np.uint8)
    assert np.array_equal(O.pack(4, codes), want)
    assert np.array_equal(O.unpack(4, want), codes)


def test_pack_2bit_fixture():
    rows = _rows("pack_2bit.txt")
    codes = {"i%4": (np.arange(128) % 4).astype(np.uint8), "3-i%4": (3 - np.arange(128) % 4).astype(np.uint8)}
    for i in range(0, len(rows), 2):
        c = codes[rows[i][1]]
        want = np.array([int(h, 16) for h in rows[i + 1][1:]], np.uint8)
        assert want.size == 32
        assert np.array_equal(O.pack(2, c), want)
        assert np.array_equal(O.unpack(2, want), c)


def test_pack_3bit_fixtures():
    with open(os.path.join(GOLD, "pack_3bit.txt")) as f:
        lines = [ln for ln in f if ln.startswith("case")]
    assert len(lines) == 5
    for ln in lines:
        parts = [p.split() for p in ln.split("|")]
        base = int(parts[1][1])
        codes = np.full(128, base, np.uint8)
        for kv in parts[2][1:]:
            dim, code = kv.split("=")
            codes[int(dim)] = int(code)
        want = np.array([int(h, 16) for h in parts[3][1:]], np.uint8)
        assert want.size == 48, parts[0]
        assert np.array_equal(O.pack(3, codes), want), parts[0]
        assert np.array_equal(O.unpack(3, want), codes), parts[0]


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_round_trip_and_sizes(bits):
    rng = np.random.default_rng(30 + bits)
    for _ in range(50):
        codes = rng.integers(0, 1 << bits, 128).astype(np.uint8)
        packed = O.pack(bits, codes)
        assert packed.size == 16 * bits
        assert np.array_equal(O.unpack(bits, packed), codes)
    assert O.page_bytes(bits, 16) == 16 * (32 * bits + 4)
    assert O.page_bytes(bits, 64) == 64 * (32 * bits + 4)


def test_v_placement_fixture():
    for bits, off, unit, offset in (map(int, r) for r in _rows("v_layout.txt")):
        assert O.v_unit_offset(bits, off, unit) == offset, (bits, off, unit)


@pytest.mark.parametrize("bits,P", [(4, 16), (4, 64), (3, 16), (2, 16), (2, 64)])
def test_v_placement_is_a_bijection_onto_the_section(bits, P):
    vb = O.vector_bytes(bits)
    ub = O.v_unit_bytes(bits)
    seen = set()
    for off in range(P):
        for u in range(vb // ub):
            o = O.v_unit_offset(bits, off, u)
            assert o % ub == 0 and 0 <= o < P * vb
            seen.add(o)
    assert len(seen) == P * vb // ub


def test_savings_printed_on_the_pages():
    for bits, pct in ((int(r[0]), int(r[1])) for r in _rows("savings_vs_fp16.txt")):
        saved = 100.0 * (1 - O.vector_bytes(bits, 128) / (128 * 2)) if bits >= 3 else 100.0 * (1 - bits / 16)
        assert int(saved) == pct, (bits, saved)


# ---------------------------------------------------------------------------------------
# Cache layout and attention
# ---------------------------------------------------------------------------------------
def _small_cache(mode, bits, P=16, hq=8, hkv=2, num_pages=6, seed=40):
    rng = np.random.default_rng(seed)
    mk = _planar_params if mode == O.PLANAR else _iso_params
    rk = np.stack([mk(rng) for _ in range(hkv)])
    rv = np.stack([mk(rng) for _ in range(hkv)])
    return O.Cache(mode, bits, hq, hkv, P, num_pages, rk, rv), rng


@pytest.mark.parametrize("bits", [3, 4])
def test_append_places_codes_and_norms_in_the_chunk(bits):
    cache, rng = _small_cache(O.ISO, bits)
    k = rng.standard_normal((3, 2, 128)).astype(np.float16)
    v = rng.standard_normal((3, 2, 128)).astype(np.float16)
    slots = np.array([5, 16 * 3 + 15, -1], np.int32)
    cache.append(k, v, slots)
    vb = O.vector_bytes(bits)
    for t, s in enumerate(slots[:2]):
        page, off = divmod(int(s), 16)
        for h in range(2):
            ch = cache.chunk(page, h)
            ck, nk, _ = O.encode(O.ISO, bits, cache.rot_k[h], cache.boundaries, k[t, h])
            cv, nv, _ = O.encode(O.ISO, bits, cache.rot_v[h], cache.boundaries, v[t, h])
            assert np.array_equal(ch[off * vb:(off + 1) * vb], O.pack(bits, ck))
            assert np.array_equal(O.v_codes_of(bits, ch, 16, off), O.pack(bits, cv))
            norms = ch[32 * vb:].view(np.uint16)
            assert norms[off] == nk and norms[16 + off] == nv
    touched = {(int(s) // 16, h) for s in slots[:2] for h in range(2)}
    for page in range(6):
        for h in range(2):
            if (page, h) not in touched:
                assert not cache.chunk(page, h).any()


def _dequantised(cache, bt, lens):
    """Dense K/V [B][L][Hkv][d] decoded token by token with the oracle's own unpack."""
    B, L = len(lens), int(max(lens))
    vb = O.vector_bytes(cache.bits)
    K = np.zeros((B, L, cache.hkv, 128))
    V = np.zeros_like(K)
    for b in range(B):
        for t in range(int(lens[b])):
            for h in range(cache.hkv):
                ch = cache.chunk(int(bt[b, t // cache.P]), h)
                off = t % cache.P
                norms = ch[2 * cache.P * vb:].view(np.uint16)
                ck = O.unpack(cache.bits, ch[off * vb:(off + 1) * vb])
                cv = O.unpack(cache.bits, O.v_codes_of(cache.bits, ch, cache.P, off))
                K[b, t, h] = O.dequant(cache.mode, cache.bits, cache.rot_k[h], cache.centroids, ck, norms[off])
                V[b, t, h] = O.dequant(cache.mode, cache.bits, cache.rot_v[h], cache.centroids, cv,
                                       norms[cache.P + off])
    return K, V


@pytest.mark.parametrize("mode,bits,T", [(O.PLANAR, 4, 1), (O.ISO, 3, 1), (O.ISO, 3, 3), (O.PLANAR, 3, 4)])
def test_attention_against_torch_sdpa(mode, bits, T):
    cache, rng = _small_cache(mode, bits, num_pages=8)
    lens = np.array([37, 16, 5], np.int32)
    bt = np.array([[3, 0, 6], [7, 0, 0], [1, 0, 0]], np.int32)
    for b, L in enumerate(lens):
        k = (rng.standard_normal((L, 2, 128)) * 2).astype(np.float16)
        v = rng.standard_normal((L, 2, 128)).astype(np.float16)
        pos = np.arange(L)
        cache.append(k, v, (bt[b, pos // 16] * 16 + pos % 16).astype(np.int32))
    q = rng.standard_normal((3, T, 8, 128)).astype(np.float16)
    got = cache.attention(q, bt, lens, T=T)
    K, V = _dequantised(cache, bt, lens)
    for b, L in enumerate(lens):
        qq = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)            # [Hq][T][d]
        kk = torch.from_numpy(K[b, :L]).permute(1, 0, 2).repeat_interleave(4, 0)   # [Hq][L][d]
        vv = torch.from_numpy(V[b, :L]).permute(1, 0, 2).repeat_interleave(4, 0)
        mask = torch.tensor([[t <= L - T + j for t in range(L)] for j in range(T)])
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask)
        assert np.allclose(got[b], ref.permute(1, 0, 2).numpy(), atol=1e-12), (b,)


def test_attention_special_cases():
    cache, rng = _small_cache(O.PLANAR, 4, num_pages=4)
    # every key the same vector: the weights are uniform, the output is the mean of the values
    k = np.repeat(rng.standard_normal((1, 2, 128)).astype(np.float16), 20, axis=0)
    v = rng.standard_normal((20, 2, 128)).astype(np.float16)
    bt = np.array([[2, 1], [0, 0]], np.int32)
    pos = np.arange(20)
    cache.append(k, v, (bt[0, pos // 16] * 16 + pos % 16).astype(np.int32))
    q = rng.standard_normal((2, 1, 8, 128)).astype(np.float16)
    lens = np.array([20, 0], np.int32)
    out = cache.attention(q, bt, lens)
    _, V = _dequantised(cache, bt[:1], lens[:1])
    for hq in range(8):
        assert np.allclose(out[0, 0, hq], V[0, :20, hq // 4].mean(axis=0), atol=1e-12)
    assert not out[1].any()                          # empty sequence -> zeros


def test_dense_attention_against_torch_sdpa():
    rng = np.random.default_rng(50)
    q = rng.standard_normal((2, 2, 8, 128)).astype(np.float16)
    k = rng.standard_normal((2, 9, 2, 128)).astype(np.float16)
    v = rng.standard_normal((2, 9, 2, 128)).astype(np.float16)
    lens = np.array([9, 4], np.int32)
    got = O.attention_dense(q, k, v, lens, 8, 2, T=2)
    for b, L in enumerate(lens):
        qq = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)
        kk = torch.from_numpy(k[b, :L].astype(np.float64)).permute(1, 0, 2).repeat_interleave(4, 0)
        vv = torch.from_numpy(v[b, :L].astype(np.float64)).permute(1, 0, 2).repeat_interleave(4, 0)
        mask = torch.tensor([[t <= L - 2 + j for t in range(L)] for j in range(2)])
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask)
        assert np.allclose(got[b], ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_rotated_space_accumulation_identity():
    """R^T (sum_t p_t c_t n_t) == sum_t p_t (n_t R^T c_t): the kernel's V path in rotated space."""
    rng = np.random.default_rng(60)
    p_rot = _iso_params(rng)
    cents, _ = O.codebook(4, 128)
    codes = rng.integers(0, 16, (10, 128)).astype(np.uint8)
    n16 = np.array([1.5, 2.0, 0.25, 3.0, 1.0, 0.5, 2.5, 1.25, 0.75, 1.75], np.float16).view(np.uint16)
    w = rng.dirichlet(np.ones(10))
    acc = sum(w[t] * float(np.uint16(n16[t]).view(np.float16)) * cents[codes[t]].astype(np.float64)
              for t in range(10))
    once, _ = O.rotate(O.ISO, p_rot, acc, inverse=True)
    each = sum(w[t] * O.dequant(O.ISO, 4, p_rot, cents, codes[t], n16[t]) for t in range(10))
    assert np.allclose(once, each, atol=1e-12)


def _random_tree_masks(rng, B, T):
    """Ancestor masks of random draft trees: draft i's parent is the root (prefix) or an earlier
    draft; draft i sees itself and its ancestors."""
    masks = np.zeros((B, T), np.uint64)
    for b in range(B):
        parent = [-1] + [int(rng.integers(-1, i)) for i in range(1, T)]
        for i in range(T):
            m, j = 0, i
            while j >= 0:
                m |= 1 << j
                j = parent[j]
            masks[b, i] = m
    return masks


def test_tree_attention_against_sdpa_and_chain():
    cache, rng = _small_cache(O.PLANAR, 4, num_pages=8)
    T = 5
    lens = np.array([37, T], np.int32)
    bt = np.array([[3, 0, 6], [7, 0, 0]], np.int32)
    for b, L in enumerate(lens):
        k = (rng.standard_normal((L, 2, 128)) * 2).astype(np.float16)
        v = rng.standard_normal((L, 2, 128)).astype(np.float16)
        pos = np.arange(L)
        cache.append(k, v, (bt[b, pos // 16] * 16 + pos % 16).astype(np.int32))
    q = rng.standard_normal((2, T, 8, 128)).astype(np.float16)
    masks = _random_tree_masks(rng, 2, T)
    got = cache.tree_attention(q, masks, bt, lens)
    K, V = _dequantised(cache, bt, lens)
    for b, L in enumerate(lens):
        qq = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)
        kk = torch.from_numpy(K[b, :L]).permute(1, 0, 2).repeat_interleave(4, 0)
        vv = torch.from_numpy(V[b, :L]).permute(1, 0, 2).repeat_interleave(4, 0)
        vis = torch.tensor([[t < L - T or bool((int(masks[b, j]) >> (t - (L - T))) & 1) for t in range(L)]
                            for j in range(T)])
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=vis)
        assert np.allclose(got[b], ref.permute(1, 0, 2).numpy(), atol=1e-12)
    chain = np.array([[(1 << (j + 1)) - 1 for j in range(T)]] * 2, np.uint64)
    assert np.array_equal(cache.tree_attention(q, chain, bt, lens), cache.attention(q, bt, lens, T=T))
