"""Pins for the float64 oracle: checks against what the pages and the
mathematics fix, never against the oracle's own formulas retyped.

Pins (each a different route to the same fact):
  rotation     scipy's Sylvester Hadamard, a textbook butterfly, orthogonality,
               the one-hot closed form, the outlier example of the RHT page
  generator    SplitMix64 reference outputs, sign balance, Gaussian moments
  codebook     scipy betainc cell masses (stationarity), a second Lloyd-Max
               written on scipy, the b=1 closed form, Max's Gaussian table
  keys         brute-force argmin on tiny inputs
  bit budget   the pages' printed bit counts and memory figures
  distortion   Monte Carlo over the sphere vs the codebook's integral distortion
  values       min/max map to the end codes, error <= scale/2, numpy restatement
  attention    a rotated-frame numpy path, len=1, identical keys, 8-bit limit
  QJL          unbiasedness over many independent Gaussian matrices
  packing      hand-built straddling 3-bit rows
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import integrate, linalg, special

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# rotation: TurboQuant deep dive (cell-devlog) -- Step 1: RHT
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d", [4, 16, 128, 256])
def test_hadamard_matches_scipy_sylvester(oracle, d):
    H = oracle.hadamard(d)
    np.testing.assert_array_equal(H, linalg.hadamard(d))
    np.testing.assert_array_equal(H @ H, d * np.eye(d))  # H symmetric, H H = d I


def _butterfly(x):
    """Textbook radix-2 Walsh-Hadamard butterfly, natural order, unnormalised."""
    x = np.array(x, dtype=np.float64)
    d, h = len(x), 1
    while h < d:
        for i in range(0, d, 2 * h):
            a = x[i:i + h].copy()
            b = x[i + h:i + 2 * h].copy()
            x[i:i + h], x[i + h:i + 2 * h] = a + b, a - b
        h *= 2
    return x


@pytest.mark.parametrize("d", [8, 128])
def test_rotation_equals_signs_then_butterfly_then_scale(oracle, d):
    rng = np.random.default_rng(1)
    s = oracle.signs(42, d)
    for _ in range(5):
        x = rng.standard_normal(d)
        np.testing.assert_allclose(oracle.rotate(s, x), _butterfly(s * x) / math.sqrt(d),
                                   rtol=0, atol=1e-13)


@pytest.mark.parametrize("d", [8, 128])
def test_rotation_orthogonal_and_inverse(oracle, d):
    rng = np.random.default_rng(2)
    s = oracle.signs(7, d)
    R = np.stack([oracle.rotate(s, e) for e in np.eye(d)], axis=1)
    np.testing.assert_allclose(R.T @ R, np.eye(d), rtol=0, atol=1e-14)
    x, y = rng.standard_normal(d), rng.standard_normal(d)
    Rx, Ry = oracle.rotate(s, x), oracle.rotate(s, y)
    assert abs(np.linalg.norm(Rx) - np.linalg.norm(x)) < 1e-13
    assert abs(Rx @ Ry - x @ y) < 1e-12
    np.testing.assert_allclose(oracle.rotate_inverse(s, Rx), x, rtol=0, atol=1e-13)
    # the unsigned transform applied twice gives the sign-flipped input back
    np.testing.assert_allclose(linalg.hadamard(d) @ Rx / math.sqrt(d), s * x, rtol=0, atol=1e-13)
    # "apply the transform again" is not the inverse once the signs are random
    assert not np.allclose(oracle.rotate(s, Rx), x, atol=1e-6)


def test_one_hot_spreads_to_equal_magnitudes(oracle):
    """RHT-effect example: energy on one coordinate ends up spread evenly."""
    d = 128
    s = oracle.signs(42, d)
    e = np.zeros(d)
    e[2] = 1.0
    np.testing.assert_allclose(np.abs(oracle.rotate(s, e)), 1 / math.sqrt(d), rtol=0, atol=1e-16)
    x = np.zeros(d)
    x[:5] = [-0.001, 0.002, 45.3, -0.003, 0.001]
    y = oracle.rotate(s, x)
    assert np.max(np.abs(x)) / np.linalg.norm(x) > 0.999
    assert np.max(np.abs(y)) / np.linalg.norm(y) < 1.01 / math.sqrt(d)


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------

def test_splitmix64_reference_outputs(oracle):
    ref = [int(h, 16) for h in _gold("splitmix64_seed0.json")["state0_outputs_hex"]]
    assert [int(v) for v in oracle.stream(0, 0, 0, 3)] == ref


def test_signs_and_gaussian_statistics(oracle):
    s = np.concatenate([oracle.signs(seed, 128) for seed in range(200)])
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.mean()) < 4 / math.sqrt(s.size)
    S = oracle.gaussian(5, 256, 128).ravel()
    n = S.size
    assert abs(S.mean()) < 4 / math.sqrt(n)
    assert abs(S.var() - 1) < 4 * math.sqrt(2 / n)
    assert abs(np.mean(S ** 4) - 3) < 4 * math.sqrt(96 / n)
    assert not np.array_equal(oracle.signs(1, 128), oracle.signs(2, 128))


# --------------------------------------------------------------------------
# codebook: OCTOPUS summary -- key idea / glossary "Lloyd-Max quantization"
# --------------------------------------------------------------------------

def _beta_cdf(d, x):
    a = (d - 1) / 2.0
    return special.betainc(a, a, (1.0 + np.asarray(x)) / 2.0)


def _moment(d, lo, hi):
    """int_lo^hi x f(x) dx for the sphere marginal, f = (1-x^2)^((d-3)/2) / B(1/2,(d-1)/2)."""
    K = 1.0 / special.beta(0.5, (d - 1) / 2.0)
    e = (d - 1) / 2.0
    return K / (d - 1) * ((1 - lo * lo) ** e - (1 - hi * hi) ** e)


@pytest.mark.parametrize("d", [16, 128])
def test_moment_closed_form_against_quadrature(d):
    K = 1.0 / special.beta(0.5, (d - 1) / 2.0)
    for lo, hi in [(-1, -0.2), (-0.05, 0.1), (0.3, 1.0)]:
        q, _ = integrate.quad(lambda x: x * K * (1 - x * x) ** ((d - 3) / 2), lo, hi,
                              epsabs=1e-16, epsrel=1e-13)
        assert abs(q - _moment(d, lo, hi)) < 1e-14


@pytest.mark.parametrize("d", [4, 16, 128, 256])
def test_density_normalised_with_variance_one_over_d(oracle, d):
    assert abs(oracle.cell_mass(d, -1, 1) - 1) < 1e-14
    var, _ = integrate.quad(lambda x: x * x * oracle.density(d, x), -1, 1, epsabs=1e-15, limit=200)
    assert abs(var - 1.0 / d) < 1e-12
    for lo, hi in [(-1, -0.3), (-0.1, 0.05), (0.2, 0.9)]:
        ref = _beta_cdf(d, hi) - _beta_cdf(d, lo)
        assert abs(oracle.cell_mass(d, lo, hi) - ref) < 1e-14


@pytest.mark.parametrize("d,b", [(16, 2), (64, 3), (128, 1), (128, 2), (128, 3), (128, 4), (256, 4)])
def test_codebook_stationary_and_symmetric(oracle, d, b):
    c, t, passes = oracle.lloyd_max(d, b)
    n = 1 << b
    assert passes < 10000
    assert np.all(np.diff(c) > 0)
    np.testing.assert_allclose(c, -c[::-1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(t, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=0)
    edges = np.concatenate([[-1.0], t, [1.0]])
    mass = np.diff(_beta_cdf(d, edges))
    for i in range(n):
        assert abs(c[i] - _moment(d, edges[i], edges[i + 1]) / mass[i]) < 1e-13


def _scipy_lloyd(d, b, tol=1e-14, max_iter=20000):
    n = 1 << b
    c = (2 * np.arange(n) + 1 - n) / n * 4 / math.sqrt(d)
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        e = np.concatenate([[-1.0], t, [1.0]])
        mass = np.diff(_beta_cdf(d, e))
        cn = _moment(d, e[:-1], e[1:]) / mass
        done = np.max(np.abs(cn - c)) < tol
        c = cn
        if done:
            break
    return c


@pytest.mark.parametrize("d,b", [(128, 2), (128, 3), (128, 4), (64, 4)])
def test_codebook_matches_independent_scipy_lloyd(oracle, d, b):
    c, _, _ = oracle.lloyd_max(d, b)
    np.testing.assert_allclose(c, _scipy_lloyd(d, b), rtol=0, atol=1e-12)


@pytest.mark.parametrize("d", [16, 128, 1024])
def test_one_bit_codebook_closed_form(oracle, d):
    """b = 1: the two cells are the half-lines, so c = +-E|X| = +-Gamma(d/2)/(sqrt(pi)Gamma((d+1)/2))."""
    c, t, _ = oracle.lloyd_max(d, 1)
    e_abs = math.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / math.sqrt(math.pi)
    assert abs(c[1] - e_abs) < 1e-14 and abs(c[0] + e_abs) < 1e-14
    assert abs(t[0]) < 1e-16


@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_codebook_tends_to_gaussian_lloyd_max(oracle, b):
    ref = np.array(_gold("gaussian_lloyd_max.json")["levels"][str(b)])
    d = 4096
    c, _, _ = oracle.lloyd_max(d, b)
    pos = c[len(c) // 2:] * math.sqrt(d)
    np.testing.assert_allclose(pos, ref, rtol=1.5e-3, atol=0)


# --------------------------------------------------------------------------
# keys: Bit-Axon -- quantization function (argmin over the codebook)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("d", [4, 8, 16])
@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_key_codes_are_brute_force_nearest_centroid(oracle, d, b):
    cache = oracle.Cache(d, b, b, 0, 16, 1, 1, seed=3)
    H = linalg.hadamard(d)
    rng = np.random.default_rng(100 * d + b)
    for _ in range(100):
        k = rng.standard_normal(d) * rng.uniform(0.1, 30)
        g, idx, _, _ = cache.encode_key_vector(k)
        assert g == pytest.approx(np.linalg.norm(k), rel=1e-15)
        u_rot = H @ (cache.s * k / np.linalg.norm(k)) / math.sqrt(d)
        expect = np.argmin(np.abs(u_rot[:, None] - cache.C[None, :]), axis=1)
        np.testing.assert_array_equal(idx, expect)


def test_zero_key_reading(oracle):
    cache = oracle.Cache(128, 4, 4, 64, 16, 1, 1, seed=0)
    g, idx, rho, sig = cache.encode_key_vector(np.zeros(128))
    assert g == 0.0 and rho == 0.0
    assert np.all(idx == 7) and np.all(sig == 1)


# --------------------------------------------------------------------------
# bit budget: deep dive -- [PolarQuant compression efficiency], [H100 benchmark];
# Bit-Axon -- KV cache memory model
# --------------------------------------------------------------------------

def test_page_arithmetic_matches_printed_figures(oracle):
    g = _gold("page_arithmetic.json")
    for key in ("key_bits_4bit", "key_bits_3bit"):
        e = g[key]
        bits = e["d"] * e["bits"] + e["norm_bits"]
        assert bits == e["printed_total_bits"]
        assert round(e["d"] * 16 / bits, 1) == e["printed_ratio_vs_fp16"]
    # one page (16 tokens x one KV head) holds exactly the printed per-vector budget
    for kb, vb, m, per_token in [(4, 4, 0, 134), (3, 3, 0, 102), (2, 2, 128, 88)]:
        assert oracle.page_bytes(128, kb, vb, m, 16) == 16 * per_token
    kv_bits = 128 * 4 + 16 + 128 * 4 + 32
    assert kv_bits == 1072 and round(2 * 128 * 16 / kv_bits, 1) == g["kv_savings_tq4"]["printed_ratio_vs_fp16"]
    tq3 = 2 * 128 * 16 / (128 * 3 + 16 + 128 * 3 + 32)
    assert round(tq3, 2) == 5.02 and round(tq3, 1) != g["kv_savings_tq3"]["printed_ratio_vs_fp16"]
    e = g["swa_memory_model"]
    fp16 = e["layers"] * 2 * e["batch"] * e["window"] * e["d_model"] * e["bytes_per_elem_fp16"]
    assert round(fp16 / 1e6, 1) == e["printed_fp16_MB"]
    assert round(fp16 / e["printed_ratio"] / 1e6, 1) == e["printed_q4_MB"]
    # the same window in this cache: 20 heads x 128 dims, codes only, 4+4 bits
    heads = e["d_model"] // 128
    assert e["layers"] * heads * e["window"] * (64 + 64) == fp16 // 4 == 83_886_080
    e = g["llama70b_kv"]
    exact = 2 * e["layers"] * e["kv_heads"] * e["head_dim"] * e["seq_len"] * e["bytes"]
    assert abs(exact / 1e9 - e["printed_GB"]) / e["printed_GB"] < 0.01
    e = g["conservative_per_layer_bits"]
    avg = (16 * 8 + 64 * 4) / e["num_layers"]
    assert avg == 4.8 and avg != e["printed_avg_bits"]


# --------------------------------------------------------------------------
# distortion (Monte Carlo over the sphere)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_sphere_distortion_matches_integral(oracle, b):
    d = 128
    cache = oracle.Cache(d, b, b, 8, 16, 1, 1, seed=11)
    c, t = cache.C, cache.T
    edges = np.concatenate([[-1.0], t, [1.0]])
    K = 1.0 / special.beta(0.5, (d - 1) / 2.0)
    Db = sum(integrate.quad(lambda x: (x - c[i]) ** 2 * K * (1 - x * x) ** ((d - 3) / 2),
                            edges[i], edges[i + 1], epsabs=1e-15, limit=200)[0]
             for i in range(len(c)))
    survey = {1: 0.3609, 2: 0.1160, 3: 0.03397, 4: 0.009315}
    assert abs(d * Db - survey[b]) / survey[b] < 2e-4
    rng = np.random.default_rng(500 + b)
    N = 8000
    err = np.empty(N)
    for i in range(N):
        u = rng.standard_normal(d)
        _, _, rho, _ = cache.encode_key_vector(u)  # rho = ||u_rot - C[idx]|| for a unit u
        err[i] = rho ** 2
    se = err.std() / math.sqrt(N)
    assert abs(err.mean() - d * Db) < 4 * se


# --------------------------------------------------------------------------
# values: deep dive -- Step 3 (min-max value codes)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("b", [2, 3, 4, 8])
def test_value_codes_min_max(oracle, b):
    d = 128
    cache = oracle.Cache(d, 4, b, 0, 16, 1, 1, seed=9)
    H = linalg.hadamard(d)
    rng = np.random.default_rng(b)
    qmax = (1 << b) - 1
    for _ in range(50):
        v = rng.standard_normal(d) * rng.uniform(0.01, 50)
        sc, zr, q = cache.encode_value_vector(v)
        vr = H @ (cache.s * v) / math.sqrt(d)
        assert zr == vr.min() or abs(zr - vr.min()) < 1e-13 * abs(vr).max()
        assert abs(sc - (vr.max() - vr.min()) / qmax) < 1e-13 * abs(vr).max()
        assert q[np.argmin(vr)] == 0 and q[np.argmax(vr)] == qmax
        assert np.all((q >= 0) & (q <= qmax))
        np.testing.assert_array_equal(q, np.clip(np.rint((vr - vr.min()) / sc), 0, qmax))
        assert np.max(np.abs(q * sc + zr - vr)) <= sc / 2 * (1 + 1e-9)


def test_constant_value_vector_gives_zero_scale(oracle):
    d = 16
    cache = oracle.Cache(d, 2, 2, 0, 16, 1, 1, seed=0)
    e = np.zeros(d)
    e[0] = 0.0
    sc, zr, q = cache.encode_value_vector(e)
    assert sc == 0.0 and zr == 0.0 and np.all(q == 0)


def test_fp16_rounding_matches_numpy(oracle):
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 6, 2000),
                         [65504.0, 65519.9, 65520.0, 1e-8, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                          0.1, -0.1, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]])
    for x in xs:
        with np.errstate(over="ignore"):
            ref = np.float16(x)
        assert oracle.fp16_round(x) == float(ref) or (np.isinf(ref) and np.isinf(oracle.fp16_round(x)))
        assert oracle.fp16_bits(x) == int(ref.view(np.uint16))
        assert oracle.fp16_value(int(ref.view(np.uint16))) == float(ref)


# --------------------------------------------------------------------------
# attention: Bit-Axon -- attention under quantized KV
# --------------------------------------------------------------------------

def _encode_simple(cache, K, V, lens, rng):
    """Write each sequence into its own randomly chosen blocks."""
    B = len(lens)
    nb_per = max(1, (max(lens) + cache.bs - 1) // cache.bs)
    perm = rng.permutation(cache.num_blocks)[: B * nb_per].reshape(B, nb_per)
    pool = cache.new_pool()
    for b in range(B):
        L = lens[b]
        slots = perm[b, np.arange(L) // cache.bs] * cache.bs + np.arange(L) % cache.bs
        assert cache.encode(K[b, :L], V[b, :L], slots, pool) == 0
    return pool, perm.astype(np.int32)


def _rotated_frame_decode(cache, pool, q, bt, lens, sm_scale):
    """Second route: logits in the rotated frame straight from the stored fields,
    values accumulated in the rotated frame, one inverse transform at the end."""
    d = cache.d
    H = linalg.hadamard(d) / math.sqrt(d)
    B, Hq, _ = q.shape
    G = Hq // cache.hkv
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(cache.hkv):
            rows = [cache.unpack_slot(pool, bt[b, t // cache.bs], h, t % cache.bs) for t in range(lens[b])]
            if not rows:
                continue
            Chat = np.stack([cache.C[r["kidx"]] for r in rows])
            gam = np.array([r["gamma"] for r in rows])
            Vr = np.stack([r["scale"] * r["vq"] + r["zero"] for r in rows])
            for g in range(G):
                qr = H @ (cache.s * q[b, h * G + g])
                logit = gam * (Chat @ qr)
                if cache.m:
                    sq = cache.S @ qr
                    sgn = np.stack([2 * r["sig"] - 1 for r in rows])
                    rho = np.array([r["rho"] for r in rows])
                    logit = logit + gam * math.sqrt(math.pi / 2) / cache.m * rho * (sgn @ sq)
                logit = logit * sm_scale
                p = np.exp(logit - logit.max())
                acc = p @ Vr / p.sum()
                out[b, h * G + g] = cache.s * (H @ acc)
    return out


@pytest.mark.parametrize("kb,vb,m,G", [(4, 4, 0, 1), (3, 3, 0, 4), (2, 2, 32, 2), (4, 2, 16, 1)])
def test_decode_matches_rotated_frame_route(oracle, kb, vb, m, G):
    d, hkv, bs = 32, 2, 16
    rng = np.random.default_rng(kb * 100 + vb * 10 + m)
    cache = oracle.Cache(d, kb, vb, m, bs, hkv, 16, seed=5)
    lens = [37, 16, 1]
    B = len(lens)
    K = rng.standard_normal((B, max(lens), hkv, d)) * 3
    V = rng.standard_normal((B, max(lens), hkv, d))
    q = rng.standard_normal((B, hkv * G, d))
    pool, bt = _encode_simple(cache, K, V, lens, rng)
    sm = 1 / math.sqrt(d)
    out, st = cache.decode(pool, q, bt, np.array(lens), sm)
    assert st == 0
    ref = _rotated_frame_decode(cache, pool, q, bt, lens, sm)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_decode_single_token_and_identical_keys(oracle):
    d, hkv = 16, 1
    cache = oracle.Cache(d, 4, 4, 0, 16, hkv, 4, seed=1)
    rng = np.random.default_rng(0)
    V = rng.standard_normal((1, 20, hkv, d))
    K = np.repeat(rng.standard_normal((1, 1, hkv, d)), 20, axis=1)
    pool, bt = _encode_simple(cache, K, V, [20], rng)
    q = rng.standard_normal((1, 1, d))
    vhat = []
    for t in range(20):
        r = cache.unpack_slot(pool, bt[0, t // 16], 0, t % 16)
        vhat.append(oracle.rotate_inverse(cache.s, r["scale"] * r["vq"] + r["zero"]))
    vhat = np.array(vhat)
    out, _ = cache.decode(pool, q, bt, np.array([1]), 0.3)
    np.testing.assert_allclose(out[0, 0], vhat[0], rtol=0, atol=1e-13)
    out, _ = cache.decode(pool, q, bt, np.array([20]), 0.3)
    np.testing.assert_allclose(out[0, 0], vhat.mean(axis=0), rtol=0, atol=1e-13)
    out, _ = cache.decode(pool, q, bt, np.array([0]), 0.3)
    assert np.all(out == 0)


def test_decode_error_within_value_quantization_bound(oracle):
    """With logits near zero the key codes hardly matter and the output error is
    the value quantisation error, bounded per coordinate by sqrt(d) * scale / 2
    (the rotation maps a rotated-frame error of at most scale/2 per coordinate to
    at most sqrt(d) scale / 2 in any original coordinate), plus fp16 effects."""
    d, hkv, T = 64, 1, 40
    rng = np.random.default_rng(4)
    K = rng.standard_normal((1, T, hkv, d))
    V = rng.standard_normal((1, T, hkv, d))
    q = rng.standard_normal((1, 1, d)) * 1e-9
    p = np.ones(T) / T
    exact = p @ V[0, :, 0]
    errs = {}
    for vb in (2, 4, 8):
        cache = oracle.Cache(d, 4, vb, 0, 16, hkv, 8, seed=2)
        pool, bt = _encode_simple(cache, K, V, [T], rng)
        out, _ = cache.decode(pool, q, bt, np.array([T]), 1 / math.sqrt(d))
        errs[vb] = np.abs(out[0, 0] - exact).max()
        scales = [cache.unpack_slot(pool, bt[0, t // 16], 0, t % 16)["scale"] for t in range(T)]
        assert errs[vb] <= math.sqrt(d) * max(scales) / 2 * 1.01 + 1e-3
    assert errs[8] < errs[4] < errs[2]
    assert errs[8] < 0.02


def test_decode_flags_bad_block(oracle):
    d = 16
    cache = oracle.Cache(d, 4, 4, 0, 16, 1, 4, seed=1)
    rng = np.random.default_rng(1)
    pool, bt = _encode_simple(cache, rng.standard_normal((1, 20, 1, d)),
                              rng.standard_normal((1, 20, 1, d)), [20], rng)
    bt2 = bt.copy()
    bt2[0, 1] = 99
    out, st = cache.decode(pool, rng.standard_normal((1, 1, d)), bt2, np.array([20]), 0.25)
    assert st & oracle.FLAG_BAD_SLOT and np.all(np.isfinite(out))
    st = cache.encode(np.zeros((1, 1, d)), np.zeros((1, 1, d)), np.array([4 * 16]), cache.new_pool())
    assert st & oracle.FLAG_BAD_SLOT


# --------------------------------------------------------------------------
# QJL: OCTOPUS summary -- "Optional 1-bit QJL residual", methodology step 8
# --------------------------------------------------------------------------

def test_qjl_correction_is_unbiased(oracle):
    d, m = 128, 64
    rng = np.random.default_rng(8)
    k = rng.standard_normal(d) * 2
    q = rng.standard_normal(d)
    base = oracle.Cache(d, 2, 2, m, 16, 1, 1, seed=0)
    qr = oracle.rotate(base.s, q)
    g, idx, _, _ = base.encode_key_vector(k)
    u_rot = oracle.rotate(base.s, k / g)
    r = u_rot - base.C[idx]
    target = g * (qr @ r)
    est = []
    for seed in range(1, 3001):
        S = oracle.gaussian(seed, m, d)
        sig = (S @ r >= 0).astype(np.float64) * 2 - 1
        est.append(g * math.sqrt(math.pi / 2) / m * np.linalg.norm(r) * ((S @ qr) @ sig))
    est = np.array(est)
    assert abs(est.mean() - target) < 4 * est.std() / math.sqrt(len(est))
    # the oracle's own sketch for one seed is the same sign pattern
    c2 = oracle.Cache(d, 2, 2, m, 16, 1, 1, seed=17)
    _, idx2, rho2, sig2 = c2.encode_key_vector(k)
    r2 = oracle.rotate(c2.s, k / g) - c2.C[idx2]
    np.testing.assert_array_equal(sig2, (c2.S @ r2 >= 0).astype(int))
    assert abs(rho2 - np.linalg.norm(r2)) < 1e-14


def test_qjl_variance_shrinks_with_m(oracle):
    d = 64
    rng = np.random.default_rng(9)
    r = rng.standard_normal(d)
    qr = rng.standard_normal(d)
    var = {}
    for m in (16, 64):
        est = []
        for seed in range(1, 801):
            S = oracle.gaussian(seed, m, d)
            est.append(math.sqrt(math.pi / 2) / m * np.linalg.norm(r) * ((S @ qr) @ np.where(S @ r >= 0, 1, -1)))
        var[m] = np.var(est)
    assert 2.5 < var[16] / var[64] < 6.5


# --------------------------------------------------------------------------
# packing
# --------------------------------------------------------------------------

def test_three_bit_rows_straddle_bytes(oracle):
    d, kb, vb = 8, 3, 3
    cache = oracle.Cache(d, kb, vb, 0, 16, 1, 1, seed=0)
    pool = cache.new_pool()
    codes = [1, 7, 2, 5, 0, 6, 3, 4]
    bits = sum(c << (3 * j) for j, c in enumerate(codes))  # LSB-first bit string
    pool[0:3] = np.frombuffer(bits.to_bytes(3, "little"), dtype=np.uint8)
    r = cache.unpack_slot(pool, 0, 0, 0)
    np.testing.assert_array_equal(r["kidx"], codes)
    # code 2 of the row occupies bits 6..8, across bytes 0 and 1
    assert (pool[0] >> 6) | ((pool[1] & 1) << 2) == codes[2]


@pytest.mark.parametrize("kb,vb,m", [(4, 4, 0), (3, 3, 0), (2, 2, 128), (1, 8, 8)])
def test_encode_then_unpack_roundtrip(oracle, kb, vb, m):
    d, hkv = 128, 3
    cache = oracle.Cache(d, kb, vb, m, 16, hkv, 4, seed=6)
    rng = np.random.default_rng(kb)
    K = rng.standard_normal((5, hkv, d)) * 4
    V = rng.standard_normal((5, hkv, d))
    slots = np.array([17, 3, 63, 40, -1])
    pool = cache.new_pool()
    assert cache.encode(K, V, slots, pool) == 0
    for t in range(4):
        for h in range(hkv):
            r = cache.unpack_slot(pool, slots[t] // 16, h, slots[t] % 16)
            g, idx, rho, sig = cache.encode_key_vector(K[t, h])
            sc, zr, q = cache.encode_value_vector(V[t, h])
            np.testing.assert_array_equal(r["kidx"], idx)
            np.testing.assert_array_equal(r["vq"], q)
            assert r["gamma"] == oracle.fp16_round(g) and r["scale"] == oracle.fp16_round(sc)
            assert r["zero"] == oracle.fp16_round(zr)
            if m:
                np.testing.assert_array_equal(r["sig"], sig)
                assert r["rho"] == oracle.fp16_round(rho)


@pytest.mark.parametrize("T", [40, 64, 112, 208])
def test_ring_window_equals_linear_window(oracle, T):
    """A sliding window kept as a ring of W slots (token t in slot t mod W)
    holds the last W tokens; since attention does not depend on token order,
    decoding the ring over min(T, W) slots equals decoding a linear cache of
    all T tokens over its last W tokens (T - W is a whole number of blocks
    here, so those tokens are whole pages of the linear cache)."""
    d, hkv, bs, W_ = 16, 2, 16, 64
    rng = np.random.default_rng(T)
    K = rng.standard_normal((T, hkv, d)) * 2
    V = rng.standard_normal((T, hkv, d))
    q = rng.standard_normal((1, 2 * hkv, d))
    lin = oracle.Cache(d, 4, 4, 0, bs, hkv, 32, seed=3)
    ring = oracle.Cache(d, 4, 4, 0, bs, hkv, 32, seed=3)
    blocks = rng.permutation(32)
    lin_bt = blocks[: (T + bs - 1) // bs].astype(np.int32)[None, :]
    ring_bt = blocks[16: 16 + W_ // bs].astype(np.int32)[None, :]
    pool_l, pool_r = lin.new_pool(), ring.new_pool()
    t = np.arange(T)
    assert lin.encode(K, V, lin_bt[0, t // bs].astype(np.int64) * bs + t % bs, pool_l) == 0
    for c0 in range(0, T, W_):  # in order, one window at a time, so no two tokens of a call share a slot
        tc = t[c0: c0 + W_]
        assert ring.encode(K[tc], V[tc], ring_bt[0, (tc % W_) // bs].astype(np.int64) * bs + tc % bs, pool_r) == 0
    n = min(T, W_)
    out_r, st = ring.decode(pool_r, q, ring_bt, np.array([n]), 0.25)
    assert st == 0
    first = (T - n) // bs
    out_l, st = lin.decode(pool_l, q, np.ascontiguousarray(lin_bt[:, first:]), np.array([n]), 0.25)
    assert st == 0
    np.testing.assert_allclose(out_r, out_l, rtol=0, atol=1e-12 * np.abs(out_l).max())
