"""Pins of the oracle's OCTOPUS triplet codec against what the OCTOPUS page and
the mathematics fix: the octahedral map is a bijection of the sphere onto the
square, the densities its codebooks are fitted to integrate to one and agree
with sampling, the codebooks are stationary, joint rounding never loses to
independent rounding, and the distortion lands near the page's printed
figures."""
import json
import math
import os

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _unit(rng, n, dim):
    x = rng.standard_normal((n, dim))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def test_octahedral_map_round_trip(oracle):
    rng = np.random.default_rng(0)
    for n in _unit(rng, 2000, 3):
        xi, eta = oracle.oct_map(n)
        assert -1.0 <= xi <= 1.0 and -1.0 <= eta <= 1.0
        np.testing.assert_allclose(oracle.oct_inverse(xi, eta), n, rtol=0, atol=1e-14)
    # the axes and the fold
    for n, want in (((0, 0, 1), (0, 0)), ((1, 0, 0), (1, 0)), ((0, -1, 0), (0, -1)), ((0, 0, -1), (1, 1))):
        assert oracle.oct_map(np.array(n, float)) == pytest.approx(want)
    # every point of the square is a unit direction
    for xi, eta in rng.uniform(-1, 1, (500, 2)):
        assert np.linalg.norm(oracle.oct_inverse(xi, eta)) == pytest.approx(1.0, abs=1e-14)


def test_octahedral_density_normalised_and_matches_sampling(oracle):
    assert oracle.oct_cell_mass(0, 128, -1.0, 1.0) == pytest.approx(1.0, abs=1e-10)
    rng = np.random.default_rng(1)
    xs = np.array([oracle.oct_map(n)[0] for n in _unit(rng, 200000, 3)])
    edges = np.linspace(-1, 1, 21)
    counts, _ = np.histogram(xs, edges)
    for i in range(20):
        p = oracle.oct_cell_mass(0, 128, edges[i], edges[i + 1])
        se = math.sqrt(len(xs) * p * (1 - p))
        assert abs(counts[i] - len(xs) * p) < 4 * se, (i, counts[i], len(xs) * p)


@pytest.mark.parametrize("d", [16, 128])
def test_triplet_norm_density(oracle, d):
    """rho^2 of three coordinates of a uniform point on S^{d-1} is Beta(3/2, (d-3)/2):
    mass 1, E[rho^2] = 3/d, and the histogram of sampled norms."""
    assert oracle.oct_cell_mass(1, d, 0.0, 1.0) == pytest.approx(1.0, abs=1e-10)
    r = np.linspace(0, 1, 200001)
    f = np.array([oracle.rho_density(d, x) for x in r])
    assert np.trapezoid(r * r * f, r) == pytest.approx(3.0 / d, rel=1e-6)
    rng = np.random.default_rng(2)
    u = _unit(rng, 100000, d)
    rho = np.linalg.norm(u[:, :3], axis=1)
    edges = np.linspace(0, rho.max() + 1e-9, 16)
    counts, _ = np.histogram(rho, edges)
    for i in range(15):
        p = oracle.oct_cell_mass(1, d, edges[i], edges[i + 1])
        se = math.sqrt(len(rho) * p * (1 - p)) + 1
        assert abs(counts[i] - len(rho) * p) < 4 * se


@pytest.mark.parametrize("kind,bits", [(0, 3), (0, 5), (1, 1), (1, 3)])
def test_codebooks_stationary(oracle, kind, bits):
    """Each level is the conditional mean of its cell (checked by trapezoid
    integration on a fine grid, independent of the quadrature the iteration
    uses); the xi codebook is symmetric."""
    d = 128
    c, t, _ = oracle.oct_codebook(kind, d, bits)
    lo = -1.0 if kind == 0 else 0.0
    dens = oracle.oct_marginal if kind == 0 else (lambda x: oracle.rho_density(d, x))
    edges = np.concatenate([[lo], t, [1.0]])
    for i in range(len(c)):
        x = np.linspace(edges[i], edges[i + 1], 4001)
        f = np.array([dens(v) for v in x])
        m = np.trapezoid(f, x)
        if m < 1e-12:
            continue
        assert np.trapezoid(x * f, x) / m == pytest.approx(c[i], abs=2e-7)
    assert np.all(np.diff(c) > 0)
    if kind == 0:
        np.testing.assert_allclose(c, -c[::-1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("b", [2, 3, 4])
def test_joint_rounding_never_loses_to_independent_rounding(oracle, b):
    c = oracle.OctCache(128, b, 4, 16, 1, 1, 0)
    rng = np.random.default_rng(b)
    for t in rng.standard_normal((3000, 3)) * 0.1:
        a, e, r, sc = c.encode_triplet(t)
        n = t / np.linalg.norm(t)
        xi, eta = oracle.oct_map(n)
        ia = int(np.searchsorted(c.Txi, xi, side="left"))
        ie = int(np.searchsorted(c.Txi, eta, side="left"))
        indep = n @ oracle.oct_inverse(c.Cxi[ia], c.Cxi[ie])
        assert sc >= indep - 1e-15
        assert n @ oracle.oct_inverse(c.Cxi[a], c.Cxi[e]) == pytest.approx(sc, abs=1e-15)
        assert abs(a - ia) <= 1 and abs(e - ie) <= 1
        assert r == int(np.searchsorted(c.Trho, np.linalg.norm(t), side="left"))


@pytest.mark.parametrize("b", [2, 3, 4])
def test_distortion_near_the_page_figures(oracle, b):
    """E||u - u^||^2 and the mean cosine for u uniform on S^127 land within 10 %
    (MSE) and 0.005 (cos) of the figures the page prints for its codec."""
    g = json.load(open(os.path.join(GOLD, "octopus_synthetic.json")))["printed"][str(b)]
    c = oracle.OctCache(128, b, 4, 16, 1, 1, 0)
    rng = np.random.default_rng(10 + b)
    errs, coss = [], []
    for x in _unit(rng, 1500, 128):
        _, a, e, r = c.encode_key_vector(x)
        uh = c.direction(a, e, r)
        u = oracle.rotate(c.s, x)
        errs.append(np.sum((u - uh) ** 2))
        coss.append(u @ uh / np.linalg.norm(uh))
    assert np.mean(errs) == pytest.approx(g["mse"], rel=0.10)
    assert np.mean(coss) == pytest.approx(g["cos"], abs=0.005)


def test_octopus_encode_unpack_and_decode_invariants(oracle):
    """Codes written to a page read back as encoded; one token gives out = V^_0;
    identical keys give the mean of the values."""
    d, hkv, b, vb = 128, 2, 3, 4
    c = oracle.OctCache(d, b, vb, 16, hkv, 4, 7)
    rng = np.random.default_rng(3)
    T = 20
    K = np.repeat(rng.standard_normal((1, hkv, d)), T, axis=0)
    V = rng.standard_normal((T, hkv, d))
    pool = c.new_pool()
    slots = np.arange(T) + 16
    assert c.encode(K, V, slots, pool) == 0
    g, a, e, r = c.encode_key_vector(K[0, 1])
    u = c.unpack_slot(pool, 1, 1, 3)
    assert np.array_equal(u["ixi"], a) and np.array_equal(u["ieta"], e) and np.array_equal(u["irho"], r)
    assert u["gamma"] == oracle.fp16_value(int(np.float16(g).view(np.uint16)))
    vhat = np.array([[oracle.rotate_inverse(c.s, v["scale"] * v["vq"] + v["zero"])
                      for v in (c.unpack_slot(pool, (16 + t) // 16, h, (16 + t) % 16) for h in range(hkv))]
                     for t in range(T)])
    bt = np.array([[1, 2]], dtype=np.int32)
    q = rng.standard_normal((1, 2 * hkv, d))
    out, st = c.decode(pool, q, bt, np.array([1]), 0.1)
    assert st == 0
    for h in range(hkv):
        np.testing.assert_allclose(out[0, 2 * h], vhat[0, h], rtol=0, atol=1e-12)
    out, st = c.decode(pool, q, bt, np.array([T]), 0.1)
    for h in range(hkv):
        np.testing.assert_allclose(out[0, 2 * h + 1], vhat[:, h].mean(axis=0), rtol=0, atol=1e-12)


def _rotated_frame_decode(oracle, c, pool, q, bt, lens, sm_scale, swap=False):
    """A second route to the OCTOPUS decode, independent of the oracle's decode
    loop: fields read by the numpy page reader, the unit keys rebuilt by
    OctCache.direction (pinned by the distortion test), logits in the rotated
    frame, gamma_t sm_scale <R q, u^_t>, values accumulated in the rotated
    frame, then one inverse rotation per output ["OCTOPUS ..." -- step 7:
    attention from the codes without materialising K^].  swap=True exchanges
    xi and eta: a planted mistake the comparison must catch."""
    from tests import parity
    B, hq, d = q.shape
    G = hq // c.hkv
    out = np.zeros_like(q)
    for b in range(B):
        n = int(lens[b])
        if n == 0:
            continue
        t = np.arange(n)
        slots = bt[b, t // c.bs].astype(np.int64) * c.bs + t % c.bs
        for h in range(c.hkv):
            f = parity.unpack_octopus(pool, d, c.b, c.vb, c.bs, c.hkv, c.page_bytes, slots, np.full(n, h))
            a_, e_ = (f["ieta"], f["ixi"]) if swap else (f["ixi"], f["ieta"])
            U = np.stack([c.direction(a_[i], e_[i], f["irho"][i]) for i in range(n)])
            Vr = f["scale"][:, None] * f["vq"] + f["zero"][:, None]
            for g in range(G):
                qh = h * G + g
                logit = sm_scale * f["gamma"] * (U @ oracle.rotate(c.s, q[b, qh]))
                p = np.exp(logit - logit.max())
                out[b, qh] = oracle.rotate_inverse(c.s, (p @ Vr) / p.sum())
    return out


@pytest.mark.parametrize("b,G", [(2, 1), (3, 4), (4, 2)])
def test_decode_matches_rotated_frame_route(oracle, b, G):
    """The oracle's OCTOPUS decode (keys rebuilt, rotated back, plain softmax)
    against the rotated-frame route above on random distinct keys, ragged
    lengths and a permuted block table: agreement to 1e-12, while the same
    route with xi and eta swapped is far off."""
    d, hkv, vb, bs = 128, 2, 4, 16
    lens = np.array([37, 70])
    nbk = 5
    c = oracle.OctCache(d, b, vb, bs, hkv, 2 * nbk, 11)
    rng = np.random.default_rng(20 + b)
    bt = rng.permutation(2 * nbk).reshape(2, nbk).astype(np.int32)
    pool = c.new_pool()
    for s in range(2):
        K = rng.standard_normal((lens[s], hkv, d))
        K[:, :, rng.choice(d, 4, replace=False)] *= 20.0
        V = rng.standard_normal((lens[s], hkv, d))
        t = np.arange(lens[s])
        assert c.encode(K, V, bt[s, t // bs].astype(np.int64) * bs + t % bs, pool) == 0
    q = rng.standard_normal((2, hkv * G, d)) * 3.0
    sm = 1.0 / math.sqrt(d)
    out, st = c.decode(pool, q, bt, lens, sm)
    assert st == 0
    ref = _rotated_frame_decode(oracle, c, pool, q, bt, lens, sm)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    bad = _rotated_frame_decode(oracle, c, pool, q, bt, lens, sm, swap=True)
    assert np.abs(bad - ref).max() > 1e-3 * np.abs(ref).max()


def test_numpy_page_reader_matches_encoder_codes(oracle):
    """The numpy reader gives back the codes and fp16 fields the oracle's key
    and value encoders produce for each slot."""
    from tests import parity
    d, b, vb, bs, hkv = 128, 3, 3, 16, 1
    c = oracle.OctCache(d, b, vb, bs, hkv, 2, 5)
    rng = np.random.default_rng(4)
    K = rng.standard_normal((20, hkv, d))
    V = rng.standard_normal((20, hkv, d))
    pool = c.new_pool()
    slots = np.arange(20) + 5
    assert c.encode(K, V, slots, pool) == 0
    f = parity.unpack_octopus(pool, d, b, vb, bs, hkv, c.page_bytes, slots, np.zeros(20, dtype=np.int64))
    for t in range(20):
        g, a, e, r = c.encode_key_vector(K[t, 0])
        assert np.array_equal(f["ixi"][t], a) and np.array_equal(f["ieta"][t], e) and np.array_equal(f["irho"][t], r)
        assert f["gamma"][t] == float(np.float16(g))
        assert np.array_equal(f["vq"][t], c.unpack_slot(pool, int(slots[t]) // bs, 0, int(slots[t]) % bs)["vq"])
