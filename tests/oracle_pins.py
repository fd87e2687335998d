"""Pins of the CPU oracle to facts outside itself (no GPU).

Each ``check_*`` takes an oracle handle (``oracle.Oracle``) and raises AssertionError when the
oracle disagrees with the fact it is pinned to.  ``test_oracle_pins.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` runs them on deliberately broken copies of the oracle source
and requires every copy to fail at least one of them.

What pins what:
  * Haar filters  -- the sign patterns printed on page 4, section 3 (tests/golden/haar_filters.txt)
  * analysis / synthesis -- perfect reconstruction and Parseval (orthonormal transform)
  * dwconv -- torch.nn.functional.conv2d in float64 (a library routine)
  * forward -- (i) zero wavelet scales reduce the layer to a scaled depthwise conv + bias;
    (ii) delta kernels with one scale a_l per level give the closed form
    y = s_b (x + b) + sum_l a_l P_(l-1) x, with P_j the 2^j x 2^j block mean;
    (iii) a dense matrix of the whole layer assembled stage by stage on 8x8 / 16x16 planes
  * backward -- dx = M^T dy from the same dense matrix; central finite differences (exact up to
    rounding, since the layer is affine in x and in each single parameter); Euler identities
"""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_haar_filters() -> tuple[float, dict[str, np.ndarray]]:
    scale, pats = None, {}
    with open(os.path.join(GOLDEN, "haar_filters.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "scale":
                scale = float(parts[1])
            else:
                pats[parts[0]] = np.array([float(v) for v in parts[1:]]).reshape(2, 2)
    return scale, pats


def random_params(rng, C, L, k, zero_wavelet_scale=False):
    p = {
        "base_w": rng.standard_normal((C, k, k)) / k,
        "base_bias": rng.standard_normal(C) * 0.3,
        "base_scale": rng.uniform(0.5, 1.5, C),
        "wavelet_w": rng.standard_normal((L, 4 * C, k, k)) / k,
        "wavelet_scale": rng.uniform(0.05, 0.2, (L, 4 * C)),
    }
    if zero_wavelet_scale:
        p["wavelet_scale"][:] = 0.0
    return p


def _close(a, b, tol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    ref = max(float(np.max(np.abs(b))) if b.size else 0.0, 1e-300)
    assert err <= tol * ref, f"{what}: max abs err {err:.3e} > {tol:.1e} * {ref:.3e}"


# ----------------------------------------------------------------------------- transform pins

def check_haar_filters(orc):
    """Each impulse in a 2x2 block reproduces the printed filter taps (x 0.5)."""
    scale, pats = load_haar_filters()
    for a in range(2):
        for b in range(2):
            x = np.zeros((2, 2))
            x[a, b] = 1.0
            y = orc.haar_analysis(x)
            for s, name in enumerate(("LL", "LH", "HL", "HH")):
                want = scale * pats[name][a, b]
                assert y[s, 0, 0] == want, f"subband {name} tap ({a},{b}): {y[s,0,0]} != {want}"


def check_perfect_reconstruction(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((12, 16))
    _close(orc.haar_synthesis(orc.haar_analysis(x)), x, 1e-14, "IWT(WT(x))")
    c = rng.standard_normal((4, 5, 3))
    _close(orc.haar_analysis(orc.haar_synthesis(c)), c, 1e-14, "WT(IWT(c))")


def check_parseval(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 8))
    e0 = float(np.sum(x * x))
    e1 = float(np.sum(orc.haar_analysis(x) ** 2))
    assert abs(e0 - e1) <= 1e-12 * e0, f"Parseval: {e0} vs {e1}"


def check_dwconv_library(orc):
    rng = np.random.default_rng(3)
    for k in (1, 3, 5, 7):
        for H, W in ((9, 13), (4, 4), (16, 6)):
            x = rng.standard_normal((H, W))
            w = rng.standard_normal((k, k))
            ref = torch.nn.functional.conv2d(torch.from_numpy(x)[None, None],
                                             torch.from_numpy(w)[None, None], padding=k // 2)
            _close(orc.dwconv(x, w), ref[0, 0].numpy(), 1e-13, f"dwconv k={k} {H}x{W}")


# ------------------------------------------------------------------------------- layer pins

def check_zero_wavelet_scale(orc):
    """wavelet_scale = 0: y = s_b * (depthwise conv(x, base_w) + b), via torch conv2d."""
    rng = np.random.default_rng(4)
    B, C, H, W, L, k = 2, 3, 16, 8, 3, 5
    p = random_params(rng, C, L, k, zero_wavelet_scale=True)
    x = rng.standard_normal((B, C, H, W))
    conv = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(p["base_w"])[:, None],
                                      padding=k // 2, groups=C).numpy()
    ref = p["base_scale"][None, :, None, None] * (conv + p["base_bias"][None, :, None, None])
    _close(orc.forward(x, p), ref, 1e-13, "forward with zero wavelet scales")


def block_mean(x, j):
    """P_j: mean over aligned 2^j x 2^j blocks, broadcast back (P_0 = identity)."""
    if j == 0:
        return x.copy()
    B, C, H, W = x.shape
    n = 1 << j
    m = x.reshape(B, C, H // n, n, W // n, n).mean(axis=(3, 5), keepdims=True)
    return np.broadcast_to(m, (B, C, H // n, n, W // n, n)).reshape(B, C, H, W)


def check_identity_kernels(orc):
    """Delta kernels, one scale a_l per level: y = s_b (x + b) + sum_l a_l P_(l-1) x."""
    rng = np.random.default_rng(5)
    for (B, C, H, W, L, k) in ((1, 2, 16, 16, 3, 5), (2, 1, 8, 24, 2, 3), (1, 1, 32, 32, 4, 1)):
        p = random_params(rng, C, L, k)
        delta = np.zeros((k, k))
        delta[k // 2, k // 2] = 1.0
        p["base_w"][:] = delta
        p["wavelet_w"][:] = delta
        a = rng.uniform(0.1, 2.0, L)
        p["wavelet_scale"][:] = a[:, None]
        x = rng.standard_normal((B, C, H, W))
        ref = p["base_scale"][None, :, None, None] * (x + p["base_bias"][None, :, None, None])
        for lvl in range(1, L + 1):
            ref = ref + a[lvl - 1] * block_mean(x, lvl - 1)
        _close(orc.forward(x, p), ref, 1e-13, f"identity-kernel closed form L={L} k={k}")


# dense-matrix brute force ----------------------------------------------------------------

def _analysis_matrix(h, w):
    """Matrix of one Haar level on an h x w plane: rows (s, i, j), cols (row, col)."""
    scale, pats = load_haar_filters()
    names = ("LL", "LH", "HL", "HH")
    hh, ww = h // 2, w // 2
    A = np.zeros((4 * hh * ww, h * w))
    for s in range(4):
        for i in range(hh):
            for j in range(ww):
                for a in range(2):
                    for b in range(2):
                        A[(s * hh + i) * ww + j, (2 * i + a) * w + 2 * j + b] = scale * pats[names[s]][a, b]
    return A


def _conv_matrix(h, w, ker):
    k = ker.shape[0]
    p = k // 2
    K = np.zeros((h * w, h * w))
    for i in range(h):
        for j in range(w):
            for u in range(k):
                for v in range(k):
                    r, c = i + u - p, j + v - p
                    if 0 <= r < h and 0 <= c < w:
                        K[i * w + j, r * w + c] += ker[u, v]
    return K


def _pad_matrix(h, w):
    """h x w plane -> the same plane with one zero row / column appended to an odd side."""
    he, we = h + (h & 1), w + (w & 1)
    Pm = np.zeros((he * we, h * w))
    for i in range(h):
        for j in range(w):
            Pm[i * we + j, i * w + j] = 1.0
    return Pm


def layer_matrix(p, c, H, W, L):
    """Dense matrix M of one channel's layer (y = M x + s_b b), stage by stage.  A level whose
    input has an odd side zero-pads it at the end before the analysis; the synthesis is the
    transpose of that (the transposed Haar conv, then the crop back to the input size)."""
    n0 = H * W
    ll = np.eye(n0)                      # maps x -> LL_(l-1)
    Zs, As = [], []
    h, w = H, W                          # sides of LL_(l-1)
    for lvl in range(1, L + 1):
        he, we = h + (h & 1), w + (w & 1)
        A = _analysis_matrix(he, we) @ _pad_matrix(h, w)
        Y = A @ ll                       # maps x -> Y^(l)
        h, w = he // 2, we // 2
        m = h * w
        Z = np.zeros_like(Y)
        for s in range(4):
            K = _conv_matrix(h, w, p["wavelet_w"][lvl - 1, 4 * c + s])
            Z[s * m:(s + 1) * m] = p["wavelet_scale"][lvl - 1, 4 * c + s] * (K @ Y[s * m:(s + 1) * m])
        Zs.append(Z)
        As.append(A)
        ll = Y[:m]
    R = np.zeros((h * w, n0))
    for lvl in range(L, 0, -1):
        Z = Zs[lvl - 1].copy()
        m = R.shape[0]
        Z[:m] += R                        # reconstruction enters the LL subband
        R = As[lvl - 1].T @ Z             # transposed stride-2 conv with the same filters
    return p["base_scale"][c] * _conv_matrix(H, W, p["base_w"][c]) + R


def check_dense_matrix(orc):
    rng = np.random.default_rng(6)
    for (C, H, W, L, k) in ((2, 8, 8, 1, 3), (2, 8, 8, 2, 5), (1, 8, 8, 3, 3), (1, 16, 16, 3, 5),
                            (2, 7, 5, 2, 3), (1, 5, 9, 3, 3), (1, 3, 6, 2, 5), (1, 11, 1, 2, 3)):
        B = 2
        p = random_params(rng, C, L, k)
        x = rng.standard_normal((B, C, H, W))
        dy = rng.standard_normal((B, C, H, W))
        y = orc.forward(x, p)
        g = orc.backward(x, dy, p)
        for c in range(C):
            M = layer_matrix(p, c, H, W, L)
            for b in range(B):
                yref = M @ x[b, c].ravel() + p["base_scale"][c] * p["base_bias"][c]
                _close(y[b, c].ravel(), yref, 1e-12, f"dense forward C={C} L={L} k={k}")
                _close(g["dx"][b, c].ravel(), M.T @ dy[b, c].ravel(), 1e-12,
                       f"dense dx = M^T dy L={L} k={k}")


def check_finite_differences(orc):
    """Central differences of <dy, y(theta)>; exact up to rounding (affine in each scalar)."""
    rng = np.random.default_rng(7)
    B, C, H, W, L, k = 2, 2, 8, 8, 2, 3
    p = random_params(rng, C, L, k)
    x = rng.standard_normal((B, C, H, W))
    dy = rng.standard_normal((B, C, H, W))
    g = orc.backward(x, dy, p)
    h = 0.5

    def loss(xx, pp):
        return float(np.sum(dy * orc.forward(xx, pp, nthreads=1)))

    for name in ("base_w", "base_bias", "base_scale", "wavelet_w", "wavelet_scale"):
        fd = np.zeros_like(p[name])
        flat = p[name].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(x, p)
            flat[i] = old - h
            lm = loss(x, p)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * h)
        _close(g["d_" + name], fd, 1e-10, f"finite differences d_{name}")
    idx = rng.choice(x.size, 40, replace=False)
    xf = x.reshape(-1)
    for i in idx:
        old = xf[i]
        xf[i] = old + h
        lp = loss(x, p)
        xf[i] = old - h
        lm = loss(x, p)
        xf[i] = old
        want = (lp - lm) / (2 * h)
        got = g["dx"].reshape(-1)[i]
        assert abs(got - want) <= 1e-10 * max(1.0, abs(want)), f"finite differences dx[{i}]: {got} vs {want}"


def check_odd_sides_match_zero_padding(orc):
    """Per-level padding of odd sides and cropping of the reconstructions equals zero-padding x
    at its end to multiples of 2^L, running the layer there and cropping y (a padded row or
    column of a level is never an ancestor of a pixel inside the plane); dx and every parameter
    gradient likewise (dy padded with zeros)."""
    rng = np.random.default_rng(11)
    for (B, C, H, W, L, k) in ((2, 3, 7, 5, 2, 3), (1, 2, 5, 11, 3, 5), (2, 1, 9, 6, 1, 3), (1, 1, 3, 3, 2, 5),
                               (1, 2, 13, 4, 2, 7)):
        p = random_params(rng, C, L, k)
        x = rng.standard_normal((B, C, H, W))
        dy = rng.standard_normal((B, C, H, W))
        Hp, Wp = -(-H // 2 ** L) * 2 ** L, -(-W // 2 ** L) * 2 ** L
        xp = np.zeros((B, C, Hp, Wp))
        xp[:, :, :H, :W] = x
        dyp = np.zeros((B, C, Hp, Wp))
        dyp[:, :, :H, :W] = dy
        tag = f"{H}x{W} L={L} k={k}"
        _close(orc.forward(x, p), orc.forward(xp, p)[:, :, :H, :W], 1e-12, f"odd sides y {tag}")
        g, gp = orc.backward(x, dy, p), orc.backward(xp, dyp, p)
        _close(g["dx"], gp["dx"][:, :, :H, :W], 1e-12, f"odd sides dx {tag}")
        for n in g:
            if n != "dx":
                _close(g[n], gp[n], 1e-11, f"odd sides {n} {tag}")


def check_finite_differences_odd_sides(orc):
    """Central differences of <dy, y(theta)> on odd sides (every level pads)."""
    rng = np.random.default_rng(12)
    B, C, H, W, L, k = 1, 2, 7, 5, 2, 3
    p = random_params(rng, C, L, k)
    x = rng.standard_normal((B, C, H, W))
    dy = rng.standard_normal((B, C, H, W))
    g = orc.backward(x, dy, p)
    h = 0.5

    def loss(xx, pp):
        return float(np.sum(dy * orc.forward(xx, pp, nthreads=1)))

    for name in ("base_w", "base_bias", "base_scale", "wavelet_w", "wavelet_scale"):
        fd = np.zeros_like(p[name])
        flat = p[name].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(x, p)
            flat[i] = old - h
            lm = loss(x, p)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * h)
        _close(g["d_" + name], fd, 1e-10, f"finite differences (odd sides) d_{name}")
    xf = x.reshape(-1)
    for i in range(x.size):
        old = xf[i]
        xf[i] = old + h
        lp = loss(x, p)
        xf[i] = old - h
        lm = loss(x, p)
        xf[i] = old
        want = (lp - lm) / (2 * h)
        got = g["dx"].reshape(-1)[i]
        assert abs(got - want) <= 1e-10 * max(1.0, abs(want)), f"finite differences (odd) dx[{i}]: {got} vs {want}"


def check_euler_identities(orc):
    """Homogeneity: sum w*dw = s*ds per subband channel; base: sum w_b dw_b + b db = s_b ds_b;
    <dx, x> = <dy, y - s_b b>."""
    rng = np.random.default_rng(8)
    B, C, H, W, L, k = 2, 3, 16, 16, 3, 5
    p = random_params(rng, C, L, k)
    x = rng.standard_normal((B, C, H, W))
    dy = rng.standard_normal((B, C, H, W))
    y = orc.forward(x, p)
    g = orc.backward(x, dy, p)
    lhs = np.sum(p["wavelet_w"] * g["d_wavelet_w"], axis=(2, 3))
    _close(lhs, p["wavelet_scale"] * g["d_wavelet_scale"], 1e-11, "Euler identity, wavelet path")
    lhs = np.sum(p["base_w"] * g["d_base_w"], axis=(1, 2)) + p["base_bias"] * g["d_base_bias"]
    _close(lhs, p["base_scale"] * g["d_base_scale"], 1e-11, "Euler identity, base path")
    shift = (p["base_scale"] * p["base_bias"])[None, :, None, None]
    a, b = float(np.sum(g["dx"] * x)), float(np.sum(dy * (y - shift)))
    assert abs(a - b) <= 1e-11 * max(abs(a), abs(b)), f"<dx,x> {a} vs <dy,y-s_b b> {b}"


def check_thread_invariance(orc):
    rng = np.random.default_rng(9)
    B, C, H, W, L, k = 3, 5, 16, 16, 2, 5
    p = random_params(rng, C, L, k)
    x = rng.standard_normal((B, C, H, W))
    dy = rng.standard_normal((B, C, H, W))
    assert np.array_equal(orc.forward(x, p, nthreads=1), orc.forward(x, p, nthreads=3))
    g1, g3 = orc.backward(x, dy, p, nthreads=1), orc.backward(x, dy, p, nthreads=4)
    for n in g1:
        assert np.array_equal(g1[n], g3[n]), n


ALL_CHECKS = [
    check_odd_sides_match_zero_padding,
    check_finite_differences_odd_sides,
    check_haar_filters,
    check_perfect_reconstruction,
    check_parseval,
    check_dwconv_library,
    check_zero_wavelet_scale,
    check_identity_kernels,
    check_dense_matrix,
    check_finite_differences,
    check_euler_identities,
    check_thread_invariance,
]
