"""Pin battery for the weight-gradient oracle (``oracle/conv2d_wgrad.c``).

Usable two ways: imported by the tests (``run_all(lib)``), or run as a script on
a library path (``python tests/oracle_wgrad_pins.py path/to/lib.so``; exit status
0 when every pin holds), which is how the mutation tests judge planted mistakes.

What pins it:

* hand-worked fixtures (tests/golden/backward/, each with its derivation), one
  with stride 2 and padding;
* adjoint identity: the weight gradient is the adjoint of the forward
  convolution in the weight, so for every weight-shaped V,
  sum(dw * V) == sum(dy * conv(x, V)); the forward convolution is the separately
  pinned forward oracle (its own library and pins);
* brute force: with integer inputs, dw == dy^T @ cols(x) exactly, the column
  matrix gathered window by window here, and with groups one such product per
  group;
* 1x1 convolutions: dy^T @ x, and with stride 2 the subsampled x;
* a library gradient: torch.nn.grad.conv2d_weight in float64;
* point queries against the full gradient, their |term| sums against the brute
  force, the bf16 entry against widened values, and a zero gradient for dy = 0.
"""
from __future__ import annotations

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import wgrad as ow  # noqa: E402

GOLDEN_BACKWARD = os.path.join(HERE, "golden", "backward")


def read_backward_fixtures(op):
    """The hand-worked fixtures of tests/golden/backward for `op` ("wgrad" or "dgrad")."""
    out = []
    for name in sorted(os.listdir(GOLDEN_BACKWARD)):
        if not name.endswith(".txt"):
            continue
        d = {}
        for line in open(os.path.join(GOLDEN_BACKWARD, name)):
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split(":", 1)
                d[key.strip()] = val.split()
        if d["op"] != [op]:
            continue
        shape = lambda k: tuple(int(v) for v in d[k])  # noqa: E731
        arr = lambda k, s: np.array([float(v) for v in d[k]]).reshape(shape(s))  # noqa: E731
        f = dict(name=name, shape_x=shape("shape_x"), shape_w=shape("shape_w"), stride=shape("stride"),
                 pad=shape("pad"), dil=shape("dil"), dy=arr("dy", "shape_dy"))
        for key, s in (("x", "shape_x"), ("w", "shape_w"), ("dw", "shape_w"), ("dx", "shape_x")):
            if key in d:
                f[key] = arr(key, s)
        out.append(f)
    assert out, f"no {op} fixtures"
    return out


GEOMS = [  # (N, H, W, C, K, R, S, stride, pad, dil, groups)
    (2, 5, 6, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1), 1),
    (1, 7, 5, 2, 3, 3, 2, (2, 1), (1, 0), (1, 2), 1),
    (2, 6, 6, 4, 2, 2, 3, (1, 2), (0, 2), (2, 1), 1),
    (1, 8, 7, 4, 6, 3, 3, (2, 2), (2, 1), (1, 1), 2),
    (1, 5, 5, 6, 6, 1, 2, (1, 3), (0, 1), (1, 1), 3),
]


def extent(in_size, pad, dil, ker, stride):
    count, start = 0, -pad
    while start + dil * (ker - 1) <= in_size - 1 + pad:
        count += 1
        start += stride
    return count


def columns(x, r, s, stride, pad, dil):
    """Column matrix [N*P*Q, R*S*C]: each output pixel's window, tap by tap (zero outside)."""
    n, h, w, c = x.shape
    (sh, sw), (ph, pw), (dh, dw) = stride, pad, dil
    p, q = extent(h, ph, dh, r, sh), extent(w, pw, dw, s, sw)
    cols = np.zeros((n * p * q, r * s * c))
    row = 0
    for ni in range(n):
        for pi in range(p):
            for qi in range(q):
                for ri in range(r):
                    for si in range(s):
                        ih, iw = pi * sh - ph + ri * dh, qi * sw - pw + si * dw
                        if 0 <= ih < h and 0 <= iw < w:
                            t = ri * s + si
                            cols[row, t * c:(t + 1) * c] = x[ni, ih, iw, :]
                row += 1
    return cols, p, q


def brute_force(x, dy, k, r, s, stride, pad, dil, groups):
    """dw [K,R,S,C/G] = per group: dy_g^T @ cols(x_g), by explicit loops over the products."""
    n, h, w, c = x.shape
    cg, kg = c // groups, k // groups
    out = np.zeros((k, r, s, cg))
    mass = np.zeros((k, r, s, cg))
    for g in range(groups):
        cols, p, q = columns(x[..., g * cg:(g + 1) * cg], r, s, stride, pad, dil)
        d = dy.reshape(-1, k)[:, g * kg:(g + 1) * kg]
        for kk in range(kg):
            for j in range(r * s * cg):
                terms = d[:, kk] * cols[:, j]
                out[g * kg + kk].reshape(-1)[j] = terms.sum()
                mass[g * kg + kk].reshape(-1)[j] = np.abs(terms).sum()
    return out, mass


def _rand(rng, shape, ints):
    return rng.integers(-3, 4, shape).astype(np.float64) if ints else rng.standard_normal(shape)


def _dy_shape(g):
    n, h, w, c, k, r, s, st, pd, dl, gr = g
    return (n, extent(h, pd[0], dl[0], r, st[0]), extent(w, pd[1], dl[1], s, st[1]), k)


def pin_adjoint(lib):
    rng = np.random.default_rng(11)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        x = _rand(rng, (n, h, w, c), False)
        dy = _rand(rng, _dy_shape(g), False)
        v = _rand(rng, (k, r, s, c // gr), False)
        dw = ow.conv2d_wgrad_f64(x, dy, (k, r, s, c // gr), st, pd, dl, gr, threads=2, lib=lib)
        y = oracle.conv2d_fwd_f64(x, v, None, st, pd, dl, threads=2, groups=gr)
        lhs, rhs = float(np.sum(dw * v)), float(np.sum(dy * y))
        assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), f"adjoint identity fails for {g}: {lhs} vs {rhs}"


def pin_bruteforce_ints(lib):
    rng = np.random.default_rng(12)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        x = _rand(rng, (n, h, w, c), True)
        dy = _rand(rng, _dy_shape(g), True)
        dw = ow.conv2d_wgrad_f64(x, dy, (k, r, s, c // gr), st, pd, dl, gr, threads=3, lib=lib)
        want, _ = brute_force(x, dy, k, r, s, st, pd, dl, gr)
        assert np.array_equal(dw, want), f"brute force differs for {g}"


def pin_1x1_matmul(lib):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, 5, 6, 7))
    dy = rng.standard_normal((2, 5, 6, 4))
    dw = ow.conv2d_wgrad_f64(x, dy, (4, 1, 1, 7), 1, 0, 1, lib=lib)
    assert np.allclose(dw.reshape(4, 7), dy.reshape(-1, 4).T @ x.reshape(-1, 7), rtol=1e-12, atol=1e-12)
    dy2 = rng.standard_normal((2, 3, 3, 4))
    dw2 = ow.conv2d_wgrad_f64(x, dy2, (4, 1, 1, 7), 2, 0, 1, lib=lib)
    sub = x[:, ::2, ::2, :].reshape(-1, 7)
    assert np.allclose(dw2.reshape(4, 7), dy2.reshape(-1, 4).T @ sub, rtol=1e-12, atol=1e-12)


def pin_library_gradient(lib):
    import torch
    rng = np.random.default_rng(14)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        x = rng.standard_normal((n, h, w, c))
        dy = rng.standard_normal(_dy_shape(g))
        dw = ow.conv2d_wgrad_f64(x, dy, (k, r, s, c // gr), st, pd, dl, gr, lib=lib)
        ref = torch.nn.grad.conv2d_weight(torch.from_numpy(x).permute(0, 3, 1, 2), (k, c // gr, r, s),
                                          torch.from_numpy(dy).permute(0, 3, 1, 2), stride=st, padding=pd,
                                          dilation=dl, groups=gr).permute(0, 2, 3, 1).numpy()
        assert np.allclose(dw, ref, rtol=1e-10, atol=1e-10), f"library gradient differs for {g}"


def pin_points_mass_bf16(lib):
    import torch
    rng = np.random.default_rng(15)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        cg = c // gr
        xi = _rand(rng, (n, h, w, c), True)
        dyi = _rand(rng, _dy_shape(g), True)
        full = ow.conv2d_wgrad_f64(xi, dyi, (k, r, s, cg), st, pd, dl, gr, lib=lib)
        want, want_mass = brute_force(xi, dyi, k, r, s, st, pd, dl, gr)
        kk = np.repeat(np.arange(k), r * s * cg)
        jj = np.tile(np.arange(r * s * cg), k)
        pts, mass = ow.conv2d_wgrad_points_f64(xi, dyi, (k, r, s, cg), st, pd, dl, kk, jj, gr, lib=lib)
        assert np.array_equal(pts, full.reshape(-1)), f"points differ from the full gradient for {g}"
        assert np.array_equal(mass, want_mass.reshape(-1)), f"|term| sums differ for {g}"
        xb = torch.from_numpy(xi).to(torch.bfloat16)
        dyb = torch.from_numpy(dyi).to(torch.bfloat16)
        got, got_mass = ow.conv2d_wgrad(xb, dyb, (k, r, s, cg), st, pd, dl, gr, threads=2, with_mass=True, lib=lib)
        assert np.array_equal(got, want) and np.array_equal(got_mass, want_mass), f"bf16 entry differs for {g}"


def pin_zero_cases(lib):
    rng = np.random.default_rng(16)
    x = rng.standard_normal((2, 4, 4, 3))
    dw = ow.conv2d_wgrad_f64(x, np.zeros((2, 4, 4, 5)), (5, 3, 3, 3), 1, 1, 1, lib=lib)
    assert np.array_equal(dw, np.zeros_like(dw))
    dw0 = ow.conv2d_wgrad_f64(np.zeros((0, 4, 4, 3)), np.zeros((0, 4, 4, 5)), (5, 3, 3, 3), 1, 1, 1, lib=lib)
    assert dw0.shape == (5, 3, 3, 3) and np.array_equal(dw0, np.zeros_like(dw0))


def pin_golden(lib):
    for f in read_backward_fixtures("wgrad"):
        got = ow.conv2d_wgrad_f64(f["x"], f["dy"], f["shape_w"], f["stride"], f["pad"], f["dil"], lib=lib)
        assert np.array_equal(got, f["dw"]), f"{f['name']}: {got.reshape(-1)} vs {f['dw'].reshape(-1)}"


ALL_PINS = [pin_golden, pin_adjoint, pin_bruteforce_ints, pin_1x1_matmul, pin_library_gradient, pin_points_mass_bf16,
            pin_zero_cases]


def run_all(lib):
    for pin in ALL_PINS:
        pin(lib)


if __name__ == "__main__":
    lib = ow.load(sys.argv[1]) if len(sys.argv) > 1 else ow.load()
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            failed.append(f"{pin.__name__}: {e}")
    for f in failed:
        print("FAIL", f)
    sys.exit(1 if failed else 0)
