"""Pin battery for the data-gradient oracle (``oracle/conv2d_dgrad.c``).

Imported by the tests (``run_all(lib)``) or run as a script on a library path
(exit status 0 when every pin holds), which is how the mutation tests judge
planted mistakes.

What pins it:

* hand-worked fixtures (tests/golden/backward/, each with its derivation), one
  with stride 2 and padding;
* adjoint identity: the data gradient is the adjoint of the forward
  convolution in the input, so for every input-shaped U,
  sum(dx * U) == sum(dy * conv(U, w)); the forward convolution is the
  separately pinned forward oracle;
* brute force: with integer inputs, dx == col2im(dy @ w_matrix) exactly, the
  columns scattered back window by window here (one product per group);
* 1x1 stride 1: dx = dy @ w;
* a library gradient: torch.nn.grad.conv2d_input in float64;
* point queries and |term| sums against the brute force, the bf16 entry, and
  zero gradients for dy = 0 and an empty batch.
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
from oracle import dgrad as od  # noqa: E402

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
    (1, 9, 8, 3, 5, 3, 3, (3, 2), (1, 1), (1, 1), 1),
]


def extent(in_size, pad, dil, ker, stride):
    count, start = 0, -pad
    while start + dil * (ker - 1) <= in_size - 1 + pad:
        count += 1
        start += stride
    return count


def col2im_bruteforce(dy, w, x_shape, stride, pad, dil, groups):
    """dx by scattering each output pixel's column (dy row times the weight matrix) back
    into the window it was read from, with |term| sums; loops over every product."""
    n, h, wd, c = x_shape
    k, r, s, cg = w.shape
    kg = k // groups
    (sh, sw), (ph, pw), (dh, dw) = stride, pad, dil
    p, q = dy.shape[1], dy.shape[2]
    out = np.zeros((n, h, wd, c))
    mass = np.zeros((n, h, wd, c))
    for ni in range(n):
        for pi in range(p):
            for qi in range(q):
                for ri in range(r):
                    for si in range(s):
                        ih, iw = pi * sh - ph + ri * dh, qi * sw - pw + si * dw
                        if not (0 <= ih < h and 0 <= iw < wd):
                            continue
                        for g in range(groups):
                            for cc in range(cg):
                                terms = dy[ni, pi, qi, g * kg:(g + 1) * kg] * w[g * kg:(g + 1) * kg, ri, si, cc]
                                out[ni, ih, iw, g * cg + cc] += terms.sum()
                                mass[ni, ih, iw, g * cg + cc] += np.abs(terms).sum()
    return out, mass


def _rand(rng, shape, ints):
    return rng.integers(-3, 4, shape).astype(np.float64) if ints else rng.standard_normal(shape)


def _dy_shape(g):
    n, h, w, c, k, r, s, st, pd, dl, gr = g
    return (n, extent(h, pd[0], dl[0], r, st[0]), extent(w, pd[1], dl[1], s, st[1]), k)


def pin_adjoint(lib):
    rng = np.random.default_rng(21)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        wt = _rand(rng, (k, r, s, c // gr), False)
        dy = _rand(rng, _dy_shape(g), False)
        u = _rand(rng, (n, h, w, c), False)
        dx = od.conv2d_dgrad_f64(dy, wt, (n, h, w, c), st, pd, dl, gr, threads=2, lib=lib)
        y = oracle.conv2d_fwd_f64(u, wt, None, st, pd, dl, threads=2, groups=gr)
        lhs, rhs = float(np.sum(dx * u)), float(np.sum(dy * y))
        assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), f"adjoint identity fails for {g}: {lhs} vs {rhs}"


def pin_bruteforce_ints(lib):
    rng = np.random.default_rng(22)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        wt = _rand(rng, (k, r, s, c // gr), True)
        dy = _rand(rng, _dy_shape(g), True)
        dx = od.conv2d_dgrad_f64(dy, wt, (n, h, w, c), st, pd, dl, gr, threads=3, lib=lib)
        want, _ = col2im_bruteforce(dy, wt, (n, h, w, c), st, pd, dl, gr)
        assert np.array_equal(dx, want), f"col2im brute force differs for {g}"


def pin_1x1_matmul(lib):
    rng = np.random.default_rng(23)
    dy = rng.standard_normal((2, 5, 6, 4))
    wt = rng.standard_normal((4, 1, 1, 7))
    dx = od.conv2d_dgrad_f64(dy, wt, (2, 5, 6, 7), 1, 0, 1, lib=lib)
    assert np.allclose(dx.reshape(-1, 7), dy.reshape(-1, 4) @ wt.reshape(4, 7), rtol=1e-12, atol=1e-12)


def pin_library_gradient(lib):
    import torch
    rng = np.random.default_rng(24)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        wt = rng.standard_normal((k, r, s, c // gr))
        dy = rng.standard_normal(_dy_shape(g))
        dx = od.conv2d_dgrad_f64(dy, wt, (n, h, w, c), st, pd, dl, gr, lib=lib)
        ref = torch.nn.grad.conv2d_input((n, c, h, w), torch.from_numpy(wt).permute(0, 3, 1, 2),
                                         torch.from_numpy(dy).permute(0, 3, 1, 2), stride=st, padding=pd,
                                         dilation=dl, groups=gr).permute(0, 2, 3, 1).numpy()
        assert np.allclose(dx, ref, rtol=1e-10, atol=1e-10), f"library gradient differs for {g}"


def pin_points_mass_bf16(lib):
    import torch
    rng = np.random.default_rng(25)
    for g in GEOMS:
        n, h, w, c, k, r, s, st, pd, dl, gr = g
        wt = _rand(rng, (k, r, s, c // gr), True)
        dy = _rand(rng, _dy_shape(g), True)
        full = od.conv2d_dgrad_f64(dy, wt, (n, h, w, c), st, pd, dl, gr, lib=lib)
        want, want_mass = col2im_bruteforce(dy, wt, (n, h, w, c), st, pd, dl, gr)
        mi = np.repeat(np.arange(n * h * w), c)
        ci = np.tile(np.arange(c), n * h * w)
        pts, mass = od.conv2d_dgrad_points_f64(dy, wt, (n, h, w, c), st, pd, dl, mi, ci, gr, lib=lib)
        assert np.array_equal(pts, full.reshape(-1)), f"points differ from the full gradient for {g}"
        assert np.array_equal(mass, want_mass.reshape(-1)), f"|term| sums differ for {g}"
        got, got_mass = od.conv2d_dgrad(torch.from_numpy(dy).to(torch.bfloat16), torch.from_numpy(wt).to(torch.bfloat16),
                                        (n, h, w, c), st, pd, dl, gr, threads=2, with_mass=True, lib=lib)
        assert np.array_equal(got, want) and np.array_equal(got_mass, want_mass), f"bf16 entry differs for {g}"


def pin_zero_cases(lib):
    rng = np.random.default_rng(26)
    wt = rng.standard_normal((5, 3, 3, 3))
    dx = od.conv2d_dgrad_f64(np.zeros((2, 4, 4, 5)), wt, (2, 4, 4, 3), 1, 1, 1, lib=lib)
    assert np.array_equal(dx, np.zeros_like(dx))
    dx0 = od.conv2d_dgrad_f64(np.zeros((0, 4, 4, 5)), wt, (0, 4, 4, 3), 1, 1, 1, lib=lib)
    assert dx0.shape == (0, 4, 4, 3)


def pin_golden(lib):
    for f in read_backward_fixtures("dgrad"):
        got = od.conv2d_dgrad_f64(f["dy"], f["w"], f["shape_x"], f["stride"], f["pad"], f["dil"], lib=lib)
        assert np.array_equal(got, f["dx"]), f"{f['name']}: {got.reshape(-1)} vs {f['dx'].reshape(-1)}"


ALL_PINS = [pin_golden, pin_adjoint, pin_bruteforce_ints, pin_1x1_matmul, pin_library_gradient, pin_points_mass_bf16,
            pin_zero_cases]


def run_all(lib):
    for pin in ALL_PINS:
        pin(lib)


if __name__ == "__main__":
    lib = od.load(sys.argv[1]) if len(sys.argv) > 1 else od.load()
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            failed.append(f"{pin.__name__}: {e}")
    for f in failed:
        print("FAIL", f)
    sys.exit(1 if failed else 0)
