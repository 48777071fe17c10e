"""Pins that tie the CPU oracle to facts fixed outside it.

Each check raises AssertionError on failure.  ``run_all(lib)`` runs the whole
battery against one build of the oracle library, which lets
``test_oracle_mutations.py`` show that a planted mistake in the oracle fails at
least one pin.  Run as a script (``python tests/oracle_pins.py LIB.so``) it
exits 0 when every pin holds and 1 otherwise.

The pins (none re-types the oracle's formula):
* hand-worked fixtures in ``tests/golden/`` (the pages print no worked values);
* delta filters: identity and shifted identity, with zero fill at the border;
* a 1x1 convolution equals a plain matrix product, and a strided 1x1 equals
  subsampling followed by that product;
* brute force: explicit im2col (column matrix built by gathering windows) and a
  naive GEMM, on integer-valued inputs so that every sum is exact in fp64;
* invariants: linearity in the input, the bias shift, zero input gives the bias,
  output extents on edge cases, thread-count independence, the point-query
  entry agreeing with the full output, bf16 widening matching float64 input;
* grouped convolution: per group, the same brute force on the group's slice of
  input channels, filters and bias (channels split into consecutive groups),
  and a depthwise case (groups = C = K) written as its own loop.
Only numpy is used here, so the battery runs quickly in a subprocess.
"""
from __future__ import annotations

import os
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import oracle  # noqa: E402

GOLDEN = os.path.join(_HERE, "golden")


# ----------------------------------------------------------------------------
# helpers independent of the oracle
# ----------------------------------------------------------------------------
def bf16_bits_of_ints(a: np.ndarray) -> np.ndarray:
    """Integer-valued array (|v| <= 256) -> bf16 bit patterns (exact: fp32 top half)."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def extent(in_size, pad, dil, ker, stride):
    """Output extent by counting window positions one by one (no closed form)."""
    count = 0
    start = -pad
    while start + dil * (ker - 1) <= in_size - 1 + pad:
        count += 1
        start += stride
    return count


def im2col_gemm(x, w, bias, stride, pad, dil):
    """Brute force: materialise the column matrix, then a naive triple-loop GEMM.

    x [N,H,W,C], w [K,R,S,C] as float64.  The column matrix has one row per output
    pixel and one column per (r, s, c) filter tap; entries outside the padded image
    are zero.  Only used on tiny shapes.
    """
    n, h, wd, c = x.shape
    k, r, s, _ = w.shape
    sh, sw = stride
    ph, pw = pad
    dh, dw = dil
    p = extent(h, ph, dh, r, sh)
    q = extent(wd, pw, dw, s, sw)
    padded = np.zeros((n, h + 2 * ph, wd + 2 * pw, c))
    padded[:, ph:ph + h, pw:pw + wd, :] = x
    cols = np.zeros((n * p * q, r * s * c))
    row = 0
    for ni in range(n):
        for pi in range(p):
            for qi in range(q):
                taps = []
                for ri in range(r):
                    for si in range(s):
                        taps.append(padded[ni, pi * sh + ri * dh, qi * sw + si * dw, :])
                cols[row] = np.concatenate(taps)
                row += 1
    wmat = w.reshape(k, r * s * c)
    out = np.zeros((n * p * q, k))
    for i in range(n * p * q):
        for j in range(k):
            acc = 0.0
            for t in range(r * s * c):
                acc += cols[i, t] * wmat[j, t]
            out[i, j] = acc
    if bias is not None:
        out += np.asarray(bias, dtype=np.float64)[None, :]
    return out.reshape(n, p, q, k)


def read_fixture(path):
    d = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            d[key.strip()] = val.split()
    def ints(key):
        return tuple(int(v) for v in d[key])
    x = np.array([float(v) for v in d["x"]]).reshape(ints("shape_x"))
    w = np.array([float(v) for v in d["w"]]).reshape(ints("shape_w"))
    bias = None if d["bias"] == ["none"] else np.array([float(v) for v in d["bias"]], dtype=np.float32)
    y = np.array([float(v) for v in d["y"]]).reshape(ints("shape_y"))
    return dict(x=x, w=w, bias=bias, y=y, stride=ints("stride"), pad=ints("pad"), dil=ints("dil"))


def fixtures():
    return sorted(os.path.join(GOLDEN, f) for f in os.listdir(GOLDEN) if f.endswith(".txt"))


# ----------------------------------------------------------------------------
# the pins
# ----------------------------------------------------------------------------
def pin_golden(lib):
    paths = fixtures()
    assert len(paths) >= 3
    for path in paths:
        fx = read_fixture(path)
        y64 = oracle.conv2d_fwd_f64(fx["x"], fx["w"], fx["bias"], fx["stride"], fx["pad"], fx["dil"], lib=lib)
        assert y64.shape == fx["y"].shape, (path, y64.shape)
        assert np.array_equal(y64, fx["y"]), (path, y64.ravel(), fx["y"].ravel())
        yb = oracle.conv2d_fwd(bf16_bits_of_ints(fx["x"]), bf16_bits_of_ints(fx["w"]), fx["bias"],
                               fx["stride"], fx["pad"], fx["dil"], lib=lib)
        assert np.array_equal(yb, fx["y"]), path


def pin_delta_identity(lib):
    rng = np.random.default_rng(1)
    x = rng.integers(-4, 5, size=(2, 5, 7, 6)).astype(np.float64)
    # 1x1 identity
    w = np.zeros((6, 1, 1, 6))
    for c in range(6):
        w[c, 0, 0, c] = 1.0
    assert np.array_equal(oracle.conv2d_fwd_f64(x, w, lib=lib), x)
    # centred 3x3 delta with padding 1 (and a 5x5 with padding 2)
    for ker, pad in ((3, 1), (5, 2)):
        w = np.zeros((6, ker, ker, 6))
        for c in range(6):
            w[c, ker // 2, ker // 2, c] = 1.0
        y = oracle.conv2d_fwd_f64(x, w, padding=pad, lib=lib)
        assert np.array_equal(y, x), (ker, pad)


def pin_shifted_delta(lib):
    rng = np.random.default_rng(2)
    x = rng.integers(-4, 5, size=(1, 6, 5, 3)).astype(np.float64)
    n, h, wd, c = x.shape
    for r0 in range(3):
        for s0 in range(3):
            w = np.zeros((c, 3, 3, c))
            for ch in range(c):
                w[ch, r0, s0, ch] = 1.0
            y = oracle.conv2d_fwd_f64(x, w, padding=1, lib=lib)
            expect = np.zeros_like(x)
            dr, ds = r0 - 1, s0 - 1
            for p in range(h):
                for q in range(wd):
                    ih, iw = p + dr, q + ds
                    if 0 <= ih < h and 0 <= iw < wd:
                        expect[:, p, q, :] = x[:, ih, iw, :]
            assert np.array_equal(y, expect), (r0, s0)


def pin_1x1_matmul(lib):
    rng = np.random.default_rng(3)
    x = rng.integers(-5, 6, size=(3, 4, 6, 7)).astype(np.float64)
    w = rng.integers(-5, 6, size=(9, 1, 1, 7)).astype(np.float64)
    y = oracle.conv2d_fwd_f64(x, w, lib=lib)
    expect = (x.reshape(-1, 7) @ w.reshape(9, 7).T).reshape(3, 4, 6, 9)
    assert np.array_equal(y, expect)
    # stride 2: subsample rows/cols 0, 2, 4, ... then the same product
    y2 = oracle.conv2d_fwd_f64(x, w, stride=2, lib=lib)
    xs = x[:, ::2, ::2, :]
    expect2 = (xs.reshape(-1, 7) @ w.reshape(9, 7).T).reshape(xs.shape[:3] + (9,))
    assert y2.shape == expect2.shape, (y2.shape, expect2.shape)
    assert np.array_equal(y2, expect2)
    # stride 3 along H only, stride 2 along W
    y3 = oracle.conv2d_fwd_f64(x, w, stride=(3, 2), lib=lib)
    xs3 = x[:, ::3, ::2, :]
    expect3 = (xs3.reshape(-1, 7) @ w.reshape(9, 7).T).reshape(xs3.shape[:3] + (9,))
    assert np.array_equal(y3, expect3)


BRUTE_CASES = [
    # (n, h, w, c, k, r, s, stride, pad, dil)
    (1, 5, 5, 1, 1, 3, 3, (1, 1), (0, 0), (1, 1)),
    (1, 6, 7, 3, 2, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 7, 6, 3, 4, 3, 2, (2, 1), (1, 0), (1, 1)),
    (1, 9, 8, 2, 3, 3, 3, (1, 2), (2, 3), (2, 1)),
    (1, 8, 9, 16, 2, 2, 3, (3, 1), (0, 2), (1, 3)),
    (1, 11, 10, 1, 2, 5, 5, (2, 2), (3, 1), (1, 2)),
    (2, 9, 9, 3, 2, 7, 7, (2, 2), (3, 3), (1, 1)),
    (1, 10, 12, 2, 3, 1, 5, (1, 3), (0, 2), (3, 2)),
    (1, 4, 4, 3, 5, 2, 2, (3, 3), (3, 3), (3, 3)),
    (1, 3, 13, 1, 1, 3, 7, (1, 1), (1, 3), (1, 2)),
]


def pin_bruteforce_im2col(lib):
    rng = np.random.default_rng(4)
    for case in BRUTE_CASES:
        n, h, wd, c, k, r, s, st, pd, dl = case
        x = rng.integers(-3, 4, size=(n, h, wd, c)).astype(np.float64)
        w = rng.integers(-3, 4, size=(k, r, s, c)).astype(np.float64)
        b = rng.integers(-8, 9, size=(k,)).astype(np.float32)
        expect = im2col_gemm(x, w, b, st, pd, dl)
        y = oracle.conv2d_fwd_f64(x, w, b, st, pd, dl, lib=lib)
        assert y.shape == expect.shape, (case, y.shape, expect.shape)
        assert np.array_equal(y, expect), case
        yb = oracle.conv2d_fwd(bf16_bits_of_ints(x), bf16_bits_of_ints(w), b, st, pd, dl, lib=lib)
        assert np.array_equal(yb, expect), case


def pin_invariants(lib):
    rng = np.random.default_rng(5)
    shape_x, shape_w = (2, 6, 5, 4), (3, 3, 2, 4)
    st, pd, dl = (2, 1), (1, 2), (1, 2)
    x1 = rng.integers(-4, 5, size=shape_x).astype(np.float64)
    x2 = rng.integers(-4, 5, size=shape_x).astype(np.float64)
    w = rng.integers(-4, 5, size=shape_w).astype(np.float64)
    y1 = oracle.conv2d_fwd_f64(x1, w, None, st, pd, dl, lib=lib)
    y2 = oracle.conv2d_fwd_f64(x2, w, None, st, pd, dl, lib=lib)
    y12 = oracle.conv2d_fwd_f64(3 * x1 - 2 * x2, w, None, st, pd, dl, lib=lib)
    assert np.array_equal(y12, 3 * y1 - 2 * y2)
    # linearity in the weight
    w2 = rng.integers(-4, 5, size=shape_w).astype(np.float64)
    yw = oracle.conv2d_fwd_f64(x1, w + w2, None, st, pd, dl, lib=lib)
    assert np.array_equal(yw, y1 + oracle.conv2d_fwd_f64(x1, w2, None, st, pd, dl, lib=lib))
    # bias shift and zero input
    b = np.array([0.5, -2.0, 7.25], dtype=np.float32)
    yb = oracle.conv2d_fwd_f64(x1, w, b, st, pd, dl, lib=lib)
    assert np.array_equal(yb - y1, np.broadcast_to(b.astype(np.float64), y1.shape))
    y0 = oracle.conv2d_fwd_f64(np.zeros(shape_x), w, b, st, pd, dl, lib=lib)
    assert np.array_equal(y0, np.broadcast_to(b.astype(np.float64), y0.shape))
    # thread count does not change a single bit (random non-integer data)
    xr = rng.standard_normal(shape_x)
    wr = rng.standard_normal(shape_w)
    ya = oracle.conv2d_fwd_f64(xr, wr, b, st, pd, dl, threads=1, lib=lib)
    yc = oracle.conv2d_fwd_f64(xr, wr, b, st, pd, dl, threads=5, lib=lib)
    assert np.array_equal(ya, yc)


def pin_extents(lib):
    # (in, pad, dil, ker, stride): compared with counting window positions.
    cases = [(8, 1, 1, 3, 1), (224, 3, 1, 7, 2), (56, 0, 1, 1, 2), (64, 2, 2, 3, 1), (7, 1, 1, 3, 1),
             (5, 0, 1, 5, 1), (4, 0, 1, 5, 1), (4, 0, 2, 3, 1), (5, 0, 2, 3, 1), (10, 0, 1, 3, 3),
             (11, 0, 1, 3, 3), (1, 0, 1, 1, 1), (3, 2, 3, 3, 2), (9, 1, 1, 2, 4), (0, 1, 1, 3, 1)]
    for c in cases:
        got = oracle.out_extent(*c, lib=lib)
        assert got == extent(*c), (c, got, extent(*c))
    # a window that does not fit gives an empty output, not an error
    x = np.ones((1, 2, 2, 1))
    w = np.ones((1, 3, 3, 1))
    assert oracle.conv2d_fwd_f64(x, w, lib=lib).shape == (1, 0, 0, 1)


def pin_points_and_bf16(lib):
    rng = np.random.default_rng(6)
    x = rng.integers(-3, 4, size=(2, 7, 9, 5)).astype(np.float64)
    w = rng.integers(-3, 4, size=(6, 3, 2, 5)).astype(np.float64)
    b = rng.integers(-3, 4, size=(6,)).astype(np.float32)
    st, pd, dl = (1, 2), (1, 0), (2, 1)
    xb, wb = bf16_bits_of_ints(x), bf16_bits_of_ints(w)
    full = oracle.conv2d_fwd(xb, wb, b, st, pd, dl, lib=lib)
    assert np.array_equal(full, oracle.conv2d_fwd_f64(x, w, b, st, pd, dl, lib=lib))
    flat = full.reshape(-1, full.shape[-1])
    mi = rng.integers(0, flat.shape[0], size=64)
    ki = rng.integers(0, flat.shape[1], size=64)
    pts = oracle.conv2d_fwd_points(xb, wb, b, st, pd, dl, mi, ki, lib=lib)
    assert np.array_equal(pts, flat[mi, ki])
    pts64 = oracle.conv2d_fwd_points_f64(x, w, b, st, pd, dl, mi, ki, lib=lib)
    assert np.array_equal(pts64, flat[mi, ki])
    # bf16 widening of non-integer patterns: 1.5, -0.375, 2^-10, 3.0e38-ish
    vals = np.array([1.5, -0.375, 2.0 ** -10, 1.0e30], dtype=np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    xv = bits.reshape(1, 1, 1, 4)
    wv = np.array([0x3F80] * 4, dtype=np.uint16).reshape(1, 1, 1, 4)  # four ones
    got = oracle.conv2d_fwd(xv, wv, lib=lib)
    widened = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert got.item() == ((widened[0] + widened[1]) + widened[2]) + widened[3]


GROUP_CASES = [
    # (n, h, w, c, k, r, s, groups, stride, pad, dil)
    (2, 5, 6, 4, 6, 3, 3, 2, (1, 1), (1, 1), (1, 1)),
    (1, 7, 5, 6, 9, 3, 2, 3, (2, 1), (1, 0), (1, 2)),
    (2, 6, 6, 8, 4, 1, 1, 4, (1, 1), (0, 0), (1, 1)),
    (1, 6, 7, 6, 12, 2, 3, 6, (1, 2), (1, 1), (2, 1)),
]


def pin_groups(lib):
    rng = np.random.default_rng(7)
    for case in GROUP_CASES:
        n, h, wd, c, k, r, s, g, st, pd, dl = case
        cg, kg = c // g, k // g
        x = rng.integers(-3, 4, size=(n, h, wd, c)).astype(np.float64)
        w = rng.integers(-3, 4, size=(k, r, s, cg)).astype(np.float64)
        b = rng.integers(-8, 9, size=(k,)).astype(np.float32)
        # consecutive groups: group i takes input channels i*cg.. and filters i*kg..
        expect = np.concatenate(
            [im2col_gemm(x[..., i * cg:(i + 1) * cg], w[i * kg:(i + 1) * kg], b[i * kg:(i + 1) * kg], st, pd, dl)
             for i in range(g)], axis=-1)
        y = oracle.conv2d_fwd_f64(x, w, b, st, pd, dl, lib=lib, groups=g)
        assert y.shape == expect.shape, (case, y.shape, expect.shape)
        assert np.array_equal(y, expect), case
        xb, wb = bf16_bits_of_ints(x), bf16_bits_of_ints(w)
        assert np.array_equal(oracle.conv2d_fwd(xb, wb, b, st, pd, dl, lib=lib, groups=g), expect), case
        flat = expect.reshape(-1, k)
        mi = rng.integers(0, flat.shape[0], size=32)
        ki = rng.integers(0, k, size=32)
        pts = oracle.conv2d_fwd_points(xb, wb, b, st, pd, dl, mi, ki, lib=lib, groups=g)
        assert np.array_equal(pts, flat[mi, ki]), case
    # depthwise: every channel filtered by its own R x S kernel, written as its own loop
    x = rng.integers(-3, 4, size=(1, 5, 4, 3)).astype(np.float64)
    w = rng.integers(-3, 4, size=(3, 3, 3, 1)).astype(np.float64)
    expect = np.zeros((1, 5, 4, 3))
    for ch in range(3):
        for pi in range(5):
            for qi in range(4):
                acc = 0.0
                for ri in range(3):
                    for si in range(3):
                        ih, iw = pi - 1 + ri, qi - 1 + si
                        if 0 <= ih < 5 and 0 <= iw < 4:
                            acc += x[0, ih, iw, ch] * w[ch, ri, si, 0]
                expect[0, pi, qi, ch] = acc
    assert np.array_equal(oracle.conv2d_fwd_f64(x, w, None, 1, 1, 1, lib=lib, groups=3), expect)


ALL_PINS = [pin_golden, pin_delta_identity, pin_shifted_delta, pin_1x1_matmul, pin_bruteforce_im2col,
            pin_invariants, pin_extents, pin_points_and_bf16, pin_groups]


def run_all(lib):
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:  # noqa: PERF203
            failed.append((pin.__name__, repr(e)[:200]))
    return failed


if __name__ == "__main__":
    path = sys.argv[1]
    failures = run_all(oracle.load(path))
    for name, why in failures:
        print(f"FAILED {name}: {why}")
    sys.exit(1 if failures else 0)
