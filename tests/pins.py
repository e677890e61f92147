"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics,
checked with code that shares nothing with oracle.c.

Each ``pin_*`` takes an oracle backend (the ctypes library, possibly a mutated
build) and raises AssertionError when the backend disagrees with the fact.
tests/test_oracle_pins.py runs them against the real oracle;
tests/test_oracle_mutations.py runs them against deliberately broken copies of
oracle.c and requires every copy to fail at least one of them.

Sources (page titles of the three Kimi-K2.6 traces):
  * l2_p50 -- fused ConvTranspose3d(k3,s2,p1) -> x0.5 -> AvgPool3d(2) -> +bias -> x1.0
  * l1_p46 -- AvgPool3d(k3, s2, p1), count_include_pad
  * l1_p74 -- ConvTranspose1d(K5, s1, p0, d3)
"""
from __future__ import annotations

import itertools
import os
import re

import numpy as np

import oracle as ora

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- fixtures
def load_worked_examples():
    """Parse golden/convt1d_worked_examples.txt -> list of (params, terms)."""
    out = []
    cur = None
    with open(os.path.join(GOLDEN, "convt1d_worked_examples.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("example"):
                kv = dict(t.split("=") for t in line.split()[2:])
                cur = ({k: int(v) for k, v in kv.items()}, [])
                out.append(cur)
                continue
            lhs, rhs = (t.strip() for t in line.split("="))
            o = int(lhs[1:])
            terms = set()
            if rhs != "0":
                for term in rhs.split("+"):
                    m = re.fullmatch(r"w(\d+)\*x(\d+)", term.strip())
                    assert m, term
                    terms.add((int(m.group(1)), int(m.group(2))))
            assert o == len(cur[1])
            cur[1].append(terms)
    return out


def load_taps():
    rows = []
    with open(os.path.join(GOLDEN, "ct3d_k3s2p1_pool2_taps.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                v = [int(t) for t in line.split()]
                rows.append((tuple(v[0:3]), tuple(v[3:6]), v[6]))
    return rows


def load_sizes():
    rows = []
    with open(os.path.join(GOLDEN, "output_sizes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            toks = line.split()
            op, L = toks[0], int(toks[1])
            params = {}
            i = 2
            while "=" in toks[i]:
                k, v = toks[i].split("=")
                params[k] = int(v)
                i += 1
            rows.append((op, L, params, int(toks[i])))
    return rows


# ------------------------------------------------- independent brute force
def forward_conv_matrix(cin, cout, L_in, L_out, w, s, p, d):
    """Dense matrix of the forward (cross-correlation) convolution that maps a
    Cout x L_out signal u to a Cin x L_in signal z in gather form:
    z[ci, j] = sum_co sum_k w[ci, co, k] * u[co, j*s - p + k*d].
    Transposed convolution is defined as the transpose (adjoint) of this map."""
    K = w.shape[2]
    M = np.zeros((cin * L_in, cout * L_out))
    for ci in range(cin):
        for j in range(L_in):
            for co in range(cout):
                for k in range(K):
                    t = j * s - p + k * d
                    if 0 <= t < L_out:
                        M[ci * L_in + j, co * L_out + t] += w[ci, co, k]
    return M


def forward_conv3d_matrix(cin, cout, Lin, Lout, w, s, p, d):
    """3-D analogue of forward_conv_matrix (tensor-product gather)."""
    M = np.zeros((cin * int(np.prod(Lin)), cout * int(np.prod(Lout))))
    K = w.shape[2:]
    for ci in range(cin):
        for j in itertools.product(*[range(n) for n in Lin]):
            r = ci * int(np.prod(Lin)) + np.ravel_multi_index(j, Lin)
            for co in range(cout):
                for k in itertools.product(*[range(n) for n in K]):
                    t = [j[a] * s[a] - p[a] + k[a] * d[a] for a in range(3)]
                    if all(0 <= t[a] < Lout[a] for a in range(3)):
                        c = co * int(np.prod(Lout)) + np.ravel_multi_index(t, Lout)
                        M[r, c] += w[(ci, co) + k]
    return M


def _exact_random(rng, shape, bits=8):
    """fp32-exact values k/2^bits in [-1, 1] (so scaled sums stay exact)."""
    return (rng.integers(-(1 << bits), (1 << bits) + 1, size=shape) / float(1 << bits)).astype(np.float32)


# ------------------------------------------------------------------- pins
def pin_output_sizes(be):
    """Every output size printed on the pages."""
    for op, L, prm, want in load_sizes():
        if op == "convt":
            got = be.ora_convt_len(L, prm["k"], prm["s"], prm["p"], prm["d"], prm["op"])
        else:
            got = be.ora_pool_len(L, prm["k"], prm["s"], prm["p"], 0)
        assert got == want, (op, L, prm, got, want)


def pin_worked_examples(be):
    """l1_p74's printed transposed-matrix examples, checked term by term with
    one-hot input and one-hot weight."""
    for prm, rows in load_worked_examples():
        K, L_in = prm["K"], prm["L_in"]
        L_out = be.ora_convt_len(L_in, K, prm["s"], prm["p"], prm["d"], prm["op"])
        assert L_out == len(rows), (prm, L_out)
        for k in range(K):
            for i in range(L_in):
                x = np.zeros((1, 1, L_in), np.float32)
                x[0, 0, i] = 1
                w = np.zeros((1, 1, K), np.float32)
                w[0, 0, k] = 1
                y = ora.convt(x, w, None, prm["s"], prm["p"], prm["d"], prm["op"], backend=be)
                want = np.array([1.0 if (k, i) in rows[o] else 0.0 for o in range(L_out)])
                assert np.array_equal(y[0, 0], want), (prm, k, i, y[0, 0], want)


def pin_fused_tap_table(be):
    """l2_p50's 27-term list: for pooled output (1,1,1) of the k3/s2/p1 +
    pool-2 geometry, weight tap t and input offset (a,b,c) meet in the pooled
    window iff the pair is in the table, and at the listed pre-pool parity."""
    table = load_taps()
    assert sorted(t for _, _, t in table) == list(range(27))
    pairs = {(off, t): pp for pp, off, t in table}
    # the page's grouping of the 27 terms by input offset: counts 8,4,4,4,2,2,2,1
    counts = sorted((sum(1 for (o, _) in pairs if o == off)
                     for off in itertools.product((0, 1), repeat=3)), reverse=True)
    assert counts == [8, 4, 4, 4, 2, 2, 2, 1], counts
    shape = (1, 1, 4, 4, 4)
    for t in range(27):
        kd, kh, kw = t // 9, (t // 3) % 3, t % 3
        w = np.zeros((1, 1, 3, 3, 3), np.float32)
        w[0, 0, kd, kh, kw] = 1
        for off in itertools.product((0, 1), repeat=3):
            x = np.zeros(shape, np.float32)
            x[0, 0, 1 + off[0], 1 + off[1], 1 + off[2]] = 1
            y = ora.ct3d_scale_pool_bias(x, w, None, np.zeros(1, np.float32), 2, 1, 0, 1, 2,
                                         1.0, 1.0, backend=be)
            want = 0.125 if (off, t) in pairs else 0.0
            assert y[0, 0, 1, 1, 1] == want, (t, off, y[0, 0, 1, 1, 1], want)
            yc = ora.convt(x, w, None, (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), backend=be)
            block = yc[0, 0, 2:4, 2:4, 2:4]
            if (off, t) in pairs:
                pp = pairs[(off, t)]
                want_block = np.zeros((2, 2, 2))
                want_block[pp] = 1.0
                assert np.array_equal(block, want_block), (t, off, block)
            else:
                assert not block.any(), (t, off, block)


def pin_fused_all_taps_in_range(be):
    """l2_p50's boundary check: for the k3/s2/p1 + pool-2 geometry every pooled
    output, edges included, sees all 27 taps per input channel, so unit
    weights on unit input give 27*Cin/8 everywhere (pooled size = input - 1)."""
    for shp in [(1, 2, 3, 5, 4), (2, 1, 2, 2, 7)]:
        x = np.ones(shp, np.float32)
        w = np.ones((shp[1], 3, 3, 3, 3), np.float32)
        y = ora.ct3d_scale_pool_bias(x, w, None, np.zeros(3, np.float32), 2, 1, 0, 1, 2,
                                     1.0, 1.0, backend=be)
        assert y.shape == (shp[0], 3, shp[2] - 1, shp[3] - 1, shp[4] - 1), y.shape
        assert np.all(y == 27.0 * shp[1] / 8.0), np.unique(y)


def pin_avgpool_constant(be):
    """l1_p46: divisor is always 27 with count_include_pad, so a constant c
    gives c in the interior, c*18/27 on a face, c*12/27 on an edge, c*8/27 at
    a corner (even sizes: only the low side touches padding; odd sizes: the
    high side too).  With count_include_pad off every output is c."""
    c = 0.75
    for shp in [(1, 1, 6, 8, 10), (1, 2, 7, 5, 9)]:
        x = np.full(shp, c, np.float32)
        y = ora.avgpool3d(x, 3, 2, 1, 1, 0, backend=be)
        P = [(n + 2 - 3) // 2 + 1 for n in shp[2:]]
        assert y.shape == (shp[0], shp[1], *P)
        for idx in itertools.product(*[range(n) for n in P]):
            inside = 1
            for a in range(3):
                lo = 2 * idx[a] - 1
                inside *= sum(1 for u in range(lo, lo + 3) if 0 <= u < shp[2 + a])
            assert abs(y[(0, 0) + idx] - c * inside / 27.0) < 1e-15, (shp, idx)
        assert y[0, 0, 0, 0, 0] == c * 8 / 27 and y[0, 0, 1, 1, 1] == c
        y2 = ora.avgpool3d(x, 3, 2, 1, 0, 0, backend=be)
        assert np.allclose(y2, c, rtol=0, atol=1e-15)


def pin_avgpool_separable(be):
    """l1_p46's separable form: W sums, then H sums, then D sums of the padded
    input, subsampled by 2 and divided by 27, equal the pool."""
    rng = np.random.default_rng(7)
    for shp in [(2, 3, 6, 7, 9), (1, 1, 9, 4, 16)]:
        x = rng.standard_normal(shp).astype(np.float32)
        xp = np.pad(x.astype(np.float64), [(0, 0), (0, 0), (1, 1), (1, 1), (1, 1)])
        sw = xp[..., :-2] + xp[..., 1:-1] + xp[..., 2:]
        sh = sw[..., :-2, :] + sw[..., 1:-1, :] + sw[..., 2:, :]
        sd = sh[:, :, :-2] + sh[:, :, 1:-1] + sh[:, :, 2:]
        want = sd[:, :, ::2, ::2, ::2] / 27.0
        y = ora.avgpool3d(x, 3, 2, 1, 1, 0, backend=be)
        assert y.shape == want.shape, (y.shape, want.shape)
        assert np.allclose(y, want, rtol=1e-13, atol=1e-13)


def pin_avgpool_general_window(be):
    """Other windows (k, s, p) and count_include_pad off: brute force over the
    window of every output."""
    rng = np.random.default_rng(11)
    for (k, s, p, cip) in [((2, 3, 3), (1, 2, 3), (1, 0, 1), 1), ((3, 3, 2), (2, 1, 2), (1, 1, 0), 0),
                           ((4, 2, 5), (3, 2, 2), (2, 1, 2), 0)]:
        x = rng.standard_normal((1, 2, 7, 6, 9)).astype(np.float32)
        y = ora.avgpool3d(x, k, s, p, cip, 0, backend=be)
        for n, c in itertools.product(range(1), range(2)):
            for idx in itertools.product(*[range(v) for v in y.shape[2:]]):
                tot, cnt = 0.0, 0
                for u in itertools.product(*[range(idx[a] * s[a] - p[a], idx[a] * s[a] - p[a] + k[a])
                                             for a in range(3)]):
                    if all(0 <= u[a] < x.shape[2 + a] for a in range(3)):
                        tot += float(x[(n, c) + u])
                        cnt += 1
                div = k[0] * k[1] * k[2] if cip else cnt
                assert abs(y[(n, c) + idx] - tot / div) < 1e-12


def pin_avgpool_ceil_mode(be):
    """Ceil mode (not used on the pages): size ceil((L+2p-k)/s)+1, dropping a
    last window that would start past L+p; with count_include_pad the divisor
    counts window cells up to L+p."""
    assert be.ora_pool_len(6, 3, 2, 1, 1) == 4 and be.ora_pool_len(6, 3, 2, 1, 0) == 3
    assert be.ora_pool_len(5, 2, 2, 0, 1) == 3 and be.ora_pool_len(4, 2, 2, 1, 1) == 3
    # a last window that would start in the right padding is dropped
    assert be.ora_pool_len(5, 2, 3, 1, 1) == 2 and be.ora_pool_len(4, 2, 3, 1, 1) == 2
    x = np.ones((1, 1, 6, 6, 6), np.float32)
    y = ora.avgpool3d(x, 3, 2, 1, 1, 1, backend=be)
    assert y.shape == (1, 1, 4, 4, 4)
    # last window per dim: cells 5,6 (6 is the right pad) -> 1 real of 2 counted
    assert abs(y[0, 0, 3, 3, 3] - 1.0 / 8.0) < 1e-15
    assert abs(y[0, 0, 0, 0, 0] - 8.0 / 27.0) < 1e-15
    y0 = ora.avgpool3d(x, 3, 2, 1, 0, 1, backend=be)
    assert np.allclose(y0, 1.0, rtol=0, atol=1e-15)


def pin_convt1d_dense_transpose(be):
    """Transposed convolution equals the transpose of the dense forward
    convolution matrix, over strides, paddings, dilations, taps and output
    paddings (l1_p74 derives the transposed form this way)."""
    rng = np.random.default_rng(3)
    cases = 0
    for s, p, d, K in itertools.product((1, 2, 3), (0, 1, 2), (1, 2, 3), (1, 2, 3, 5)):
        for op in range(max(s, d)):
            L_in = int(rng.integers(1, 6))
            cin, cout = 2, 3
            L_out = (L_in - 1) * s - 2 * p + d * (K - 1) + op + 1
            if L_out <= 0:
                continue
            x = rng.standard_normal((1, cin, L_in)).astype(np.float32)
            w = rng.standard_normal((cin, cout, K)).astype(np.float32)
            b = rng.standard_normal(cout).astype(np.float32)
            M = forward_conv_matrix(cin, cout, L_in, L_out, w.astype(np.float64), s, p, d)
            want = (M.T @ x.reshape(-1).astype(np.float64)).reshape(cout, L_out) + b[:, None]
            y = ora.convt(x, w, b, s, p, d, op, backend=be)
            assert y.shape == (1, cout, L_out), (y.shape, L_out, (s, p, d, K, op))
            assert np.allclose(y[0], want, rtol=1e-12, atol=1e-12), (s, p, d, K, op)
            cases += 1
    assert cases > 100


def pin_convt3d_dense_transpose(be):
    """3-D transposed convolution equals the transpose of the dense 3-D forward
    convolution matrix (mixed strides/paddings/dilations per dim)."""
    rng = np.random.default_rng(5)
    for (Lin, K, s, p, d, op) in [((2, 3, 2), (3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0)),
                                  ((2, 2, 3), (2, 3, 1), (1, 2, 3), (0, 1, 0), (2, 1, 1), (1, 1, 2)),
                                  ((3, 2, 2), (3, 2, 2), (3, 1, 2), (2, 0, 1), (1, 3, 2), (2, 0, 1))]:
        cin, cout = 2, 2
        Lout = tuple((Lin[a] - 1) * s[a] - 2 * p[a] + d[a] * (K[a] - 1) + op[a] + 1 for a in range(3))
        x = rng.standard_normal((1, cin) + Lin).astype(np.float32)
        w = rng.standard_normal((cin, cout) + K).astype(np.float32)
        M = forward_conv3d_matrix(cin, cout, Lin, Lout, w.astype(np.float64), s, p, d)
        want = (M.T @ x.reshape(-1).astype(np.float64)).reshape((cout,) + Lout)
        y = ora.convt(x, w, None, s, p, d, op, backend=be)
        assert y.shape == (1, cout) + Lout, (y.shape, Lout)
        assert np.allclose(y[0], want, rtol=1e-12, atol=1e-12), (Lin, K, s, p, d, op)


def pin_adjoint_identity(be):
    """<conv(u), v> = <u, convT(v)> (l1_p74's adjoint argument), with the
    forward convolution evaluated directly in gather form."""
    rng = np.random.default_rng(9)
    for s, p, d, K, L_in in [(1, 0, 3, 5, 9), (2, 1, 2, 4, 7), (3, 2, 1, 5, 6)]:
        cin, cout = 3, 2
        L_out = (L_in - 1) * s - 2 * p + d * (K - 1) + 1
        u = rng.standard_normal((cout, L_out))
        v = rng.standard_normal((1, cin, L_in)).astype(np.float32)
        w = rng.standard_normal((cin, cout, K)).astype(np.float32)
        conv_u = np.zeros((cin, L_in))
        for ci, j, co, k in itertools.product(range(cin), range(L_in), range(cout), range(K)):
            t = j * s - p + k * d
            if 0 <= t < L_out:
                conv_u[ci, j] += float(w[ci, co, k]) * u[co, t]
        lhs = float(np.sum(conv_u * v[0].astype(np.float64)))
        rhs = float(np.sum(u * ora.convt(v, w, None, s, p, d, 0, backend=be)[0]))
        assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs)), (lhs, rhs)


def pin_stride1_flipped_conv(be):
    """l1_p74: with stride 1 and no padding, the transposed convolution is a
    plain correlation with the tap order reversed over an input zero-padded by
    (K-1)*d on both sides."""
    rng = np.random.default_rng(13)
    for K, d, L in [(5, 3, 20), (2, 1, 6), (3, 2, 5), (4, 1, 11)]:
        x = rng.standard_normal((1, 2, L)).astype(np.float32)
        w = rng.standard_normal((2, 3, K)).astype(np.float32)
        P = (K - 1) * d
        xp = np.pad(x[0].astype(np.float64), [(0, 0), (P, P)])
        wf = w[:, :, ::-1].astype(np.float64)
        want = np.zeros((3, L + P))
        for o in range(L + P):
            for k in range(K):
                want[:, o] += np.einsum("c,cq->q", xp[:, o + k * d], wf[:, :, k])
        y = ora.convt(x, w, None, 1, 0, d, 0, backend=be)
        assert y.shape == (1, 3, L + P)
        assert np.allclose(y[0], want, rtol=1e-12, atol=1e-12), (K, d, L)


def effective_fused(x, w, conv_bias, bias, s1, s2):
    """Second derivation of the k3/s2/p1 + pool-2 chain (l2_p50's collapsed
    form): group the 27 taps by the input neighbour they read -- offset 0 in a
    dim takes taps {1, 2}, offset 1 takes tap {0} -- and run the resulting
    2x2x2 valid correlation, then the affine epilogue."""
    x = x.astype(np.float64)
    w = w.astype(np.float64)
    N, cin, D, H, W = x.shape
    cout = w.shape[1]
    T = {0: (1, 2), 1: (0,)}
    y = np.zeros((N, cout, D - 1, H - 1, W - 1))
    for a, b, c in itertools.product((0, 1), repeat=3):
        g = np.zeros((cin, cout))
        for kd in T[a]:
            for kh in T[b]:
                for kw in T[c]:
                    g += w[:, :, kd, kh, kw]
        xs = x[:, :, a:a + D - 1, b:b + H - 1, c:c + W - 1]
        y += np.einsum("nidhw,io->nodhw", xs, g)
    cb = np.zeros(cout) if conv_bias is None else conv_bias.astype(np.float64)
    return ((y / 8.0 + cb[None, :, None, None, None]) * s1 + bias.astype(np.float64)[None, :, None, None, None]) * s2


def pin_fused_effective_conv(be):
    """The literal chain equals the collapsed 2x2x2 form to 1e-12."""
    rng = np.random.default_rng(17)
    for shp, cout in [((2, 3, 3, 4, 5), 4), ((1, 2, 5, 2, 6), 3), ((1, 3, 2, 3, 2), 16)]:
        x = rng.uniform(-1, 1, shp).astype(np.float32)
        w = rng.uniform(-0.05, 0.05, (shp[1], cout, 3, 3, 3)).astype(np.float32)
        cb = rng.uniform(-0.05, 0.05, cout).astype(np.float32)
        b = (0.02 * rng.standard_normal(cout)).astype(np.float32)
        want = effective_fused(x, w, cb, b, 0.5, 1.5)
        y = ora.ct3d_scale_pool_bias(x, w, cb, b, 2, 1, 0, 1, 2, 0.5, 1.5, backend=be)
        assert y.shape == want.shape, (y.shape, want.shape)
        assert np.allclose(y, want, rtol=1e-12, atol=1e-13), np.abs(y - want).max()


def pin_zero_input_affine(be):
    """x = 0: the fused output is (conv_bias*s1 + bias)*s2 everywhere and the
    transposed convolution is its bias."""
    rng = np.random.default_rng(19)
    cb = rng.uniform(-1, 1, 5).astype(np.float32)
    b = rng.uniform(-1, 1, 5).astype(np.float32)
    y = ora.ct3d_scale_pool_bias(np.zeros((1, 2, 3, 3, 3), np.float32),
                                 rng.uniform(-1, 1, (2, 5, 3, 3, 3)).astype(np.float32),
                                 cb, b, 2, 1, 0, 1, 2, 0.5, 1.25, backend=be)
    want = (cb.astype(np.float64) * 0.5 + b) * 1.25
    assert np.array_equal(y[0], np.broadcast_to(want[:, None, None, None], y.shape[1:]))
    y1 = ora.convt(np.zeros((2, 3, 7), np.float32), rng.uniform(-1, 1, (3, 5, 4)).astype(np.float32),
                   b, 2, 1, 2, 1, backend=be)
    assert np.array_equal(y1, np.broadcast_to(b.astype(np.float64)[None, :, None], y1.shape))


def pin_linearity(be):
    """f(a*u + b*v) - f(0) = a*(f(u) - f(0)) + b*(f(v) - f(0)) for the fused chain
    and for the transposed convolution (inputs chosen so a*u + b*v is exact in
    fp32)."""
    rng = np.random.default_rng(23)
    shp = (1, 2, 3, 4, 3)
    u, v = _exact_random(rng, shp), _exact_random(rng, shp)
    w = _exact_random(rng, (2, 3, 3, 3, 3))
    cb, bb = _exact_random(rng, 3), _exact_random(rng, 3)
    f = lambda z: ora.ct3d_scale_pool_bias(z, w, cb, bb, 2, 1, 0, 1, 2, 0.5, 1.5, backend=be)
    z = (np.float32(2.0) * u - np.float32(0.5) * v).astype(np.float32)
    f0 = f(np.zeros(shp, np.float32))
    assert np.allclose(f(z) - f0, 2.0 * (f(u) - f0) - 0.5 * (f(v) - f0), rtol=0, atol=1e-12)
    u1, v1 = _exact_random(rng, (2, 3, 9)), _exact_random(rng, (2, 3, 9))
    w1 = _exact_random(rng, (3, 4, 4))
    g = lambda q: ora.convt(q, w1, cb[:1].repeat(4), 2, 1, 2, 1, backend=be)
    z1 = (np.float32(2.0) * u1 - np.float32(0.5) * v1).astype(np.float32)
    g0 = g(np.zeros_like(u1))
    assert np.allclose(g(z1) - g0, 2.0 * (g(u1) - g0) - 0.5 * (g(v1) - g0), rtol=0, atol=1e-12)


def pin_strided_even_outputs_are_bias(be):
    """Stride 2, dilation 2, padding 1: o + 1 - 2k is odd for even o, so no tap
    reaches an even output; it equals the bias exactly.  Each odd output has at
    most K = 4 taps, all at inputs (o + 1)/2 - k."""
    rng = np.random.default_rng(29)
    L = 9
    x = rng.standard_normal((2, 3, L)).astype(np.float32)
    w = rng.standard_normal((3, 4, 4)).astype(np.float32)
    b = rng.standard_normal(4).astype(np.float32)
    y = ora.convt(x, w, b, 2, 1, 2, 1, backend=be)
    assert y.shape == (2, 4, 2 * L + 4), y.shape  # (L-1)*2 - 2 + 2*3 + 1 + 1
    assert np.array_equal(y[:, :, 0::2], np.broadcast_to(b.astype(np.float64)[None, :, None],
                                                         y[:, :, 0::2].shape))
    xx = x.astype(np.float64)
    ww = w.astype(np.float64)
    for o in range(1, y.shape[2], 2):
        want = b.astype(np.float64).copy()
        for k in range(4):
            i = (o + 1) // 2 - k
            if 0 <= i < L:
                want = want + np.einsum("nc,co->no", xx[:, :, i], ww[:, :, k])
        assert np.allclose(y[:, :, o], want, rtol=1e-12, atol=1e-12), o


ALL_PINS = [pin_output_sizes, pin_worked_examples, pin_fused_tap_table,
            pin_fused_all_taps_in_range, pin_avgpool_constant, pin_avgpool_separable,
            pin_avgpool_general_window, pin_avgpool_ceil_mode, pin_convt1d_dense_transpose,
            pin_convt3d_dense_transpose, pin_adjoint_identity, pin_stride1_flipped_conv,
            pin_fused_effective_conv, pin_zero_input_affine, pin_linearity,
            pin_strided_even_outputs_are_bias]
