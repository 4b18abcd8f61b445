"""Pins for the fp64 reference of the input preparation and output norm: each ties it to
a closed form, a brute-force loop or an identity, not to itself."""
import math

import numpy as np

from oracle import prep


def _rand(rng, T, H, D, W=4):
    xq, xk, xv = (rng.standard_normal((T, H, D)) for _ in range(3))
    w = rng.standard_normal((3, H, D, W)) * 0.5
    a = rng.standard_normal((T, H, D))
    b = rng.standard_normal((T, H))
    return xq, xk, xv, w, a, b


def test_identity_taps_reduce_to_norm_and_copy():
    """Taps (0, 0, 0, 1), no activation: q and k are just normalised, v is copied."""
    rng = np.random.default_rng(1)
    T, H, D = 9, 2, 8
    xq, xk, xv, _, a, b = _rand(rng, T, H, D)
    w = np.zeros((3, H, D, 4)); w[..., 3] = 1.0
    q, k, v, la, beta = prep.prepare_inputs(xq, xk, xv, w, a, b, [0, T], act=0)
    np.testing.assert_allclose(q, xq / np.linalg.norm(xq, axis=-1, keepdims=True), rtol=1e-6)
    np.testing.assert_allclose(k, xk / np.linalg.norm(xk, axis=-1, keepdims=True), rtol=1e-6)
    np.testing.assert_array_equal(v, xv)


def test_impulse_response_is_the_taps_in_time_order():
    """A unit impulse at token 2 of v, no activation: v[2 + i] = w[W-1-i] (tap order)."""
    T, H, D, W = 8, 1, 2, 4
    x = np.zeros((T, H, D)); x[2, 0, :] = 1.0
    w = np.arange(1.0, 1.0 + 3 * H * D * W).reshape(3, H, D, W)
    _, _, v, _, _ = prep.prepare_inputs(np.ones((T, H, D)), np.ones((T, H, D)), x, w, np.zeros((T, H, D)),
                                        np.zeros((T, H)), [0, T], act=0)
    for i in range(W):
        np.testing.assert_array_equal(v[2 + i, 0], w[2, 0, :, W - 1 - i])
    assert not v[:2].any() and not v[2 + W:].any()


def test_brute_force_single_element():
    """One output element written out from the definition, with SiLU."""
    rng = np.random.default_rng(2)
    T, H, D = 6, 2, 4
    xq, xk, xv, w, a, b = _rand(rng, T, H, D)
    _, k, _, _, _ = prep.prepare_inputs(xq, xk, xv, w, a, b, [0, T], act=1)
    t, h = 4, 1
    raw = [sum(w[1, h, c, j] * xk[t - 3 + j, h, c] for j in range(4)) for c in range(D)]
    act = [r / (1.0 + math.exp(-r)) for r in raw]
    nrm = math.sqrt(sum(x * x for x in act) + prep.L2_EPS)
    np.testing.assert_allclose(k[t, h], np.array(act) / nrm, rtol=1e-12)


def test_sequences_do_not_leak_and_carry_state():
    """Packed sequences convolve independently; a continuation given the last W-1 raw
    inputs of its prefix as conv_state equals one pass over prefix + continuation."""
    rng = np.random.default_rng(3)
    T, H, D = 14, 2, 4
    xq, xk, xv, w, a, b = _rand(rng, T, H, D)
    one = prep.prepare_inputs(xq, xk, xv, w, a, b, [0, T])
    packed = prep.prepare_inputs(xq, xk, xv, w, a, b, [0, 5, T])
    sep = prep.prepare_inputs(xq[5:], xk[5:], xv[5:], w, a[5:], b[5:], [0, T - 5])
    for x, y in zip(packed, sep):
        np.testing.assert_allclose(x[5:], y, rtol=1e-12)
    state = np.stack([xq[2:5], xk[2:5], xv[2:5]])[None]          # [1, 3, W-1, H, D]
    cont = prep.prepare_inputs(xq[5:], xk[5:], xv[5:], w, a[5:], b[5:], [0, T - 5], conv_state=state)
    for x, y in zip(one, cont):
        np.testing.assert_allclose(x[5:], y, rtol=1e-12)


def test_gate_closed_forms():
    z = np.array([[0.0, -40.0, 40.0, 3.0]])
    _, _, _, la, beta = prep.prepare_inputs(np.ones((1, 1, 4)), np.ones((1, 1, 4)), np.ones((1, 1, 4)),
                                            np.ones((3, 1, 4, 4)), z[:, None, :], np.array([[0.0]]), [0, 1])
    np.testing.assert_allclose(la[0, 0], [-math.log(2.0), -math.exp(-40.0), -40.0 - math.exp(-40.0),
                                          -math.log1p(math.exp(3.0))], rtol=1e-12)
    assert beta[0, 0] == 0.5
    assert np.all(la <= 0)


def test_output_norm_unit_rms_and_weight():
    rng = np.random.default_rng(4)
    o = rng.standard_normal((5, 3, 16)) * 7.0
    g = rng.uniform(0.5, 2.0, (3, 16))
    y = prep.output_norm(o, np.ones((3, 16)), eps=0.0)
    np.testing.assert_allclose(np.sqrt((y * y).mean(-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(prep.output_norm(o, g, eps=0.0), y * g[None], rtol=1e-12)
    np.testing.assert_allclose(prep.output_norm(3.0 * o, g, eps=0.0), prep.output_norm(o, g, eps=0.0), rtol=1e-12)
