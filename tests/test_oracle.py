"""Pins of the fp64 oracle against what the pages and the mathematics fix.

No expected value here comes from the CUDA library.  Each pin is an
independent route to the same number: a hand-derived closed form, a special
case that reduces to a textbook computation (prefix sum, geometric decay,
numpy's correlate), the brute-force chunk form of TensorRT-Model-Connect
#2207 ("Implementation") against the row-by-row recurrence of TensorSharp
"nemotron.md" section 4.1, or an invariant (linearity, group expansion,
split invariance).
"""
import math

import numpy as np
import pytest

import oracle
import ssd_inputs as si

TINY = si.TINY


def _tiny_problem(seed=0, z=False, h0=False, shape=TINY, stress=False):
    p = si.params(shape, seed=seed, stress=stress)
    a = si.prefill_inputs(shape, seed=seed, act_dtype=__import__("torch").float32,
                          initial_state=h0, with_z=z, stress=stress)
    conv = {k: p[k].double().numpy() for k in ("conv_w", "conv_b")}
    xbc_raw = a["xbc"].double().numpy()
    xbc, _ = oracle.conv1d(xbc_raw, conv["conv_w"], conv["conv_b"], None)
    out = dict(xbc=xbc, dt_raw=a["dt_raw"].double().numpy(),
               dt_bias=p["dt_bias"].double().numpy(), A=p["A"].double().numpy(),
               D=p["D"].double().numpy(),
               z=None if a["z"] is None else a["z"].double().numpy(),
               h0=None if a["ssm_state"] is None else a["ssm_state"].double().numpy())
    return out


def _dims(shape):
    return dict(H=shape.nheads, P=shape.headdim, N=shape.dstate, G=shape.ngroups)


def _relerr(a, b):
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / (den if den > 0 else 1.0))


# --------------------------------------------------------------------------
# hand-derived closed forms (H = P = N = G = 1)

def _scalar_xbc(xs, Bs, Cs):
    return np.array([[[x, b, c] for x, b, c in zip(xs, Bs, Cs)]], dtype=np.float64)


def test_single_step_hand_values():
    # dt passed directly, A = -ln 2 so the decay is exactly 1/2.
    # h1 = 0.5*2 + 1*1*2 = 3 ; y1 = 3*3 + 0.5*1 = 9.5   (post-update state)
    # h2 = 0.5*3 + 1*2*2 = 5.5 ; y2 = 3*5.5 + 0.5*2 = 17.5
    xbc = _scalar_xbc([1.0, 2.0], [2.0, 2.0], [3.0, 3.0])
    dt = np.ones((1, 2, 1))
    y, hS = oracle.ssd_sequential(xbc, dt, np.array([-math.log(2.0)]), H=1, P=1, N=1, G=1,
                                  D=np.array([0.5]), h0=np.array([[[[2.0]]]]),
                                  dt_softplus=False)
    assert y[0, :, 0, 0] == pytest.approx([9.5, 17.5], abs=1e-14)
    assert hS[0, 0, 0, 0] == pytest.approx(5.5, abs=1e-14)


def test_softplus_and_bias_hand_values():
    # dt = softplus(0.3 + 0.2) = ln(1 + e^0.5); decay e^{dt*A}; N = P = 1
    sp = math.log1p(math.exp(0.5))
    A = -0.7
    h1 = math.exp(sp * A) * 1.5 + sp * 0.4 * -1.1
    y1 = 0.9 * h1
    xbc = _scalar_xbc([0.4], [-1.1], [0.9])
    y, hS = oracle.ssd_sequential(xbc, np.full((1, 1, 1), 0.3), np.array([A]), H=1, P=1,
                                  N=1, G=1, dt_bias=np.array([0.2]),
                                  h0=np.array([[[[1.5]]]]))
    assert y[0, 0, 0, 0] == pytest.approx(y1, rel=1e-14)
    assert hS[0, 0, 0, 0] == pytest.approx(h1, rel=1e-14)


def test_three_step_unrolled_sum():
    # Three steps unrolled by hand into the convolutional sum:
    # h3 = e^{a1+a2+a3} h0 + e^{a2+a3} dt1 x1 B1 + e^{a3} dt2 x2 B2 + dt3 x3 B3
    rng = np.random.default_rng(3)
    xs, Bs, Cs = rng.normal(size=3), rng.normal(size=3), rng.normal(size=3)
    dts = rng.uniform(0.1, 1.0, size=3)
    A, h0 = -0.8, 0.37
    a = dts * A
    h3 = (math.exp(a.sum()) * h0 + math.exp(a[1] + a[2]) * dts[0] * xs[0] * Bs[0]
          + math.exp(a[2]) * dts[1] * xs[1] * Bs[1] + dts[2] * xs[2] * Bs[2])
    h2 = (math.exp(a[0] + a[1]) * h0 + math.exp(a[1]) * dts[0] * xs[0] * Bs[0]
          + dts[1] * xs[1] * Bs[1])
    y, hS = oracle.ssd_sequential(_scalar_xbc(xs, Bs, Cs), dts.reshape(1, 3, 1),
                                  np.array([A]), H=1, P=1, N=1, G=1,
                                  h0=np.array([[[[h0]]]]), dt_softplus=False)
    assert hS[0, 0, 0, 0] == pytest.approx(h3, rel=1e-13)
    assert y[0, 1, 0, 0] == pytest.approx(Cs[1] * h2, rel=1e-13)


# --------------------------------------------------------------------------
# special cases with textbook answers

def test_dt_zero_leaves_state_unchanged():
    prob = _tiny_problem(h0=True)
    dt0 = np.zeros_like(prob["dt_raw"])
    y, hS = oracle.ssd_sequential(prob["xbc"], dt0, prob["A"], **_dims(TINY), D=prob["D"],
                                  h0=prob["h0"], dt_softplus=False)
    assert np.array_equal(hS, prob["h0"])
    H, P, N, G = TINY.nheads, TINY.headdim, TINY.dstate, TINY.ngroups
    x = prob["xbc"][..., : H * P].reshape(1, -1, H, P)
    Cm = prob["xbc"][..., H * P + G * N:].reshape(1, -1, G, N)
    Ch = np.repeat(Cm, H // G, axis=2)
    expect = np.einsum("bthn,bhpn->bthp", Ch, prob["h0"]) + prob["D"][None, None, :, None] * x
    assert _relerr(y, expect) < 1e-13


def test_zero_input_is_geometric_decay():
    prob = _tiny_problem(h0=True)
    H, P = TINY.nheads, TINY.headdim
    xbc = prob["xbc"].copy()
    xbc[..., : H * P] = 0.0
    y, hS = oracle.ssd_sequential(xbc, prob["dt_raw"], prob["A"], **_dims(TINY),
                                  dt_bias=prob["dt_bias"], h0=prob["h0"])
    dt = np.log1p(np.exp(prob["dt_raw"] + prob["dt_bias"]))  # softplus, moderate values
    total = dt.sum(axis=1)[0]  # [H]
    expect = np.exp(prob["A"] * total)[:, None, None] * prob["h0"][0]
    assert _relerr(hS[0], expect) < 1e-12


def test_A_zero_is_prefix_sum():
    prob = _tiny_problem(h0=True)
    H, P, N, G = TINY.nheads, TINY.headdim, TINY.dstate, TINY.ngroups
    A0 = np.zeros(H)
    y, hS = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], A0, **_dims(TINY),
                                  dt_bias=prob["dt_bias"], D=prob["D"], h0=prob["h0"])
    dt = np.log1p(np.exp(prob["dt_raw"] + prob["dt_bias"]))[0]  # [S,H]
    x = prob["xbc"][0, :, : H * P].reshape(-1, H, P)
    Bm = np.repeat(prob["xbc"][0, :, H * P: H * P + G * N].reshape(-1, G, N), H // G, axis=1)
    Cm = np.repeat(prob["xbc"][0, :, H * P + G * N:].reshape(-1, G, N), H // G, axis=1)
    inc = dt[:, :, None, None] * x[:, :, :, None] * Bm[:, :, None, :]  # [S,H,P,N]
    states = prob["h0"][0][None] + np.cumsum(inc, axis=0)
    assert _relerr(hS[0], states[-1]) < 1e-13
    y_expect = np.einsum("thn,thpn->thp", Cm, states) + prob["D"][None, :, None] * x
    assert _relerr(y[0], y_expect) < 1e-13


# --------------------------------------------------------------------------
# chunk form == recurrence (TensorRT-Model-Connect #2207: 11 rows as 7 + 4)

@pytest.mark.parametrize("parts", [[11], [7, 4], [1] * 11, [3, 1, 5, 2], [4, 7]])
@pytest.mark.parametrize("with_z", [False, True])
def test_chunked_equals_sequential(parts, with_z):
    prob = _tiny_problem(z=with_z, h0=True)
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"], z=prob["z"], h0=prob["h0"])
    y1, h1 = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], **_dims(TINY), **kw)
    y2, h2 = oracle.ssd_chunked(prob["xbc"], prob["dt_raw"], prob["A"], parts, **_dims(TINY),
                                **kw)
    assert y1.size == 1 * 11 * 4 * 16 and h1.size == 4 * 16 * 16
    assert _relerr(y2, y1) < 1e-12
    assert _relerr(h2, h1) < 1e-12


def test_chunk_form_clamp_hand_values():
    """The clamp of the chunk form where gamma rises (TensorRT-Model-Connect
    #2207 "Implementation": every exponent of the chunk form is at most 0).

    One chunk of 3 rows, H = P = N = G = 1, dt taken as given, A = -1,
    dt = (1, -2, 0.5): a = (-1, 2, -0.5), gamma = (-1, 1, 0.5), gamma_L = 0.5.
    x = (1.5, -0.5, 2), B = (0.5, 2, -1), C = (1, -1.5, 0.25), D = 0.5, h0 = 0.75,
    so dt*x = (1.5, 1, 1).  Clamped exponents min(gamma_t - gamma_s, 0):
      t=0: s=0 -> 0;         h0 term min(-1, 0) = -1
      t=1: s=0 -> min(2,0)=0, s=1 -> 0;           h0 term min(1, 0) = 0
      t=2: s=0 -> min(1.5,0)=0, s=1 -> -0.5, s=2 -> 0; h0 term 0
      state: L - s: min(1.5,0)=0, min(-0.5,0)=-0.5, 0;  h0 term min(0.5, 0) = 0
    y0 = 0.5*1.5 + e^-1*1*0.75 + 0.5*1.5              = 1.5 + 0.75 e^-1
    y1 = -0.75*1.5 + -3*1 + 1*(-1.5*0.75) + 0.5*(-0.5) = -5.5
    y2 = 0.125*1.5 + 0.5*e^-0.5*1 + -0.25*1 + 0.25*0.75 + 0.5*2 = 1.125 + 0.5 e^-0.5
    h  = 0.75 + 1.5*0.5 + e^-0.5*1*2 + 1*(-1)          = 0.5 + 2 e^-0.5
    Without the clamp (or with gamma_t and gamma_s clamped one by one) rows 1
    and 2 and the state pick up factors e^1, e^1.5 or e^2 instead."""
    xbc = _scalar_xbc([1.5, -0.5, 2.0], [0.5, 2.0, -1.0], [1.0, -1.5, 0.25])
    dt = np.array([1.0, -2.0, 0.5]).reshape(1, 3, 1)
    y, hS = oracle.ssd_chunked(xbc, dt, np.array([-1.0]), [3], H=1, P=1, N=1, G=1,
                               D=np.array([0.5]), h0=np.array([[[[0.75]]]]), dt_softplus=False)
    y_expect = np.array([1.5 + 0.75 * math.exp(-1.0), -5.5, 1.125 + 0.5 * math.exp(-0.5)])
    assert _relerr(y.reshape(3), y_expect) < 1e-14
    assert abs(hS.item() - (0.5 + 2.0 * math.exp(-0.5))) < 1e-14


def test_chunk_form_clamp_carries_across_chunks():
    """The same 3 rows as two chunks 2 + 1: gamma restarts at each chunk.
    Chunk 1 (rows 0,1): gamma = (-1, 1), gamma_L = 1.
      y0 = 1.5 + 0.75 e^-1 (as in one chunk); y1 = -5.5 (as in one chunk);
      h1 = e^min(1,0)*0.75 + e^min(2,0)*1.5*0.5 + e^0*1*2 = 0.75 + 0.75 + 2 = 3.5
    Chunk 2 (row 2): gamma = (-0.5), gamma_L = -0.5.
      y2 = -0.25*1 + e^-0.5*0.25*3.5 + 0.5*2 = 0.75 + 0.875 e^-0.5
      h  = e^-0.5*3.5 + 1*(-1) = 3.5 e^-0.5 - 1"""
    xbc = _scalar_xbc([1.5, -0.5, 2.0], [0.5, 2.0, -1.0], [1.0, -1.5, 0.25])
    dt = np.array([1.0, -2.0, 0.5]).reshape(1, 3, 1)
    y, hS = oracle.ssd_chunked(xbc, dt, np.array([-1.0]), [2, 1], H=1, P=1, N=1, G=1,
                               D=np.array([0.5]), h0=np.array([[[[0.75]]]]), dt_softplus=False)
    y_expect = np.array([1.5 + 0.75 * math.exp(-1.0), -5.5, 0.75 + 0.875 * math.exp(-0.5)])
    assert _relerr(y.reshape(3), y_expect) < 1e-14
    assert abs(hS.item() - (3.5 * math.exp(-0.5) - 1.0)) < 1e-14


def test_chunked_rejects_bad_partition():
    prob = _tiny_problem()
    with pytest.raises(ValueError):
        oracle.ssd_chunked(prob["xbc"], prob["dt_raw"], prob["A"], [5, 5], **_dims(TINY))


def test_split_calls_equal_one_call():
    """Two calls chained through the final state == one call over all rows."""
    prob = _tiny_problem(h0=True)
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"])
    y, h = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], **_dims(TINY),
                                 h0=prob["h0"], **kw)
    ya, ha = oracle.ssd_sequential(prob["xbc"][:, :7], prob["dt_raw"][:, :7], prob["A"],
                                   **_dims(TINY), h0=prob["h0"], **kw)
    yb, hb = oracle.ssd_sequential(prob["xbc"][:, 7:], prob["dt_raw"][:, 7:], prob["A"],
                                   **_dims(TINY), h0=ha, **kw)
    assert np.array_equal(np.concatenate([ya, yb], axis=1), y)
    assert np.array_equal(hb, h)


# --------------------------------------------------------------------------
# decay of about 1e6 per row (TensorRT-Model-Connect #2207 Tests)

@pytest.mark.parametrize("form", ["sequential", "chunked"])
def test_huge_decay_limit(form):
    shape = TINY.with_(seqlen=9)
    prob = _tiny_problem(h0=True, shape=shape, stress=True)
    dt_raw = np.full_like(prob["dt_raw"], 300.0)  # dt ~ 300, |A| >= 1e3 -> |dt A| >= 3e5
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"], h0=prob["h0"])
    if form == "sequential":
        y, hS = oracle.ssd_sequential(prob["xbc"], dt_raw, prob["A"], **_dims(shape), **kw)
    else:
        y, hS = oracle.ssd_chunked(prob["xbc"], dt_raw, prob["A"], [4, 5], **_dims(shape), **kw)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(hS))
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    dt = dt_raw[0] + prob["dt_bias"][None, :]  # softplus(v) == v to 1e-130 at v ~ 300
    x = prob["xbc"][0, :, : H * P].reshape(-1, H, P)
    Bm = np.repeat(prob["xbc"][0, :, H * P: H * P + G * N].reshape(-1, G, N), H // G, axis=1)
    Cm = np.repeat(prob["xbc"][0, :, H * P + G * N:].reshape(-1, G, N), H // G, axis=1)
    h_last = dt[-1][:, None, None] * x[-1][:, :, None] * Bm[-1][:, None, :]
    assert _relerr(hS[0], h_last) < 1e-12
    cb = np.einsum("thn,thn->th", Cm, Bm)
    y_expect = (cb * dt)[:, :, None] * x + prob["D"][None, :, None] * x
    assert _relerr(y[0], y_expect) < 1e-12


# --------------------------------------------------------------------------
# invariants

def test_linearity_in_x_and_h0():
    prob = _tiny_problem(h0=True)
    H, P = TINY.nheads, TINY.headdim
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"])
    y, h = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], **_dims(TINY),
                                 h0=prob["h0"], **kw)
    xbc2 = prob["xbc"].copy()
    xbc2[..., : H * P] *= -2.5
    y2, h2 = oracle.ssd_sequential(xbc2, prob["dt_raw"], prob["A"], **_dims(TINY),
                                   h0=-2.5 * prob["h0"], **kw)
    assert _relerr(y2, -2.5 * y) < 1e-13
    assert _relerr(h2, -2.5 * h) < 1e-13


def test_group_mapping_equals_expanded_groups():
    """G=2 over H=4 (heads_per_group 2) == G=4 with each head's group copied
    (the head -> group map of vllm.cpp #1362: g = h / heads_per_group)."""
    shape = TINY.with_(ngroups=2)
    prob = _tiny_problem(h0=True, shape=shape)
    H, P, N = shape.nheads, shape.headdim, shape.dstate
    xbc = prob["xbc"]
    x = xbc[..., : H * P]
    Bm = xbc[..., H * P: H * P + 2 * N].reshape(1, -1, 2, N)
    Cm = xbc[..., H * P + 2 * N:].reshape(1, -1, 2, N)
    gmap = [h // (H // 2) for h in range(H)]
    Bx = Bm[:, :, gmap, :].reshape(1, -1, H * N)
    Cx = Cm[:, :, gmap, :].reshape(1, -1, H * N)
    xbc_exp = np.concatenate([x, Bx, Cx], axis=-1)
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"], h0=prob["h0"])
    y1, h1 = oracle.ssd_sequential(xbc, prob["dt_raw"], prob["A"], H=H, P=P, N=N, G=2, **kw)
    y2, h2 = oracle.ssd_sequential(xbc_exp, prob["dt_raw"], prob["A"], H=H, P=P, N=N, G=H,
                                   **kw)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)
    # heads of different groups must see different B/C (guards a clamped index)
    assert not np.allclose(y1[..., 0, :], y1[..., 3, :])


def test_z_gate_is_silu_product():
    prob = _tiny_problem(z=True, h0=True)
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"], h0=prob["h0"])
    y0, _ = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], **_dims(TINY), **kw)
    yz, _ = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], **_dims(TINY),
                                  z=prob["z"], **kw)
    zz = prob["z"].reshape(y0.shape)
    assert _relerr(yz, y0 * zz * 0.5 * (1.0 + np.tanh(0.5 * zz))) < 1e-13


# --------------------------------------------------------------------------
# conv

def test_conv_matches_numpy_correlate():
    rng = np.random.default_rng(5)
    B, S, C, W = 2, 9, 5, 4
    xbc = rng.normal(size=(B, S, C))
    w = rng.normal(size=(C, W))
    bias = rng.normal(size=C)
    st = rng.normal(size=(B, W - 1, C))
    out, st_out = oracle.conv1d(xbc, w, bias, st, apply_silu=False)
    for b in range(B):
        for c in range(C):
            u = np.concatenate([st[b, :, c], xbc[b, :, c]])
            ref = np.correlate(u, w[c], mode="valid") + bias[c]
            assert np.allclose(out[b, :, c], ref, rtol=1e-13, atol=1e-13)
    assert np.array_equal(st_out, xbc[:, -(W - 1):, :])
    out_s, _ = oracle.conv1d(xbc, w, bias, st, apply_silu=True)
    assert np.allclose(out_s, out / (1.0 + np.exp(-out)), rtol=1e-14, atol=1e-15)


def test_conv_impulse_returns_reversed_taps():
    W, C = 4, 3
    w = np.arange(1.0, 1.0 + C * W).reshape(C, W)
    xbc = np.zeros((1, 6, C))
    xbc[0, 1, :] = 1.0
    out, _ = oracle.conv1d(xbc, w, None, None, apply_silu=False)
    # the impulse at row 1 meets tap W-1 (newest) at row 1, tap 0 at row 1+W-1
    for c in range(C):
        assert np.array_equal(out[0, 1:1 + W, c], w[c, ::-1])
        assert out[0, 0, c] == 0.0 and out[0, 5, c] == 0.0


@pytest.mark.parametrize("split", [1, 2, 3, 5])
def test_conv_split_invariance(split):
    rng = np.random.default_rng(11)
    xbc = rng.normal(size=(2, 8, 6))
    w = rng.normal(size=(6, 4))
    st = rng.normal(size=(2, 3, 6))
    out, so = oracle.conv1d(xbc, w, None, st)
    o1, s1 = oracle.conv1d(xbc[:, :split], w, None, st)
    o2, s2 = oracle.conv1d(xbc[:, split:], w, None, s1)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), out)
    assert np.array_equal(s2, so)


def test_conv_state_short_call_keeps_old_rows():
    rng = np.random.default_rng(2)
    st = rng.normal(size=(1, 3, 2))
    xbc = rng.normal(size=(1, 1, 2))
    _, so = oracle.conv1d(xbc, rng.normal(size=(2, 4)), None, st)
    assert np.array_equal(so[0, :2], st[0, 1:]) and np.array_equal(so[0, 2], xbc[0, 0])


# --------------------------------------------------------------------------
# decode at slots == one row of the recurrence

def test_decode_steps_equal_sequential_rows():
    shape = TINY.with_(ngroups=2)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    prob = _tiny_problem(h0=True, z=True, shape=shape)
    pool = np.random.default_rng(1).normal(size=(5, H, P, N))
    slot = 3
    pool[slot] = prob["h0"][0]
    before = pool.copy()
    ys = []
    for t in range(shape.seqlen):
        y, pool, rc = oracle.decode_step(prob["xbc"][0, t:t + 1], prob["dt_raw"][0, t:t + 1],
                                         prob["A"], [slot], pool, H=H, P=P, N=N, G=G,
                                         dt_bias=prob["dt_bias"], D=prob["D"],
                                         z=prob["z"][0, t:t + 1])
        assert rc == 0
        ys.append(y[0])
    yseq, hseq = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], H=H, P=P, N=N,
                                       G=G, dt_bias=prob["dt_bias"], D=prob["D"],
                                       z=prob["z"], h0=prob["h0"])
    assert np.array_equal(np.stack(ys), yseq[0])
    assert np.array_equal(pool[slot], hseq[0])
    for s in (0, 1, 2, 4):
        assert np.array_equal(pool[s], before[s])


def test_decode_rejects_out_of_range_slot():
    shape = TINY
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    prob = _tiny_problem()
    pool = np.zeros((2, H, P, N))
    _, pool2, rc = oracle.decode_step(prob["xbc"][0, :2], prob["dt_raw"][0, :2], prob["A"],
                                      [1, 7], pool, H=H, P=P, N=N, G=G)
    assert rc == -1
    assert not np.array_equal(pool2[1], pool[1])  # the valid row still ran
    assert np.array_equal(pool2[0], pool[0])


# --------------------------------------------------------------------------
# group RMSNorm then SiLU gate (TensorSharp "nemotron.md" sections 3, 4.1, 6)

def _norm_inputs(rows=5, C=24, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((rows, C)), rng.standard_normal((rows, C)), \
        rng.uniform(0.5, 1.5, C)


def test_rmsnorm_constant_group_hand_value():
    """A group of equal values a: the norm gives a / sqrt(a^2 + eps); with
    a = 0.003 and eps = 0.000016, a^2 + eps = 0.000025 and the norm is 0.6."""
    from scipy.special import expit
    C, G = 8, 2
    y = np.concatenate([np.full(4, 0.003), np.full(4, -2.0)])[None, :]
    z = np.linspace(-1.5, 2.0, C)[None, :]
    w = np.linspace(0.5, 1.25, C)
    out = oracle.gated_group_rmsnorm(y, z, w, 0.000016, G)
    silu = z * expit(z)
    assert np.allclose(out[0, :4], 0.6 * silu[0, :4] * w[:4], rtol=1e-12, atol=0)
    # the second group: -2 / sqrt(4 + 0.000016) = -1 / sqrt(1 + 0.000004)
    assert np.allclose(out[0, 4:], -silu[0, 4:] * w[4:] / math.sqrt(1.000004), rtol=1e-12,
                       atol=0)


def test_rmsnorm_scale_invariance():
    """With eps = 0 the norm ignores the scale of y and is odd in y."""
    y, z, w = _norm_inputs()
    base = oracle.gated_group_rmsnorm(y, z, w, 0.0, 3)
    assert np.allclose(oracle.gated_group_rmsnorm(3.7 * y, z, w, 0.0, 3), base, rtol=1e-13)
    assert np.array_equal(oracle.gated_group_rmsnorm(-y, z, w, 0.0, 3), -base)


def test_rmsnorm_unit_rms_when_gate_is_one():
    """silu(50) = 50 to within 1e-20, so with w = 1/50 and eps = 0 every group
    of the output has root-mean-square 1."""
    y, _, _ = _norm_inputs(rows=4, C=32)
    out = oracle.gated_group_rmsnorm(y, np.full_like(y, 50.0), np.full(32, 1.0 / 50.0), 0.0, 4)
    rms = np.sqrt(np.mean(out.reshape(4, 4, 8) ** 2, axis=2))
    assert np.allclose(rms, 1.0, rtol=1e-13)


def test_rmsnorm_groups_are_independent():
    """Changing y in one group leaves every other group's output unchanged."""
    y, z, w = _norm_inputs()
    base = oracle.gated_group_rmsnorm(y, z, w, 1e-5, 3)
    y2 = y.copy()
    y2[:, 8:16] *= 5.0
    y2[:, 9] += 1.0
    out = oracle.gated_group_rmsnorm(y2, z, w, 1e-5, 3)
    assert np.array_equal(out[:, :8], base[:, :8]) and np.array_equal(out[:, 16:], base[:, 16:])
    assert not np.array_equal(out[:, 8:16], base[:, 8:16])


def test_rmsnorm_gate_acts_after_the_norm():
    """The norm is taken over y alone, so a change of z in one channel changes
    that channel's output only (and by the ratio of the two silu values)."""
    from scipy.special import expit
    y, z, w = _norm_inputs()
    base = oracle.gated_group_rmsnorm(y, z, w, 1e-5, 3)
    z2 = z.copy()
    z2[:, 5] = 2.5
    out = oracle.gated_group_rmsnorm(y, z2, w, 1e-5, 3)
    others = [c for c in range(24) if c != 5]
    assert np.array_equal(out[:, others], base[:, others])
    ratio = (2.5 * expit(2.5)) / (z[:, 5] * expit(z[:, 5]))
    assert np.allclose(out[:, 5], base[:, 5] * ratio, rtol=1e-12)


# --------------------------------------------------------------------------
# packed sequences with states at pool slots (vllm.cpp #1362 summary;
# TensorSharp "nemotron.md" section 11)

def _varlen_problem(lens, nslots=6, seed=0):
    shape = TINY.with_(batch=1, seqlen=sum(lens))
    p = si.params(shape, seed=seed)
    a = si.prefill_inputs(shape, seed=seed, act_dtype=__import__("torch").float32, with_z=True)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    rng = np.random.default_rng(seed)
    pools = (rng.standard_normal((nslots, H, P, N)) * 0.1,
             rng.standard_normal((nslots, shape.conv_width - 1, shape.cdim)))
    prm = {k: p[k].double().numpy() for k in ("conv_w", "conv_b", "dt_bias", "A", "D")}
    return shape, prm, a["xbc"][0].double().numpy(), a["dt_raw"][0].double().numpy(), \
        a["z"][0].double().numpy(), pools


def test_varlen_equals_one_call_per_sequence_and_leaves_other_slots():
    """Each packed sequence equals a call of its own from its slot's states; a
    fresh sequence (has_initial_state 0) equals a call from zero states; slots
    no sequence names are untouched."""
    lens, slots, init = [5, 1, 7], [4, 0, 2], [1, 0, 1]
    shape, prm, xbc, dt, z, (spool, cpool) = _varlen_problem(lens)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    cu = np.concatenate([[0], np.cumsum(lens)])
    y, sp, cp = oracle.mixer_prefill_varlen(
        xbc, prm["conv_w"], dt, prm["A"], cu, slots, spool, cpool, H=H, P=P, N=N, G=G,
        has_initial_state=init, conv_b=prm["conv_b"], dt_bias=prm["dt_bias"], D=prm["D"], z=z)
    for i, (r0, r1) in enumerate(zip(cu[:-1], cu[1:])):
        s = slots[i]
        yi, hi, ci = oracle.mixer_prefill(
            xbc[None, r0:r1], prm["conv_w"], dt[None, r0:r1], prm["A"], H=H, P=P, N=N, G=G,
            conv_b=prm["conv_b"], conv_state=cpool[s][None] if init[i] else None,
            dt_bias=prm["dt_bias"], D=prm["D"], z=z[None, r0:r1],
            h0=spool[s][None] if init[i] else None)
        assert np.array_equal(y[r0:r1], yi[0])
        assert np.array_equal(sp[s], hi[0]) and np.array_equal(cp[s], ci[0])
    for s in (1, 3, 5):
        assert np.array_equal(sp[s], spool[s]) and np.array_equal(cp[s], cpool[s])


def test_varlen_of_equal_lengths_equals_the_batched_call():
    """Equal lengths at slots 0..B-1 with initial states: the batched mixer."""
    lens = [4, 4, 4]
    shape, prm, xbc, dt, z, (spool, cpool) = _varlen_problem(lens, nslots=3, seed=2)
    H, P, N, G = shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    cu = np.array([0, 4, 8, 12])
    y, sp, cp = oracle.mixer_prefill_varlen(
        xbc, prm["conv_w"], dt, prm["A"], cu, [0, 1, 2], spool, cpool, H=H, P=P, N=N, G=G,
        conv_b=prm["conv_b"], dt_bias=prm["dt_bias"], D=prm["D"], z=z)
    yb, hb, cb = oracle.mixer_prefill(
        xbc.reshape(3, 4, -1), prm["conv_w"], dt.reshape(3, 4, -1), prm["A"], H=H, P=P, N=N,
        G=G, conv_b=prm["conv_b"], conv_state=cpool, dt_bias=prm["dt_bias"], D=prm["D"],
        z=z.reshape(3, 4, -1), h0=spool)
    assert np.array_equal(y.reshape(yb.shape), yb)
    assert np.array_equal(sp, hb) and np.array_equal(cp, cb)



# --------------------------------------------------------------------------
# sequence-parallel state passing: segments scanned from a zero state, then
# chained by the decay of each segment (TensorRT-Model-Connect #2207
# "Implementation": the chunk form's carry with a segment as the chunk)

def test_segment_decay_hand_values():
    # dt as given: gamma = (0.5 + 1.5) * -2 = -4 ; with softplus and bias 0:
    # softplus(0) = ln 2, softplus(ln 3) = ln 4 -> gamma = (ln 2 + ln 4) * -1 = -ln 8
    g = oracle.segment_decay(np.array([[[0.5], [1.5]]]), np.array([-2.0]), dt_softplus=False)
    assert g.shape == (1, 1) and g[0, 0] == -4.0
    g = oracle.segment_decay(np.array([[[0.0], [math.log(3.0)]]]), np.array([-1.0]),
                             dt_bias=np.array([0.0]))
    assert abs(g[0, 0] + math.log(8.0)) < 1e-15


def test_state_combine_hand_values():
    hp = np.arange(8, dtype=np.float64).reshape(1, 2, 2, 2)
    hs = np.ones((1, 2, 2, 2))
    out = oracle.state_combine(np.array([[0.0, -math.log(2.0)]]), hp, hs)
    assert np.array_equal(out[0, 0], hp[0, 0] + 1.0)
    assert np.allclose(out[0, 1], 0.5 * hp[0, 1] + 1.0, rtol=0, atol=1e-15)
    assert np.array_equal(oracle.state_combine(np.array([[-3.0, -1.0]]), None, hs), hs)


@pytest.mark.parametrize("cuts", [[5], [3, 8], [1, 2, 9]])
def test_segments_chained_by_combine_equal_one_call(cuts):
    """Split the 11 rows at ``cuts``; scan every segment from a zero state;
    chain: h <- state_combine(gamma_k, h, h_k) from h0.  The result is the
    final state of one row-by-row call over all rows, and rescanning each
    segment from the chained state gives that call's y."""
    prob = _tiny_problem(h0=True)
    kw = dict(dt_bias=prob["dt_bias"], D=prob["D"])
    y, hS = oracle.ssd_sequential(prob["xbc"], prob["dt_raw"], prob["A"], **_dims(TINY),
                                  h0=prob["h0"], **kw)
    edges = [0] + list(cuts) + [11]
    h = prob["h0"]
    ys = []
    for a, b in zip(edges[:-1], edges[1:]):
        xs, ds = prob["xbc"][:, a:b], prob["dt_raw"][:, a:b]
        _, h_k = oracle.ssd_sequential(xs, ds, prob["A"], **_dims(TINY), **kw)  # zero start
        g_k = oracle.segment_decay(ds, prob["A"], dt_bias=prob["dt_bias"])
        y_k, _ = oracle.ssd_sequential(xs, ds, prob["A"], **_dims(TINY), h0=h, **kw)
        ys.append(y_k)
        h = oracle.state_combine(g_k, h, h_k)
    assert _relerr(h, hS) < 1e-13
    assert _relerr(np.concatenate(ys, axis=1), y) < 1e-13
