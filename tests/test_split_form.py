"""The algebra behind the exact form's split column blocks, on the CPU.

The chunk form of TensorRT-Model-Connect #2207 ("Implementation") weights
the pair (t, s <= t) by exp(gamma_t - gamma_s) dt_s.  With gamma never rising
(every a <= 0), that factor splits at any row m between s and t, or with s
and t on either side of m inside one block, as exp(gamma_t - gamma_m) times
exp(gamma_m - gamma_s).  The tensor-core scan evaluates a 32-row block j of
columns that way, with m the block's middle row.  The column factor
V_s = exp(gamma_m - gamma_s) dt_s goes on the x rows, the row factor
R_t = exp(gamma_t - gamma_m) on the mask, and the skip term D R_t / dt_t on
the diagonal.  The split is taken when neither half of the block decays by
more than 2^60.  These tests check, in fp64, that this evaluation equals
the per-element definition at decays far past fp32's range.  They also check
that the split condition keeps every factor within 2^±60, and that an fp32
evaluation stays finite and close.  No GPU code is involved."""
import numpy as np
import pytest

Q, P, BLK = 128, 16, 32
SPLIT_MAX_LOG2 = 60.0


def _chunk(seed, scale):
    rng = np.random.default_rng(seed)
    dt = np.log1p(np.exp(rng.normal(-3.0, 1.0, Q))) * scale  # softplus, > 0
    A = -rng.uniform(1.0, 16.0)
    g = np.cumsum(dt * A)                                      # natural units, falling
    CB = rng.normal(0.0, 3.0, (Q, Q))
    x = rng.normal(0.0, 1.0, (Q, P))
    D = rng.normal(0.0, 1.0)
    return dt, g, CB, x, D


def _chunk_with_decay(seed, total_log2):
    """As _chunk, dt rescaled so that the chunk decays by 2^-total_log2."""
    dt, g, CB, x, D = _chunk(seed, 1.0)
    k = total_log2 / (-g[-1] / np.log(2.0))
    return dt * k, g * k, CB, x, D


def _per_element(dt, g, CB, x, D):
    """y_t = sum_{s<=t} CB[t,s] exp(min(g_t - g_s, 0)) dt_s x_s + D x_t."""
    dec = np.exp(np.minimum(g[:, None] - g[None, :], 0.0))
    M = np.tril(CB * dec * dt[None, :]) + np.diag(np.full(Q, D))
    return M @ x


def _split_blocks(dt, g, D):
    """Which 32-row column blocks split (both halves within 2^60, dt > 0,
    |D| < dt 2^60), as the scan decides it."""
    l2 = g / np.log(2.0)
    out = []
    for j in range(Q // BLK):
        f, m, e = l2[BLK * j], l2[BLK * j + 16], l2[BLK * j + BLK - 1]
        rows = slice(BLK * j, BLK * j + BLK)
        ok = (f - m <= SPLIT_MAX_LOG2 and m - e <= SPLIT_MAX_LOG2 and
              np.all(dt[rows] > 0) and np.all(abs(D) < dt[rows] * 2.0 ** 60))
        out.append(bool(ok))
    return out


def _split_form(dt, g, CB, x, D, dtype=np.float64):
    """M and x' per column block: split blocks carry V on x and R in the mask
    (D R_t / dt_t on the diagonal); the others keep the per-element factor."""
    split = _split_blocks(dt, g, D)
    M = np.zeros((Q, Q), dtype)
    xv = np.zeros((Q, P), dtype)
    t = np.arange(Q)
    for j in range(Q // BLK):
        cols = slice(BLK * j, BLK * j + BLK)
        s = np.arange(BLK * j, BLK * j + BLK)
        if split[j]:
            m = BLK * j + 16
            # per row, for the block's rows and the rows below it (the rows above
            # are masked out and never evaluated)
            R = np.exp(np.where(t >= BLK * j, g[t] - g[m], 0.0).astype(dtype))
            V = (np.exp((g[m] - g[s]).astype(dtype)) * dt[s]).astype(dtype)
            blk = (CB[:, cols].astype(dtype) * R[:, None]).astype(dtype)
            xv[cols] = (V[:, None] * x[cols]).astype(dtype)
            diag = (D * R[s] / dt[s]).astype(dtype)
        else:
            dec = np.exp(np.minimum(g[:, None] - g[None, s], 0.0)).astype(dtype)
            blk = (CB[:, cols] * dec * dt[None, s]).astype(dtype)
            xv[cols] = x[cols].astype(dtype)
            diag = np.full(BLK, D, dtype)
        blk = np.where(t[:, None] >= s[None, :], blk, 0.0).astype(dtype)
        blk[s, s - BLK * j] += diag
        M[:, cols] = blk
    return M @ xv, split


@pytest.mark.parametrize("scale", [0.05, 1.0, 6.0, 30.0])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_evaluation_equals_per_element_definition(scale, seed):
    dt, g, CB, x, D = _chunk(seed, scale)
    ref = _per_element(dt, g, CB, x, D)
    got, split = _split_form(dt, g, CB, x, D)
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err < 1e-12, (err, split)


def test_strong_decays_still_split_and_chunks_past_fp32_range_are_covered():
    """A chunk whose total decay is far past what exp(gamma_t) exp(-gamma_s)
    can hold in fp32 still splits most of its blocks."""
    dt, g, CB, x, D = _chunk_with_decay(3, 300.0)  # well beyond the factored form's 2^90
    got, split = _split_form(dt, g, CB, x, D)
    assert sum(split) >= 2
    ref = _per_element(dt, g, CB, x, D)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 1e-12


def test_split_factors_stay_within_2_pow_60():
    for seed in range(6):
        for scale in (0.5, 3.0, 10.0):
            dt, g, CB, x, D = _chunk(seed, scale)
            for j, ok in enumerate(_split_blocks(dt, g, D)):
                if not ok:
                    continue
                m = BLK * j + 16
                rows = np.arange(BLK * j, BLK * j + BLK)
                l2R = (g[rows] - g[m]) / np.log(2.0)      # the block's own rows
                l2V = (g[m] - g[rows]) / np.log(2.0)
                assert l2R.max() <= SPLIT_MAX_LOG2 + 1e-9 and l2V.max() <= SPLIT_MAX_LOG2 + 1e-9
                # rows below the block: R <= 1
                later = np.arange(BLK * j + BLK, Q)
                assert np.all(g[later] - g[m] <= 1e-12)


def test_fp32_split_evaluation_is_finite_and_close():
    """In fp32 (the kernel's mask and x-row precision before bf16) the split
    blocks give no inf or NaN at decays that overflow a whole-chunk factoring."""
    for seed in range(3):
        dt, g, CB, x, D = _chunk_with_decay(seed, 300.0)
        ref = _per_element(dt, g, CB, x, D)
        got, split = _split_form(dt, g, CB, x, D, dtype=np.float32)
        assert any(split)
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) < 1e-4


def test_rising_gamma_does_not_factor():
    """Where gamma rises the clamp at 0 breaks the identity, which is why the
    scan splits no block of such a chunk: min(a + b, 0) != min(a, 0) + min(b, 0)."""
    g = np.array([0.0, -5.0, 3.0])  # rises from row 1 to row 2
    t, m, s = 2, 1, 0
    whole = np.exp(min(g[t] - g[s], 0.0))
    parts = np.exp(min(g[t] - g[m], 0.0)) * np.exp(min(g[m] - g[s], 0.0))
    assert not np.isclose(whole, parts)
