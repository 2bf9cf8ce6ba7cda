"""Pins for the CPU oracle: every oracle function is checked against something
other than itself -- closed forms, invariants the pages state, library
routines (numpy / torch / scipy) on tiny inputs, and an independently written
vector form of the Sinkhorn-Knopp iteration.  A plausible slip anywhere in the
oracle (a dropped term, a wrong sign or index, a transposed operand, an extra
or missing round, a misplaced eps) fails at least one test here.

No GPU: these run with -m "not gpu".
"""
import math

import numpy as np
import pytest
import torch

import oracle
from hyper_connection_residual_mixes_gb300 import inputs

RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------- bf16 cast
def _torch_bf16_bits_from_f32(v32):
    t = torch.from_numpy(np.asarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch_on_fp32_values():
    # fp32-representable doubles: torch's fp32 -> bf16 (round to nearest even)
    # is a library reference with no double rounding on these inputs.
    v = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32),
        (RNG.standard_normal(5000) * 1e-3).astype(np.float32),
        (RNG.standard_normal(5000) * 1e30).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-39).astype(np.float32),   # fp32 subnormals
        np.array([3.38e38, -3.38e38, 3.3961e38, 1.1754944e-38, 0.0, -0.0], np.float32),
    ])
    got = oracle.bf16_from_f64(v.astype(np.float64))
    want = _torch_bf16_bits_from_f32(v)
    assert np.array_equal(got, want)


def test_bf16_round_ties_to_even_and_specials():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2.0 ** -8: 0x3F80,             # tie -> even (1.0)
        one + 3 * 2.0 ** -8: 0x3F82,         # tie -> even (1 + 2^-6)
        one + 2.0 ** -8 + 2.0 ** -40: 0x3F81,  # just above the tie (not fp32-representable)
        one + 2.0 ** -8 - 2.0 ** -40: 0x3F80,  # just below the tie
        -2.5: 0xC020,
        float("inf"): 0x7F80,
        -float("inf"): 0xFF80,
        1e39: 0x7F80,                         # overflows bf16
        2.0 ** -133: 0x0001,                  # smallest bf16 subnormal
        2.0 ** -134: 0x0000,                  # tie between 0 and the smallest subnormal -> 0 (even)
        3 * 2.0 ** -134: 0x0002,              # tie between 1 and 2 subnormal units -> 2 (even)
        -0.0: 0x8000,
    }
    for v, bits in cases.items():
        assert int(oracle.bf16_from_f64(np.array([v]))[0]) == bits, (v, hex(bits))
    assert (int(oracle.bf16_from_f64(np.array([float("nan")]))[0]) & 0x7FFF) > 0x7F80


def test_bf16_to_f64_is_exact():
    bits = RNG.integers(0, 1 << 16, size=50000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite values only
    got = oracle.bf16_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want)


# ------------------------------------------------------------- a1: mixes
def _rand_x(n, hc, d, scale=1.0):
    return inputs.bf16_bits_np((torch.from_numpy(RNG.standard_normal((n, hc, d))) * scale)
                               .to(torch.bfloat16))


def test_mixes_matches_numpy_gemv_tiny():
    n, hc, d = 5, 4, 24
    x = _rand_x(n, hc, d)
    w = (RNG.standard_normal(((2 + hc) * hc, hc * d)) * 0.1).astype(np.float32)
    got = oracle.mixes(x, w, norm_eps=1e-20)
    xf = oracle.bf16_to_f64(x).reshape(n, hc * d)
    r = 1.0 / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + 1e-20)
    want = (xf @ w.astype(np.float64).T) * r
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("hc", [1, 2, 3, 4])
def test_mixes_generic_hc_matches_numpy(hc):
    n, d = 3, 16
    x = _rand_x(n, hc, d)
    w = (RNG.standard_normal(((2 + hc) * hc, hc * d)) * 0.1).astype(np.float32)
    got = oracle.mixes(x, w, norm_eps=1e-6)
    xf = oracle.bf16_to_f64(x).reshape(n, hc * d)
    want = (xf @ w.astype(np.float64).T) / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


def test_mixes_power_of_two_scale_invariance_bitwise():
    n, hc, d = 4, 4, 64
    x = _rand_x(n, hc, d)
    w = (RNG.standard_normal((24, hc * d)) * 0.01).astype(np.float32)
    base = oracle.mixes(x, w)
    for k in (-3, 1, 5):
        xs = oracle.bf16_from_f64(oracle.bf16_to_f64(x) * 2.0 ** k).reshape(x.shape)
        assert np.array_equal(oracle.mixes(xs, w), base)


def test_mixes_zero_input_is_exactly_zero():
    x = np.zeros((3, 4, 32), np.uint16)
    w = (RNG.standard_normal((24, 128))).astype(np.float32)
    assert np.array_equal(oracle.mixes(x, w, 1e-20), np.zeros((3, 24)))


def test_mixes_statistic_uses_all_streams():
    # one statistic per token over all hc*d values: a stream of zeros still
    # counts in the mean (a per-stream norm would give a different value).
    hc, d = 4, 8
    x = np.zeros((1, hc, d), np.uint16)
    x[0, 0, :] = 0x3F80  # stream 0 all ones, others zero
    w = np.zeros((24, hc * d), np.float32)
    w[0, 0] = 1.0
    m = oracle.mixes(x, w, norm_eps=0.0)
    # mean(x^2) over 32 values = 8/32 = 1/4 -> r = 2; m0 = 1 * r
    assert m[0, 0] == 2.0


# --------------------------------------------- a2 + a3: split + Sinkhorn
def _vector_form_sinkhorn(logits, iters, eps):
    """Independent restatement: the row softmax + eps gives K0; every later
    step only rescales rows (u) or columns (v), so P = diag(u) K0 diag(v).
    Rows use sums of P along axis 1, columns along axis 0, each divided by
    (sum + eps).  Written as matrix-vector products on the fixed K0."""
    z = logits - logits.max(axis=1, keepdims=True)
    e = np.exp(z)
    K0 = e / e.sum(axis=1, keepdims=True) + eps
    hc = K0.shape[0]
    u = np.ones(hc)
    v = np.ones(hc)
    steps = ["col"] + ["row", "col"] * (iters - 1)
    for s in steps:
        if s == "row":
            rs = u * (K0 @ v)
            u = u / (rs + eps)
        else:
            cs = v * (K0.T @ u)
            v = v / (cs + eps)
    return u[:, None] * K0 * v[None, :]


@pytest.mark.parametrize("hc", [2, 3, 4])
@pytest.mark.parametrize("iters", [1, 2, 3, 20, 57])
@pytest.mark.parametrize("eps", [1e-6, 0.0, 0.05])
def test_sinkhorn_matches_vector_form(hc, iters, eps):
    mix = (2 + hc) * hc
    n = 6
    m = RNG.standard_normal((n, mix)) * 3.0
    scale = np.array([0.7, 1.3, 1.9], np.float32)
    base = RNG.standard_normal(mix).astype(np.float32)
    pre, post, comb = oracle.split_sinkhorn(m, scale, base, hc=hc, iters=iters, eps=eps)
    for t in range(n):
        logits = (m[t, 2 * hc:] * float(scale[2]) + base[2 * hc:].astype(np.float64)).reshape(hc, hc)
        want = _vector_form_sinkhorn(logits, iters, eps)
        np.testing.assert_allclose(comb[t], want, rtol=1e-12, atol=1e-15)


def test_split_pre_post_closed_forms():
    from scipy.special import expit  # library logistic function
    hc, n = 4, 50
    m = RNG.standard_normal((n, 24)) * 3.0
    scale = np.array([0.6, 1.7, 1.1], np.float32)
    base = RNG.standard_normal(24).astype(np.float32)
    pre, post, _ = oracle.split_sinkhorn(m, scale, base, hc=hc, iters=20, eps=1e-6)
    sc = scale.astype(np.float64)
    b = base.astype(np.float64)
    np.testing.assert_allclose(pre, expit(m[:, :4] * sc[0] + b[:4]) + 1e-6, rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(post, 2.0 * expit(m[:, 4:8] * sc[1] + b[4:8]), rtol=1e-14, atol=1e-16)


def test_split_reads_comb_row_major_from_offset_2hc():
    # comb[j][k] = m[2hc + j*hc + k]: put a single large logit at one index.
    # iters=1, eps=0: after the softmax row j is (almost exactly) the unit
    # vector e_k and the other rows are uniform 1/4, so column k sums to 7/4
    # and the entry becomes 4/7; the other columns sum to 3/4 and their
    # uniform-row entries become 1/3.
    hc = 4
    for j, k in [(0, 3), (2, 1), (3, 0)]:
        m = np.zeros((1, 24))
        m[0, 2 * hc + j * hc + k] = 50.0
        _, _, comb = oracle.split_sinkhorn(m, np.ones(3, np.float32), np.zeros(24, np.float32),
                                           hc=hc, iters=1, eps=0.0)
        assert abs(comb[0, j, k] - 4.0 / 7.0) < 1e-12
        other_row = (j + 1) % hc
        assert abs(comb[0, other_row, k] - 1.0 / 7.0) < 1e-12
        assert abs(comb[0, other_row, (k + 1) % hc] - 1.0 / 3.0) < 1e-12
        assert comb[0, j, (k + 1) % hc] < 1e-20


def test_sinkhorn_uniform_logits_scalar_recursion():
    # all 16 logits equal: the softmax gives 1/4, + eps; every later
    # normalisation maps a constant matrix c to c / (4c + eps).
    eps = 1e-6
    for iters in (1, 2, 20):
        m = np.zeros((1, 24))
        _, _, comb = oracle.split_sinkhorn(m, np.ones(3, np.float32), np.zeros(24, np.float32),
                                           hc=4, iters=iters, eps=eps)
        c = 0.25 + eps
        for _ in range(1 + 2 * (iters - 1)):
            c = c / (4.0 * c + eps)
        assert np.all(comb[0] == comb[0, 0, 0])
        assert abs(comb[0, 0, 0] - c) < 1e-15
    # the fixed point of c -> c / (4c + eps) is (1 - eps) / 4
    assert abs(comb[0, 0, 0] - (1 - eps) / 4) < 1e-15


def test_sinkhorn_2x2_limit_closed_form():
    # eps = 0: scaling preserves the cross ratio P00 P11 / (P01 P10) = exp(delta),
    # delta = c00 + c11 - c01 - c10; the doubly stochastic 2x2 limit is
    # [[p, 1-p], [1-p, p]] with p / (1 - p) = exp(delta / 2).
    # The limit is reached within the 400 rounds only for moderate logits (std 1:
    # worst error 2e-16 over 300 draws; std 2 leaves up to 1e-4), and the pin uses
    # its own stream so that it does not depend on which tests ran before it.
    hc = 2
    rng = np.random.default_rng(218)
    for _ in range(10):
        m = rng.standard_normal((1, 8)) * 1.0
        _, _, comb = oracle.split_sinkhorn(m, np.ones(3, np.float32), np.zeros(8, np.float32),
                                           hc=hc, iters=400, eps=0.0)
        c = m[0, 4:].reshape(2, 2)
        delta = c[0, 0] + c[1, 1] - c[0, 1] - c[1, 0]
        p = 1.0 / (1.0 + math.exp(-delta / 2.0))
        np.testing.assert_allclose(comb[0], [[p, 1 - p], [1 - p, p]], rtol=0, atol=1e-12)


@pytest.mark.parametrize("iters", [1, 2, 7, 20])
def test_sinkhorn_cross_ratios_preserved_eps0(iters):
    # with eps = 0 every step is a diagonal scaling, so every cross ratio
    # P[i,j] P[k,l] / (P[i,l] P[k,j]) equals exp(c[i,j] + c[k,l] - c[i,l] - c[k,j]).
    m = RNG.standard_normal((1, 24)) * 2.0
    _, _, comb = oracle.split_sinkhorn(m, np.ones(3, np.float32), np.zeros(24, np.float32),
                                       hc=4, iters=iters, eps=0.0)
    P = comb[0]
    c = m[0, 8:].reshape(4, 4)
    for (i, k) in [(0, 1), (1, 3), (2, 0)]:
        for (j, l) in [(0, 2), (3, 1)]:
            got = P[i, j] * P[k, l] / (P[i, l] * P[k, j])
            want = math.exp(c[i, j] + c[k, l] - c[i, l] - c[k, j])
            assert abs(got / want - 1) < 1e-11


def test_page_invariants_on_tiny_like_data(golden_constants):
    # columns sum to 1 within 1e-5 after the final column step; all entries
    # positive; pre > eps; 0 < post < 2 (strict, fp64 oracle).
    case = inputs.tiny(seed=0, n=16, d=256)
    p = case.params[0]
    m = oracle.mixes(inputs.bf16_bits_np(case.x), p.hc_fn.numpy())
    eps = golden_constants["hc_eps"]
    pre, post, comb = oracle.split_sinkhorn(m, p.hc_scale.numpy(), p.hc_base.numpy(),
                                            hc=golden_constants["hc_mult"],
                                            iters=golden_constants["hc_sinkhorn_iters"], eps=eps)
    colsum = comb.sum(axis=1)
    assert np.max(np.abs(colsum - 1)) <= golden_constants["comb_col_sum_tolerance_after_final_column_step"]
    assert np.all(comb > 0)
    assert np.all(pre > eps)
    assert np.all((post > 0) & (post < 2))


def test_rows_sum_to_one_on_convergent_fixture(golden_constants):
    # logits of std <= 0.5: 20 rounds converge, rows sum to 1 within 1e-3.
    n = 2000
    m = RNG.standard_normal((n, 24)) * 0.5
    pre, post, comb = oracle.split_sinkhorn(m, np.ones(3, np.float32), np.zeros(24, np.float32),
                                            hc=4, iters=20, eps=1e-6)
    rows = comb.sum(axis=2)
    assert np.max(np.abs(rows - 1)) <= golden_constants["comb_row_sum_tolerance_convergent"]
    assert np.max(np.abs(comb.sum(axis=1) - 1)) <= 1e-5


def test_rows_need_not_converge_on_wide_logits():
    # documents the reading: on N(0,3) logits, 20 rounds leave some rows off by
    # more than 1e-3 even in fp64 (so that check is scoped to convergent data).
    m = RNG.standard_normal((4000, 24)) * 3.0
    _, _, comb = oracle.split_sinkhorn(m, np.array([1.5, 1.5, 1.5], np.float32),
                                       np.zeros(24, np.float32), hc=4, iters=20, eps=1e-6)
    rows = comb.sum(axis=2)
    assert np.max(np.abs(rows - 1)) > 1e-3
    assert np.max(np.abs(comb.sum(axis=1) - 1)) <= 1e-5


# -------------------------------------------------------------- a4: pre
def test_pre_matches_numpy_then_round():
    n, hc, d = 7, 4, 40
    x = _rand_x(n, hc, d)
    pm = RNG.uniform(0.1, 1.0, (n, hc))
    got = oracle.pre(x, pm)
    xf = oracle.bf16_to_f64(x)
    want = oracle.bf16_from_f64(np.einsum("ts,tsd->td", pm, xf))
    # einsum may sum in another order: allow a 1-ulp tie flip, never more
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1 and np.mean(diff) < 1e-3


def test_pre_identical_streams_closed_form():
    n, hc, d = 3, 4, 32
    v = _rand_x(n, 1, d)
    x = np.repeat(v, hc, axis=1)
    pm = np.array([[0.5, 0.25, 0.125, 0.0625]] * n)  # dyadic: exact sums
    got = oracle.pre(x, pm)
    want = oracle.bf16_from_f64(oracle.bf16_to_f64(v[:, 0, :]) * 0.9375)
    assert np.array_equal(got, want)


# ---------------------------------------------------------- a5: RMSNorm
def test_rmsnorm_matches_torch_rms_norm():
    n, d = 6, 64
    h = _rand_x(n, 1, d)[:, 0, :]
    w = RNG.uniform(0.5, 1.5, d).astype(np.float32)
    got = oracle.rmsnorm(h, w, eps=1e-20)
    hf = torch.from_numpy(oracle.bf16_to_f64(h))
    ref = torch.nn.functional.rms_norm(hf, (d,), weight=torch.from_numpy(w.astype(np.float64)),
                                       eps=1e-20).numpy()
    want = oracle.bf16_from_f64(ref)
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1 and np.mean(diff) < 1e-2


def test_rmsnorm_scale_invariance_and_constant_vector():
    n, d = 4, 128
    h = _rand_x(n, 1, d)[:, 0, :]
    w = RNG.uniform(0.5, 1.5, d).astype(np.float32)
    base = oracle.rmsnorm(h, w)
    for k in (-4, 3):
        hs = oracle.bf16_from_f64(oracle.bf16_to_f64(h) * 2.0 ** k)
        assert np.array_equal(oracle.rmsnorm(hs, w), base)
    # a constant vector normalises to +-1, so the output is the rounded gain
    c = oracle.bf16_from_f64(np.full((1, d), -3.0))
    assert np.array_equal(oracle.rmsnorm(c, w), oracle.bf16_from_f64(-w.astype(np.float64))[None])


def test_rmsnorm_eps_matters_only_near_zero():
    d = 16
    z = np.zeros((1, d), np.uint16)
    w = np.ones(d, np.float32)
    assert np.array_equal(oracle.rmsnorm(z, w, 1e-20), np.zeros((1, d), np.uint16))


# ------------------------------------------------------------- a6: post
def test_post_matches_numpy_einsum():
    n, hc, d = 5, 4, 48
    r = _rand_x(n, hc, d)
    f = _rand_x(n, 1, d)[:, 0, :]
    post = RNG.uniform(0, 2, (n, hc))
    comb = RNG.uniform(0, 1, (n, hc, hc))
    got = oracle.post(f, r, post, comb)
    rf = oracle.bf16_to_f64(r)
    ff = oracle.bf16_to_f64(f)
    ref = post[:, :, None] * ff[:, None, :] + np.einsum("tjk,tjd->tkd", comb, rf)
    want = oracle.bf16_from_f64(ref)
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1 and np.mean(diff) < 1e-3


def test_post_column_k_feeds_output_k():
    # comb = permutation matrix (j -> k) with post = 0 routes stream j to output k
    n, hc, d = 1, 4, 16
    r = _rand_x(n, hc, d)
    f = _rand_x(n, 1, d)[:, 0, :]
    perm = [2, 0, 3, 1]  # input j goes to output perm[j]
    comb = np.zeros((1, 4, 4))
    for j, k in enumerate(perm):
        comb[0, j, k] = 1.0
    y = oracle.post(f, r, np.zeros((1, 4)), comb)
    for j, k in enumerate(perm):
        assert np.array_equal(y[0, k], r[0, j])


def test_post_identical_streams_and_stream_sum():
    n, hc, d = 2, 4, 32
    v = _rand_x(n, 1, d)
    r = np.repeat(v, hc, axis=1)
    f = _rand_x(n, 1, d)[:, 0, :]
    post = np.array([[0.5, 1.0, 1.5, 0.25]] * n)
    comb = np.full((n, hc, hc), 0.25)  # column sums exactly 1
    y = oracle.post(f, r, post, comb)
    want = oracle.bf16_from_f64(post[:, :, None] * oracle.bf16_to_f64(f)[:, None, :]
                                + oracle.bf16_to_f64(v))
    assert np.array_equal(y, want)


# -------------------------------------------------- a7: the side step / block
def test_block_step_stream_permutation_equivariance():
    # relabel the streams by a permutation pi consistently (x streams,
    # hc_fn column blocks, pre/post base entries, comb rows and columns,
    # pre_mix): pre/post/comb/y are relabelled, h_norm is unchanged.
    hc, d, n = 4, 32, 3
    case = inputs.tiny(seed=5, n=n, d=d)
    p = case.params[0]
    x = inputs.bf16_bits_np(case.x)
    f = inputs.bf16_bits_np(case.fs[0])
    pm = case.pre_mix.numpy().astype(np.float64)
    W = p.hc_fn.numpy()
    base = p.hc_base.numpy()
    out = oracle.block_step(x, pm, f, W, p.hc_scale.numpy(), base, p.norm_w.numpy())
    pi = np.array([2, 0, 3, 1])
    xp = x[:, pi, :]
    pmp = pm[:, pi]
    Wb = W.reshape(24, hc, d)[:, pi, :]
    rows = np.concatenate([pi, 4 + pi, (8 + (pi[:, None] * 4 + pi[None, :])).reshape(-1)])
    Wp = Wb[rows].reshape(24, hc * d)
    bp = base[rows]
    o2 = oracle.block_step(xp, pmp, f, Wp, p.hc_scale.numpy(), bp, p.norm_w.numpy())
    np.testing.assert_allclose(o2["pre"], out["pre"][:, pi], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o2["post"], out["post"][:, pi], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o2["comb"], out["comb"][:, pi][:, :, pi], rtol=1e-10, atol=1e-14)
    assert np.abs(o2["y"].astype(np.int32) - out["y"][:, pi].astype(np.int32)).max() <= 1
    assert np.abs(o2["h_norm"].astype(np.int32) - out["h_norm"].astype(np.int32)).max() <= 1


def test_block_layer_wiring():
    # the FFN side reads with the attention side's pre and consumes its y
    hc, d, n = 4, 16, 2
    case = inputs.decode(seed=1, n=n, d=d)
    pa, pf = (p.astuple() for p in case.params)
    pa = tuple(t.numpy() for t in pa)
    pf = tuple(t.numpy() for t in pf)
    x = inputs.bf16_bits_np(case.x)
    fa, ff = (inputs.bf16_bits_np(f) for f in case.fs)
    pm = case.pre_mix.numpy().astype(np.float64)
    a, b = oracle.block_layer(x, pm, fa, ff, pa, pf)
    a2 = oracle.block_step(x, pm, fa, *pa)
    b2 = oracle.block_step(a2["y"], a2["pre"], ff, *pf)
    assert np.array_equal(b["y"], b2["y"]) and np.array_equal(b["h_norm"], b2["h_norm"])
    # the FFN side's h_norm depends on the attention side's pre, not its own
    h_expected = oracle.rmsnorm(oracle.pre(a["y"], a["pre"]), pf[3])
    assert np.array_equal(b["h_norm"], h_expected)


def test_param_counts_match_pages(golden_constants):
    g = golden_constants
    p = inputs.side_params(torch.Generator().manual_seed(0), hc=g["hc_mult"], d=g["dim"])
    n_params = p.hc_fn.numel() + p.hc_base.numel() + p.hc_scale.numel()
    assert n_params == g["stream_weights_params_per_sublayer"] == 491547
    assert p.norm_w.numel() == g["rmsnorm_params"]
    hc = g["hc_mult"]
    assert hc * hc + 1 == g["comb_params_per_instance"]
    assert (2 + hc) * hc == g["comb_in_out_shapes"]["in_mix_numbers"]


# ---------------------------------------------------------------- MXFP8 cast
# DeepSeek V4.1 Flash diagram, block "Cast to MXFP8": groups of 32 channels,
# UE8M0 scale = the group's largest magnitude (at least 1e-4) over 448 rounded
# up to a power of two, E4M3 elements of x / scale kept within [-448, 448].

def _torch_e4m3_bits(v32):
    t = torch.from_numpy(np.asarray(v32, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _all_e4m3_values():
    codes = np.arange(0, 0x7F, dtype=np.uint8)   # 0x7F is NaN
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_e4m3_round_matches_torch():
    # torch's fp32 -> float8_e4m3fn conversion rounds to nearest, ties to even:
    # a library reference.  Values: log-uniform magnitudes across the normal and
    # subnormal range, every representable value, and every midpoint (ties).
    rng = np.random.default_rng(4321)   # its own stream: the shared one feeds other pins
    mags = np.exp2(rng.uniform(-12.0, math.log2(448.0), 6000))
    vals = _all_e4m3_values()
    mids = (vals[1:] + vals[:-1]) / 2.0
    v = np.concatenate([mags, -mags, vals, -vals, mids, -mids, [448.0, -448.0, 0.0, -0.0]])
    v = v.astype(np.float32).astype(np.float64)     # fp32 inputs, as the cast sees them
    assert np.array_equal(oracle.e4m3_from_f64(v), _torch_e4m3_bits(v))


@pytest.mark.parametrize("value, code", [
    (448.0, 0x7E), (-448.0, 0xFE), (1.0, 0x38), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01),
    (0.75 * 2.0 ** -9, 0x01), (0.5 * 2.0 ** -9, 0x00), (1.5 * 2.0 ** -9, 0x02),
    (2.5 * 2.0 ** -9, 0x02), (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80), (240.0, 0x77),
])
def test_e4m3_hand_values(value, code):
    # field 0: m * 2^-9; field e > 0: (1 + m/8) * 2^(e-7); ties go to the even mantissa
    assert int(oracle.e4m3_from_f64(np.array([value]))[0]) == code


def _bits(v):
    return _torch_bf16_bits_from_f32(np.asarray(v, dtype=np.float32)).reshape(1, -1)


def test_mxfp8_scale_closed_forms():
    g = np.zeros(32)
    g[5] = 448.0          # 448 / 448 = 1 = 2^0
    codes, sc = oracle.mxfp8(_bits(g))
    assert sc[0, 0] == 127 and codes[0, 5] == 0x7E and not codes[0, np.arange(32) != 5].any()
    g[5] = 449.0 - 1.0    # 448 again (bf16 of 448 exactly)
    g[7] = -452.0         # 452/448 > 1 -> 2^1; -452/2 = -226 -> nearest E4M3 -224
    codes, sc = oracle.mxfp8(_bits(g))
    assert sc[0, 0] == 128 and codes[0, 7] == 0xF6 and codes[0, 5] == 0x76  # 448/2 = 224 = 1.75 * 2^7
    g = np.zeros(32)
    g[0] = 224.0          # 224/448 = 0.5 exactly -> 2^-1, and 224 / 0.5 = 448
    codes, sc = oracle.mxfp8(_bits(g))
    assert sc[0, 0] == 126 and codes[0, 0] == 0x7E
    # all zeros: the largest magnitude is kept at 1e-4; fp32(1e-4)/448 = 2.23e-7
    # lies in (2^-23, 2^-22], so the scale is 2^-22 (byte 105); -0 keeps its sign
    z = np.zeros(32)
    z[3] = -0.0
    codes, sc = oracle.mxfp8(_bits(z))
    assert sc[0, 0] == 127 - 22 and codes[0, 3] == 0x80 and not (codes[0] & 0x7F).any()
    # a tiny group is scaled by the same 2^-22: 1e-5 * 2^22 = 41.9 -> E4M3 40 (0x64)
    t = np.zeros(32)
    t[1] = 1e-5
    codes, sc = oracle.mxfp8(_bits(t))
    assert sc[0, 0] == 105 and codes[0, 1] == _torch_e4m3_bits(
        [float(inputs_bf16_value(1e-5)) * 2.0 ** 22])[0]


def inputs_bf16_value(v):
    return oracle.bf16_to_f64(_torch_bf16_bits_from_f32(np.array([v], np.float32)))[0]


def _decode(codes, scales):
    vals = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).float().numpy()
    return vals.astype(np.float64) * np.exp2(np.repeat(scales.astype(np.float64) - 127.0, 32, axis=1))


def test_mxfp8_round_trip_bound_and_minimal_scale():
    g = torch.Generator().manual_seed(7)
    x = inputs.streams(g, 24, 1, 256, outlier_p=0.02).reshape(24, 256)
    x[3, :32] = 0                                              # an all-zero group
    x[4, 32:64] *= 1e-6                                        # a group below the 1e-4 floor
    bits = oracle.bf16_bits(x)
    codes, scales = oracle.mxfp8(bits)
    xv = oracle.bf16_to_f64(bits)
    back = _decode(codes, scales)
    scale = np.exp2(np.repeat(scales.astype(np.float64) - 127.0, 32, axis=1))
    q = np.abs(xv) / scale
    # half an E4M3 step at q's binade (normal: 2^(e-3); subnormal: 2^-9), scaled back
    e = np.floor(np.log2(np.maximum(q, 2.0 ** -6)))
    half_step = np.exp2(e - 4.0) * scale
    assert np.all(np.abs(back - xv) <= half_step * (1 + 1e-12))
    # the scale is the smallest power of two with every |x| / scale <= 448
    amax = np.maximum(np.abs(xv).reshape(24, -1, 32).max(-1), np.float32(1e-4))
    s = np.exp2(scales.astype(np.float64) - 127.0)
    assert np.all(amax / s <= 448.0) and np.all(amax / (s / 2) > 448.0 * (1 - 2.0 ** -23))


def test_mxfp8_power_of_two_invariance():
    # scaling a row by 2^k leaves every code unchanged and moves every scale by k
    # (groups well above the 1e-4 floor)
    g = torch.Generator().manual_seed(9)
    x = inputs.streams(g, 8, 1, 128).reshape(8, 128)
    c0, s0 = oracle.mxfp8(oracle.bf16_bits(x))
    for k in (-5, -1, 3, 7):
        ck, sk = oracle.mxfp8(oracle.bf16_bits(x * 2.0 ** k))
        assert np.array_equal(ck, c0) and np.array_equal(sk.astype(int), s0.astype(int) + k)


def test_mxfp8_every_e4m3_value_round_trips():
    # a group holding exactly v * 2^ex for every representable v reproduces v's code
    vals = _all_e4m3_values()
    codes_all = np.arange(0, 0x7F, dtype=np.uint8)
    for ex in (-3, 0, 5):
        for start in range(0, len(vals), 31):
            v = vals[start:start + 31]
            grp = np.zeros(32)
            grp[:len(v)] = v * 2.0 ** ex
            grp[31] = 448.0 * 2.0 ** ex                 # pins the scale to 2^ex
            codes, sc = oracle.mxfp8(_bits(grp))
            assert sc[0, 0] == 127 + ex
            assert np.array_equal(codes[0, :len(v)], codes_all[start:start + 31])


# ------------------------------------------------ other stream counts (hc = 8)
# The oracle is written for any hc; these pins repeat the library and
# independent-restatement checks at hc = 8 (mix = 80), each on its own random
# stream.

def test_hc8_mixes_matches_numpy():
    rng = np.random.default_rng(801)
    n, hc, d = 3, 8, 16
    x = inputs.bf16_bits_np(torch.from_numpy(rng.standard_normal((n, hc, d))).to(torch.bfloat16))
    w = (rng.standard_normal(((2 + hc) * hc, hc * d)) * 0.1).astype(np.float32)
    got = oracle.mixes(x, w, norm_eps=1e-6)
    xf = oracle.bf16_to_f64(x).reshape(n, hc * d)
    want = (xf @ w.astype(np.float64).T) / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("iters", [1, 2, 20])
@pytest.mark.parametrize("eps", [1e-6, 0.0])
def test_hc8_sinkhorn_matches_vector_form(iters, eps):
    rng = np.random.default_rng(802 + iters)
    hc = 8
    mix = (2 + hc) * hc
    m = rng.standard_normal((4, mix)) * 2.0
    scale = np.array([0.7, 1.3, 0.9], np.float32)
    base = rng.standard_normal(mix).astype(np.float32)
    from scipy.special import expit
    pre, post, comb = oracle.split_sinkhorn(m, scale, base, hc=hc, iters=iters, eps=eps)
    for t in range(4):
        logits = (m[t, 2 * hc:] * float(scale[2]) + base[2 * hc:].astype(np.float64)).reshape(hc, hc)
        np.testing.assert_allclose(comb[t], _vector_form_sinkhorn(logits, iters, eps), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(pre, expit(m[:, :hc] * float(scale[0]) + base[:hc]) + eps, rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(post, 2.0 * expit(m[:, hc:2 * hc] * float(scale[1]) + base[hc:2 * hc]),
                               rtol=1e-14, atol=1e-16)


def test_hc8_pre_and_post_match_numpy():
    rng = np.random.default_rng(803)
    n, hc, d = 5, 8, 40
    x = inputs.bf16_bits_np(torch.from_numpy(rng.standard_normal((n, hc, d))).to(torch.bfloat16))
    pm = rng.uniform(0.1, 1.0, (n, hc))
    got = oracle.pre(x, pm)
    xf = oracle.bf16_to_f64(x)
    want = oracle.bf16_from_f64(np.einsum("ts,tsd->td", pm, xf))
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1 and np.mean(diff) < 1e-3
    f = inputs.bf16_bits_np(torch.from_numpy(rng.standard_normal((n, d))).to(torch.bfloat16))
    post = rng.uniform(0, 2, (n, hc))
    comb = rng.uniform(0, 1, (n, hc, hc))
    got = oracle.post(f, x, post, comb)
    ref = post[:, :, None] * oracle.bf16_to_f64(f)[:, None, :] + np.einsum("tjk,tjd->tkd", comb, xf)
    diff = np.abs(got.astype(np.int32) - oracle.bf16_from_f64(ref).astype(np.int32))
    assert diff.max() <= 1 and np.mean(diff) < 1e-3


# --------------------------------------------------- f3: the side step backward
# The pages give no backward; the oracle's is the derivative of a1-a6.  Pinned
# by central finite differences of the (separately pinned) forward, with the
# bf16 casts switched off so that the forward is smooth.

def test_side_f64_with_casts_equals_block_step():
    case = inputs.tiny(n=3, d=64, seed=31)
    p = case.params[0]
    xb, fb = oracle.bf16_bits(case.x), oracle.bf16_bits(case.fs[0])
    pm = case.pre_mix.numpy().astype(np.float64)
    ref = oracle.block_step(xb, pm, fb, *(t.numpy() for t in p.astuple()))
    got = oracle.side_f64(oracle.bf16_to_f64(xb), pm, oracle.bf16_to_f64(fb),
                          *(t.numpy().astype(np.float64) for t in p.astuple()), rounded=True)
    assert np.array_equal(got["h_norm"], oracle.bf16_to_f64(ref["h_norm"]))
    assert np.array_equal(got["y"], oracle.bf16_to_f64(ref["y"]))
    for k in ("pre", "post", "comb"):
        assert np.array_equal(got[k], ref[k])


def _bwd_case(rng, n, hc, d):
    mix = (2 + hc) * hc
    return dict(x=rng.standard_normal((n, hc, d)), pre_mix=rng.uniform(0.1, 1.0, (n, hc)),
                f=rng.standard_normal((n, d)), hc_fn=rng.standard_normal((mix, hc * d)) * 0.3,
                hc_scale=rng.uniform(0.5, 2.0, 3), hc_base=rng.standard_normal(mix),
                norm_w=rng.uniform(0.5, 1.5, d))


@pytest.mark.parametrize("hc", [2, 4, 8])
@pytest.mark.parametrize("iters,eps", [(1, 1e-6), (3, 0.05), (20, 1e-6)])
def test_side_backward_matches_finite_differences(hc, iters, eps):
    rng = np.random.default_rng(1000 + 10 * hc + iters)
    n, d = 2, 8
    inp = _bwd_case(rng, n, hc, d)
    g_hn, g_y, g_pre = rng.standard_normal((n, d)), rng.standard_normal((n, hc, d)), rng.standard_normal((n, hc))

    def loss(v):
        o = oracle.side_f64(**v, iters=iters, eps=eps, norm_eps=1e-6, rounded=False)
        return float(np.sum(o["h_norm"] * g_hn) + np.sum(o["y"] * g_y) + np.sum(o["pre"] * g_pre))

    grads = oracle.side_backward(**inp, g_h_norm=g_hn, g_y=g_y, g_pre=g_pre, iters=iters, eps=eps,
                                 norm_eps=1e-6, rounded=False)
    names = {"x": "g_x", "pre_mix": "g_pre_mix", "f": "g_f", "hc_fn": "g_hc_fn",
             "hc_scale": "g_hc_scale", "hc_base": "g_hc_base", "norm_w": "g_norm_w"}
    for name, gname in names.items():
        flat = inp[name].reshape(-1)
        picks = rng.choice(flat.size, size=min(flat.size, 8), replace=False)
        for i in picks:
            h = 1e-5 * max(1.0, abs(flat[i]))
            up, dn = {k: v.copy() for k, v in inp.items()}, {k: v.copy() for k, v in inp.items()}
            up[name].reshape(-1)[i] += h
            dn[name].reshape(-1)[i] -= h
            fd = (loss(up) - loss(dn)) / (2 * h)
            got = grads[gname].reshape(-1)[i]
            assert abs(got - fd) <= 1e-6 * max(1.0, abs(fd)), (name, int(i), got, fd)


def test_side_backward_casts_enter_only_through_h():
    # With pre_mix one-hot and x bf16-representable, h = x_s is exactly a bf16
    # value, so casting h changes nothing; the backward never reads h_norm or y
    # themselves, so the rounded and unrounded backward are then identical.
    rng = np.random.default_rng(77)
    n, hc, d = 3, 4, 16
    inp = _bwd_case(rng, n, hc, d)
    inp["x"] = oracle.bf16_to_f64(oracle.bf16_from_f64(inp["x"]))
    inp["pre_mix"] = np.zeros((n, hc))
    inp["pre_mix"][:, 2] = 1.0
    g = dict(g_h_norm=rng.standard_normal((n, d)), g_y=rng.standard_normal((n, hc, d)),
             g_pre=rng.standard_normal((n, hc)))
    a = oracle.side_backward(**inp, **g, rounded=True)
    b = oracle.side_backward(**inp, **g, rounded=False)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
