"""Pins of the CPU oracle against things other than itself (no GPU).

Each test states what fixes the expected value: a hand-derived table, brute
force from an independent characterisation of the window, a library routine
for a special case, or an invariant of the definition.

The definition: "[Triton/Gluon] Add 3D neighborhood flash attention
(na3d_flash)" (ROCm/aiter pull request 5230), Motivation and Technical Details.
"""
import math
import os

import numpy as np
import pytest
import torch

import na3d_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(a):
    return na3d_inputs.bf16_bits_to_f64(a)


def nearest_centre_starts(N, K):
    """Window starts from a characterisation that does not use a clamp: among
    all length-K intervals inside [0, N), the one whose centre is nearest to i.
    For odd K the nearest centre is unique."""
    s = np.arange(N - K + 1)
    centres = s + (K - 1) / 2.0
    return np.array([s[np.argmin(np.abs(centres - i))] for i in range(N)])


def brute_dense(q, k, v, kernel):
    """Dense L x L attention per (batch, head) with a boolean window mask,
    fp64, windows from ``nearest_centre_starts``."""
    B, T, H, W, NH, HD = q.shape
    KT, KH, KW = kernel
    qd, kd, vd = f64(q), f64(k), f64(v)
    st, sh, sw = (nearest_centre_starts(T, KT), nearest_centre_starts(H, KH),
                  nearest_centre_starts(W, KW))
    tt, hh, ww = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")
    tt, hh, ww = tt.ravel(), hh.ravel(), ww.ravel()
    mask = ((tt[None, :] >= st[tt][:, None]) & (tt[None, :] < st[tt][:, None] + KT)
            & (hh[None, :] >= sh[hh][:, None]) & (hh[None, :] < sh[hh][:, None] + KH)
            & (ww[None, :] >= sw[ww][:, None]) & (ww[None, :] < sw[ww][:, None] + KW))
    out = np.empty_like(qd)
    L = T * H * W
    for b in range(B):
        for n in range(NH):
            Q = qd[b, ..., n, :].reshape(L, HD)
            Kt = kd[b, ..., n, :].reshape(L, HD)
            V = vd[b, ..., n, :].reshape(L, HD)
            S = Q @ Kt.T
            S = np.where(mask, S, -np.inf)
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P /= P.sum(axis=1, keepdims=True)
            out[b, ..., n, :] = (P @ V).reshape(T, H, W, HD)
    return out


def rel_l2(a, b):
    return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))


# ---------------------------------------------------------------- generator

def test_generator_deterministic_and_seeded():
    a = na3d_inputs.make_qkv(1, 2, 3, 4, 2, 16, seed=0)
    b = na3d_inputs.make_qkv(1, 2, 3, 4, 2, 16, seed=0)
    c = na3d_inputs.make_qkv(1, 2, 3, 4, 2, 16, seed=1)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a[1], c[1])
    # q, k and v come from disjoint parts of one stream
    assert not np.array_equal(a[1], a[2])


def test_generator_thread_count_independent():
    a = na3d_inputs.make_qkv(1, 3, 5, 7, 2, 32, seed=3, nthreads=1)
    b = na3d_inputs.make_qkv(1, 3, 5, 7, 2, 32, seed=3, nthreads=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_generator_is_standard_normal():
    z = na3d_inputs.normals_f64(1 << 20, seed=0)
    n = z.size
    assert abs(z.mean()) < 5.0 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 5.0 * math.sqrt(2.0 / n)
    # tail mass beyond 2 sigma: 2 * (1 - Phi(2)) = 0.0455
    frac = np.mean(np.abs(z) > 2.0)
    assert abs(frac - 0.0455) < 0.003


def test_generator_recipe_rounding_and_q_scale():
    B, T, H, W, NH, HD = 1, 2, 2, 3, 2, 32
    q, k, v = na3d_inputs.make_qkv(B, T, H, W, NH, HD, seed=7)
    n = q.size
    z = na3d_inputs.normals_f64(3 * n, seed=7)
    s = np.float32(1.0 / math.sqrt(HD))
    q_expect = na3d_inputs.f64_to_bf16_bits(
        (z[:n].astype(np.float32) * s).astype(np.float64)).reshape(q.shape)
    k_expect = na3d_inputs.f64_to_bf16_bits(z[n:2 * n].astype(np.float32)).reshape(q.shape)
    v_expect = na3d_inputs.f64_to_bf16_bits(z[2 * n:].astype(np.float32)).reshape(q.shape)
    np.testing.assert_array_equal(q, q_expect)
    np.testing.assert_array_equal(k, k_expect)
    np.testing.assert_array_equal(v, v_expect)


# ---------------------------------------------------------------- windows

def load_golden_starts():
    rows = []
    with open(os.path.join(GOLDEN, "window_starts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            vals = [int(x) for x in line.split()]
            rows.append((vals[0], vals[1], vals[2:]))
    return rows


@pytest.mark.parametrize("N,K,starts", load_golden_starts())
def test_window_starts_match_hand_table(N, K, starts):
    assert len(starts) == N
    assert [oracle.window_start(i, K, N) for i in range(N)] == starts
    # the independent characterisation agrees with the table as well
    assert list(nearest_centre_starts(N, K)) == starts


def test_window_starts_sweep_against_nearest_centre():
    for N in range(1, 40):
        for K in range(1, N + 1, 2):
            got = [oracle.window_start(i, K, N) for i in range(N)]
            assert got == list(nearest_centre_starts(N, K)), (N, K)


# ---------------------------------------------------------------- P1 brute force

BRUTE_CASES = [
    ((2, 3, 5, 7, 2, 16), (3, 3, 5)),
    ((1, 4, 8, 16, 2, 32), (3, 5, 5)),     # the tiny benchmark configuration
    ((1, 5, 6, 9, 1, 16), (5, 1, 3)),
    ((1, 1, 7, 9, 2, 16), (1, 7, 3)),      # one frame: 2-D neighbourhoods
    ((1, 9, 1, 1, 2, 16), (5, 1, 1)),      # 1-D along T
    ((1, 3, 4, 33, 1, 16), (3, 3, 33)),    # window as wide as the grid on W
    ((1, 2, 3, 5, 3, 64), (1, 3, 5)),
]


@pytest.mark.parametrize("shape,kernel", BRUTE_CASES)
def test_oracle_matches_brute_force_dense(shape, kernel):
    q, k, v = na3d_inputs.make_qkv(*shape, seed=11)
    got = oracle.na3d_fwd(q, k, v, kernel)
    want = brute_dense(q, k, v, kernel)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_oracle_random_odd_kernels_against_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(6):
        T, H, W = (int(x) for x in rng.integers(1, 8, size=3))
        kernel = tuple(int(rng.choice(np.arange(1, n + 1, 2))) for n in (T, H, W))
        shape = (int(rng.integers(1, 3)), T, H, W, int(rng.integers(1, 3)), 16)
        q, k, v = na3d_inputs.make_qkv(*shape, seed=int(rng.integers(1 << 30)))
        np.testing.assert_allclose(oracle.na3d_fwd(q, k, v, kernel),
                                   brute_dense(q, k, v, kernel), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- P2 full grid

@pytest.mark.parametrize("shape", [(1, 3, 5, 7, 2, 16), (2, 2, 4, 6, 3, 32)])
def test_full_grid_window_is_full_attention(shape):
    B, T, H, W, NH, HD = shape
    q, k, v = na3d_inputs.make_qkv(*shape, seed=2)
    got = oracle.na3d_fwd(q, k, v, (T, H, W))

    def heads(x):  # (B, T, H, W, NH, HD) -> (B, NH, L, HD)
        return torch.from_numpy(f64(x)).permute(0, 4, 1, 2, 3, 5).reshape(B, NH, -1, HD)

    ref = torch.nn.functional.scaled_dot_product_attention(
        heads(q), heads(k), heads(v), scale=1.0)
    ref = ref.reshape(B, NH, T, H, W, HD).permute(0, 2, 3, 4, 1, 5).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- P3, P4

def test_unit_kernel_returns_v_exactly():
    q, k, v = na3d_inputs.make_qkv(2, 3, 4, 5, 2, 16, seed=4)
    np.testing.assert_array_equal(oracle.na3d_fwd(q, k, v, (1, 1, 1)), f64(v))


def test_constant_v_returns_the_constant():
    q, k, v = na3d_inputs.make_qkv(1, 5, 6, 7, 2, 32, seed=9)
    c = na3d_inputs.f64_to_bf16_bits(np.array([0.75]))[0]
    v[...] = c
    out = oracle.na3d_fwd(q, k, v, (3, 5, 3))
    np.testing.assert_allclose(out, 0.75, rtol=0, atol=1e-14)


def test_zero_q_gives_window_mean_of_v():
    """q = 0 makes every score 0, so each output is the plain mean of v over
    the window: a box filter, computed here by 3-D prefix sums over windows
    from the nearest-centre characterisation."""
    shape = (1, 7, 9, 11, 2, 16)
    kernel = (3, 5, 7)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=12)
    q[...] = 0
    got = oracle.na3d_fwd(q, k, v, kernel)
    vd = f64(v)[0]  # (T, H, W, NH, HD)
    T, H, W = shape[1:4]
    cs = np.zeros((T + 1, H + 1, W + 1) + vd.shape[3:])
    cs[1:, 1:, 1:] = vd.cumsum(0).cumsum(1).cumsum(2)
    st, sh, sw = (nearest_centre_starts(T, kernel[0]), nearest_centre_starts(H, kernel[1]),
                  nearest_centre_starts(W, kernel[2]))
    want = np.empty_like(vd)
    for t in range(T):
        for h in range(H):
            for w in range(W):
                a0, a1 = st[t], st[t] + kernel[0]
                b0, b1 = sh[h], sh[h] + kernel[1]
                c0, c1 = sw[w], sw[w] + kernel[2]
                box = (cs[a1, b1, c1] - cs[a0, b1, c1] - cs[a1, b0, c1] - cs[a1, b1, c0]
                       + cs[a0, b0, c1] + cs[a0, b1, c0] + cs[a1, b0, c0] - cs[a0, b0, c0])
                want[t, h, w] = box / np.prod(kernel)
    np.testing.assert_allclose(got[0], want, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- P5 flips

@pytest.mark.parametrize("axis", [1, 2, 3])
def test_axis_flip_equivariance(axis):
    q, k, v = na3d_inputs.make_qkv(1, 6, 7, 8, 2, 16, seed=21)
    kernel = (3, 5, 3)
    out = oracle.na3d_fwd(q, k, v, kernel)
    fl = [np.ascontiguousarray(np.flip(x, axis=axis)) for x in (q, k, v)]
    out_f = oracle.na3d_fwd(*fl, kernel)
    np.testing.assert_allclose(out_f, np.flip(out, axis=axis), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- P6 dimension reduction

def test_one_frame_window_isolates_frames():
    """KT = 1 is 2-D neighborhood attention in each frame: the 3-D result of
    frame t equals the oracle on that frame alone (a grid with T = 1)."""
    shape = (2, 4, 6, 7, 2, 16)
    kernel = (1, 3, 5)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=31)
    out = oracle.na3d_fwd(q, k, v, kernel)
    for t in range(shape[1]):
        sl = [np.ascontiguousarray(x[:, t:t + 1]) for x in (q, k, v)]
        np.testing.assert_allclose(out[:, t:t + 1], oracle.na3d_fwd(*sl, kernel), rtol=1e-13, atol=1e-14)


def test_one_dimensional_grid_is_a_sliding_window_along_t():
    """H = W = 1 is 1-D neighborhood attention along T: for each frame t the
    K frames starting at clamp(t - K//2, 0, T - K), a softmax over their
    scores and the weighted sum of their values, written out here with
    numpy for each (batch, head, frame)."""
    B, T, NH, HD, K = 2, 23, 3, 16, 5
    q, k, v = na3d_inputs.make_qkv(B, T, 1, 1, NH, HD, seed=32)
    got = oracle.na3d_fwd(q, k, v, (K, 1, 1))
    qd, kd, vd = f64(q)[:, :, 0, 0], f64(k)[:, :, 0, 0], f64(v)[:, :, 0, 0]
    want = np.empty_like(qd)
    for b in range(B):
        for n in range(NH):
            for t in range(T):
                s0 = min(max(t - K // 2, 0), T - K)
                x = kd[b, s0:s0 + K, n] @ qd[b, t, n]
                p = np.exp(x - x.max())
                want[b, t, n] = (p / p.sum()) @ vd[b, s0:s0 + K, n]
    np.testing.assert_allclose(got[:, :, 0, 0], want, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- P7 isolation

def test_batch_head_isolation():
    shape = (2, 3, 4, 5, 3, 16)
    kernel = (3, 3, 3)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=8)
    base = oracle.na3d_fwd(q, k, v, kernel)
    k2 = k.copy()
    k2[1, :, :, :, 2, :] ^= 0x0040  # flip a mantissa bit in one (batch, head) slice
    v2 = v.copy()
    v2[1, :, :, :, 2, :] ^= 0x0040
    out = oracle.na3d_fwd(q, k2, v2, kernel)
    changed = np.zeros(base.shape[:5], dtype=bool)
    changed |= np.any(out != base, axis=-1)
    assert changed[1, :, :, :, 2].all()
    changed[1, :, :, :, 2] = False
    assert not changed.any()


# ---------------------------------------------------------------- P8 internals

def test_row_detail_window_and_weights():
    shape = (2, 5, 6, 7, 2, 16)
    kernel = (3, 5, 3)
    B, T, H, W, NH, HD = shape
    q, k, v = na3d_inputs.make_qkv(*shape, seed=13)
    full = oracle.na3d_fwd(q, k, v, kernel)
    st, sh, sw = (nearest_centre_starts(T, 3), nearest_centre_starts(H, 5),
                  nearest_centre_starts(W, 3))
    rng = np.random.default_rng(0)
    for row in rng.integers(0, B * T * H * W * NH, size=25):
        toks, wts, o = oracle.na3d_row_detail(q, k, v, kernel, int(row))
        n = row % NH
        b, t, h, w = np.unravel_index(row // NH, (B, T, H, W))
        assert len(set(toks.tolist())) == 45
        kb, kt, kh, kw = np.unravel_index(toks, (B, T, H, W))
        assert (kb == b).all()
        assert ((kt >= st[t]) & (kt < st[t] + 3)).all()
        assert ((kh >= sh[h]) & (kh < sh[h] + 5)).all()
        assert ((kw >= sw[w]) & (kw < sw[w] + 3)).all()
        assert abs(wts.sum() - 1.0) < 1e-12
        # weights are proportional to exp(q.k)
        qd = f64(q)[b, t, h, w, n]
        x = np.array([qd @ f64(k)[kb[j], kt[j], kh[j], kw[j], n] for j in range(45)])
        np.testing.assert_allclose(wts, np.exp(x - x.max()) / np.exp(x - x.max()).sum(),
                                   rtol=1e-12)
        np.testing.assert_allclose(o, full[b, t, h, w, n], rtol=1e-13, atol=1e-15)


def test_rows_entry_matches_full():
    shape = (1, 4, 8, 16, 2, 32)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=0)
    full = oracle.na3d_fwd(q, k, v, (3, 5, 5)).reshape(-1, 32)
    rows = np.array([0, 5, 17, 255, 511, 1023], dtype=np.int64)
    np.testing.assert_array_equal(oracle.na3d_fwd_rows(q, k, v, (3, 5, 5), rows), full[rows])


def test_oracle_rejects_invalid():
    q, k, v = na3d_inputs.make_qkv(1, 3, 3, 3, 1, 16)
    with pytest.raises(ValueError):
        oracle.na3d_fwd(q, k, v, (5, 1, 1))  # K > N
    with pytest.raises(ValueError):
        oracle.na3d_fwd(q, k, v, (0, 1, 1))
