"""The fused QKV projection on the GPU (through the C ABI) against the fp64
oracle, and the projection feeding the attention through its strided views.

Bar for the projection: every output within one bf16 ulp of the fp64 value
plus the fp32 accumulation error, |gpu - ref| <= 2^-7 |ref| +
2^-16 sum_c |x_c w_c| (the q block scaled alike), and at least 99 % of the
outputs equal to the fp64 value rounded to bf16 (nearest even).
"""
import numpy as np
import pytest
import torch

import na3d_inputs
import neighborhood_attention_video_gb300 as na
import oracle

pytestmark = pytest.mark.gpu


def bits(a):
    return na3d_inputs.f64_to_bf16_bits(np.asarray(a, dtype=np.float64))


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def from_dev(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make(M, C, NH, HD, seed, with_bias):
    rng = np.random.default_rng(seed)
    N = 3 * NH * HD
    x = bits(rng.normal(size=(M, C)))
    w = bits(rng.normal(size=(N, C)) / np.sqrt(C))
    b = bits(rng.normal(size=N) * 0.5) if with_bias else None
    return x, w, b


def check_projection(got_bits, x, w, b, NH, HD, label):
    ref = oracle.qkv_projection(x, w, b, NH, HD)
    mag = oracle.qkv_projection(x & 0x7FFF, w & 0x7FFF, None, NH, HD)   # sum |x||w|, q block scaled
    got = na3d_inputs.bf16_bits_to_f64(got_bits).reshape(ref.shape)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    bound = 2.0 ** -7 * np.abs(ref) + 2.0 ** -16 * mag
    exact = float(np.mean(got_bits.reshape(ref.shape) == bits(ref)))
    print(f"{label}: max err/bound {float((err / bound).max()):.3f}, equal to the rounded oracle {exact:.4f}")
    assert (err <= bound).all(), label
    assert exact >= 0.99, (label, exact)


CASES = [
    # M, C, NH, HD, bias     what it covers
    (4096, 512, 8, 64, True),     # the benchmark head layout, six N tiles
    (1000, 64, 2, 32, False),     # ragged M, one K block, no bias
    (300, 40, 3, 16, True),       # K tail inside the only K block, N = 144 < one tile
    (777, 256, 4, 128, True),     # HD 128
    (2048, 1032, 1, 64, False),   # 17 K blocks with a tail of 8
]


@pytest.mark.parametrize("M,C,NH,HD,with_bias", CASES, ids=lambda v: str(v))
def test_projection_matches_the_oracle(M, C, NH, HD, with_bias):
    x, w, b = make(M, C, NH, HD, seed=M + C, with_bias=with_bias)
    qkv = torch.empty((M, 3 * NH * HD), dtype=torch.bfloat16, device="cuda")
    na.na3d_qkv_proj(to_dev(x), to_dev(w), to_dev(b) if b is not None else None, qkv, NH, HD)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    check_projection(from_dev(qkv), x, w, b, NH, HD, f"proj M={M} C={C} NH={NH} HD={HD}")


def test_full_size_projection_on_sampled_rows():
    """The benchmark's projection (65536 tokens, C = 512, 8 heads of 64: the
    headline attention's q, k, v) in its own launch configuration; rows are
    independent, so the oracle checks a random sample of them plus the first
    and last tile."""
    M, C, NH, HD = 65536, 512, 8, 64
    x, w, b = make(M, C, NH, HD, seed=5, with_bias=True)
    qkv = torch.empty((M, 3 * NH * HD), dtype=torch.bfloat16, device="cuda")
    na.na3d_qkv_proj(to_dev(x), to_dev(w), to_dev(b), qkv, NH, HD)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    got = from_dev(qkv)
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(M - 128, M), rng.integers(0, M, 768)]))
    check_projection(got[rows], x[rows], w, b, NH, HD, f"proj M={M} sampled {rows.size} rows")


def test_projection_beyond_2_31_output_elements():
    """The benchmark's own projection shape (393216 tokens, C = 2048, 16 heads of
    128): 2.4e9 output elements, so the last rows sit past 2^31. x is drawn on
    the device (seeded); the oracle checks the first and last tiles and a
    random sample of rows from their x rows."""
    M, C, NH, HD = 393216, 2048, 16, 128
    N = 3 * NH * HD
    assert M * N > 2 ** 31
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    xd = torch.randn((M, C), generator=gen, device="cuda").to(torch.bfloat16)
    _, w, b = make(8, C, NH, HD, seed=10, with_bias=True)
    qkv = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    na.na3d_qkv_proj(xd, to_dev(w), to_dev(b), qkv, NH, HD)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(M - 128, M), rng.integers(0, M, 512)]))
    idx = torch.from_numpy(rows).cuda()
    got = from_dev(qkv.index_select(0, idx))
    x_rows = from_dev(xd.index_select(0, idx))
    check_projection(got, x_rows, w, b, NH, HD, f"proj M={M} C={C}: sampled {rows.size} rows")
    del xd, qkv
    torch.cuda.empty_cache()


def test_unaligned_output_uses_16_byte_stores():
    M, C, NH, HD = 513, 128, 2, 64
    x, w, b = make(M, C, NH, HD, seed=5, with_bias=True)
    N = 3 * NH * HD
    buf = torch.full((M * N + 8 + 4096,), 3.0, dtype=torch.bfloat16, device="cuda")
    qkv = buf[8:8 + M * N]                      # 16-byte but not 32-byte aligned
    na.na3d_qkv_proj(to_dev(x), to_dev(w), to_dev(b), qkv, NH, HD)
    torch.cuda.synchronize()
    assert bool((buf[:8] == 3.0).all()) and bool((buf[8 + M * N:] == 3.0).all())
    check_projection(from_dev(qkv), x, w, b, NH, HD, "proj, 16-byte aligned output")


def test_projection_feeds_the_attention():
    """x -> na3d_qkv_proj -> q, k, v views -> na3d_fwd_strided: the attention
    output matches the oracle attention of the projected q, k, v."""
    B, T, H, W, NH, HD, C = 1, 6, 12, 20, 2, 64, 96
    kernel = (3, 5, 7)
    M = B * T * H * W
    x, w, b = make(M, C, NH, HD, seed=31, with_bias=True)
    qkv = torch.empty((B, T, H, W, 3, NH, HD), dtype=torch.bfloat16, device="cuda")
    na.na3d_qkv_proj(to_dev(x), to_dev(w), to_dev(b), qkv, NH, HD)
    q, k, v = na.qkv_views(qkv)
    out = torch.empty((B, T, H, W, NH, HD), dtype=torch.bfloat16, device="cuda")
    na.na3d_fwd_strided(q, k, v, out, kernel)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    pb = from_dev(qkv)
    check_projection(pb.reshape(M, -1), x, w, b, NH, HD, "proj for attention")
    qb, kb, vb = (np.ascontiguousarray(pb[:, :, :, :, j]) for j in range(3))
    want = oracle.na3d_fwd(qb, kb, vb, kernel)
    got = na3d_inputs.bf16_bits_to_f64(from_dev(out))
    rel = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    print(f"attention on the projection: rel_l2 {rel:.3e}")
    assert rel <= 5e-3 and float(np.abs(got - want).max()) <= 3e-2
