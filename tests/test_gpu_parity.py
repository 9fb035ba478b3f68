"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Bar: relative L2 error <= 5e-3 and max abs error <= 3e-2 against the
unrounded fp64 oracle, on the same seeded inputs. Small and medium shapes are
compared element by element over the whole output; the full benchmark shapes
are compared on sampled rows (random rows plus every grid corner and edge
row), which the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import na3d_inputs
from instance_cases import INSTANCE_CASES
import neighborhood_attention_video_gb300 as na
import oracle

pytestmark = pytest.mark.gpu

REL_L2_MAX = 5e-3
MAX_ABS_MAX = 3e-2


def to_dev(a):
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def from_dev(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(q, k, v, kernel, stream=None):
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = torch.empty_like(qd)
    na.na3d_fwd(qd, kd, vd, out, kernel, stream=stream)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    return from_dev(out)


def errors(got_bits, want):
    got = na3d_inputs.bf16_bits_to_f64(got_bits)
    assert np.isfinite(got).all()
    rel = float(np.linalg.norm((got - want).ravel()) / np.linalg.norm(want.ravel()))
    mabs = float(np.abs(got - want).max())
    return rel, mabs


def check(got_bits, want, label):
    rel, mabs = errors(got_bits, want)
    print(f"{label}: rel_l2 {rel:.3e} max_abs {mabs:.3e}")
    assert rel <= REL_L2_MAX, (label, rel)
    assert mabs <= MAX_ABS_MAX, (label, mabs)


# ------------------------------------------------------------ whole-output parity

FULL_CASES = [
    # (B, T, H, W, NH, HD), kernel          what it covers
    ((1, 4, 8, 16, 2, 32), (3, 5, 5)),       # the tiny benchmark configuration, seed 0
    ((1, 6, 20, 36, 2, 64), (3, 7, 7)),      # several bricks, ragged tails on every axis
    ((2, 5, 13, 19, 3, 128), (3, 5, 7)),     # HD 128, B and NH > 1, ragged
    ((1, 3, 6, 40, 2, 128), (3, 5, 33)),     # HD 128 with per-key masks (W union over 32 keys)
    ((1, 8, 14, 14, 4, 128), (7, 9, 9)),     # HD 128, many chunks per unit, head groups
    ((1, 4, 9, 40, 2, 256), (3, 3, 11)),     # HD 256 (64-key chunks)
    ((1, 3, 7, 11, 2, 16), (3, 5, 5)),       # HD 16
    ((1, 16, 64, 5, 8, 64), (3, 5, 5)),      # narrow edge tile: W = KW = 5
    ((1, 8, 24, 33, 2, 64), (3, 7, 33)),     # W = KW = 33
    ((1, 16, 20, 20, 2, 64), (11, 11, 11)),  # large window
    ((1, 3, 4, 150, 1, 64), (1, 3, 141)),    # W halo wider than one chunk: split W segments
    ((1, 1, 12, 20, 2, 32), (1, 5, 7)),      # one frame (2-D)
    ((1, 40, 1, 1, 2, 32), (7, 1, 1)),       # 1-D along T
    ((1, 3, 5, 7, 2, 64), (3, 5, 7)),        # window = whole grid: full attention
    ((1, 16, 64, 64, 8, 64), (3, 7, 7)),     # benchmark shape, (3,7,7)
    ((1, 16, 64, 96, 8, 64), (3, 5, 5)),     # benchmark shape, (3,5,5)
    ((1, 3, 6, 10, 64, 16), (3, 3, 5)),      # 64 heads of 16
    ((64, 2, 3, 5, 2, 32), (1, 3, 5)),       # 64 small batches: many units over tiny grids
    ((1, 4, 8, 128, 8, 64), (3, 5, 27)),     # the pages' wide-KW benchmark shape (NH 8)
    ((1, 16, 80, 32, 8, 64), (11, 11, 11)),  # the pages' small (11,11,11) benchmark shape (NH 8)
    ((1, 4, 9, 20, 2, 512), (3, 5, 7)),      # HD 512: two passes over 256 output columns
    ((1, 3, 5, 40, 1, 512), (3, 3, 33)),     # HD 512 with per-key masks
    ((2, 3, 6, 12, 3, 1024), (3, 3, 5)),     # HD 1024: four passes, B and NH > 1
    ((1, 2, 4, 6, 1, 2048), (1, 3, 5)),      # HD 2048
    ((1, 1, 2, 3, 1, 4096), (1, 1, 3)),      # HD 4096: sixteen passes
    ((1, 2, 4, 40, 1, 1024), (1, 3, 33)),    # HD 1024 with per-key masks
    # whole-row W windows (KW = W): H windows applied by the tensor core
    ((1, 4, 10, 21, 2, 128), (3, 5, 21)),    # HD 128
    ((1, 5, 12, 9, 3, 32), (3, 3, 9)),       # HD 32
    ((1, 3, 8, 13, 2, 256), (3, 5, 13)),     # HD 256 (one CTA per SM)
    ((1, 4, 20, 3, 2, 16), (3, 7, 3)),       # HD 16, W = 3
    ((2, 6, 30, 1, 2, 64), (3, 5, 1)),       # W = KW = 1
    ((1, 7, 40, 17, 2, 64), (5, 11, 17)),    # tall H windows: many h-chunks per brick
] + [(shape, kernel) for shape, kernel, _, _ in INSTANCE_CASES]   # one problem per kernel instance


@pytest.mark.parametrize("shape,kernel", FULL_CASES, ids=lambda x: "x".join(map(str, x)))
def test_parity_whole_output(shape, kernel):
    q, k, v = na3d_inputs.make_qkv(*shape, seed=0)
    got = run_gpu(q, k, v, kernel)
    want = oracle.na3d_fwd(q, k, v, kernel)
    check(got, want, f"{shape} {kernel}")


def random_cases(n, seed):
    """Seeded random problems over every mask mode: grids up to 16 x 24 x 60,
    odd windows (a quarter of them spanning the whole W axis), head dims 16
    to 512, one or two batches and heads."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        T, H = (int(x) for x in rng.integers(1, 17, size=2))
        W = int(rng.integers(1, 61))
        KT, KH, KW = (int(rng.choice(np.arange(1, N + 1, 2))) for N in (T, H, W))
        if W % 2 == 1 and rng.random() < 0.25:
            KW = W
        HD = int(rng.choice([16, 32, 64, 64, 128, 128, 256, 512]))
        B, NH = (int(x) for x in rng.integers(1, 3, size=2))
        out.append(((B, T, H, W, NH, HD), (KT, KH, KW)))
    return out


@pytest.mark.parametrize("shape,kernel", random_cases(32, 2024), ids=lambda x: "x".join(map(str, x)))
def test_parity_random_problems(shape, kernel):
    q, k, v = na3d_inputs.make_qkv(*shape, seed=sum(shape) + sum(kernel))
    got = run_gpu(q, k, v, kernel)
    check(got, oracle.na3d_fwd(q, k, v, kernel), f"random {shape} {kernel}")


# ------------------------------------------------------------ full sizes, sampled rows

def sample_rows(shape, n_random, seed=0):
    B, T, H, W, NH, HD = shape
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, B * T * H * W * NH, size=n_random).tolist())
    # corners and edge lines of the grid, for every batch and a few heads
    for b in {0, B - 1}:
        for n in {0, NH - 1}:
            for t in {0, 1, T // 2, T - 2, T - 1}:
                for h in {0, 1, H // 2, H - 2, H - 1}:
                    for w in range(W):
                        if t in (0, T - 1) or h in (0, H - 1) or w in (0, 1, W - 2, W - 1):
                            tt, hh = min(max(t, 0), T - 1), min(max(h, 0), H - 1)
                            rows.add(((((b * T + tt) * H + hh) * W + w) * NH) + n)
    return np.array(sorted(rows), dtype=np.int64)


BIG_CASES = [
    ((1, 16, 48, 48, 8, 64), (11, 11, 11)),
    ((2, 16, 96, 128, 16, 128), (3, 7, 7)),
    ((2, 8, 64, 33, 8, 64), (3, 7, 33)),
]


@pytest.mark.parametrize("shape,kernel", BIG_CASES, ids=lambda x: "x".join(map(str, x)))
def test_parity_full_size_sampled(shape, kernel):
    q, k, v = na3d_inputs.make_qkv(*shape, seed=0)
    got = run_gpu(q, k, v, kernel).reshape(-1, shape[-1])
    rows = sample_rows(shape, 20000)
    want = oracle.na3d_fwd_rows(q, k, v, kernel, rows)
    check(got[rows], want, f"{shape} {kernel} ({rows.size} sampled rows)")


def test_parity_beyond_2_31_elements():
    """Tensors of more than 2^31 elements (6 GB each): every offset past 2^31
    must be computed in 64 bits. The inputs are drawn on the device (seeded).
    Each sampled row, including the last rows of the tensor, is checked by the
    oracle on its own window box: a (1, KT, KH, KW, 1, HD) problem whose
    windows cover the whole box, so its output there is the whole-grid one."""
    shape, kernel = (2, 79, 192, 192, 8, 64), (3, 5, 5)
    B, T, H, W, NH, HD = shape
    KT, KH, KW = kernel
    n = int(np.prod(shape))
    assert n > 2 ** 31
    gen = torch.Generator(device="cuda")
    gen.manual_seed(31)

    def draw(scale):
        t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        flat = t.view(-1)
        step = 1 << 28
        for i in range(0, n, step):
            m = min(step, n - i)
            flat[i:i + m] = (torch.randn(m, generator=gen, device="cuda") * scale).to(torch.bfloat16)
        return t

    q, k, v = draw(HD ** -0.5), draw(1.0), draw(1.0)
    out = torch.full_like(q, float("nan"))
    na.na3d_fwd(q, k, v, out, kernel)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0

    total = B * T * H * W * NH
    rng = np.random.default_rng(5)
    rows = sorted(set(rng.integers(0, total, size=200).tolist()) | set(range(total - 40, total)) | {0})
    got, want = [], []
    for r in rows:
        b, t, h, w, head = (int(x) for x in np.unravel_index(r, (B, T, H, W, NH)))
        sT, sH, sW = (oracle.window_start(i, K, N) for i, K, N in ((t, KT, T), (h, KH, H), (w, KW, W)))
        box = (b, slice(sT, sT + KT), slice(sH, sH + KH), slice(sW, sW + KW), head)
        kb = from_dev(k[box].contiguous()).reshape(1, KT, KH, KW, 1, HD)
        vb = from_dev(v[box].contiguous()).reshape(1, KT, KH, KW, 1, HD)
        qb = np.zeros_like(kb)
        qb[0, t - sT, h - sH, w - sW, 0] = from_dev(q[b, t, h, w, head].contiguous())
        want.append(oracle.na3d_fwd(qb, kb, vb, kernel)[0, t - sT, h - sH, w - sW, 0])
        got.append(from_dev(out[b, t, h, w, head].contiguous()))
    check(np.stack(got), np.stack(want), f"{shape} {kernel} ({len(rows)} sampled rows, last ones included)")
    del q, k, v, out
    torch.cuda.empty_cache()


# ------------------------------------------------------------ exact special cases

def test_unit_window_returns_v_bit_exactly():
    shape = (2, 5, 9, 13, 3, 64)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=4)
    got = run_gpu(q, k, v, (1, 1, 1))
    np.testing.assert_array_equal(got, v)


def test_constant_v_returns_the_constant():
    shape = (1, 6, 17, 23, 2, 64)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=9)
    c = na3d_inputs.f64_to_bf16_bits(np.array([0.75]))[0]
    v[...] = c
    got = na3d_inputs.bf16_bits_to_f64(run_gpu(q, k, v, (3, 5, 7)))
    # within one bf16 ulp of 0.75 (2^-8)
    assert np.abs(got - 0.75).max() <= 2.0 ** -8
    print("constant-V exact fraction:", float(np.mean(got == 0.75)))


def test_axis_flip_equivariance():
    shape = (1, 7, 12, 18, 2, 64)
    kernel = (3, 5, 7)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=21)
    base = na3d_inputs.bf16_bits_to_f64(run_gpu(q, k, v, kernel))
    for axis in (1, 2, 3):
        fl = [np.ascontiguousarray(np.flip(x, axis=axis)) for x in (q, k, v)]
        got = na3d_inputs.bf16_bits_to_f64(run_gpu(*fl, kernel))
        ref = np.flip(base, axis=axis)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 5e-3, (axis, rel)


@pytest.mark.parametrize("hd", [64, 128, 512])
@pytest.mark.parametrize("kernel", [(3, 5, 7), (3, 7, 33)], ids=lambda x: "x".join(map(str, x)))
def test_score_spike_in_a_later_chunk(kernel, hd):
    """Keys of the last frames are scaled up, so rows meet scores tens of log2
    units above everything they saw in earlier chunks: the kept reference
    maximum must be raised mid-row and O rescaled (the exact pass taken when a
    chunk's probabilities sum past 2^32). With HD 128 the two halves of each
    score row must take these steps together."""
    shape = (1, 6, 12, 36, 2, hd)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=13)
    kf = na3d_inputs.bf16_bits_to_f64(k)
    kf[:, 4:] *= 40.0
    k = na3d_inputs.f64_to_bf16_bits(kf)
    got = run_gpu(q, k, v, kernel)
    check(got, oracle.na3d_fwd(q, k, v, kernel), f"spike {shape} {kernel}")


@pytest.mark.parametrize("shape,kernel", [
    ((1, 6, 8, 16, 2, 64), (3, 3, 3)),     # tensor-core W mask, 16-key rows
    ((1, 6, 8, 48, 2, 64), (3, 3, 33)),    # per-key masks, 48-key rows
    ((1, 6, 8, 48, 2, 32), (3, 3, 33)),    # HD 32
], ids=lambda x: "x".join(map(str, x)))
def test_score_spike_on_paired_score_tiles(shape, kernel):
    """The score spike on problems that run on the 96-key tiles in pairs of
    tensor-memory slots (two tiles in flight): the rescale of O waits for the
    previous product through that ring's barriers."""
    assert na.na3d_plan(*shape[1:], *kernel)["tile_cap"] == 96
    q, k, v = na3d_inputs.make_qkv(*shape, seed=17)
    kf = na3d_inputs.bf16_bits_to_f64(k)
    kf[:, 4:] *= 40.0
    k = na3d_inputs.f64_to_bf16_bits(kf)
    got = run_gpu(q, k, v, kernel)
    check(got, oracle.na3d_fwd(q, k, v, kernel), f"spike {shape} {kernel}")


def test_score_spike_with_whole_row_windows():
    """As above, with KW = W: the H window comes from the tensor core, and
    the spiking rows must still raise the kept reference maximum."""
    shape, kernel = (1, 6, 14, 33, 2, 64), (3, 7, 33)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=31)
    kf = na3d_inputs.bf16_bits_to_f64(k)
    kf[:, 4:] *= 40.0
    k = na3d_inputs.f64_to_bf16_bits(kf)
    got = run_gpu(q, k, v, kernel)
    check(got, oracle.na3d_fwd(q, k, v, kernel), f"spike {shape} {kernel}")


# ------------------------------------------------------------ launch behaviour

def test_deterministic_and_stream_independent():
    shape, kernel = (1, 6, 20, 36, 2, 64), (3, 7, 7)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=3)
    a = run_gpu(q, k, v, kernel)
    b = run_gpu(q, k, v, kernel)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = run_gpu(q, k, v, kernel, stream=s)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)


@pytest.mark.parametrize("shape,kernel", [((1, 16, 64, 64, 8, 64), (3, 7, 7)),
                                          ((1, 16, 64, 96, 8, 64), (3, 5, 5)),   # paired 96-key tiles
                                          ((1, 16, 64, 5, 8, 64), (3, 5, 5)),
                                          ((2, 8, 48, 48, 8, 128), (3, 7, 7)),
                                          ((1, 8, 32, 40, 8, 256), (3, 5, 7)),
                                          ((1, 6, 24, 40, 8, 512), (3, 5, 7)),
                                          ((2, 8, 64, 33, 8, 64), (3, 7, 33)),
                                          ((1, 16, 48, 48, 8, 64), (11, 11, 11))],
                         ids=lambda x: "x".join(map(str, x)))
def test_repeated_launches_are_bit_identical(shape, kernel):
    """Shapes with many work units per CTA: every per-chunk pipeline barrier
    goes through many phases, and softmax warps can drift a chunk apart. A
    barrier that lets one warp complete another chunk's phase shows up as
    rows that differ between launches."""
    q, k, v = na3d_inputs.make_qkv(*shape, seed=11)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    first = None
    for _ in range(6):
        out = torch.full_like(qd, float("nan"))
        na.na3d_fwd(qd, kd, vd, out, kernel)
        torch.cuda.synchronize()
        assert na.na3d_device_status() == 0
        got = from_dev(out)
        assert np.isfinite(na3d_inputs.bf16_bits_to_f64(got)).all()
        if first is None:
            first = got
        else:
            np.testing.assert_array_equal(got, first)


def test_concurrent_launches_on_several_streams():
    """Launches in flight at once on different streams (HD-64 problems on
    both tile families and an HD-128 problem, several units per CTA): their
    CTAs may share SMs and the tensor memory of an SM. Each result equals its
    launch alone, bit for bit, and the device reports no wait that ran out."""
    cases = [((1, 8, 32, 48, 4, 64), (3, 7, 7), 41), ((1, 6, 24, 40, 4, 128), (3, 5, 7), 42),
             ((1, 8, 32, 48, 4, 64), (3, 5, 5), 43)]
    alone, dev = [], []
    for shape, kernel, seed in cases:
        q, k, v = na3d_inputs.make_qkv(*shape, seed=seed)
        alone.append(run_gpu(q, k, v, kernel))
        dev.append((to_dev(q), to_dev(k), to_dev(v), kernel))
    streams = [torch.cuda.Stream() for _ in cases]
    for _ in range(3):
        outs = [torch.full_like(d[0], float("nan")) for d in dev]
        torch.cuda.synchronize()
        for (qd, kd, vd, kernel), out, st in zip(dev, outs, streams):
            na.na3d_fwd(qd, kd, vd, out, kernel, stream=st)
        torch.cuda.synchronize()
        assert na.na3d_device_status() == 0
        for out, want in zip(outs, alone):
            np.testing.assert_array_equal(from_dev(out), want)


def test_cuda_graph_capture_and_replay():
    """na3d_fwd launches into a CUDA graph being captured on the current
    stream (one kernel, host-encoded tensor maps passed by value); replays
    recompute the same bits, including after the inputs change in place."""
    shape, kernel = (1, 6, 20, 36, 2, 64), (3, 7, 7)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=37)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    want = run_gpu(q, k, v, kernel)
    out = torch.empty_like(qd)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):           # a launch outside capture first (lazy set-up)
        na.na3d_fwd(qd, kd, vd, out, kernel)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        na.na3d_fwd(qd, kd, vd, out, kernel)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(from_dev(out), want)
    q2, k2, v2 = na3d_inputs.make_qkv(*shape, seed=38)
    qd.copy_(to_dev(q2)); kd.copy_(to_dev(k2)); vd.copy_(to_dev(v2))
    g.replay()
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    np.testing.assert_array_equal(from_dev(out), run_gpu(q2, k2, v2, kernel))


def test_attention_returns_what_na3d_fwd_writes():
    shape, kernel = (1, 6, 20, 36, 2, 64), (3, 7, 7)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=23)
    want = run_gpu(q, k, v, kernel)
    out = na.na3d_attention(to_dev(q), to_dev(k), to_dev(v), kernel)
    torch.cuda.synchronize()
    assert out.shape == shape and out.dtype == torch.bfloat16 and out.is_contiguous()
    np.testing.assert_array_equal(from_dev(out), want)


def test_invalid_device_arguments_are_rejected():
    shape = (1, 4, 8, 16, 2, 32)
    x = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    with pytest.raises(na.NA3DError) as e:
        na.na3d_fwd(x, x, x, out, (4, 5, 5))
    assert e.value.status == 3
    with pytest.raises(na.NA3DError) as e:
        na.na3d_fwd(x, x, x, x, (3, 5, 5))
    assert e.value.status == 6
    # a view starting 2 bytes into a buffer is not 16-byte aligned
    flat = torch.zeros(x.numel() + 8, dtype=torch.bfloat16, device="cuda")
    mis = flat[1:1 + x.numel()].view(shape)
    with pytest.raises(na.NA3DError) as e:
        na.na3d_fwd(mis, x, x, out, (3, 5, 5))
    assert e.value.status == 5


def test_empty_batch_is_rejected():
    x = torch.zeros((0, 4, 8, 16, 2, 32), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(na.NA3DError) as e:
        na.na3d_fwd(x, x, x, torch.empty_like(x), (3, 5, 5))
    assert e.value.status == 2


@pytest.mark.parametrize("hd", [64, 128, 512])
@pytest.mark.parametrize("shift", [0, 8], ids=["out32B", "out16B"])
def test_output_untouched_outside_the_tensor(shift, hd):
    """The kernel writes exactly the output tensor: guard bands around it keep
    their sentinel values. `shift` elements move the output off a 32-byte
    boundary (16-byte stores instead of 32-byte ones)."""
    shape, kernel = (1, 5, 11, 13, 3, hd), (3, 5, 5)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=5)
    n = int(np.prod(shape))
    guard = 4096 + shift
    buf = torch.full((n + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(shape)
    na.na3d_fwd(to_dev(q), to_dev(k), to_dev(v), out, kernel)
    torch.cuda.synchronize()
    assert bool((buf[:guard] == 7.0).all()) and bool((buf[guard + n:] == 7.0).all())
    check(from_dev(out.contiguous()), oracle.na3d_fwd(q, k, v, kernel), "guarded")


# ------------------------------------------------------------ query boxes (global coordinates)

REGION_CASES = [
    # (B, T, H, W, NH, HD), kernel, (t0, h0, w0, Tq, Hq, Wq)
    ((1, 6, 12, 40, 2, 64), (3, 5, 7), (0, 0, 24, 6, 12, 16)),     # right W tile, as in tiled decode
    ((1, 8, 16, 20, 2, 64), (3, 5, 5), (2, 3, 5, 4, 8, 9)),        # interior box on every axis
    ((1, 5, 9, 30, 2, 32), (3, 5, 11), (1, 2, 10, 2, 4, 4)),       # box narrower than the window
    ((1, 6, 10, 24, 2, 64), (5, 5, 5), (3, 5, 20, 3, 5, 4)),       # box at the far borders
    ((2, 5, 13, 19, 3, 128), (3, 5, 7), (1, 2, 3, 3, 8, 10)),      # HD 128, B and NH > 1
    ((1, 5, 9, 21, 2, 512), (3, 5, 7), (1, 2, 6, 3, 5, 9)),        # HD 512
    ((1, 5, 14, 25, 2, 64), (3, 5, 25), (1, 3, 0, 3, 8, 25)),      # whole-row W windows
    ((1, 5, 14, 25, 2, 64), (3, 5, 25), (0, 4, 5, 5, 7, 10)),      # whole-row W windows, W sub-box
    ((2, 4, 11, 9, 3, 128), (3, 5, 9), (1, 3, 0, 2, 6, 9)),        # whole-row W windows, HD 128
    ((1, 4, 9, 50, 2, 64), (3, 3, 33), (0, 0, 7, 4, 9, 30)),       # wide window: per-key masks
    ((1, 6, 16, 40, 2, 64), (3, 5, 5), (1, 2, 8, 4, 12, 24)),      # interior box, HD 64 (3,5,5)
]


def region_oracle(q_full, k, v, kernel, box):
    """The oracle on the whole grid, restricted to the box: a query's output
    depends only on its own q and on k, v (global windows)."""
    t0, h0, w0, Tq, Hq, Wq = box
    full = oracle.na3d_fwd(q_full, k, v, kernel)
    return full[:, t0:t0 + Tq, h0:h0 + Hq, w0:w0 + Wq]


@pytest.mark.parametrize("shape,kernel,box", REGION_CASES, ids=lambda x: "x".join(map(str, x)))
def test_region_matches_the_whole_grid_oracle(shape, kernel, box):
    q_full, k, v = na3d_inputs.make_qkv(*shape, seed=17)
    t0, h0, w0, Tq, Hq, Wq = box
    q = np.ascontiguousarray(q_full[:, t0:t0 + Tq, h0:h0 + Hq, w0:w0 + Wq])
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = torch.empty_like(qd)
    na.na3d_fwd_region(qd, kd, vd, out, kernel, (t0, h0, w0))
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    check(from_dev(out), region_oracle(q_full, k, v, kernel, box), f"region {shape} {kernel} {box}")


def test_region_of_the_whole_grid_is_na3d_fwd():
    shape, kernel = (1, 6, 20, 36, 2, 64), (3, 7, 7)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=19)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = torch.empty_like(qd)
    na.na3d_fwd_region(qd, kd, vd, out, kernel, (0, 0, 0))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(from_dev(out), run_gpu(q, k, v, kernel))


def test_w_tiles_reassemble_the_whole_output():
    """Tiled decode: the W axis cut into tiles, each tile's queries attending
    to the whole grid, reassembles the untiled result (within the bar)."""
    shape, kernel = (1, 6, 16, 48, 2, 64), (3, 7, 9)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=23)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    tiles = []
    for w0, w1 in ((0, 20), (20, 29), (29, 48)):
        out = torch.empty((1, 6, 16, w1 - w0, 2, 64), dtype=torch.bfloat16, device="cuda")
        na.na3d_fwd_region(qd[:, :, :, w0:w1].contiguous(), kd, vd, out, kernel, (0, 0, w0))
        tiles.append(out)
    torch.cuda.synchronize()
    got = from_dev(torch.cat(tiles, dim=3).contiguous())
    check(got, oracle.na3d_fwd(q, k, v, kernel), "W tiles")


def test_region_with_strided_views():
    """The box's q and the whole grid's k, v as slices of fused projection outputs."""
    shape, kernel, box = (1, 6, 12, 28, 2, 64), (3, 5, 7), (1, 2, 9, 4, 8, 12)
    t0, h0, w0, Tq, Hq, Wq = box
    q_full, k, v = na3d_inputs.make_qkv(*shape, seed=29)
    fused = np.stack([q_full, k, v], axis=4)          # (B, T, H, W, 3, NH, HD)
    fd = torch.from_numpy(fused.view(np.int16)).cuda().view(torch.bfloat16)
    qv = fd[:, t0:t0 + Tq, h0:h0 + Hq, w0:w0 + Wq, 0]
    assert not qv.is_contiguous()
    out = torch.empty((1, Tq, Hq, Wq, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):          # a box view of the grid has no single token stride
        na.na3d_fwd_region(qv, fd[:, :, :, :, 1], fd[:, :, :, :, 2], out, kernel, (t0, h0, w0))
    qb = torch.from_numpy(np.stack([q_full[:, t0:t0 + Tq, h0:h0 + Hq, w0:w0 + Wq]] * 3, axis=4)
                          .view(np.int16)).cuda().view(torch.bfloat16)[:, :, :, :, 1]
    na.na3d_fwd_region(qb, fd[:, :, :, :, 1], fd[:, :, :, :, 2], out, kernel, (t0, h0, w0))
    torch.cuda.synchronize()
    check(from_dev(out), region_oracle(q_full, k, v, kernel, box), "strided region")


# ------------------------------------------------------------ strided (fused QKV) inputs

@pytest.mark.parametrize("shape,kernel", [((1, 6, 20, 36, 2, 64), (3, 7, 7)),
                                          ((2, 5, 13, 19, 3, 128), (3, 5, 7)),
                                          ((1, 8, 24, 33, 2, 64), (3, 7, 33)),
                                          ((1, 4, 9, 20, 2, 1024), (3, 5, 7))],
                         ids=lambda x: "x".join(map(str, x)))
def test_fused_qkv_views_match_contiguous(shape, kernel):
    """q, k, v as the three slices of one fused [B,T,H,W,3,NH,HD] projection
    output: same result as contiguous inputs, and parity with the oracle."""
    B, T, H, W, NH, HD = shape
    q, k, v = na3d_inputs.make_qkv(*shape, seed=6)
    fused = np.stack([q, k, v], axis=4)          # (B, T, H, W, 3, NH, HD)
    fd = torch.from_numpy(fused.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    na.na3d_fwd_strided(fd[:, :, :, :, 0], fd[:, :, :, :, 1], fd[:, :, :, :, 2], out, kernel)
    torch.cuda.synchronize()
    got = from_dev(out)
    np.testing.assert_array_equal(got, run_gpu(q, k, v, kernel))
    check(got, oracle.na3d_fwd(q, k, v, kernel), f"fused {shape} {kernel}")
