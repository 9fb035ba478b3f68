"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol that include/na3d.h declares, validates arguments before touching
CUDA, and its tiling plans cover every window (host-side box arithmetic)."""
import ctypes
import os
import re

import numpy as np
import pytest

import neighborhood_attention_video_gb300 as na
from neighborhood_attention_video_gb300 import build as na_build
from instance_cases import INSTANCE_CASES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "na3d.h")

# status codes, as include/na3d.h numbers them
OK, ERR_NULL, ERR_SHAPE, ERR_KERNEL, ERR_HEAD_DIM, ERR_ALIGN, ERR_ALIAS = 0, 1, 2, 3, 4, 5, 6
ERR_OVERFLOW, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = 7, 8, 9, 10, 11


@pytest.fixture(scope="module")
def lib():
    na_build.build()
    return na.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(na3d_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    assert declared_functions() == sorted(na.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {na.library_path()}").read()
    exported = set(re.findall(r" T (na3d_\w+)", out))
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for code in range(12):
        s = na.na3d_status_string(code)
        assert s.startswith("NA3D_")
    assert "unknown" in na.na3d_status_string(999)


def call_fwd(lib, ptrs=(16, 32, 48, 1 << 20), dims=(1, 4, 8, 16, 2, 32), kernel=(3, 5, 5)):
    return lib.na3d_fwd(*[ctypes.c_void_p(p) for p in ptrs], *dims, *kernel, None)


@pytest.mark.parametrize("dims,kernel,code", [
    ((1, 0, 8, 16, 2, 32), (1, 5, 5), ERR_SHAPE),
    ((-1, 4, 8, 16, 2, 32), (3, 5, 5), ERR_SHAPE),
    ((1, 4, 8, 16, -2, 32), (3, 5, 5), ERR_SHAPE),
    ((1, 4, 8, 16, 2, 32), (2, 5, 5), ERR_KERNEL),      # even
    ((1, 4, 8, 16, 2, 32), (5, 5, 5), ERR_KERNEL),      # KT > T
    ((1, 4, 8, 16, 2, 32), (3, 5, 0), ERR_KERNEL),
    ((1, 4, 8, 16, 2, 32), (3, 9, 5), ERR_KERNEL),      # KH > H
    ((1, 4, 8, 16, 2, 48), (3, 5, 5), ERR_HEAD_DIM),
    ((1, 4, 8, 16, 2, 8), (3, 5, 5), ERR_HEAD_DIM),
    ((1, 4, 8, 16, 1 << 22, 512), (3, 5, 5), ERR_OVERFLOW),   # NH * HD = 2^31 columns
    ((1 << 40, 4, 8, 16, 2, 32), (3, 5, 5), ERR_OVERFLOW),
])
def test_shape_validation(lib, dims, kernel, code):
    ptrs = (1 << 20, 2 << 20, 3 << 20, 4 << 30)
    assert call_fwd(lib, ptrs, dims, kernel) == code


def test_pointer_validation(lib):
    assert call_fwd(lib, (0, 32, 48, 64)) == ERR_NULL
    assert call_fwd(lib, (16, 32, 48, 0)) == ERR_NULL
    assert call_fwd(lib, (16, 40, 64, 1 << 30)) == ERR_ALIGN
    n_bytes = 1 * 4 * 8 * 16 * 2 * 32 * 2
    base = 1 << 20
    assert call_fwd(lib, (base, base + n_bytes, base + 2 * n_bytes, base + n_bytes - 16)) == ERR_ALIAS
    # q, k, v may alias one another
    assert call_fwd(lib, (base, base, base, base + n_bytes)) not in (ERR_ALIAS, ERR_NULL, ERR_ALIGN)


def call_strided(lib, ptrs, strides, dims=(1, 4, 8, 16, 2, 32), kernel=(3, 5, 5)):
    return lib.na3d_fwd_strided(*[ctypes.c_void_p(p) for p in ptrs], *dims, *kernel, *strides, None)


def test_strided_validation(lib):
    nhd = 2 * 32
    base = 1 << 20
    ok = (base, base + 2 * nhd, base + 4 * nhd, 1 << 30)
    # a fused [.., 3, NH, HD] layout passes validation (fails later only for want of a GPU)
    import torch
    expect = OK if torch.cuda.is_available() else ERR_CUDA
    assert call_strided(lib, ok, (3 * nhd, 3 * nhd, 3 * nhd)) == expect
    assert call_strided(lib, ok, (nhd - 8, 3 * nhd, 3 * nhd)) == ERR_SHAPE
    assert call_strided(lib, ok, (3 * nhd + 4, 3 * nhd, 3 * nhd)) == ERR_ALIGN
    # out overlapping the strided span of v
    n_tokens = 4 * 8 * 16
    inside_v = base + 4 * nhd + 2 * (3 * nhd) * (n_tokens // 2)
    assert call_strided(lib, (base, base + 2 * nhd, base + 4 * nhd, inside_v - inside_v % 16),
                        (3 * nhd,) * 3) == ERR_ALIAS


def call_region(lib, ptrs, box, dims=(1, 4, 8, 16, 2, 32), kernel=(3, 5, 5), strides=None):
    nhd = dims[4] * dims[5]
    strides = strides or (nhd, nhd, nhd)
    return lib.na3d_fwd_region(*[ctypes.c_void_p(p) for p in ptrs], *dims, *kernel, *box,
                               *strides, None)


def test_region_validation(lib):
    """The query box (t0, h0, w0, Tq, Hq, Wq) must lie inside the grid."""
    import torch
    expect = OK if torch.cuda.is_available() else ERR_CUDA
    base = 1 << 20
    ptrs = (base, base + (1 << 22), base + (2 << 22), base + (3 << 22))
    T, H, W = 4, 8, 16
    assert call_region(lib, ptrs, (0, 0, 0, T, H, W)) == expect          # the whole grid
    assert call_region(lib, ptrs, (1, 2, 9, 2, 5, 7)) == expect          # an interior box
    assert call_region(lib, ptrs, (0, 0, 12, T, H, 2)) == expect         # narrower than KW
    for box in [(0, 0, 10, T, H, 7), (1, 0, 0, T, H, W), (-1, 0, 0, 2, H, W), (0, 0, 0, 0, H, W),
                (0, 8, 0, T, 1, W), (0, 0, 0, T, H, 17)]:
        assert call_region(lib, ptrs, box) == ERR_SHAPE, box
    # the window is checked against the grid, not the box
    assert call_region(lib, ptrs, (0, 0, 0, T, H, 3), kernel=(3, 5, 17)) == ERR_KERNEL
    # an empty batch is a size below 1
    assert call_region(lib, ptrs, (0, 0, 4, T, H, 4), dims=(0, T, H, W, 2, 32)) == ERR_SHAPE
    # out overlapping k, which spans the whole grid
    n_kv = 1 * T * H * W * 2 * 32 * 2
    assert call_region(lib, (base, base + (1 << 22), base + (2 << 22), base + (1 << 22) + n_kv // 2),
                       (0, 0, 0, 2, 2, 2)) == ERR_ALIAS


def test_qkv_proj_validation(lib):
    import torch
    expect = OK if torch.cuda.is_available() else ERR_CUDA
    base = 1 << 20
    x, w, qkv = base, base + (1 << 24), base + (2 << 24)
    P = ctypes.c_void_p
    call = lambda x_, w_, b_, o_, M, C, NH, HD: lib.na3d_qkv_proj(P(x_), P(w_), P(b_), P(o_), M, C,  # noqa: E731
                                                                    NH, HD, None)
    assert call(x, w, None, qkv, 1000, 64, 2, 32) == expect
    assert call(x, w, None, qkv, 1000, 60, 2, 32) == ERR_ALIGN    # rows of 120 bytes
    assert call(x, w, None, qkv, 1000, 64, 2, 48) == ERR_HEAD_DIM
    assert call(x, w, None, qkv, -1, 64, 2, 32) == ERR_SHAPE
    assert call(x, w, None, qkv, 0, 64, 2, 32) == ERR_SHAPE          # no tokens
    assert call(x, w, None, qkv, 10, 64, 0, 32) == ERR_SHAPE         # no heads
    assert call(0, w, None, qkv, 10, 64, 2, 32) == ERR_NULL
    assert call(x + 8, w, None, qkv, 10, 64, 2, 32) == ERR_ALIGN
    assert call(x, w, None, x + 64, 10, 64, 2, 32) == ERR_ALIAS   # qkv over x
    assert call(x, w, qkv + 64, qkv, 10, 64, 2, 32) == ERR_ALIAS  # bias inside qkv


@pytest.mark.parametrize("shape,kernel,cap,stride", INSTANCE_CASES + [
    ((1, 16, 48, 48, 8, 64), (11, 11, 11), 128, 14),
])
def test_each_instance_is_selected_by_its_problem(lib, shape, kernel, cap, stride):
    """The problems the GPU parity tests use to exercise each kernel instance
    do select that instance (score-tile cap and W row stride)."""
    p = na.na3d_plan(*shape[1:], *kernel)
    assert (p["tile_cap"], p["w_stride"]) == (cap, stride)
    if stride not in (0, 1):
        assert p["cw"] == stride


@pytest.mark.parametrize("grid,kernel,cap,brick", [
    ((16, 64, 96), (3, 5, 5), 96, (4, 8, 4)),      # same plan in both families: paired tiles
    ((36, 64, 96), (3, 5, 5), 96, (4, 8, 4)),
    ((16, 64, 64), (3, 7, 7), 128, (2, 8, 8)),     # the 96-key cap would force 2x10x6 bricks
    ((16, 48, 48), (11, 11, 11), 128, (4, 8, 4)),  # ... or 16x4x2 bricks
    ((16, 32, 32), (7, 7, 7), 128, (8, 8, 2)),
    ((4, 8, 128), (3, 5, 27), 128, (4, 8, 4)),     # ... or 3 rows of 32 keys instead of 4
])
def test_paired_tiles_only_where_they_keep_the_plan(lib, grid, kernel, cap, brick):
    """HD 64: the 96-key paired family is chosen when its plan costs no more
    than the 128-key family's (the same plan runs faster on paired tiles; a
    plan the smaller cap forces measured slower)."""
    p = na.na3d_plan(*grid, 8, 64, *kernel)
    assert p["tile_cap"] == cap
    assert (p["bt"], p["bh"], p["bw"]) == brick


def test_every_power_of_two_head_dim_is_planned(lib):
    """HD > 256 is served by one wide instance: 64-key tiles, 64-column boxes."""
    for hd in (512, 1024, 2048, 4096):
        p = na.na3d_plan(4, 8, 16, 2, hd, 3, 5, 5)
        assert p["hd_box"] == 64 and p["n_mma"] <= 64


def test_empty_problem_is_rejected(lib):
    """Every size must be at least 1: an empty batch or no heads is a shape
    error, returned before the pointers are looked at."""
    assert call_fwd(lib, (16, 32, 48, 64), dims=(0, 4, 8, 16, 2, 32)) == ERR_SHAPE
    assert call_fwd(lib, (16, 32, 48, 64), dims=(1, 4, 8, 16, 0, 32)) == ERR_SHAPE
    assert call_fwd(lib, (0, 0, 0, 0), dims=(0, 4, 8, 16, 2, 32)) == ERR_SHAPE
    info = na.PlanInfo()
    assert lib.na3d_plan(4, 8, 16, 0, 32, 3, 5, 5, ctypes.byref(info)) == ERR_SHAPE


def test_valid_call_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    n_bytes = 1 * 4 * 8 * 16 * 2 * 32 * 2
    base = 1 << 20
    rc = call_fwd(lib, (base, base + n_bytes, base + 2 * n_bytes, base + 3 * n_bytes))
    assert rc == ERR_CUDA


def test_binding_requires_cuda_bf16_tensors():
    import torch
    x = torch.zeros(1, 4, 8, 16, 2, 32, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        na.na3d_fwd(x, x, x, x.clone(), (3, 5, 5))


# ------------------------------------------------------------------ planner

def nearest_centre_starts(N, K):
    s = np.arange(N - K + 1)
    return np.array([s[np.argmin(np.abs(s + (K - 1) / 2.0 - i))] for i in range(N)])


def check_plan_covers_windows(T, H, W, HD, kernel):
    """Every key of every query's window lies in one of its brick's chunks;
    chunks stay inside the TMA limits; the score tile fits its cap. The
    chunk enumeration is the kernel's: frames of the brick's window union,
    then groups of cr rows, then segments of cw keys, from the union's start."""
    KT, KH, KW = kernel
    p = na.na3d_plan(T, H, W, 1, HD, *kernel)
    bt, bh, bw, cw, cr = p["bt"], p["bh"], p["bw"], p["cw"], p["cr"]
    ncap = p["tile_cap"]
    assert ncap == (64 if HD >= 128 else 128) or (HD <= 64 and ncap == 96)
    assert 1 <= bt * bh * bw <= 128
    assert cr * cw <= ncap and p["n_mma"] % 16 == 0 and cr * cw <= p["n_mma"] <= ncap
    assert max(bt, bh, bw, cw, cr) <= 256
    starts = [nearest_centre_starts(N, K) for N, K in ((T, KT), (H, KH), (W, KW))]
    total_chunks = 0
    for t0 in range(0, T, bt):
        for h0 in range(0, H, bh):
            for w0 in range(0, W, bw):
                qs = [np.arange(o, min(o + b, N)) for o, b, N in ((t0, bt, T), (h0, bh, H), (w0, bw, W))]
                lo = [starts[a][qs[a][0]] for a in range(3)]
                hi = [starts[a][qs[a][-1]] + kernel[a] for a in range(3)]
                n_hc = -(-(hi[1] - lo[1]) // cr)
                n_wc = -(-(hi[2] - lo[2]) // cw)
                if p["w_stride"] == 1:
                    # whole-row W windows: one W segment, and the halo's rows
                    # (chunk padding included) fit the 15 row-mask columns
                    # and the 5 per-h-chunk mask tiles
                    assert KW == W and cw == W and n_wc == 1
                    assert n_hc * cr <= 15 and n_hc <= 5
                total_chunks += (hi[0] - lo[0]) * n_hc * n_wc
                cov_h = set()
                for hc in range(n_hc):
                    cov_h |= set(range(lo[1] + hc * cr, lo[1] + hc * cr + cr))
                cov_w = set()
                for wc in range(n_wc):
                    cov_w |= set(range(lo[2] + wc * cw, lo[2] + wc * cw + cw))
                for a, cov in ((1, cov_h), (2, cov_w)):
                    for i in qs[a]:
                        assert set(range(starts[a][i], starts[a][i] + kernel[a])) <= cov
                for i in qs[0]:
                    assert lo[0] <= starts[0][i] and starts[0][i] + KT <= hi[0]
    assert total_chunks == p["chunks_per_slice"]


@pytest.mark.parametrize("T,H,W,HD,kernel", [
    (4, 8, 16, 32, (3, 5, 5)),
    (16, 64, 64, 64, (3, 7, 7)),
    (16, 64, 96, 64, (3, 5, 5)),
    (16, 64, 5, 64, (3, 5, 5)),
    (16, 48, 48, 64, (11, 11, 11)),
    (16, 96, 128, 128, (3, 7, 7)),
    (8, 64, 33, 64, (3, 7, 33)),
    (5, 7, 200, 256, (3, 3, 161)),
    (6, 9, 20, 512, (3, 5, 7)),
    (3, 6, 40, 1024, (3, 3, 33)),
    (7, 40, 17, 64, (5, 11, 17)),
    (6, 30, 1, 64, (3, 5, 1)),
    (8, 64, 33, 128, (3, 7, 33)),
    (1, 1, 9, 16, (1, 1, 9)),
    (9, 1, 1, 16, (5, 1, 1)),
])
def test_plan_covers_every_window(lib, T, H, W, HD, kernel):
    check_plan_covers_windows(T, H, W, HD, kernel)


def test_plan_random_sweep(lib):
    rng = np.random.default_rng(1)
    for _ in range(40):
        T, H, W = (int(x) for x in rng.integers(1, 40, size=3))
        kernel = tuple(int(rng.choice(np.arange(1, n + 1, 2))) for n in (T, H, W))
        HD = int(rng.choice([16, 32, 64, 128, 256, 512, 2048]))
        check_plan_covers_windows(T, H, W, HD, kernel)
