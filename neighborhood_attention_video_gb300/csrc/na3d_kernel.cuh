// Host/device interface between the NA3D launcher and its kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace na3d {

// Division by a runtime constant for dividends below 2^31: q = (n * mul) >> shift
// with mul = floor(2^shift / d) + 1 and shift = 31 + ceil(log2 d), which is
// exact for every 0 <= n < 2^31 (Granlund & Montgomery, PLDI 1994, sec. 4).
struct FastDiv {
    uint64_t mul;
    uint32_t shift;
    int32_t d;
};

inline FastDiv make_fastdiv(int32_t d) {
    uint32_t l = 0;
    while ((int64_t(1) << l) < d) ++l;
    FastDiv f;
    f.shift = 31 + l;
    f.mul = ((uint64_t(1) << f.shift) / uint64_t(d)) + 1;
    f.d = d;
    return f;
}

// Everything the kernel needs besides the three TMA descriptors.
struct KernelParams {
    int32_t B, T, H, W, NH;          // key/value grid
    int32_t Tq, Hq, Wq;              // query box extents (the whole grid unless a region is given)
    int32_t t_off, h_off, w_off;     // query box origin in the grid
    int32_t KT, KH, KW;
    int32_t bt, bh, bw;      // query brick
    int32_t nbt, nbh, nbw;   // bricks per axis of the query box
    int32_t cw, cr, n_mma;   // chunk geometry and score-tile width
    int32_t n_units;         // B * nbt * nbh * nbw * NH (head fastest)
    int32_t hg;              // heads per group (a power of two dividing NH): a CTA runs the
                             // hg heads of one brick back to back (1 for HD < 128); for
                             // HD > 256 a "head" here is one (head, pass) pair
    int32_t hd;              // head dimension (the instance's own unless HD > 256)
    int32_t nreg;            // HD > 256: 64-column regions of a head (HD / 64)
    int32_t npass_log2;      // HD > 256: log2 of the passes over 256 output columns
    uint16_t* out;           // bf16 output, (B,Tq,Hq,Wq,NH,HD)
    int32_t out_v8;          // 1: out is 32-byte aligned (32-byte stores), 0: 16-byte stores
    int32_t withhold_k;      // self-test: CTA 0 skips its K load number withhold_k (-1: none)
    FastDiv div_nh, div_nbw, div_nbh, div_nbt;   // unit index decomposition
    FastDiv div_cr, div_cw;                      // chunks per halo row group / W segment
};

// Compile-time shape of one kernel instance, as the planner needs it.
struct VariantInfo {
    int ncap;      // max keys per chunk (score-tile width cap)
    int stages;    // K/V pipeline depth
    int hd_box;    // head-dim columns per TMA box
    int smem;      // dynamic shared memory bytes
    int ctas_per_sm;  // resident CTAs per SM the instance is sized for
};

// Instances exist for HD in {16, 32, 64, 128, 256, >= 512 (one instance for
// every larger power of two)}, chunk stride cwp in {0 (generic per-key masks),
// 8, 12, 14, 16, 32 (W window applied by the tensor core), 1 (H window applied
// by the tensor core)} and score-tile cap ncap (default_ncap(hd), and 96 for
// HD 64: paired tiles). info may be null: then only whether it exists.
int default_ncap(int hd);
bool variant_info(int hd, int cwp, int ncap, VariantInfo* info);

// Launch the instance for (hd, cwp, ncap) on `stream` with `grid` persistent CTAs.
cudaError_t launch_fwd(int hd, int cwp, int ncap, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const KernelParams& kp, int grid,
                       cudaStream_t stream);

// After the work already on `stream`, take (read and clear in one atomic
// step) the timeout flag of the current device, then synchronize `stream`.
cudaError_t take_device_error(cudaStream_t stream, unsigned int* flag);

}  // namespace na3d
