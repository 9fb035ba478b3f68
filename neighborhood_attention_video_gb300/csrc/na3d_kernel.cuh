// Host/device interface between the NA3D launcher and its kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace na3d {

// Everything the kernel needs besides the three TMA descriptors.
struct KernelParams {
    int32_t B, T, H, W, NH;
    int32_t KT, KH, KW;
    int32_t bt, bh, bw;      // query brick
    int32_t nbt, nbh, nbw;   // bricks per axis
    int32_t cw, cr, n_mma;   // chunk geometry and score-tile width
    int32_t n_units;         // B * nbt * nbh * nbw * NH
    uint16_t* out;           // bf16 output, (B,T,H,W,NH,HD)
};

// Compile-time shape of one kernel instance, as the planner needs it.
struct VariantInfo {
    int ncap;      // max keys per chunk (score-tile width cap)
    int stages;    // K/V pipeline depth
    int hd_box;    // head-dim columns per TMA box
    int smem;      // dynamic shared memory bytes
    int ctas_per_sm;  // resident CTAs per SM the instance is sized for
};

bool variant_info(int hd, VariantInfo* info);

// Launch the instance for `hd` on `stream` with `grid` persistent CTAs.
cudaError_t launch_fwd(int hd, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const KernelParams& kp, int grid,
                       cudaStream_t stream);

// Read (and clear) the device-side timeout flag of the current device.
cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* flag);

}  // namespace na3d
