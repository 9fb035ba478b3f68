// Host/device interface of the QKV projection kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace na3d {

struct ProjParams {
    int32_t M;          // tokens (rows of x and qkv)
    int32_t C;          // input channels (contraction length)
    int32_t N;          // output columns, 3 * NH * HD
    int32_t Nq;         // columns of the q block, NH * HD (scaled by q_scale)
    int32_t n_tiles_n;  // ceil(N / 256)
    int32_t n_tiles;    // ceil(M / 128) * n_tiles_n
    int32_t k_blocks;   // ceil(C / 64)
    int32_t out_v8;     // 1: qkv is 32-byte aligned (32-byte stores)
    float q_scale;      // HD^-0.5 rounded to fp32
    const uint16_t* bias;   // bf16 [N] or null
    uint16_t* qkv;          // bf16 [M][N]
};

// Launch the persistent projection kernel with `grid` CTAs (one per SM).
cudaError_t launch_qkv_proj(const CUtensorMap& tx, const CUtensorMap& tw, const ProjParams& pp,
                            int grid, cudaStream_t stream);

// After the work already on `stream`, take (read and clear in one atomic
// step) the projection kernel's timeout flag, then synchronize `stream`.
cudaError_t take_proj_error(cudaStream_t stream, unsigned int* flag);

}  // namespace na3d
