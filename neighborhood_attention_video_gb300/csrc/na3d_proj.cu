// QKV projection on GB300 (sm_103a): qkv = x W^T (+ bias), q block scaled.
//
// The producer of the attention inputs ("LTX-2.5 optimization: integrate
// faster AITER NA3D flash attention for diffusion decoder", xDiT pull request
// 773, Summary and Notes: one concatenated Q/K/V weight, q, k and v are views
// of its output). The output row of a token holds its q, k and v heads in the
// layout na3d_fwd_strided reads with a token stride of 3 * NH * HD, and the q
// block is multiplied by HD^-0.5 before the single rounding to bf16, as the
// attention expects ("[Triton/Gluon] Add 3D neighborhood flash attention
// (na3d_flash)", Technical Details, launcher).
//
// A persistent, warp-specialised tcgen05 GEMM, one CTA per SM:
//   warps 0..3  epilogue: one output row per thread (its TMEM lane): fp32
//               accumulator + bias (staged per tile in shared memory, read
//               as broadcasts), q scale, bf16, 32-byte stores;
//   warp 4      TMA producer: 128 x 64 tiles of x and 256 x 64 tiles of W into
//               a ring of four stages;
//   warp 5      MMA issuer (M = 128, N = 256, K = 16), owns the tensor memory.
// Output tiles are 128 x 256 with two TMEM accumulators (2 x 256 columns),
// so a tile's epilogue overlaps the next tile's MMAs. Tiles run N-fastest:
// CTAs working at the same time share the x tile through L2, and W stays in
// L2. Every wait is bounded as in the attention kernel.
#include <atomic>
#include "na3d_proj.cuh"
#include "sm103_ptx.cuh"

namespace na3d {

__device__ unsigned int g_proj_timeout_flag = 0;

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 256;
constexpr int A_TILE = kBM * kBK * 2;   // 16 KB, 128-byte rows, 128-byte swizzle
constexpr int B_TILE = kBN * kBK * 2;   // 32 KB
constexpr int STAGE = A_TILE + B_TILE;
constexpr int OFF_BAR = kStages * STAGE;
constexpr int B_FULL = 0, B_EMPTY = kStages, B_AFULL = 2 * kStages, B_AEMPTY = B_AFULL + 2,
              B_DRAIN = B_AEMPTY + 2, NBAR = B_DRAIN + 1;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_BIAS = (OFF_MISC + 16 + 15) & ~15;   // per epilogue warp: the tile's bias, fp32
constexpr int SMEM_ALLOC = OFF_BIAS + 4 * kBN * 4 + 1024;
constexpr uint32_t TM_COLS = 512;   // two 256-column accumulators
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 500000000ull;

struct Sync {
    uint32_t bar0;
    volatile uint32_t* abort_flag;
    __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * i; }
    // Wait for a barrier phase; false once this CTA has given up.
    __device__ __forceinline__ bool wait(uint32_t b, uint32_t parity) const {
        if (mbar_try_wait(b, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait(b, parity)) return true;
            if ((it & 1023u) == 0u) {
                if (*abort_flag) return false;
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    *abort_flag = 1u;
                    atomicOr(&g_proj_timeout_flag, 1u);
                    return false;
                }
            }
        }
    }
};

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
qkv_proj_sm103(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
               const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(base_ptr + OFF_MISC);
    Sync sy{base + OFF_BAR, misc + 1};
    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i)
            mbar_init(sy.bar(i), (i >= B_AEMPTY && i < B_AEMPTY + 2) ? 128u : 1u);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 5) {
        tmem_alloc(base + OFF_MISC, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 4 && lane == 0) {
        // ---------------------------------------------------------- producer
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.n_tiles; t += gridDim.x) {
            const int m0 = (t / p.n_tiles_n) * kBM, n0 = (t % p.n_tiles_n) * kBN;
            for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
                const uint32_t st = it % kStages;
                if (!sy.wait(sy.bar(B_EMPTY + st), ((it / kStages) & 1u) ^ 1u)) { ok = false; break; }
                const uint32_t full = sy.bar(B_FULL + st);
                mbar_arrive_expect_tx(full, STAGE);
                tma_load_2d(base + st * STAGE, &tm_x, full, kb * kBK, m0);
                tma_load_2d(base + st * STAGE + A_TILE, &tm_w, full, kb * kBK, n0);
            }
        }
        // every issued load lands before the CTA may exit
        for (uint32_t s = 0; s < kStages; ++s) {
            const uint32_t f = it / kStages + (s < it % kStages ? 1u : 0u);
            if (f && !mbar_wait_bounded(sy.bar(B_FULL + s), (f - 1u) & 1u, kDrainLimitNs))
                atomicOr(&g_proj_timeout_flag, 1u);
        }
    } else if (warp == 5 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        const uint32_t idesc = make_idesc_bf16(kBM, kBN, 0, 0);
        const uint64_t ad0 = make_smem_desc(base, 16, 1024, kSwizzle128B);
        const uint64_t bd0 = make_smem_desc(base + A_TILE, 16, 1024, kSwizzle128B);
        const uint32_t a_hi = static_cast<uint32_t>(ad0 >> 32), b_hi = static_cast<uint32_t>(bd0 >> 32);
        uint32_t it = 0, lt = 0;
        for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++lt) {
            const uint32_t buf = lt & 1u;
            // the epilogue has read this accumulator's previous tile
            if (!sy.wait(sy.bar(B_AEMPTY + buf), ((lt >> 1) & 1u) ^ 1u)) break;
            tc_fence_after();
            const uint32_t d = tmem + buf * kBN;
            bool ok = true;
            for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
                const uint32_t st = it % kStages;
                if (!sy.wait(sy.bar(B_FULL + st), (it / kStages) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a_lo = static_cast<uint32_t>(ad0) + ((st * STAGE) >> 4);
                const uint32_t b_lo = static_cast<uint32_t>(bd0) + ((st * STAGE) >> 4);
                // K = 16 per MMA: 32 bytes further along the swizzled 128-byte rows
                if (kb == 0) umma_ss_halves<0>(d, a_lo, a_hi, b_lo, b_hi, idesc);
                else umma_ss_halves<1>(d, a_lo, a_hi, b_lo, b_hi, idesc);
                umma_ss_halves<1>(d, a_lo + 2, a_hi, b_lo + 2, b_hi, idesc);
                umma_ss_halves<1>(d, a_lo + 4, a_hi, b_lo + 4, b_hi, idesc);
                umma_ss_halves<1>(d, a_lo + 6, a_hi, b_lo + 6, b_hi, idesc);
                umma_commit(sy.bar(B_EMPTY + st));
            }
            if (!ok) break;
            umma_commit(sy.bar(B_AFULL + buf));
        }
        umma_commit(sy.bar(B_DRAIN));
        if (!mbar_wait_bounded(sy.bar(B_DRAIN), 0, kDrainLimitNs)) atomicOr(&g_proj_timeout_flag, 1u);
    } else if (warp < 4) {
        // ---------------------------------------------------------- epilogue
        const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float* bias_s = reinterpret_cast<float*>(base_ptr + OFF_BIAS) + warp * kBN;   // this warp's copy
        const uint32_t bias_addr = smem_u32(bias_s);
        uint32_t lt = 0;
        for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++lt) {
            const uint32_t buf = lt & 1u;
            if (!sy.wait(sy.bar(B_AFULL + buf), (lt >> 1) & 1u)) break;
            tc_fence_after();
            const int m0 = (t / p.n_tiles_n) * kBM, n0 = (t % p.n_tiles_n) * kBN;
            const int row = m0 + warp * 32 + lane;
            uint16_t* orow = p.qkv + static_cast<int64_t>(row) * p.N;
            // the tile's bias (0 past N or without bias), one coalesced pass per warp
#pragma unroll
            for (int i = 0; i < kBN / 32; ++i) {
                const int c = n0 + 32 * i + lane;
                bias_s[32 * i + lane] = (p.bias && c < p.N) ? bf16_to_f32(p.bias[c]) : 0.f;
            }
            __syncwarp();
#pragma unroll 1
            for (int q = 0; q < kBN / 32; ++q) {
                const int c0 = n0 + 32 * q;
                if (c0 >= p.N) break;   // ragged last tile (uniform over the CTA)
                float acc[32];
                tmem_ld32(t_row + buf * kBN + 32 * q, acc);
                tmem_wait_ld();
                float bv[32];   // bias of these 32 columns: same address in every lane
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(bv[4 * i]), "=f"(bv[4 * i + 1]), "=f"(bv[4 * i + 2]), "=f"(bv[4 * i + 3])
                                 : "r"(bias_addr + (32 * q + 4 * i) * 4));
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c0 + 2 * j;   // columns c, c + 1
                    float v0 = acc[2 * j] + bv[2 * j], v1 = acc[2 * j + 1] + bv[2 * j + 1];
                    // the q block (columns below NH * HD) carries the HD^-0.5 scale
                    v0 *= c < p.Nq ? p.q_scale : 1.f;
                    v1 *= c + 1 < p.Nq ? p.q_scale : 1.f;
                    pk[j] = pack_bf16x2(v0, v1);
                }
                if (row < p.M) {
                    const int nval = p.N - c0 >= 32 ? 32 : p.N - c0;   // a multiple of 16
                    if (p.out_v8) {
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            if (16 * i < nval) st_global_v8(orow + c0 + 16 * i, pk + 8 * i);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (8 * i < nval)
                                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
            __syncwarp();   // the bias copy is rewritten for the next tile
            tc_fence_before();
            mbar_arrive(sy.bar(B_AEMPTY + buf));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

cudaError_t launch_qkv_proj(const CUtensorMap& tx, const CUtensorMap& tw, const ProjParams& pp,
                            int grid, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(qkv_proj_sm103, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    qkv_proj_sm103<<<grid, kThreads, SMEM_ALLOC, stream>>>(tx, tw, pp);
    return cudaGetLastError();
}

// The flag is taken as for the attention kernel: one atomic exchange per
// status request, its old value left in a slot of that request's own.
constexpr unsigned int kStatusSlots = 256;
__device__ unsigned int g_proj_status_slots[kStatusSlots];

__global__ void take_proj_flag(unsigned int slot) {
    g_proj_status_slots[slot] = atomicExch(&g_proj_timeout_flag, 0u);
}

cudaError_t take_proj_error(cudaStream_t stream, unsigned int* flag) {
    static std::atomic<unsigned int> next{0};
    const unsigned int slot = next.fetch_add(1u) % kStatusSlots;
    take_proj_flag<<<1, 1, 0, stream>>>(slot);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbolAsync(flag, g_proj_status_slots, sizeof(unsigned int),
                                  slot * sizeof(unsigned int), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace na3d
