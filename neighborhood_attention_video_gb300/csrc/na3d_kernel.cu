// NA3D forward on GB300 (sm_103a): persistent, warp-specialised kernel.
//
// The operation ("[Triton/Gluon] Add 3D neighborhood flash attention
// (na3d_flash)", ROCm/aiter pull request 5230, Motivation and Technical
// Details): each query (t,h,w) of a (B,T,H,W,NH,HD) bf16 tensor attends to the
// KT x KH x KW keys of its inward-shifted window; q is pre-scaled; the softmax
// is online and runs in log2 space with the log2(e) factor folded into the
// exponent; the output is bf16 in the input layout.
//
// Work decomposition. One work unit is one query brick (bt x bh x bw <= 128
// grid positions of the query box, which is the whole grid unless a region is
// given) of one (batch, head). Its keys are the union of its queries' windows
// (the halo, in grid coordinates), a box that is streamed through shared
// memory in chunks: a chunk is cr consecutive rows (h) of cw consecutive keys
// (w) in one frame (t), loaded with one TMA box per 64 head-dim columns.
// Queries are the M = 128 rows of every tensor-core tile; a chunk's keys are
// its N columns. Persistent CTAs take units round-robin; for HD >= 128 a CTA
// takes the heads of one brick back to back (see next_unit).
//
// Roles (256 threads; two CTAs per SM for HD <= 128, one for HD = 256):
//   warps 0..3  softmax (warpgroup 0): one query row per thread (its TMEM
//               lane): window mask, running max and sum in log2 space, P as
//               bf16 into tensor memory, occasional O rescale, and the
//               epilogue O / l -> bf16 -> HBM.
//   warp 4      TMA producer: the Q brick once per unit; K and V of each chunk
//               into rings of NS stages with separate barriers, K one chunk
//               ahead of V.
//   warp 5      score issuer: S = Q K^T (+ the W-mask block) into the TMEM
//               score tile, one chunk ahead; owns the tensor-memory allocation.
//   warp 6      product issuer: O += P V with P read from tensor memory.
//   warp 7      idle (it completes warpgroup 1 for the register hand-over).
//
// Tensor memory per CTA: O (HD fp32 columns) and a ring of NSLOT slots of
// NCAP/2 columns. A score tile S (NCAP fp32 columns) takes two consecutive
// slots; once the softmax has read it into registers, it writes P (NCAP/2
// columns of bf16 pairs) over the first of them and the second is free. So the
// next score tile is computed while the softmax works on the current one, and
// the softmax never waits for the previous product: P(g) and P(g-1) sit in
// different slots. A score tile waits only for the product that last read its
// slots, LAG chunks back. With three slots the ring wraps every third chunk;
// that tile is issued as two halves.
//
// Every pipeline wait is bounded: a wait that runs out sets a device flag, all
// roles drop out of their loops, in-flight copies and MMAs are drained, and
// the tensor memory is freed before the CTA exits.
#include <cuda_bf16.h>

#include <atomic>

#include "na3d_kernel.cuh"
#include "sm103_ptx.cuh"

namespace na3d {

__device__ unsigned int g_na3d_timeout_flag = 0;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 500000000ull;
constexpr float kLog2e = 1.4426950408889634f;
// When the maximum is recomputed, the reference maximum (log2 units) is raised
// only if the chunk's maximum exceeds it by more than this, so the O rescale
// (a TMEM round trip) stays rare.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kSumLimit = 4294967296.0f;  // 2^32: bound on one chunk's probability sum
constexpr int kThreads = 256;

// bf16 -2^40: the score offset that masks a key through the extra
// contraction block (exact: valid keys get +0, masked ones vanish in exp2).
constexpr uint16_t kMaskBf16 = 0xD380u;

template <int HD_, int NCAP_, int NS_, int CPS_, int CWP_>
struct Cfg {
    static constexpr int HD = HD_, NCAP = NCAP_, NS = NS_, CPS = CPS_, CWP = CWP_;
    // CWP > 1: chunk rows have a fixed stride of CWP keys and the W window is
    // applied by the tensor core (extra contraction block Qx Kx^T); CWP == 0:
    // per-element window masks in the softmax (any chunk geometry).
    // CWP == 1 (ROWS): every W window is the whole axis (KW = W), chunk rows
    // are whole grid rows, and the tensor core applies the H window instead:
    // Kx marks each key's row within the brick's halo (one Kx tile per h-chunk
    // index), Qx marks the halo rows outside each query's H window.
    static constexpr bool FAST = CWP > 0;
    static constexpr bool ROWS = CWP == 1;
    // CWP 12 or 14: chunk rows of CWP keys that do not tile a 32-key word
    // (exact fits of 11- to 14-key W unions, instead of padding them to 16)
    static constexpr bool ODD = FAST && !ROWS && (CWP & (CWP - 1)) != 0;
    // softmax: columns per uniformly masked group (ROWS: 16, so that the
    // validity bits end at the tile width, a multiple of 16)
    static constexpr int RW = ROWS ? 16 : CWP;
    static constexpr int NKX = ROWS ? 5 : 1;        // Kx tiles (ROWS: one per h-chunk index)
    static constexpr int XDEAD = 15;                // ROWS: the Kx column of padding keys
    // WIDE (HD > 256): O of a whole row does not fit in tensor memory next to
    // the score tiles. A work unit then computes one block of OB output
    // columns (a "pass"; the head's NPASS passes are consecutive units), and
    // the score contraction streams Q and K through one ring, one 64-column
    // region of each per stage, instead of keeping the Q brick resident. Every
    // pass recomputes the same scores (same MMA sequence, same probabilities).
    // The one WIDE instance (HD = 512) serves every HD >= 512: the head size,
    // its region count and its pass count come from the kernel parameters.
    static constexpr bool WIDE = HD > 256;
    static constexpr int OB = WIDE ? 256 : HD;      // output columns of a unit
    static constexpr int KEXT = FAST ? (CWP < 16 ? 16 : CWP) : 0;   // extra contraction columns (ROWS: 16)
    static constexpr int XROWB = KEXT * 2;
    static constexpr uint32_t XSWZ = KEXT == 32 ? kSwizzle64B : kSwizzle32B;
    static constexpr int XSBO = 8 * XROWB;
    static constexpr int QX_TILE = 128 * XROWB;
    static constexpr int KX_TILE = NCAP * XROWB;
    static constexpr int RPW = FAST && !ODD ? 32 / RW : 0;   // uniformly masked groups per 32-column word
    static constexpr int NROWS = FAST ? (NCAP + RW - 1) / RW : 0;   // groups in a tile
    // bits of the groups with a column in 32-column word q
    static constexpr uint32_t word_rows(int q) {
        return FAST ? ((0xFFFFFFFFu >> (31 - (32 * q + 31) / RW)) >> ((32 * q) / RW)) << ((32 * q) / RW) : 0u;
    }
    static constexpr int HDB = HD < 64 ? HD : 64;   // head-dim columns per TMA box / smem row
    static constexpr int NREG = HD / HDB;           // boxes (smem regions) of a Q or K row (not WIDE)
    static constexpr int VREG = OB / HDB;           // boxes of a V row block (= NREG unless WIDE)
    static constexpr int ROWB = HDB * 2;            // bytes per smem row
    static constexpr uint32_t SWZ = HDB == 64 ? kSwizzle128B : (HDB == 32 ? kSwizzle64B : kSwizzle32B);
    static constexpr int SBO = 8 * ROWB;            // stride between 8-row core groups
    static constexpr int Q_REG = 128 * ROWB;
    static constexpr int Q_TILE = WIDE ? 0 : NREG * Q_REG;   // the resident Q brick
    static constexpr int KV_REG = NCAP * ROWB;
    // one K stage: all regions of a chunk's K rows, or (WIDE) one region of the
    // Q brick followed by the same region of the chunk's K rows
    static constexpr int K_TILE = WIDE ? Q_REG + KV_REG : NREG * KV_REG;
    static constexpr int V_TILE = VREG * KV_REG;
    static constexpr int NSV = WIDE ? 2 : NS;       // V stages (K stages: NS)
    static constexpr int NW = NCAP / 32;            // 32-column words per score row
    static constexpr int OPIECES = (OB + 31) / 32;  // 32-column TMEM loads per output row
    static constexpr uint32_t TM_COLS = CPS == 2 ? 256 : 512;
    static constexpr uint32_t TM_O = 0;                              // OB fp32 output columns
    static constexpr uint32_t OCOLS = OPIECES * 32 < 64 ? 64 : OPIECES * 32;
    static constexpr uint32_t SW = NCAP / 2;                         // slot width = P columns
    static constexpr uint32_t TM_R = OCOLS;                          // first ring column
    static constexpr int NSLOT = static_cast<int>((TM_COLS - OCOLS) / SW);
    static constexpr int STEP = NSLOT % 2 == 0 ? 2 : 1;   // slots a chunk advances the ring by
    static constexpr int RING = NSLOT / STEP;             // distinct P slots in rotation
    static constexpr int LAG = STEP == 1 ? NSLOT - 1 : RING;   // S(g) reuses P(g - LAG)'s slot
    // S(g) overwrites columns of S(g - SLAG): with pairs of slots (STEP 2) the
    // next tile goes to other columns and is issued before the softmax has
    // read the current one
    static constexpr int SLAG = STEP == 1 ? 1 : RING;
    // Head groups (several heads of one brick back to back) pay for HD >= 128,
    // where a unit boundary is a large share of a unit; smaller HD keeps the
    // plain round-robin unit order (and its smaller code).
    static constexpr bool GROUPED = HD >= 128;
    // first slot of chunk g's score tile (and of its P)
    static __device__ __forceinline__ uint32_t slot_of(uint32_t g) { return (g * STEP) % NSLOT; }
    // Shared memory: double-buffer Q and Qx where the per-SM share allows it.
    static constexpr int LIMIT = (CPS == 2 ? 115712 : 232448) - 1024 - 512;
    static constexpr int FIXED = NS * K_TILE + NSV * V_TILE + (FAST ? NKX * KX_TILE : 0);
    static constexpr int NQ = WIDE ? 0 : (FIXED + 2 * Q_TILE + (FAST ? 2 * QX_TILE : 0) <= LIMIT ? 2 : 1);
    static constexpr int NQX = !FAST ? 0 : (FIXED + NQ * Q_TILE + 2 * QX_TILE <= LIMIT ? 2 : 1);
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NQ * Q_TILE;
    static constexpr int OFF_V = OFF_K + NS * K_TILE;
    static constexpr int OFF_QX = OFF_V + NSV * V_TILE;
    static constexpr int OFF_KX = OFF_QX + NQX * QX_TILE;
    static constexpr int OFF_BAR = OFF_KX + (FAST ? NKX * KX_TILE : 0);
    // barrier indices
    static constexpr int B_QFULL = 0, B_QEMPTY = NQ;
    static constexpr int B_KFULL = 2 * NQ, B_KEMPTY = B_KFULL + NS;
    static constexpr int B_VFULL = B_KEMPTY + NS, B_VEMPTY = B_VFULL + NSV;
    static constexpr int B_XFULL = B_VEMPTY + NSV, B_XEMPTY = B_XFULL + NQX;
    // For chunk c: S(c) ready, S(c) read, P(c) written and the product of c
    // done are signalled on B_SFULL, B_SEMPTY, B_PFULL and B_PFREE + c % RING:
    // one barrier per ring position, so a softmax warp that runs ahead of the
    // others never completes another chunk's phase, and no waiter ever sees a
    // phase alias (the next use of a barrier needs the current one consumed).
    static constexpr int B_OFULL = B_XEMPTY + NQX, B_OEMPTY = B_OFULL + 1, B_DRAIN = B_OFULL + 2,
                         B_DRAIN2 = B_OFULL + 3, B_SFULL = B_OFULL + 4, B_SEMPTY = B_SFULL + RING,
                         B_PFULL = B_SEMPTY + RING, B_PFREE = B_PFULL + RING, NBAR = B_PFREE + RING;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // The floor keeps the CTA count per SM at CPS (tensor memory is sized for it).
    static constexpr int MIN_SMEM = CPS == 2 ? 80 * 1024 : 120 * 1024;
    static constexpr int SMEM_ALLOC = (SMEM_USED + 1024) > MIN_SMEM ? (SMEM_USED + 1024) : MIN_SMEM;
    // registers: warpgroup 1 gives its share to the softmax warpgroup
    static constexpr uint32_t REGS_LAUNCH = 65536 / (kThreads * CPS) >= 256 ? 255 : 65536 / (kThreads * CPS);
    static constexpr uint32_t REGS_LOW = 56;
    static constexpr uint32_t REGS_HIGH = CPS == 2 ? 200 : 232;
    static_assert(CPS == 1 || (REGS_HIGH + REGS_LOW) * 128 <= REGS_LAUNCH * kThreads, "register split");
    static_assert(TM_COLS * CPS <= 512, "TMEM budget");
    static_assert(NSLOT >= 3 && TM_R + NSLOT * SW <= TM_COLS && OPIECES * 32 <= OCOLS, "TMEM ring");
    static_assert(LAG <= RING, "a product barrier never runs a phase ahead of its waiter");
    static_assert(SMEM_ALLOC * CPS <= 232448 && SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(NCAP == 64 || NCAP == 96 || NCAP == 128, "score tile width");
    static_assert(SW >= 64 || STEP == 2, "pairs of score words are adjacent in tensor memory");
    static_assert(NS >= 2 && NSV >= 2, "K/V rings need two stages");
    static_assert(!FAST || (CWP == 1 || CWP == 8 || CWP == 12 || CWP == 14 || CWP == 16 || CWP == 32),
                  "fast-path chunk stride");
    static_assert(NROWS <= 32, "group bits");
    static_assert(!ROWS || (KEXT == 16 && !WIDE), "row-mask instances");
    static_assert(!WIDE || (CPS == 1 && HDB == 64 && OB == 256 && STEP == 2), "wide instances");
};

// ------------------------------------------------------------------ geometry

__device__ __forceinline__ int win_start(int i, int K, int N) {
    int s = i - (K >> 1);
    s = s < 0 ? 0 : s;
    return s > N - K ? N - K : s;
}

struct Unit {
    int b, n, t0, h0, w0;
    int lo_t, lo_h, lo_w;
    int n_hc, n_wc, nch;
};

// n = q * d + r for 0 <= n < 2^31 (see FastDiv).
__device__ __forceinline__ int fast_divmod(int n, const FastDiv& f, int* r) {
    const int q = static_cast<int>((static_cast<uint64_t>(n) * f.mul) >> f.shift);
    *r = n - q * f.d;
    return q;
}

__device__ __forceinline__ Unit unit_of(const KernelParams& p, int u) {
    Unit U;
    int iw, ih, it;
    u = fast_divmod(u, p.div_nh, &U.n);
    u = fast_divmod(u, p.div_nbw, &iw);
    u = fast_divmod(u, p.div_nbh, &ih);
    U.b = fast_divmod(u, p.div_nbt, &it);
    U.t0 = it * p.bt;   // brick origin in the query box
    U.h0 = ih * p.bh;
    U.w0 = iw * p.bw;
    // halo in grid coordinates: windows of the brick's first and last queries
    U.lo_t = win_start(p.t_off + U.t0, p.KT, p.T);
    U.lo_h = win_start(p.h_off + U.h0, p.KH, p.H);
    U.lo_w = win_start(p.w_off + U.w0, p.KW, p.W);
    const int hi_t = win_start(p.t_off + min(U.t0 + p.bt, p.Tq) - 1, p.KT, p.T) + p.KT;
    const int hi_h = win_start(p.h_off + min(U.h0 + p.bh, p.Hq) - 1, p.KH, p.H) + p.KH;
    const int hi_w = win_start(p.w_off + min(U.w0 + p.bw, p.Wq) - 1, p.KW, p.W) + p.KW;
    int rem;
    U.n_hc = fast_divmod(hi_h - U.lo_h + p.cr - 1, p.div_cr, &rem);
    U.n_wc = fast_divmod(hi_w - U.lo_w + p.cw - 1, p.div_cw, &rem);
    U.nch = (hi_t - U.lo_t) * U.n_hc * U.n_wc;
    return U;
}

// Unit order of a CTA: the hg heads of one brick back to back (one head group),
// then the group gridDim.x groups further on. Neighbouring CTAs work on
// neighbouring bricks at the same head, so their halos meet in L2, and the
// per-brick work (W masks, row set-up) is done once per group.
// Instances without head groups (hg = 1) use u, u + gridDim.x, ...
template <class C>
__device__ __forceinline__ int first_unit(const KernelParams& p) {
    if constexpr (C::GROUPED) return blockIdx.x * p.hg;
    else return blockIdx.x;
}
template <class C>
__device__ __forceinline__ bool group_end(const KernelParams& p, int u) {
    if constexpr (C::GROUPED) return ((u + 1) & (p.hg - 1)) == 0;
    else return true;
}
template <class C>
__device__ __forceinline__ int next_unit(const KernelParams& p, int u) {
    if constexpr (C::GROUPED)
        return group_end<C>(p, u) ? u + 1 + (static_cast<int>(gridDim.x) - 1) * p.hg : u + 1;
    else return u + static_cast<int>(gridDim.x);
}

// The first unit of the head group after the one unit u belongs to.
template <class C>
__device__ __forceinline__ int next_group_unit(const KernelParams& p, int u) {
    if constexpr (C::GROUPED) return (u | (p.hg - 1)) + 1 + (static_cast<int>(gridDim.x) - 1) * p.hg;
    else return u + static_cast<int>(gridDim.x);
}

// Chunk order inside a unit: w-segment fastest, then h-row group, then frame.
struct ChunkCursor {
    int kt, hc, wc;
    __device__ __forceinline__ void advance(const Unit& U) {
        if (++wc == U.n_wc) {
            wc = 0;
            if (++hc == U.n_hc) {
                hc = 0;
                ++kt;
            }
        }
    }
};

// bits [a, b) of a 128-bit mask held in four words (0 <= a, b <= 128)
__device__ __forceinline__ void bit_range128(uint32_t m[4], int a, int b) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const int lo = max(a - 32 * w, 0), hi = min(b - 32 * w, 32);
        m[w] = hi > lo ? static_cast<uint32_t>(((1ull << (hi - lo)) - 1ull) << lo) : 0u;
    }
}

// ------------------------------------------------------------------ waits

// Spin on a barrier phase for at most kWaitLimitNs; on timeout, flag the CTA
// (abort_flag, shared by all roles) and the device (g_na3d_timeout_flag).
__device__ __forceinline__ bool wait_spin(uint32_t b, uint32_t parity, volatile uint32_t* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(b, parity)) return true;
        if ((it & 1023u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1u;
                atomicOr(&g_na3d_timeout_flag, 1u);
                return false;
            }
        }
    }
}
// Wait for copies or MMAs in flight before the CTA frees its tensor memory
// and exits; a drain that gives up is recorded like any other timeout.
__device__ __forceinline__ void drain_wait(uint32_t b, uint32_t parity) {
    if (!mbar_wait_bounded(b, parity, kDrainLimitNs)) atomicOr(&g_na3d_timeout_flag, 1u);
}

struct Sync {
    uint32_t bar0;                     // smem address of barrier 0
    volatile uint32_t* abort_flag;     // smem, shared by all roles
    __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * i; }

    // Wait for a barrier phase; false once this CTA has given up.
    __device__ __forceinline__ bool wait(uint32_t b, uint32_t parity) const {
        if (mbar_try_wait(b, parity)) return true;
        return wait_spin(b, parity, abort_flag);
    }
};

// ------------------------------------------------------------------ producer

struct ChunkCoords {
    int x, kw0, kh0, kt, b;
};

template <class C>
__device__ void producer_role(const KernelParams& p, const CUtensorMap* tq, const CUtensorMap* tk,
                              const CUtensorMap* tv, const Sync& sy, uint32_t base) {
    // K stages, V stages, chunks and Q bricks issued (WIDE: a K stage is one
    // region of Q and K, so gk counts regions)
    uint32_t gk = 0, gv = 0, gc = 0, nq = 0;
    ChunkCoords prev{0, 0, 0, 0, 0};
    // bytes of one K stage, one V stage and one Q brick (WIDE: of one region
    // of the Q brick and of the K rows, which share a stage)
    const uint32_t k_bytes = (C::WIDE ? 1 : C::NREG) * C::ROWB * p.cw * p.cr;
    const uint32_t v_bytes = C::VREG * C::ROWB * p.cw * p.cr;
    const uint32_t q_bytes = (C::WIDE ? 1 : C::NREG) * C::ROWB * p.bt * p.bh * p.bw;

    auto load_v = [&](const ChunkCoords& cc) -> bool {
        const uint32_t st = gv % C::NSV;
        if (!sy.wait(sy.bar(C::B_VEMPTY + st), ((gv / C::NSV) & 1u) ^ 1u)) return false;
        const uint32_t full = sy.bar(C::B_VFULL + st);
        mbar_arrive_expect_tx(full, v_bytes);
#pragma unroll
        for (int r = 0; r < C::VREG; ++r)
            tma_load_5d(base + C::OFF_V + st * C::V_TILE + r * C::KV_REG, tv, full,
                        cc.x + r * C::HDB, cc.kw0, cc.kh0, cc.kt, cc.b);
        ++gv;
        return true;
    };
    // one K stage; self-test of the bounded waits: CTA 0 may withhold one,
    // whose barrier then never completes
    auto begin_k = [&](uint32_t* full_out) -> int {
        const uint32_t st = gk % C::NS;
        if (!sy.wait(sy.bar(C::B_KEMPTY + st), ((gk / C::NS) & 1u) ^ 1u)) return -1;
        *full_out = sy.bar(C::B_KFULL + st);
        const bool send = blockIdx.x != 0 || static_cast<int>(gk) != p.withhold_k;
        ++gk;
        return send ? static_cast<int>(st) : -2;
    };

    bool ok = true;
    uint32_t ul = 0;
    for (int u = first_unit<C>(p); ok && u < p.n_units; u = next_unit<C>(p, u), ++ul) {
        const Unit U = unit_of(p, u);
        // U.n counts (head, pass) pairs when WIDE; the head's columns start at xq
        const int head = C::WIDE ? U.n >> p.npass_log2 : U.n;
        const int xq = head * (C::WIDE ? p.hd : C::HD);
        const int xv = C::WIDE ? xq + (U.n & ((1 << p.npass_log2) - 1)) * C::OB : xq;
        ChunkCursor cur{U.lo_t, 0, 0};
        for (int c = 0; c < U.nch; ++c) {
            const ChunkCoords cc{xv, U.lo_w + cur.wc * p.cw, U.lo_h + cur.hc * p.cr, cur.kt, U.b};
            cur.advance(U);
            if constexpr (C::WIDE) {
                // region r of the Q brick and of the chunk's K rows, per stage
                for (int r = 0; r < p.nreg; ++r) {
                    uint32_t full;
                    const int st = begin_k(&full);
                    if (st == -1) { ok = false; break; }
                    if (st >= 0) {
                        const uint32_t dst = base + C::OFF_K + st * C::K_TILE;
                        mbar_arrive_expect_tx(full, q_bytes + k_bytes);
                        tma_load_5d(dst, tq, full, xq + r * C::HDB, U.w0, U.h0, U.t0, U.b);
                        tma_load_5d(dst + C::Q_REG, tk, full, xq + r * C::HDB, cc.kw0, cc.kh0, cc.kt, cc.b);
                    }
                }
                if (!ok) break;
            } else {
                uint32_t full;
                const int st = begin_k(&full);
                if (st == -1) { ok = false; break; }
                if (st >= 0) {
                    mbar_arrive_expect_tx(full, k_bytes);
#pragma unroll
                    for (int r = 0; r < C::NREG; ++r)
                        tma_load_5d(base + C::OFF_K + st * C::K_TILE + r * C::KV_REG, tk, full,
                                    xq + r * C::HDB, cc.kw0, cc.kh0, cc.kt, cc.b);
                }
            }
            ++gc;
            // V trails K by one chunk; it goes before the unit's Q brick, whose
            // buffer may still be read by the previous unit's last score tile
            if (gc >= 2 && !load_v(prev)) { ok = false; break; }
            prev = cc;
            if constexpr (!C::WIDE) {
                if (c == 0) {  // the Q brick goes right behind the unit's first K chunk
                    const uint32_t qb = ul % C::NQ;
                    if (!sy.wait(sy.bar(C::B_QEMPTY + qb), ((ul / C::NQ) & 1u) ^ 1u)) { ok = false; break; }
                    const uint32_t qf = sy.bar(C::B_QFULL + qb);
                    mbar_arrive_expect_tx(qf, q_bytes);
#pragma unroll
                    for (int r = 0; r < C::NREG; ++r)
                        tma_load_5d(base + C::OFF_Q + qb * C::Q_TILE + r * C::Q_REG, tq, qf,
                                    xq + r * C::HDB, U.w0, U.h0, U.t0, U.b);
                    ++nq;
                }
            }
        }
    }
    if (ok && gc > gv) load_v(prev);
    // Drain: every issued load must land before the CTA may exit.
    for (uint32_t s = 0; s < C::NS; ++s) {
        const uint32_t fk = gk / C::NS + (s < gk % C::NS ? 1u : 0u);
        if (fk) drain_wait(sy.bar(C::B_KFULL + s), (fk - 1u) & 1u);
    }
    for (uint32_t s = 0; s < C::NSV; ++s) {
        const uint32_t fv = gv / C::NSV + (s < gv % C::NSV ? 1u : 0u);
        if (fv) drain_wait(sy.bar(C::B_VFULL + s), (fv - 1u) & 1u);
    }
    if constexpr (C::NQ > 0) {
        for (uint32_t s = 0; s < C::NQ; ++s) {
            const uint32_t fq = nq / C::NQ + (s < nq % C::NQ ? 1u : 0u);
            if (fq) drain_wait(sy.bar(C::B_QFULL + s), (fq - 1u) & 1u);
        }
    }
}

// ------------------------------------------------------------------ tensor-core issuer

// Walks the CTA's chunks in order: unit u (see next_unit), chunk c.
// The unit's chunk count is decoded once, at its first chunk (one call site).
template <class C>
struct ChunkWalk {
    int u, c, nch;
    int hc, n_hc;         // ROWS: h-chunk index of chunk c (one W segment per row)
    uint32_t ul, g, gl;   // local unit, global chunk and local head-group counters
    bool gfirst;          // the unit opens its head group
    __device__ __forceinline__ void start(const KernelParams& p) {
        u = first_unit<C>(p);
        c = 0;
        ul = 0;
        g = 0;
        gl = 0;
        gfirst = true;
        nch = 0;
        hc = 0;
        n_hc = 1;
    }
    // false when the CTA has no units left; decodes a new unit's chunk count
    __device__ __forceinline__ bool more(const KernelParams& p) {
        if (u >= p.n_units) return false;
        if (c == 0) {
            const Unit U = unit_of(p, u);
            nch = U.nch;
            if constexpr (C::ROWS) {
                n_hc = U.n_hc;
                hc = 0;
            }
        }
        return true;
    }
    __device__ __forceinline__ void next(const KernelParams& p) {
        ++g;
        if constexpr (C::ROWS) {
            if (++hc == n_hc) hc = 0;
        }
        if (++c == nch) {
            c = 0;
            ++ul;
            gfirst = group_end<C>(p, u);
            if (gfirst) ++gl;
            u = next_unit<C>(p, u);
        }
    }
};

// Score tiles: S = Q K^T (+ Qx Kx^T), one chunk after another. Issued by one
// thread of warp 5; the products are issued by warp 6 (disjoint TMEM columns,
// each thread commits its own MMAs), so the two streams do not wait for each
// other's issue and sit on different SM sub-partitions.
template <class C>
__device__ void mma_s_role(const KernelParams& p, const Sync& sy, uint32_t base, uint32_t tmem) {
    // a tile that wraps around the ring is issued as two halves of SW keys
    const int n_lo = p.n_mma < static_cast<int>(C::SW) ? p.n_mma : static_cast<int>(C::SW);
    const int n_hi = p.n_mma - n_lo;
    const uint32_t idesc_s = make_idesc_bf16(128, p.n_mma, 0, 0);
    const uint32_t idesc_lo = make_idesc_bf16(128, n_lo, 0, 0);
    const uint32_t idesc_hi = n_hi > 0 ? make_idesc_bf16(128, n_hi, 0, 0) : 0u;
    const uint64_t qd0 = make_smem_desc(base + C::OFF_Q, 16, C::SBO, C::SWZ);
    const uint64_t kd0 = make_smem_desc(base + C::OFF_K, 16, C::SBO, C::SWZ);
    const uint32_t q_hi = static_cast<uint32_t>(qd0 >> 32), k_hi = static_cast<uint32_t>(kd0 >> 32);
    uint32_t x_hi = 0, x_lo0 = 0, y_lo = 0;
    if constexpr (C::FAST) {
        const uint64_t xd0 = make_smem_desc(base + C::OFF_QX, 16, C::XSBO, C::XSWZ);
        const uint64_t yd0 = make_smem_desc(base + C::OFF_KX, 16, C::XSBO, C::XSWZ);
        x_hi = static_cast<uint32_t>(xd0 >> 32);
        x_lo0 = static_cast<uint32_t>(xd0);
        y_lo = static_cast<uint32_t>(yd0);
    }
    // S = Q K^T + Qx Kx^T for the keys whose K and Kx rows start at k_lo and
    // y_l, into TMEM column d
    auto issue = [&](uint32_t d, uint32_t q_lo, uint32_t k_lo, uint32_t x_lo, uint32_t y_l,
                     uint32_t idesc) {
#pragma unroll
        for (int kk = 0; kk < C::HD / 16; ++kk) {
            constexpr int kPer = C::HDB / 16;   // k-steps per swizzle row
            const uint32_t qo = ((kk / kPer) * C::Q_REG + (kk % kPer) * 32) >> 4;
            const uint32_t ko = ((kk / kPer) * C::KV_REG + (kk % kPer) * 32) >> 4;
            if (kk == 0) umma_ss_halves<0>(d, q_lo + qo, q_hi, k_lo + ko, k_hi, idesc);
            else umma_ss_halves<1>(d, q_lo + qo, q_hi, k_lo + ko, k_hi, idesc);
        }
        if constexpr (C::FAST) {   // -2^40 on keys outside each row's W window
#pragma unroll
            for (int kk = 0; kk < C::KEXT / 16; ++kk)
                umma_ss_halves<1>(d, x_lo + kk * 2, x_hi, y_l + kk * 2, x_hi, idesc);
        }
    };
    ChunkWalk<C> w;
    w.start(p);
    if constexpr (C::WIDE) {
        // S(g) = sum over the NREG regions r of Q_r K_r^T, each region pair one
        // stage of the K ring; never wraps (pairs of slots)
        uint32_t gk = 0;   // K stages consumed
        while (w.more(p)) {
            uint32_t xb = 0;
            if constexpr (C::FAST) {
                xb = w.gl % C::NQX;
                if (w.c == 0 && w.gfirst && !sy.wait(sy.bar(C::B_XFULL + xb), (w.gl / C::NQX) & 1u)) break;
            }
            if (w.g >= static_cast<uint32_t>(C::SLAG)) {
                const uint32_t sc = w.g - C::SLAG;
                if (!sy.wait(sy.bar(C::B_SEMPTY + sc % C::RING), (sc / C::RING) & 1u)) break;
            }
            if (w.g >= static_cast<uint32_t>(C::LAG)) {
                const uint32_t pc = w.g - C::LAG;
                if (!sy.wait(sy.bar(C::B_PFREE + pc % C::RING), (pc / C::RING) & 1u)) break;
            }
            const uint32_t d = tmem + C::TM_R + C::slot_of(w.g) * C::SW;
            bool ok = true;
            for (int r = 0; r < p.nreg; ++r, ++gk) {
                const uint32_t st = gk % C::NS;
                if (!sy.wait(sy.bar(C::B_KFULL + st), (gk / C::NS) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t q_lo = static_cast<uint32_t>(kd0) + ((st * C::K_TILE) >> 4);
                const uint32_t k_lo = q_lo + (C::Q_REG >> 4);
                if (r == 0) umma_ss_halves<0>(d, q_lo, k_hi, k_lo, k_hi, idesc_s);
                else umma_ss_halves<1>(d, q_lo, k_hi, k_lo, k_hi, idesc_s);
#pragma unroll
                for (int kk = 1; kk < C::HDB / 16; ++kk)
                    umma_ss_halves<1>(d, q_lo + kk * 2, k_hi, k_lo + kk * 2, k_hi, idesc_s);
                umma_commit(sy.bar(C::B_KEMPTY + st));
            }
            if (!ok) break;
            if constexpr (C::FAST) {   // -2^40 on keys outside each row's W window
                const uint32_t x_lo = x_lo0 + ((xb * C::QX_TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < C::KEXT / 16; ++kk)
                    umma_ss_halves<1>(d, x_lo + kk * 2, x_hi, y_lo + kk * 2, x_hi, idesc_s);
            }
            umma_commit(sy.bar(C::B_SFULL + w.g % C::RING));
            if constexpr (C::FAST) {
                if (w.c == w.nch - 1 && group_end<C>(p, w.u)) umma_commit(sy.bar(C::B_XEMPTY + xb));
            }
            w.next(p);
        }
    } else while (w.more(p)) {
        const uint32_t qb = w.ul % C::NQ, st = w.g % C::NS;
        if (w.c == 0 && !sy.wait(sy.bar(C::B_QFULL + qb), (w.ul / C::NQ) & 1u)) break;
        uint32_t xb = 0;
        if constexpr (C::FAST) {
            xb = w.gl % C::NQX;   // one W-mask tile per head group
            if (w.c == 0 && w.gfirst && !sy.wait(sy.bar(C::B_XFULL + xb), (w.gl / C::NQX) & 1u)) break;
        }
        if (!sy.wait(sy.bar(C::B_KFULL + st), (w.g / C::NS) & 1u)) break;
        // the tile that last used these columns has been read, and the
        // product that last read them has completed
        if (w.g >= static_cast<uint32_t>(C::SLAG)) {
            const uint32_t sc = w.g - C::SLAG;
            if (!sy.wait(sy.bar(C::B_SEMPTY + sc % C::RING), (sc / C::RING) & 1u)) break;
        }
        if (w.g >= static_cast<uint32_t>(C::LAG)) {
            const uint32_t pc = w.g - C::LAG;
            if (!sy.wait(sy.bar(C::B_PFREE + pc % C::RING), (pc / C::RING) & 1u)) break;
        }
        tc_fence_after();
        const uint32_t q_lo = static_cast<uint32_t>(qd0) + ((qb * C::Q_TILE) >> 4);
        const uint32_t k_lo = static_cast<uint32_t>(kd0) + ((st * C::K_TILE) >> 4);
        const uint32_t x_lo = C::FAST ? x_lo0 + ((xb * C::QX_TILE) >> 4) : 0u;
        const uint32_t slot = C::slot_of(w.g);
        const uint32_t d = tmem + C::TM_R + slot * C::SW;
        // A tile that wraps around the ring goes out as two halves, keys SW..
        // to the first slot. With the tensor-core W mask one copy of the MMA
        // sequence serves both (smaller code measured faster there); the
        // per-key-mask instances measured faster with the halves written out.
        const bool wrap = C::STEP == 1 && slot + 1 == static_cast<uint32_t>(C::NSLOT);
        if constexpr (C::FAST) {
            // ROWS: the Kx tile of this chunk's h-chunk index
            const uint32_t y0 = C::ROWS ? y_lo + static_cast<uint32_t>(w.hc) * (C::KX_TILE >> 4) : y_lo;
            const int halves = wrap && n_hi > 0 ? 2 : 1;
#pragma unroll 1
            for (int hh = 0; hh < halves; ++hh) {
                const uint32_t dd = hh == 0 ? d : tmem + C::TM_R;
                const uint32_t kl = hh == 0 ? k_lo : k_lo + ((C::SW * C::ROWB) >> 4);
                const uint32_t yl = hh == 0 ? y0 : y0 + ((C::SW * C::XROWB) >> 4);
                const uint32_t id = !wrap ? idesc_s : (hh == 0 ? idesc_lo : idesc_hi);
                issue(dd, q_lo, kl, x_lo, yl, id);
            }
        } else if (wrap) {
            issue(d, q_lo, k_lo, x_lo, y_lo, idesc_lo);
            if (n_hi > 0)
                issue(tmem + C::TM_R, q_lo, k_lo + ((C::SW * C::ROWB) >> 4), x_lo,
                      y_lo + ((C::SW * C::XROWB) >> 4), idesc_hi);
        } else {
            issue(d, q_lo, k_lo, x_lo, y_lo, idesc_s);
        }
        umma_commit(sy.bar(C::B_SFULL + w.g % C::RING));
        umma_commit(sy.bar(C::B_KEMPTY + st));
        if (w.c == w.nch - 1) {
            umma_commit(sy.bar(C::B_QEMPTY + qb));
            if constexpr (C::FAST) {
                if (group_end<C>(p, w.u)) umma_commit(sy.bar(C::B_XEMPTY + xb));
            }
        }
        w.next(p);
    }
    // Drain: all MMAs issued by this thread complete before TMEM is freed.
    umma_commit(sy.bar(C::B_DRAIN));
    drain_wait(sy.bar(C::B_DRAIN), 0);
}

// Products: O += P V with P read from tensor memory; the unit's first
// product overwrites O, its last one signals the epilogue.
template <class C>
__device__ void mma_pv_role(const KernelParams& p, const Sync& sy, uint32_t base, uint32_t tmem) {
    const uint32_t idesc_o = make_idesc_bf16(128, C::OB, 0, 1);
    const uint32_t d_o = tmem + C::TM_O;
    const uint64_t vd0 = make_smem_desc(base + C::OFF_V, C::KV_REG, C::SBO, C::SWZ);
    const uint32_t v_hi = static_cast<uint32_t>(vd0 >> 32);
    const int ksteps = p.n_mma >> 4;
    ChunkWalk<C> w;
    w.start(p);
    while (w.more(p)) {
        const uint32_t st = w.g % C::NSV;
        if (w.c == 0 && !sy.wait(sy.bar(C::B_OEMPTY), (w.ul & 1u) ^ 1u)) break;
        if (!sy.wait(sy.bar(C::B_VFULL + st), (w.g / C::NSV) & 1u)) break;
        if (!sy.wait(sy.bar(C::B_PFULL + w.g % C::RING), (w.g / C::RING) & 1u)) break;
        tc_fence_after();
        const uint32_t v_lo = static_cast<uint32_t>(vd0) + ((st * C::V_TILE) >> 4);
        const uint32_t a_p = tmem + C::TM_R + C::slot_of(w.g) * C::SW;
        if (w.c == 0) umma_ts_halves<0>(d_o, a_p, v_lo, v_hi, idesc_o);
        else umma_ts_halves<1>(d_o, a_p, v_lo, v_hi, idesc_o);
#pragma unroll
        for (int kk = 1; kk < C::NCAP / 16; ++kk)
            if (kk < ksteps)
                umma_ts_halves<1>(d_o, a_p + kk * 8, v_lo + ((kk * 16 * C::ROWB) >> 4), v_hi, idesc_o);
        umma_commit(sy.bar(C::B_PFREE + w.g % C::RING));
        umma_commit(sy.bar(C::B_VEMPTY + st));
        if (w.c == w.nch - 1) umma_commit(sy.bar(C::B_OFULL));
        w.next(p);
    }
    umma_commit(sy.bar(C::B_DRAIN2));
    drain_wait(sy.bar(C::B_DRAIN2), 0);
}

// ------------------------------------------------------------------ softmax

// P = 2^(s log2e - moff) for the masked score row (masked keys give 0), as
// bf16 pairs into tensor memory; returns the fp32 sum of the probabilities.
template <class C>
__device__ __forceinline__ float write_probabilities(const float* s, const uint32_t* m,
                                                     const bool* live, int n_mma, float moff,
                                                     uint32_t p_addr) {
    const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
    const uint64_t neg2 = f2_pack(-moff, -moff);
    uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int q = 0; q < C::NW; ++q) {
        if (q * 32 < n_mma) {
            uint32_t pk[16];
            if (live[q] && __all_sync(0xffffffffu, m[q] == 0xffffffffu)) {
                // every key of this word is in every row's window: no selects
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float e0, e1;
                    f2_unpack(f2_fma(f2_pack(s[32 * q + 2 * j], s[32 * q + 2 * j + 1]), l2e2, neg2), e0, e1);
                    e0 = ex2_approx(e0);
                    e1 = ex2_approx(e1);
                    pk[j] = pack_bf16x2(e0, e1);
                    if (j & 1) acc1 = f2_add(acc1, f2_pack(e0, e1));
                    else acc0 = f2_add(acc0, f2_pack(e0, e1));
                }
            } else if (live[q]) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float x0 = ((m[q] >> (2 * j)) & 1u) ? s[32 * q + 2 * j] : -INFINITY;
                    const float x1 = ((m[q] >> (2 * j + 1)) & 1u) ? s[32 * q + 2 * j + 1] : -INFINITY;
                    float e0, e1;
                    f2_unpack(f2_fma(f2_pack(x0, x1), l2e2, neg2), e0, e1);
                    e0 = ex2_approx(e0);
                    e1 = ex2_approx(e1);
                    pk[j] = pack_bf16x2(e0, e1);
                    if (j & 1) acc1 = f2_add(acc1, f2_pack(e0, e1));
                    else acc0 = f2_add(acc0, f2_pack(e0, e1));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) pk[j] = 0u;
            }
            tmem_st16(p_addr + q * 16, pk);
        }
    }
    float a0, a1, b0, b1;
    f2_unpack(acc0, a0, a1);
    f2_unpack(acc1, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

// Maximum of the masked score row (-inf when the row has no key here).
template <class C>
__device__ __forceinline__ float masked_row_max(const float* s, const uint32_t* m, const bool* live) {
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < C::NW; ++q) {
        if (live[q]) {
#pragma unroll
            for (int b = 0; b < 32; b += 2) {
                const float x0 = ((m[q] >> b) & 1u) ? s[32 * q + b] : -INFINITY;
                const float x1 = ((m[q] >> (b + 1)) & 1u) ? s[32 * q + b + 1] : -INFINITY;
                mx = max3f(mx, x0, x1);
            }
        }
    }
    return mx;
}

// Byte offset of 16-byte chunk k of row `row` in a K-major operand tile with
// rows of `rowb` bytes and the matching swizzle (the 16-byte chunk index is
// XORed with address bits 7.. of the row start, over rowb/16 chunks).
__device__ __forceinline__ uint32_t swizzled_chunk(int row, int k, int rowb) {
    return static_cast<uint32_t>(row * rowb + ((k ^ (((row * rowb) >> 7) & (rowb / 16 - 1))) << 4));
}

// Probabilities for the fast path: chunk row i holds keys [i*CWP, (i+1)*CWP)
// and is either wholly in this row's H/T window (bit i of rowbits) or not;
// keys outside the W window already carry -2^40 from the tensor core.
template <class C>
__device__ __forceinline__ float fast_probabilities(const float* s, uint32_t rowbits, const bool* live,
                                                    int n_mma, float moff, uint32_t p_addr) {
    const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
    uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int q = 0; q < C::NW; ++q) {
        if constexpr (C::ODD) {   // a row's keys may straddle words: the row of each pair is fixed
            if (q * 32 < n_mma) {
                uint32_t pk[16];
                if (live[q]) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int i = (32 * q + 2 * j) / C::RW;   // both keys of a pair share a row
                        const float nm = ((rowbits >> i) & 1u) ? -moff : -INFINITY;
                        float e0, e1;
                        f2_unpack(f2_fma(f2_pack(s[32 * q + 2 * j], s[32 * q + 2 * j + 1]), l2e2,
                                         f2_pack(nm, nm)),
                                  e0, e1);
                        e0 = ex2_approx(e0);
                        e1 = ex2_approx(e1);
                        pk[j] = pack_bf16x2(e0, e1);
                        if (j & 1) acc1 = f2_add(acc1, f2_pack(e0, e1));
                        else acc0 = f2_add(acc0, f2_pack(e0, e1));
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[j] = 0u;
                }
                tmem_st16(p_addr + q * 16, pk);
            }
            continue;
        }
        if (q * 32 < n_mma) {
            uint32_t pk[16];
            if (live[q]) {
#pragma unroll
                for (int rr = 0; rr < C::RPW; ++rr) {
                    const int i = q * C::RPW + rr;
                    const float nm = ((rowbits >> i) & 1u) ? -moff : -INFINITY;
                    const uint64_t nm2 = f2_pack(nm, nm);
#pragma unroll
                    for (int jj = 0; jj < C::RW / 2; ++jj) {
                        const int j = rr * (C::RW / 2) + jj;
                        float e0, e1;
                        f2_unpack(f2_fma(f2_pack(s[32 * q + 2 * j], s[32 * q + 2 * j + 1]), l2e2, nm2),
                                  e0, e1);
                        e0 = ex2_approx(e0);
                        e1 = ex2_approx(e1);
                        pk[j] = pack_bf16x2(e0, e1);
                        if (j & 1) acc1 = f2_add(acc1, f2_pack(e0, e1));
                        else acc0 = f2_add(acc0, f2_pack(e0, e1));
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) pk[j] = 0u;
            }
            tmem_st16(p_addr + q * 16, pk);
        }
    }
    float a0, a1, b0, b1;
    f2_unpack(acc0, a0, a1);
    f2_unpack(acc1, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

// Maximum over the valid chunk rows (W-masked keys sit at -2^40 and never win:
// every valid row holds the whole W window of its query).
template <class C>
__device__ __forceinline__ float fast_row_max(const float* s, uint32_t rowbits, const bool* live) {
    float mx = -INFINITY;
    if constexpr (C::ODD) {
        float rm[C::NROWS];
#pragma unroll
        for (int i = 0; i < C::NROWS; ++i) rm[i] = -INFINITY;
#pragma unroll
        for (int q = 0; q < C::NW; ++q) {
            if (live[q]) {
#pragma unroll
                for (int b = 32 * q; b < 32 * q + 32; b += 2) rm[b / C::RW] = max3f(rm[b / C::RW], s[b], s[b + 1]);
            }
        }
#pragma unroll
        for (int i = 0; i < C::NROWS; ++i) mx = ((rowbits >> i) & 1u) ? fmaxf(mx, rm[i]) : mx;
    } else {
#pragma unroll
        for (int q = 0; q < C::NW; ++q) {
            if (live[q]) {
#pragma unroll
                for (int rr = 0; rr < C::RPW; ++rr) {
                    const int i = q * C::RPW + rr;
                    float rm = -INFINITY;
#pragma unroll
                    for (int jj = 0; jj < C::RW; jj += 2) {
                        const int b = 32 * q + rr * C::RW + jj;
                        rm = max3f(rm, s[b], s[b + 1]);
                    }
                    mx = ((rowbits >> i) & 1u) ? fmaxf(mx, rm) : mx;
                }
            }
        }
    }
    return mx;
}

template <class C>
__device__ void softmax_role(const KernelParams& p, const Sync& sy, uint32_t base, uint32_t tmem,
                             int warp, int lane) {
    const int r = warp * 32 + lane;             // tile row = query of the brick = TMEM lane
    const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int M = p.bt * p.bh * p.bw;
    const int iw = r % p.bw, ih = (r / p.bw) % p.bh, it = r / (p.bw * p.bh);
    uint32_t g = 0, ul = 0;
    // A wait whose outcome the whole warp shares (the .sync.aligned tensor
    // memory instructions that follow need every lane); a warp that gives up
    // first waits for its own tensor-memory stores, then leaves.
    auto swait = [&](uint32_t b, uint32_t parity) -> bool {
        const bool ok = __all_sync(0xffffffffu, sy.wait(b, parity));
        if (!ok) tmem_wait_st();
        return ok;
    };

    // Qx row of the brick of unit X (local head-group index `v`): -2^40 where
    // this row's query does not see the chunk column, 0 elsewhere; published
    // for the tensor core once per head group.
    auto publish_qx = [&](uint32_t v, const Unit& X) -> bool {
        if constexpr (C::FAST) {
            const uint32_t xb = v % C::NQX;
            if (!swait(sy.bar(C::B_XEMPTY + xb), ((v / C::NQX) & 1u) ^ 1u)) return false;
            const int t = X.t0 + it, h = X.h0 + ih, w = X.w0 + iw;
            const bool ok = r < M && t < p.Tq && h < p.Hq && w < p.Wq;
            // column c masks W position c of a chunk row (the window starts at
            // c_lo), or with ROWS halo row c (the H window starts at c_lo)
            const int c_lo = C::ROWS ? win_start(p.h_off + h, p.KH, p.H) - X.lo_h
                                     : win_start(p.w_off + w, p.KW, p.W) - X.lo_w;
            const int klen = C::ROWS ? p.KH : p.KW;
            const int ncol = C::ROWS ? C::XDEAD : C::CWP;   // columns that can be valid
            const uint32_t tile = base + C::OFF_QX + xb * C::QX_TILE;
#pragma unroll
            for (int k = 0; k < C::XROWB / 16; ++k) {
                uint32_t wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c0 = 8 * k + 2 * e, c1 = c0 + 1;
                    bool m0 = ok && c0 < ncol && static_cast<unsigned>(c0 - c_lo) >= static_cast<unsigned>(klen);
                    bool m1 = ok && c1 < ncol && static_cast<unsigned>(c1 - c_lo) >= static_cast<unsigned>(klen);
                    if constexpr (C::ROWS) {   // padding keys are masked for every row
                        m0 = m0 || c0 == C::XDEAD;
                        m1 = m1 || c1 == C::XDEAD;
                    }
                    wd[e] = (m0 ? kMaskBf16 : 0u) | ((m1 ? kMaskBf16 : 0u) << 16);
                }
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + swizzled_chunk(r, k, C::XROWB)),
                             "r"(wd[0]), "r"(wd[1]), "r"(wd[2]), "r"(wd[3])
                             : "memory");
            }
            fence_proxy_async_smem();
            mbar_arrive(sy.bar(C::B_XFULL + xb));
        }
        return true;
    };

    int u = first_unit<C>(p);
    uint32_t gl = 0;   // local head-group counter (W-mask tiles)
    Unit U{};          // the unit being processed
    Unit Un{};         // mask instances: the next head group's first unit
    // Mask tiles go out one head group ahead of use: a group's tile is
    // published when the group two before it ends (that group's buffer is
    // then free), so a group's first score tile never waits for the softmax
    // to finish the previous group.
    if (u < p.n_units) {
        U = unit_of(p, u);
        if (!publish_qx(0, U)) return;
        if constexpr (C::FAST) {
            const int u1 = next_group_unit<C>(p, u);
            if (u1 < p.n_units) {
                Un = unit_of(p, u1);
                if (!publish_qx(1, Un)) return;
            }
        }
    }
    // A finished unit's output is written once the next unit is set up, so its
    // last product completes meanwhile; then the tensor memory O is released.
    uint16_t* e_orow = nullptr;
    float e_l = 0.f;
    uint32_t e_ul = 0;
    bool e_valid = false, e_live = false;

    for (;; ++ul) {
        const bool have = u < p.n_units;
        const int t = U.t0 + it, h = U.h0 + ih, w = U.w0 + iw;
        const bool valid = have && r < M && t < p.Tq && h < p.Hq && w < p.Wq;
        // this row's window, in grid coordinates
        const int sT = win_start(p.t_off + t, p.KT, p.T), sH = win_start(p.h_off + h, p.KH, p.H),
                  sW = win_start(p.w_off + w, p.KW, p.W);
        // Generic path: column pattern of this row's window inside one chunk
        // (when a chunk holds several h-rows, the W extent of the halo fits in cw).
        uint32_t rowpat[4] = {0u, 0u, 0u, 0u};
        if constexpr (!C::FAST) {
            if (have && p.cr > 1) {
                const int c0 = max(sW - U.lo_w, 0), c1 = min(sW + p.KW - U.lo_w, p.cw);
                for (int i = 0; i < p.cr; ++i) {
                    uint32_t tmp[4];
                    bit_range128(tmp, i * p.cw + c0, i * p.cw + c1);
#pragma unroll
                    for (int q = 0; q < 4; ++q) rowpat[q] |= tmp[q];
                }
            }
        }
        if (e_live) {   // the previous unit's epilogue: O / l -> bf16 -> global
            if (!swait(sy.bar(C::B_OFULL), e_ul & 1u)) return;
            tc_fence_after();
            const float inv = (e_valid && e_l > 0.f) ? rcp_approx(e_l) : 0.f;
            // HD >= 128 (a 32-byte aligned output): lanes 2i and 2i + 1 store rows 2i and 2i + 1
            // together, so each store instruction writes 64 contiguous bytes per row
            // instead of 32 scattered ones (fewer, larger write requests)
            bool paired = false;
            const bool odd = (lane & 1) != 0;
            uint16_t* p_orow = nullptr;   // the partner lane's row
            bool p_valid = false;
            if constexpr (C::HD >= 128) {
                paired = p.out_v8 != 0;
                p_orow = reinterpret_cast<uint16_t*>(
                    __shfl_xor_sync(0xffffffffu, reinterpret_cast<unsigned long long>(e_orow), 1));
                p_valid = __shfl_xor_sync(0xffffffffu, e_valid ? 1 : 0, 1) != 0;
            }
#pragma unroll 1
            for (int q = 0; q < C::OPIECES; ++q) {
                float o[32];
                tmem_ld32(t_row + C::TM_O + q * 32, o);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(o[2 * j] * inv, o[2 * j + 1] * inv);
                if (paired) {
                    // even lane: the first 32 bytes of its row, then of the odd partner's row;
                    // odd lane: the last 32 bytes of the even partner's row, then of its row
                    uint32_t snd[8], rcv[8], d1[8], d2[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) snd[j] = odd ? pk[j] : pk[8 + j];
#pragma unroll
                    for (int j = 0; j < 8; ++j) rcv[j] = __shfl_xor_sync(0xffffffffu, snd[j], 1);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        d1[j] = odd ? rcv[j] : pk[j];
                        d2[j] = odd ? pk[8 + j] : rcv[j];
                    }
                    const int off = odd ? 16 : 0;
                    if (odd ? p_valid : e_valid) st_global_v8((odd ? p_orow : e_orow) + q * 32 + off, d1);
                    if (odd ? e_valid : p_valid) st_global_v8((odd ? e_orow : p_orow) + q * 32 + off, d2);
                } else if (e_valid) {
                    constexpr int kBytes = (C::HD < 32 ? C::HD : 32) * 2;   // bytes per piece
                    if (p.out_v8) {   // whole 32-byte sectors per lane
#pragma unroll
                        for (int i = 0; i < kBytes / 32; ++i) st_global_v8(e_orow + q * 32 + 16 * i, pk + 8 * i);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(e_orow + q * 32);
#pragma unroll
                        for (int i = 0; i < kBytes / 16; ++i)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(sy.bar(C::B_OEMPTY));
            e_live = false;
        }
        if (!have) break;

        float m_ref = -INFINITY;   // reference maximum, log2 units
        float l = 0.f;             // running sum of the probabilities
        ChunkCursor cur{U.lo_t, 0, 0};

        for (int c = 0; c < U.nch; ++c, ++g) {
            // The window mask of this chunk depends only on its position: it is
            // built before the wait for its scores, off the chain from S to P.
            const int kh0 = U.lo_h + cur.hc * p.cr, kw0 = U.lo_w + cur.wc * p.cw;
            const bool t_ok = valid && static_cast<unsigned>(cur.kt - sT) < static_cast<unsigned>(p.KT);
            uint32_t m[4] = {0u, 0u, 0u, 0u};   // generic path: per-key mask
            uint32_t rowbits = 0u;              // fast path: valid chunk rows
            if (t_ok) {
                const int i0 = max(sH - kh0, 0), i1 = min(sH + p.KH - kh0, p.cr);
                if constexpr (C::ROWS) {
                    // the tensor core masks single keys; a chunk with no row of
                    // this query's H window is skipped as a whole; the groups
                    // of 16 columns past the tile width hold no scores
                    if (i0 < i1) rowbits = (1u << (p.n_mma >> 4)) - 1u;
                } else if constexpr (C::FAST) {
                    if (i0 < i1) rowbits = ((1u << (i1 - i0)) - 1u) << i0;
                } else {
                    const int c0 = max(sW - kw0, 0), c1 = min(sW + p.KW - kw0, p.cw);
                    if (i0 < i1 && c0 < c1) {
                        if (p.cr == 1) {
                            bit_range128(m, c0, c1);
                        } else {
                            bit_range128(m, i0 * p.cw, i1 * p.cw);
#pragma unroll
                            for (int q = 0; q < 4; ++q) m[q] &= rowpat[q];
                        }
                    }
                }
            }
            cur.advance(U);
            bool live[C::NW];
#pragma unroll
            for (int q = 0; q < C::NW; ++q) {
                bool mine;
                if constexpr (C::ODD) mine = (rowbits & C::word_rows(q)) != 0u;
                else if constexpr (C::FAST) mine = (rowbits >> (q * C::RPW)) & ((1u << C::RPW) - 1u);
                else mine = m[q] != 0u;
                live[q] = (q * 32 < p.n_mma) && __any_sync(0xffffffffu, mine);
            }
            bool has_keys;
            if constexpr (C::FAST) has_keys = rowbits != 0u;
            else has_keys = (m[0] | m[1] | m[2] | m[3]) != 0u;

            if (!swait(sy.bar(C::B_SFULL + g % C::RING), (g / C::RING) & 1u)) return;
            tc_fence_after();
            // this chunk's ring slot: S words 0.. start there (wrapping to the
            // first slot after the last), and P goes over its first SW columns
            const uint32_t slot = C::slot_of(g);
            const uint32_t p_addr = t_row + C::TM_R + slot * C::SW;
            float s[C::NCAP];   // loaded asynchronously; not read before tmem_wait_ld
            // words 2k and 2k+1 are adjacent columns (in one slot, or in a
            // pair of slots that never wraps): one load each
#pragma unroll
            for (int q = 0; q < C::NW; q += 2) {
                if (q * 32 < p.n_mma) {
                    uint32_t sl = slot + (32u * q) / C::SW;
                    sl = sl >= static_cast<uint32_t>(C::NSLOT) ? sl - C::NSLOT : sl;
                    if (q + 1 < C::NW) tmem_ld64(t_row + C::TM_R + sl * C::SW + (32u * q) % C::SW, s + 32 * q);
                    else tmem_ld32(t_row + C::TM_R + sl * C::SW + (32u * q) % C::SW, s + 32 * q);
                }
            }

            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(sy.bar(C::B_SEMPTY + g % C::RING));   // these S columns may be overwritten now


            // Probabilities against the kept reference maximum, with no max
            // pass. A row meeting its first keys, or a chunk whose
            // probabilities sum past 2^32 (its maximum grew by ~32 in log2
            // units), takes an exact pass: maximum, reference update, redo.
            // Probabilities keep their relative precision at any scale, so
            // both passes give the same result.
            bool exact = __any_sync(0xffffffffu, has_keys && m_ref == -INFINITY);
            float lsum = 0.f, alpha = 1.f;
            bool rescale = false;
            // the reference update of an exact pass
            auto exact_max = [&]() {
                float mx;
                if constexpr (C::FAST) mx = fast_row_max<C>(s, rowbits, live);
                else mx = masked_row_max<C>(s, m, live);
                const float mx2 = mx * kLog2e;
                if (mx2 > m_ref + kRescaleThreshold) {
                    if (m_ref != -INFINITY) {
                        alpha = ex2_approx(m_ref - mx2);
                        rescale = true;
                    }
                    m_ref = mx2;
                }
            };
            if constexpr (C::FAST) {
                // one copy of the probability code serves both passes (the
                // loop is not unrolled), which keeps the loop body small
#pragma unroll 1
                for (;;) {
                    if (exact) exact_max();
                    lsum = fast_probabilities<C>(s, rowbits, live, p.n_mma,
                                                 m_ref == -INFINITY ? 0.f : m_ref, p_addr);
                    // after an exact pass every probability is at most 2^8
                    if (exact || !__any_sync(0xffffffffu, !(lsum <= kSumLimit))) break;
                    exact = true;
                    tmem_wait_st();   // the exact pass overwrites this P
                }
            } else {
                // per-key masks: the rolled form spills, so the passes are written out
                if (!exact) {
                    lsum = write_probabilities<C>(s, m, live, p.n_mma, m_ref == -INFINITY ? 0.f : m_ref,
                                                  p_addr);
                    exact = __any_sync(0xffffffffu, !(lsum <= kSumLimit));
                    if (exact) tmem_wait_st();   // the exact pass overwrites this P
                }
                if (exact) {
                    exact_max();
                    lsum = write_probabilities<C>(s, m, live, p.n_mma, m_ref == -INFINITY ? 0.f : m_ref,
                                                  p_addr);
                }
            }
            l = l * alpha + lsum;

            if (__any_sync(0xffffffffu, rescale)) {
                // O holds the products up to chunk g-1 (one of this unit: the
                // reference maximum was finite); the last of them must be done
                const uint32_t pc = g - 1u;
                if (!swait(sy.bar(C::B_PFREE + pc % C::RING), (pc / C::RING) & 1u)) return;
                tc_fence_after();
                const float a = rescale ? alpha : 1.f;
#pragma unroll 1
                for (int q = 0; q < C::OPIECES; ++q) {  // HD = 16 also scales 16 unused columns
                    float o[32];
                    tmem_ld32(t_row + C::TM_O + q * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= a;
                    tmem_st32(t_row + C::TM_O + q * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(sy.bar(C::B_PFULL + g % C::RING));
        }

        // this unit's output is written at the top of the next iteration, once
        // the next unit is set up
        const int64_t tok = ((static_cast<int64_t>(U.b) * p.Tq + t) * p.Hq + h) * p.Wq + w;
        if constexpr (C::WIDE)   // U.n counts (head, pass) pairs; a pass writes OB columns
            e_orow = p.out + (tok * p.NH + (U.n >> p.npass_log2)) * p.hd +
                     (U.n & ((1 << p.npass_log2) - 1)) * C::OB;
        else
            e_orow = p.out + (tok * p.NH + U.n) * C::HD;
        e_l = l;
        e_ul = ul;
        e_valid = valid;
        e_live = true;
        const bool new_group = group_end<C>(p, u);
        u = next_unit<C>(p, u);
        if (u < p.n_units) {
            if (new_group) {   // another brick (its mask tile is already out)
                ++gl;
                if constexpr (C::FAST) {
                    U = Un;
                    const int u2 = next_group_unit<C>(p, u);
                    if (u2 < p.n_units) {   // the group after it, into the finished group's buffer
                        Un = unit_of(p, u2);
                        if (!publish_qx(gl + 1, Un)) return;
                    }
                } else {
                    U = unit_of(p, u);
                }
            } else {           // the next head of the same brick
                ++U.n;
            }
        }
    }
}

// ------------------------------------------------------------------ kernel

template <int HD, int NCAP, int NS, int CPS, int CWP>
__global__ void __launch_bounds__(kThreads, CPS)
na3d_fwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const KernelParams p) {
    using C = Cfg<HD, NCAP, NS, CPS, CWP>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Zero the Q and K/V tiles once: pad rows are never written by TMA and
    // must hold finite values (a zero probability times NaN is NaN).
    {
        uint4* z = reinterpret_cast<uint4*>(base_ptr);
        for (int i = threadIdx.x; i < C::OFF_KX / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    }
    if constexpr (C::FAST) {
        // Kx: key j of a chunk has a one in column j % CWP (its W position);
        // with ROWS, tile hc has it in the column of the key's row within the
        // brick's halo (hc * cr + j / cw), or in the dead column for padding
        // keys and rows past the last one a mask column can name.
        const int j = threadIdx.x;
        if (j < C::NCAP) {
#pragma unroll 1
            for (int x = 0; x < C::NKX; ++x) {
                int col = j % CWP;
                if constexpr (C::ROWS) {
                    col = j < p.cr * p.cw ? x * p.cr + j / p.cw : C::XDEAD;
                    col = col < C::XDEAD ? col : C::XDEAD;
                }
#pragma unroll
                for (int k = 0; k < C::XROWB / 16; ++k) {
                    uint32_t wd[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c0 = 8 * k + 2 * e;
                        wd[e] = (c0 == col ? 0x3F80u : 0u) | ((c0 + 1 == col ? 0x3F80u : 0u) << 16);
                    }
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     base + C::OFF_KX + x * C::KX_TILE + swizzled_chunk(j, k, C::XROWB)),
                                 "r"(wd[0]), "r"(wd[1]), "r"(wd[2]), "r"(wd[3])
                                 : "memory");
                }
            }
        }
    }
    fence_proxy_async_smem();

    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_MISC);
    Sync sy{base + C::OFF_BAR, misc + 1};
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NBAR; ++i) {
            const bool softmax_arrives = i == C::B_OEMPTY ||
                                         (i >= C::B_SEMPTY && i < C::B_SEMPTY + C::RING) ||
                                         (i >= C::B_PFULL && i < C::B_PFULL + C::RING) ||
                                         (i >= C::B_XFULL && i < C::B_XFULL + C::NQX);
            mbar_init(sy.bar(i), softmax_arrives ? 128u : 1u);
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 5) {
        tmem_alloc(base + C::OFF_MISC, C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // The score ring starts as zeros: a tile narrower than its last 32-column
    // word leaves columns that the softmax reads (and masks) unwritten, and
    // fresh tensor memory may hold any bit pattern.
    if (warp < 4) {
        float z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0.f;
        for (uint32_t c = C::TM_R; c + 32 <= C::TM_COLS; c += 32)
            tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, z);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp < 4) {
        if (C::CPS == 2) regs_increase<C::REGS_HIGH>();
        softmax_role<C>(p, sy, base, tmem, warp, lane);
    } else {
        if (C::CPS == 2) regs_decrease<C::REGS_LOW>();
        if (warp == 4 && lane == 0) producer_role<C>(p, &tm_q, &tm_k, &tm_v, sy, base);
        if (warp == 5 && lane == 0) mma_s_role<C>(p, sy, base, tmem);
        if (warp == 6 && lane == 0) mma_pv_role<C>(p, sy, base, tmem);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// ------------------------------------------------------------------ host side

template <int HD, int NCAP, int NS, int CPS, int CWP>
static cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const KernelParams& kp, int grid, cudaStream_t stream) {
    using C = Cfg<HD, NCAP, NS, CPS, CWP>;
    auto kern = na3d_fwd_sm103<HD, NCAP, NS, CPS, CWP>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::SMEM_ALLOC, stream>>>(tq, tk, tv, kp);
    return cudaGetLastError();
}

template <int HD, int NCAP, int NS, int CPS, int CWP>
static void info_t(VariantInfo* v) {
    using C = Cfg<HD, NCAP, NS, CPS, CWP>;
    v->ncap = NCAP;
    v->stages = NS;
    v->hd_box = C::HDB;
    v->smem = C::SMEM_ALLOC;
    v->ctas_per_sm = CPS;
}

// The instance table: (HD, score-tile cap, K/V stages, CTAs per SM) x chunk
// stride CWP (0: generic masks; 8, 16, 32 and, for HD 64 and 128, 12 and 14: W
// window applied by the tensor core; 1: whole-row W windows, H window applied
// by the tensor core). HD <= 64 has a second family of 96-key score tiles: O
// (64 columns) and four 48-column slots fill the CTA's 256 tensor-memory
// columns, and the slots are used as pairs, so the next score tile is
// computed while the softmax works on the current one.
#define NA3D_HD_TABLE(X, CWP) \
    X(16, 128, 4, 2, CWP)     \
    X(32, 128, 3, 2, CWP)     \
    X(64, 128, 2, 2, CWP)     \
    X(128, 64, 2, 2, CWP)     \
    X(256, 64, 2, 1, CWP)     \
    X(512, 64, 4, 1, CWP)
#define NA3D_EXACT_TABLE(X)  \
    X(64, 128, 2, 2, 12)     \
    X(64, 128, 2, 2, 14)     \
    X(128, 64, 2, 2, 12)     \
    X(128, 64, 2, 2, 14)
#define NA3D_PAIRED_TABLE(X)  \
    X(16, 96, 4, 2, 0)     \
    X(16, 96, 4, 2, 8)     \
    X(16, 96, 4, 2, 16)    \
    X(16, 96, 4, 2, 32)    \
    X(32, 96, 3, 2, 0)     \
    X(32, 96, 3, 2, 8)     \
    X(32, 96, 3, 2, 16)    \
    X(32, 96, 3, 2, 32)    \
    X(64, 96, 3, 2, 0)     \
    X(64, 96, 3, 2, 8)     \
    X(64, 96, 3, 2, 12)    \
    X(64, 96, 3, 2, 14)    \
    X(64, 96, 3, 2, 16)    \
    X(64, 96, 3, 2, 32)
#define NA3D_ROWS_TABLE(X)  \
    X(16, 128, 4, 2, 1)     \
    X(32, 128, 3, 2, 1)     \
    X(64, 128, 2, 2, 1)     \
    X(128, 64, 2, 2, 1)     \
    X(256, 64, 2, 1, 1)
#define NA3D_VARIANTS(X) \
    NA3D_HD_TABLE(X, 0) NA3D_HD_TABLE(X, 8) NA3D_HD_TABLE(X, 16) NA3D_HD_TABLE(X, 32) NA3D_ROWS_TABLE(X) \
    NA3D_EXACT_TABLE(X) NA3D_PAIRED_TABLE(X)

int default_ncap(int hd) { return hd <= 64 ? 128 : 64; }

bool variant_info(int hd, int cwp, int ncap, VariantInfo* info) {
    if (hd > 256) hd = 512;   // the wide instance serves every HD >= 512
#define X(hd_, n_, s_, c_, w_)                   \
    if (hd == hd_ && cwp == w_ && ncap == n_) {  \
        if (info) info_t<hd_, n_, s_, c_, w_>(info); \
        return true;                             \
    }
    NA3D_VARIANTS(X)
#undef X
    return false;
}

cudaError_t launch_fwd(int hd, int cwp, int ncap, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const KernelParams& kp, int grid,
                       cudaStream_t stream) {
    if (hd > 256) hd = 512;
#define X(hd_, n_, s_, c_, w_) \
    if (hd == hd_ && cwp == w_ && ncap == n_) return launch_t<hd_, n_, s_, c_, w_>(tq, tk, tv, kp, grid, stream);
    NA3D_VARIANTS(X)
#undef X
    return cudaErrorInvalidValue;
}

// Each status request takes the flag with one atomic exchange (so a timeout is
// reported to exactly one request, never lost between a read and a clear) and
// leaves the old value in a slot of its own, which the host then reads.
constexpr unsigned int kStatusSlots = 256;
__device__ unsigned int g_na3d_status_slots[kStatusSlots];

__global__ void take_timeout_flag(unsigned int slot) {
    g_na3d_status_slots[slot] = atomicExch(&g_na3d_timeout_flag, 0u);
}

cudaError_t take_device_error(cudaStream_t stream, unsigned int* flag) {
    static std::atomic<unsigned int> next{0};
    const unsigned int slot = next.fetch_add(1u) % kStatusSlots;
    take_timeout_flag<<<1, 1, 0, stream>>>(slot);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbolAsync(flag, g_na3d_status_slots, sizeof(unsigned int),
                                  slot * sizeof(unsigned int), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace na3d
