// C ABI of the NA3D forward pass: argument validation, the brick/chunk
// planner, TMA descriptor encoding and the launch. Declared in include/na3d.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "na3d.h"
#include "na3d_kernel.cuh"
#include "na3d_proj.cuh"

namespace {

using na3d::KernelParams;
using na3d::VariantInfo;

// ------------------------------------------------------------------ validation

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

int validate_shape(int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT,
                   int64_t KH, int64_t KW) {
    if (B < 1 || NH < 1 || T < 1 || H < 1 || W < 1 || HD < 1) return NA3D_ERR_SHAPE;
    const int64_t ks[3] = {KT, KH, KW}, ns[3] = {T, H, W};
    for (int a = 0; a < 3; ++a)
        if (ks[a] < 1 || (ks[a] & 1) == 0 || ks[a] > ns[a]) return NA3D_ERR_KERNEL;
    if (!is_pow2(HD) || HD < 16) return NA3D_ERR_HEAD_DIM;
    // element count and byte size of one tensor must fit int64; TMA limits:
    // every global dimension < 2^32, every stride < 2^40 bytes.
    int64_t n = 1;
    const int64_t dims[6] = {B, T, H, W, NH, HD};
    for (int i = 0; i < 6; ++i)
        if (!mul_ok(n, dims[i], &n)) return NA3D_ERR_OVERFLOW;
    if (!mul_ok(n, 2, &n)) return NA3D_ERR_OVERFLOW;
    // a head's column offset is a signed 32-bit TMA coordinate
    if (NH * HD >= (int64_t(1) << 31) || W >= (int64_t(1) << 31) || H >= (int64_t(1) << 31) ||
        T >= (int64_t(1) << 31) || B >= (int64_t(1) << 31))
        return NA3D_ERR_OVERFLOW;
    if (n / dims[0] >= (int64_t(1) << 40)) return NA3D_ERR_OVERFLOW;  // batch stride in bytes
    return NA3D_OK;
}

// ------------------------------------------------------------------ planner

int64_t win_start(int64_t i, int64_t K, int64_t N) {
    int64_t s = i - K / 2;
    if (s < 0) s = 0;
    if (s > N - K) s = N - K;
    return s;
}

// One axis of the problem: `nq` query positions starting at `off` of an axis
// of length `n` (the whole axis: off = 0, nq = n), windows of length `k`.
struct Axis {
    int64_t nq, off, n, k;
};

// Sum over the bricks of one axis of ceil(extent / unit), where extent is the
// length of the union of the windows of the brick's queries (unit 1: the
// union length itself). Also returns the number of bricks.
int64_t axis_sum(const Axis& a, int64_t b, int64_t unit, int64_t* nbricks) {
    int64_t sum = 0, cnt = 0;
    for (int64_t p0 = 0; p0 < a.nq; p0 += b, ++cnt) {
        const int64_t last = a.off + (p0 + b < a.nq ? p0 + b : a.nq) - 1;
        const int64_t ext = win_start(last, a.k, a.n) + a.k - win_start(a.off + p0, a.k, a.n);
        sum += (ext + unit - 1) / unit;
    }
    *nbricks = cnt;
    return sum;
}

struct Plan {
    int bt = 0, bh = 0, bw = 0, cw = 0, cr = 0, n_mma = 0;
    int cwp = 0;   // fixed chunk stride of the tensor-core W-mask path (0: generic masks)
    int ncap = 0;  // score-tile cap of the instance family
    int64_t bricks = 0, chunks = 0;
    double cost = 0;
};

// Costs in units of score columns of a 128-row tile: every chunk costs its
// tile width (tensor-core and exp work) plus a fixed overhead (the latency of
// its score -> softmax -> product chain); every brick adds the unit boundary
// (epilogue, last product, set-up: about 2.7 chunks of a 128-key tile on
// GB300). Columns of the tensor-core mask paths cost about half as much
// softmax work as columns masked key by key.
constexpr double kChunkOverhead = 60.0;
constexpr double kBrickOverhead = 250.0;
constexpr double kFastColumn = 0.55;
// Tensor-core work per tile column: the softmax works in 32-key words, the
// MMAs in 16-key steps, so of two tiles with the same words the narrower
// one is cheaper.
constexpr double kMmaColumn = 0.05;

// Row-mask plans (every W window is the whole axis): the tensor core masks
// the H window through halo-row columns, so a brick's halo may span at most
// kRowsCols rows including chunk padding, in at most kRowsTiles h-chunks.
constexpr int64_t kRowsCols = 15;
constexpr int64_t kRowsTiles = 5;

Plan make_plan(const Axis& at, const Axis& ah, const Axis& aw, int ncap, bool allow_rows,
               bool allow_exact) {
    const int64_t H = ah.n, W = aw.n, KH = ah.k, KW = aw.k;
    Plan best;
    // mode 0: W windows by the tensor core (W unions up to 32 keys, a fixed
    // power-of-two chunk stride) or per-key masks (wider unions);
    // mode 1: whole-row W windows (KW == W), H windows by the tensor core
    for (int mode = 0; mode < 2; ++mode) {
    if (mode == 1 && !(allow_rows && KW == W && W <= ncap)) break;
    for (int64_t bw = 1; bw <= (aw.nq < 128 ? aw.nq : 128); ++bw) {
        const int64_t ew = (bw + KW - 1 < W) ? bw + KW - 1 : W;   // widest W union
        int64_t cwp = 0;
        if (mode == 1) cwp = 1;
        else if (ew <= 32) {
            cwp = ew <= 8 ? 8 : (ew <= 16 ? 16 : 32);
            // unions of 9 to 14 keys: rows of 12 or 14 keys where instances exist
            if (allow_exact && ew > 8 && ew <= 14) cwp = ew <= 12 ? 12 : 14;
        }
        const int64_t cw = cwp == 1 ? W : cwp ? cwp : (ew > ncap ? ncap : ew);
        const double col_cost = cwp ? kFastColumn : 1.0;
        int64_t nbw;
        const int64_t sw = axis_sum(aw, bw, cw, &nbw);
        for (int64_t bh = 1; bh <= ah.nq && bw * bh <= 128; ++bh) {
            const int64_t eh = (bh + KH - 1 < H) ? bh + KH - 1 : H;
            int64_t cr_max = (!cwp && ew > ncap) ? 1 : ncap / cw;
            if (cr_max > eh) cr_max = eh;
            // any row count up to the cap (fewer rows can mean fewer 32-key words)
            for (int64_t cr = cr_max; cr >= 1; --cr) {
                if (cwp == 1) {   // the widest halo's rows must fit the mask columns
                    const int64_t n_hc = (eh + cr - 1) / cr;
                    if (n_hc > kRowsTiles || n_hc * cr > kRowsCols) continue;
                }
                const int64_t n_mma = (cr * cw + 15) / 16 * 16;
                int64_t nbh;
                const int64_t sh = axis_sum(ah, bh, cr, &nbh);
                for (int64_t bt = 1; bt <= at.nq && bw * bh * bt <= 128; ++bt) {
                    int64_t nbt;
                    const int64_t st = axis_sum(at, bt, 1, &nbt);
                    const int64_t chunks = st * sh * sw;
                    const int64_t bricks = nbt * nbh * nbw;
                    // the softmax works in 32-key words, so a tile costs its width
                    // rounded up to a word
                    const int64_t n_words = (n_mma + 31) / 32 * 32;
                    const double cost =
                        double(chunks) * (double(n_words) * col_cost + double(n_mma) * kMmaColumn +
                                          kChunkOverhead) +
                        double(bricks) * kBrickOverhead;
                    const bool better =
                        best.bt == 0 || cost < best.cost - 1e-9 ||
                        (cost < best.cost + 1e-9 && bw * bh * bt > int64_t(best.bw) * best.bh * best.bt);
                    if (better) {
                        best.bt = int(bt); best.bh = int(bh); best.bw = int(bw);
                        best.cw = int(cw); best.cr = int(cr); best.n_mma = int(n_mma);
                        best.cwp = int(cwp);
                        best.bricks = bricks; best.chunks = chunks; best.cost = cost;
                    }
                }
            }
        }
    }
    }
    return best;
}

// Plans depend only on the grid, the query box, the window and the
// score-tile cap; they are cached (bounded, mutex-guarded) because the search
// takes ~0.1 ms.
Plan cached_plan(const Axis& at, const Axis& ah, const Axis& aw, int ncap, bool allow_rows,
                 bool allow_exact) {
    using Key = std::tuple<int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t,
                           int64_t, int64_t, int64_t, int64_t, int, bool, bool>;
    static std::mutex mu;
    static std::map<Key, Plan> cache;
    const Key key{at.nq, at.off, at.n, at.k, ah.nq, ah.off, ah.n, ah.k,
                  aw.nq, aw.off, aw.n, aw.k, ncap, allow_rows, allow_exact};
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    Plan pl = make_plan(at, ah, aw, ncap, allow_rows, allow_exact);
    pl.ncap = ncap;
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() >= 1024) cache.clear();
    cache.emplace(key, pl);
    return pl;
}

// The plan of a problem over the instance families of its head dim. HD <= 64
// has two: tiles of up to 128 keys (three single slots), and tiles of up to
// 96 keys in pairs of slots, where the next score tile is computed while the
// softmax works on the current one. The same plan runs 5-13 % faster on the
// paired tiles, but where the 96-key cap forces a plan the cost model rates
// worse, the extra chunks cost more than the overlap saves (measured on
// GB300 up to 16 % slower even at a 1 % higher modelled cost). So the paired
// family serves a problem exactly when its best plan costs no more than the
// 128-key family's. Whole-row W windows and 12/14-key rows are offered where
// the family has those instances.
Plan choose_plan(const Axis& at, const Axis& ah, const Axis& aw, int hd) {
    const int caps[2] = {na3d::default_ncap(hd), 96};
    Plan best;
    for (int i = 0; i < 2; ++i) {
        const int ncap = caps[i];
        if (i == 1 && (ncap == caps[0] || !na3d::variant_info(hd, 0, ncap, nullptr))) continue;
        const bool rows = na3d::variant_info(hd, 1, ncap, nullptr);
        const bool exact = na3d::variant_info(hd, 12, ncap, nullptr) && na3d::variant_info(hd, 14, ncap, nullptr);
        const Plan pl = cached_plan(at, ah, aw, ncap, rows, exact);
        if (best.bt == 0 || pl.cost <= best.cost) best = pl;
    }
    return best;
}

// ------------------------------------------------------------------ TMA descriptors

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The (B,T,H,W,NH,HD) tensor viewed as 5-D (NH*HD, W, H, T, B), with
// `token_stride` elements between consecutive grid positions: a box of
// {hd_box, bx, by, bz, 1} at x = head*HD + column picks one head's rows.
bool encode_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t H, int64_t W,
                int64_t NH, int64_t HD, int64_t token_stride, int hd_box, int bx, int by, int bz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[5] = {cuuint64_t(NH * HD), cuuint64_t(W), cuuint64_t(H), cuuint64_t(T),
                                cuuint64_t(B)};
    const cuuint64_t row = cuuint64_t(token_stride * 2);
    const cuuint64_t strides[4] = {row, row * W, row * W * H, row * W * H * T};
    const cuuint32_t box[5] = {cuuint32_t(hd_box), cuuint32_t(bx), cuuint32_t(by), cuuint32_t(bz), 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUtensorMapSwizzle swz = hd_box == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : hd_box == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major (outer, inner) bf16 matrix as a 2-D tensor map with a
// (box_inner, box_outer) box and the 128-byte swizzle (box_inner = 64).
bool encode_map_2d(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int box_inner,
                   int box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    const cuuint64_t strides[1] = {cuuint64_t(inner * 2)};
    const cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Do the byte ranges [a, a + a_bytes) and [b, b + b_bytes) intersect?
bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + uintptr_t(b_bytes) && y < x + uintptr_t(a_bytes);
}

}  // namespace

extern "C" {

const char* na3d_status_string(int status) {
    switch (status) {
        case NA3D_OK: return "NA3D_OK";
        case NA3D_ERR_NULL: return "NA3D_ERR_NULL: a required pointer is NULL";
        case NA3D_ERR_SHAPE: return "NA3D_ERR_SHAPE: every size must be >= 1 (and a query box inside the grid)";
        case NA3D_ERR_KERNEL: return "NA3D_ERR_KERNEL: window lengths must be odd and within 1..axis length";
        case NA3D_ERR_HEAD_DIM: return "NA3D_ERR_HEAD_DIM: head dimension must be a power of two >= 16";
        case NA3D_ERR_ALIGN: return "NA3D_ERR_ALIGN: tensor pointers must be 16-byte aligned";
        case NA3D_ERR_ALIAS: return "NA3D_ERR_ALIAS: out overlaps q, k or v";
        case NA3D_ERR_OVERFLOW: return "NA3D_ERR_OVERFLOW: sizes exceed int64 or TMA descriptor limits";
        case NA3D_ERR_ARCH: return "NA3D_ERR_ARCH: the current device is not sm_103 (GB300)";
        case NA3D_ERR_CUDA: return "NA3D_ERR_CUDA: a CUDA call failed";
        case NA3D_ERR_DEVICE_TIMEOUT: return "NA3D_ERR_DEVICE_TIMEOUT: a pipeline wait in the kernel gave up";
        case NA3D_ERR_UNSUPPORTED: return "NA3D_ERR_UNSUPPORTED: valid arguments this library does not implement";
        default: return "unknown na3d status";
    }
}

int na3d_plan(int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT, int64_t KH,
              int64_t KW, na3d_plan_info* info) {
    if (!info) return NA3D_ERR_NULL;
    const int rc = validate_shape(1, T, H, W, NH, HD, KT, KH, KW);
    if (rc != NA3D_OK) return rc;
    VariantInfo vi;
    const Plan pl = choose_plan(Axis{T, 0, T, KT}, Axis{H, 0, H, KH}, Axis{W, 0, W, KW}, int(HD));
    if (!na3d::variant_info(int(HD), pl.cwp, pl.ncap, &vi)) return NA3D_ERR_UNSUPPORTED;
    info->bt = pl.bt; info->bh = pl.bh; info->bw = pl.bw;
    info->cw = pl.cw; info->cr = pl.cr; info->n_mma = pl.n_mma;
    info->hd_box = vi.hd_box; info->stages = vi.stages;
    info->bricks_per_slice = pl.bricks;
    info->chunks_per_slice = pl.chunks;
    info->smem_bytes = vi.smem;
    info->w_stride = pl.cwp;
    info->tile_cap = pl.ncap;
    return NA3D_OK;
}

}  // extern "C"

namespace {

int fwd_region(const void* q, const void* k, const void* v, void* out, int64_t B, int64_t T,
               int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT, int64_t KH, int64_t KW,
               int64_t t0, int64_t h0, int64_t w0, int64_t Tq, int64_t Hq, int64_t Wq,
               int64_t q_token_stride, int64_t k_token_stride, int64_t v_token_stride, void* stream,
               int32_t withhold_k) {
    int rc = validate_shape(B, T, H, W, NH, HD, KT, KH, KW);
    if (rc != NA3D_OK) return rc;
    // the query box lies inside the grid
    if (Tq < 1 || Hq < 1 || Wq < 1 || t0 < 0 || h0 < 0 || w0 < 0 || t0 > T - Tq || h0 > H - Hq ||
        w0 > W - Wq)
        return NA3D_ERR_SHAPE;
    const int64_t kv_tokens = B * T * H * W, q_tokens = B * Tq * Hq * Wq;
    const int64_t out_bytes = q_tokens * NH * HD * 2;
    if (!q || !k || !v || !out) return NA3D_ERR_NULL;
    const int64_t strides[3] = {q_token_stride, k_token_stride, v_token_stride};
    const int64_t tokens[3] = {q_tokens, kv_tokens, kv_tokens};
    const int64_t grid_tokens[3] = {Tq * Hq * Wq, T * H * W, T * H * W};
    int64_t spans[3];
    for (int i = 0; i < 3; ++i) {
        if (strides[i] < NH * HD) return NA3D_ERR_SHAPE;
        if ((strides[i] * 2) % 16 != 0) return NA3D_ERR_ALIGN;
        int64_t span;
        if (!mul_ok(tokens[i] - 1, strides[i], &span) || !mul_ok(span + NH * HD, 2, &spans[i]) ||
            strides[i] * 2 >= (int64_t(1) << 40) / grid_tokens[i])
            return NA3D_ERR_OVERFLOW;
    }
    const void* ptrs[4] = {q, k, v, out};
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return NA3D_ERR_ALIGN;
    if (overlaps(out, out_bytes, q, spans[0]) || overlaps(out, out_bytes, k, spans[1]) ||
        overlaps(out, out_bytes, v, spans[2]))
        return NA3D_ERR_ALIAS;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NA3D_ERR_CUDA;
    if (major != 10 || minor != 3) return NA3D_ERR_ARCH;

    VariantInfo vi;
    const Plan pl = choose_plan(Axis{Tq, t0, T, KT}, Axis{Hq, h0, H, KH}, Axis{Wq, w0, W, KW}, int(HD));
    if (!na3d::variant_info(int(HD), pl.cwp, pl.ncap, &vi)) return NA3D_ERR_UNSUPPORTED;

    KernelParams kp;
    kp.B = int32_t(B); kp.T = int32_t(T); kp.H = int32_t(H); kp.W = int32_t(W); kp.NH = int32_t(NH);
    kp.Tq = int32_t(Tq); kp.Hq = int32_t(Hq); kp.Wq = int32_t(Wq);
    kp.t_off = int32_t(t0); kp.h_off = int32_t(h0); kp.w_off = int32_t(w0);
    kp.KT = int32_t(KT); kp.KH = int32_t(KH); kp.KW = int32_t(KW);
    kp.bt = pl.bt; kp.bh = pl.bh; kp.bw = pl.bw;
    kp.nbt = int32_t((Tq + pl.bt - 1) / pl.bt);
    kp.nbh = int32_t((Hq + pl.bh - 1) / pl.bh);
    kp.nbw = int32_t((Wq + pl.bw - 1) / pl.bw);
    kp.cw = pl.cw; kp.cr = pl.cr; kp.n_mma = pl.n_mma;
    // HD > 256: every head is cut into passes over 256 output columns, and a
    // work unit is one (head, pass) pair of a brick
    const int64_t npass = HD > 256 ? HD / 256 : 1;
    int npass_log2 = 0;
    while ((int64_t(1) << npass_log2) < npass) ++npass_log2;
    const int64_t nv = NH * npass;   // (head, pass) pairs per token
    kp.hd = int32_t(HD);
    kp.nreg = int32_t(HD > 256 ? HD / 64 : 0);
    kp.npass_log2 = npass_log2;
    const int64_t units = B * int64_t(kp.nbt) * kp.nbh * kp.nbw * nv;
    if (units >= (int64_t(1) << 31)) return NA3D_ERR_OVERFLOW;
    kp.n_units = int32_t(units);
    kp.out = static_cast<uint16_t*>(out);
    // rows are HD * 2 >= 32 bytes: 32-byte stores when the base allows them
    kp.out_v8 = (reinterpret_cast<uintptr_t>(out) % 32u) == 0u ? 1 : 0;
    kp.withhold_k = withhold_k;
    kp.div_nh = na3d::make_fastdiv(int32_t(nv));
    kp.div_nbw = na3d::make_fastdiv(kp.nbw);
    kp.div_nbh = na3d::make_fastdiv(kp.nbh);
    kp.div_nbt = na3d::make_fastdiv(kp.nbt);
    kp.div_cr = na3d::make_fastdiv(kp.cr);
    kp.div_cw = na3d::make_fastdiv(kp.cw);

    // Head groups: the largest power of two dividing NH whose groups still
    // fill the persistent grid within 3 % of the best balance.
    const int64_t slots = int64_t(sms) * vi.ctas_per_sm;   // persistent CTAs
    auto balance = [&](int64_t hg) {
        const int64_t groups = units / hg;
        const int64_t waves = (groups + slots - 1) / slots;
        return double(groups) / double(waves * slots);
    };
    double best = 0;
    for (int64_t d = 1; d <= nv; d *= 2)
        if (nv % d == 0 && balance(d) > best) best = balance(d);
    kp.hg = 1;
    for (int64_t d = 1; HD >= 128 && d <= nv; d *= 2)   // the kernel groups heads for HD >= 128
        if (nv % d == 0 && balance(d) >= best - 0.03) kp.hg = int32_t(d);

    // Q over the query box, K and V over the whole grid
    CUtensorMap tq, tk, tv;
    if (!encode_map(&tq, q, B, Tq, Hq, Wq, NH, HD, q_token_stride, vi.hd_box, pl.bw, pl.bh, pl.bt) ||
        !encode_map(&tk, k, B, T, H, W, NH, HD, k_token_stride, vi.hd_box, pl.cw, pl.cr, 1) ||
        !encode_map(&tv, v, B, T, H, W, NH, HD, v_token_stride, vi.hd_box, pl.cw, pl.cr, 1))
        return NA3D_ERR_CUDA;

    const int64_t groups = units / kp.hg;
    const int grid = int(groups < slots ? groups : slots);
    if (na3d::launch_fwd(int(HD), pl.cwp, pl.ncap, tq, tk, tv, kp, grid, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return NA3D_ERR_CUDA;
    return NA3D_OK;
}

}  // namespace

extern "C" {

int na3d_fwd_region(const void* q, const void* k, const void* v, void* out, int64_t B, int64_t T,
                    int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT, int64_t KH, int64_t KW,
                    int64_t t0, int64_t h0, int64_t w0, int64_t Tq, int64_t Hq, int64_t Wq,
                    int64_t q_token_stride, int64_t k_token_stride, int64_t v_token_stride,
                    void* stream) {
    return fwd_region(q, k, v, out, B, T, H, W, NH, HD, KT, KH, KW, t0, h0, w0, Tq, Hq, Wq,
                      q_token_stride, k_token_stride, v_token_stride, stream, -1);
}

int na3d_selftest_withhold(const void* q, const void* k, const void* v, void* out, int64_t B,
                           int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT,
                           int64_t KH, int64_t KW, int64_t chunk, void* stream) {
    if (chunk < 0 || chunk >= (int64_t(1) << 30)) return NA3D_ERR_SHAPE;
    return fwd_region(q, k, v, out, B, T, H, W, NH, HD, KT, KH, KW, 0, 0, 0, T, H, W, NH * HD,
                      NH * HD, NH * HD, stream, int32_t(chunk));
}

int na3d_fwd_strided(const void* q, const void* k, const void* v, void* out, int64_t B, int64_t T,
                     int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT, int64_t KH,
                     int64_t KW, int64_t q_token_stride, int64_t k_token_stride,
                     int64_t v_token_stride, void* stream) {
    return na3d_fwd_region(q, k, v, out, B, T, H, W, NH, HD, KT, KH, KW, 0, 0, 0, T, H, W,
                           q_token_stride, k_token_stride, v_token_stride, stream);
}

int na3d_fwd(const void* q, const void* k, const void* v, void* out, int64_t B, int64_t T,
             int64_t H, int64_t W, int64_t NH, int64_t HD, int64_t KT, int64_t KH, int64_t KW,
             void* stream) {
    return na3d_fwd_strided(q, k, v, out, B, T, H, W, NH, HD, KT, KH, KW, NH * HD, NH * HD,
                            NH * HD, stream);
}

int na3d_qkv_proj(const void* x, const void* w, const void* bias, void* qkv, int64_t M, int64_t C,
                  int64_t NH, int64_t HD, void* stream) {
    if (M < 1 || NH < 1 || C < 1 || HD < 1) return NA3D_ERR_SHAPE;
    if (!is_pow2(HD) || HD < 16) return NA3D_ERR_HEAD_DIM;
    if (C % 8 != 0) return NA3D_ERR_ALIGN;   // rows of x and W must be 16-byte aligned
    int64_t N, xb, wb, ob;
    if (!mul_ok(3 * NH, HD, &N) || !mul_ok(M, C, &xb) || !mul_ok(xb, 2, &xb) || !mul_ok(N, C, &wb) ||
        !mul_ok(wb, 2, &wb) || !mul_ok(M, N, &ob) || !mul_ok(ob, 2, &ob))
        return NA3D_ERR_OVERFLOW;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || C >= (int64_t(1) << 31))
        return NA3D_ERR_OVERFLOW;
    if (!x || !w || !qkv) return NA3D_ERR_NULL;
    const void* ptrs[3] = {x, w, qkv};
    for (const void* p : ptrs)
        if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return NA3D_ERR_ALIGN;
    if (bias && reinterpret_cast<uintptr_t>(bias) % 2 != 0) return NA3D_ERR_ALIGN;
    if (overlaps(qkv, ob, x, xb) || overlaps(qkv, ob, w, wb) || (bias && overlaps(qkv, ob, bias, N * 2)))
        return NA3D_ERR_ALIAS;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NA3D_ERR_CUDA;
    if (major != 10 || minor != 3) return NA3D_ERR_ARCH;

    na3d::ProjParams pp;
    pp.M = int32_t(M);
    pp.C = int32_t(C);
    pp.N = int32_t(N);
    pp.Nq = int32_t(NH * HD);
    pp.n_tiles_n = int32_t((N + 255) / 256);
    const int64_t tiles = ((M + 127) / 128) * pp.n_tiles_n;
    if (tiles >= (int64_t(1) << 31)) return NA3D_ERR_OVERFLOW;
    pp.n_tiles = int32_t(tiles);
    pp.k_blocks = int32_t((C + 63) / 64);
    pp.out_v8 = (reinterpret_cast<uintptr_t>(qkv) % 32u) == 0u ? 1 : 0;   // rows: N * 2 = 96k bytes
    pp.q_scale = float(1.0 / __builtin_sqrt(double(HD)));
    pp.bias = static_cast<const uint16_t*>(bias);
    pp.qkv = static_cast<uint16_t*>(qkv);
    CUtensorMap tx, tw;
    if (!encode_map_2d(&tx, x, C, M, 64, 128) || !encode_map_2d(&tw, w, C, N, 64, 256))
        return NA3D_ERR_CUDA;
    const int grid = int(tiles < sms ? tiles : sms);
    if (na3d::launch_qkv_proj(tx, tw, pp, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return NA3D_ERR_CUDA;
    return NA3D_OK;
}

int na3d_device_status(void* stream) {
    unsigned int flag = 0, pflag = 0;
    if (na3d::take_device_error(static_cast<cudaStream_t>(stream), &flag) != cudaSuccess ||
        na3d::take_proj_error(static_cast<cudaStream_t>(stream), &pflag) != cudaSuccess)
        return NA3D_ERR_CUDA;
    return (flag || pflag) ? NA3D_ERR_DEVICE_TIMEOUT : NA3D_OK;
}

}  // extern "C"
