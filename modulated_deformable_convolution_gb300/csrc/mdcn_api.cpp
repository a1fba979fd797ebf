// C ABI of libmdcn (include/mdcn.h): argument validation following
// "TensorRT plugin walkthrough: modulatedDeformConvPlugin" (section 2 shape
// rule, section 3 attribute ranges, section 4 type and dimension bindings),
// the execution plan, and dispatch to the kernels. No exception leaves this
// file; every entry point returns an mdcn_status.
#include "mdcn.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "mdcn_backward.h"
#include "mdcn_launch.h"
#include "mdcn_plan.h"

struct mdcn_handle_ {
    mdcn_attrs attrs;
    mdcn_tuning tuning;
};

namespace {

using mdcn::Plan;

thread_local int g_last_cuda_error = 0;

mdcn_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return MDCN_ERR_CUDA;
}

constexpr int64_t kI31 = (int64_t(1) << 31) - 1;
constexpr int64_t kI62 = int64_t(1) << 62;

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// a*b*... with overflow detection against kI62
bool mul_ok(int64_t& acc, int64_t v) {
    if (v < 0 || (v != 0 && acc > kI62 / v)) return false;
    acc *= v;
    return true;
}

bool attrs_valid(const mdcn_attrs& a) {
    for (int i = 0; i < 2; ++i) {
        if (a.stride[i] < 1 || a.dilation[i] < 1 || a.padding[i] < 0) return false;
        if (a.stride[i] > kI31 || a.dilation[i] > kI31 || a.padding[i] > kI31) return false;
    }
    return a.group >= 1 && a.deformable_group >= 1 && a.group <= kI31 && a.deformable_group <= kI31;
}

// Section 2/4 bindings and the section-2 output rule.
mdcn_status check_dims(const mdcn_attrs& a, const mdcn_dims& d, int64_t out[4]) {
    for (int i = 0; i < 4; ++i)
        if (d.x[i] < 1 || d.offset[i] < 1 || d.mask[i] < 1 || d.weight[i] < 1) return MDCN_ERR_SHAPE;
    const int64_t N = d.x[0], Cin = d.x[1];
    const int64_t Cout = d.weight[0], Cg = d.weight[1], kh = d.weight[2], kw = d.weight[3];
    const int64_t Ho = d.offset[2], Wo = d.offset[3];
    for (int i = 0; i < 4; ++i)
        if (d.x[i] > kI31 || d.offset[i] > kI31 || d.mask[i] > kI31 || d.weight[i] > kI31) return MDCN_ERR_UNSUPPORTED;
    int64_t K = kh;
    if (!mul_ok(K, kw)) return MDCN_ERR_UNSUPPORTED;
    const int64_t dg = a.deformable_group, g = a.group;
    if (d.offset[0] != N || d.mask[0] != N) return MDCN_ERR_SHAPE;          // offset_0 = mask_0 = x_0
    if (d.mask[2] != Ho || d.mask[3] != Wo) return MDCN_ERR_SHAPE;          // mask_2 = offset_2, mask_3 = offset_3
    int64_t oc = 2 * dg;
    if (!mul_ok(oc, K)) return MDCN_ERR_UNSUPPORTED;
    if (d.offset[1] != oc) return MDCN_ERR_SHAPE;                           // 2*dg*kh*kw offset channels
    if (d.mask[1] != dg * K) return MDCN_ERR_SHAPE;                         // dg*kh*kw mask channels
    if (Cin % g != 0 || Cout % g != 0 || Cg != Cin / g) return MDCN_ERR_SHAPE;  // weight [Cout, Cin/group, kh, kw]
    if (Cin % dg != 0) return MDCN_ERR_SHAPE;
    if (d.bias != 0 && d.bias != Cout) return MDCN_ERR_SHAPE;               // bias_0 = weight_0
    // element counts
    int64_t n;
    n = N; if (!mul_ok(n, Cin) || !mul_ok(n, d.x[2]) || !mul_ok(n, d.x[3])) return MDCN_ERR_UNSUPPORTED;
    n = N; if (!mul_ok(n, oc) || !mul_ok(n, Ho) || !mul_ok(n, Wo)) return MDCN_ERR_UNSUPPORTED;
    n = N; if (!mul_ok(n, Cout) || !mul_ok(n, Ho) || !mul_ok(n, Wo)) return MDCN_ERR_UNSUPPORTED;
    n = Cout; if (!mul_ok(n, Cg) || !mul_ok(n, K)) return MDCN_ERR_UNSUPPORTED;
    out[0] = N;
    out[1] = Cout;
    out[2] = Ho;
    out[3] = Wo;
    return MDCN_OK;
}

// One CTA's fp32 partial accumulator of a split tile: acc_cols x 128 rows.
size_t partial_slot_bytes(const Plan& p) {
    return static_cast<size_t>(p.acc_cols) * mdcn::kTileM * sizeof(float);
}

mdcn_status make_plan(const mdcn_attrs& a, const mdcn_tuning& tuning, const mdcn_dims* d, mdcn_dtype dtype,
                      Plan* pl) {
    if (!d || !pl) return MDCN_ERR_NULL;
    if (dtype != MDCN_F32 && dtype != MDCN_F16 && dtype != MDCN_BF16) return MDCN_ERR_DTYPE;
    int64_t od[4];
    mdcn_status s = check_dims(a, *d, od);
    if (s != MDCN_OK) return s;
    Plan p;
    std::memset(&p, 0, sizeof(p));
    p.N = d->x[0];
    p.Cin = d->x[1];
    p.H = d->x[2];
    p.W = d->x[3];
    p.Cout = d->weight[0];
    p.kh = d->weight[2];
    p.kw = d->weight[3];
    p.Ho = d->offset[2];
    p.Wo = d->offset[3];
    p.sh = static_cast<int32_t>(a.stride[0]);
    p.sw = static_cast<int32_t>(a.stride[1]);
    p.ph = static_cast<int32_t>(a.padding[0]);
    p.pw = static_cast<int32_t>(a.padding[1]);
    p.dh = static_cast<int32_t>(a.dilation[0]);
    p.dw = static_cast<int32_t>(a.dilation[1]);
    p.group = static_cast<int32_t>(a.group);
    p.dg = static_cast<int32_t>(a.deformable_group);
    p.dtype = static_cast<int32_t>(dtype);
    p.has_bias = d->bias != 0;
    const int64_t K = p.kh * p.kw;
    const int64_t Cg = p.Cin / a.group, Og = p.Cout / a.group, Cd = p.Cin / a.deformable_group;
    // positions are compared in fp32: keep every coordinate exactly representable
    if (p.H >= (1 << 24) || p.W >= (1 << 24)) return MDCN_ERR_UNSUPPORTED;
    if ((p.Ho - 1) * a.stride[0] + (p.kh - 1) * a.dilation[0] >= (1 << 24) ||
        (p.Wo - 1) * a.stride[1] + (p.kw - 1) * a.dilation[1] >= (1 << 24))
        return MDCN_ERR_UNSUPPORTED;
    if (K > kI31 || Cg > kI31 || Og > kI31) return MDCN_ERR_UNSUPPORTED;
    p.K = static_cast<int32_t>(K);
    p.Cg = static_cast<int32_t>(Cg);
    p.Og = static_cast<int32_t>(Og);
    p.Cd = static_cast<int32_t>(Cd);
    p.P = p.Ho * p.Wo;
    p.NP = p.N * p.P;
    if (p.NP > kI31) return MDCN_ERR_UNSUPPORTED;  // 32-bit pixel arithmetic in the kernels

    // The direct CUDA-core kernel where each output sums over few products per
    // tap (Cin/group x Cout/group <= 16, e.g. depthwise): the implicit GEMM would
    // pad each channel unit to a 128-byte k-tile and each group's outputs to 16
    // MMA columns (measured: a depthwise 128-channel 80x80 layer 1343 us fused,
    // ~250 us direct; groups of 8 x 8 channels are faster fused, 158 against
    // 258 us). It needs no workspace beyond the status word.
    {
        const bool fits = Og <= mdcn::kDirectMaxOg &&
                          mdcn::direct_groups_per_thread(Og) * Og * Cg * K * 4 <= mdcn::kDirectMaxSmem &&
                          p.group <= 65535 && p.N <= 65535;
        if (tuning.path == 2 && !fits) return MDCN_ERR_UNSUPPORTED;
        if (fits && (tuning.path == 2 || (tuning.path == 0 && Cg * Og <= 16))) {
            p.direct = 1;
            p.off_xt = p.off_wp = p.off_part = p.ws_bytes = mdcn::kStatusBytes;
            // depthwise with deformable groups of whole 4-channel chunks: the
            // channels-last form, on a copy of x [N*H*W + 1][Cin] in the workspace
            const int64_t elem_b = dtype == MDCN_F32 ? 4 : 2;
            int64_t xt_bytes = p.N * p.H;  // N <= 65535, H < 2^24
            bool xt_ok = mul_ok(xt_bytes, p.W);
            xt_bytes += 1;  // the zero pixel
            xt_ok = xt_ok && mul_ok(xt_bytes, p.Cin) && mul_ok(xt_bytes, elem_b);
            if (Cg == 1 && Og == 1 && p.Cin % 4 == 0 && Cd % 4 == 0 && K <= mdcn::kDirectClMaxTaps &&
                p.Cin <= 65535ll * 128 && xt_ok && tuning.path != 2) {
                p.direct_cl = 1;
                p.ws_bytes = align256(p.off_xt + static_cast<size_t>(xt_bytes));
            }
            *pl = p;
            return MDCN_OK;
        }
    }

    const int64_t elem = dtype == MDCN_F32 ? 4 : 2;
    p.BKc = static_cast<int32_t>(128 / elem);
    const int64_t U = gcd64(Cg, Cd);
    const int64_t UP = round_up(U, p.BKc);
    p.U = static_cast<int32_t>(U);
    p.UP = static_cast<int32_t>(UP);
    p.Ug = static_cast<int32_t>(Cg / U);
    p.nch = static_cast<int32_t>(UP / p.BKc);
    p.ntb = static_cast<int32_t>(ceil_div(K, mdcn::kTapBlock));
    int64_t KT = Cg / U;
    if (!mul_ok(KT, K) || !mul_ok(KT, p.nch) || KT * p.BKc > kI31) return MDCN_ERR_UNSUPPORTED;
    p.KT = static_cast<int32_t>(KT);
    p.KP = KT * p.BKc;
    p.Cp = (p.Cin / U) * UP;
    if (ceil_div(p.Cp, 32) > 65535) return MDCN_ERR_UNSUPPORTED;

    // N tiling: up to 256 output channels per MMA, two MMAs (512 TMEM columns) per
    // tile; tuning.ntile caps the output channels of one tile
    {
        const int64_t cap = tuning.ntile > 0 ? tuning.ntile : 512;
        p.ntiles_n = static_cast<int32_t>(ceil_div(Og, cap));
        const int64_t per = ceil_div(Og, p.ntiles_n);
        p.nsub = per <= 256 ? 1 : 2;
        p.BNs = static_cast<int32_t>(round_up(ceil_div(per, p.nsub), 16));
    }
    p.acc_cols = p.nsub * p.BNs;
    p.nacc = 2 * p.acc_cols <= 512 ? 2 : 1;

    // pixel tiles: 8 x 16 blocks of one image when they waste (almost) no rows,
    // else 128 consecutive pixels of N*Ho*Wo
    p.TH = mdcn::kTileH;
    p.TW = mdcn::kTileW;
    p.tiles_x = ceil_div(p.Wo, p.TW);
    p.tiles_y = ceil_div(p.Ho, p.TH);
    const double waste = 1.0 - static_cast<double>(p.P) / static_cast<double>(p.tiles_x * p.TW * p.tiles_y * p.TH);
    int32_t mode = tuning.tile_mode >= 0 ? tuning.tile_mode : (waste <= 0.06 ? 1 : 0);
    p.tile_mode = mode;
    p.plain = 0;
    p.mtiles = mode == 1 ? p.N * p.tiles_x * p.tiles_y : ceil_div(p.NP, mdcn::kTileM);
    int64_t tt = p.mtiles;
    if (!mul_ok(tt, p.ntiles_n) || !mul_ok(tt, p.group)) return MDCN_ERR_UNSUPPORTED;
    p.tiles_total = tt;

    const int64_t halves = dtype == MDCN_F32 ? 2 : 1;
    p.a_bytes = static_cast<int32_t>(mdcn::kTileM * 128 * halves);
    p.b_bytes = static_cast<int32_t>(p.nsub * p.BNs * 128 * halves);
    p.desc_size = dtype == MDCN_F32 ? 32 : 16;
    p.desc_slot_bytes = mdcn::kTileM * mdcn::kTapBlock * p.desc_size;
    // TMA-store epilogue: 2-D tiles whose 16-channel boxes stay inside a group
    // and whose output rows are 16-byte multiples
    {
        // vector epilogue: every group of 16/elem consecutive output pixels that
        // it stores is inside one row (2-D tiles) or one image, and 16-byte aligned
        const int64_t v = 16 / elem;
        p.epi_vec = (p.P % v == 0 && (mode == 0 || p.Wo % v == 0)) ? 1 : 0;
    }
    p.epi_bytes = mdcn::kEpiWarps * 16 * 32 * static_cast<int32_t>(elem);
    const int32_t fixed = 1024 + 2 * p.desc_slot_bytes + p.epi_bytes + mdcn::kBiasBytes + 512;
    // automatic: 2 k-tiles in production at once, which hides the gather's
    // latency while the contraction of a k-tile is short; 1 (all 8 warps on
    // one k-tile) when the accumulator is wider than 256 columns and each
    // k-tile's contraction takes about as long as its gather (measured on
    // the named workloads)
    p.kgroups = tuning.kgroups > 0 ? tuning.kgroups : (p.acc_cols > 256 ? 1 : 2);
    // A stages in tensor memory (32 columns each, after the accumulators):
    // 16-bit types whose gather warps form 2 groups (each warp then writes the
    // tile rows of its own tensor-memory lane quarter), with one accumulator
    // where two leave no room (measured: multi-dg bf16, 256 columns, 41.6 ->
    // 39.7 us with one accumulator and the A stages in tensor memory).
    {
        const int32_t st_req = tuning.stages > 0 ? tuning.stages : 4;
        const int32_t room = 512 - 32 * st_req;
        int32_t a_tmem = 0;
        if (tuning.a_operand != 1 && elem == 2 && p.kgroups == 2) {
            if (p.nacc * p.acc_cols <= room) {
                a_tmem = 1;
            } else if (p.acc_cols <= room) {
                p.nacc = 1;
                a_tmem = 1;
            }
        }
        if (tuning.a_operand == 2 && !a_tmem) return MDCN_ERR_UNSUPPORTED;
        p.a_tmem = a_tmem;
        if (a_tmem) p.a_bytes = 0;  // no A stages in shared memory
    }
    const int32_t per_stage = p.a_bytes + p.b_bytes;
    // stages: 2, 4, 6 or 8; the gather produces kgroups k-tiles at once (1, 2
    // or 4, dividing the stage count)
    const int32_t max_stages = (mdcn::kSmemLimit - fixed) / per_stage;
    int32_t stages = tuning.stages > 0 ? tuning.stages : (max_stages >= 4 ? 4 : 2);
    if (stages < 2 || stages > 8 || (stages & 1) || stages > max_stages) return MDCN_ERR_UNSUPPORTED;
    p.stages = stages;
    if (stages % p.kgroups != 0) return MDCN_ERR_UNSUPPORTED;
    p.smem_bytes = fixed + stages * per_stage;
    p.a_col0 = p.nacc * p.acc_cols;
    {
        const int32_t used = p.a_col0 + (p.a_tmem ? 32 * stages : 0);
        if (used > 512) return MDCN_ERR_UNSUPPORTED;
        int32_t cols = 32;
        while (cols < used) cols <<= 1;
        p.tmem_cols = cols;
    }
    p.grid = 0;  // set at launch from the SM count

    // workspace: [status word, split-tile counters: 1 KB][x channels-last][packed weight][partials]
    // channels-last conversion stages whole pixels in 40 KB of shared memory
    if ((p.Cp + 16 / elem) * elem > 40 * 1024) return MDCN_ERR_UNSUPPORTED;
    if (p.N * p.H * p.W > kI31) return MDCN_ERR_UNSUPPORTED;
    // channels-last x, plus one all-zero pixel that the gather reads for
    // corners outside the image
    int64_t xt = p.N * p.H;
    if (!mul_ok(xt, p.W)) return MDCN_ERR_UNSUPPORTED;
    xt += 1;
    if (!mul_ok(xt, p.Cp) || !mul_ok(xt, elem)) return MDCN_ERR_UNSUPPORTED;
    int64_t rows = p.Cout * halves;
    if (rows < p.BNs) rows = p.BNs;
    p.wp_rows = rows;
    int64_t wpb = rows;
    if (!mul_ok(wpb, p.KP) || !mul_ok(wpb, elem) || rows > kI31) return MDCN_ERR_UNSUPPORTED;
    {
        // register-blocked channels-last conversion: H*W and the unit in whole
        // 16-byte vectors, grid within limits
        const int64_t vec = 16 / elem;
        const int64_t pblocks = (p.H * p.W / vec + 3) / 4;
        const int64_t cblocks = (p.Cp / vec + 7) / 8;
        p.xt_block = ((p.H * p.W) % vec == 0 && p.U % vec == 0 && p.N <= 65535 && cblocks <= 65535 &&
                      (pblocks + 7) / 8 <= 65535)
                         ? 1
                         : 0;
    }
    // stream-K: fp32 partial accumulators of split tiles, one slot per CTA.
    // Whether any tile is split depends on the grid (the SM count), which
    // finish_plan sets; until then the workspace size is the bound for the
    // largest grid.
    p.total_kt = p.tiles_total;
    if (!mul_ok(p.total_kt, p.KT) || p.total_kt > kI31) return MDCN_ERR_UNSUPPORTED;  // 32-bit tile arithmetic
    p.off_xt = mdcn::kStatusBytes;
    p.off_wp = align256(p.off_xt + static_cast<size_t>(xt));
    p.off_part = align256(p.off_wp + static_cast<size_t>(wpb));
    p.ws_bytes = align256(p.off_part + partial_slot_bytes(p) * mdcn::kMaxCtas);
    *pl = p;
    return MDCN_OK;
}

// Finishes a plan for a device with `sms` SMs: the persistent grid, each
// CTA's range of the k-tile sequence, and the workspace size, which holds the
// partial-sum slots (one per CTA) only when some tile is split between CTAs.
void finish_plan(Plan* p, const mdcn_tuning& tuning, int sms) {
    if (p->direct) return;  // no persistent grid, no partial sums
    int64_t grid = sms > 0 ? sms : 1;
    if (grid > mdcn::kMaxCtas) grid = mdcn::kMaxCtas;
    if (tuning.max_ctas > 0 && tuning.max_ctas < grid) grid = tuning.max_ctas;
    if (grid > p->total_kt) grid = p->total_kt;
    // stream-K split: equal consecutive k-tile ranges, none empty. Splitting a
    // tile costs its other CTAs an fp32 partial write each and its owner a
    // read of them, so ranges stay whole tiles unless the busiest CTA's share
    // drops clearly (measured break-even: about 15% plus 4 k-tiles).
    const int64_t split = (p->total_kt + grid - 1) / grid;
    const int64_t whole = (p->tiles_total + grid - 1) / grid * p->KT;
    p->kt_per_cta = split * 115 / 100 + 4 < whole ? split : whole;
    p->grid = static_cast<int32_t>((p->total_kt + p->kt_per_cta - 1) / p->kt_per_cta);
    p->ws_bytes = mdcn::splitk_needed(*p) ? align256(p->off_part + partial_slot_bytes(*p) * p->grid) : p->off_part;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// compute capability 10.3 check, cached per device; *sms = SM count
mdcn_status check_device(int* sms = nullptr) {
    static std::atomic<int> cached[64];
    static std::atomic<int> sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return MDCN_ERR_UNSUPPORTED;
    int v = cached[dev].load(std::memory_order_acquire);
    if (v == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        sm_count[dev].store(nsm, std::memory_order_relaxed);
        v = (major == 10 && minor == 3) ? 1 : 2;
        if (v == 1) {
            for (int dt = 0; dt < 3; ++dt) {
                e = mdcn::prepare_fused_attributes(dt, mdcn::kSmemLimit);
                if (e != cudaSuccess) return cuda_fail(e);
            }
        }
        cached[dev].store(v, std::memory_order_release);
    }
    if (sms) *sms = sm_count[dev].load(std::memory_order_relaxed);
    return v == 1 ? MDCN_OK : MDCN_ERR_ARCH;
}

mdcn_status check_forward_args(mdcn_handle h, const void* x, const void* offset, const void* mask, const void* weight,
                               const void* bias, void* out, void* ws, const mdcn_dims* dims) {
    if (!h || !x || !offset || !mask || !weight || !out || !ws || !dims) return MDCN_ERR_NULL;
    if ((bias == nullptr) != (dims->bias == 0)) return bias ? MDCN_ERR_SHAPE : MDCN_ERR_NULL;
    if (!aligned16(x) || !aligned16(offset) || !aligned16(mask) || !aligned16(weight) || !aligned16(out) ||
        !aligned16(ws) || (bias && !aligned16(bias)))
        return MDCN_ERR_ALIGN;
    return MDCN_OK;
}

// Plan + workspace-size + device checks shared by the fused-path entry points.
mdcn_status plan_for(const mdcn_attrs& attrs, const mdcn_tuning& tuning, const mdcn_dims* dims, mdcn_dtype dtype,
                     size_t ws_bytes, Plan* p) {
    mdcn_status s = make_plan(attrs, tuning, dims, dtype, p);
    if (s != MDCN_OK) return s;
    // below the size of any plan (no partial slots): refused before the device check
    if (ws_bytes < p->off_part) return MDCN_ERR_WORKSPACE;
    int sms = 0;
    s = check_device(&sms);
    if (s != MDCN_OK) return s;
    finish_plan(p, tuning, sms);
    if (ws_bytes < p->ws_bytes) return MDCN_ERR_WORKSPACE;
    return MDCN_OK;
}

// Workspace bytes of a forward on the current device, or, where no usable
// device is current, the bound for any device.
size_t forward_ws_bytes(const mdcn_tuning& tuning, Plan p) {
    const int last = g_last_cuda_error;  // a size query does not report the device probe's error
    int sms = 0;
    if (check_device(&sms) == MDCN_OK) finish_plan(&p, tuning, sms);
    g_last_cuda_error = last;
    return p.ws_bytes;
}

mdcn_status plan_for_call(mdcn_handle h, const mdcn_dims* dims, mdcn_dtype dtype, size_t ws_bytes, Plan* p) {
    return plan_for(h->attrs, h->tuning, dims, dtype, ws_bytes, p);
}

// The offset/mask front end of the pack form, as an ordinary convolution:
// the layer's stride, padding and dilation, group 1, no deformation, and
// 3*dg*kh*kw output channels with a bias. Its spatial size is the
// convolution's, which the layer's offset and mask dims must match.
mdcn_status front_end_problem(const mdcn_attrs& a, const mdcn_dims* d, mdcn_attrs* fa, mdcn_dims* fd) {
    if (!d) return MDCN_ERR_NULL;
    const int64_t kh = d->weight[2], kw = d->weight[3], K = kh * kw;
    const int64_t H = d->x[2], W = d->x[3];
    if (kh < 1 || kw < 1 || H < 1 || W < 1 || K > kI31) return MDCN_ERR_SHAPE;
    const int64_t Ho = (H + 2 * a.padding[0] - a.dilation[0] * (kh - 1) - 1) / a.stride[0] + 1;
    const int64_t Wo = (W + 2 * a.padding[1] - a.dilation[1] * (kw - 1) - 1) / a.stride[1] + 1;
    if (H + 2 * a.padding[0] < a.dilation[0] * (kh - 1) + 1 || W + 2 * a.padding[1] < a.dilation[1] * (kw - 1) + 1)
        return MDCN_ERR_SHAPE;  // empty convolution output
    if (d->offset[2] != Ho || d->offset[3] != Wo) return MDCN_ERR_SHAPE;
    *fa = a;
    fa->group = 1;
    fa->deformable_group = 1;
    *fd = *d;
    const int64_t com = 3 * a.deformable_group * K;
    fd->weight[0] = com;
    fd->weight[1] = d->x[1];
    fd->offset[1] = 2 * K;
    fd->mask[1] = K;
    fd->bias = com;
    return MDCN_OK;
}

// Problem of a backward call: the forward's checks (section 2/4 bindings,
// section 3 attributes) plus the limits of the backward's kernels and of the
// cuBLAS dimensions (32-bit), then the chunking and workspace layout.
// Per-chunk buffers (columns, their gradients, x and grad_x of the chunk's
// images). Measured on the named workloads: chunks of 256 MB (one chunk for
// neck and multi-dg, two for large-channel) run 16-20% faster than chunks that
// stay in the 129 MB L2, from fewer launches and larger GEMMs.
constexpr size_t kBwdChunkBudget = size_t(256) << 20;

mdcn_status make_bwd_plan(const mdcn_attrs& a, const mdcn_dims* d, mdcn_dtype dtype, mdcn::BwdPlan* p) {
    if (!d || !p) return MDCN_ERR_NULL;
    if (dtype != MDCN_F32 && dtype != MDCN_F16 && dtype != MDCN_BF16) return MDCN_ERR_DTYPE;
    int64_t od[4];
    mdcn_status s = check_dims(a, *d, od);
    if (s != MDCN_OK) return s;
    mdcn::BwdPlan b;
    std::memset(&b, 0, sizeof(b));
    b.N = d->x[0];
    b.Cin = d->x[1];
    b.H = d->x[2];
    b.W = d->x[3];
    b.Cout = d->weight[0];
    b.kh = d->weight[2];
    b.kw = d->weight[3];
    b.Ho = d->offset[2];
    b.Wo = d->offset[3];
    b.sh = static_cast<int32_t>(a.stride[0]);
    b.sw = static_cast<int32_t>(a.stride[1]);
    b.ph = static_cast<int32_t>(a.padding[0]);
    b.pw = static_cast<int32_t>(a.padding[1]);
    b.dh = static_cast<int32_t>(a.dilation[0]);
    b.dw = static_cast<int32_t>(a.dilation[1]);
    b.group = static_cast<int32_t>(a.group);
    b.dg = static_cast<int32_t>(a.deformable_group);
    b.dtype = static_cast<int32_t>(dtype);
    b.has_bias = d->bias != 0;
    const int64_t K = b.kh * b.kw;
    // positions are formed in fp32: keep every coordinate exactly representable
    if (b.H >= (1 << 24) || b.W >= (1 << 24)) return MDCN_ERR_UNSUPPORTED;
    if ((b.Ho - 1) * a.stride[0] + (b.kh - 1) * a.dilation[0] >= (1 << 24) ||
        (b.Wo - 1) * a.stride[1] + (b.kw - 1) * a.dilation[1] >= (1 << 24))
        return MDCN_ERR_UNSUPPORTED;
    b.P = b.Ho * b.Wo;
    int64_t kcg = K;
    if (!mul_ok(kcg, b.Cin / a.group) || kcg > kI31 || b.P > kI31 || b.Cout / a.group > kI31 || K > kI31)
        return MDCN_ERR_UNSUPPORTED;  // cuBLAS dimensions are 32-bit
    b.K = static_cast<int32_t>(K);
    b.Cg = static_cast<int32_t>(b.Cin / a.group);
    b.Og = static_cast<int32_t>(b.Cout / a.group);
    b.Cd = static_cast<int32_t>(b.Cin / a.deformable_group);
    int64_t cols = b.P;  // column elements of one image, and its x
    if (!mul_ok(cols, K) || !mul_ok(cols, b.Cin) || !mul_ok(cols, 32)) return MDCN_ERR_UNSUPPORTED;
    // the sampling backward's grid: (pixel blocks, dg*K, images of a chunk)
    if (static_cast<int64_t>(b.dg) * K > 65535) return MDCN_ERR_UNSUPPORTED;
    mdcn::plan_backward(&b, kBwdChunkBudget);
    // the transposes' tile counts fit 32-bit block indices
    if ((b.H * b.W / 32 + 1) * (b.Cin / 32 + 1) >= kI31) return MDCN_ERR_UNSUPPORTED;
    *p = b;
    return MDCN_OK;
}

}  // namespace

extern "C" {

mdcn_status mdcn_create_tuned(const mdcn_attrs* attrs, const mdcn_tuning* tuning, mdcn_handle* out) {
    if (!attrs || !out) return MDCN_ERR_NULL;
    if (!attrs_valid(*attrs)) return MDCN_ERR_ATTR;
    mdcn_tuning tu{0, -1, 0, 0, 0, 0, 0};
    if (tuning) {
        tu = *tuning;
        if (tu.stages < 0 || tu.stages == 1 || tu.stages > 8 || tu.tile_mode < -1 || tu.tile_mode > 1 ||
            tu.max_ctas < 0 || !(tu.kgroups == 0 || tu.kgroups == 1 || tu.kgroups == 2 || tu.kgroups == 4) ||
            tu.a_operand < 0 || tu.a_operand > 2 || tu.ntile < 0 || tu.ntile > 512 || tu.ntile % 16 != 0 ||
            tu.path < 0 || tu.path > 2)
            return MDCN_ERR_ATTR;
    }
    mdcn_handle h = new (std::nothrow) mdcn_handle_;
    if (!h) return MDCN_ERR_UNSUPPORTED;
    h->attrs = *attrs;
    h->tuning = tu;
    *out = h;
    return MDCN_OK;
}

mdcn_status mdcn_create(const mdcn_attrs* attrs, mdcn_handle* out) { return mdcn_create_tuned(attrs, nullptr, out); }

mdcn_status mdcn_destroy(mdcn_handle handle) {
    delete handle;
    return MDCN_OK;
}

mdcn_status mdcn_output_dims(mdcn_handle handle, const mdcn_dims* dims, int64_t out_dims[4]) {
    if (!handle || !dims || !out_dims) return MDCN_ERR_NULL;
    int64_t od[4];
    mdcn_status s = check_dims(handle->attrs, *dims, od);
    if (s != MDCN_OK) return s;
    for (int i = 0; i < 4; ++i) out_dims[i] = od[i];
    return MDCN_OK;
}

mdcn_status mdcn_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes) {
    if (!handle || !dims || !bytes) return MDCN_ERR_NULL;
    Plan p;
    mdcn_status s = make_plan(handle->attrs, handle->tuning, dims, dtype, &p);
    if (s != MDCN_OK) return s;
    *bytes = forward_ws_bytes(handle->tuning, p);
    return MDCN_OK;
}

mdcn_status mdcn_query_plan(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, mdcn_plan_info* info) {
    if (!handle || !dims || !info) return MDCN_ERR_NULL;
    Plan p;
    mdcn_status s = make_plan(handle->attrs, handle->tuning, dims, dtype, &p);
    if (s != MDCN_OK) return s;
    s = plan_for_call(handle, dims, dtype, p.ws_bytes, &p);
    if (s != MDCN_OK) return s;
    info->tiles = p.tiles_total;
    info->ktiles_per_tile = p.KT;
    info->ktiles_per_cta = p.kt_per_cta;
    info->ctas = p.grid;
    info->split = mdcn::splitk_needed(p) ? 1 : 0;
    info->stages = p.stages;
    info->kgroups = p.kgroups;
    info->tile_mode = p.tile_mode;
    info->launches = p.direct ? (p.direct_cl ? 2 : 1) : (p.xt_block ? 2 : 3);
    info->a_operand = p.direct ? 0 : (p.a_tmem ? 2 : 1);
    info->path = p.direct ? 2 : 1;
    return MDCN_OK;
}

mdcn_status mdcn_forward(mdcn_handle handle, const void* x, const void* offset, const void* mask, const void* weight,
                         const void* bias_or_null, void* out, void* workspace, size_t workspace_bytes,
                         const mdcn_dims* dims, mdcn_dtype dtype, void* stream) {
    mdcn_status s = check_forward_args(handle, x, offset, mask, weight, bias_or_null, out, workspace, dims);
    if (s != MDCN_OK) return s;
    Plan p;
    s = plan_for_call(handle, dims, dtype, workspace_bytes, &p);
    if (s != MDCN_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p.direct) {
        const cudaError_t e = mdcn::launch_direct(p, x, offset, mask, weight, bias_or_null, out, workspace, st);
        return e == cudaSuccess ? MDCN_OK : cuda_fail(e);
    }
    const size_t elem = dtype == MDCN_F32 ? 4 : 2;
    const size_t plane = static_cast<size_t>(p.N) * static_cast<size_t>(p.P) * elem;
    cudaError_t e = mdcn::launch_prep_both(p, x, weight, offset, plane * 2 * p.dg * p.K, mask, plane * p.dg * p.K,
                                           workspace, st);
    if (e == cudaSuccess) e = mdcn::launch_fused(p, offset, mask, bias_or_null, out, workspace, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

// Device-buffer layout of mdcn_forward_host: the device copies of x, offset,
// mask, weight and bias, the output, and the workspace, each 256-byte
// aligned (so every part meets the 16-byte rule of the device entry points).
struct HostLayout {
    size_t off[7];
    size_t bytes[7];
    size_t total;
};

static mdcn_status host_layout(mdcn_handle h, const mdcn_dims* d, mdcn_dtype dt, HostLayout* L) {
    Plan p;
    const mdcn_status s = make_plan(h->attrs, h->tuning, d, dt, &p);
    if (s != MDCN_OK) return s;
    const int64_t elem = dt == MDCN_F32 ? 4 : 2;
    const int64_t* dims4[4] = {d->x, d->offset, d->mask, d->weight};
    for (int i = 0; i < 4; ++i) {
        int64_t n = elem;
        for (int k = 0; k < 4; ++k)
            if (!mul_ok(n, dims4[i][k])) return MDCN_ERR_UNSUPPORTED;
        L->bytes[i] = static_cast<size_t>(n);
    }
    L->bytes[4] = static_cast<size_t>(d->bias * elem);
    int64_t nout = elem;
    if (!mul_ok(nout, p.N) || !mul_ok(nout, p.Cout) || !mul_ok(nout, p.Ho) || !mul_ok(nout, p.Wo))
        return MDCN_ERR_UNSUPPORTED;
    L->bytes[5] = static_cast<size_t>(nout);
    L->bytes[6] = forward_ws_bytes(h->tuning, p);
    size_t at = 0;
    for (int i = 0; i < 7; ++i) {
        L->off[i] = at;
        at = align256(at + L->bytes[i]);
    }
    L->total = at;
    return MDCN_OK;
}

mdcn_status mdcn_host_buffer_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes) {
    if (!handle || !dims || !bytes) return MDCN_ERR_NULL;
    HostLayout L;
    const mdcn_status s = host_layout(handle, dims, dtype, &L);
    if (s != MDCN_OK) return s;
    *bytes = L.total;
    return MDCN_OK;
}

mdcn_status mdcn_forward_host(mdcn_handle handle, const void* x_host, const void* offset_host, const void* mask_host,
                              const void* weight_host, const void* bias_host_or_null, void* out_host,
                              void* device_buffer, size_t device_buffer_bytes, const mdcn_dims* dims,
                              mdcn_dtype dtype, void* stream) {
    if (!handle || !x_host || !offset_host || !mask_host || !weight_host || !out_host || !device_buffer || !dims)
        return MDCN_ERR_NULL;
    if ((bias_host_or_null == nullptr) != (dims->bias == 0)) return bias_host_or_null ? MDCN_ERR_SHAPE : MDCN_ERR_NULL;
    if (!aligned16(device_buffer)) return MDCN_ERR_ALIGN;
    HostLayout L;
    mdcn_status s = host_layout(handle, dims, dtype, &L);
    if (s != MDCN_OK) return s;
    if (device_buffer_bytes < L.total) return MDCN_ERR_WORKSPACE;
    Plan p;
    s = plan_for_call(handle, dims, dtype, L.bytes[6], &p);  // everything checked before the first copy
    if (s != MDCN_OK) return s;
    uint8_t* base = static_cast<uint8_t*>(device_buffer);
    void* dev[7];
    for (int i = 0; i < 7; ++i) dev[i] = base + L.off[i];
    const void* src[5] = {x_host, offset_host, mask_host, weight_host, bias_host_or_null};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < 5; ++i) {
        if (L.bytes[i] == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(dev[i], src[i], L.bytes[i], cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    s = mdcn_forward(handle, dev[0], dev[1], dev[2], dev[3], bias_host_or_null ? dev[4] : nullptr, dev[5], dev[6],
                     L.bytes[6], dims, dtype, stream);
    if (s != MDCN_OK) return s;
    const cudaError_t e = cudaMemcpyAsync(out_host, dev[5], L.bytes[5], cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

// The pack form's front end uses its own workspace and, after it, the buffer
// of its raw output om [N, 3*dg*K, Ho, Wo]; the deformable convolution then
// reuses the whole workspace.
static size_t pack_front_bytes(const Plan& pf, mdcn_dtype dtype) {
    const size_t elem = dtype == MDCN_F32 ? 4 : 2;
    return align256(pf.ws_bytes) +
           align256(static_cast<size_t>(pf.N) * static_cast<size_t>(pf.Cout) * static_cast<size_t>(pf.P) * elem);
}

mdcn_status mdcn_pack_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes) {
    if (!handle || !dims || !bytes) return MDCN_ERR_NULL;
    mdcn_attrs fa;
    mdcn_dims fd;
    mdcn_status s = front_end_problem(handle->attrs, dims, &fa, &fd);
    if (s != MDCN_OK) return s;
    Plan pf, pd;
    s = make_plan(fa, handle->tuning, &fd, dtype, &pf);
    if (s != MDCN_OK) return s;
    s = make_plan(handle->attrs, handle->tuning, dims, dtype, &pd);
    if (s != MDCN_OK) return s;
    pf.ws_bytes = forward_ws_bytes(handle->tuning, pf);
    pd.ws_bytes = forward_ws_bytes(handle->tuning, pd);
    const size_t front = pack_front_bytes(pf, dtype);
    *bytes = front > pd.ws_bytes ? front : pd.ws_bytes;
    return MDCN_OK;
}

mdcn_status mdcn_forward_pack(mdcn_handle handle, const void* x, const void* weight_om, const void* bias_om,
                              const void* weight, const void* bias_or_null, void* offset_out, void* mask_out,
                              void* out, void* workspace, size_t workspace_bytes, const mdcn_dims* dims,
                              mdcn_dtype dtype, void* stream) {
    if (!weight_om || !bias_om || !offset_out || !mask_out) return MDCN_ERR_NULL;
    mdcn_status s = check_forward_args(handle, x, offset_out, mask_out, weight, bias_or_null, out, workspace, dims);
    if (s != MDCN_OK) return s;
    if (!aligned16(weight_om) || !aligned16(bias_om)) return MDCN_ERR_ALIGN;
    mdcn_attrs fa;
    mdcn_dims fd;
    s = front_end_problem(handle->attrs, dims, &fa, &fd);
    if (s != MDCN_OK) return s;
    Plan pf, pd;
    s = plan_for(fa, handle->tuning, &fd, dtype, workspace_bytes, &pf);
    if (s != MDCN_OK) return s;
    s = plan_for_call(handle, dims, dtype, workspace_bytes, &pd);
    if (s != MDCN_OK) return s;
    if (workspace_bytes < pack_front_bytes(pf, dtype)) return MDCN_ERR_WORKSPACE;
    pf.plain = 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void* om = static_cast<uint8_t*>(workspace) + align256(pf.ws_bytes);
    // 1: the front end's raw output, then offset and sigmoid(mask) from it
    cudaError_t e;
    if (pf.direct) {
        e = mdcn::launch_direct(pf, x, nullptr, nullptr, weight_om, bias_om, om, workspace, st);
    } else {
        e = mdcn::launch_prep_both(pf, x, weight_om, nullptr, 0, nullptr, 0, workspace, st);
        if (e == cudaSuccess) e = mdcn::launch_fused(pf, nullptr, nullptr, bias_om, om, workspace, st);
    }
    if (e == cudaSuccess)
        e = mdcn::launch_split_offset_mask(pf, om, offset_out, mask_out, 2 * pd.dg * pd.K, pd.dg * pd.K, st);
    // 2: the deformable convolution; when its channels-last x has the front
    // end's layout, the copy already in the workspace is reused
    const bool same_xt = !pf.direct && !pd.direct && pf.Cp == pd.Cp && pf.U == pd.U && pf.UP == pd.UP &&
                         pf.off_xt == pd.off_xt && pf.off_wp == pd.off_wp && pf.a_tmem == pd.a_tmem;
    const size_t elem = dtype == MDCN_F32 ? 4 : 2;
    const size_t plane = static_cast<size_t>(pd.N) * static_cast<size_t>(pd.P) * elem;
    if (pd.direct) {
        if (e == cudaSuccess)
            e = mdcn::launch_direct(pd, x, offset_out, mask_out, weight, bias_or_null, out, workspace, st);
    } else {
        if (e == cudaSuccess)
            e = same_xt ? mdcn::launch_pack_weight(pd, weight, workspace, st)
                        : mdcn::launch_prep_both(pd, x, weight, offset_out, plane * 2 * pd.dg * pd.K, mask_out,
                                                 plane * pd.dg * pd.K, workspace, st);
        if (e == cudaSuccess) e = mdcn::launch_fused(pd, offset_out, mask_out, bias_or_null, out, workspace, st);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

mdcn_status mdcn_prepare_input(mdcn_handle handle, const void* x, void* workspace, size_t workspace_bytes,
                               const mdcn_dims* dims, mdcn_dtype dtype, void* stream) {
    if (!handle || !x || !workspace || !dims) return MDCN_ERR_NULL;
    if (!aligned16(x) || !aligned16(workspace)) return MDCN_ERR_ALIGN;
    Plan p;
    mdcn_status s = plan_for_call(handle, dims, dtype, workspace_bytes, &p);
    if (s != MDCN_OK) return s;
    if (p.direct) return MDCN_ERR_UNSUPPORTED;  // a direct plan runs whole, in mdcn_forward
    cudaError_t e = mdcn::launch_prep_input(p, x, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

mdcn_status mdcn_pack_weight(mdcn_handle handle, const void* weight, void* workspace, size_t workspace_bytes,
                             const mdcn_dims* dims, mdcn_dtype dtype, void* stream) {
    if (!handle || !weight || !workspace || !dims) return MDCN_ERR_NULL;
    if (!aligned16(weight) || !aligned16(workspace)) return MDCN_ERR_ALIGN;
    Plan p;
    mdcn_status s = plan_for_call(handle, dims, dtype, workspace_bytes, &p);
    if (s != MDCN_OK) return s;
    if (p.direct) return MDCN_ERR_UNSUPPORTED;  // a direct plan runs whole, in mdcn_forward
    cudaError_t e = mdcn::launch_pack_weight(p, weight, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

mdcn_status mdcn_forward_prepared(mdcn_handle handle, const void* offset, const void* mask, const void* bias_or_null,
                                  void* out, void* workspace, size_t workspace_bytes, const mdcn_dims* dims,
                                  mdcn_dtype dtype, void* stream) {
    if (!handle || !offset || !mask || !out || !workspace || !dims) return MDCN_ERR_NULL;
    if ((bias_or_null == nullptr) != (dims->bias == 0)) return bias_or_null ? MDCN_ERR_SHAPE : MDCN_ERR_NULL;
    if (!aligned16(offset) || !aligned16(mask) || !aligned16(out) || !aligned16(workspace) ||
        (bias_or_null && !aligned16(bias_or_null)))
        return MDCN_ERR_ALIGN;
    Plan p;
    mdcn_status s = plan_for_call(handle, dims, dtype, workspace_bytes, &p);
    if (s != MDCN_OK) return s;
    if (p.direct) return MDCN_ERR_UNSUPPORTED;  // a direct plan runs whole, in mdcn_forward
    cudaError_t e = mdcn::launch_fused(p, offset, mask, bias_or_null, out, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

mdcn_status mdcn_im2col_gemm_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype,
                                            size_t* bytes) {
    if (!handle || !dims || !bytes) return MDCN_ERR_NULL;
    Plan p;
    mdcn_status s = make_plan(handle->attrs, handle->tuning, dims, dtype, &p);
    if (s != MDCN_OK) return s;
    if (p.P > kI31 || static_cast<int64_t>(p.Cg) * p.K > kI31 || p.N > kI31) return MDCN_ERR_UNSUPPORTED;
    *bytes = mdcn::im2col_workspace_bytes(p);
    return MDCN_OK;
}

mdcn_status mdcn_forward_im2col_gemm(mdcn_handle handle, const void* x, const void* offset, const void* mask,
                                     const void* weight, const void* bias_or_null, void* out, void* workspace,
                                     size_t workspace_bytes, const mdcn_dims* dims, mdcn_dtype dtype, void* stream) {
    mdcn_status s = check_forward_args(handle, x, offset, mask, weight, bias_or_null, out, workspace, dims);
    if (s != MDCN_OK) return s;
    size_t need = 0;
    s = mdcn_im2col_gemm_workspace_size(handle, dims, dtype, &need);
    if (s != MDCN_OK) return s;
    if (workspace_bytes < need) return MDCN_ERR_WORKSPACE;
    Plan p;
    s = make_plan(handle->attrs, handle->tuning, dims, dtype, &p);
    if (s != MDCN_OK) return s;
    s = check_device();
    if (s != MDCN_OK) return s;
    cudaError_t e = mdcn::launch_im2col_gemm(p, x, offset, mask, weight, bias_or_null, out, workspace,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

mdcn_status mdcn_backward_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes) {
    if (!handle || !dims || !bytes) return MDCN_ERR_NULL;
    mdcn::BwdPlan b;
    mdcn_status s = make_bwd_plan(handle->attrs, dims, dtype, &b);
    if (s != MDCN_OK) return s;
    *bytes = b.ws_bytes;
    return MDCN_OK;
}

mdcn_status mdcn_backward_launches(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, int32_t* launches) {
    if (!handle || !dims || !launches) return MDCN_ERR_NULL;
    mdcn::BwdPlan b;
    mdcn_status s = make_bwd_plan(handle->attrs, dims, dtype, &b);
    if (s != MDCN_OK) return s;
    *launches = mdcn::backward_launch_count(b);
    return MDCN_OK;
}

mdcn_status mdcn_backward(mdcn_handle handle, const void* x, const void* offset, const void* mask, const void* weight,
                          const void* grad_out, void* grad_x, void* grad_offset, void* grad_mask, void* grad_weight,
                          void* grad_bias_or_null, void* workspace, size_t workspace_bytes, const mdcn_dims* dims,
                          mdcn_dtype dtype, void* stream) {
    if (!handle || !x || !offset || !mask || !weight || !grad_out || !grad_x || !grad_offset || !grad_mask ||
        !grad_weight || !workspace || !dims)
        return MDCN_ERR_NULL;
    if ((grad_bias_or_null == nullptr) != (dims->bias == 0)) return grad_bias_or_null ? MDCN_ERR_SHAPE : MDCN_ERR_NULL;
    const void* ptrs[] = {x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask, grad_weight, workspace};
    for (const void* q : ptrs)
        if (!aligned16(q)) return MDCN_ERR_ALIGN;
    if (grad_bias_or_null && !aligned16(grad_bias_or_null)) return MDCN_ERR_ALIGN;
    mdcn::BwdPlan b;
    mdcn_status s = make_bwd_plan(handle->attrs, dims, dtype, &b);
    if (s != MDCN_OK) return s;
    if (workspace_bytes < b.ws_bytes) return MDCN_ERR_WORKSPACE;
    s = check_device();
    if (s != MDCN_OK) return s;
    cudaError_t e = mdcn::launch_backward(b, x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask,
                                          grad_weight, grad_bias_or_null, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return MDCN_OK;
}

mdcn_status mdcn_query_status(const void* workspace, void* stream, uint32_t* device_bits) {
    if (!workspace) return MDCN_ERR_NULL;
    if (!aligned16(workspace)) return MDCN_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    cudaError_t e = cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(bits), st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (device_bits) *device_bits = bits;
    return (bits & 1u) ? MDCN_ERR_TIMEOUT : MDCN_OK;
}

mdcn_status mdcn_selftest_wait_timeout(void* status_word, uint32_t limit_us, void* stream) {
    if (!status_word) return MDCN_ERR_NULL;
    if (!aligned16(status_word)) return MDCN_ERR_ALIGN;
    if (limit_us < 1 || limit_us > 10000000u) return MDCN_ERR_ATTR;
    mdcn_status s = check_device();
    if (s != MDCN_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // limit in SM cycles at the 2.07 GHz maximum clock (longer in time at lower clocks)
    cudaError_t e = mdcn::launch_wait_selftest(static_cast<uint32_t*>(status_word), uint64_t(limit_us) * 2070u, st);
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t bits = 0;
    e = cudaMemcpyAsync(&bits, status_word, sizeof(bits), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (bits & (1u << 31)) return MDCN_OK;  // the wait completed: the bound is broken
    return (bits & 1u) ? MDCN_ERR_TIMEOUT : MDCN_OK;
}

int mdcn_last_cuda_error(void) { return g_last_cuda_error; }

const char* mdcn_status_string(mdcn_status status) {
    switch (status) {
        case MDCN_OK: return "ok";
        case MDCN_ERR_NULL: return "a required pointer is NULL";
        case MDCN_ERR_ATTR: return "attribute out of range (stride, dilation >= 1; padding >= 0; group, deformable_group >= 1)";
        case MDCN_ERR_SHAPE: return "tensor dims are inconsistent";
        case MDCN_ERR_DTYPE: return "unknown dtype";
        case MDCN_ERR_ALIGN: return "device pointer not 16-byte aligned";
        case MDCN_ERR_WORKSPACE: return "workspace too small";
        case MDCN_ERR_ARCH: return "current device is not compute capability 10.3";
        case MDCN_ERR_CUDA: return "CUDA runtime error";
        case MDCN_ERR_TIMEOUT: return "device pipeline wait timed out";
        case MDCN_ERR_UNSUPPORTED: return "size beyond the library's limits";
    }
    return "unknown status";
}

}  // extern "C"
