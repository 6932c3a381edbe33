// Host side of the C ABI declared in tfq.h: argument validation, the launch
// planner and the entry points. Nothing here allocates, synchronises or prints
// (except the two documented diagnostics that read device memory back).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>

#include "tfq_internal.h"

namespace tfq {

namespace {
thread_local char g_last_error[512] = "";
// planner overrides of tf_tune_set: per host thread, so that one caller's tuning
// never changes another caller's schedule or workspace needs
thread_local int g_tune[7] = {-1, -1, -1, -1, -1, -1, -1};
int g_sms_cache[64] = {0};

constexpr size_t kStatusBytes = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The kernels' BITS argument for a descriptor's weight code.
int kernel_bits(const tf_qweight* w) { return w->code == TF_CODE_NVFP4 ? kNvfp4 : w->bits; }

int fail(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(TF_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Validate a descriptor filled by tf_qlinear_pack or tf_qlinear_pack_nvfp4.
int check_desc(const tf_qweight* w, const char* name)
{
    if (w == nullptr)
        return fail(TF_E_INVALID_ARG, "%s: descriptor is NULL", name);
    if (w->magic != TF_QWEIGHT_MAGIC || w->version != TF_PACK_VERSION)
        return fail(TF_E_BAD_PACK, "%s: descriptor magic/version mismatch (not filled by tf_qlinear_pack?)", name);
    const bool nvfp4 = w->code == TF_CODE_NVFP4;
    if (w->code != TF_CODE_AFFINE && !nvfp4)
        return fail(TF_E_BAD_PACK, "%s: unknown weight code %d", name, w->code);
    if (nvfp4 ? (w->bits != 4 || w->group != 16 || !std::isfinite(w->global_scale))
              : ((w->bits != 4 && w->bits != 8) || w->group != kGroup))
        return fail(TF_E_BAD_PACK, "%s: bits=%d group=%d do not match the weight code", name, w->bits, w->group);
    if (w->K <= 0 || w->K % kGroup != 0 || w->N <= 0 || w->batch <= 0)
        return fail(TF_E_BAD_PACK, "%s: bad shape", name);
    if (w->n_pad != (w->N + 15) / 16 * 16 || w->tile_bytes != tile_bytes_for(kernel_bits(w)) ||
        w->matrix_bytes != w->n_pad / 16 * (w->K / kGroup) * w->tile_bytes)
        return fail(TF_E_BAD_PACK, "%s: inconsistent sizes", name);
    if (w->data == nullptr || !aligned(w->data, 16))
        return fail(TF_E_INVALID_ARG, "%s: data pointer NULL or not 16-byte aligned", name);
    if (w->N > INT32_MAX / 2 || w->K > INT32_MAX / 2 ||
        (w->n_pad / 16) * (w->K / kGroup) * (w->batch > 64 ? 64 : w->batch) >= (int64_t)1 << 30)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: dimension too large", name);
    return TF_OK;
}

int check_act(const void* x, int64_t ldx, int64_t K, const char* name)
{
    if (x == nullptr)
        return fail(TF_E_INVALID_ARG, "%s is NULL", name);
    if (!aligned(x, 16) || ldx < K || ldx % 8 != 0)
        return fail(TF_E_INVALID_ARG, "%s must be 16-byte aligned with a leading dimension >= K and a multiple of 8",
                    name);
    return TF_OK;
}

const uint8_t* tiles_of(const tf_qweight* w)
{
    return static_cast<const uint8_t*>(w->data) + TF_PACK_HEADER_BYTES;
}

// The per-matrix fp32 scale table of an NVFP4 pack (after its matrices); null for affine codes.
const float* nvfp4_scales_of(const tf_qweight* w)
{
    if (w->code != TF_CODE_NVFP4)
        return nullptr;
    return reinterpret_cast<const float*>(tiles_of(w) + w->batch * w->matrix_bytes);
}

size_t plan_scratch(const Plan& p) { return p.ws_counters + p.ws_partials; }

// For the calls whose kernels read MLX affine codes only (the MoE layer).

void fill_common(QProjParams& p, const Plan& pl, void* ws, uint8_t* scratch)
{
    p.S = pl.S;
    p.Gs = pl.Gs;
    p.P = 1;
    p.C = pl.C;
    p.aligned = pl.aligned;
    p.kmax = pl.kmax;
    p.cg = pl.cg;
    p.nst = pl.nst;
    p.segmax = pl.segmax;
    p.red_off = pl.red_off;
    p.seg_off = pl.seg_off;
    p.round_off = pl.round_off;
    p.last_off = pl.last_off;
    p.nw = pl.nw;
    p.pw = pl.pw;
    p.xsum1_off = pl.xsum1_off;
    p.xraw1_off = pl.xraw1_off;
    p.gamma_off = pl.gamma_off;
    p.x_direct = pl.x_direct;
    p.xraw_off = pl.xraw_off;
    p.x_rs = pl.x_rs;
    p.stage_off = pl.stage_off;
    p.status = static_cast<int*>(ws);
    p.counters = reinterpret_cast<int*>(scratch);
    p.partials = reinterpret_cast<float*>(scratch + pl.ws_counters);
    p.limit_ns = kDefaultWaitLimitNs;
}

}  // namespace

void set_error(const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
}

// A fingerprint of the calling thread's tuning overrides (they change launch plans).
uint64_t tune_fingerprint()
{
    uint64_t h = 1469598103934665603ull;
    for (int v : g_tune) {
        h ^= (uint64_t)(uint32_t)v;
        h *= 1099511628211ull;
    }
    return h;
}

int device_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    if (g_sms_cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
            cudaGetLastError();
            sms = 152;
        }
        g_sms_cache[dev] = sms;
    }
    return g_sms_cache[dev];
}

// Streaming plan (tfq_stream.cuh) for one matrix of one problem: false when the call
// does not suit it (an RMSNorm over K > 1024, or more K splits than SMs).
bool plan_stream(int n_rb, int groups, int bits, int k_full, int sms, Plan& pl)
{
    const int tile = tile_bytes_for(bits);
    if (k_full > 1024)  // the normalised rows are staged by warps holding at most 4 chunks a lane
        return false;
    // 8 compute warps and at most 110 KB: the next kernel's CTA fits beside this one's,
    // so its weight copies start while this kernel finishes; 16 warps take a whole SM
    const int W = g_tune[TF_TUNE_WARPS] == 16 ? 16 : 8;
    const size_t budget = W == 8 ? 110 * 1024 : 227 * 1024;
    // K splits: 8 rows of a split's slice within 28 KB (the same split for every M)
    int S = 1;
    if (k_full == 0) {
        while (S < groups && (groups % S != 0 || (int64_t)kMaxM * ((groups / S) * kGroup * 2 + 16) > 28 * 1024))
            ++S;
        if (g_tune[TF_TUNE_SPLITK] > 0 && groups % g_tune[TF_TUNE_SPLITK] == 0)
            S = g_tune[TF_TUNE_SPLITK];
    }
    if (S > sms)
        return false;
    const int Gs = groups / S;
    pl = Plan{};
    pl.mode = 2;
    pl.slots = 1;
    pl.S = S;
    pl.Gs = Gs;
    pl.nw = W;
    pl.KW = 1;
    pl.R = 1;
    const int64_t Us = (int64_t)n_rb * Gs;
    // S groups of C / S CTAs, one split each, every CTA with at least one unit
    pl.C = S * (int)std::min<int64_t>(sms / S, Us);
    const int64_t upc_min = Us / (pl.C / S);
    pl.kmax = upc_min >= 1 ? (int)std::min<int64_t>(Gs, (Gs - 1) / upc_min + 2) : Gs;
    pl.aligned = 0;
    // chunks of 32 tiles (a multiple of 2 W: a warp's two tiles share a chunk)
    int CH = g_tune[TF_TUNE_STAGE_GROUPS] > 0 ? g_tune[TF_TUNE_STAGE_GROUPS] : 32;
    CH = std::max(2 * W, (CH + 2 * W - 1) / (2 * W) * (2 * W));
    pl.cg = CH;
    pl.pw = 4;  // hand-off slots of the reducer
    const int xg = k_full > 0 ? groups : Gs;  // groups staged
    pl.xraw_off = (int)align_up(384 + (size_t)xg * kMaxM * 4, 128);
    pl.x_rs = xg * kGroup * 2 + 16;
    pl.red_off = (int)align_up(pl.xraw_off + (size_t)kMaxM * pl.x_rs, 128);  // all 8 rows (zero past M)
    const int64_t upc_max = (Us + pl.C / S - 1) / (pl.C / S);
    pl.segmax = (int)(upc_max / Gs + 2);  // row blocks a CTA touches
    pl.last_off = (int)align_up(pl.red_off + (size_t)pl.pw * W * 32 * 16, 128);
    pl.stage_off = (int)align_up(pl.last_off + (size_t)pl.segmax * 4, 128);
    const size_t slot = (size_t)CH * tile;
    int NS = pl.stage_off + 2 * slot <= budget ? (int)((budget - pl.stage_off) / slot) : 0;
    NS = std::min(NS, 8);
    if (g_tune[TF_TUNE_STAGES] > 0)
        NS = std::min(NS, g_tune[TF_TUNE_STAGES]);
    if (NS < 2)
        return false;
    pl.nst = NS;
    pl.smem = pl.stage_off + (size_t)NS * slot;
    pl.ws_counters = align_up((size_t)n_rb * sizeof(int), 256);
    pl.ws_partials = align_up((size_t)S * n_rb * pl.kmax * 32 * 4 * sizeof(float), 256);
    return true;
}

// Plan of one projection launch (persistent grid, at most one CTA per SM).
//   n_rb, groups  16-row blocks and 64-column groups of one matrix
//   mats          2 for gate + up, else 1
//   slots         independent problems (MoE expert slots, an upper bound); 1 otherwise
//   k_full        K when whole activation rows are staged (RMSNorm prologue), else 0
//   rows          activation rows to reserve shared memory for
// The workspace size depends only on (n_rb, groups, mats, bits, slots).
Plan plan_qproj(int n_rb, int groups, int mats, int bits, int slots, int k_full, int rows)
{
    const int sms = device_sms();
    const int tile = tile_bytes_for(bits);
    const int vals = mats == 2 ? 8 : 4;
    Plan pl{};
    pl.slots = slots;

    // K splits: the split's activation slice for 8 rows must stay within 112 KB (the same
    // split for every M, so a row gives the same bits alone or in a block of 8)
    // long rows of one plain matrix (few row blocks, many groups, bandwidth-bound):
    // warp workers over K splits of at most 40 groups, 8 workers a CTA (on GB300 this
    // measured 12.8 / 14.8 us at M = 1 / 8 for K = 12800, N = 2560, against 14.6 / 17.0
    // for lock-step teams over two splits)
    const bool nvfp4 = bits == kNvfp4;  // no streaming schedule
    const bool long_plain = slots == 1 && mats == 1 && k_full == 0 && groups >= 64 && n_rb <= 2 * sms &&
                            (double)n_rb * groups * tile > 8.0 * 1024 * 1024 && g_tune[TF_TUNE_MODE] <= 0;
    int S = 1;
    while ((int64_t)kMaxM * (groups / S) * kGroup * 2 > 112 * 1024 || groups % S != 0)
        ++S;
    while (long_plain && (groups / S > 40 || groups % S != 0))
        ++S;
    if (g_tune[TF_TUNE_SPLITK] > 0 && groups % g_tune[TF_TUNE_SPLITK] == 0)
        S = g_tune[TF_TUNE_SPLITK];
    pl.S = S;
    pl.Gs = groups / S;

    // partition: whole row blocks when that balances within ~10 % (or the call is
    // small enough to be latency-bound), else exact stream-K shares
    const int64_t items = (int64_t)slots * S * n_rb;
    const int64_t U = items * pl.Gs;
    pl.C = sms;
    const double per_cta = (double)items / pl.C;
    const double imbalance = items >= pl.C ? (double)((items + pl.C - 1) / pl.C) / per_cta : 1.0;
    const bool small = (double)U * tile * mats <= 6.0 * 1024 * 1024;
    pl.aligned = (small || imbalance <= 1.10) ? 1 : 0;

    // segments per CTA (capacity of its list) and partial slots per row block
    const int64_t C_items = std::min<int64_t>(pl.C, std::max<int64_t>(items, 1));
    const int64_t C_units = std::min<int64_t>(pl.C, std::max<int64_t>(U, 1));
    const int64_t per_ps = (int64_t)n_rb * pl.Gs;
    double segs_per_cta;
    if (pl.aligned) {
        pl.segmax = (int)((items + C_items - 1) / C_items);
        pl.kmax = 1;
        segs_per_cta = (double)items / C_items;
    } else {
        const int64_t upc_max = (U + C_units - 1) / C_units;
        const int64_t U_min = (int64_t)S * n_rb * pl.Gs;  // one problem
        const int64_t upc_min = U_min / std::min<int64_t>(pl.C, U_min);
        pl.segmax = (int)(upc_max / pl.Gs + 4 + 2 * (upc_max / per_ps));
        pl.kmax = upc_min >= 1 ? (int)std::min<int64_t>(pl.Gs, (pl.Gs - 1) / upc_min + 2) : pl.Gs;
        segs_per_cta = (double)U / C_units / pl.Gs + 1.0;
    }

    // long rows (a plain problem with few, long segments per CTA and enough bytes to be
    // bandwidth-bound): one segment at a time, all warps on it, stages of about 27 KB
    const bool long_rows = !long_plain && slots == 1 && items <= 8LL * sms &&
                           (double)U * tile * mats > 8.0 * 1024 * 1024 && pl.Gs >= 2 * kConsumerWarps;

    // teams: R segments side by side, KW warps per segment, at least two tiles a warp
    int R = 1;
    while (!long_rows && R < kConsumerWarps && 2 * R <= segs_per_cta)
        R *= 2;
    while (kConsumerWarps / R > std::max(1, pl.Gs / 2))
        R *= 2;
    if (g_tune[TF_TUNE_ROWBLOCKS] > 0)
        R = g_tune[TF_TUNE_ROWBLOCKS];
    pl.R = R;
    pl.KW = kConsumerWarps / R;

    // stages of about 16 KB (27 KB for long rows), a multiple of KW groups per segment
    int cg = std::max(1, (long_rows ? 27648 : 16384) / (mats * pl.R * tile));
    cg = (cg + pl.KW - 1) / pl.KW * pl.KW;
    if (g_tune[TF_TUNE_STAGE_GROUPS] > 0)
        cg = g_tune[TF_TUNE_STAGE_GROUPS];
    pl.cg = std::min(cg, std::max(1, pl.Gs));
    const size_t stage = (size_t)mats * pl.R * pl.cg * tile;

    // shared memory: fixed part, xsum, reduction buffer, segment lists, activations, ring
    const size_t fixed = 256 + kMaxSlots * 8 + kMaxSlots * kMaxM * 4;
    pl.red_off = (int)align_up(fixed + (size_t)pl.Gs * kMaxM * 4, 128);
    pl.seg_off = (int)align_up(pl.red_off + (size_t)kConsumerWarps * 32 * vals * 4, 128);
    pl.round_off = (int)align_up(pl.seg_off + (size_t)pl.segmax * 16, 128);
    pl.last_off = (int)align_up(pl.round_off + (size_t)(pl.segmax + 1) * 8, 128);
    pl.gamma_off = (int)align_up(pl.last_off + (size_t)pl.segmax * 4, 128);
    pl.xraw_off = (int)align_up(pl.gamma_off + (size_t)std::max(k_full, 0) * 2, 128);
    const int xcols = k_full > 0 ? k_full : pl.Gs * kGroup;
    pl.x_rs = xcols * 2 + 16;
    pl.stage_off = (int)align_up(pl.xraw_off + (size_t)rows * pl.x_rs, 128);
    const size_t budget = 227 * 1024;
    int nst = budget > pl.stage_off + stage ? (int)((budget - pl.stage_off) / stage) : 1;
    nst = std::min(nst, kMaxStages);
    if (g_tune[TF_TUNE_STAGES] > 0)
        nst = std::min(g_tune[TF_TUNE_STAGES], nst);
    pl.nst = std::max(nst, 1);
    pl.smem = pl.stage_off + (size_t)pl.nst * stage;

    // ---- small calls (latency-bound): light teams, one whole item per CTA, the item
    // fetched in one stage, small enough for several CTAs (and the next kernel's) per SM
    const bool light_ok = S == 1 && items <= 4LL * sms && (double)U * tile * mats <= 8.0 * 1024 * 1024;
    bool light = light_ok && g_tune[TF_TUNE_MODE] <= 0;
    if (g_tune[TF_TUNE_MODE] == 3 || g_tune[TF_TUNE_MODE] == 4)
        light = light_ok;
    // ---- the stage kernel: one CTA per whole row block (all of K), the activations loaded
    // straight into registers (with an RMSNorm: K <= 1024), no weight ring, no partial sums;
    // small enough for two CTAs an SM (the next kernel's CTAs start beside the running ones)
    if (light && slots == 1 && k_full <= 1024 && g_tune[TF_TUNE_MODE] <= 0) {
        const size_t fixed = 256 + kMaxSlots * 8 + kMaxSlots * kMaxM * 4;  // barrier, flags, slots
        Plan sp = pl;
        sp.mode = 3;
        sp.C = n_rb;
        sp.aligned = 1;
        sp.kmax = 1;
        sp.nst = 1;
        sp.cg = groups;
        sp.nw = n_rb <= sms ? 16 : 8;  // 16 warps when one CTA an SM holds every row block
        sp.KW = sp.nw;
        sp.R = 1;
        sp.red_off = (int)align_up(fixed + (size_t)groups * kMaxM * 4, 128);
        sp.xraw_off = (int)align_up(sp.red_off + (size_t)2 * sp.nw * 32 * 16, 128);
        sp.x_rs = groups * kGroup * 2 + 16;
        sp.stage_off = (int)align_up(sp.xraw_off + (size_t)rows * sp.x_rs, 128);
        sp.smem = sp.stage_off + (size_t)mats * groups * tile;
        sp.ws_counters = 0;
        sp.ws_partials = 0;
        sp.x_direct = 1;
        if (sp.smem <= 110 * 1024)
            return sp;
    }
    if (light) {
        pl.nw = 8;
        pl.C = (int)std::max<int64_t>(items, 1);
        pl.aligned = 1;
        pl.kmax = 1;
        pl.segmax = 1;
        int KW = 8;
        while (KW > 1 && pl.Gs < 2 * KW)
            KW /= 2;
        pl.KW = KW;
        pl.R = 8 / KW;
        pl.cg = pl.Gs;
        pl.nst = 1;
        const size_t stage = (size_t)mats * pl.R * pl.cg * tile;
        const size_t fixed = 256 + kMaxSlots * 8 + kMaxSlots * kMaxM * 4;
        pl.red_off = (int)align_up(fixed + (size_t)pl.Gs * kMaxM * 4, 128);
        pl.seg_off = (int)align_up(pl.red_off + (size_t)8 * 32 * vals * 4, 128);
        pl.round_off = (int)align_up(pl.seg_off + 16, 128);
        pl.last_off = (int)align_up(pl.round_off + 16, 128);
        pl.gamma_off = (int)align_up(pl.last_off + 4, 128);
        pl.xraw_off = (int)align_up(pl.gamma_off + (size_t)std::max(k_full, 0) * 2, 128);
        const int xcols = k_full > 0 ? k_full : pl.Gs * kGroup;
        pl.x_rs = xcols * 2 + 16;
        pl.stage_off = (int)align_up(pl.xraw_off + (size_t)rows * pl.x_rs, 128);
        pl.smem = pl.stage_off + stage;
        pl.ws_counters = 0;
        pl.ws_partials = 0;
        // plain rows (one problem) come straight from global memory: with an RMSNorm the
        // row must fit four 8-column chunks per lane (K <= 1024)
        pl.x_direct = slots == 1 && (k_full == 0 || k_full <= 1024) && g_tune[TF_TUNE_MODE] != 4 ? 1 : 0;
        return pl;
    }
    // ---- one large matrix: streaming CTAs (selected with TF_TUNE_MODE 5; on GB300 it
    // measured no faster than the long-row teams and warp workers below: every schedule
    // is bound by the instructions per tile, ~90-110, not by the memory system)
    if (slots == 1 && mats == 1 && g_tune[TF_TUNE_MODE] == 5 && !nvfp4) {
        Plan sp;
        if (plan_stream(n_rb, groups, bits, k_full, sms, sp))
            return sp;
    }
    pl.nw = kConsumerWarps;

    // ---- bandwidth-bound calls: warp workers with private ring slots
    // MoE layers (many problems, each with its own activation rows): 8 workers a CTA
    // measured fastest; otherwise all 16
    const int nw_default = slots > 1 || long_plain ? 8 : kConsumerWarps;
    int nw = g_tune[TF_TUNE_WARPS] > 0 ? std::min(g_tune[TF_TUNE_WARPS], kConsumerWarps) : nw_default;
    int64_t W = (int64_t)sms * nw;
    const int64_t upc_max_all = (U + pl.C - 1) / pl.C;  // units per CTA with every slot active
    bool warp_mode = (long_plain || (!long_rows && U >= 4 * W)) && upc_max_all <= per_ps;
    if (g_tune[TF_TUNE_MODE] > 0)
        warp_mode = g_tune[TF_TUNE_MODE] == 2 && upc_max_all <= per_ps;
    // the activation buffers (two unless a single problem and split, or an RMSNorm)
    // and two ring slots per worker must fit, else lock-step teams
    auto warp_fits = [&](int nw_) {
        const bool norm_rows = k_full > 0;
        const int bufs = (!norm_rows && (int64_t)slots * S > 1) ? 2 : 1;
        const int xcols = norm_rows ? k_full : pl.Gs * kGroup;
        const int Tw = std::max(1, (mats == 2 && slots == 1 ? 2304 : 4608) / tile);
        const size_t need = 16384 + (size_t)bufs * kMaxM * (xcols * 2 + 16) +
                            (size_t)2 * nw_ * mats * std::min(Tw, pl.Gs) * tile;
        return need <= 227 * 1024;
    };
    if (warp_mode) {
        warp_mode = warp_fits(nw);
        W = (int64_t)sms * nw;
    }
    if (warp_mode) {
        pl.mode = 1;
        pl.nw = nw;
        const int64_t W_items = std::min<int64_t>(W, std::max<int64_t>(items, 1));
        // stream-K workers (as the kernel counts them): at least Gs / 2 units each
        auto workers_for = [&](int64_t units) {
            return std::min<int64_t>(W, std::max<int64_t>(units / std::max(1, pl.Gs / 2), 1));
        };
        const int64_t W_units = workers_for(U);
        const double per_w = (double)items / W_items;
        const double imb = (double)((items + W_items - 1) / W_items) / per_w;
        pl.aligned = imb <= 1.10 ? 1 : 0;
        const int64_t U_min = (int64_t)S * n_rb * pl.Gs;
        if (pl.aligned) {
            pl.kmax = 1;
            pl.pw = S > 1 ? (int)((items + W_items - 1) / W_items) + 1 : 1;
        } else {
            const int64_t upw_min = U_min / workers_for(U_min);
            const int64_t upw_max = std::max<int64_t>((U + W_units - 1) / W_units, pl.Gs);
            pl.kmax = upw_min >= 1 ? (int)std::min<int64_t>(pl.Gs, (pl.Gs - 1) / upw_min + 2) : pl.Gs;
            pl.pw = (int)(upw_max / pl.Gs + 4);
        }
        // chunks of ~4.5 KB per matrix (~2.3 KB for gate + up of one problem; one bulk copy
        // each), two or more slots per worker
        int T = std::max(1, 4608 / tile);
        if (mats == 2 && slots == 1)
            T = std::max(1, T / 2);
        if (g_tune[TF_TUNE_STAGE_GROUPS] > 0)
            T = g_tune[TF_TUNE_STAGE_GROUPS];
        pl.cg = std::min(T, pl.Gs);
        const size_t slot = (size_t)mats * pl.cg * tile;
        const bool norm = k_full > 0;
        const bool two_bufs = !norm && (int64_t)slots * S > 1;
        const int xs_groups = norm ? groups : pl.Gs;
        const size_t fixed = 256 + kMaxSlots * 8 + kMaxSlots * kMaxM * 4;
        pl.xsum1_off = (int)align_up(fixed + (size_t)xs_groups * kMaxM * 4, 128);
        pl.red_off = (int)align_up(pl.xsum1_off + (size_t)pl.Gs * kMaxM * 4, 128);  // ring barriers
        pl.round_off = (int)align_up(pl.red_off + (size_t)2 * nw * kMaxStages * 8, 128);  // inv1, rows1, npend
        pl.seg_off = (int)align_up(pl.round_off + 128, 128);                              // pending
        pl.last_off = (int)align_up(pl.seg_off + (size_t)nw * pl.pw * 16, 128);
        pl.gamma_off = (int)align_up(pl.last_off + (size_t)nw * pl.pw * 4, 128);
        pl.xraw_off = (int)align_up(pl.gamma_off + (size_t)std::max(k_full, 0) * 2, 128);
        const int xcols = norm ? k_full : pl.Gs * kGroup;
        pl.x_rs = xcols * 2 + 16;
        // M rows of each buffer and a zero row that the fragment loads of rows M..7 read
        // (8 rows for MoE, whose problems stage up to 8); only the ring depth below
        // depends on M, never the partition, so a row's result does not
        const int xrows = std::min(rows + 1, kMaxM);
        pl.xraw1_off = (int)align_up(pl.xraw_off + (size_t)xrows * pl.x_rs, 128);
        pl.stage_off = (int)align_up(pl.xraw1_off + (two_bufs ? (size_t)xrows * pl.x_rs : 0), 128);
        const size_t budget = 227 * 1024;
        int SW = budget > pl.stage_off + 2 * nw * slot ? (int)((budget - pl.stage_off) / (nw * slot)) : 1;
        SW = std::min(SW, kMaxStages);
        if (g_tune[TF_TUNE_STAGES] > 0)
            SW = std::min(g_tune[TF_TUNE_STAGES], SW);
        pl.nst = std::max(SW, 1);
        pl.smem = pl.stage_off + (size_t)nw * pl.nst * slot;
        pl.KW = 1;
        pl.R = nw;
    }

    const bool partials = S > 1 || !pl.aligned;
    pl.ws_counters = partials ? align_up((size_t)slots * n_rb * sizeof(int), 256) : 0;
    pl.ws_partials =
        partials ? align_up((size_t)slots * S * n_rb * pl.kmax * 32 * vals * sizeof(float), 256) : 0;
    return pl;
}

// For the other translation units of the library: set the calling thread's error
// message and return the status; validate a descriptor as every entry point does.
int report_error(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int validate_desc(const tf_qweight* w, const char* name) { return check_desc(w, name); }

}  // namespace tfq

using namespace tfq;

extern "C" {

const char* tf_status_str(int status)
{
    switch (status) {
    case TF_OK: return "TF_OK";
    case TF_E_INVALID_ARG: return "TF_E_INVALID_ARG";
    case TF_E_UNSUPPORTED_SHAPE: return "TF_E_UNSUPPORTED_SHAPE";
    case TF_E_WORKSPACE_TOO_SMALL: return "TF_E_WORKSPACE_TOO_SMALL";
    case TF_E_BAD_PACK: return "TF_E_BAD_PACK";
    case TF_E_CUDA: return "TF_E_CUDA";
    case TF_E_TIMEOUT: return "TF_E_TIMEOUT";
    case TF_E_INTERNAL: return "TF_E_INTERNAL";
    default: return "TF_E_UNKNOWN";
    }
}

const char* tf_last_error(void) { return g_last_error; }

int tf_version(void) { return 1 * 10000 + 0 * 100 + 0; }

int tf_tune_set(int key, int value)
{
    if (key < 0 || key > 6)
        return fail(TF_E_INVALID_ARG, "tf_tune_set: unknown key %d", key);
    if (key == TF_TUNE_ROWBLOCKS && value > 0 && value != 1 && value != 2 && value != 4 && value != 8 && value != 16)
        return fail(TF_E_INVALID_ARG, "tf_tune_set: row blocks per round must be 1, 2, 4, 8 or 16");
    g_tune[key] = value > 0 ? value : -1;
    return TF_OK;
}

size_t tf_qlinear_packed_bytes(int64_t batch, int64_t N, int64_t K, int bits, int group)
{
    const bool ok_code = (group == kGroup && (bits == 4 || bits == 8)) || (group == 16 && bits == 4);
    if (!ok_code || K <= 0 || K % kGroup != 0 || N < 1 || batch < 1)
        return 0;
    const int64_t n_pad = (N + 15) / 16 * 16;
    const bool nvfp4 = group == 16;
    return (size_t)TF_PACK_HEADER_BYTES + (size_t)batch * (n_pad / 16) * (K / kGroup) * tile_bytes_for(bits) +
           (nvfp4 ? nvfp4_scale_table_bytes(batch) : 0);
}

int tf_qlinear_pack(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases, int64_t batch, int64_t N,
                    int64_t K, int bits, int group, void* packed, size_t packed_bytes, tf_qweight* desc,
                    void* stream)
{
    if (bits != 4 && bits != 8)
        return fail(TF_E_UNSUPPORTED_SHAPE, "tf_qlinear_pack: bits must be 4 or 8 (got %d)", bits);
    if (group != kGroup)
        return fail(TF_E_UNSUPPORTED_SHAPE, "tf_qlinear_pack: group must be 64 (got %d)", group);
    if (K <= 0 || K % kGroup != 0)
        return fail(TF_E_UNSUPPORTED_SHAPE, "tf_qlinear_pack: K must be a positive multiple of 64");
    if (N < 1 || batch < 1)
        return fail(TF_E_INVALID_ARG, "tf_qlinear_pack: N and batch must be >= 1");
    if (wq == nullptr || scales == nullptr || biases == nullptr || packed == nullptr || desc == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_qlinear_pack: NULL pointer");
    if (!aligned(packed, 16) || !aligned(wq, 4) || !aligned(scales, 2) || !aligned(biases, 2))
        return fail(TF_E_INVALID_ARG, "tf_qlinear_pack: misaligned pointer (packed needs 16 bytes)");
    const size_t need = tf_qlinear_packed_bytes(batch, N, K, bits, group);
    if (packed_bytes < need)
        return fail(TF_E_WORKSPACE_TOO_SMALL, "tf_qlinear_pack: packed buffer has %zu bytes, needs %zu", packed_bytes,
                    need);
    cudaError_t e = launch_pack(wq, scales, biases, batch, N, K, bits, static_cast<uint8_t*>(packed),
                                static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qlinear_pack");
    desc->magic = TF_QWEIGHT_MAGIC;
    desc->version = TF_PACK_VERSION;
    desc->bits = bits;
    desc->group = group;
    desc->code = TF_CODE_AFFINE;
    desc->global_scale = 1.f;
    desc->batch = batch;
    desc->N = N;
    desc->K = K;
    desc->n_pad = (N + 15) / 16 * 16;
    desc->tile_bytes = tile_bytes_for(bits);
    desc->matrix_bytes = desc->n_pad / 16 * (K / kGroup) * desc->tile_bytes;
    desc->data = packed;
    return TF_OK;
}

static int pack_nvfp4_impl(const uint8_t* codes, const uint8_t* block_scales, float global_scale,
                           const float* global_scales, int64_t batch, int64_t N, int64_t K, void* packed,
                           size_t packed_bytes, tf_qweight* desc, void* stream, const char* name)
{
    if (K <= 0 || K % kGroup != 0)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: K must be a positive multiple of 64", name);
    if (N < 1 || batch < 1)
        return fail(TF_E_INVALID_ARG, "%s: N and the number of matrices must be >= 1", name);
    if (!std::isfinite(global_scale))
        return fail(TF_E_INVALID_ARG, "%s: global_scale must be finite", name);
    if (codes == nullptr || block_scales == nullptr || packed == nullptr || desc == nullptr)
        return fail(TF_E_INVALID_ARG, "%s: NULL pointer", name);
    if (!aligned(packed, 16))
        return fail(TF_E_INVALID_ARG, "%s: packed must be 16-byte aligned", name);
    const size_t need = tf_qlinear_packed_bytes(batch, N, K, 4, 16);
    if (packed_bytes < need)
        return fail(TF_E_WORKSPACE_TOO_SMALL, "%s: packed buffer has %zu bytes, needs %zu", name, packed_bytes, need);
    PackHeader h{};
    h.magic = TF_QWEIGHT_MAGIC;
    h.version = TF_PACK_VERSION;
    h.bits = 4;
    h.group = 16;
    h.code = TF_CODE_NVFP4;
    h.global_scale = global_scale;
    h.batch = batch;
    h.N = N;
    h.K = K;
    h.n_pad = (N + 15) / 16 * 16;
    h.tile_bytes = tile_bytes_for(kNvfp4);
    h.matrix_bytes = h.n_pad / 16 * (K / kGroup) * h.tile_bytes;
    cudaError_t e = launch_pack_nvfp4(codes, block_scales, global_scales, batch, N, K, static_cast<uint8_t*>(packed),
                                      h, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, name);
    desc->magic = h.magic;
    desc->version = h.version;
    desc->bits = h.bits;
    desc->group = h.group;
    desc->code = h.code;
    desc->global_scale = h.global_scale;
    desc->batch = h.batch;
    desc->N = N;
    desc->K = K;
    desc->n_pad = h.n_pad;
    desc->tile_bytes = h.tile_bytes;
    desc->matrix_bytes = h.matrix_bytes;
    desc->data = packed;
    return TF_OK;
}

int tf_qlinear_pack_nvfp4(const uint8_t* codes, const uint8_t* block_scales, float global_scale, int64_t N, int64_t K,
                          void* packed, size_t packed_bytes, tf_qweight* desc, void* stream)
{
    return pack_nvfp4_impl(codes, block_scales, global_scale, nullptr, 1, N, K, packed, packed_bytes, desc, stream,
                           "tf_qlinear_pack_nvfp4");
}

int tf_qlinear_pack_nvfp4_experts(const uint8_t* codes, const uint8_t* block_scales, const float* global_scales,
                                  int64_t E, int64_t N, int64_t K, void* packed, size_t packed_bytes, tf_qweight* desc,
                                  void* stream)
{
    if (global_scales == nullptr || !aligned(global_scales, 4))
        return fail(TF_E_INVALID_ARG, "tf_qlinear_pack_nvfp4_experts: global_scales NULL or misaligned");
    // the descriptor's own global_scale is not used for a batch: each matrix's comes from the
    // scale table in the packed buffer
    return pack_nvfp4_impl(codes, block_scales, 1.f, global_scales, E, N, K, packed, packed_bytes, desc, stream,
                           "tf_qlinear_pack_nvfp4_experts");
}

int tf_qlinear_unpack_debug(const tf_qweight* w, uint32_t* wq, uint16_t* scales, uint16_t* biases, void* stream)
{
    int rc = check_desc(w, "tf_qlinear_unpack_debug");
    if (rc)
        return rc;
    if (w->code == TF_CODE_NVFP4) {
        if (wq == nullptr || scales == nullptr)
            return fail(TF_E_INVALID_ARG, "tf_qlinear_unpack_debug: NULL output");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaSuccess;
        for (int64_t b = 0; b < w->batch && e == cudaSuccess; ++b)
            e = launch_unpack_nvfp4(static_cast<const uint8_t*>(w->data) + b * w->matrix_bytes, w->N, w->K,
                                    reinterpret_cast<uint8_t*>(wq) + b * w->N * (w->K / 2),
                                    reinterpret_cast<uint8_t*>(scales) + b * w->N * (w->K / 16), st);
        if (e == cudaSuccess && biases != nullptr)  // the per-matrix fp32 scales, when asked for
            e = cudaMemcpyAsync(biases, nvfp4_scales_of(w), (size_t)w->batch * sizeof(float),
                                cudaMemcpyDeviceToDevice, st);
        return e == cudaSuccess ? TF_OK : cuda_fail(e, "tf_qlinear_unpack_debug");
    }
    if (wq == nullptr || scales == nullptr || biases == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_qlinear_unpack_debug: NULL output");
    cudaError_t e = launch_unpack(static_cast<const uint8_t*>(w->data), w->batch, w->N, w->K, w->bits, wq, scales,
                                  biases, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qlinear_unpack_debug");
    return TF_OK;
}

int tf_qweight_check(const tf_qweight* w, void* stream)
{
    int rc = check_desc(w, "tf_qweight_check");
    if (rc)
        return rc;
    PackHeader h;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, w->data, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qweight_check");
    if (h.magic != w->magic || h.version != w->version || h.bits != w->bits || h.group != w->group ||
        h.code != w->code || !(h.global_scale == w->global_scale) ||
        h.batch != w->batch || h.N != w->N || h.K != w->K || h.n_pad != w->n_pad || h.tile_bytes != w->tile_bytes ||
        h.matrix_bytes != w->matrix_bytes)
        return fail(TF_E_BAD_PACK, "tf_qweight_check: device header does not match the descriptor");
    return TF_OK;
}

// ------------------------------------------------------------------ projections

// Split-K scratch of the plans for every activation row count up to 8, with and without
// an RMSNorm prologue, so one workspace serves any call of these weights.
static size_t qlinear_scratch_all_m(const tf_qweight* w, const tf_qweight* w_up)
{
    size_t r = 0;
    for (int rows = 1; rows <= kMaxM; ++rows)
        for (int k_full : {0, (int)w->K}) {  // with and without an RMSNorm prologue
            const Plan pl =
                plan_qproj((int)(w->n_pad / 16), (int)(w->K / kGroup), w_up ? 2 : 1, kernel_bits(w), 1, k_full, rows);
            r = std::max(r, plan_scratch(pl));
        }
    return r;
}

size_t tf_qlinear_workspace_bytes(const tf_qweight* w, int64_t M)
{
    (void)M;
    if (check_desc(w, "tf_qlinear_workspace_bytes"))
        return 0;
    return kStatusBytes + qlinear_scratch_all_m(w, nullptr);
}

// `ws` holds the status word; `scratch` (scratch_bytes) the split-K counters and partials.
static int qlinear_impl(const tf_qweight* w, const tf_qweight* w_up, const uint16_t* x, int64_t ldx, int64_t M,
                        const uint16_t* gamma, float eps, const uint16_t* residual, void* y, int64_t ldy, int y_dtype,
                        void* ws, uint8_t* scratch, size_t scratch_bytes, bool pdl, cudaStream_t stream,
                        const char* name, const uint8_t* rht = nullptr)
{
    const bool dual = w_up != nullptr;
    const Plan pl = plan_qproj((int)(w->n_pad / 16), (int)(w->K / kGroup), dual ? 2 : 1, kernel_bits(w), 1,
                               gamma != nullptr ? (int)w->K : 0, (int)M);
    if (pl.smem > 227 * 1024)
        return fail(TF_E_UNSUPPORTED_SHAPE,
                    gamma != nullptr ? "%s: K too large for the RMSNorm prologue (rows do not fit on chip)"
                                     : "%s: the activation rows of a K split do not fit on chip",
                    name);
    if (scratch_bytes < plan_scratch(pl))
        return fail(TF_E_WORKSPACE_TOO_SMALL, "%s: workspace too small for the launch plan", name);
    QProjParams p{};
    p.w0 = tiles_of(w);
    p.w1 = dual ? tiles_of(w_up) : nullptr;
    p.matrix_bytes = w->matrix_bytes;
    p.n_rb = (int)(w->n_pad / 16);
    p.groups = (int)(w->K / kGroup);
    p.N = (int)w->N;
    p.K = (int)w->K;
    p.x = x;
    p.ldx = ldx;
    p.M = (int)M;
    p.gamma = gamma;
    p.eps = eps;
    p.residual = residual;
    p.ldr = w->N;
    p.y = y;
    p.ldy = ldy;
    p.y_f32 = y_dtype == TF_DTYPE_F32;
    fill_common(p, pl, ws, scratch);
    p.rht = rht;
    p.wscale0 = w->global_scale;
    p.wscale1 = dual ? w_up->global_scale : 1.f;
    cudaError_t e = launch_qproj(kernel_bits(w), dual, false, pl, p, stream, pdl);
    if (e != cudaSuccess)
        return cuda_fail(e, name);
    return TF_OK;
}

static int qlinear_entry(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint8_t* rht,
                         const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual, void* y, int y_dtype,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream, const char* name);

int tf_qlinear_run(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint16_t* rms_gamma,
                   float rms_eps, const uint16_t* residual, void* y, int y_dtype, void* ws, size_t ws_bytes,
                   unsigned flags, void* stream)
{
    return qlinear_entry(w, x, ldx, M, nullptr, rms_gamma, rms_eps, residual, y, y_dtype, ws, ws_bytes, flags, stream,
                         "tf_qlinear_run");
}

int tf_qlinear_run_rht(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint8_t* rht_signs,
                       const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual, void* y, int y_dtype,
                       void* ws, size_t ws_bytes, unsigned flags, void* stream)
{
    if (rht_signs == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_qlinear_run_rht: rht_signs is NULL");
    return qlinear_entry(w, x, ldx, M, rht_signs, rms_gamma, rms_eps, residual, y, y_dtype, ws, ws_bytes, flags,
                         stream, "tf_qlinear_run_rht");
}

static int qlinear_entry(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint8_t* rht,
                         const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual, void* y, int y_dtype,
                         void* ws, size_t ws_bytes, unsigned flags, void* stream, const char* name)
{
    int rc = check_desc(w, name);
    if (rc)
        return rc;
    if (w->batch != 1)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: batch must be 1 (use tf_qmoe_run for experts)", name);
    if (M < 1 || M > kMaxM)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: M must be in [1, 8] (got %lld)", name, (long long)M);
    char what[96];
    snprintf(what, sizeof what, "%s: x", name);
    if ((rc = check_act(x, ldx, w->K, what)))
        return rc;
    if (rms_gamma != nullptr && (!aligned(rms_gamma, 16) || !(rms_eps >= 0.f)))
        return fail(TF_E_INVALID_ARG, "%s: rms_gamma must be 16-byte aligned and rms_eps >= 0", name);
    if (y == nullptr || (y_dtype != TF_DTYPE_BF16 && y_dtype != TF_DTYPE_F32))
        return fail(TF_E_INVALID_ARG, "%s: y NULL or bad y_dtype", name);
    if (ws == nullptr || !aligned(ws, 256))
        return fail(TF_E_INVALID_ARG, "%s: workspace NULL or not 256-byte aligned", name);
    if (ws_bytes < kStatusBytes)
        return fail(TF_E_WORKSPACE_TOO_SMALL, "%s: workspace too small", name);
    return qlinear_impl(w, nullptr, x, ldx, M, rms_gamma, rms_eps, residual, y, w->N, y_dtype, ws,
                        static_cast<uint8_t*>(ws) + kStatusBytes, ws_bytes - kStatusBytes, (flags & TF_RUN_PDL) != 0,
                        static_cast<cudaStream_t>(stream), name, rht);
}

extern "C++" {
namespace tfq {
int qlinear_run_named(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint16_t* rms_gamma,
                      float rms_eps, const uint16_t* residual, void* y, int y_dtype, void* ws, size_t ws_bytes,
                      unsigned flags, void* stream, const char* name)
{
    return qlinear_entry(w, x, ldx, M, nullptr, rms_gamma, rms_eps, residual, y, y_dtype, ws, ws_bytes, flags, stream,
                         name);
}
}  // namespace tfq
}  // extern "C++"

size_t tf_qmlp_gateup_workspace_bytes(const tf_qweight* gate, const tf_qweight* up, int64_t M)
{
    (void)M;
    if (check_desc(gate, "gate") || check_desc(up, "up"))
        return 0;
    return kStatusBytes + qlinear_scratch_all_m(gate, up);
}

int tf_qmlp_gateup_run(const tf_qweight* gate, const tf_qweight* up, const uint16_t* x, int64_t ldx, int64_t M,
                       const uint16_t* rms_gamma, float rms_eps, uint16_t* h, void* ws, size_t ws_bytes,
                       unsigned flags, void* stream)
{
    int rc = check_desc(gate, "tf_qmlp_gateup_run: gate");
    if (rc || (rc = check_desc(up, "tf_qmlp_gateup_run: up")))
        return rc;
    if (gate->batch != 1 || up->batch != 1 || gate->N != up->N || gate->K != up->K || gate->bits != up->bits ||
        gate->code != up->code)
        return fail(TF_E_UNSUPPORTED_SHAPE,
                    "tf_qmlp_gateup_run: gate and up must have equal N, K, bits, weight code and batch 1");
    if (M < 1 || M > kMaxM)
        return fail(TF_E_UNSUPPORTED_SHAPE, "tf_qmlp_gateup_run: M must be in [1, 8]");
    if ((rc = check_act(x, ldx, gate->K, "tf_qmlp_gateup_run: x")))
        return rc;
    if (rms_gamma != nullptr && (!aligned(rms_gamma, 16) || !(rms_eps >= 0.f)))
        return fail(TF_E_INVALID_ARG, "tf_qmlp_gateup_run: rms_gamma must be 16-byte aligned and rms_eps >= 0");
    if (h == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_qmlp_gateup_run: h is NULL");
    if (ws == nullptr || !aligned(ws, 256))
        return fail(TF_E_INVALID_ARG, "%s: workspace NULL or not 256-byte aligned", "tf_qmlp_gateup_run");
    if (ws_bytes < kStatusBytes)
        return fail(TF_E_WORKSPACE_TOO_SMALL, "%s: workspace too small", "tf_qmlp_gateup_run");
    return qlinear_impl(gate, up, x, ldx, M, rms_gamma, rms_eps, nullptr, h, gate->N, TF_DTYPE_BF16, ws,
                        static_cast<uint8_t*>(ws) + kStatusBytes, ws_bytes - kStatusBytes, (flags & TF_RUN_PDL) != 0,
                        static_cast<cudaStream_t>(stream), "tf_qmlp_gateup_run");
}

// ------------------------------------------------------------------ MoE

namespace {
struct MoeLayout {
    Plan pgu, pdn;
    size_t meta, h, o, gu, dn, total;
    int slots;
};

MoeLayout moe_layout(const tf_qweight* gate, const tf_qweight* down, int64_t M, int top_k)
{
    MoeLayout L{};
    const int E = (int)gate->batch;
    L.slots = (int)(M * top_k < E ? M * top_k : E);
    L.pgu = plan_qproj((int)(gate->n_pad / 16), (int)(gate->K / kGroup), 2, kernel_bits(gate), L.slots, 0, kMaxM);
    L.pdn = plan_qproj((int)(down->n_pad / 16), (int)(down->K / kGroup), 1, kernel_bits(down), L.slots, 0, kMaxM);
    L.meta = kStatusBytes;
    L.h = align_up(L.meta + sizeof(MoeMeta), 256);
    L.o = align_up(L.h + (size_t)L.slots * kMaxM * gate->N * sizeof(uint16_t), 256);
    L.gu = align_up(L.o + (size_t)L.slots * kMaxM * down->N * sizeof(float), 256);
    L.dn = align_up(L.gu + plan_scratch(L.pgu), 256);
    L.total = align_up(L.dn + plan_scratch(L.pdn), 256);
    return L;
}

int check_moe(const tf_qweight* gate, const tf_qweight* up, const tf_qweight* down, int64_t M, int top_k,
              const char* name)
{
    int rc = check_desc(gate, "gate");
    if (rc || (rc = check_desc(up, "up")) || (rc = check_desc(down, "down")))
        return rc;
    if (up->code != gate->code || down->code != gate->code)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: gate, up and down must share one weight code", name);
    if (up->batch != gate->batch || down->batch != gate->batch || up->N != gate->N || up->K != gate->K ||
        down->K != gate->N || down->N != gate->K || up->bits != gate->bits || down->bits != gate->bits)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: expert shapes must be gate/up [E][I][H], down [E][H][I]", name);
    if (gate->batch > 1024)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: at most 1024 experts", name);
    if (M < 1 || M > kMaxM || top_k < 1 || top_k > 8 || top_k > gate->batch)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: need 1 <= M <= 8 and 1 <= top_k <= min(8, E)", name);
    if (gate->N % 8 != 0)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: expert intermediate size must be a multiple of 8", name);
    return TF_OK;
}
}  // namespace

size_t tf_qmoe_workspace_bytes(const tf_qweight* gate, const tf_qweight* up, const tf_qweight* down, int64_t M,
                               int top_k)
{
    if (check_moe(gate, up, down, M, top_k, "tf_qmoe_workspace_bytes"))
        return 0;
    return moe_layout(gate, down, M, top_k).total;
}

int tf_qmoe_run(const tf_qweight* gate, const tf_qweight* up, const tf_qweight* down, const float* router_logits,
                int64_t M, int top_k, const uint16_t* x, uint16_t* y, int32_t* topk_idx, float* topk_w, void* ws,
                size_t ws_bytes, unsigned flags, void* stream)
{
    int rc = check_moe(gate, up, down, M, top_k, "tf_qmoe_run");
    if (rc)
        return rc;
    if (router_logits == nullptr || y == nullptr || topk_idx == nullptr || topk_w == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_qmoe_run: NULL pointer");
    if ((rc = check_act(x, gate->K, gate->K, "tf_qmoe_run: x")))
        return rc;
    const MoeLayout L = moe_layout(gate, down, M, top_k);
    if (ws == nullptr || !aligned(ws, 256))
        return fail(TF_E_INVALID_ARG, "tf_qmoe_run: workspace NULL or not 256-byte aligned");
    if (ws_bytes < L.total)
        return fail(TF_E_WORKSPACE_TOO_SMALL, "tf_qmoe_run: workspace has %zu bytes, needs %zu", ws_bytes, L.total);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    MoeMeta* meta = reinterpret_cast<MoeMeta*>(wsb + L.meta);
    uint16_t* hbuf = reinterpret_cast<uint16_t*>(wsb + L.h);
    float* obuf = reinterpret_cast<float*>(wsb + L.o);
    const int H = (int)gate->K, I = (int)gate->N;

    cudaError_t e = launch_moe_route(router_logits, (int)M, (int)gate->batch, top_k, topk_idx, topk_w, meta, s,
                                     (flags & TF_RUN_PDL) != 0);
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qmoe_run: route");

    QProjParams p{};
    p.w0 = tiles_of(gate);
    p.w1 = tiles_of(up);
    p.matrix_bytes = gate->matrix_bytes;
    p.n_rb = (int)(gate->n_pad / 16);
    p.groups = H / kGroup;
    p.N = I;
    p.K = H;
    p.x = x;
    p.ldx = H;
    p.M = (int)M;
    p.y = hbuf;
    p.ldy = I;
    p.y_f32 = 0;
    p.y_slot_stride = (int64_t)kMaxM * I;
    p.meta = meta;
    p.gather = 1;
    fill_common(p, L.pgu, ws, wsb + L.gu);
    p.wscales0 = nvfp4_scales_of(gate);
    p.wscales1 = nvfp4_scales_of(up);
    e = launch_qproj(kernel_bits(gate), true, true, L.pgu, p, s, true);
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qmoe_run: gate/up");

    QProjParams q{};
    q.w0 = tiles_of(down);
    q.matrix_bytes = down->matrix_bytes;
    q.n_rb = (int)(down->n_pad / 16);
    q.groups = I / kGroup;
    q.N = H;
    q.K = I;
    q.x = hbuf;
    q.ldx = I;
    q.M = (int)M;
    q.x_slot_stride = (int64_t)kMaxM * I;
    q.y = obuf;
    q.ldy = H;
    q.y_f32 = 1;
    q.y_slot_stride = (int64_t)kMaxM * H;
    q.meta = meta;
    q.meta_ready = 1;  // written by the routing kernel, which the gate/up launch waited for
    q.gather = 0;
    fill_common(q, L.pdn, ws, wsb + L.dn);
    q.wscales0 = nvfp4_scales_of(down);
    e = launch_qproj(kernel_bits(down), false, true, L.pdn, q, s, true);
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qmoe_run: down");

    e = launch_moe_combine(meta, obuf, (int)M, top_k, H, y, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_qmoe_run: combine");
    return TF_OK;
}

// ------------------------------------------------------------------ decoder step

namespace {
struct StepLayout {
    Plan p_qkv, p_o, p_gu, p_dn, p_ro;
    size_t bar, ssq, act, red, total;
    size_t qkv_e, h_e, a_e;  // elements per activation buffer
};

int check_decoder(const tf_decoder_desc* d, int64_t M, const char* name)
{
    if (d == nullptr || d->layers == nullptr || d->final_norm == nullptr)
        return fail(TF_E_INVALID_ARG, "%s: NULL descriptor, layers or final_norm", name);
    if (d->n_layers < 0 || M < 1 || M > kMaxM)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: need n_layers >= 0 and 1 <= M <= 8", name);
    const int64_t D = d->d_model, F = d->d_ff, Q = d->q_dim, KV = d->kv_dim;
    if (D <= 0 || D % kGroup || F <= 0 || F % kGroup || Q <= 0 || Q % kGroup || KV < 0 || KV % 8 || d->vocab <= 0)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: dimensions must be positive multiples of 64", name);
    int rc;
    for (int l = 0; l < d->n_layers; ++l) {
        const tf_decoder_layer& L = d->layers[l];
        if ((rc = check_desc(&L.qkv, "qkv")) || (rc = check_desc(&L.o, "o")) || (rc = check_desc(&L.gate, "gate")) ||
            (rc = check_desc(&L.up, "up")) || (rc = check_desc(&L.down, "down")))
            return rc;
        // one weight code for the whole step (the workspace is planned from layer 0)
        const int code = d->layers[0].qkv.code;
        if (L.qkv.code != code || L.o.code != code || L.gate.code != code || L.up.code != code ||
            L.down.code != code || d->readout.code != code)
            return fail(TF_E_UNSUPPORTED_SHAPE, "%s: layer %d mixes weight codes", name, l);
        if (L.qkv.N != Q + 2 * KV || L.qkv.K != D || L.o.N != D || L.o.K != Q || L.gate.N != F || L.gate.K != D ||
            L.up.N != F || L.up.K != D || L.down.N != D || L.down.K != F || L.gate.bits != L.up.bits ||
            L.qkv.batch != 1 || L.o.batch != 1 || L.gate.batch != 1 || L.up.batch != 1 || L.down.batch != 1)
            return fail(TF_E_UNSUPPORTED_SHAPE, "%s: layer %d weight shapes do not match the dimensions", name, l);
        if (L.attn_norm == nullptr || L.mlp_norm == nullptr || !aligned(L.attn_norm, 16) || !aligned(L.mlp_norm, 16))
            return fail(TF_E_INVALID_ARG, "%s: layer %d norm weights NULL or misaligned", name, l);
    }
    if ((rc = check_desc(&d->readout, "readout")))
        return rc;
    if (d->readout.N != d->vocab || d->readout.K != D || d->readout.batch != 1)
        return fail(TF_E_UNSUPPORTED_SHAPE, "%s: readout must be [vocab][d_model]", name);
    if (!aligned(d->final_norm, 16))
        return fail(TF_E_INVALID_ARG, "%s: final_norm misaligned", name);
    return TF_OK;
}

StepLayout step_layout(const tf_decoder_desc* d, int64_t M)
{
    StepLayout L{};
    const int bits = d->n_layers > 0 ? d->layers[0].qkv.bits : d->readout.bits;
    const int D = (int)d->d_model, F = (int)d->d_ff, Q = (int)d->q_dim, KV = (int)d->kv_dim;
    (void)bits;
    if (d->n_layers > 0) {
        const tf_decoder_layer& l0 = d->layers[0];
        L.p_qkv = plan_qproj((int)(l0.qkv.n_pad / 16), D / kGroup, 1, kernel_bits(&l0.qkv), 1, 0, kMaxM);
        L.p_o = plan_qproj((int)(l0.o.n_pad / 16), Q / kGroup, 1, kernel_bits(&l0.o), 1, 0, kMaxM);
        L.p_gu = plan_qproj((int)(l0.gate.n_pad / 16), D / kGroup, 2, kernel_bits(&l0.gate), 1, 0, kMaxM);
        L.p_dn = plan_qproj((int)(l0.down.n_pad / 16), F / kGroup, 1, kernel_bits(&l0.down), 1, 0, kMaxM);
    }
    L.p_ro = plan_qproj((int)(d->readout.n_pad / 16), D / kGroup, 1, kernel_bits(&d->readout), 1, 0, kMaxM);
    L.qkv_e = (size_t)kMaxM * (Q + 2 * KV);
    L.h_e = (size_t)kMaxM * D;
    L.a_e = (size_t)kMaxM * F;
    (void)M;
    L.bar = kStatusBytes;  // stage arrival counters of the single-kernel step: 4 per layer + 1
    L.ssq = align_up(L.bar + (size_t)(4 * d->n_layers + 1) * sizeof(unsigned), 256);  // [2 L][8] u64
    L.act = align_up(L.ssq + (size_t)2 * d->n_layers * kMaxM * sizeof(unsigned long long), 256);
    // qkv | h1 | a | h ping | h pong
    const size_t act_bytes = (L.qkv_e + L.h_e + L.a_e + 2 * L.h_e) * sizeof(uint16_t) + 5 * 256;
    L.red = align_up(L.act + act_bytes, 256);
    size_t r = qlinear_scratch_all_m(&d->readout, nullptr);
    if (d->n_layers > 0) {
        const tf_decoder_layer& l0 = d->layers[0];
        const size_t c[4] = {qlinear_scratch_all_m(&l0.qkv, nullptr), qlinear_scratch_all_m(&l0.o, nullptr),
                             qlinear_scratch_all_m(&l0.gate, &l0.up), qlinear_scratch_all_m(&l0.down, nullptr)};
        for (size_t v : c)
            r = v > r ? v : r;
    }
    L.total = align_up(L.red + r, 256);
    return L;
}
}  // namespace

size_t tf_decode_step_workspace_bytes(const tf_decoder_desc* d, int64_t M)
{
    if (check_decoder(d, M, "tf_decode_step_workspace_bytes"))
        return 0;
    return step_layout(d, M).total;
}

size_t tf_decode_step_debug_elems(const tf_decoder_desc* d, int64_t M)
{
    if (check_decoder(d, M, "tf_decode_step_debug_elems"))
        return 0;
    return (size_t)d->n_layers * M * (d->q_dim + 2 * d->kv_dim + d->d_model + d->d_ff + d->d_model);
}

int tf_decode_step_run(const tf_decoder_desc* d, const uint16_t* x, int64_t M, uint16_t* logits, void* ws,
                       size_t ws_bytes, uint16_t* debug, unsigned flags, void* stream)
{
    int rc = check_decoder(d, M, "tf_decode_step_run");
    if (rc)
        return rc;
    if ((rc = check_act(x, d->d_model, d->d_model, "tf_decode_step_run: x")))
        return rc;
    if (logits == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_decode_step_run: logits is NULL");
    if (debug != nullptr && !aligned(debug, 16))
        return fail(TF_E_INVALID_ARG, "tf_decode_step_run: debug buffer must be 16-byte aligned");
    const StepLayout L = step_layout(d, M);
    if (ws == nullptr || !aligned(ws, 256))
        return fail(TF_E_INVALID_ARG, "tf_decode_step_run: workspace NULL or not 256-byte aligned");
    if (ws_bytes < L.total)
        return fail(TF_E_WORKSPACE_TOO_SMALL, "tf_decode_step_run: workspace has %zu bytes, needs %zu", ws_bytes,
                    L.total);
    const int64_t D = d->d_model, F = d->d_ff, Q = d->q_dim, KV = d->kv_dim;
    const int64_t QKV = Q + 2 * KV;
    if (debug != nullptr && ((M * QKV) % 8 || (M * D) % 8 || (M * F) % 8))
        return fail(TF_E_UNSUPPORTED_SHAPE, "tf_decode_step_run: debug blocks need M*dim to be a multiple of 8");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint8_t* red = wsb + L.red;
    const size_t red_bytes = ws_bytes - L.red;
    uint16_t* act = reinterpret_cast<uint16_t*>(wsb + L.act);
    uint16_t* qkv_ws = act;
    uint16_t* h1_ws = reinterpret_cast<uint16_t*>(align_up(reinterpret_cast<uintptr_t>(qkv_ws + L.qkv_e), 256));
    uint16_t* a_ws = reinterpret_cast<uint16_t*>(align_up(reinterpret_cast<uintptr_t>(h1_ws + L.h_e), 256));
    uint16_t* hp_ws[2];
    hp_ws[0] = reinterpret_cast<uint16_t*>(align_up(reinterpret_cast<uintptr_t>(a_ws + L.a_e), 256));
    hp_ws[1] = reinterpret_cast<uint16_t*>(align_up(reinterpret_cast<uintptr_t>(hp_ws[0] + L.h_e), 256));

    const size_t per_layer = (size_t)M * (QKV + D + F + D);

    // ---- the whole step as one persistent kernel, on request (TF_TUNE_CHAIN = 2): on GB300
    // its grid-wide stage barriers cost more than the kernel boundaries of the chain of
    // projections with programmatic dependent launch, which is therefore the default
    int bits = d->readout.bits;
    bool chain = g_tune[TF_TUNE_CHAIN] == 2 && d->readout.code == TF_CODE_AFFINE && d->n_layers <= kChainMaxLayers &&
                 D >= kGroup &&
                 std::max<int64_t>(D, std::max<int64_t>(Q, F)) <= (int64_t)kChainMaxGroups * kGroup &&
                 d->vocab <= INT32_MAX;
    for (int l = 0; chain && l < d->n_layers; ++l) {
        const tf_decoder_layer& Ly = d->layers[l];
        chain = Ly.qkv.bits == bits && Ly.o.bits == bits && Ly.gate.bits == bits && Ly.up.bits == bits &&
                Ly.down.bits == bits;
    }
    ChainParams cp{};
    size_t chain_smem_bytes = 0;
    if (chain) {
        chain_smem_bytes = chain_smem(bits, (int)std::max<int64_t>(D, std::max<int64_t>(Q, F)), (int)D, &cp.nst,
                                      &cp.x_rs, &cp.xsum_off, &cp.red_off, &cp.gamma_off, &cp.xraw_off, &cp.ring_off);
        chain = cp.nst >= 2 && chain_fits(bits, chain_smem_bytes);
    }
    if (!chain && g_tune[TF_TUNE_CHAIN] == 2)
        return fail(TF_E_UNSUPPORTED_SHAPE, "tf_decode_step_run: the single-kernel step cannot run for these shapes "
                                            "on this device (and it was required)");
    if (chain && d->n_layers > 0) {
        cp.L = d->n_layers;
        cp.M = (int)M;
        cp.D = (int)D;
        cp.F = (int)F;
        cp.Q = (int)Q;
        cp.KV = (int)KV;
        cp.eps = d->eps;
        cp.C = device_sms();
        cp.limit_ns = kDefaultWaitLimitNs;
        cp.x = x;
        if (debug != nullptr) {
            cp.buf[0] = debug;
            cp.buf[1] = debug + M * QKV;
            cp.buf[2] = debug + M * (QKV + D);
            cp.buf[3] = debug + M * (QKV + D + F);
            for (int r = 0; r < 4; ++r)
                cp.lstride[r] = (int64_t)per_layer;
        } else {
            cp.buf[0] = qkv_ws;
            cp.buf[1] = h1_ws;
            cp.buf[2] = a_ws;
            cp.buf[3] = hp_ws[0];
            cp.astride[3] = hp_ws[1] - hp_ws[0];
        }
        cp.bar = reinterpret_cast<unsigned*>(wsb + L.bar);
        cp.ssq = reinterpret_cast<unsigned long long*>(wsb + L.ssq);
        cp.status = static_cast<int*>(ws);
        for (int l = 0; l < d->n_layers; ++l) {
            const tf_decoder_layer& Ly = d->layers[l];
            cp.layer[l] = ChainLayerW{tiles_of(&Ly.qkv), tiles_of(&Ly.o), tiles_of(&Ly.gate), tiles_of(&Ly.up),
                                      tiles_of(&Ly.down), Ly.attn_norm, Ly.mlp_norm};
        }
        const cudaError_t e = launch_chain(bits, cp, chain_smem_bytes, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "tf_decode_step_run: single-kernel step");
        // the final RMSNorm + readout: its own kernel, streaming its weights while the
        // layers finish (programmatic dependent launch)
        const int Ll = d->n_layers - 1;
        const uint16_t* h_last = debug != nullptr ? debug + (size_t)Ll * per_layer + M * (QKV + D + F) : hp_ws[Ll & 1];
        return qlinear_impl(&d->readout, nullptr, h_last, D, M, d->final_norm, d->eps, nullptr, logits, d->vocab,
                            TF_DTYPE_BF16, ws, red, red_bytes, true, s, "tf_decode_step_run: readout");
    }

    // ---- one kernel per projection
    bool pdl = (flags & TF_RUN_PDL) != 0;
    const uint16_t* h = x;
    for (int l = 0; l < d->n_layers; ++l) {
        const tf_decoder_layer& Ly = d->layers[l];
        uint16_t *qkv, *h1, *a, *h2;
        if (debug != nullptr) {
            qkv = debug + l * per_layer;
            h1 = qkv + M * QKV;
            a = h1 + M * D;
            h2 = a + M * F;
        } else {
            qkv = qkv_ws;
            h1 = h1_ws;
            a = a_ws;
            h2 = hp_ws[l & 1];
        }
        if ((rc = qlinear_impl(&Ly.qkv, nullptr, h, D, M, Ly.attn_norm, d->eps, nullptr, qkv, QKV, TF_DTYPE_BF16, ws, red,
                               red_bytes, pdl, s, "tf_decode_step_run: qkv")))
            return rc;
        pdl = true;
        // the q part of qkv stands in for the attention output
        if ((rc = qlinear_impl(&Ly.o, nullptr, qkv, QKV, M, nullptr, 0.f, h, h1, D, TF_DTYPE_BF16, ws, red,
                               red_bytes, pdl, s, "tf_decode_step_run: o")))
            return rc;
        if ((rc = qlinear_impl(&Ly.gate, &Ly.up, h1, D, M, Ly.mlp_norm, d->eps, nullptr, a, F, TF_DTYPE_BF16, ws, red,
                               red_bytes, pdl, s, "tf_decode_step_run: gate/up")))
            return rc;
        if ((rc = qlinear_impl(&Ly.down, nullptr, a, F, M, nullptr, 0.f, h1, h2, D, TF_DTYPE_BF16, ws, red,
                               red_bytes, pdl, s, "tf_decode_step_run: down")))
            return rc;
        h = h2;
    }
    return qlinear_impl(&d->readout, nullptr, h, D, M, d->final_norm, d->eps, nullptr, logits, d->vocab, TF_DTYPE_BF16,
                        ws, red, red_bytes, pdl, s, "tf_decode_step_run: readout");
}

// ------------------------------------------------------------------ diagnostics

int tf_workspace_status(void* ws, void* stream)
{
    if (ws == nullptr)
        return fail(TF_E_INVALID_ARG, "tf_workspace_status: NULL workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, ws, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && st != 0) {
        e = cudaMemsetAsync(ws, 0, sizeof st, s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_workspace_status");
    if (st != 0)
        fail(st, "a device-side wait gave up (status recorded in the workspace)");
    return st;
}

int tf_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream)
{
    if (ws == nullptr) {  // the status word of tf_qlinear_run_noalloc's fixed array
        size_t bytes = 0;
        const int rc = noalloc_scratch(&ws, &bytes);
        if (rc)
            return rc;
    }
    if (!aligned(ws, 4))
        return fail(TF_E_INVALID_ARG, "tf_selftest_wait_timeout: misaligned workspace");
    if (limit_ns > 5000000000ull)
        return fail(TF_E_INVALID_ARG, "tf_selftest_wait_timeout: limit above 5 s");
    cudaError_t e = launch_timeout_probe(static_cast<int*>(ws), limit_ns, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "tf_selftest_wait_timeout");
    return TF_OK;
}

}  // extern "C"
