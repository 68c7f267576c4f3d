// C ABI of libqmv: argument validation, launch-geometry choice and launches.
// The public contract is documented in include/qmv.h.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "../../include/qmv.h"
#include "../../include/qmv_debug.h"
#include "gemv_tiles.cuh"
#include "kernels.h"

namespace qmv {

const void *gemv_tiles_fn_q4_0(int mode, int nc, int rw);
const void *gemv_tiles_fn_q4_K(int mode, int nc, int rw);
const void *gemv_tiles_mma_fn_q4_K(int mode);
const void *gemv_tiles_fn_q6_K(int mode, int nc, int rw);
const void *gemv_tiles_probe_fn_q4_0(int mode, int nc);
const void *gemv_tiles_probe_fn_q4_K(int mode, int nc);
const void *gemv_tiles_probe_fn_q6_K(int mode, int nc);
const void *gemv_tiles_yq_fn_q4_0(int mode, bool probe);
const void *gemv_tiles_yq_fn_q4_K(int mode, bool probe);
const void *gemv_tiles_yq_fn_q6_K(int mode, bool probe);
const void *gemv_tiles_rowrun_fn_q6_K(int mode, int nc);
const void *gemv_generic_fn_q4_0(int mode);
const void *gemv_generic_fn_q4_K(int mode);
const void *gemv_generic_fn_q6_K(int mode);

const void *gemv_tiles_fn(int type, int mode, int nc, int rw)
{
    switch (type) {
    case FMT_Q4_0: return gemv_tiles_fn_q4_0(mode, nc, rw);
    case FMT_Q4_K: return gemv_tiles_fn_q4_K(mode, nc, rw);
    case FMT_Q6_K: return gemv_tiles_fn_q6_K(mode, nc, rw);
    default: return nullptr;
    }
}

// The instrumented twin of the tile kernel gemv_tiles_fn(type, mode, nc, 4)
// (timeline and withheld share of qmv_debug.h); nullptr where none exists.
const void *gemv_tiles_probe_fn(int type, int mode, int nc)
{
    switch (type) {
    case FMT_Q4_0: return gemv_tiles_probe_fn_q4_0(mode, nc);
    case FMT_Q4_K: return gemv_tiles_probe_fn_q4_K(mode, nc);
    case FMT_Q6_K: return gemv_tiles_probe_fn_q6_K(mode, nc);
    default: return nullptr;
    }
}

// The tile kernel of the plain or gate/up GEMV of one column that also writes
// y as q8_1 blocks (qmv_mul_mat_vec_fused_q8_1), or its instrumented twin.
const void *gemv_tiles_yq_fn(int type, int mode, bool probe)
{
    switch (type) {
    case FMT_Q4_0: return gemv_tiles_yq_fn_q4_0(mode, probe);
    case FMT_Q4_K: return gemv_tiles_yq_fn_q4_K(mode, probe);
    case FMT_Q6_K: return gemv_tiles_yq_fn_q6_K(mode, probe);
    default: return nullptr;
    }
}

const void *gemv_generic_fn(int type, int mode)
{
    switch (type) {
    case FMT_Q4_0: return gemv_generic_fn_q4_0(mode);
    case FMT_Q4_K: return gemv_generic_fn_q4_K(mode);
    case FMT_Q6_K: return gemv_generic_fn_q6_K(mode);
    default: return nullptr;
    }
}

static int block_elems(int type) { return type == FMT_Q4_0 ? QK4_0 : QK_K; }
static int block_bytes(int type)
{
    return type == FMT_Q4_0 ? Q4_0_BYTES : type == FMT_Q4_K ? Q4_K_BYTES : Q6_K_BYTES;
}
static bool weight_type(int t) { return t == FMT_Q4_0 || t == FMT_Q4_K || t == FMT_Q6_K; }

// Sticky device fault word, reserved for kernels that detect a fault themselves
// (a bounded wait that ran out); read and cleared by qmv_device_fault.
__device__ unsigned int g_fault_word;

namespace {

constexpr int MAX_DEVICES = 64;
constexpr size_t SMEM_RESERVE = 2048;  // static shared memory (MoE token lists) and alignment slack per CTA
constexpr int F32_CLUSTER = 2;         // CTAs that share the quantization of fp32 activations (a TPC pair)
constexpr int MAX_CLUSTER = 8;         // portable cluster size limit
// MoE experts per call: the generic kernel gives every expert one grid row
// plus one for the invalid ids, and gridDim.y is at most 65535
constexpr int64_t MAX_EXPERTS = 65534;
// Delay of the early weight requests of launches that request their whole
// matrix early (q8_1 input), and of launches with fp32 input (plan_tiles).
constexpr int EARLY_DELAY_NS = 400;
constexpr int EARLY_DELAY_F32_NS = 700;

std::atomic<int> g_pdl{1};

// Diagnostic timeline (qmv_debug_trace): the next g_trace_slots launches that
// have an instrumented twin run it, each with a slot of TRACE_MAX_CTAS x
// TRACE_WORDS timestamps.
constexpr int TRACE_MAX_CTAS = 1024;
std::atomic<unsigned long long *> g_trace_buf{nullptr};
std::atomic<int64_t> g_trace_slots{0}, g_trace_next{0};

struct Tuning {
    std::atomic<int> threads{0}, slice_units{0}, stages{0}, ctas_per_sm{0}, smem_share{0}, cluster{0};
    std::atomic<int> dec_warps{0}, pre_tiles{0};
    std::atomic<int> mma_min_cols{0};  // 0: MMA_MIN_COLS; 9: never
    std::atomic<int> early_warps{0};   // 0: every decoding warp requests its early tiles
    std::atomic<int> early_delay_ns{0};  // 0: EARLY_DELAY_NS / EARLY_DELAY_F32_NS; -1: no delay
};
Tuning g_tuning[3];

int tidx(int type) { return type == FMT_Q4_0 ? 0 : type == FMT_Q4_K ? 1 : 2; }

std::mutex g_mu;
std::map<std::tuple<int, const void *, int, size_t>, int> g_occupancy;  // (dev, fn, threads, smem) -> CTAs/SM
std::map<std::tuple<int, const void *, int, size_t, int>, int> g_clusters;  // (..., cluster size) -> resident clusters
std::map<std::pair<int, const void *>, bool> g_smem_attr;
int g_num_sms[MAX_DEVICES];
int g_clock_khz[MAX_DEVICES];
int g_smem_optin[MAX_DEVICES];
int g_smem_sm[MAX_DEVICES];
int g_smem_resv[MAX_DEVICES];
std::map<const void *, size_t> g_static_smem;  // kernel -> static shared bytes
unsigned int *g_fault_ptr[MAX_DEVICES];

qmv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QMV_OK : QMV_ERR_CUDA; }

struct DevInfo {
    int dev;
    int num_sms;
    int clock_khz;      // peak SM clock
    size_t smem_limit;  // dynamic shared memory a CTA may use
    size_t smem_per_sm; // shared memory of one SM
    size_t smem_resv;   // shared memory the hardware reserves per CTA
    unsigned int *fault;
};

// ---- QMV_GEOM: launch-geometry overrides from the environment (tuning) ----
// "type:key=value,key=value;type:..." with type q4_0, q4_K or q6_K and keys
// threads, slice_units, stages, ctas_per_sm, smem_share, cluster (as for
// qmv_set_tuning), dec_warps, pre_tiles (qmv_set_stream_tuning),
// early_warps (qmv_set_early_warps), early_delay_ns (qmv_set_early_delay) and
// mma_min_cols (qmv_set_mma_min_cols).
// Read once, before the first GEMV call is planned; values go through the
// setters' range checks.
std::once_flag g_geom_once;
std::atomic<int> g_geom_status{QMV_OK};

bool parse_int(const std::string &s, int &v)
{
    if (s.empty() || s.size() > 9) return false;
    char *end = nullptr;
    const long x = strtol(s.c_str(), &end, 10);
    if (end != s.c_str() + s.size()) return false;
    v = static_cast<int>(x);
    return true;
}

bool apply_geom_entry(const std::string &entry)
{
    const size_t colon = entry.find(':');
    if (colon == std::string::npos) return false;
    const std::string tname = entry.substr(0, colon);
    const int type = tname == "q4_0" ? FMT_Q4_0 : tname == "q4_K" ? FMT_Q4_K : tname == "q6_K" ? FMT_Q6_K : -1;
    if (type < 0) return false;
    const Tuning &cur = g_tuning[tidx(type)];
    constexpr int NK = 11;
    int v[NK] = {cur.threads.load(),     cur.slice_units.load(), cur.stages.load(),
                 cur.ctas_per_sm.load(), cur.smem_share.load(),  cur.cluster.load(),
                 cur.dec_warps.load(),   cur.pre_tiles.load(),   cur.mma_min_cols.load(),
                 cur.early_warps.load(), cur.early_delay_ns.load()};
    static const char *const keys[NK] = {"threads",   "slice_units", "stages",       "ctas_per_sm", "smem_share",
                                         "cluster",   "dec_warps",   "pre_tiles",    "mma_min_cols",
                                         "early_warps", "early_delay_ns"};
    size_t pos = colon + 1;
    while (pos <= entry.size()) {
        size_t comma = entry.find(',', pos);
        if (comma == std::string::npos) comma = entry.size();
        const std::string kv = entry.substr(pos, comma - pos);
        const size_t eq = kv.find('=');
        if (eq == std::string::npos) return false;
        int k = 0;
        while (k < NK && kv.compare(0, eq, keys[k]) != 0) ++k;
        if (k == NK || !parse_int(kv.substr(eq + 1), v[k])) return false;
        pos = comma + 1;
    }
    return qmv_set_tuning(type, v[0], v[1], v[2], v[3], v[4], v[5]) == QMV_OK &&
           qmv_set_stream_tuning(type, v[6], v[7]) == QMV_OK && qmv_set_mma_min_cols(type, v[8]) == QMV_OK &&
           qmv_set_early_warps(type, v[9]) == QMV_OK && qmv_set_early_delay(type, v[10]) == QMV_OK;
}

qmv_status geom_env()
{
    std::call_once(g_geom_once, [] {
        const char *e = getenv("QMV_GEOM");
        if (!e || !*e) return;
        const std::string spec(e);
        size_t pos = 0;
        while (pos <= spec.size()) {
            size_t semi = spec.find(';', pos);
            if (semi == std::string::npos) semi = spec.size();
            if (semi > pos && !apply_geom_entry(spec.substr(pos, semi - pos))) {
                g_geom_status = QMV_ERR_CONFIG;
                return;
            }
            pos = semi + 1;
        }
    });
    return static_cast<qmv_status>(g_geom_status.load());
}

qmv_status device_info(DevInfo &d)
{
    const qmv_status g = geom_env();
    if (g != QMV_OK) return g;
    if (cudaGetDevice(&d.dev) != cudaSuccess) return QMV_ERR_CUDA;
    if (d.dev < 0 || d.dev >= MAX_DEVICES) return QMV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_num_sms[d.dev]) {
        int n = 0, optin = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d.dev) != cudaSuccess) return QMV_ERR_CUDA;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.dev) != cudaSuccess)
            return QMV_ERR_CUDA;
        g_smem_optin[d.dev] = optin;
        int per_sm = 0;
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d.dev) != cudaSuccess)
            return QMV_ERR_CUDA;
        g_smem_sm[d.dev] = per_sm;
        int resv = 0;
        if (cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, d.dev) != cudaSuccess) resv = 1024;
        g_smem_resv[d.dev] = resv;
        int khz = 0;
        if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, d.dev) != cudaSuccess || khz <= 0) khz = 2000000;
        g_clock_khz[d.dev] = khz;
        void *f = nullptr;
        if (cudaGetSymbolAddress(&f, g_fault_word) != cudaSuccess) return QMV_ERR_CUDA;
        g_fault_ptr[d.dev] = static_cast<unsigned int *>(f);
        g_num_sms[d.dev] = n;
    }
    d.num_sms = g_num_sms[d.dev];
    d.clock_khz = g_clock_khz[d.dev];
    d.smem_limit = static_cast<size_t>(g_smem_optin[d.dev]) - SMEM_RESERVE;
    d.smem_per_sm = static_cast<size_t>(g_smem_sm[d.dev]);
    d.smem_resv = static_cast<size_t>(g_smem_resv[d.dev]);
    d.fault = g_fault_ptr[d.dev];
    return QMV_OK;
}

size_t static_smem(const void *fn);

// Lets fn use as much dynamic shared memory as the opt-in limit leaves beside
// its static shared memory (at most d.smem_limit).
qmv_status ensure_smem_attr(const DevInfo &d, const void *fn)
{
    const size_t st = static_smem(fn);
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(d.dev, fn);
    if (g_smem_attr.count(key)) return QMV_OK;
    const size_t optin = static_cast<size_t>(g_smem_optin[d.dev]);
    const size_t lim = std::min(d.smem_limit, optin > st ? optin - st : size_t(0));
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(lim)) != cudaSuccess)
        return QMV_ERR_CUDA;
    g_smem_attr[key] = true;
    return QMV_OK;
}

size_t static_smem(const void *fn)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_static_smem.find(fn);
    if (it != g_static_smem.end()) return it->second;
    cudaFuncAttributes a{};
    const size_t v = cudaFuncGetAttributes(&a, fn) == cudaSuccess ? a.sharedSizeBytes : 2048;
    g_static_smem[fn] = v;
    return v;
}

int occupancy(int dev, const void *fn, int threads, size_t smem)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(dev, fn, threads, smem);
    auto it = g_occupancy.find(key);
    if (it != g_occupancy.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) n = 0;
    g_occupancy[key] = n;
    return n;
}

// Clusters of `cl` CTAs of fn that can be resident at once (0: none fits).
int cluster_occupancy(int dev, const void *fn, int threads, size_t smem, int cl)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_tuple(dev, fn, threads, smem, cl);
    auto it = g_clusters.find(key);
    if (it != g_clusters.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cl));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    g_clusters[key] = n;
    return n;
}

int round_nc(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Launch {
    const void *fn = nullptr;
    const void *probe = nullptr;  // fn's instrumented twin (qmv_debug.h), if it has one
    bool stream = false;
    int rw = 0;       // tile kernel: weight rows per warp tile
    int cluster = 1;  // CTAs per cluster (1: no cluster dimension)
    GemvParams p{};
    dim3 grid, block;
    size_t smem = 0;
};

int pow2_at_least(int v)
{
    int p2 = 1;
    while (p2 < v) p2 <<= 1;
    return p2;
}

// Rows the tile kernel takes: whole 16-byte pieces per row and whole tile
// units (Q4_0 / Q4_K: K % 256 == 0; Q6_K: K % 2048 == 0, eight 210-byte
// super-blocks per tile row), 16-byte aligned weights.
bool tile_shape_ok(int type, int64_t K, int64_t row_bytes)
{
    return row_bytes % 16 == 0 && K % (type == FMT_Q6_K ? 2048 : 256) == 0;
}

// Geometry of the tile kernel: warp tiles of RW rows x 32/RW units, a ring of
// `stages` tile buffers per warp; the grid covers every SM (one CTA per SM
// unless tuned) with up to 12 warps per CTA, every warp owning a balanced
// contiguous range of RW-row groups.  NoFit: the activations do not fit in
// shared memory (the caller may fall back to the generic kernel); Error: a
// CUDA call failed or the kernel is missing (never a silent fallback).
enum class TilePlan { Ok, NoFit, Error };

TilePlan plan_tiles(int type, int mode, const DevInfo &dev, GemvParams &p, int nc_t, int n_potential_experts,
                    Launch &L, bool allow_mma = true)
{
    const Tuning &tu = g_tuning[tidx(type)];
    const int U = static_cast<int>(p.K / 256);
    // the tensor-core decode (16-row tiles) for the plain Q4_K GEMV from
    // mma_min columns on; the same choice for q8_1 and fp32 input, so the two
    // stay bit-identical
    const int mma_min = tu.mma_min_cols.load() > 0 ? tu.mma_min_cols.load() : MMA_MIN_COLS;
    const bool yq = p.yq != nullptr;  // y also as q8_1 blocks: one column, 4-row tiles, dp4a decode
    const bool mma = !yq && allow_mma && type == FMT_Q4_K && mode == MODE_PLAIN && nc_t >= mma_min;
    int rw = 4;
    if (mma) rw = MMA_RW;
    else if (tu.slice_units.load() && !yq) rw = 32 / std::max(4, std::min(16, pow2_at_least(tu.slice_units.load())));
    const void *fn = yq    ? gemv_tiles_yq_fn(type, mode, false)
                     : mma ? gemv_tiles_mma_fn_q4_K(mode)
                           : gemv_tiles_fn(type, mode, nc_t, rw);
    if (!fn && rw != 4 && !mma) {
        rw = 4;
        fn = gemv_tiles_fn(type, mode, nc_t, rw);
    }
    if (!fn) return TilePlan::Error;
    // Q6_K, one plain column, two tiles or fewer per row group (short rows:
    // the stream bounds the launch, not the decode): tiles copied one row at a
    // time by the whole warp (on GB300, 32000x4096: 21.75 -> 20.94 us; on
    // 4096x14336 the same copy was 3 % slower)
    if (type == FMT_Q6_K && mode == MODE_PLAIN && nc_t == 1 && !yq && !mma && rw == 4 && U <= 2 * (32 / rw)) {
        const void *f2 = gemv_tiles_rowrun_fn_q6_K(mode, nc_t);
        if (f2) fn = f2;
    }
    const int sc_stride = type == FMT_Q6_K ? act_sc_stride<FMT_Q6_K>() : act_sc_stride<FMT_Q4_K>();
    const size_t packed = mma ? align_up(static_cast<size_t>(mma_act_bytes(nc_t, static_cast<int64_t>(U) * 8)), 128)
                              : align_up(static_cast<size_t>(nc_t) * U * (ACT_QS_STRIDE + sc_stride), 128);
    const size_t raw = align_up(static_cast<size_t>(nc_t) * U * 8 * Q8_1_BYTES, 128);
    // per warp: its ring of tile buffers, plus the row-factor scratch of the tensor-core decode
    const size_t tb = static_cast<size_t>(tile_bytes_rt(type, rw, mma));
    const size_t warp_extra = mma ? static_cast<size_t>(MMA_FAC_BYTES) : 0;
    int stages = tu.stages.load() ? tu.stages.load() : 2;
    stages = std::max(1, std::min(TILE_MAX_STAGES, stages));
    int max_wpc = tu.threads.load() ? tu.threads.load() / 32 : TILE_MAX_THREADS / 32;
    max_wpc = std::max(1, std::min(TILE_MAX_THREADS / 32, max_wpc));
    // every CTA has this many warps: all of them stage the activations (a
    // latency-bound phase that wants many warps), the first wpc of them also
    // stream and decode weight tiles
    const int cta_warps = max_wpc;

    // grid: every SM first (MoE: the SMs shared among the experts that may be
    // picked), then more warps per CTA; warps own whole row groups
    const int cps = tu.ctas_per_sm.load() > 0 ? tu.ctas_per_sm.load() : 1;
    const int64_t max_ctas = static_cast<int64_t>(cps) * dev.num_sms;
    const int64_t G = (p.M + rw - 1) / rw;
    int64_t gx = std::min(max_ctas, G);
    int64_t groups_per_cta = (G + gx - 1) / gx;
    // q8_1 output: every CTA owns whole 32-row blocks of y and keeps their fp32
    // values in shared memory until it quantizes them
    const int64_t n_yblk = (p.M + 31) / 32;
    size_t ybuf = 0;
    if (yq) {
        const int64_t blk_per_cta = (n_yblk + gx - 1) / gx;
        groups_per_cta = blk_per_cta * (32 / rw);
        p.ybuf_rows = static_cast<int>(blk_per_cta * 32);
        p.yq_nb_pad = static_cast<int>((p.M + ROW_PAD - 1) / ROW_PAD * ROW_PAD / QK8_1);
        p.yq_col_bytes = static_cast<int64_t>(p.yq_nb_pad) * Q8_1_BYTES;
        ybuf = align_up(static_cast<size_t>(nc_t) * p.ybuf_rows * 4, 16);
    }
    const bool is_moe = mode == MODE_MOE || mode == MODE_MOE_GATE;
    if (is_moe) {
        // the kernel shares the grid among the experts the ids pick (at most
        // n_potential_experts); at least one CTA per possible expert
        gx = std::max<int64_t>(max_ctas, static_cast<int64_t>(p.n_tokens) * p.top_k + (p.W2 ? 1 : 0));
        groups_per_cta = (G * n_potential_experts + gx - 1) / gx;
    }
    max_wpc = static_cast<int>(std::min<int64_t>(max_wpc, std::max<int64_t>(1, groups_per_cta)));
    if (tu.dec_warps.load() > 0) max_wpc = std::min(max_wpc, tu.dec_warps.load());
    // Budget: by default half of an SM's shared memory, so that the next
    // kernel's CTA fits beside this one and streams its first tiles early --
    // unless that would give some warp more row groups than the whole SM's
    // budget would (more serial work outweighs the overlap).  Warps and stages
    // are fixed from the packed activations alone, so the fp32-input and
    // q8_1-input launches of a shape share one geometry (and produce
    // bit-identical results).
    const size_t st_smem = static_smem(fn);
    const size_t fn_limit = std::min(dev.smem_limit, dev.smem_limit + SMEM_RESERVE - st_smem);
    auto need = [&](int w, int st, size_t act) {
        return act + ybuf + static_cast<size_t>(w) * (st * tb + warp_extra) + 128;
    };
    auto fit = [&](size_t budget, int &w, int &st) {
        w = max_wpc;
        st = stages;
        while (w > 1 && need(w, st, packed) > budget) --w;
        while (st > 1 && need(w, st, packed) > budget) --st;
        // When the staged activations squeeze the rings (many columns of a long
        // row) so that some warp would own two row groups where single-tile
        // rings leave every warp at most one, take the single-tile rings: the
        // busiest warp's serial work halves (Q6_K 4096x14336 at 7-8 columns,
        // 7 groups of 7 tiles per CTA: 34 -> 25-27 us).
        if (st > 1 && !tu.stages.load()) {
            int w1 = max_wpc;
            while (w1 > 1 && need(w1, 1, packed) > budget) --w1;
            const int64_t g2 = (groups_per_cta + w - 1) / w, g1 = (groups_per_cta + w1 - 1) / w1;
            if (g2 == 2 && g1 == 1) {
                w = w1;
                st = 1;
            }
        }
        return need(w, st, packed) <= budget;
    };
    auto share_budget = [&](int share) {
        return std::min(fn_limit, dev.smem_per_sm / share - dev.smem_resv - st_smem);
    };
    int wpc_f = 0, st_f = 0;
    const bool tuned_share = tu.smem_share.load() > 0;
    // The half-SM share only helps if a second CTA fits the SM at all: kernels
    // whose registers allow one CTA per SM (more than one column) take it whole
    const bool one_cta = occupancy(dev.dev, fn, cta_warps * 32, 0) < 2;
    size_t budget = share_budget(tuned_share ? tu.smem_share.load() : (one_cta ? 1 : 2));
    if (!fit(budget, wpc_f, st_f)) {
        budget = fn_limit;
        if (!fit(budget, wpc_f, st_f))
            return mma ? plan_tiles(type, mode, dev, p, nc_t, n_potential_experts, L, false) : TilePlan::NoFit;
    } else if (!tuned_share && !is_moe) {
        int wpc_1 = 0, st_1 = 0;
        const int64_t gpc = (G + gx - 1) / gx;  // most row groups a CTA owns
        if (fit(fn_limit, wpc_1, st_1) && (gpc + wpc_1 - 1) / wpc_1 < (gpc + wpc_f - 1) / wpc_f) {
            budget = fn_limit;
            wpc_f = wpc_1;
            st_f = st_1;
        }
    }
    max_wpc = wpc_f;
    stages = st_f;
    // the raw copy of the q8_1 blocks (coalesced staging) only if it still fits;
    // fp32 input is quantized straight into the packed layout
    size_t act = packed;
    if (p.xf == nullptr && !mma && need(max_wpc, stages, packed + raw) <= budget) act = packed + raw;
    const size_t act_staged = act;  // the q8_1 output's row buffer follows the staged activations
    act += ybuf;
    const int wpc = max_wpc;
    const size_t smem = need(wpc, stages, act_staged);  // need() adds the row buffer
    if (ensure_smem_attr(dev, fn) != QMV_OK) return TilePlan::Error;
    if (occupancy(dev.dev, fn, cta_warps * 32, smem) <= 0) return TilePlan::Error;
    // fp32 input: clusters of CTAs share the quantization of the activations
    // (the grid becomes a whole number of clusters; CTAs without row groups
    // still take their share); one CTA per cluster if no such cluster fits
    // The tensor-core decode shares its staging (a conversion of every block of
    // every column) the same way, from q8_1 input too.
    int cl = 1;
    if ((p.xf != nullptr || mma) && (mode == MODE_PLAIN || mode == MODE_GATE)) {
        cl = tu.cluster.load() ? tu.cluster.load() : F32_CLUSTER;
        cl = std::max(1, std::min(MAX_CLUSTER, cl));
        if (cl > 1) {
            const int64_t gx_cl = (gx + cl - 1) / cl * cl;
            if (cluster_occupancy(dev.dev, fn, cta_warps * 32, smem, cl) > 0) gx = gx_cl;
            else cl = 1;
        }
    }
    p.fault = dev.fault;
    p.units_per_row = U;
    p.n_groups = G;
    p.stages = stages;
    p.dec_warps = wpc;
    // Tiles each warp requests before the dependency wait: all of its ring when
    // the ring holds all of its tiles, else one.  Every tile requested early
    // lands ahead of this kernel's activations and of the previous kernel's
    // staging on the SM's return path; a warp with more tiles than its ring
    // refills as soon as its activations are staged, which keeps the stream
    // going for less delay (measured on GB300: qkv, gate/up and down launches
    // 1.5-3 % faster, the 4096x4096 launch, two tiles per warp, slower).
    const int64_t tiles_per_warp =
        (groups_per_cta + wpc - 1) / wpc * ((U + 32 / rw - 1) / (32 / rw)) *
        ((mode == MODE_GATE || mode == MODE_MOE_GATE) ? 2 : 1);
    // Held-back early requests (see the kernel): where the next kernel's CTA
    // can sit beside this one, and either every warp requests all of its
    // tiles early or the activations are fp32, the early requests wait a few
    // hundred ns after the CTA starts, so that the neighbour's activation
    // loads reach the memory system first.  Measured on GB300:
    // - whole matrix early (q8_1 input), EARLY_DELAY_NS: 4096x4096 Q4_K
    //   chained 3.59 -> 3.00 us per call, no launch slower; on launches that
    //   stream more than their rings hold (q8_1 input) 14336x4096 and Q6_K
    //   4096x14336 went 1-5 % slower, so those keep none;
    // - fp32 input, EARLY_DELAY_F32_NS, and then every warp requests its
    //   whole ring early: their neighbours are mostly fp32-input launches,
    //   whose activation loads (4x the bytes, quantized on arrival) gain most
    //   from going first.  The step 0.996 -> 0.990 ms with the hold-back of
    //   400 ns and one early tile per warp, 0.981 with the whole ring, 0.976
    //   to 0.979 with the whole ring and 700 ns (500: 0.978, 900: 0.980, 1200:
    //   0.988; the whole ring without the hold-back: slower).
    const bool beside = !is_moe && occupancy(dev.dev, fn, cta_warps * 32, smem) >= 2;
    const bool hold_f32 = beside && p.xf != nullptr && tu.early_delay_ns.load() >= 0;
    p.pre_tiles = tu.pre_tiles.load() > 0 ? std::min(stages, tu.pre_tiles.load())
                                          : ((tiles_per_warp <= stages || hold_f32) ? stages : 1);
    p.early_warps = tu.early_warps.load() > 0 ? tu.early_warps.load() : wpc;
    p.early_delay = 0;
    if (beside && (tiles_per_warp <= p.pre_tiles || p.xf != nullptr) && tu.early_delay_ns.load() >= 0) {
        const int ns = tu.early_delay_ns.load() > 0 ? tu.early_delay_ns.load()
                       : p.xf != nullptr              ? EARLY_DELAY_F32_NS
                                                      : EARLY_DELAY_NS;
        p.early_delay = static_cast<int>(static_cast<int64_t>(ns) * dev.clock_khz / 1000000);
    }
    p.act_bytes = static_cast<uint32_t>(act);
    p.raw_off = act_staged > packed ? static_cast<uint32_t>(packed) : 0u;
    p.ybuf_off = static_cast<uint32_t>(act_staged);
    L.fn = fn;
    L.probe = yq ? gemv_tiles_yq_fn(type, mode, true) : (!mma && rw == 4) ? gemv_tiles_probe_fn(type, mode, nc_t) : nullptr;
    L.stream = true;
    L.rw = rw;
    L.cluster = cl;
    L.p = p;
    L.block = dim3(static_cast<unsigned>(cta_warps * 32));
    L.grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, gx)));
    L.smem = smem;
    return TilePlan::Ok;
}

// Host checks of the fused fp32-input path (before any CUDA call): the tile
// kernel only (Q4_0 / Q4_K: K % 256 == 0; Q6_K: K % 2048 == 0), 16-byte aligned
// weights.
qmv_status check_f32(int type, const void *W, const void *W2, int64_t K, int64_t ldx)
{
    if (K % (type == FMT_Q6_K ? 2048 : 256) != 0 || ldx < K) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(W) % 16 != 0 || (W2 && reinterpret_cast<uintptr_t>(W2) % 16 != 0))
        return QMV_ERR_ALIGN;
    return QMV_OK;
}

qmv_status plan_f32(int type, int mode, const DevInfo &dev, GemvParams p, int nc_active, int n_potential_experts,
                    Launch &L)
{
    const int nc_t = (mode == MODE_PLAIN) ? nc_active : round_nc(nc_active);
    if (!tile_shape_ok(type, p.K, p.row_bytes)) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(p.W) % 16 != 0 ||
        (mode == MODE_GATE && reinterpret_cast<uintptr_t>(p.W2) % 16 != 0) ||
        (mode == MODE_MOE_GATE && reinterpret_cast<uintptr_t>(p.W3) % 16 != 0))
        return QMV_ERR_ALIGN;
    switch (plan_tiles(type, mode, dev, p, nc_t, n_potential_experts, L)) {
    case TilePlan::Ok: return QMV_OK;
    case TilePlan::NoFit: return QMV_ERR_SHAPE;
    default: return QMV_ERR_CUDA;
    }
}

qmv_status plan(int type, int mode, const DevInfo &dev, GemvParams p, int nc_active, int n_potential_experts,
                Launch &L)
{
    const int nc_t = (mode == MODE_PLAIN) ? nc_active : round_nc(nc_active);
    if (tile_shape_ok(type, p.K, p.row_bytes) && reinterpret_cast<uintptr_t>(p.W) % 16 == 0 &&
        (mode != MODE_GATE || reinterpret_cast<uintptr_t>(p.W2) % 16 == 0)) {
        const TilePlan tp = plan_tiles(type, mode, dev, p, nc_t, n_potential_experts, L);
        if (tp == TilePlan::Ok) return QMV_OK;
        if (tp == TilePlan::Error) return QMV_ERR_CUDA;
    }
    L.fn = gemv_generic_fn(type, mode);
    if (!L.fn) return QMV_ERR_TYPE;
    L.stream = false;
    L.p = p;
    const int threads = 128;
    const int64_t need = (p.M + 3) / 4;
    int64_t gx = std::min<int64_t>(need, static_cast<int64_t>(dev.num_sms) * 16);
    if (mode == MODE_MOE) gx = std::min<int64_t>(need, std::max<int64_t>(1, dev.num_sms * 16 / n_potential_experts));
    L.block = dim3(threads);
    L.grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, gx)), mode == MODE_MOE ? p.n_expert + 1 : 1);
    L.smem = 0;
    return QMV_OK;
}

qmv_status launch(const Launch &L, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = L.block;
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (g_pdl.load()) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    if (L.cluster > 1) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = static_cast<unsigned>(L.cluster);
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    GemvParams p = L.p;
    const void *fn = L.fn;
    unsigned long long *tb = g_trace_buf.load();
    if (tb && L.probe && L.grid.x <= static_cast<unsigned>(TRACE_MAX_CTAS)) {
        const int64_t k = g_trace_next.fetch_add(1);
        if (k < g_trace_slots.load()) {
            DevInfo dev;
            qmv_status s = device_info(dev);
            if (s == QMV_OK) s = ensure_smem_attr(dev, L.probe);
            if (s != QMV_OK) return s;
            p.trace = tb + k * TRACE_MAX_CTAS * TRACE_WORDS;
            fn = L.probe;
        }
    }
    void *args[1] = {&p};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    return cuda_status(e);
}


// ---- checked mode: byte ranges of the arguments inside device allocations ----
std::atomic<int> g_checked{-1};  // -1: QMV_CHECKED not read yet

bool checked_mode()
{
    int v = g_checked.load();
    if (v < 0) {
        const char *e = getenv("QMV_CHECKED");
        int want = (e && *e && *e != '0') ? 1 : 0, expect = -1;
        g_checked.compare_exchange_strong(expect, want);
        v = g_checked.load();
    }
    return v == 1;
}

// cuMemGetAddressRange, looked up at run time (the library does not link the driver)
using AddrRangeFn = int (*)(unsigned long long *, size_t *, unsigned long long);

AddrRangeFn addr_range_fn()
{
    static const AddrRangeFn f = [] {
        void *fp = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fp, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<AddrRangeFn>(nullptr);
        return reinterpret_cast<AddrRangeFn>(fp);
    }();
    return f;
}

// In checked mode [p, p + bytes) must lie inside one device allocation;
// QMV_ERR_RANGE otherwise (also for memory the driver does not know).
qmv_status check_range(const void *p, uint64_t bytes)
{
    if (!checked_mode() || p == nullptr || bytes == 0) return QMV_OK;
    const AddrRangeFn f = addr_range_fn();
    if (!f) return QMV_ERR_CUDA;
    unsigned long long base = 0;
    size_t size = 0;
    const unsigned long long a = reinterpret_cast<unsigned long long>(p);
    if (f(&base, &size, a) != 0 || a < base) return QMV_ERR_RANGE;
    const unsigned long long off = a - base;
    if (off > size || bytes > size - off) return QMV_ERR_RANGE;
    return QMV_OK;
}

#define QMV_RANGE(ptr, nbytes)                                          \
    do {                                                                \
        const qmv_status r_ = check_range((ptr), (nbytes));             \
        if (r_ != QMV_OK) return r_;                                    \
    } while (0)

// bytes of ncols fp32 columns of K values, column stride ldx
uint64_t f32_cols_bytes(int64_t K, int ncols, int64_t ldx)
{
    return (static_cast<uint64_t>(ncols - 1) * static_cast<uint64_t>(ldx) + static_cast<uint64_t>(K)) * 4u;
}

qmv_status check_common(int type, const void *W, int64_t M, int64_t K, const void *xq, const void *out)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (!W || !xq || !out) return QMV_ERR_NULL;
    if (M <= 0 || K <= 0 || K % block_elems(type) != 0) return QMV_ERR_SHAPE;
    if (K > (int64_t(1) << 28) || M > (int64_t(1) << 40)) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(W) % 2 || reinterpret_cast<uintptr_t>(xq) % 4 ||
        reinterpret_cast<uintptr_t>(out) % 4)
        return QMV_ERR_ALIGN;
    return QMV_OK;
}

// Checked mode: the byte ranges a GEMV-family call reads and writes.  n_mat
// weight matrices of M rows each; ncols activation columns (q8_1 from xq, or
// fp32 from x with column stride ldx); y_elems fp32 outputs.
qmv_status check_gemv_ranges(int type, int64_t M, int64_t K, const void *const *Ws, int n_W, int64_t n_mat,
                             const void *xq, const float *x, int64_t ldx, int ncols, const void *y, uint64_t y_elems)
{
    if (!checked_mode()) return QMV_OK;
    const uint64_t w_bytes = static_cast<uint64_t>(n_mat) * static_cast<uint64_t>(M) * qmv_row_bytes(type, K);
    for (int i = 0; i < n_W; ++i) QMV_RANGE(Ws[i], w_bytes);
    QMV_RANGE(xq, qmv_q8_1_bytes(K, ncols));
    QMV_RANGE(x, f32_cols_bytes(K, ncols, ldx));
    QMV_RANGE(y, y_elems * 4u);
    return QMV_OK;
}

GemvParams base_params(int type, const void *W, int64_t M, int64_t K, const void *xq, int ncols)
{
    GemvParams p{};
    p.W = static_cast<const uint8_t *>(W);
    p.xq = static_cast<const uint8_t *>(xq);
    p.M = M;
    p.ldy = M;
    p.K = static_cast<int>(K);
    p.ncols = ncols;
    p.row_bytes = K / block_elems(type) * block_bytes(type);
    p.xq_col_bytes = (K + ROW_PAD - 1) / ROW_PAD * ROW_PAD / QK8_1 * Q8_1_BYTES;
    return p;
}

}  // namespace
}  // namespace qmv

using namespace qmv;

extern "C" {

const char *qmv_status_str(int s)
{
    switch (s) {
    case QMV_OK: return "ok";
    case QMV_ERR_NULL: return "null pointer";
    case QMV_ERR_TYPE: return "unsupported type";
    case QMV_ERR_SHAPE: return "bad shape";
    case QMV_ERR_NCOLS: return "ncols out of range";
    case QMV_ERR_ALIGN: return "misaligned pointer";
    case QMV_ERR_CUDA: return "CUDA error";
    case QMV_ERR_IDS: return "invalid expert id";
    case QMV_ERR_DEVICE_FAULT: return "device wait timed out";
    case QMV_ERR_RANGE: return "argument outside its device allocation";
    case QMV_ERR_CONFIG: return "malformed or out-of-range QMV_GEOM override";
    default: return "unknown status";
    }
}

int qmv_version(void) { return 10000; }

size_t qmv_row_bytes(int type, int64_t K)
{
    if (!weight_type(type) || K <= 0 || K % block_elems(type)) return 0;
    return static_cast<size_t>(K / block_elems(type) * block_bytes(type));
}

int64_t qmv_q8_1_padded_k(int64_t K) { return K <= 0 ? 0 : (K + ROW_PAD - 1) / ROW_PAD * ROW_PAD; }

size_t qmv_q8_1_bytes(int64_t K, int ncols)
{
    if (K <= 0 || ncols <= 0) return 0;
    return static_cast<size_t>(ncols) * static_cast<size_t>(qmv_q8_1_padded_k(K) / QK8_1 * Q8_1_BYTES);
}

qmv_status qmv_quantize_q8_1(const float *x, int64_t K, int ncols, int64_t ldx, void *xq, void *stream)
{
    if (!x || !xq) return QMV_ERR_NULL;
    if (K <= 0 || ncols <= 0 || ldx < K || K > (int64_t(1) << 28)) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(xq) % 4) return QMV_ERR_ALIGN;
    QMV_RANGE(x, f32_cols_bytes(K, ncols, ldx));
    QMV_RANGE(xq, qmv_q8_1_bytes(K, ncols));
    return cuda_status(launch_quantize_q8_1(x, K, ncols, ldx, static_cast<uint8_t *>(xq),
                                            static_cast<cudaStream_t>(stream), g_pdl.load() != 0));
}

qmv_status qmv_quantize_weights(int type, const float *w, int64_t M, int64_t K, int64_t ldw, void *W, void *stream)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (!w || !W) return QMV_ERR_NULL;
    if (M <= 0 || K <= 0 || K % block_elems(type) || ldw < K) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(w) % 4 || reinterpret_cast<uintptr_t>(W) % 2) return QMV_ERR_ALIGN;
    QMV_RANGE(w, static_cast<uint64_t>(M - 1) * static_cast<uint64_t>(ldw) * 4u + static_cast<uint64_t>(K) * 4u);
    QMV_RANGE(W, static_cast<uint64_t>(M) * qmv_row_bytes(type, K));
    return cuda_status(launch_quantize_weights(type, w, M, K, ldw, static_cast<uint8_t *>(W),
                                               static_cast<int64_t>(qmv_row_bytes(type, K)),
                                               static_cast<cudaStream_t>(stream)));
}

qmv_status qmv_mul_mat_vec(int type, const void *W, int64_t M, int64_t K, const void *xq, int ncols, float *y,
                           void *stream)
{
    qmv_status s = check_common(type, W, M, K, xq, y);
    if (s != QMV_OK) return s;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, 1, xq, nullptr, 0, ncols, y, uint64_t(ncols) * M)) != QMV_OK)
        return s;
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, xq, ncols);
    p.y = y;
    Launch L;
    if ((s = plan(type, MODE_PLAIN, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_gate_up_swiglu(int type, const void *W_gate, const void *W_up, int64_t M, int64_t K,
                                          const void *xq, int ncols, float *y, void *stream)
{
    qmv_status s = check_common(type, W_up, M, K, xq, y);
    if (s != QMV_OK) return s;
    if (!W_gate) return QMV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(W_gate) % 2) return QMV_ERR_ALIGN;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    {
        const void *Ws[2] = {W_up, W_gate};
        if ((s = check_gemv_ranges(type, M, K, Ws, 2, 1, xq, nullptr, 0, ncols, y, uint64_t(ncols) * M)) != QMV_OK)
            return s;
    }
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W_up, M, K, xq, ncols);
    p.W2 = static_cast<const uint8_t *>(W_gate);
    p.y = y;
    Launch L;
    if ((s = plan(type, MODE_GATE, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_id(int type, const void *W, int64_t n_expert, int64_t M, int64_t K, const void *xq,
                              const int32_t *ids, int n_tokens, int top_k, float *y, int32_t *dev_status, void *stream)
{
    qmv_status s = check_common(type, W, M, K, xq, y);
    if (s != QMV_OK) return s;
    if (!ids) return QMV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(ids) % 4 || reinterpret_cast<uintptr_t>(dev_status) % 4) return QMV_ERR_ALIGN;
    if (n_tokens < 1 || n_tokens > 8) return QMV_ERR_NCOLS;
    if (top_k < 1 || top_k > 32 || n_expert < 1 || n_expert > MAX_EXPERTS) return QMV_ERR_SHAPE;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, n_expert, xq, nullptr, 0, n_tokens, y,
                               uint64_t(n_tokens) * top_k * M)) != QMV_OK)
        return s;
    QMV_RANGE(ids, uint64_t(n_tokens) * top_k * 4u);
    QMV_RANGE(dev_status, 4u);
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, xq, n_tokens);
    p.y = y;
    p.ids = ids;
    p.status = dev_status;
    p.n_tokens = n_tokens;
    p.top_k = top_k;
    p.n_expert = static_cast<int>(n_expert);
    p.expert_bytes = M * p.row_bytes;
    const int potential = static_cast<int>(std::min<int64_t>(n_expert, static_cast<int64_t>(n_tokens) * top_k));
    Launch L;
    if ((s = plan(type, MODE_MOE, dev, p, n_tokens, potential, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_f32(int type, const void *W, int64_t M, int64_t K, const float *x, int64_t ldx, int ncols,
                               float *y, void *stream)
{
    qmv_status s = check_common(type, W, M, K, x, y);
    if (s != QMV_OK) return s;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    if ((s = check_f32(type, W, nullptr, K, ldx)) != QMV_OK) return s;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, 1, nullptr, x, ldx, ncols, y, uint64_t(ncols) * M)) != QMV_OK)
        return s;
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, nullptr, ncols);
    p.xf = x;
    p.ldx = ldx;
    p.y = y;
    Launch L;
    if ((s = plan_f32(type, MODE_PLAIN, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_debug_f32_withheld_share(int type, const void *W, int64_t M, int64_t K, const float *x, int64_t ldx,
                                        int ncols, float *y, uint64_t wait_ns, void *stream)
{
    qmv_status s = check_common(type, W, M, K, x, y);
    if (s != QMV_OK) return s;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    if (wait_ns < 1 || wait_ns > WAIT_LIMIT_NS) return QMV_ERR_SHAPE;
    if ((s = check_f32(type, W, nullptr, K, ldx)) != QMV_OK) return s;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, 1, nullptr, x, ldx, ncols, y, uint64_t(ncols) * M)) != QMV_OK)
        return s;
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, nullptr, ncols);
    p.xf = x;
    p.ldx = ldx;
    p.y = y;
    Launch L;
    if ((s = plan_f32(type, MODE_PLAIN, dev, p, ncols, 1, L)) != QMV_OK) return s;
    if (L.cluster < 2 || !L.probe) return QMV_ERR_CONFIG;
    if ((s = ensure_smem_attr(dev, L.probe)) != QMV_OK) return s;
    L.fn = L.probe;
    L.probe = nullptr;  // not traced: the timeline is of the ordinary launches
    L.p.withhold = 1;
    L.p.withhold_wait_ns = wait_ns;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_debug_f32_withheld_share_q8_1(int type, const void *W, int64_t M, int64_t K, const float *x, float *y,
                                             void *yq, uint64_t wait_ns, void *stream)
{
    qmv_status s = check_common(type, W, M, K, x, y ? static_cast<void *>(y) : yq);
    if (s != QMV_OK) return s;
    if (!yq) return QMV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(yq) % 4) return QMV_ERR_ALIGN;
    if (wait_ns < 1 || wait_ns > WAIT_LIMIT_NS) return QMV_ERR_SHAPE;
    if (M > (int64_t(1) << 31)) return QMV_ERR_SHAPE;
    if ((s = check_f32(type, W, nullptr, K, K)) != QMV_OK) return s;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, 1, nullptr, x, K, 1, y, y ? uint64_t(M) : 0u)) != QMV_OK) return s;
    QMV_RANGE(yq, qmv_q8_1_bytes(M, 1));
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, nullptr, 1);
    p.xf = x;
    p.ldx = K;
    p.y = y;
    p.yq = static_cast<uint8_t *>(yq);
    Launch L;
    if ((s = plan_f32(type, MODE_PLAIN, dev, p, 1, 1, L)) != QMV_OK) return s;
    if (L.cluster < 2 || !L.probe) return QMV_ERR_CONFIG;
    if ((s = ensure_smem_attr(dev, L.probe)) != QMV_OK) return s;
    L.fn = L.probe;
    L.probe = nullptr;
    L.p.withhold = 1;
    L.p.withhold_wait_ns = wait_ns;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_gate_up_swiglu_f32(int type, const void *W_gate, const void *W_up, int64_t M, int64_t K,
                                              const float *x, int64_t ldx, int ncols, float *y, void *stream)
{
    qmv_status s = check_common(type, W_up, M, K, x, y);
    if (s != QMV_OK) return s;
    if (!W_gate) return QMV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(W_gate) % 2) return QMV_ERR_ALIGN;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    if ((s = check_f32(type, W_up, W_gate, K, ldx)) != QMV_OK) return s;
    {
        const void *Ws[2] = {W_up, W_gate};
        if ((s = check_gemv_ranges(type, M, K, Ws, 2, 1, nullptr, x, ldx, ncols, y, uint64_t(ncols) * M)) != QMV_OK)
            return s;
    }
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W_up, M, K, nullptr, ncols);
    p.W2 = static_cast<const uint8_t *>(W_gate);
    p.xf = x;
    p.ldx = ldx;
    p.y = y;
    Launch L;
    if ((s = plan_f32(type, MODE_GATE, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_id_f32(int type, const void *W, int64_t n_expert, int64_t M, int64_t K, const float *x,
                                  int64_t ldx, const int32_t *ids, int n_tokens, int top_k, float *y, int32_t *dev_status,
                                  void *stream)
{
    qmv_status s = check_common(type, W, M, K, x, y);
    if (s != QMV_OK) return s;
    if (!ids) return QMV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(ids) % 4 || reinterpret_cast<uintptr_t>(dev_status) % 4) return QMV_ERR_ALIGN;
    if (n_tokens < 1 || n_tokens > 8) return QMV_ERR_NCOLS;
    if (top_k < 1 || top_k > 32 || n_expert < 1 || n_expert > MAX_EXPERTS) return QMV_ERR_SHAPE;
    if ((s = check_f32(type, W, nullptr, K, ldx)) != QMV_OK) return s;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, n_expert, nullptr, x, ldx, n_tokens, y,
                               uint64_t(n_tokens) * top_k * M)) != QMV_OK)
        return s;
    QMV_RANGE(ids, uint64_t(n_tokens) * top_k * 4u);
    QMV_RANGE(dev_status, 4u);
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, nullptr, n_tokens);
    p.xf = x;
    p.ldx = ldx;
    p.y = y;
    p.ids = ids;
    p.status = dev_status;
    p.n_tokens = n_tokens;
    p.top_k = top_k;
    p.n_expert = static_cast<int>(n_expert);
    p.expert_bytes = M * p.row_bytes;
    const int potential = static_cast<int>(std::min<int64_t>(n_expert, static_cast<int64_t>(n_tokens) * top_k));
    Launch L;
    if ((s = plan_f32(type, MODE_MOE, dev, p, n_tokens, potential, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_fused(int type, const void *W_up, const void *W_gate, int64_t M, int64_t K, const void *xq,
                                 const float *x, int64_t ldx, int ncols, const float *bias, const float *gate_bias, float *y,
                                 void *stream)
{
    if (!xq && !x) return QMV_ERR_NULL;
    if (xq && x) return QMV_ERR_SHAPE;
    qmv_status s = check_common(type, W_up, M, K, xq ? xq : static_cast<const void *>(x), y);
    if (s != QMV_OK) return s;
    if (gate_bias && !W_gate) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(bias) % 4 || reinterpret_cast<uintptr_t>(gate_bias) % 4) return QMV_ERR_ALIGN;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    if ((s = check_f32(type, W_up, W_gate, K, x ? ldx : K)) != QMV_OK) return s;
    {
        const void *Ws[2] = {W_up, W_gate};
        if ((s = check_gemv_ranges(type, M, K, Ws, W_gate ? 2 : 1, 1, xq, x, ldx, ncols, y, uint64_t(ncols) * M)) !=
            QMV_OK)
            return s;
    }
    QMV_RANGE(bias, uint64_t(M) * 4u);
    QMV_RANGE(gate_bias, uint64_t(M) * 4u);
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W_up, M, K, xq, ncols);
    if (x) {
        p.xf = x;
        p.ldx = ldx;
    }
    p.W2 = static_cast<const uint8_t *>(W_gate);
    p.bias = bias;
    p.gate_bias = gate_bias;
    p.y = y;
    Launch L;
    if ((s = plan_f32(type, W_gate ? MODE_GATE : MODE_PLAIN, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_fused_q8_1(int type, const void *W_up, const void *W_gate, int64_t M, int64_t K,
                                      const void *xq, const float *x, int64_t ldx, int ncols, const float *bias,
                                      const float *gate_bias, float *y, void *yq, void *stream)
{
    if (!xq && !x) return QMV_ERR_NULL;
    if (xq && x) return QMV_ERR_SHAPE;
    if (!yq) return QMV_ERR_NULL;
    qmv_status s = check_common(type, W_up, M, K, xq ? xq : static_cast<const void *>(x), y ? y : yq);
    if (s != QMV_OK) return s;
    if (reinterpret_cast<uintptr_t>(yq) % 4) return QMV_ERR_ALIGN;
    if (gate_bias && !W_gate) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(bias) % 4 || reinterpret_cast<uintptr_t>(gate_bias) % 4) return QMV_ERR_ALIGN;
    if (ncols != 1) return QMV_ERR_NCOLS;
    if (M > (int64_t(1) << 31)) return QMV_ERR_SHAPE;
    if ((s = check_f32(type, W_up, W_gate, K, x ? ldx : K)) != QMV_OK) return s;
    {
        const void *Ws[2] = {W_up, W_gate};
        if ((s = check_gemv_ranges(type, M, K, Ws, W_gate ? 2 : 1, 1, xq, x, ldx, ncols, y, y ? uint64_t(M) : 0u)) !=
            QMV_OK)
            return s;
    }
    QMV_RANGE(bias, uint64_t(M) * 4u);
    QMV_RANGE(gate_bias, uint64_t(M) * 4u);
    QMV_RANGE(yq, qmv_q8_1_bytes(M, 1));
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W_up, M, K, xq, ncols);
    if (x) {
        p.xf = x;
        p.ldx = ldx;
    }
    p.W2 = static_cast<const uint8_t *>(W_gate);
    p.bias = bias;
    p.gate_bias = gate_bias;
    p.y = y;
    p.yq = static_cast<uint8_t *>(yq);
    Launch L;
    if ((s = plan_f32(type, W_gate ? MODE_GATE : MODE_PLAIN, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_mul_mat_vec_id_fused(int type, const void *W_up, const void *W_gate, int64_t n_expert, int64_t M, int64_t K,
                                    const void *xq, const float *x, int64_t ldx, const int32_t *ids, int n_tokens, int top_k,
                                    float *y, const void *W_shared_up, const void *W_shared_gate, float *y_shared,
                                    int32_t *dev_status, void *stream)
{
    if (!xq && !x) return QMV_ERR_NULL;
    if (xq && x) return QMV_ERR_SHAPE;
    qmv_status s = check_common(type, W_up, M, K, xq ? xq : static_cast<const void *>(x), y);
    if (s != QMV_OK) return s;
    if (!ids) return QMV_ERR_NULL;
    if (!W_shared_up != !y_shared) return QMV_ERR_NULL;
    // a gated launch gates the shared expert too, a plain one does not
    if (W_shared_up && (!W_gate != !W_shared_gate)) return QMV_ERR_NULL;
    if (!W_shared_up && W_shared_gate) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(ids) % 4 || reinterpret_cast<uintptr_t>(dev_status) % 4 ||
        reinterpret_cast<uintptr_t>(y_shared) % 4)
        return QMV_ERR_ALIGN;
    if (n_tokens < 1 || n_tokens > 8) return QMV_ERR_NCOLS;
    if (top_k < 1 || top_k > 32 || n_expert < 1 || n_expert > MAX_EXPERTS) return QMV_ERR_SHAPE;
    if ((s = check_f32(type, W_up, W_gate, K, x ? ldx : K)) != QMV_OK) return s;
    if ((s = check_f32(type, W_shared_up, W_shared_gate, K, x ? ldx : K)) != QMV_OK) return s;
    {
        const void *Ws[2] = {W_up, W_gate};
        if ((s = check_gemv_ranges(type, M, K, Ws, W_gate ? 2 : 1, n_expert, xq, x, ldx, n_tokens, y,
                                   uint64_t(n_tokens) * top_k * M)) != QMV_OK)
            return s;
        const void *Ss[2] = {W_shared_up, W_shared_gate};
        if ((s = check_gemv_ranges(type, M, K, Ss, 2, 1, nullptr, nullptr, 0, n_tokens, y_shared,
                                   uint64_t(n_tokens) * M)) != QMV_OK)
            return s;
    }
    QMV_RANGE(ids, uint64_t(n_tokens) * top_k * 4u);
    QMV_RANGE(dev_status, 4u);
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W_up, M, K, xq, n_tokens);
    if (x) {
        p.xf = x;
        p.ldx = ldx;
    }
    p.W2 = static_cast<const uint8_t *>(W_shared_up);
    p.W3 = static_cast<const uint8_t *>(W_gate);
    p.W4 = static_cast<const uint8_t *>(W_shared_gate);
    p.y_shared = y_shared;
    p.y = y;
    p.ids = ids;
    p.status = dev_status;
    p.n_tokens = n_tokens;
    p.top_k = top_k;
    p.n_expert = static_cast<int>(n_expert);
    p.expert_bytes = M * p.row_bytes;
    const int potential = static_cast<int>(std::min<int64_t>(n_expert, static_cast<int64_t>(n_tokens) * top_k)) +
                          (W_shared_up ? 1 : 0);
    Launch L;
    if ((s = plan_f32(type, W_gate ? MODE_MOE_GATE : MODE_MOE, dev, p, n_tokens, potential, L)) != QMV_OK) return s;
    return launch(L, static_cast<cudaStream_t>(stream));
}

qmv_status qmv_debug_subblock_sums(int type, const void *W, int64_t M, int64_t K, const void *xq, int ncols, int32_t *out,
                                   void *stream)
{
    qmv_status s = check_common(type, W, M, K, xq, out);
    if (s != QMV_OK) return s;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    const int64_t per_row = (type == FMT_Q4_0) ? K / 32 : K / 16;
    if ((s = check_gemv_ranges(type, M, K, &W, 1, 1, xq, nullptr, 0, ncols, out, uint64_t(ncols) * M * per_row)) !=
        QMV_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(out, 0, static_cast<size_t>(ncols) * M * per_row * sizeof(int32_t), st) != cudaSuccess)
        return QMV_ERR_CUDA;
    GemvParams p = base_params(type, W, M, K, xq, ncols);
    p.dbg = out;
    Launch L;
    if ((s = plan(type, MODE_DEBUG, dev, p, ncols, 1, L)) != QMV_OK) return s;
    return launch(L, st);
}

qmv_status qmv_device_fault(unsigned int *code)
{
    if (!code) return QMV_ERR_NULL;
    DevInfo dev;
    qmv_status s = device_info(dev);
    if (s != QMV_OK) return s;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpy(&v, dev.fault, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return QMV_ERR_CUDA;
    if (cudaMemcpy(dev.fault, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return QMV_ERR_CUDA;
    *code = v;
    return QMV_OK;
}

qmv_status qmv_set_tuning(int type, int threads, int slice_units, int stages, int ctas_per_sm, int smem_share, int cluster)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (threads < 0 || threads > TILE_MAX_THREADS || threads % 32 || slice_units < 0 || stages < 0 || stages > 16 ||
        ctas_per_sm < 0 || smem_share < 0 || smem_share > 4 || cluster < 0 || cluster > MAX_CLUSTER)
        return QMV_ERR_SHAPE;
    Tuning &t = g_tuning[tidx(type)];
    t.threads = threads;
    t.slice_units = slice_units;
    t.stages = stages;
    t.ctas_per_sm = ctas_per_sm;
    t.smem_share = smem_share;
    t.cluster = cluster;
    return QMV_OK;
}

qmv_status qmv_set_stream_tuning(int type, int dec_warps, int pre_tiles)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (dec_warps < 0 || dec_warps > TILE_MAX_THREADS / 32 || pre_tiles < 0 || pre_tiles > TILE_MAX_STAGES)
        return QMV_ERR_SHAPE;
    Tuning &t = g_tuning[tidx(type)];
    t.dec_warps = dec_warps;
    t.pre_tiles = pre_tiles;
    return QMV_OK;
}

qmv_status qmv_read_bandwidth_probe(const void *buf, size_t bytes, unsigned int *sink, void *stream)
{
    if (!buf || !sink) return QMV_ERR_NULL;
    if (bytes == 0 || bytes % 16) return QMV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(buf) % 16 || reinterpret_cast<uintptr_t>(sink) % 4) return QMV_ERR_ALIGN;
    QMV_RANGE(buf, bytes);
    QMV_RANGE(sink, 4u);
    DevInfo dev;
    qmv_status s = device_info(dev);
    if (s != QMV_OK) return s;
    return cuda_status(launch_read_probe(buf, static_cast<int64_t>(bytes), sink, dev.num_sms,
                                         static_cast<cudaStream_t>(stream)));
}

qmv_status qmv_describe_gemv(int type, int gate_up, int64_t M, int64_t K, int ncols, int fp32_input, qmv_launch_info *info)
{
    if (!info) return QMV_ERR_NULL;
    *info = qmv_launch_info{};
    // stand-in addresses, 256-byte aligned: only their alignment is looked at
    const void *W = reinterpret_cast<const void *>(uintptr_t(1) << 20);
    const void *W2 = reinterpret_cast<const void *>(uintptr_t(2) << 20);
    const void *act = reinterpret_cast<const void *>(uintptr_t(3) << 20);
    float *y = reinterpret_cast<float *>(uintptr_t(4) << 20);
    qmv_status s = check_common(type, W, M, K, act, y);
    if (s != QMV_OK) return s;
    if (ncols < 1 || ncols > 8) return QMV_ERR_NCOLS;
    if (fp32_input && (s = check_f32(type, W, gate_up ? W2 : nullptr, K, K)) != QMV_OK) return s;
    DevInfo dev;
    if ((s = device_info(dev)) != QMV_OK) return s;
    GemvParams p = base_params(type, W, M, K, fp32_input ? nullptr : act, ncols);
    if (fp32_input) {
        p.xf = static_cast<const float *>(act);
        p.ldx = K;
    }
    if (gate_up) p.W2 = static_cast<const uint8_t *>(W2);
    p.y = y;
    const int mode = gate_up ? MODE_GATE : MODE_PLAIN;
    Launch L;
    s = fp32_input ? plan_f32(type, mode, dev, p, ncols, 1, L) : plan(type, mode, dev, p, ncols, 1, L);
    if (s != QMV_OK) return s;
    info->tile_kernel = L.stream ? 1 : 0;
    info->tensor_cores = (L.stream && type == FMT_Q4_K && L.fn == gemv_tiles_mma_fn_q4_K(mode)) ? 1 : 0;
    info->rows_per_tile = L.stream ? L.rw : 0;
    info->grid = static_cast<int>(L.grid.x * L.grid.y);
    info->block = static_cast<int>(L.block.x);
    info->cluster = L.cluster;
    info->stages = L.stream ? L.p.stages : 0;
    info->dec_warps = L.stream ? L.p.dec_warps : 0;
    info->pre_tiles = L.stream ? L.p.pre_tiles : 0;
    info->smem = L.smem;
    return QMV_OK;
}

qmv_status qmv_set_early_warps(int type, int early_warps)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (early_warps < 0 || early_warps > TILE_MAX_THREADS / 32) return QMV_ERR_SHAPE;
    g_tuning[tidx(type)].early_warps = early_warps;
    return QMV_OK;
}

qmv_status qmv_set_early_delay(int type, int ns)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (ns < -1 || ns > 100000) return QMV_ERR_SHAPE;
    g_tuning[tidx(type)].early_delay_ns = ns;
    return QMV_OK;
}

qmv_status qmv_set_mma_min_cols(int type, int min_cols)
{
    if (!weight_type(type)) return QMV_ERR_TYPE;
    if (min_cols < 0 || min_cols > 9) return QMV_ERR_SHAPE;
    g_tuning[tidx(type)].mma_min_cols = min_cols;
    return QMV_OK;
}

qmv_status qmv_debug_trace(unsigned long long *buf, int64_t slots)
{
    if (slots < 0) return QMV_ERR_SHAPE;
    if (buf && reinterpret_cast<uintptr_t>(buf) % 8) return QMV_ERR_ALIGN;
    g_trace_buf = nullptr;
    g_trace_slots = buf ? slots : 0;
    g_trace_next = 0;
    g_trace_buf = slots ? buf : nullptr;
    return QMV_OK;
}

qmv_status qmv_set_pdl(int enable)
{
    g_pdl = enable ? 1 : 0;
    return QMV_OK;
}

qmv_status qmv_set_checked(int enable)
{
    g_checked = enable ? 1 : 0;
    return QMV_OK;
}

}  // extern "C"
