// api.cu -- the C ABI declared in include/fp8gemm.h: argument validation,
// tile-configuration choice, TMA descriptor encoding and launch.
//
// Source of the launch shape: DeepGEMM fp8_gemm.cuh, Gemm::run (a persistent
// grid of at most one CTA per SM) and the make_2d_tma_*_desc factories (the
// operand and output layouts).  Unlike the page's launcher, nothing here
// aborts: every failure is returned as a status code.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fp8gemm.h"
#include "launch.h"

namespace {

using fp8g::LaunchArgs;
using fp8g::Params;

constexpr int kVersion = 10000;          // 1.0.0
constexpr int kDefaultSms = 152;
constexpr int kMaxDevices = 64;
constexpr long long kMaxDim = 1ll << 30;  // rows, N and K limits (int32-safe indexing)

__device__ int g_error_word;              // sticky device-side error bits, per device

std::atomic<int> g_override_bn{0};
std::atomic<int> g_override_split{0};
// CTA pairs: 0 = automatic choice, 1 = the cta_group::2 pair kernel wherever
// it applies, 2 = clusters of two one-CTA kernels sharing A over DSMEM,
// -1 = never
std::atomic<int> g_override_pair{0};

// FP8G_FORCE_CONFIG="block_n[,split_ctas]" sets the tuning overrides when the
// library loads (the values fp8_gemm_set_override accepts); a malformed value
// is ignored, leaving the automatic choice.
struct EnvOverride {
    EnvOverride()
    {
        const char *v = std::getenv("FP8G_FORCE_CONFIG");
        if (!v || !*v)
            return;
        char *end = nullptr;
        const long bn = std::strtol(v, &end, 10);
        long split = 0;
        if (end == v || (bn != 0 && bn != 128 && bn != 256))
            return;
        if (*end == ',') {
            const char *s = end + 1;
            split = std::strtol(s, &end, 10);
            if (end == s || split < -1000000 || split > 1000000)
                return;
        }
        if (*end != '\0')
            return;
        g_override_bn.store((int)bn);
        g_override_split.store((int)split);
    }
} g_env_override;

// FP8G_PAIR_MODE="-1" | "0" | "1" | "2" sets the CTA-pair choice when the library
// loads (the values fp8_gemm_set_pair_mode accepts); anything else is ignored.
struct EnvPairMode {
    EnvPairMode()
    {
        const char *v = std::getenv("FP8G_PAIR_MODE");
        if (!v)
            return;
        if (!std::strcmp(v, "-1"))
            g_override_pair.store(-1);
        else if (!std::strcmp(v, "0"))
            g_override_pair.store(0);
        else if (!std::strcmp(v, "1"))
            g_override_pair.store(1);
        else if (!std::strcmp(v, "2"))
            g_override_pair.store(2);
    }
} g_env_pair_mode;

// The narrow-slice kernel (plain GEMM, M <= 128): 0 = automatic choice,
// 1 = wherever it applies, -1 = never.  FP8G_NARROW_MODE="-1" | "0" | "1" sets
// it when the library loads (anything else is ignored).
std::atomic<int> g_narrow_mode{0};
struct EnvNarrowMode {
    EnvNarrowMode()
    {
        const char *v = std::getenv("FP8G_NARROW_MODE");
        if (!v)
            return;
        if (!std::strcmp(v, "-1"))
            g_narrow_mode.store(-1);
        else if (!std::strcmp(v, "0"))
            g_narrow_mode.store(0);
        else if (!std::strcmp(v, "1"))
            g_narrow_mode.store(1);
    }
} g_env_narrow_mode;
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};

// ------------------------------------------------------------ device facts

struct DeviceInfo {
    int id = 0;
    int sms = 0;
    int *error_word = nullptr;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

int current_device_info(DeviceInfo &out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return FP8G_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (d.sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return FP8G_ERR_CUDA;
        void *w = nullptr;
        if (cudaGetSymbolAddress(&w, g_error_word) != cudaSuccess)
            return FP8G_ERR_CUDA;
        d.error_word = static_cast<int *>(w);
        d.id = dev;
        d.sms = sms;
    }
    out = d;
    return FP8G_OK;
}

int sms_or_default()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
        return sms;
    cudaGetLastError();  // clear a "no device" error left by the probe
    return kDefaultSms;
}

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A 2-D row-major view: `inner` contiguous elements per row, `outer` rows,
// `row_bytes` between rows; tiles of box_inner x box_outer elements.
// outer == 0 makes a 1-D view of `inner` elements with boxes of box_inner.
// Reads outside the view return zeros.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const cuuint32_t rank = outer ? 2 : 1;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    std::memset(m, 0, sizeof(*m));
    return enc(m, dt, rank, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An e4m3 operand [rows][K] viewed as [K/128][rows][128 B] (K-block stride
// 128 bytes), with boxes of box_rows rows x `depth` K blocks: one copy fills
// `depth` consecutive 128-byte-swizzled K-block tiles (K blocks past the end
// arrive as zeros).
bool make_kblock_map(CUtensorMap *m, const void *base, uint64_t rows, int K, uint32_t box_rows, uint32_t depth)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {128, rows, (cuuint64_t)(K / 128)};
    cuuint64_t strides[2] = {(cuuint64_t)K, 128};
    cuuint32_t box[3] = {128, box_rows, depth};
    cuuint32_t es[3] = {1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Two K blocks per box (the one-CTA kernel's paired stages).
bool make_pair_map(CUtensorMap *m, const void *base, uint64_t rows, int K, uint32_t box_rows)
{
    return make_kblock_map(m, base, rows, K, box_rows, 2);
}

// The fp32 addend C [rows][N] viewed as [N/16][rows][16] (slab stride 64
// bytes), with boxes of 4 slabs x 32 rows, 64-byte swizzled: one copy brings
// 32 rows x 64 columns of C into one epilogue warp's staging area.
bool make_c_map(CUtensorMap *m, const float *C, uint64_t rows, int N)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {16, rows, (cuuint64_t)(N / 16)};
    cuuint64_t strides[2] = {(cuuint64_t)N * 4, 64};
    cuuint32_t box[3] = {16, 32, 4};
    cuuint32_t es[3] = {1, 1, 1};
    std::memset(m, 0, sizeof(*m));
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(C), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ validation

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_common(const void *A, const float *SFA, const void *B, const float *SFB, void *D, long long rows,
                 int N, int K)
{
    if (!A || !SFA || !B || !SFB || !D)
        return FP8G_ERR_INVALID_ARG;
    if (rows < 0 || N < 0 || K <= 0)
        return FP8G_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 16 != 0)
        return FP8G_ERR_UNSUPPORTED;
    if (rows > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16) || !aligned(SFA, 16) || !aligned(SFB, 16))
        return FP8G_ERR_MISALIGNED;
    return FP8G_OK;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

int pick_block_n(int N, bool many_tiles)
{
    const int o = g_override_bn.load();
    if (o)
        return o;
    if (N <= 128)
        return 128;
    return many_tiles ? 256 : 128;
}

size_t split_workspace_bytes(int M, int N, int K, int block_n, int ctas)
{
    const long long tiles = (long long)ceil_div(M, 128) * ceil_div(N, block_n);
    const size_t counters = ((size_t)tiles * 8 * sizeof(int) + 255) / 256 * 256;
    const size_t partials = (size_t)2 * ctas * 128 * block_n * sizeof(float);
    (void)K;
    return counters + partials;
}

struct NtChoice {
    int block_n;
    int split_ctas;   // 0: not split
    int grid;
    int tiles;
    bool narrow = false;   // the narrow-slice kernel (block_n = its slice width)
};

// The narrow-slice kernel's launch shape for M rows: A box height, slice
// width, K parts and work units.
struct NarrowShape {
    int a_rows, block_n, ksplit, slices, units;
};

NarrowShape narrow_shape(int M, int N)
{
    NarrowShape n;
    n.a_rows = M <= 64 ? 64 : 128;
    n.block_n = fp8g::narrow_block_n(n.a_rows);
    n.ksplit = fp8g::narrow_ksplit(n.a_rows);
    n.slices = ceil_div(N, n.block_n);
    n.units = n.slices * n.ksplit;
    return n;
}

// Whether the narrow-slice kernel runs a plain GEMM (no addend) of M x N x K
// on `sms` SMs: asked for (fp8_gemm_set_narrow_mode(1)) with M <= 128 and at
// least 4 K blocks (its copies are up to 4 K blocks deep), or, automatically,
// with at least 8 K blocks (16 with two K parts) when its units keep at least
// half the SMs busy without needing a second round.  Measured on 64 / 128 x
// 7168 x 16384 against the split-K schedule (30.5 / 32.2 us): 96-column
// slices in two K parts, 25.6 / 27.6 us.  A forced tile width or split rules
// it out.
bool want_narrow(int M, int N, int K, int sms)
{
    const int mode = g_narrow_mode.load();
    if (mode < 0 || M > 128 || K / 128 < 4 || g_override_bn.load() != 0 || g_override_split.load() > 0)
        return false;
    const NarrowShape n = narrow_shape(M, N);
    if (mode > 0)
        return true;
    const int cap = n.ksplit == 1 ? sms : (sms & ~1);
    return 2 * n.units >= sms && n.units <= cap && K / 128 >= 8 * n.ksplit;
}

// Tile shape and schedule for a plain GEMM on a device with `sms` SMs.
// workspace_bytes < 0 means "as much as it needs".  With fewer output tiles
// than SMs the K blocks of all tiles are shared evenly over the SMs (split-K)
// with 128-column tiles (6 operand stages keep more of B in flight than the 3
// of 256-column tiles; measured faster on small-M shapes), else 256-column
// ones, whichever workspace fits first.  With allow_narrow (no addend) small
// M may go to the narrow-slice kernel instead (want_narrow).
int choose_nt(int M, int N, int K, int sms, long long workspace_bytes, NtChoice &c, bool allow_narrow = false)
{
    const int mb = ceil_div(M, 128);
    const int kb = K / 128;
    const int obn = g_override_bn.load();
    const int osplit = g_override_split.load();
    if (allow_narrow && want_narrow(M, N, K, sms)) {
        const NarrowShape n = narrow_shape(M, N);
        c.narrow = true;
        c.block_n = n.block_n;
        c.split_ctas = 0;
        c.tiles = n.units;
        // the launch sets the grid (two K parts: whole clusters that fit)
        c.grid = std::min(sms, n.units);
        return FP8G_OK;
    }
    auto tiles_for = [&](int bn) { return mb * ceil_div(N, bn); };
    // the kernel's split arithmetic is 32-bit: units * CTAs must stay below 2^31
    auto fits32 = [&](int bn, long long P) { return (long long)tiles_for(bn) * kb * P < (1ll << 31); };
    auto bytes_ok = [&](int bn, long long P) {
        return workspace_bytes < 0 || (long long)split_workspace_bytes(M, N, K, bn, (int)P) <= workspace_bytes;
    };
    auto set = [&](int bn, int P) {
        c.block_n = bn;
        c.tiles = tiles_for(bn);
        c.split_ctas = P;
        c.grid = P ? P : std::min(sms, c.tiles);
    };
    if (osplit > 0) {
        // every CTA of a split schedule must be resident at once (one CTA per
        // SM): a tile's reducer waits for the partials of the others
        if (osplit > sms)
            return FP8G_ERR_UNSUPPORTED;
        const int bn = obn ? obn : 128;
        const long long P = std::min<long long>(osplit, (long long)tiles_for(bn) * kb);
        if (!fits32(bn, P))
            return FP8G_ERR_UNSUPPORTED;
        if (!bytes_ok(bn, P))
            return FP8G_ERR_WORKSPACE;
        set(bn, (int)P);
        return FP8G_OK;
    }
    if (osplit == 0 && kb >= 8) {
        for (int bn : {128, 256}) {
            if ((obn && bn != obn) || (bn == 256 && N <= 128))
                continue;
            const int t = tiles_for(bn);
            if (t >= sms)
                break;          // enough tiles to fill the SMs: no split
            // at least 4 K blocks per CTA
            const long long P = std::min<long long>(sms, (long long)t * kb / 4);
            if (P > t && fits32(bn, P) && bytes_ok(bn, P)) {
                set(bn, (int)P);
                return FP8G_OK;
            }
        }
    }
    set(pick_block_n(N, (long long)mb * ceil_div(N, 256) >= sms), 0);
    return FP8G_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? FP8G_OK : FP8G_ERR_CUDA; }

void fill_common(Params &p, long long rows, int N, int K, int G, const float *SFA, const float *SFB, void *D,
                 const int *layout, int block_n, const DeviceInfo &dev)
{
    std::memset(&p, 0, sizeof(p));
    p.rows = (int)rows;
    p.N = N;
    p.K = K;
    p.G = G;
    p.kb = K / 128;
    p.nb = ceil_div(N, 128);
    p.sfa_ld = (int)((rows + 3) / 4 * 4);
    p.sfa = SFA;
    p.sfb = SFB;
    p.layout = layout;
    p.d = static_cast<__nv_bfloat16 *>(D);
    p.num_n_blocks = ceil_div(N, block_n);
    p.error_word = dev.error_word;
    p.timeout_ns = g_timeout_ns.load();
    // 2-D view extents (the masked launch paths scale A's and D's by G)
    p.a_box_rows = 128;
    p.a_rows_total = (int)rows;
    p.d_rows_total = (int)rows;
    p.b_rows_total = (int)((long long)G * N);
}

// The TMA swizzle that matches a staging panel's row width (2 bytes a column).
CUtensorMapSwizzle panel_swizzle(int cols)
{
    return cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}

// Operand, output and scale views of one launch.  SFA is viewed as
// [sfa_rows][sfa_ld] fp32 (sfa_rows = K/128, or G*K/128 when masked) and
// loaded 128 rows x kScaleChunk K blocks at a time; SFB as one flat fp32
// vector of G*ceil(N/128)*K/128 values, loaded kScaleChunk + 4 at a time from
// a 16-byte aligned start.
bool make_maps(LaunchArgs &a, const void *A, const float *SFA, const void *B, const float *SFB, void *D,
               long long a_rows, long long b_rows, long long d_rows, long long sfa_rows, int sfa_ld,
               long long sfb_count, int N, int K, int block_n)
{
    const int pc = fp8g::panel_cols_for(block_n);
    return make_map(&a.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, a_rows, K, 128, (uint32_t)a.p.a_box_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&a.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, b_rows, K, 128, block_n,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&a.tmap_d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, d_rows, (uint64_t)N * 2, pc, 32,
                    panel_swizzle(pc)) &&
           make_map(&a.tmap_sfa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SFA, sfa_ld, sfa_rows, (uint64_t)sfa_ld * 4,
                    128, fp8g::kScaleChunk, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(&a.tmap_sfb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SFB, sfb_count, 0, 0, fp8g::kScaleChunk + 4, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE) &&
           (K < 256 ? (std::memset(&a.tmap_a2, 0, sizeof(a.tmap_a2)), std::memset(&a.tmap_b2, 0, sizeof(a.tmap_b2)), true)
                    : (make_pair_map(&a.tmap_a2, A, (uint64_t)a_rows, K, 128) &&
                       make_pair_map(&a.tmap_b2, B, (uint64_t)b_rows, K, (uint32_t)block_n)));
}

// The views of a CTA-pair launch: A boxes of 128 rows (each CTA its half of a
// 256-row pair tile), B boxes of half the pair tile's columns, D panels of
// pair_panel_cols() columns; the scale views are those of make_maps.
bool make_pair_maps(LaunchArgs &a, const void *A, const float *SFA, const void *B, const float *SFB, void *D,
                    long long a_rows, long long b_rows, long long d_rows, long long sfa_rows, int sfa_ld,
                    long long sfb_count, int N, int K, int block_n)
{
    const int pc = fp8g::pair_panel_cols();
    std::memset(&a.tmap_a2, 0, sizeof(a.tmap_a2));
    std::memset(&a.tmap_b2, 0, sizeof(a.tmap_b2));
    return make_map(&a.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, a_rows, K, 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&a.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, b_rows, K, 128, (uint32_t)block_n / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&a.tmap_d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, d_rows, (uint64_t)N * 2, pc, 32,
                    panel_swizzle(pc)) &&
           make_map(&a.tmap_sfa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SFA, sfa_ld, sfa_rows, (uint64_t)sfa_ld * 4,
                    128, fp8g::kScaleChunk, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(&a.tmap_sfb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SFB, sfb_count, 0, 0, fp8g::kScaleChunk + 4, 1,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
}

// The pair tile width: the block_n override when one is set, else 256.
int pair_bn() { return g_override_bn.load() ? g_override_bn.load() : 256; }

// Whether the automatic choice may put the plain GEMM, with or without the
// addend (not split), on CTA pairs: its 256 x 256 pair tiles must cover no
// more than an eighth more of the output than the one-CTA kernel's
// 128 x block_n tiles (M = 384 would compute 512 rows for 384).  Measured at
// 1.9 GHz: 4096 x 7168 x 2048 50.8 -> 49.0 us, 4096 x 24576 x 1536
// 134.7 -> 127.2 us, with the addend 65.5 -> 62.1 us.  The grouped GEMMs
// stay on one CTA (contiguous 512 -> 566 us and masked 53.3 -> 58.6 us on
// pairs: their groups' row blocks fill 256-row tiles less well), and so does
// a launch with a forced block_n.
bool pair_auto_ok(int M, int N, int block_n)
{
    if (g_override_bn.load() != 0)
        return false;     // a forced block_n keeps the one-CTA kernel
    const long long pair_area = (long long)ceil_div(M, 256) * 256 * ceil_div(N, 256) * 256;
    const long long one_area = (long long)ceil_div(M, 128) * 128 * ceil_div(N, block_n) * block_n;
    return pair_area * 8 <= one_area * 9;
}

// Whether an unsplit launch runs on CTA pairs, and over how many pairs.
// `pair_tiles` is the number of 256 x pair_bn() pair tiles the problem has;
// mode 0 takes pairs when `automatic` allows them and there is at least one
// pair tile per resident pair.
bool want_pair(long long pair_tiles, const DeviceInfo &dev, int &pairs, bool automatic)
{
    const int mode = g_override_pair.load();
    if (mode < 0 || mode == 2 || pair_tiles <= 0 || (mode == 0 && !automatic))
        return false;
    pairs = fp8g::max_active_pairs(dev.id, pair_bn());
    if (pairs <= 0)
        return false;
    return mode > 0 || pair_tiles >= pairs;
}

// Whether an unsplit launch runs as clusters of two CTAs sharing A over DSMEM
// (only when asked for: fp8_gemm_set_pair_mode(2)), and over how many
// clusters.  Tiles are 128 x 256; `share_tiles` counts (m-block, pair of
// n-blocks) tiles.
bool want_share(long long share_tiles, const DeviceInfo &dev, int &pairs)
{
    if (g_override_pair.load() != 2 || share_tiles <= 0)
        return false;
    const int obn = g_override_bn.load();
    if (obn != 0 && obn != 256)
        return false;
    pairs = fp8g::max_active_share_pairs(dev.id);
    return pairs > 0;
}

int share_n_pairs(int N) { return (ceil_div(N, 256) + 1) / 2; }

// The plain GEMM as A-sharing clusters (no split, no addend).
int run_nt_share(const void *A, const float *SFA, const void *B, const float *SFB, void *D, int M, int N, int K,
                 int pairs, const DeviceInfo &dev, fp8g_stream_t stream)
{
    LaunchArgs a;
    fill_common(a.p, M, N, K, 1, SFA, SFB, D, nullptr, 256, dev);
    a.p.num_m_blocks = ceil_div(M, 128);
    a.p.group_m = 8;
    a.p.num_tiles = a.p.num_m_blocks * share_n_pairs(N);
    if (!make_maps(a, A, SFA, B, SFB, D, M, N, M, a.p.kb, a.p.sfa_ld, (long long)a.p.nb * a.p.kb, N, K, 256))
        return FP8G_ERR_CUDA;
    a.grid = 2 * std::min(pairs, a.p.num_tiles);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return to_status(fp8g::launch_share(fp8g::kKindNT, a));
}

// The plain GEMM on CTA pairs (no split), with or without the addend C.
int run_nt_pair(const void *A, const float *SFA, const void *B, const float *SFB, const float *C, void *D, int M,
                int N, int K, int pairs, const DeviceInfo &dev, fp8g_stream_t stream)
{
    const int bn = pair_bn();
    LaunchArgs a;
    fill_common(a.p, M, N, K, 1, SFA, SFB, D, nullptr, bn, dev);
    a.p.c = C;
    a.p.num_m_blocks = ceil_div(M, 256);
    a.p.group_m = 8;
    a.p.num_tiles = a.p.num_m_blocks * a.p.num_n_blocks;
    if (!make_pair_maps(a, A, SFA, B, SFB, D, M, N, M, a.p.kb, a.p.sfa_ld, (long long)a.p.nb * a.p.kb, N, K, bn))
        return FP8G_ERR_CUDA;
    // 256-column tiles copy the addend through the staging area by TMA
    if (C && bn == 256 && !make_c_map(&a.tmap_c, C, (uint64_t)M, N))
        return FP8G_ERR_CUDA;
    a.grid = 2 * std::min(pairs, a.p.num_tiles);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return to_status(fp8g::launch_pair(C ? fp8g::kKindNTAcc : fp8g::kKindNT, bn, a));
}

// The plain GEMM (M <= 128, no addend) on the narrow-slice kernel.
int run_nt_narrow(const void *A, const float *SFA, const void *B, const float *SFB, void *D, int M, int N, int K,
                  const NtChoice &c, const DeviceInfo &dev, fp8g_stream_t stream)
{
    const NarrowShape n = narrow_shape(M, N);
    LaunchArgs a;
    fill_common(a.p, M, N, K, 1, SFA, SFB, D, nullptr, c.block_n, dev);
    a.p.a_box_rows = n.a_rows;    // with M <= 64 rows past M are never stored: load only the first 64
    a.p.num_m_blocks = 1;
    a.p.num_tiles = c.tiles;
    int grid = c.grid;
    if (n.ksplit == 2) {
        // clusters of two that are all resident at once; an even grid keeps
        // both CTAs of a slice in the same round
        const int clusters = fp8g::narrow_max_clusters(dev.id, n.a_rows);
        if (clusters <= 0)
            return FP8G_ERR_CUDA;
        grid = std::min(n.units, 2 * clusters);
    }
    const uint32_t kd = (uint32_t)fp8g::narrow_kd(a.p.a_box_rows);
    std::memset(&a.tmap_d, 0, sizeof(a.tmap_d));
    std::memset(&a.tmap_a2, 0, sizeof(a.tmap_a2));
    std::memset(&a.tmap_b2, 0, sizeof(a.tmap_b2));
    if (!make_kblock_map(&a.tmap_a, A, (uint64_t)M, K, (uint32_t)a.p.a_box_rows, kd) ||
        !make_kblock_map(&a.tmap_b, B, (uint64_t)N, K, (uint32_t)c.block_n, kd) ||
        !make_map(&a.tmap_sfa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SFA, a.p.sfa_ld, a.p.kb, (uint64_t)a.p.sfa_ld * 4,
                  128, (uint32_t)fp8g::narrow_scale_chunk(), CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&a.tmap_sfb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, SFB, (uint64_t)a.p.nb * a.p.kb, 0, 0,
                  (uint32_t)fp8g::narrow_scale_chunk() + 4, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return FP8G_ERR_CUDA;
    a.grid = grid;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return to_status(fp8g::launch_narrow(a));
}

// The plain GEMM, with or without the fp32 addend C (validated by the caller).
int run_nt(const void *A, const float *SFA, const void *B, const float *SFB, const float *C, void *D, int M, int N,
           int K, void *workspace, size_t workspace_bytes, fp8g_stream_t stream)
{
    DeviceInfo dev;
    int st;
    if ((st = current_device_info(dev)) != FP8G_OK)
        return st;
    NtChoice c;
    const long long ws = workspace ? (long long)workspace_bytes : 0;
    if ((st = choose_nt(M, N, K, dev.sms, ws, c, C == nullptr)) != FP8G_OK)
        return st;
    if (c.narrow)
        return run_nt_narrow(A, SFA, B, SFB, D, M, N, K, c, dev, stream);
    if (c.split_ctas && !aligned(workspace, 256))
        return FP8G_ERR_MISALIGNED;
    int pairs = 0;
    if (!c.split_ctas && want_pair((long long)ceil_div(M, 256) * ceil_div(N, pair_bn()), dev, pairs,
                                   pair_auto_ok(M, N, c.block_n)))
        return run_nt_pair(A, SFA, B, SFB, C, D, M, N, K, pairs, dev, stream);
    if (!c.split_ctas && !C && want_share((long long)ceil_div(M, 128) * share_n_pairs(N), dev, pairs))
        return run_nt_share(A, SFA, B, SFB, D, M, N, K, pairs, dev, stream);

    LaunchArgs a;
    fill_common(a.p, M, N, K, 1, SFA, SFB, D, nullptr, c.block_n, dev);
    a.p.c = C;
    a.p.a_box_rows = M <= 64 ? 64 : 128;    // rows past M are never stored: load only the first 64
    a.p.num_m_blocks = ceil_div(M, 128);
    a.p.group_m = 8;
    a.p.num_tiles = c.tiles;
    if (c.split_ctas) {
        a.p.units = c.tiles * a.p.kb;
        const size_t counters = ((size_t)c.tiles * 8 * sizeof(int) + 255) / 256 * 256;
        a.p.counters = static_cast<int *>(workspace);
        a.p.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + counters);
    }
    if (!make_maps(a, A, SFA, B, SFB, D, M, N, M, a.p.kb, a.p.sfa_ld, (long long)a.p.nb * a.p.kb, N, K,
                   c.block_n))
        return FP8G_ERR_CUDA;
    // the accumulate kernel with whole-tile staging copies C by TMA (unsplit)
    if (C && c.block_n == 256 && !c.split_ctas && !make_c_map(&a.tmap_c, C, (uint64_t)M, N))
        return FP8G_ERR_CUDA;
    a.grid = c.grid;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return to_status(C ? fp8g::launch_nt_acc(c.block_n, c.split_ctas != 0, a)
                       : fp8g::launch_nt(c.block_n, c.split_ctas != 0, a));
}

}  // namespace

// ============================================================================ C ABI

extern "C" {

int fp8_gemm_nt(const void *A, const float *SFA, const void *B, const float *SFB, void *D, int M, int N, int K,
                void *workspace, size_t workspace_bytes, fp8g_stream_t stream)
{
    int st = check_common(A, SFA, B, SFB, D, M, N, K);
    if (st != FP8G_OK)
        return st;
    if (M == 0 || N == 0)
        return FP8G_OK;
    return run_nt(A, SFA, B, SFB, nullptr, D, M, N, K, workspace, workspace_bytes, stream);
}

int fp8_gemm_nt_accumulate(const void *A, const float *SFA, const void *B, const float *SFB, const float *C,
                           void *D, int M, int N, int K, void *workspace, size_t workspace_bytes,
                           fp8g_stream_t stream)
{
    int st = check_common(A, SFA, B, SFB, D, M, N, K);
    if (st != FP8G_OK)
        return st;
    if (!C)
        return FP8G_ERR_INVALID_ARG;
    if (!aligned(C, 16))
        return FP8G_ERR_MISALIGNED;
    if (M == 0 || N == 0)
        return FP8G_OK;
    // the kernel reads C through the read-only path while other CTAs write D
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(C), c1 = c0 + (uintptr_t)M * N * 4;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(D), d1 = d0 + (uintptr_t)M * N * 2;
    if (c0 < d1 && d0 < c1)
        return FP8G_ERR_INVALID_ARG;
    return run_nt(A, SFA, B, SFB, C, D, M, N, K, workspace, workspace_bytes, stream);
}

int fp8_gemm_grouped_contiguous(const void *A, const float *SFA, const void *B, const float *SFB, void *D,
                                const int *m_indices, int M_total, int N, int K, int G, void *workspace,
                                size_t workspace_bytes, fp8g_stream_t stream)
{
    (void)workspace;
    (void)workspace_bytes;
    int st = check_common(A, SFA, B, SFB, D, M_total, N, K);
    if (st != FP8G_OK)
        return st;
    if (!m_indices || G <= 0)
        return FP8G_ERR_INVALID_ARG;
    if (!aligned(m_indices, 4))
        return FP8G_ERR_MISALIGNED;
    if (M_total % 128 != 0 || (long long)G * N > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    if (M_total == 0 || N == 0)
        return FP8G_OK;
    DeviceInfo dev;
    if ((st = current_device_info(dev)) != FP8G_OK)
        return st;
    int pairs = 0;
    if (want_pair((long long)ceil_div(M_total, 256) * ceil_div(N, pair_bn()), dev, pairs, false)) {
        const int bn = pair_bn();
        LaunchArgs a;
        fill_common(a.p, M_total, N, K, G, SFA, SFB, D, m_indices, bn, dev);
        a.p.num_m_blocks = ceil_div(M_total, 256);
        a.p.group_m = 8;
        const int pair_tiles = a.p.num_m_blocks * a.p.num_n_blocks;
        a.p.num_tiles = 2 * pair_tiles;     // two passes (see the pair scheduler)
        if (!make_pair_maps(a, A, SFA, B, SFB, D, M_total, (long long)G * N, M_total, a.p.kb, a.p.sfa_ld,
                            (long long)G * a.p.nb * a.p.kb, N, K, bn))
            return FP8G_ERR_CUDA;
        a.grid = 2 * std::min(pairs, pair_tiles);
        a.stream = reinterpret_cast<cudaStream_t>(stream);
        return to_status(fp8g::launch_pair(fp8g::kKindContiguous, bn, a));
    }
    if (want_share((long long)(M_total / 128) * share_n_pairs(N), dev, pairs)) {
        LaunchArgs a;
        fill_common(a.p, M_total, N, K, G, SFA, SFB, D, m_indices, 256, dev);
        a.p.num_m_blocks = M_total / 128;
        a.p.group_m = 8;
        a.p.num_tiles = a.p.num_m_blocks * share_n_pairs(N);
        if (!make_maps(a, A, SFA, B, SFB, D, M_total, (long long)G * N, M_total, a.p.kb, a.p.sfa_ld,
                       (long long)G * a.p.nb * a.p.kb, N, K, 256))
            return FP8G_ERR_CUDA;
        a.grid = 2 * std::min(pairs, a.p.num_tiles);
        a.stream = reinterpret_cast<cudaStream_t>(stream);
        return to_status(fp8g::launch_share(fp8g::kKindContiguous, a));
    }
    const int mb = M_total / 128;
    const int block_n = pick_block_n(N, (long long)mb * ceil_div(N, 256) >= dev.sms);
    LaunchArgs a;
    fill_common(a.p, M_total, N, K, G, SFA, SFB, D, m_indices, block_n, dev);
    a.p.num_m_blocks = mb;
    a.p.group_m = 8;
    a.p.num_tiles = mb * a.p.num_n_blocks;
    if (!make_maps(a, A, SFA, B, SFB, D, M_total, (long long)G * N, M_total, a.p.kb, a.p.sfa_ld,
                   (long long)G * a.p.nb * a.p.kb, N, K, block_n))
        return FP8G_ERR_CUDA;
    a.grid = std::min(dev.sms, a.p.num_tiles);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return to_status(fp8g::launch_contiguous(block_n, a));
}

int fp8_gemm_grouped_masked(const void *A, const float *SFA, const void *B, const float *SFB, void *D,
                            const int *masked_m, int G, int M_max, int N, int K, void *workspace,
                            size_t workspace_bytes, fp8g_stream_t stream)
{
    (void)workspace;
    (void)workspace_bytes;
    int st = check_common(A, SFA, B, SFB, D, M_max, N, K);
    if (st != FP8G_OK)
        return st;
    if (!masked_m || G <= 0)
        return FP8G_ERR_INVALID_ARG;
    if (!aligned(masked_m, 4))
        return FP8G_ERR_MISALIGNED;
    if ((long long)G * M_max > kMaxDim || (long long)G * N > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    if (M_max == 0 || N == 0)
        return FP8G_OK;
    DeviceInfo dev;
    if ((st = current_device_info(dev)) != FP8G_OK)
        return st;
    int pairs = 0;
    if (want_pair((long long)G * ceil_div(M_max, 256) * ceil_div(N, pair_bn()), dev, pairs, false)) {
        const int bn = pair_bn();
        LaunchArgs a;
        fill_common(a.p, M_max, N, K, G, SFA, SFB, D, masked_m, bn, dev);
        a.p.a_rows_total = a.p.d_rows_total = (int)((long long)G * M_max);
        a.p.num_m_blocks = ceil_div(M_max, 256);
        a.p.group_m = a.p.num_m_blocks;
        const long long tiles_max = (long long)G * a.p.num_m_blocks * a.p.num_n_blocks;
        if (!make_pair_maps(a, A, SFA, B, SFB, D, (long long)G * M_max, (long long)G * N, (long long)G * M_max,
                            (long long)G * a.p.kb, a.p.sfa_ld, (long long)G * a.p.nb * a.p.kb, N, K, bn))
            return FP8G_ERR_CUDA;
        a.grid = 2 * (int)std::min<long long>(pairs, tiles_max);
        a.stream = reinterpret_cast<cudaStream_t>(stream);
        return to_status(fp8g::launch_pair(fp8g::kKindMasked, bn, a));
    }
    if (want_share((long long)G * ceil_div(M_max, 128) * share_n_pairs(N), dev, pairs)) {
        LaunchArgs a;
        fill_common(a.p, M_max, N, K, G, SFA, SFB, D, masked_m, 256, dev);
        a.p.a_rows_total = a.p.d_rows_total = (int)((long long)G * M_max);
        a.p.num_m_blocks = ceil_div(M_max, 128);
        a.p.group_m = a.p.num_m_blocks;
        const long long tiles_max = (long long)G * a.p.num_m_blocks * share_n_pairs(N);
        if (!make_maps(a, A, SFA, B, SFB, D, (long long)G * M_max, (long long)G * N, (long long)G * M_max,
                       (long long)G * a.p.kb, a.p.sfa_ld, (long long)G * a.p.nb * a.p.kb, N, K, 256))
            return FP8G_ERR_CUDA;
        a.grid = 2 * (int)std::min<long long>(pairs, tiles_max);
        a.stream = reinterpret_cast<cudaStream_t>(stream);
        return to_status(fp8g::launch_share(fp8g::kKindMasked, a));
    }
    const int mb = ceil_div(M_max, 128);
    const long long tiles_max256 = (long long)G * mb * ceil_div(N, 256);
    const int block_n = pick_block_n(N, tiles_max256 >= dev.sms);
    LaunchArgs a;
    fill_common(a.p, M_max, N, K, G, SFA, SFB, D, masked_m, block_n, dev);
    a.p.a_rows_total = a.p.d_rows_total = (int)((long long)G * M_max);
    a.p.num_m_blocks = mb;
    a.p.group_m = mb;   // all m-blocks of a (group, n-block) run together: B is read once
    const long long tiles_max = (long long)G * mb * a.p.num_n_blocks;
    if (!make_maps(a, A, SFA, B, SFB, D, (long long)G * M_max, (long long)G * N, (long long)G * M_max,
                   (long long)G * a.p.kb, a.p.sfa_ld, (long long)G * a.p.nb * a.p.kb, N, K, block_n))
        return FP8G_ERR_CUDA;
    a.grid = (int)std::min<long long>(dev.sms, tiles_max);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    return to_status(fp8g::launch_masked(block_n, a));
}

int fp8_gemm_nt_ue8m0(const void *A, const void *SFA_e, const void *B, const void *SFB_e, void *D, int M, int N,
                      int K, fp8g_stream_t stream)
{
    if (!A || !SFA_e || !B || !SFB_e || !D)
        return FP8G_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K <= 0)
        return FP8G_ERR_INVALID_ARG;
    if (K % 128 != 0 || N % 16 != 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8G_ERR_UNSUPPORTED;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 16))
        return FP8G_ERR_MISALIGNED;
    if (M == 0 || N == 0)
        return FP8G_OK;
    DeviceInfo dev;
    int st;
    if ((st = current_device_info(dev)) != FP8G_OK)
        return st;
    // CTA pairs (256 x 256 tiles): with fp8_gemm_set_pair_mode(1), and by
    // default once there are two 128-row blocks (4096 x 7168 x 2048: 46.3 ->
    // 44.2 us; 4096 x 24576 x 1536: 126.7 -> 117.1 us); never with mode -1
    // or 2.  With one row block the pair's second CTA would have no rows.
    const int mode = g_override_pair.load();
    const bool want = mode == 1 || (mode == 0 && M > 128);
    const int pairs = want ? fp8g::ue8m0_pair_max_active(dev.id) : 0;
    const bool pair = pairs > 0;
    const int bn = pair ? fp8g::ue8m0_pair_block_n() : fp8g::ue8m0_block_n();
    LaunchArgs a;
    fill_common(a.p, M, N, K, 1, nullptr, nullptr, D, nullptr, bn, dev);
    a.p.sfa_e = static_cast<const uint8_t *>(SFA_e);
    a.p.sfb_e = static_cast<const uint8_t *>(SFB_e);
    a.p.num_m_blocks = ceil_div(M, pair ? 256 : 128);
    a.p.group_m = pair ? 4 : 8;
    a.p.num_tiles = a.p.num_m_blocks * a.p.num_n_blocks;
    const int pc = fp8g::ue8m0_panel_cols();
    std::memset(&a.tmap_sfa, 0, sizeof(a.tmap_sfa));
    std::memset(&a.tmap_sfb, 0, sizeof(a.tmap_sfb));
    std::memset(&a.tmap_a2, 0, sizeof(a.tmap_a2));
    std::memset(&a.tmap_b2, 0, sizeof(a.tmap_b2));
    if (!make_map(&a.tmap_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, K, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&a.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, K, 128, (uint32_t)(pair ? bn / 2 : bn),
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&a.tmap_d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, M, (uint64_t)N * 2, pc, 32, panel_swizzle(pc)))
        return FP8G_ERR_CUDA;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    if (pair) {
        a.grid = 2 * std::min(pairs, a.p.num_tiles);
        return to_status(fp8g::launch_ue8m0_pair(a));
    }
    a.grid = std::min(dev.sms, a.p.num_tiles);
    return to_status(fp8g::launch_ue8m0(a));
}

size_t fp8_gemm_workspace_size(int kind, int M, int N, int K, int G)
{
    (void)G;
    if (kind != FP8G_KIND_NT || M <= 0 || N <= 0 || K <= 0 || K % 128 != 0)
        return 0;
    // the split-K schedule's (fp8_gemm_nt_accumulate never runs the
    // narrow-slice kernel, and that kernel needs none)
    NtChoice c;
    if (choose_nt(M, N, K, sms_or_default(), -1, c) != FP8G_OK || !c.split_ctas)
        return 0;
    return split_workspace_bytes(M, N, K, c.block_n, c.split_ctas);
}

size_t fp8_gemm_workspace_size_for(int M, int N, int K, int block_n, int split_ctas)
{
    if (M <= 0 || N <= 0 || K <= 0 || split_ctas <= 0 || (block_n != 128 && block_n != 256))
        return 0;
    return split_workspace_bytes(M, N, K, block_n, split_ctas);
}

int fp8_gemm_get_device_error(fp8g_stream_t stream)
{
    DeviceInfo dev;
    int st = current_device_info(dev);
    if (st != FP8G_OK)
        return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FP8G_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, dev.error_word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return FP8G_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev.error_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8G_ERR_CUDA;
    }
    if (v & fp8g::kErrBoundsBit)
        return FP8G_ERR_BOUNDS;
    if (v & fp8g::kErrTimeoutBit)
        return FP8G_ERR_TIMEOUT;
    if (v & fp8g::kErrBadGroupBit)
        return FP8G_ERR_BAD_GROUP;
    return FP8G_OK;
}

const char *fp8_gemm_status_string(int status)
{
    switch (status) {
    case FP8G_OK: return "ok";
    case FP8G_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or G <= 0)";
    case FP8G_ERR_UNSUPPORTED: return "unsupported shape (needs K % 128 == 0, N % 16 == 0, M_total % 128 == 0)";
    case FP8G_ERR_MISALIGNED: return "misaligned pointer (A, B, D, SFA, SFB need 16 bytes, workspace 256)";
    case FP8G_ERR_CUDA: return "a CUDA call failed";
    case FP8G_ERR_TIMEOUT: return "a pipeline wait on the device ran out of time";
    case FP8G_ERR_BAD_GROUP: return "a group index or count was out of range";
    case FP8G_ERR_WORKSPACE: return "workspace too small for the forced split";
    case FP8G_ERR_SCRATCH_LIMIT:
        return "problem needs more split-K scratch than fp8_gemm_nt_noalloc's static buffer holds";
    case FP8G_ERR_BOUNDS: return "a device-side bounds check failed (bounds-checking build)";
    default: return "unknown status";
    }
}

int fp8_gemm_sfa_ld(int M) { return M < 0 ? 0 : (M + 3) / 4 * 4; }

int fp8_gemm_set_override(int block_n, int split_ctas)
{
    if (block_n != 0 && block_n != 128 && block_n != 256)
        return FP8G_ERR_INVALID_ARG;
    g_override_bn.store(block_n);
    g_override_split.store(split_ctas);
    return FP8G_OK;
}

int fp8_gemm_set_pair_mode(int mode)
{
    if (mode < -1 || mode > 2)
        return FP8G_ERR_INVALID_ARG;
    g_override_pair.store(mode);
    return FP8G_OK;
}

int fp8_gemm_set_narrow_mode(int mode)
{
    if (mode < -1 || mode > 1)
        return FP8G_ERR_INVALID_ARG;
    g_narrow_mode.store(mode);
    return FP8G_OK;
}

int fp8_gemm_set_wait_timeout_ns(uint64_t ns)
{
    if (ns < 1000000ull)
        return FP8G_ERR_INVALID_ARG;
    g_timeout_ns.store(ns);
    return FP8G_OK;
}

int fp8_gemm_version(void) { return kVersion; }

}  // extern "C"

// ============================================================================
// fp8_gemm_nt_noalloc: the plain GEMM for callers that cannot call cudaMalloc
// (code running inside an allocator callback, plug-ins whose host framework
// owns all device memory, loops that forbid allocation after start-up) and so
// cannot hand over a workspace.  The split-K schedule's scratch (counter
// counters and fp32 partials) lives in the static array below instead.

namespace {

// Largest scratch the split-K schedule may use through fp8_gemm_nt_noalloc.
// It covers the schedule fp8_gemm_nt picks for any plain GEMM on a GPU with
// up to 190 SMs (2 fp32 slots of 128 x 128 per CTA plus the counters).
constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];

// Set-up, once per device, with that device current: the device address of
// the static scratch.  (In host code the array's name is only a host-side
// stand-in; the kernel must be given this address.)
int noalloc_scratch(int dev, void **out)
{
    std::lock_guard<std::mutex> lk(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return FP8G_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return FP8G_OK;
}

}  // namespace

extern "C" int fp8_gemm_nt_noalloc(const void *A, const float *SFA, const void *B, const float *SFB,
                                   void *D, int M, int N, int K, fp8g_stream_t stream)
{
    int st = check_common(A, SFA, B, SFB, D, M, N, K);
    if (st != FP8G_OK)
        return st;
    if (M == 0 || N == 0)
        return FP8G_OK;
    DeviceInfo dev;
    if ((st = current_device_info(dev)) != FP8G_OK)
        return st;
    int dev_id = 0;
    if (cudaGetDevice(&dev_id) != cudaSuccess)
        return FP8G_ERR_CUDA;
    void *scratch = nullptr;
    if ((st = noalloc_scratch(dev_id, &scratch)) != FP8G_OK)
        return st;

    // the schedule fp8_gemm_nt picks when given all the workspace it asks
    // for, or, when that needs more than the static scratch, the best one
    // that fits it; a forced split that does not fit is refused
    NtChoice c;
    if ((st = choose_nt(M, N, K, dev.sms, -1, c, true)) != FP8G_OK)
        return st;
    if (c.narrow)
        return run_nt_narrow(A, SFA, B, SFB, D, M, N, K, c, dev, stream);
    if (c.split_ctas && split_workspace_bytes(M, N, K, c.block_n, c.split_ctas) > kNoAllocScratchBytes) {
        if (g_override_split.load() > 0)
            return FP8G_ERR_SCRATCH_LIMIT;
        if ((st = choose_nt(M, N, K, dev.sms, (long long)kNoAllocScratchBytes, c)) != FP8G_OK)
            return st;
    }
    int pairs = 0;
    if (!c.split_ctas && want_pair((long long)ceil_div(M, 256) * ceil_div(N, pair_bn()), dev, pairs,
                                   pair_auto_ok(M, N, c.block_n)))
        return run_nt_pair(A, SFA, B, SFB, nullptr, D, M, N, K, pairs, dev, stream);
    if (!c.split_ctas && want_share((long long)ceil_div(M, 128) * share_n_pairs(N), dev, pairs))
        return run_nt_share(A, SFA, B, SFB, D, M, N, K, pairs, dev, stream);
    const size_t counters = ((size_t)c.tiles * 8 * sizeof(int) + 255) / 256 * 256;

    LaunchArgs a;
    fill_common(a.p, M, N, K, 1, SFA, SFB, D, nullptr, c.block_n, dev);
    a.p.a_box_rows = M <= 64 ? 64 : 128;    // as fp8_gemm_nt
    a.p.num_m_blocks = ceil_div(M, 128);
    a.p.group_m = 8;
    a.p.num_tiles = c.tiles;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    if (c.split_ctas) {
        a.p.units = c.tiles * a.p.kb;
        a.p.counters = static_cast<int *>(scratch);
        a.p.partials = reinterpret_cast<float *>(static_cast<char *>(scratch) + counters);
        // the array keeps the previous call's contents: the counters start at zero
        if (cudaMemsetAsync(scratch, 0, counters, a.stream) != cudaSuccess)
            return FP8G_ERR_CUDA;
    }
    if (!make_maps(a, A, SFA, B, SFB, D, M, N, M, a.p.kb, a.p.sfa_ld, (long long)a.p.nb * a.p.kb, N, K,
                   c.block_n))
        return FP8G_ERR_CUDA;
    a.grid = c.grid;
    return to_status(fp8g::launch_nt(c.block_n, c.split_ctas != 0, a));
}
