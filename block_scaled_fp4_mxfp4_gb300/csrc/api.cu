// extern "C" entry points of libmxfp4 (declared in include/mxfp4.h): argument
// validation, per-device facts, the TMA descriptor cache, workspace layout and
// path selection. Nothing here allocates device memory or synchronizes.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "internal.h"
#include "mxfp4.h"

using namespace mxfp4;

namespace {

std::atomic<uint64_t> g_wait_limit_ns{kWaitTimeoutNs};

}  // namespace

namespace mxfp4 {

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : kWaitTimeoutNs, std::memory_order_relaxed); }

}  // namespace mxfp4

namespace {

// Split-K and path plans assume this many SMs so that the workspace size is a
// function of the shape alone (GB300 has 152; fewer SMs only change occupancy).
constexpr int kPlanSms = 152;
constexpr int kMaxSplitK = 16;

// --------------------------------------------------------------- device info
struct DevInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

mxfp4_status_t current_device(int *sms)
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return MXFP4_ERR_NO_DEVICE;
    if (d < 0 || d >= 64) return MXFP4_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo &di = g_dev[d];
    if (!di.probed) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
            return MXFP4_ERR_NO_DEVICE;
        di.supported = (major == 10 && minor == 3);
        di.sms = n;
        di.probed = true;
    }
    if (!di.supported) return MXFP4_ERR_NO_DEVICE;
    *sms = di.sms;
    return MXFP4_OK;
}

// ------------------------------------------------------- TMA descriptor cache
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool encoder()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

struct MapKey {
    uintptr_t ptr;
    int64_t inner, rows, stride;
    int box_rows, dev, kind;   // kind 0: packed FP4 (u8, 128B swizzle); 1: scale blocks (u32); 2: C (16-bit)
    bool operator==(const MapKey &o) const
    {
        return ptr == o.ptr && inner == o.inner && rows == o.rows && stride == o.stride &&
               box_rows == o.box_rows && dev == o.dev && kind == o.kind;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        uint64_t h = 1469598103934665603ull;
        auto mix = [&](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
        mix(k.ptr);
        mix(static_cast<uint64_t>(k.inner));
        mix(static_cast<uint64_t>(k.rows));
        mix(static_cast<uint64_t>(k.stride));
        mix(static_cast<uint64_t>(k.box_rows));
        mix(static_cast<uint64_t>(k.dev));
        mix(static_cast<uint64_t>(k.kind));
        return static_cast<size_t>(h);
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

mxfp4_status_t cached_map(const MapKey &key, const void *base, CUtensorMapDataType dtype, cuuint64_t inner,
                          cuuint32_t box_inner, CUtensorMapSwizzle swz, CUtensorMap *out,
                          CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
{
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return MXFP4_OK;
        }
    }
    if (!encoder()) return MXFP4_ERR_CUDA;
    CUtensorMap tm;
    cuuint64_t dims[2] = {inner, static_cast<cuuint64_t>(key.rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(key.stride)};
    cuuint32_t box[2] = {box_inner, static_cast<cuuint32_t>(key.box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = g_encode(&tm, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MXFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 4096) g_maps.clear();
    g_maps.emplace(key, tm);
    *out = tm;
    return MXFP4_OK;
}

// Tensor map of a packed FP4 matrix [rows, inner bytes] (row stride `stride`
// bytes), box {128 bytes, box_rows}, 128-byte swizzle, zero fill out of bounds.
mxfp4_status_t fp4_map(const void *base, int64_t inner, int64_t rows, int64_t stride, int box_rows,
                       CUtensorMap *out)
{
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey key{reinterpret_cast<uintptr_t>(base), inner, rows, stride, box_rows, dev, 0};
    return cached_map(key, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint64_t>(inner), 128u,
                      CU_TENSOR_MAP_SWIZZLE_128B, out);
}

// Tensor map of a blocked scale buffer viewed as [blocks, 128 u32] (one
// 512-byte block per row), box {128, box_blocks}: box_blocks consecutive
// K-blocks of one 128-row chunk in one copy; zero fill past the last block.
mxfp4_status_t sf_map(const void *base, int64_t blocks, int box_blocks, CUtensorMap *out)
{
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey key{reinterpret_cast<uintptr_t>(base), 128, blocks, 512, box_blocks, dev, 1};
    return cached_map(key, base, CU_TENSOR_MAP_DATA_TYPE_UINT32, 128u, 128u, CU_TENSOR_MAP_SWIZZLE_NONE, out);
}

// Tensor map of a 16-bit C [rows, cols] (row stride ld elements) for the
// single-CTA GEMM's TMA-store epilogue: box {32, 32}, 64-byte swizzle. Sets
// *usable = false (and succeeds) when C's base or row stride is not 16-byte
// aligned; the kernel then stores C directly.
mxfp4_status_t c_map(void *C, int64_t cols, int64_t rows, int64_t ld, CUtensorMap *out, bool *usable)
{
    *usable = false;
    if ((reinterpret_cast<uintptr_t>(C) & 15u) != 0 || (ld * 2) % 16 != 0) return MXFP4_OK;
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey key{reinterpret_cast<uintptr_t>(C), cols, rows, ld * 2, 32, dev, 2};
    const mxfp4_status_t st = cached_map(key, C, CU_TENSOR_MAP_DATA_TYPE_UINT16, static_cast<cuuint64_t>(cols), 32u,
                                         CU_TENSOR_MAP_SWIZZLE_64B, out, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (st == MXFP4_OK) *usable = true;
    return st;
}

// ------------------------------------------------------------- validation
inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool al2(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

mxfp4_status_t check_quant(const void *A, int64_t M, int64_t K, int64_t lda, const void *Aq, int64_t ldq,
                           const void *sf, int vec)
{
    if (!A || !Aq || !sf) return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || M > kMaxDim || K > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (K % vec != 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    if (lda < K || ldq < K / 2) return MXFP4_ERR_INVALID_ARG;
    // 16-byte vector loads of A; 4-byte stores of codes and scale words
    if ((lda * 2) % 16 != 0 || ldq % 4 != 0) return MXFP4_ERR_MISALIGNED;
    if (!al16(A) || !al4(Aq) || !al4(sf)) return MXFP4_ERR_MISALIGNED;
    return MXFP4_OK;
}

mxfp4_status_t check_gemm_common(const void *Bq, int64_t ldbq, const void *B_sf, const void *C, int64_t ldc,
                                 int64_t M, int64_t N, int64_t K)
{
    if (!Bq || !B_sf || !C) return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (K % 32 != 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    if (ldbq < K / 2 || ldc < N) return MXFP4_ERR_INVALID_ARG;
    // TMA operands: 16-byte base and row stride; C needs only element alignment
    if (ldbq % 16 != 0) return MXFP4_ERR_MISALIGNED;
    if (!al16(Bq) || !al16(B_sf) || !al2(C)) return MXFP4_ERR_MISALIGNED;
    return MXFP4_OK;
}

inline mxfp4_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA; }

// --------------------------------------------------------- workspace layout
inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

size_t sf_bytes(int64_t rows, int64_t k, int vec)
{
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((k / vec + 3) / 4) * 512;
}

// ------------------------------------------------------- split-K choices
#include "split_table.inc"

// Process-wide tuning override of the K-splits (0: none), per path: 0 the
// two-kernel GEMM, 1 the fused MXFP4 kernel, 2 the fused NVFP4 kernel.
std::atomic<int> g_split_override[3] = {};

int split_bucket(int which, int64_t M)
{
    if (which == 0) return static_cast<int>((M + 127) / 128);
    return M <= 16 ? 16 : M <= 32 ? 32 : 64;
}

// K-splits asked for (M, N, K) on a path: the override, else the measured
// table's entry, else 0 (the shape-derived rule decides).
int split_choice(int which, int64_t M, int64_t N, int64_t K)
{
    const int o = g_split_override[which].load(std::memory_order_relaxed);
    if (o > 0) return o;
    const int b = split_bucket(which, M);
    for (const SplitEntry *e = kSplitTable; e->which >= 0; ++e)
        if (e->which == which && e->bucket == b && e->n == N && e->k == K) return e->splits;
    return 0;
}

struct GemmPlan {
    bool pair;     // CTA-pair kernel (256 x 256 tiles); else single-CTA 128 x bn tiles
    int bn;        // single-CTA tile width along N: 256, or 128 when 256-wide tiles leave
                   // most SMs idle (and the B box rows: 128 for the pair kernel)
    int splits;
    int tiles;
    int n_tiles;
};

// The pair kernel needs at least one 256 x 256 tile per SM pair.
bool use_pair(int64_t pair_tile_count) { return pair_tile_count >= kPlanSms / 2; }

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K)
{
    GemmPlan p;
    if (use_pair(pair_tiles(M, N))) {
        p.pair = true;
        p.bn = 128;
        p.splits = 1;
        p.tiles = pair_tiles(M, N);
        p.n_tiles = static_cast<int>((N + 255) / 256);
        return p;
    }
    p.pair = false;
    const int64_t m_tiles = (M + 127) / 128;
    p.bn = 2 * m_tiles * ((N + 255) / 256) <= kPlanSms ? 128 : 256;
    const int bn = p.bn;
    p.n_tiles = static_cast<int>((N + bn - 1) / bn);
    p.tiles = static_cast<int>(m_tiles * p.n_tiles);
    const int64_t k_stages = (K + 255) / 256;
    // No K-split unless the measured table or an override asks for one: on
    // GB300 one split was the fastest for every shape of the tuning sweep
    // (M 128 / 256, N 512-7168, K 512-7168) and for long-K shapes with few
    // tiles (16 x 640 x 4096, 128 x 2112 x 7168): summing fp32 partial tiles,
    // through the workspace or through a cluster's shared memory (measured
    // too), costs more than the shorter mainloop saves.
    int64_t s = 1;
    const int want = split_choice(0, M, N, K);
    if (want > 0) {
        s = want;
        if (s > kMaxSplitK) s = kMaxSplitK;
        if (s > k_stages) s = k_stages;
        if (s < 1) s = 1;
    }
    p.splits = static_cast<int>(s);
    return p;
}

struct WsLayout {
    size_t aq_off, sf_off, part_off, ticket_off, total;
    int64_t ldq;
};

WsLayout ws_layout(int64_t M, int64_t N, int64_t K)
{
    WsLayout w;
    w.ldq = ((K / 2) + 15) / 16 * 16;
    const GemmPlan gp = plan_gemm(M, N, K);
    const int bn = gp.bn;
    w.aq_off = 0;
    w.sf_off = up256(static_cast<size_t>(M) * w.ldq);
    w.part_off = w.sf_off + up256(sf_bytes(M, K, 32));
    size_t part = 0;
    if (gp.splits > 1) part = static_cast<size_t>(gp.splits) * gp.n_tiles * bn * static_cast<size_t>(M) * 4;
    w.ticket_off = w.part_off + up256(part);
    w.total = w.ticket_off + up256(static_cast<size_t>(gp.tiles) * 4);
    return w;
}

// Optional GEMM epilogue (mxfp4_gemm_a4w4_ex): C = alpha * acc + beta * C + bias.
struct Epilogue {
    bool on;
    float alpha, beta;
    const void *bias;
};
constexpr Epilogue kNoEpilogue{false, 1.0f, 0.0f, nullptr};

mxfp4_status_t run_gemm(const void *Aq, int64_t ldaq, const void *A_sf, const void *Bq, int64_t ldbq,
                        const void *B_sf, void *C, int64_t ldc, int64_t M, int64_t N, int64_t K, void *ws,
                        const WsLayout &wl, cudaStream_t stream, const Epilogue &epi = kNoEpilogue)
{
    GemmProblemHost h;
    memset(&h, 0, sizeof(h));
    h.epi = epi.on;
    h.alpha = epi.alpha;
    h.beta = epi.beta;
    h.bias = epi.bias;
    mxfp4_status_t st = fp4_map(Aq, K / 2, M, ldaq, 128, &h.tma);
    if (st != MXFP4_OK) return st;
    const GemmPlan gp = plan_gemm(M, N, K);
    st = fp4_map(Bq, K / 2, N, ldbq, gp.bn, &h.tmb);
    if (st != MXFP4_OK) return st;
    h.sfa = static_cast<const uint8_t *>(A_sf);
    h.sfb = static_cast<const uint8_t *>(B_sf);
    h.c = C;
    h.ldc = ldc;
    h.m = static_cast<int>(M);
    h.n = static_cast<int>(N);
    h.k = static_cast<int>(K);
    uint8_t *w = static_cast<uint8_t *>(ws);
    float *part = gp.splits > 1 ? reinterpret_cast<float *>(w + wl.part_off) : nullptr;
    int *tickets = reinterpret_cast<int *>(w + wl.ticket_off);
    if (gp.pair) {
        st = sf_map(A_sf, static_cast<int64_t>(sf_bytes(M, K, 32) / 512), 2, &h.tmsfa);
        if (st != MXFP4_OK) return st;
        st = sf_map(B_sf, static_cast<int64_t>(sf_bytes(N, K, 32) / 512), 2, &h.tmsfb);
        if (st != MXFP4_OK) return st;
        return cuda_status(launch_gemm_mx_pair(h, stream));
    }
    if (gp.splits == 1 && !epi.on) {
        st = c_map(C, N, M, ldc, &h.tmc, &h.c_tma);
        if (st != MXFP4_OK) return st;
    }
    return cuda_status(launch_gemm_mx(h, gp.bn, gp.splits, part, tickets, stream));
}

// ------------------------------------------------------------ grouped GEMMs
// nvfp4_group_gemm (E4M3 per 16, fp16 C) and mxfp4_group_gemm (E8M0 per 32,
// bf16 C) share the validation, the tensor maps and the kernel choice. Up to
// kMaxGroups problems travel in kernel parameters; longer lists in a device
// table at the start of the caller's workspace.
constexpr int kMaxGroupsAny = 1 << 20;   // sanity bound on a problem list's length

size_t group_ws_bytes(int num_groups)
{
    return num_groups > kMaxGroups ? group_table_bytes(num_groups) : 0;
}

inline bool al64(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 63u) == 0; }

template <typename Problem>
mxfp4_status_t check_groups(const Problem *problems, int num_groups, int vec, bool pointers, int64_t *tiles,
                            int64_t *pair_tile_count)
{
    if (!problems || num_groups < 1) return MXFP4_ERR_INVALID_ARG;
    if (num_groups > kMaxGroupsAny) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    const int bn = gemm_block_n_nv();
    *tiles = 0;
    *pair_tile_count = 0;
    for (int g = 0; g < num_groups; ++g) {
        const Problem &p = problems[g];
        if (pointers && (!p.a || !p.sfa || !p.b || !p.sfb || !p.c)) return MXFP4_ERR_INVALID_ARG;
        if (p.m < 1 || p.n < 1 || p.k < 1 || p.m > kMaxDim || p.n > kMaxDim || p.k > kMaxDim)
            return MXFP4_ERR_INVALID_ARG;
        if (p.k % vec != 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
        if (pointers) {
            if (p.lda < p.k / 2 || p.ldb < p.k / 2 || p.ldc < p.n) return MXFP4_ERR_INVALID_ARG;
            if (p.lda % 16 != 0 || p.ldb % 16 != 0) return MXFP4_ERR_MISALIGNED;
            if (!al16(p.a) || !al16(p.sfa) || !al16(p.b) || !al16(p.sfb) || !al2(p.c)) return MXFP4_ERR_MISALIGNED;
        }
        *tiles += ((p.m + 127) / 128) * ((p.n + bn - 1) / bn);
        *pair_tile_count += pair_tiles(p.m, p.n);
    }
    if (*tiles > kMaxDim) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    return MXFP4_OK;
}

// `table`: device memory of group_ws_bytes(num_groups) bytes (64-byte
// aligned) for lists longer than kMaxGroups, else unused.
template <typename Problem>
mxfp4_status_t group_gemm(const Problem *problems, int num_groups, bool nv, void *table, size_t table_bytes,
                          void *stream)
{
    const int vec = nv ? 16 : 32;
    int64_t tiles = 0, pair_tile_count = 0;
    mxfp4_status_t st = check_groups(problems, num_groups, vec, true, &tiles, &pair_tile_count);
    if (st != MXFP4_OK) return st;
    if (num_groups > kMaxGroups) {
        if (!table) return MXFP4_ERR_INVALID_ARG;
        if (!al64(table)) return MXFP4_ERR_MISALIGNED;
        if (table_bytes < group_ws_bytes(num_groups)) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
    }
    const bool pair = use_pair(pair_tile_count);
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    std::vector<GemmProblemHost> hp(static_cast<size_t>(num_groups));
    memset(hp.data(), 0, hp.size() * sizeof(GemmProblemHost));
    const int bn = gemm_block_n_nv();
    for (int g = 0; g < num_groups; ++g) {
        const Problem &p = problems[g];
        st = fp4_map(p.a, p.k / 2, p.m, p.lda, 128, &hp[g].tma);
        if (st != MXFP4_OK) return st;
        st = fp4_map(p.b, p.k / 2, p.n, p.ldb, pair ? 128 : bn, &hp[g].tmb);
        if (st != MXFP4_OK) return st;
        if (pair) {
            st = sf_map(p.sfa, static_cast<int64_t>(sf_bytes(p.m, p.k, vec) / 512), pair_sf_box_blocks(nv),
                        &hp[g].tmsfa);
            if (st != MXFP4_OK) return st;
            st = sf_map(p.sfb, static_cast<int64_t>(sf_bytes(p.n, p.k, vec) / 512), pair_sf_box_blocks(nv),
                        &hp[g].tmsfb);
            if (st != MXFP4_OK) return st;
        }
        if (!pair) {
            st = c_map(p.c, p.n, p.m, p.ldc, &hp[g].tmc, &hp[g].c_tma);
            if (st != MXFP4_OK) return st;
        }
        hp[g].sfa = static_cast<const uint8_t *>(p.sfa);
        hp[g].sfb = static_cast<const uint8_t *>(p.sfb);
        hp[g].c = p.c;
        hp[g].ldc = p.ldc;
        hp[g].m = static_cast<int>(p.m);
        hp[g].n = static_cast<int>(p.n);
        hp[g].k = static_cast<int>(p.k);
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (nv)
        return cuda_status(pair ? launch_gemm_nv_grouped_pair(hp.data(), num_groups, table, s)
                                : launch_gemm_nv_grouped(hp.data(), num_groups, table, s));
    return cuda_status(pair ? launch_gemm_mx_grouped_pair(hp.data(), num_groups, table, s)
                            : launch_gemm_mx_grouped(hp.data(), num_groups, table, s));
}

template <typename Problem>
mxfp4_status_t group_gemm_plan(const Problem *problems, int num_groups, bool nv, mxfp4_plan_t *out)
{
    if (!out) return MXFP4_ERR_INVALID_ARG;
    int64_t tiles = 0, pair_tile_count = 0;
    mxfp4_status_t st = check_groups(problems, num_groups, nv ? 16 : 32, false, &tiles, &pair_tile_count);
    if (st != MXFP4_OK) return st;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    memset(out, 0, sizeof(*out));
    const bool pair = use_pair(pair_tile_count);
    out->kernel = pair ? MXFP4_KERNEL_GEMM_PAIR : MXFP4_KERNEL_GEMM;
    out->tile_m = pair ? 256 : 128;
    out->tile_n = pair ? 256 : gemm_block_n_nv();
    out->splits = 1;
    out->tiles = static_cast<int>(pair ? pair_tile_count : tiles);
    out->quant_launch = 0;
    return MXFP4_OK;
}

// nvfp4_group_quant_gemm: validation of the bf16 problem list and the
// workspace layout (per group: packed A with 16-byte rows, then its scales,
// each at a 256-byte offset; then, for lists longer than kMaxGroups, the
// grouped GEMM's problem table).
struct ActWorkspace {
    std::vector<size_t> aq_off, sf_off;
    std::vector<int64_t> ldq;
    size_t table_off, total;
};

mxfp4_status_t check_act_groups(const nvfp4_act_problem_t *problems, int num_groups, bool pointers,
                                ActWorkspace *ws)
{
    if (!problems || num_groups < 1) return MXFP4_ERR_INVALID_ARG;
    if (num_groups > kMaxGroupsAny) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    ws->aq_off.resize(num_groups);
    ws->sf_off.resize(num_groups);
    ws->ldq.resize(num_groups);
    size_t off = 0;
    for (int g = 0; g < num_groups; ++g) {
        const nvfp4_act_problem_t &p = problems[g];
        if (pointers && (!p.a || !p.b || !p.sfb || !p.c)) return MXFP4_ERR_INVALID_ARG;
        if (p.m < 1 || p.n < 1 || p.k < 1 || p.m > kMaxDim || p.n > kMaxDim || p.k > kMaxDim)
            return MXFP4_ERR_INVALID_ARG;
        if (p.k % 16 != 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
        if (pointers) {
            if (p.lda < p.k || p.ldb < p.k / 2 || p.ldc < p.n) return MXFP4_ERR_INVALID_ARG;
            if ((p.lda * 2) % 16 != 0 || p.ldb % 16 != 0) return MXFP4_ERR_MISALIGNED;
            if (!al16(p.a) || !al16(p.b) || !al16(p.sfb) || !al2(p.c)) return MXFP4_ERR_MISALIGNED;
        }
        ws->ldq[g] = (p.k / 2 + 15) / 16 * 16;
        ws->aq_off[g] = off;
        off += up256(static_cast<size_t>(p.m) * static_cast<size_t>(ws->ldq[g]));
        ws->sf_off[g] = off;
        off += up256(sf_bytes(p.m, p.k, 16));
    }
    ws->table_off = off;
    ws->total = off + group_ws_bytes(num_groups);
    return MXFP4_OK;
}

}  // namespace

extern "C" {

const char *mxfp4_status_string(mxfp4_status_t s)
{
    switch (s) {
    case MXFP4_OK: return "MXFP4_OK";
    case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG";
    case MXFP4_ERR_UNSUPPORTED_SHAPE: return "MXFP4_ERR_UNSUPPORTED_SHAPE";
    case MXFP4_ERR_MISALIGNED: return "MXFP4_ERR_MISALIGNED";
    case MXFP4_ERR_WORKSPACE_TOO_SMALL: return "MXFP4_ERR_WORKSPACE_TOO_SMALL";
    case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA";
    case MXFP4_ERR_DEVICE_TIMEOUT: return "MXFP4_ERR_DEVICE_TIMEOUT";
    case MXFP4_ERR_NO_DEVICE: return "MXFP4_ERR_NO_DEVICE";
    }
    return "MXFP4_UNKNOWN_STATUS";
}

int mxfp4_abi_version(void) { return 2; }

size_t mxfp4_sf_bytes(int64_t rows, int64_t k, int vec)
{
    if ((vec != 16 && vec != 32) || rows < 1 || k < 1 || k % vec != 0) return 0;
    return sf_bytes(rows, k, vec);
}

size_t mxfp4_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || N < 1 || K < 1 || K % 32 != 0) return 0;
    return ws_layout(M, N, K).total;
}

size_t nvfp4_group_workspace_bytes(int num_groups)
{
    return num_groups < 1 || num_groups > kMaxGroupsAny ? 0 : group_ws_bytes(num_groups);
}

size_t mxfp4_group_workspace_bytes(int num_groups)
{
    return num_groups < 1 || num_groups > kMaxGroupsAny ? 0 : group_ws_bytes(num_groups);
}

mxfp4_status_t mxfp4_quantize(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq, int64_t ldq,
                              void *A_sf, void *stream)
{
    mxfp4_status_t st = check_quant(A, M, K, lda, Aq, ldq, A_sf, 32);
    if (st != MXFP4_OK) return st;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    return cuda_status(launch_quant_mx(A, M, K, lda, Aq, ldq, A_sf, sms, static_cast<cudaStream_t>(stream)));
}

mxfp4_status_t nvfp4_quantize(const void *A, int64_t M, int64_t K, int64_t lda, void *Aq, int64_t ldq,
                              void *A_sf, void *stream)
{
    mxfp4_status_t st = check_quant(A, M, K, lda, Aq, ldq, A_sf, 16);
    if (st != MXFP4_OK) return st;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    return cuda_status(launch_quant_nv(A, M, K, lda, Aq, ldq, A_sf, sms, static_cast<cudaStream_t>(stream)));
}

mxfp4_status_t mxfp4_gemm_a4w4(const void *Aq, int64_t ldaq, const void *A_sf, const void *Bq, int64_t ldbq,
                               const void *B_sf, void *C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                               void *workspace, size_t ws_bytes, void *stream)
{
    mxfp4_status_t st = check_gemm_common(Bq, ldbq, B_sf, C, ldc, M, N, K);
    if (st != MXFP4_OK) return st;
    if (!Aq || !A_sf || !workspace) return MXFP4_ERR_INVALID_ARG;
    if (ldaq < K / 2) return MXFP4_ERR_INVALID_ARG;
    if (ldaq % 16 != 0 || !al16(Aq) || !al16(A_sf) || !al16(workspace)) return MXFP4_ERR_MISALIGNED;
    const WsLayout wl = ws_layout(M, N, K);
    if (ws_bytes < wl.total) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    return run_gemm(Aq, ldaq, A_sf, Bq, ldbq, B_sf, C, ldc, M, N, K, workspace, wl,
                    static_cast<cudaStream_t>(stream));
}

mxfp4_status_t mxfp4_gemm_a4w4_ex(const void *Aq, int64_t ldaq, const void *A_sf, const void *Bq, int64_t ldbq,
                                  const void *B_sf, void *C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                  float alpha, float beta, const void *bias, void *workspace, size_t ws_bytes,
                                  void *stream)
{
    mxfp4_status_t st = check_gemm_common(Bq, ldbq, B_sf, C, ldc, M, N, K);
    if (st != MXFP4_OK) return st;
    if (!Aq || !A_sf || !workspace) return MXFP4_ERR_INVALID_ARG;
    if (ldaq < K / 2) return MXFP4_ERR_INVALID_ARG;
    if (!std::isfinite(alpha) || !std::isfinite(beta)) return MXFP4_ERR_INVALID_ARG;
    if (ldaq % 16 != 0 || !al16(Aq) || !al16(A_sf) || !al16(workspace)) return MXFP4_ERR_MISALIGNED;
    if (bias && !al2(bias)) return MXFP4_ERR_MISALIGNED;
    const WsLayout wl = ws_layout(M, N, K);
    if (ws_bytes < wl.total) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    const Epilogue epi{!(alpha == 1.0f && beta == 0.0f && bias == nullptr), alpha, beta, bias};
    return run_gemm(Aq, ldaq, A_sf, Bq, ldbq, B_sf, C, ldc, M, N, K, workspace, wl,
                    static_cast<cudaStream_t>(stream), epi);
}

mxfp4_status_t mxfp4_quant_gemm_fused(const void *A, int64_t lda, const void *Bq, int64_t ldbq, const void *B_sf,
                                      void *C, int64_t ldc, int64_t M, int64_t N, int64_t K, void *workspace,
                                      size_t ws_bytes, void *stream)
{
    mxfp4_status_t st = check_gemm_common(Bq, ldbq, B_sf, C, ldc, M, N, K);
    if (st != MXFP4_OK) return st;
    if (!A || !workspace) return MXFP4_ERR_INVALID_ARG;
    if (lda < K) return MXFP4_ERR_INVALID_ARG;
    if ((lda * 2) % 16 != 0 || !al16(A) || !al16(workspace)) return MXFP4_ERR_MISALIGNED;
    const WsLayout wl = ws_layout(M, N, K);
    if (ws_bytes < wl.total) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    FusedPlan fp;
    if (plan_fused(M, N, K, sms, &fp, false, split_choice(1, M, N, K))) {
        CUtensorMap tmw;
        st = fp4_map(Bq, K / 2, N, ldbq, 128, &tmw);
        if (st != MXFP4_OK) return st;
        return cuda_status(launch_fused(tmw, A, lda, static_cast<const uint8_t *>(B_sf), C, ldc,
                                        static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), fp, false, s));
    }
    // two-kernel path: quantize A into the workspace, then the GEMM
    uint8_t *w = static_cast<uint8_t *>(workspace);
    void *aq = w + wl.aq_off;
    void *asf = w + wl.sf_off;
    st = cuda_status(launch_quant_mx(A, M, K, lda, aq, wl.ldq, asf, sms, s, true));
    if (st != MXFP4_OK) return st;
    return run_gemm(aq, wl.ldq, asf, Bq, ldbq, B_sf, C, ldc, M, N, K, workspace, wl, s);
}

mxfp4_status_t nvfp4_quant_gemm_fused(const void *A, int64_t lda, const void *Bq, int64_t ldbq, const void *B_sf,
                                      void *C, int64_t ldc, int64_t M, int64_t N, int64_t K, void *stream)
{
    if (!A || !Bq || !B_sf || !C) return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || N > kMaxDim || K > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (K % 16 != 0 || M > 64) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    if (lda < K || ldbq < K / 2 || ldc < N) return MXFP4_ERR_INVALID_ARG;
    if ((lda * 2) % 16 != 0 || ldbq % 16 != 0) return MXFP4_ERR_MISALIGNED;
    if (!al16(A) || !al16(Bq) || !al16(B_sf) || !al2(C)) return MXFP4_ERR_MISALIGNED;
    int sms = 0;
    mxfp4_status_t st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    FusedPlan fp;
    if (!plan_fused(M, N, K, sms, &fp, true, split_choice(2, M, N, K))) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap tmw;
    st = fp4_map(Bq, K / 2, N, ldbq, 128, &tmw);
    if (st != MXFP4_OK) return st;
    return cuda_status(launch_fused(tmw, A, lda, static_cast<const uint8_t *>(B_sf), C, ldc, static_cast<int>(M),
                                    static_cast<int>(N), static_cast<int>(K), fp, true,
                                    static_cast<cudaStream_t>(stream)));
}

mxfp4_status_t nvfp4_group_gemm(const nvfp4_problem_t *problems, int num_groups, void *workspace, size_t ws_bytes,
                                void *stream)
{
    return group_gemm(problems, num_groups, true, workspace, ws_bytes, stream);
}

mxfp4_status_t mxfp4_rmsnorm_quantize_ex(const void *X, int64_t M, int64_t K, int64_t ldx, const void *weight,
                                         float eps, void *Aq, int64_t ldq, void *A_sf, float *rstd, double *sumsq,
                                         void *stream)
{
    mxfp4_status_t st = check_quant(X, M, K, ldx, Aq, ldq, A_sf, 32);
    if (st != MXFP4_OK) return st;
    if (!weight) return MXFP4_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return MXFP4_ERR_INVALID_ARG;
    if (!al16(weight) || !al4(rstd) || (reinterpret_cast<uintptr_t>(sumsq) & 7u) != 0) return MXFP4_ERR_MISALIGNED;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    return cuda_status(launch_rmsnorm_mx_quant(X, M, K, ldx, weight, eps, Aq, ldq, A_sf, rstd, sumsq, sms,
                                               static_cast<cudaStream_t>(stream)));
}

mxfp4_status_t mxfp4_rmsnorm_quantize(const void *X, int64_t M, int64_t K, int64_t ldx, const void *weight,
                                      float eps, void *Aq, int64_t ldq, void *A_sf, void *stream)
{
    return mxfp4_rmsnorm_quantize_ex(X, M, K, ldx, weight, eps, Aq, ldq, A_sf, nullptr, nullptr, stream);
}

size_t nvfp4_group_quant_gemm_workspace_bytes(const nvfp4_act_problem_t *problems, int num_groups)
{
    ActWorkspace ws;
    return check_act_groups(problems, num_groups, false, &ws) == MXFP4_OK ? ws.total : 0;
}

mxfp4_status_t nvfp4_group_quant_gemm(const nvfp4_act_problem_t *problems, int num_groups, void *workspace,
                                      size_t ws_bytes, void *stream)
{
    ActWorkspace wl;
    mxfp4_status_t st = check_act_groups(problems, num_groups, true, &wl);
    if (st != MXFP4_OK) return st;
    if (!workspace) return MXFP4_ERR_INVALID_ARG;
    if (!al16(workspace)) return MXFP4_ERR_MISALIGNED;
    if (ws_bytes < wl.total) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    std::vector<nvfp4_problem_t> q(static_cast<size_t>(num_groups));
    std::vector<QuantGroupHost> qg(static_cast<size_t>(num_groups));
    for (int g = 0; g < num_groups; ++g) {
        const nvfp4_act_problem_t &p = problems[g];
        q[g].m = p.m;
        q[g].n = p.n;
        q[g].k = p.k;
        q[g].a = w + wl.aq_off[g];
        q[g].sfa = w + wl.sf_off[g];
        q[g].b = p.b;
        q[g].sfb = p.sfb;
        q[g].c = p.c;
        q[g].lda = wl.ldq[g];
        q[g].ldb = p.ldb;
        q[g].ldc = p.ldc;
        qg[g] = QuantGroupHost{p.a, p.m, p.k, p.lda, w + wl.aq_off[g], wl.ldq[g], w + wl.sf_off[g]};
    }
    // the GEMM half's own checks, so that nothing is enqueued on a bad list
    int64_t tiles = 0, pair_tile_count = 0;
    st = check_groups(q.data(), num_groups, 16, true, &tiles, &pair_tile_count);
    if (st != MXFP4_OK) return st;
    if (num_groups > kMaxGroups && !al64(w + wl.table_off)) return MXFP4_ERR_MISALIGNED;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    // one quantization launch per kMaxGroups groups
    for (int g0 = 0; g0 < num_groups; g0 += kMaxGroups) {
        st = cuda_status(launch_quant_nv_grouped(qg.data() + g0, std::min(kMaxGroups, num_groups - g0), sms,
                                                 static_cast<cudaStream_t>(stream), g0 + kMaxGroups >= num_groups));
        if (st != MXFP4_OK) return st;
    }
    return group_gemm(q.data(), num_groups, true, w + wl.table_off, ws_bytes - wl.table_off, stream);
}

mxfp4_status_t mxfp4_group_gemm(const mxfp4_problem_t *problems, int num_groups, void *workspace, size_t ws_bytes,
                                void *stream)
{
    return group_gemm(problems, num_groups, false, workspace, ws_bytes, stream);
}

mxfp4_status_t mxfp4_gemm_plan(int64_t M, int64_t N, int64_t K, int which, mxfp4_plan_t *out)
{
    if (!out || which < 0 || which > 2) return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (K % (which == 2 ? 16 : 32) != 0 || (which == 2 && M > 64)) return MXFP4_ERR_UNSUPPORTED_SHAPE;
    int sms = 0;
    const mxfp4_status_t st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    memset(out, 0, sizeof(*out));
    FusedPlan fp;
    if (which >= 1 && plan_fused(M, N, K, sms, &fp, which == 2, split_choice(which, M, N, K))) {
        out->kernel = MXFP4_KERNEL_FUSED;
        out->tile_m = fp.mma_n;   // activation rows (padded) x 128 weight rows
        out->tile_n = 128;
        out->splits = fp.splits;
        out->tiles = fp.n_tiles;
        out->quant_launch = 0;
        return MXFP4_OK;
    }
    const GemmPlan gp = plan_gemm(M, N, K);
    out->kernel = gp.pair ? MXFP4_KERNEL_GEMM_PAIR : MXFP4_KERNEL_GEMM;
    out->tile_m = gp.pair ? 256 : 128;
    out->tile_n = gp.pair ? 256 : gp.bn;
    out->splits = gp.splits;
    out->tiles = gp.tiles;
    out->quant_launch = which;
    return MXFP4_OK;
}

mxfp4_status_t nvfp4_group_gemm_plan(const nvfp4_problem_t *problems, int num_groups, mxfp4_plan_t *out)
{
    return group_gemm_plan(problems, num_groups, true, out);
}

mxfp4_status_t mxfp4_group_gemm_plan(const mxfp4_problem_t *problems, int num_groups, mxfp4_plan_t *out)
{
    return group_gemm_plan(problems, num_groups, false, out);
}

int mxfp4_set_split_override(int path, int splits)
{
    if (path < 0 || path > 2 || splits < 0) return -1;
    return g_split_override[path].exchange(splits);
}

int mxfp4_split_table_entry(int index, int *path, int *bucket, int64_t *n, int64_t *k, int *splits)
{
    int count = 0;
    while (kSplitTable[count].which >= 0) ++count;
    if (index < 0 || index >= count) return count;
    const SplitEntry &e = kSplitTable[index];
    if (path) *path = e.which;
    if (bucket) *bucket = e.bucket;
    if (n) *n = e.n;
    if (k) *k = e.k;
    if (splits) *splits = e.splits;
    return count;
}

uint64_t mxfp4_set_wait_limit_ns(uint64_t ns)
{
    const uint64_t old = wait_limit_ns();
    set_wait_limit_ns(ns);
    return old;
}

mxfp4_status_t mxfp4_get_device_error(int *code)
{
    if (!code) return MXFP4_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MXFP4_ERR_CUDA;
    const int g = read_and_clear_gemm_error();
    const int f = read_and_clear_fused_error();
    const int pg = read_and_clear_gemm_pair_error();
    if (g < 0 || f < 0 || pg < 0) return MXFP4_ERR_CUDA;
    *code = g != 0 ? g : (f != 0 ? 16 + f : (pg != 0 ? 32 + pg : 0));
    return MXFP4_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// mxfp4_gemm_a4w4_noalloc: the MXFP4 GEMM with its split-K scratch (fp32
// partial sums and per-tile tickets) in a fixed device array owned by this
// library, for callers that cannot allocate device memory themselves.

namespace {

// Scratch of the no-allocation GEMM. Every GPU that loads the library holds
// these bytes until the process exits; all calls share them.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device (host code only
// sees a stand-in symbol, never the address). Looked up again on every call
// made outside stream capture, so that a device reset or a new primary
// context never leaves a stale address behind; a call made while `stream` is
// being captured uses the address of the last call on that device.
mxfp4_status_t noalloc_scratch(cudaStream_t stream, void **out)
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return MXFP4_ERR_NO_DEVICE;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return MXFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MXFP4_ERR_CUDA;
        g_noalloc_ptr[d] = p;
    } else if (!g_noalloc_ptr[d]) {
        return MXFP4_ERR_CUDA;   // the first call on a device must come before any capture
    }
    *out = g_noalloc_ptr[d];
    return MXFP4_OK;
}

}  // namespace

extern "C" {

size_t mxfp4_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

mxfp4_status_t mxfp4_gemm_a4w4_noalloc(const void *Aq, int64_t ldaq, const void *A_sf, const void *Bq,
                                       int64_t ldbq, const void *B_sf, void *C, int64_t ldc, int64_t M,
                                       int64_t N, int64_t K, void *stream)
{
    mxfp4_status_t st = check_gemm_common(Bq, ldbq, B_sf, C, ldc, M, N, K);
    if (st != MXFP4_OK) return st;
    if (!Aq || !A_sf) return MXFP4_ERR_INVALID_ARG;
    if (ldaq < K / 2) return MXFP4_ERR_INVALID_ARG;
    if (ldaq % 16 != 0 || !al16(Aq) || !al16(A_sf)) return MXFP4_ERR_MISALIGNED;
    // scratch this shape needs: split-K partials, then one ticket per tile
    const GemmPlan gp = plan_gemm(M, N, K);
    WsLayout wl;
    memset(&wl, 0, sizeof(wl));
    size_t part = 0;
    if (gp.splits > 1)
        part = static_cast<size_t>(gp.splits) * gp.n_tiles * gp.bn * static_cast<size_t>(M) * 4;
    wl.part_off = 0;
    wl.ticket_off = up256(part);
    wl.total = wl.ticket_off + up256(static_cast<size_t>(gp.tiles) * 4);
    if (wl.total > kNoAllocScratchBytes) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    st = current_device(&sms);
    if (st != MXFP4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    st = noalloc_scratch(s, &scratch);
    if (st != MXFP4_OK) return st;
    // the tile tickets must start at zero; the array keeps whatever the last call left
    if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + wl.ticket_off, 0, static_cast<size_t>(gp.tiles) * 4, s) !=
        cudaSuccess)
        return MXFP4_ERR_CUDA;
    return run_gemm(Aq, ldaq, A_sf, Bq, ldbq, B_sf, C, ldc, M, N, K, scratch, wl, s);
}

}  // extern "C"
