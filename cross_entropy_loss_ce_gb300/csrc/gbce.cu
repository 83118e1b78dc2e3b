// C ABI of the library (declared in include/gbce.h): argument validation, the
// launch plan chosen from the row length, stream-ordered scratch, the sticky
// device error flags and the optional kernel-timing events.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/gbce.h"
#include "row_kernels.cuh"
#include "bsr_kernels.cuh"

static_assert(gbce::kStatusBadTable == GBCE_STATUS_BAD_TABLE, "status bits of the ABI");

namespace gbce {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kWarpMaxVpl = 16;               // rows of <= 32 * 16 16-byte vectors: warp kernel
constexpr int64_t kResidentMax = 64 * 1024;   // rows up to this many staged bytes: resident kernel
constexpr int64_t kSmallCtaVecFwd = 1024;      // softmax forward rows of up to 16 KB: 128-thread
                                               // CTAs, 16 per SM (measured +4% at 4096 x 4096 fp32)
constexpr int64_t kResidentMaxFwd = 32 * 1024;  // the same for the softmax forward (measured: the
                                               // ring streams 64 KB fp32 rows 3% faster there,
                                               // while CE rows of 64 KB lose 17% on it)
constexpr int64_t kSliceMax = 200 * 1024;     // dynamic shared memory limit set on every kernel
constexpr int kMaxCluster = 16;
constexpr int64_t kStreamSlice = 64 * 1024;   // bytes of a row per CTA in the streaming fallback
constexpr int64_t kRingBytes = 192 * 1024;    // ring capacity per CTA (one CTA per SM)
constexpr int kRingWarps = 16;                // consumer warps of the ring kernel
constexpr int kRingWarpsCluster = 15;         // ... when rows are split across a cluster: with
                                              // the producer, 16 warps (4 per SM sub-partition)
                                              // may hold 128 registers each, where 17 warps
                                              // hold 96 and the cluster exchange spilled
constexpr int kRingVpt1 = 4;                  // vectors per consumer thread and slot, one operand
constexpr int kRingVpt2 = 2;                  // the same, two operands (softmax backward)
constexpr int64_t kL2Budget = 40ll << 20;     // bytes of rows between their two reads, all SMs
constexpr int64_t kSmallBatchStaged = 32 * 1024;  // small batches: rows staging more take the
                                              // ring (measured: 64 KB rows, 1-152 of them,
                                              // 5-21% faster there)
constexpr int64_t kMinClusterRow = 64 * 1024; // ... split across a cluster from this row length
                                              // on (shorter: the exchange costs more than the
                                              // split saves, measured on 36-48 KB rows)
constexpr int64_t kMinSlice = 16 * 1024;      // ... in slices of at least this many bytes
constexpr int64_t kBsrTarget = 32 * 1024;     // block-sparse: bytes per slab stage aimed at
constexpr int kBsrThreads = 256;              // block-sparse kernels' CTA size
constexpr int kBsrMaxRows = 64;               // rows per slab (<= kBsrThreads / 4)
constexpr int kBsrStages = 2;                 // slab stages in shared memory
constexpr int kBsrMaxLog2Split = 2;           // at most 4 CTAs per block-row and batch item
constexpr int kBsrLog2MinSlabs = 3;           // ... each keeping >= 8 slabs of the longest block-row

size_t elem_size(int dtype) { return dtype == GBCE_F32 ? 4 : 2; }

// The library's one-time set-up (the scratch pool, kernel attributes,
// occupancy queries, the static scratch array's address) may run while the
// calling thread captures a CUDA graph: a first call can be a captured one.
// The default (global) capture mode refuses such calls; none of them touches
// a stream, so they run with the thread switched to relaxed mode, which
// allows them, and the thread's mode is restored after.
class RelaxedCapture {
public:
    RelaxedCapture() : switched_(cudaThreadExchangeStreamCaptureMode(&mode_) == cudaSuccess) {}
    ~RelaxedCapture()
    {
        if (switched_)  // give the thread back the mode it had
            cudaThreadExchangeStreamCaptureMode(&mode_);
    }
    RelaxedCapture(const RelaxedCapture &) = delete;
    RelaxedCapture &operator=(const RelaxedCapture &) = delete;

private:
    cudaStreamCaptureMode mode_ = cudaStreamCaptureModeRelaxed;
    bool switched_;
};

std::mutex g_sm_mu;
int g_sm_count[kMaxDevices] = {};

// Multiprocessors of the current device (cached per device; 0 if unknown).
int64_t current_sm_count()
{
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
        return 0;
    std::lock_guard<std::mutex> lk(g_sm_mu);
    if (!g_sm_count[device]) {
        RelaxedCapture relaxed;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
            return 0;
        g_sm_count[device] = n;
    }
    return g_sm_count[device];
}

// ---------------------------------------------------------------------------
// launch plan: the kernel regime is chosen by the row length

enum class Kind { Warp, Resident, Ring, Streaming };

struct Plan {
    Kind kind;
    int vpl;        // warp: 16-byte vectors per lane
    int C;          // CTAs per row = cluster size
    int nt;         // threads per CTA
    int per_vec;    // resident: 16-byte vectors staged per operand
    int chunk_vec;  // resident: vectors per bulk copy; ring: vectors per slot
    int nslot;      // ring: slots
    bool hold;      // ring: every slice fits half the ring and is loaded once
    size_t smem;    // dynamic shared memory per CTA
};

// The ring plan for rows of nvec 16-byte vectors per operand split across a
// cluster of C CTAs.
Plan ring_plan(int64_t nvec, int nbuf, int C)
{
    Plan p{};
    p.kind = Kind::Ring;
    p.C = C;
    const int ncw = p.C > 1 ? kRingWarpsCluster : kRingWarps;
    p.nt = (ncw + 1) * 32;
    const int vpt = nbuf == 2 ? kRingVpt2 : kRingVpt1;
    const int64_t chunk_bytes = static_cast<int64_t>(ncw) * 32 * vpt * 16;
    p.chunk_vec = static_cast<int>(chunk_bytes / 16);
    p.nslot = static_cast<int>(kRingBytes / (chunk_bytes * nbuf));
    if (p.nslot > kRingMaxSlots)
        p.nslot = kRingMaxSlots;
    p.smem = static_cast<size_t>(p.nslot) * chunk_bytes * nbuf;
    // the most chunks any row slice needs: rows with a head have fewer vectors
    const int64_t per_max = (nvec + p.C - 1) / p.C;
    const int64_t nch_max = (per_max + p.chunk_vec - 1) / p.chunk_vec;
    p.hold = 2 * nch_max <= p.nslot;
    return p;
}

// cols elements of esize bytes per operand, nbuf operands per row; `aligned`:
// all operands of every row share their address modulo 16 bytes.
Plan make_plan(int64_t cols, size_t esize, int nbuf, bool aligned,
               int64_t resident_max = kResidentMax, int64_t small_cta_vec = 511)
{
    Plan p{};
    const int64_t row_bytes = cols * static_cast<int64_t>(esize);
    if (!aligned) {
        // streaming fallback: a cluster per row, each CTA streaming ~64 KB of it
        p.kind = Kind::Streaming;
        p.C = 1;
        while (p.C < kMaxCluster && row_bytes / p.C > kStreamSlice)
            p.C *= 2;
        p.nt = 512;
        return p;
    }
    const int64_t nvec = row_bytes / 16;  // >= whole vectors of any row
    if (nvec <= 32 * kWarpMaxVpl) {
        // very short rows: one warp per row, the row in registers
        p.kind = Kind::Warp;
        p.C = 1;
        p.nt = kWarpRowsPerCta * 32;
        p.vpl = 1;
        while (32 * p.vpl < nvec)
            p.vpl *= 2;
        return p;
    }
    if (nvec * 16 * nbuf <= resident_max) {
        // short rows: one CTA per row holds the row, three CTAs per SM
        p.kind = Kind::Resident;
        p.C = 1;
        p.per_vec = static_cast<int>(nvec > 0 ? nvec : 1);
        p.nt = p.per_vec > small_cta_vec ? 256 : 128;
        int64_t chunk = (p.per_vec + kMaxChunks - 1) / kMaxChunks;
        chunk = (chunk + p.nt - 1) / p.nt * p.nt;
        p.chunk_vec = static_cast<int>(chunk);
        p.smem = static_cast<size_t>(p.per_vec) * 16 * nbuf;
        return p;
    }
    // long rows: each SM streams one row slice at a time through the ring and
    // reads it twice; split rows across a cluster until the slices between
    // their two reads fit in L2
    const int64_t sms = current_sm_count();
    int C = 1;
    while (C < kMaxCluster && sms * row_bytes * nbuf / C > kL2Budget)
        ++C;
    return ring_plan(nvec, nbuf, C);
}

// ---------------------------------------------------------------------------
// kernel selection

using KernelFn = void (*)(const RowArgs);

// Failure-path test: the copy CTA 0 of later staged row-kernel launches leaves
// out (gbce_test_failure_path); -1 for none.
std::atomic<int> g_drop_copy{-1};

template <Op OP, typename T>
KernelFn pick_kernel(const Plan &p)
{
    switch (p.kind) {
    case Kind::Warp:
        switch (p.vpl) {
        case 1: return rows_warp_kernel<OP, T, 1>;
        case 2: return rows_warp_kernel<OP, T, 2>;
        case 4: return rows_warp_kernel<OP, T, 4>;
        case 8: return rows_warp_kernel<OP, T, 8>;
        default: return rows_warp_kernel<OP, T, 16>;
        }
    case Kind::Resident:
        if (g_drop_copy.load(std::memory_order_relaxed) >= 0)  // failure-path tests only
            return p.nt == 128 ? rows_resident_kernel<OP, T, 128, true>
                               : rows_resident_kernel<OP, T, 256, true>;
        return p.nt == 128 ? rows_resident_kernel<OP, T, 128, false>
                           : rows_resident_kernel<OP, T, 256, false>;
    case Kind::Ring: {
        constexpr int vpt = OP == Op::SoftmaxBwd ? kRingVpt2 : kRingVpt1;
        if (p.C > 1)
            return p.hold ? rows_ring_kernel<OP, T, kRingWarpsCluster, vpt, true, true>
                          : rows_ring_kernel<OP, T, kRingWarpsCluster, vpt, true, false>;
        return p.hold ? rows_ring_kernel<OP, T, kRingWarps, vpt, false, true>
                      : rows_ring_kernel<OP, T, kRingWarps, vpt, false, false>;
    }
    default:
        return rows_streaming_kernel<OP, T, 512>;
    }
}

template <Op OP>
KernelFn pick(int dtype, const Plan &p)
{
    switch (dtype) {
    case GBCE_F32: return pick_kernel<OP, float>(p);
    case GBCE_F16: return pick_kernel<OP, __half>(p);
    default: return pick_kernel<OP, __nv_bfloat16>(p);
    }
}

// Per-device one-time function attributes (large dynamic shared memory,
// cluster sizes above the portable 8).
struct FnConfig {
    const void *fn;
    int device;
};
struct GridCache {
    KernelFn fn;
    int device, C, nt;
    size_t smem;
    int64_t clusters;  // clusters (or CTAs when C == 1) resident at once
};
std::vector<GridCache> g_grid;
std::mutex g_cfg_mu;
std::vector<FnConfig> g_cfg;

cudaError_t configure(const void *fn, int device)
{
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    for (const FnConfig &c : g_cfg)
        if (c.fn == fn && c.device == device)
            return cudaSuccess;
    RelaxedCapture relaxed;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSliceMax));
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess)
        return e;
    g_cfg.push_back({fn, device});
    return cudaSuccess;
}

cudaError_t configure(KernelFn fn, int device)
{
    return configure(reinterpret_cast<const void *>(fn), device);
}

// ---------------------------------------------------------------------------
// stream-ordered scratch from a library-owned pool per device (kept warm)

std::mutex g_pool_mu;
cudaMemPool_t g_pool[kMaxDevices] = {};

cudaError_t pool_for(int device, cudaMemPool_t *out)
{
    if (device < 0 || device >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pool[device]) {
        RelaxedCapture relaxed;
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t pool;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess)
            return e;
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pool[device] = pool;
    }
    *out = g_pool[device];
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// kernel timing (benchmarks)

std::atomic<int> g_timing_on{0};
std::mutex g_timing_mu;
std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_timing_pending;
std::vector<cudaEvent_t> g_event_free;

cudaEvent_t take_event()
{
    if (!g_event_free.empty()) {
        cudaEvent_t e = g_event_free.back();
        g_event_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess)
        return nullptr;
    return e;
}

struct TimedRegion {
    cudaEvent_t start = nullptr, stop = nullptr;
    cudaStream_t stream;
    explicit TimedRegion(cudaStream_t s) : stream(s)
    {
        if (g_timing_on.load(std::memory_order_relaxed)) {
            std::lock_guard<std::mutex> lk(g_timing_mu);
            start = take_event();
            stop = take_event();
            if (!start || !stop || cudaEventRecord(start, stream) != cudaSuccess) {
                if (start)
                    g_event_free.push_back(start);
                if (stop)
                    g_event_free.push_back(stop);
                start = stop = nullptr;  // this call goes untimed
            }
        }
    }
    ~TimedRegion()
    {
        if (start) {
            cudaEventRecord(stop, stream);
            std::lock_guard<std::mutex> lk(g_timing_mu);
            g_timing_pending.emplace_back(start, stop);
        }
    }
};

// ---------------------------------------------------------------------------

int map_error(cudaError_t e)
{
    if (e == cudaSuccess)
        return GBCE_OK;
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver)
        return GBCE_ERR_NO_DEVICE;
    return GBCE_ERR_CUDA;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// How many clusters of the persistent kernel fit on the device at once.
cudaError_t resident_clusters(KernelFn fn, const Plan &p, int device, int64_t *out)
{
    {
        std::lock_guard<std::mutex> lk(g_cfg_mu);
        for (const GridCache &c : g_grid)
            if (c.fn == fn && c.device == device && c.C == p.C && c.nt == p.nt && c.smem == p.smem) {
                *out = c.clusters;
                return cudaSuccess;
            }
    }
    RelaxedCapture relaxed;
    int n = 0;
    cudaError_t e;
    if (p.C == 1) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, p.nt, p.smem);
        n *= sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(p.C), 1, 1);
        cfg.blockDim = dim3(static_cast<unsigned>(p.nt), 1, 1);
        cfg.dynamicSmemBytes = p.smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(p.C);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    }
    if (e != cudaSuccess)
        return e;
    if (n < 1)
        return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lk(g_cfg_mu);
    g_grid.push_back({fn, device, p.C, p.nt, p.smem, n});
    *out = n;
    return cudaSuccess;
}

// The plan for a batch of M rows.  make_plan's plan assumes enough rows to
// fill the device; a batch of at most one row per SM instead goes to the ring
// (rows that stage more than 32 KB), each row of 64 KB or more per operand
// split across the largest cluster of which M fit on the device at once, with
// slices of at least 16 KB: every row is then in flight in one wave, on up to
// 16 SMs each.  Batches no such cluster takes keep make_plan's plan.
template <Op OP>
Plan batch_plan(int dtype, int64_t M, int64_t cols, int nbuf, bool aligned,
                int64_t resident_max = kResidentMax, int64_t small_cta_vec = 511)
{
    const int64_t row_bytes = cols * static_cast<int64_t>(elem_size(dtype));
    const Plan p = make_plan(cols, elem_size(dtype), nbuf, aligned, resident_max, small_cta_vec);
    const bool streamed = p.kind == Kind::Ring ||
                          (p.kind == Kind::Resident && row_bytes * nbuf > kSmallBatchStaged);
    if (!streamed || M < 1 || M > current_sm_count())
        return p;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess)
        return p;
    const int64_t by_slice = row_bytes < kMinClusterRow ? 1 : row_bytes / kMinSlice;
    const int cmax = by_slice < 1 ? 1 : (by_slice > kMaxCluster ? kMaxCluster : static_cast<int>(by_slice));
    const int cmin = p.kind == Kind::Ring ? p.C : 1;
    for (int C = cmax; C >= cmin; --C) {  // fewer clusters fit as they grow
        const Plan q = ring_plan(row_bytes / 16, nbuf, C);
        const KernelFn fn = pick<OP>(dtype, q);
        int64_t fit = 0;
        if (configure(fn, device) != cudaSuccess || resident_clusters(fn, q, device, &fit) != cudaSuccess)
            return p;
        if (fit >= M)
            return q;
    }
    return p;
}

// `after_count`: the row kernel follows ce_count_kernel on the stream and may
// start while it runs (programmatic dependent launch); it waits for it on the
// device before it reads n.
cudaError_t launch_rows(KernelFn fn, const Plan &p, const RowArgs &a_in, cudaStream_t stream,
                        bool after_count = false)
{
    RowArgs a = a_in;
    a.drop_copy = g_drop_copy.load(std::memory_order_relaxed);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return e;
    if (device < 0 || device >= kMaxDevices)
        return cudaErrorInvalidDevice;
    e = configure(fn, device);
    if (e != cudaSuccess)
        return e;
    int64_t clusters = a.M;  // resident and streaming kernels: one CTA / cluster per row
    if (p.kind == Kind::Warp)
        clusters = (a.M + kWarpRowsPerCta - 1) / kWarpRowsPerCta;
    if (p.kind == Kind::Ring) {
        int64_t fit = 0;
        if ((e = resident_clusters(fn, p, device, &fit)) != cudaSuccess)
            return e;
        clusters = fit < a.M ? fit : a.M;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * p.C), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(p.nt), 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    if (p.C > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = static_cast<unsigned>(p.C);
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (after_count) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = nattr ? attr : nullptr;
    cfg.numAttrs = nattr;
    TimedRegion timed(stream);
    return cudaLaunchKernelEx(&cfg, fn, a);
}

// Largest row count such that M * C fits a 1-D grid.
constexpr int64_t kMaxRows = (int64_t{1} << 31) / kMaxCluster - 1;
// Largest row stride in elements: keeps row * stride * element size far from
// int64 overflow (no device has 2^48 bytes).
constexpr int64_t kMaxStride = int64_t{1} << 46;

int check_matrix(const void *p, int64_t stride, int64_t M, int64_t cols, int dtype)
{
    if (M > 0 && !p)
        return GBCE_ERR_NULL;
    if (stride < cols || stride > kMaxStride)
        return GBCE_ERR_SIZE;
    if (!aligned_to(p, elem_size(dtype)))
        return GBCE_ERR_ALIGN;
    return GBCE_OK;
}

int check_common(int64_t M, int64_t cols, int dtype)
{
    if (dtype != GBCE_F32 && dtype != GBCE_BF16 && dtype != GBCE_F16)
        return GBCE_ERR_DTYPE;
    if (M < 0 || cols < 1 || cols > INT32_MAX || M > kMaxRows)
        return GBCE_ERR_SIZE;
    return GBCE_OK;
}

// Do the rows of two operands start at the same address modulo 16 bytes?
bool same_phase(const void *a, int64_t sa, const void *b, int64_t sb, size_t esize, int64_t M)
{
    if ((reinterpret_cast<uintptr_t>(a) - reinterpret_cast<uintptr_t>(b)) % 16 != 0)
        return false;
    if (M <= 1)
        return true;
    return ((sa - sb) * static_cast<int64_t>(esize)) % 16 == 0;
}

// Temporary storage of one cross-entropy call: [0, 4) the non-ignored count
// n, [4, 8) the call's failure word, [kCeScratchHeader, + 4 M) the row losses.
constexpr size_t kCeScratchHeader = 256;

unsigned *fail_word(void *scratch) { return reinterpret_cast<unsigned *>(static_cast<char *>(scratch) + 4); }

// The cross-entropy launches on `stream`: the count kernel (n; the reduced
// loss itself when M == 0), the row kernel, then (mean, sum) the mean kernel,
// each of the last two a programmatic dependent of the one before.  scratch
// holds n at [0, 4); row losses go to `row_loss` when given, else to scratch
// at [kCeScratchHeader, + 4 M).
cudaError_t launch_ce(void *logits, int64_t stride, const int64_t *targets, float *loss,
                      float *row_loss, const float *grad_scale, int64_t M, int64_t V,
                      int64_t ignore_index, int dtype, int reduction, void *scratch,
                      cudaStream_t stream)
{
    int *n_ptr = static_cast<int *>(scratch);
    unsigned *fail = fail_word(scratch);
    if (!row_loss)
        row_loss = reinterpret_cast<float *>(static_cast<char *>(scratch) + kCeScratchHeader);
    ce_count_kernel<1024><<<1, 1024, 0, stream>>>(targets, M, V, ignore_index, n_ptr, fail, loss,
                                                   reduction);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || M == 0)
        return e;
    const Plan p = batch_plan<Op::CE>(dtype, M, V, 1, true);
    RowArgs a{};
    a.in0 = logits;
    a.s0 = stride;
    a.out = logits;
    a.so = stride;
    a.M = M;
    a.cols = V;
    a.targets = targets;
    a.ignore_index = ignore_index;
    a.n_ptr = n_ptr;
    a.row_loss = row_loss;
    a.reduction = reduction;
    a.grad_scale = grad_scale;
    a.fail = fail;
    a.C = p.C;
    a.per_vec = p.per_vec;
    a.chunk_vec = p.chunk_vec;
    a.nslot = p.nslot;
    e = launch_rows(pick<Op::CE>(dtype, p), p, a, stream, true);
    if (e != cudaSuccess || reduction == GBCE_NONE)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(1024, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ce_mean_kernel<1024>, static_cast<const float *>(row_loss), M,
                              static_cast<const int *>(n_ptr), static_cast<const unsigned *>(fail),
                              loss, reduction);
}

// ce_fwd_bwd_ex with its temporary storage from the pool.
int ce_call(void *logits, int64_t stride, const int64_t *targets, float *loss, float *row_loss,
            const float *grad_scale, int64_t M, int64_t V, int64_t ignore_index, int dtype,
            int reduction, cudaStream_t stream)
{
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return map_error(e);
    cudaMemPool_t pool;
    if ((e = pool_for(device, &pool)) != cudaSuccess)
        return map_error(e);
    void *scratch = nullptr;
    const size_t bytes =
        kCeScratchHeader + (row_loss ? 0 : static_cast<size_t>(M) * sizeof(float));
    if ((e = cudaMallocFromPoolAsync(&scratch, bytes, pool, stream)) != cudaSuccess)
        return map_error(e);
    e = launch_ce(logits, stride, targets, loss, row_loss, grad_scale, M, V, ignore_index, dtype,
                  reduction, scratch, stream);
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e == cudaSuccess)
        e = ef;
    return map_error(e);
}

// ---------------------------------------------------------------------------
// block-sparse softmax backward

struct BsrPlan {
    bool staged;     // bsr_bwd_staged_kernel, else bsr_bwd_unstaged_kernel
    bool vec;        // 16-byte accesses, else one element at a time
    int log2_R;      // staged: rows per slab = 2^log2_R
    int ids_bytes;   // staged: shared bytes for the block ids
    int stage_bytes; // staged: one of the kBsrStages slab stages
    int log2_split;  // staged: CTAs per block-row and batch item, log2
    int64_t smem;    // staged: dynamic shared memory per CTA
};

int log2_exact(int64_t v)
{
    int l = 0;
    while ((int64_t{1} << l) < v)
        ++l;
    return l;
}

// Rows of sizemax * block elements.  Staged when the block ids and kBsrStages
// stages of one row each (both operands) fit kSliceMax; R = the largest power of two
// <= min(block, kBsrMaxRows) whose stage stays within kBsrTarget (one row at
// least).  Longer rows go to the unstaged kernel.  `aligned`: the operands'
// bases and batch strides allow 16-byte accesses.
BsrPlan make_bsr_plan(int64_t block, int64_t sizemax, size_t es, bool aligned)
{
    BsrPlan p{};
    const int log2_block = log2_exact(block);
    p.vec = aligned && block * static_cast<int64_t>(es) >= 16;
    p.ids_bytes = static_cast<int>((sizemax * 4 + 15) / 16 * 16);
    const int64_t row2 = sizemax * block * static_cast<int64_t>(es) * 2;
    auto stage = [&](int l) { return ((row2 << l) + 15) / 16 * 16; };
    if (p.ids_bytes + kBsrStages * stage(0) > kSliceMax) {
        p.staged = false;
        return p;
    }
    p.staged = true;
    const int64_t budget = kBsrTarget > stage(0) ? kBsrTarget : stage(0);
    int l = 0;
    while (l < log2_block && (1 << (l + 1)) <= kBsrMaxRows && stage(l + 1) <= budget &&
           p.ids_bytes + kBsrStages * stage(l + 1) <= kSliceMax)
        ++l;
    p.log2_R = l;
    // split long block-rows across CTAs (finer work, a shorter tail), keeping enough slabs
    // per CTA for the stages to overlap
    p.log2_split = log2_block - l - kBsrLog2MinSlabs;
    p.log2_split = p.log2_split < 0 ? 0 : (p.log2_split > kBsrMaxLog2Split ? kBsrMaxLog2Split
                                                                           : p.log2_split);
    p.stage_bytes = static_cast<int>(stage(l));
    p.smem = p.ids_bytes + kBsrStages * int64_t{p.stage_bytes};
    return p;
}

using BsrFn = void (*)(const BsrArgs);

template <typename T>
BsrFn pick_bsr_t(const BsrPlan &p)
{
    constexpr int V = 16 / sizeof(T);
    if (p.staged)
        return p.vec ? bsr_bwd_staged_kernel<T, V, kBsrThreads, kBsrStages>
                     : bsr_bwd_staged_kernel<T, 1, kBsrThreads, kBsrStages>;
    return p.vec ? bsr_bwd_unstaged_kernel<T, V, kBsrThreads>
                 : bsr_bwd_unstaged_kernel<T, 1, kBsrThreads>;
}

BsrFn pick_bsr(int dtype, const BsrPlan &p)
{
    switch (dtype) {
    case GBCE_F32: return pick_bsr_t<float>(p);
    case GBCE_F16: return pick_bsr_t<__half>(p);
    default: return pick_bsr_t<__nv_bfloat16>(p);
    }
}

bool valid_dtype(int dtype) { return dtype == GBCE_F32 || dtype == GBCE_BF16 || dtype == GBCE_F16; }

// Shape checks of softmax_bwd_bsr that need no pointer.
int check_bsr_shape(int64_t y_zstride, int64_t dy_zstride, int64_t dx_zstride, int64_t lut_len,
                    int64_t n_block_rows, int64_t nblocks, int64_t block, int64_t sizemax,
                    int64_t Z, int dtype)
{
    if (!valid_dtype(dtype))
        return GBCE_ERR_DTYPE;
    if (block < 1 || block > 1024 || (block & (block - 1)) || Z < 0 || n_block_rows < 0 ||
        nblocks < 0 || sizemax < 0 || sizemax > INT32_MAX / block || lut_len < 2 * n_block_rows)
        return GBCE_ERR_SIZE;
    const int64_t bb = block * block;
    if (nblocks > kMaxStride / bb)
        return GBCE_ERR_SIZE;
    if (Z > 1) {
        const int64_t need = nblocks * bb;
        for (int64_t st : {y_zstride, dy_zstride, dx_zstride})
            if (st < need || st > kMaxStride)
                return GBCE_ERR_SIZE;
    }
    return GBCE_OK;
}

// ---------------------------------------------------------------------------
// the fused cross-entropy from host buffers: copies overlapped with the rows

constexpr int kHostChunks = 8;  // row chunks whose copy overlaps the previous chunk's kernel

std::mutex g_copy_mu;
cudaStream_t g_copy_stream[kMaxDevices] = {};

// The library's host-to-device copy stream of `device` (created once).
cudaError_t copy_stream_for(int device, cudaStream_t *out)
{
    if (device < 0 || device >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_copy_mu);
    if (!g_copy_stream[device]) {
        cudaStream_t s;
        cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
        if (e != cudaSuccess)
            return e;
        g_copy_stream[device] = s;
    }
    *out = g_copy_stream[device];
    return cudaSuccess;
}

// Scratch of one host call: n and the device loss in the header, the row
// losses at kCeScratchHeader, then the targets (8-byte aligned).
cudaError_t launch_ce_host(const void *logits_host, int64_t host_stride,
                           const int64_t *targets_host, void *grad, int64_t stride,
                           float *loss_host, int64_t M, int64_t V, int64_t ignore_index,
                           int dtype, void *scratch, cudaStream_t stream, cudaStream_t copy)
{
    const size_t es = elem_size(dtype);
    int *n_ptr = static_cast<int *>(scratch);
    float *loss_dev = reinterpret_cast<float *>(static_cast<char *>(scratch) + 16);
    float *row_loss = reinterpret_cast<float *>(static_cast<char *>(scratch) + kCeScratchHeader);
    int64_t *targets = reinterpret_cast<int64_t *>(
        static_cast<char *>(scratch) + kCeScratchHeader + (static_cast<size_t>(M) * 4 + 7) / 8 * 8);
    cudaError_t e = cudaSuccess;
    if (M > 0)
        e = cudaMemcpyAsync(targets, targets_host, static_cast<size_t>(M) * 8,
                            cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return e;
    ce_count_kernel<1024><<<1, 1024, 0, stream>>>(targets, M, V, ignore_index, n_ptr,
                                                   fail_word(scratch), loss_dev, GBCE_MEAN);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    if (M > 0) {
        // the copies start once the stream's earlier work is done (grad may be in use)
        cudaEvent_t ready = nullptr;
        if ((e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming)) != cudaSuccess)
            return e;
        e = cudaEventRecord(ready, stream);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(copy, ready, 0);
        cudaEventDestroy(ready);
        if (e != cudaSuccess)
            return e;
        // the device call's plan for all M rows: the same kernel, so the same bits
        const Plan p = batch_plan<Op::CE>(dtype, M, V, 1, true);
        const KernelFn fn = pick<Op::CE>(dtype, p);
        const int64_t chunks = M < kHostChunks ? M : kHostChunks;
        const int64_t per = (M + chunks - 1) / chunks;
        for (int64_t r0 = 0; r0 < M; r0 += per) {
            const int64_t rows = r0 + per < M ? per : M - r0;
            char *dst = static_cast<char *>(grad) + r0 * stride * es;
            const char *src = static_cast<const char *>(logits_host) + r0 * host_stride * es;
            if (host_stride == V && stride == V)  // contiguous rows: one linear copy
                e = cudaMemcpyAsync(dst, src, rows * V * es, cudaMemcpyHostToDevice, copy);
            else
                e = cudaMemcpy2DAsync(dst, stride * es, src, host_stride * es, V * es, rows,
                                      cudaMemcpyHostToDevice, copy);
            cudaEvent_t landed = nullptr;
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&landed, cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventRecord(landed, copy);
            if (e == cudaSuccess)
                e = cudaStreamWaitEvent(stream, landed, 0);
            if (landed)
                cudaEventDestroy(landed);
            if (e != cudaSuccess)
                return e;
            RowArgs a{};
            void *rows0 = static_cast<char *>(grad) + r0 * stride * es;
            a.in0 = rows0;
            a.s0 = stride;
            a.out = rows0;
            a.so = stride;
            a.M = rows;
            a.cols = V;
            a.targets = targets + r0;
            a.ignore_index = ignore_index;
            a.n_ptr = n_ptr;
            a.row_loss = row_loss + r0;
            a.reduction = GBCE_MEAN;
            a.grad_scale = nullptr;
            a.fail = fail_word(scratch);
            a.C = p.C;
            a.per_vec = p.per_vec;
            a.chunk_vec = p.chunk_vec;
            a.nslot = p.nslot;
            if ((e = launch_rows(fn, p, a, stream)) != cudaSuccess)
                return e;
        }
        ce_mean_kernel<1024><<<1, 1024, 0, stream>>>(row_loss, M, n_ptr, fail_word(scratch),
                                                     loss_dev, GBCE_MEAN);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    return cudaMemcpyAsync(loss_host, loss_dev, sizeof(float), cudaMemcpyDeviceToHost, stream);
}

}  // namespace
}  // namespace gbce

using namespace gbce;

extern "C" int ce_fwd_bwd(void *logits, int64_t stride, const int64_t *targets, float *loss,
                          int64_t M, int64_t V, int64_t ignore_index, int dtype,
                          gbce_stream_t stream_)
{
    int st = check_common(M, V, dtype);
    if (st)
        return st;
    if (!loss || (M > 0 && !targets))
        return GBCE_ERR_NULL;
    if ((st = check_matrix(logits, stride, M, V, dtype)))
        return st;
    if (!aligned_to(targets, 8) || !aligned_to(loss, 4))
        return GBCE_ERR_ALIGN;
    return ce_call(logits, stride, targets, loss, nullptr, nullptr, M, V, ignore_index, dtype,
                   GBCE_MEAN, reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int ce_fwd_bwd_ex(void *logits, int64_t stride, const int64_t *targets, float *loss,
                             float *row_loss, const float *grad_scale, int64_t M, int64_t V,
                             int64_t ignore_index, int dtype, int reduction,
                             gbce_stream_t stream_)
{
    int st = check_common(M, V, dtype);
    if (st)
        return st;
    if (reduction != GBCE_MEAN && reduction != GBCE_SUM && reduction != GBCE_NONE)
        return GBCE_ERR_REDUCTION;
    if ((reduction != GBCE_NONE && !loss) || (reduction == GBCE_NONE && M > 0 && !row_loss) ||
        (M > 0 && !targets))
        return GBCE_ERR_NULL;
    if ((st = check_matrix(logits, stride, M, V, dtype)))
        return st;
    if (!aligned_to(targets, 8) || !aligned_to(loss, 4) || !aligned_to(row_loss, 16) ||
        !aligned_to(grad_scale, 4))
        return GBCE_ERR_ALIGN;
    return ce_call(logits, stride, targets, reduction == GBCE_NONE ? nullptr : loss, row_loss,
                   grad_scale, M, V, ignore_index, dtype, reduction,
                   reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" int scale_rows(void *x, int64_t stride, int64_t M, int64_t N, int dtype,
                          const float *scale, int per_row, gbce_stream_t stream_)
{
    int st = check_common(M, N, dtype);
    if (st)
        return st;
    if (M > 0 && !scale)
        return GBCE_ERR_NULL;
    if ((st = check_matrix(x, stride, M, N, dtype)))
        return st;
    if (!aligned_to(scale, 4))
        return GBCE_ERR_ALIGN;
    if (M == 0)
        return GBCE_OK;
    const int64_t sms = current_sm_count();
    const int64_t grid = M < sms * 8 ? M : (sms > 0 ? sms * 8 : M);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const unsigned g = static_cast<unsigned>(grid);
    switch (dtype) {
    case GBCE_F32:
        scale_rows_kernel<float, 256><<<g, 256, 0, stream>>>(x, stride, M, N, scale, per_row);
        break;
    case GBCE_F16:
        scale_rows_kernel<__half, 256><<<g, 256, 0, stream>>>(x, stride, M, N, scale, per_row);
        break;
    default:
        scale_rows_kernel<__nv_bfloat16, 256><<<g, 256, 0, stream>>>(x, stride, M, N, scale,
                                                                      per_row);
    }
    return map_error(cudaGetLastError());
}

extern "C" int softmax_fwd_ex(const void *x, int64_t x_stride, void *y, int64_t y_stride,
                              int64_t M, int64_t N, int dtype, unsigned int *status,
                              gbce_stream_t stream_)
{
    int st = check_common(M, N, dtype);
    if (st)
        return st;
    if ((st = check_matrix(x, x_stride, M, N, dtype)) || (st = check_matrix(y, y_stride, M, N, dtype)))
        return st;
    if (!aligned_to(status, alignof(unsigned int)))
        return GBCE_ERR_ALIGN;
    if (M == 0)
        return GBCE_OK;
    const size_t es = elem_size(dtype);
    const Plan p = batch_plan<Op::SoftmaxFwd>(dtype, M, N, 1,
                                              same_phase(x, x_stride, y, y_stride, es, M),
                                              kResidentMaxFwd, kSmallCtaVecFwd);
    RowArgs a{};
    a.in0 = x;
    a.s0 = x_stride;
    a.out = y;
    a.so = y_stride;
    a.M = M;
    a.cols = N;
    a.fail = status;
    a.C = p.C;
    a.per_vec = p.per_vec;
    a.chunk_vec = p.chunk_vec;
    a.nslot = p.nslot;
    return map_error(launch_rows(pick<Op::SoftmaxFwd>(dtype, p), p, a,
                                 reinterpret_cast<cudaStream_t>(stream_)));
}

extern "C" int softmax_fwd(const void *x, int64_t x_stride, void *y, int64_t y_stride, int64_t M,
                           int64_t N, int dtype, gbce_stream_t stream)
{
    return softmax_fwd_ex(x, x_stride, y, y_stride, M, N, dtype, nullptr, stream);
}

extern "C" int softmax_bwd_ex(const void *y, int64_t y_stride, const void *dy, int64_t dy_stride,
                              void *dx, int64_t dx_stride, int64_t M, int64_t N, int dtype,
                              unsigned int *status, gbce_stream_t stream_)
{
    int st = check_common(M, N, dtype);
    if (st)
        return st;
    if ((st = check_matrix(y, y_stride, M, N, dtype)) ||
        (st = check_matrix(dy, dy_stride, M, N, dtype)) ||
        (st = check_matrix(dx, dx_stride, M, N, dtype)))
        return st;
    if (!aligned_to(status, alignof(unsigned int)))
        return GBCE_ERR_ALIGN;
    if (M == 0)
        return GBCE_OK;
    const size_t es = elem_size(dtype);
    const bool aligned = same_phase(y, y_stride, dy, dy_stride, es, M) &&
                         same_phase(y, y_stride, dx, dx_stride, es, M);
    const Plan p = batch_plan<Op::SoftmaxBwd>(dtype, M, N, 2, aligned);
    RowArgs a{};
    a.in0 = y;
    a.s0 = y_stride;
    a.in1 = dy;
    a.s1 = dy_stride;
    a.out = dx;
    a.so = dx_stride;
    a.M = M;
    a.cols = N;
    a.fail = status;
    a.C = p.C;
    a.per_vec = p.per_vec;
    a.chunk_vec = p.chunk_vec;
    a.nslot = p.nslot;
    return map_error(launch_rows(pick<Op::SoftmaxBwd>(dtype, p), p, a,
                                 reinterpret_cast<cudaStream_t>(stream_)));
}

extern "C" int softmax_bwd(const void *y, int64_t y_stride, const void *dy, int64_t dy_stride,
                           void *dx, int64_t dx_stride, int64_t M, int64_t N, int dtype,
                           gbce_stream_t stream)
{
    return softmax_bwd_ex(y, y_stride, dy, dy_stride, dx, dx_stride, M, N, dtype, nullptr, stream);
}

extern "C" const char *gbce_plan(int op, int64_t M, int64_t cols, int dtype, int same_phase,
                                 int *ctas_per_row)
{
    if (op < 0 || op > 2 || M < 0 || cols < 1 ||
        (dtype != GBCE_F32 && dtype != GBCE_BF16 && dtype != GBCE_F16))
        return nullptr;
    const bool aligned = same_phase != 0;
    const Plan p = op == 0   ? batch_plan<Op::CE>(dtype, M, cols, 1, aligned)
                   : op == 1 ? batch_plan<Op::SoftmaxFwd>(dtype, M, cols, 1, aligned,
                                                          kResidentMaxFwd, kSmallCtaVecFwd)
                             : batch_plan<Op::SoftmaxBwd>(dtype, M, cols, 2, aligned);
    if (ctas_per_row)
        *ctas_per_row = p.C;
    switch (p.kind) {
    case Kind::Warp: return "rows_warp_kernel";
    case Kind::Resident: return "rows_resident_kernel";
    case Kind::Ring: return "rows_ring_kernel";
    default: return "rows_streaming_kernel";
    }
}

extern "C" int gbce_last_error(gbce_stream_t stream_)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_));
    if (e != cudaSuccess)
        return map_error(e);
    unsigned int flags = 0;
    const unsigned int zero = 0;
    e = cudaMemcpyFromSymbol(&flags, g_flags, sizeof flags);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(g_flags, &zero, sizeof zero);
    if (e != cudaSuccess)
        return map_error(e);
    if (flags & kFlagBadTarget)
        return GBCE_ERR_BAD_TARGET;
    if (flags & kFlagBadTable)
        return GBCE_ERR_BAD_TABLE;
    if (flags & kFlagTimeout)
        return GBCE_ERR_TIMEOUT;
    return GBCE_OK;
}

extern "C" const char *gbce_status_string(int status)
{
    switch (status) {
    case GBCE_OK: return "success";
    case GBCE_ERR_NULL: return "a required pointer is NULL";
    case GBCE_ERR_SIZE: return "invalid size: M < 0, cols < 1, stride < cols, or beyond the limits";
    case GBCE_ERR_DTYPE: return "unknown dtype";
    case GBCE_ERR_ALIGN: return "a pointer is not aligned to its element size";
    case GBCE_ERR_CUDA: return "a CUDA runtime call failed";
    case GBCE_ERR_BAD_TARGET: return "a target is outside [0, V) and is not ignore_index";
    case GBCE_ERR_TIMEOUT: return "a bounded wait for an asynchronous copy gave up";
    case GBCE_ERR_NO_DEVICE: return "no usable CUDA device";
    case GBCE_ERR_REDUCTION: return "reduction is not a gbce_reduction";
    case GBCE_ERR_BAD_TABLE: return "a block-sparse look-up table entry is malformed";
    default: return "unknown status";
    }
}

extern "C" int gbce_pool_reserved(int device, uint64_t *bytes)
{
    if (!bytes)
        return GBCE_ERR_NULL;
    if (device < 0 || device >= kMaxDevices)
        return GBCE_ERR_SIZE;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        pool = g_pool[device];
    }
    *bytes = 0;
    if (!pool)
        return GBCE_OK;
    uint64_t v = 0;  // the attribute is a 64-bit unsigned value
    cudaError_t e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &v);
    if (e == cudaSuccess)
        *bytes = static_cast<uint64_t>(v);
    return map_error(e);
}

extern "C" int gbce_test_failure_path(int64_t drop_copy)
{
    if (drop_copy > INT32_MAX)
        return GBCE_ERR_SIZE;
    g_drop_copy.store(drop_copy < 0 ? -1 : static_cast<int>(drop_copy));
    return GBCE_OK;
}

extern "C" int gbce_timing_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_timing_mu);
    g_timing_on.store(on ? 1 : 0);
    if (!on) {
        for (auto &pr : g_timing_pending) {
            g_event_free.push_back(pr.first);
            g_event_free.push_back(pr.second);
        }
        g_timing_pending.clear();
    }
    return GBCE_OK;
}

extern "C" int gbce_timing_read(double *total_ms, int64_t *launches)
{
    if (!total_ms || !launches)
        return GBCE_ERR_NULL;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    double sum = 0.0;
    int64_t count = 0;
    cudaError_t err = cudaSuccess;
    for (auto &pr : g_timing_pending) {
        cudaError_t e = cudaEventSynchronize(pr.second);
        float ms = 0.f;
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&ms, pr.first, pr.second);
        if (e != cudaSuccess && err == cudaSuccess)
            err = e;
        sum += ms;
        ++count;
        g_event_free.push_back(pr.first);
        g_event_free.push_back(pr.second);
    }
    g_timing_pending.clear();
    *total_ms = sum;
    *launches = count;
    return map_error(err);
}

// ---------------------------------------------------------------------------
// ce_fwd_bwd_noalloc: the same three launches as ce_fwd_bwd, with their
// temporary storage in a fixed static device array instead of the pool.

namespace gbce {
namespace {

constexpr int64_t kNoAllocMaxRows = GBCE_NOALLOC_MAX_ROWS;
// Laid out like the pool scratch of ce_fwd_bwd: the count, then
// kNoAllocMaxRows row losses.
static __device__ __align__(256) unsigned char
    g_noalloc_scratch[kCeScratchHeader + kNoAllocMaxRows * sizeof(float)];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `device` (the current device),
// looked up once per device.  The symbol's name in host code is only a
// host-side handle and must never be handed to a kernel.
cudaError_t noalloc_scratch(int device, void **out)
{
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[device]) {
        RelaxedCapture relaxed;
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_noalloc_addr[device] = p;
    }
    *out = g_noalloc_addr[device];
    return cudaSuccess;
}

}  // namespace
}  // namespace gbce

extern "C" int ce_fwd_bwd_noalloc(void *logits, int64_t stride, const int64_t *targets,
                                  float *loss, int64_t M, int64_t V, int64_t ignore_index,
                                  int dtype, gbce_stream_t stream_)
{
    int st = check_common(M, V, dtype);
    if (st)
        return st;
    if (!loss || (M > 0 && !targets))
        return GBCE_ERR_NULL;
    if ((st = check_matrix(logits, stride, M, V, dtype)))
        return st;
    if (!aligned_to(targets, 8) || !aligned_to(loss, 4))
        return GBCE_ERR_ALIGN;
    if (M > kNoAllocMaxRows)
        return GBCE_ERR_SIZE;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return map_error(e);
    if (device < 0 || device >= kMaxDevices)
        return GBCE_ERR_CUDA;
    void *scratch = nullptr;
    if ((e = noalloc_scratch(device, &scratch)) != cudaSuccess)
        return map_error(e);
    // ce_count_kernel overwrites the count and the row kernel writes the loss
    // of every row 0..M-1 before the mean kernel reads them: nothing left by
    // an earlier call is read.
    e = launch_ce(logits, stride, targets, loss, nullptr, nullptr, M, V, ignore_index, dtype,
                  GBCE_MEAN, scratch, stream);
    return map_error(e);
}

extern "C" int softmax_bwd_bsr_ex(const void *y, int64_t y_zstride, const void *dy,
                                  int64_t dy_zstride, void *dx, int64_t dx_zstride,
                                  const int32_t *lut, int64_t lut_len, int64_t n_block_rows,
                                  int64_t nblocks, int64_t block, int64_t sizemax, int64_t Z,
                                  float scale, int dtype, unsigned int *status,
                                  gbce_stream_t stream_)
{
    int st = check_bsr_shape(y_zstride, dy_zstride, dx_zstride, lut_len, n_block_rows, nblocks,
                             block, sizemax, Z, dtype);
    if (st)
        return st;
    if (!aligned_to(status, alignof(unsigned int)))
        return GBCE_ERR_ALIGN;
    if (Z == 0 || n_block_rows == 0 || sizemax == 0)
        return GBCE_OK;
    if (!y || !dy || !dx || !lut)
        return GBCE_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned_to(y, es) || !aligned_to(dy, es) || !aligned_to(dx, es) || !aligned_to(lut, 4))
        return GBCE_ERR_ALIGN;
    const bool aligned =
        aligned_to(y, 16) && aligned_to(dy, 16) && aligned_to(dx, 16) &&
        (Z <= 1 || ((y_zstride * static_cast<int64_t>(es)) % 16 == 0 &&
                    (dy_zstride * static_cast<int64_t>(es)) % 16 == 0 &&
                    (dx_zstride * static_cast<int64_t>(es)) % 16 == 0));
    const BsrPlan p = make_bsr_plan(block, sizemax, es, aligned);
    const int log2_block = log2_exact(block);
    const int per_row_block = p.staged ? p.log2_split : log2_block;
    // CTAs = Z * n_block_rows * 2^per_row_block must fit a 1-D grid (staged:
    // 2^log2_split per block-row and batch item; unstaged: one per row)
    const int64_t kGridMax = INT32_MAX;
    if (n_block_rows > (kGridMax >> per_row_block) ||
        Z > (kGridMax >> per_row_block) / n_block_rows)
        return GBCE_ERR_SIZE;
    const int64_t units = (Z * n_block_rows) << per_row_block;

    BsrArgs a{};
    a.y = y;
    a.ys = y_zstride;
    a.dy = dy;
    a.dys = dy_zstride;
    a.dx = dx;
    a.dxs = dx_zstride;
    a.lut = lut;
    a.lut_len = lut_len;
    a.nbr = n_block_rows;
    a.nblocks = nblocks;
    a.log2_block = log2_block;
    a.log2_R = p.log2_R;
    a.sizemax = static_cast<int>(sizemax);
    a.ids_bytes = p.ids_bytes;
    a.scale = scale;
    a.status = status;

    a.stage_bytes = p.stage_bytes;
    a.log2_split = p.log2_split;
    a.max_log2_R = log2_block < log2_exact(kBsrMaxRows) ? log2_block : log2_exact(kBsrMaxRows);

    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return map_error(e);
    const BsrFn fn = pick_bsr(dtype, p);
    if ((e = configure(reinterpret_cast<const void *>(fn), device)) != cudaSuccess)
        return map_error(e);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    TimedRegion timed(stream);
    fn<<<static_cast<unsigned>(units), kBsrThreads, p.staged ? p.smem : 0, stream>>>(a);
    return map_error(cudaGetLastError());
}

extern "C" int softmax_bwd_bsr(const void *y, int64_t y_zstride, const void *dy,
                               int64_t dy_zstride, void *dx, int64_t dx_zstride,
                               const int32_t *lut, int64_t lut_len, int64_t n_block_rows,
                               int64_t nblocks, int64_t block, int64_t sizemax, int64_t Z,
                               float scale, int dtype, gbce_stream_t stream)
{
    return softmax_bwd_bsr_ex(y, y_zstride, dy, dy_zstride, dx, dx_zstride, lut, lut_len,
                              n_block_rows, nblocks, block, sizemax, Z, scale, dtype, nullptr,
                              stream);
}

extern "C" const char *gbce_bsr_plan(int64_t block, int64_t sizemax, int dtype, int aligned,
                                     int *rows_per_slab)
{
    if (check_bsr_shape(0, 0, 0, 0, 0, 0, block, sizemax, 0, dtype) != GBCE_OK || sizemax < 1)
        return nullptr;
    const BsrPlan p = make_bsr_plan(block, sizemax, elem_size(dtype), aligned != 0);
    if (rows_per_slab)
        *rows_per_slab = p.staged ? 1 << p.log2_R : 1;
    if (p.staged)
        return p.vec ? "bsr_bwd_staged_kernel" : "bsr_bwd_staged_kernel (element accesses)";
    return p.vec ? "bsr_bwd_unstaged_kernel" : "bsr_bwd_unstaged_kernel (element accesses)";
}

extern "C" int ce_fwd_bwd_host(const void *logits_host, int64_t host_stride,
                               const int64_t *targets_host, void *grad, int64_t stride,
                               float *loss_host, int64_t M, int64_t V, int64_t ignore_index,
                               int dtype, gbce_stream_t stream_)
{
    int st = check_common(M, V, dtype);
    if (st)
        return st;
    if (!loss_host || (M > 0 && (!targets_host || !logits_host)))
        return GBCE_ERR_NULL;
    if (host_stride < V || host_stride > kMaxStride)
        return GBCE_ERR_SIZE;
    if ((st = check_matrix(grad, stride, M, V, dtype)))
        return st;
    const size_t es = elem_size(dtype);
    if (!aligned_to(logits_host, es) || !aligned_to(targets_host, 8) || !aligned_to(loss_host, 4))
        return GBCE_ERR_ALIGN;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return map_error(e);
    cudaStream_t copy;
    if ((e = copy_stream_for(device, &copy)) != cudaSuccess)
        return map_error(e);
    cudaMemPool_t pool;
    if ((e = pool_for(device, &pool)) != cudaSuccess)
        return map_error(e);
    void *scratch = nullptr;
    const size_t bytes = kCeScratchHeader + (static_cast<size_t>(M) * 4 + 7) / 8 * 8 +
                         static_cast<size_t>(M) * 8;
    if ((e = cudaMallocFromPoolAsync(&scratch, bytes, pool, stream)) != cudaSuccess)
        return map_error(e);
    e = launch_ce_host(logits_host, host_stride, targets_host, grad, stride, loss_host, M, V,
                       ignore_index, dtype, scratch, stream, copy);
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e == cudaSuccess)
        e = ef;
    return map_error(e);
}
