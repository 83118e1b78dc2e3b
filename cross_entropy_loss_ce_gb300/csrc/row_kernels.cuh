// Row kernels: fused cross-entropy forward+backward, softmax forward, softmax
// backward, in four regimes chosen on the host by the row length:
//   rows_warp_kernel      rows of <= 8 KB per operand: one warp per row, the row
//                         in registers;
//   rows_resident_kernel  rows of <= 64 KB: one CTA per row, the row staged in
//                         shared memory by 1-D bulk (TMA) copies;
//   rows_ring_kernel      longer rows: persistent, a producer warp streams each
//                         row twice through a shared-memory ring (the second
//                         read served by L2), split across a thread-block
//                         cluster when the rows between reads would not fit L2;
//   rows_streaming_kernel operands whose rows start at different 16-byte
//                         phases: element loads from global memory.
// HBM sees one read and one write per element in the first three.
//
// Per row (cross-entropy; the softmax forward is the same without the target):
//   1. target load and ignore test (Liger-Kernel cross_entropy.py,
//      liger_cross_entropy_kernel, steps 1-2).  Ignored rows are zero-filled
//      with no read; a target outside [0, V) raises a flag and leaves the row.
//   2. pass 1, the online normaliser (same kernel, step 3, "Algorithm 3" of
//      the online-softmax paper it cites): running maxima m and rescaled sums
//      d = sum exp(x - m), kept as (s, d) pairs with s = fl(m log2 e) the shift
//      in log2 units (see exp2_shift), merged by warp shuffles, through shared
//      memory, and across a cluster, each sum rescaled to the larger shift.
//   3. pass 2, the gradient in place (steps 4 and 6): exp(x_i - M) / D times
//      the row's factor k (1/n for the mean), and (exp(x_y - M) / D - 1) k at
//      the target, written from the staged copy or registers.
//   4. the row loss M + ln D - x_y (step 5), evaluated as
//      ln D - (x_y log2 e - S) ln 2, x_y read before any store.
#pragma once

#include <type_traits>

#include "device.cuh"

namespace gbce {

constexpr int kMaxChunks = 8;  // bulk copies (one mbarrier each) per staged row

enum class Op { CE, SoftmaxFwd, SoftmaxBwd };

// Reductions of the cross-entropy (the values of gbce_reduction).
enum : int { kReduceMean = 0, kReduceSum = 1, kReduceNone = 2 };

struct RowArgs {
    const void *in0;  // logits (CE), x (softmax fwd), y (softmax bwd)
    int64_t s0;
    const void *in1;  // dy (softmax bwd)
    int64_t s1;
    void *out;        // logits again (CE, in place), y (softmax fwd), dx (softmax bwd)
    int64_t so;
    int64_t M, cols;
    // cross-entropy only
    const int64_t *targets;
    int64_t ignore_index;
    const int *n_ptr;   // non-ignored row count, written by ce_count_kernel
    float *row_loss;    // [M]
    int reduction;      // kReduceMean / kReduceSum / kReduceNone
    const float *grad_scale;  // NULL (1), one value, or one per row (kReduceNone)
    unsigned *fail;     // this call's failure word, cleared by ce_count_kernel (NULL: none)
    // Failure-path test (gbce_test_failure_path): the bulk copy, counted from 0,
    // that CTA 0 of the launch leaves out; -1 (always, outside such tests) for none.
    // The copy's barrier phase then never completes and the waits for it give up.
    int drop_copy;
    // launch plan
    int C;          // CTAs per row (cluster size; ring and streaming kernels)
    int per_vec;    // resident: 16-byte vectors staged per operand
    int chunk_vec;  // resident: vectors per bulk copy, a multiple of the thread count
    int nslot;      // ring: slots of the shared-memory ring
};

// Sticky error flags of this device (kFlag* bits); defined once per library.
__device__ unsigned int g_flags = 0;

// A bounded wait of this call gave up: the device flag, and for the
// cross-entropy the call's own failure word, which makes its reduced loss NaN.
// A cross-entropy caller has passed wait_prerequisite_grid() (the count kernel
// clears the word).
__device__ __forceinline__ void raise_timeout(unsigned *fail)
{
    atomicOr(&g_flags, kFlagTimeout);
    if (fail)
        atomicOr(fail, 1u);
}

template <Op OP>
struct Partial {
    // Combine two partial results of pass 1 (commutative, so butterflies agree).
    __device__ static __forceinline__ void merge(float &a, float &b, float a2, float b2)
    {
        if constexpr (OP == Op::SoftmaxBwd) {
            a += a2;
        } else {
            md_merge(a, b, a2, b2);
        }
    }
    __device__ static __forceinline__ float2 empty()
    {
        return OP == Op::SoftmaxBwd ? make_float2(0.f, 0.f) : make_float2(-INFINITY, 0.f);
    }
    __device__ static __forceinline__ void warp_reduce(float &a, float &b)
    {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float a2 = __shfl_xor_sync(0xffffffffu, a, off);
            const float b2 = __shfl_xor_sync(0xffffffffu, b, off);
            merge(a, b, a2, b2);
        }
    }
};

__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Wait for the kernel this one depends on (launched before it with
// programmatic stream serialisation) to complete and publish its writes.
//
// ce_row_exit_order: every CTA of a cross-entropy row kernel executes this
// before it exits, also on the early exits of ignored rows and bad targets
// that read no n.  The mean kernel waits only for the row kernel; because no
// row-kernel CTA can finish before the count kernel has, the row kernel's
// completion implies the count kernel's, and the mean kernel reads this
// call's n even when every row was ignored.
__device__ __forceinline__ void wait_prerequisite_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// A cross-entropy gradient row is (p - onehot) * k with k = s / n (mean) or s
// (sum, none), s the incoming grad_output (1 when absent, per row for none).
// Returns scale = k / D (for exp(x - M)) and sub = k (the one-hot term); for
// the mean without a grad_output these are 1 / (D n) and 1 / n.
__device__ __forceinline__ void ce_row_factor(const RowArgs &a, int64_t row, float D, float n,
                                              float &scale, float &sub)
{
    const float kn = a.reduction == kReduceMean ? n : 1.f;
    const float s = a.grad_scale ? __ldg(a.grad_scale + (a.reduction == kReduceNone ? row : 0)) : 1.f;
    scale = s / (D * kn);
    sub = s / kn;
}

// sum_{r < M} row_loss[r] by NTH threads (tid < NTH, all calling, synchronised
// by named barrier `bar`) in a fixed order, so the same inputs give the same
// bits: thread t adds the 16-byte groups t, t + NTH, ... (each group's four
// values in order) with Neumaier's compensated summation, then the threads'
// sums meet in fixed butterflies.  Row losses are >= 0 (or NaN), so there is
// no cancellation: the relative error stays below ~(log2(NTH) + 2) * 2^-24.
// fp32 throughout: fp64 throughput is a small fraction of fp32 on this GPU.
// Returns the total in thread 0.  row_loss is 16-byte aligned; loads go
// through L2.
__device__ __forceinline__ void neumaier_add(float &s, float &c, float v)
{
    const float t = s + v;
    c += (fabsf(s) >= fabsf(v)) ? (s - t) + v : (v - t) + s;
    s = t;
}

template <int NTH>
__device__ __forceinline__ float sum_row_losses(const float *row_loss, int64_t M, int tid, int bar)
{
    __shared__ float part[NTH / 32];
    const float4 *v = reinterpret_cast<const float4 *>(row_loss);
    const int64_t nv = M / 4;
    float s = 0.f, c = 0.f;
    int64_t i = tid;
    for (; i + 3 * NTH < nv; i += 4 * NTH) {  // four independent 16-byte loads in flight
        const float4 a = __ldcg(v + i), b = __ldcg(v + i + NTH);
        const float4 e = __ldcg(v + i + 2 * NTH), f = __ldcg(v + i + 3 * NTH);
        neumaier_add(s, c, a.x), neumaier_add(s, c, a.y), neumaier_add(s, c, a.z), neumaier_add(s, c, a.w);
        neumaier_add(s, c, b.x), neumaier_add(s, c, b.y), neumaier_add(s, c, b.z), neumaier_add(s, c, b.w);
        neumaier_add(s, c, e.x), neumaier_add(s, c, e.y), neumaier_add(s, c, e.z), neumaier_add(s, c, e.w);
        neumaier_add(s, c, f.x), neumaier_add(s, c, f.y), neumaier_add(s, c, f.z), neumaier_add(s, c, f.w);
    }
    for (; i < nv; i += NTH) {
        const float4 a = __ldcg(v + i);
        neumaier_add(s, c, a.x), neumaier_add(s, c, a.y), neumaier_add(s, c, a.z), neumaier_add(s, c, a.w);
    }
    if (tid == 0)
        for (int64_t j = nv * 4; j < M; ++j)
            neumaier_add(s, c, __ldcg(row_loss + j));
    float t = s + c;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, off);
    if ((tid & 31) == 0)
        part[tid >> 5] = t;
    named_barrier_sync(bar, NTH);
    if (tid < 32) {
        t = tid < NTH / 32 ? part[tid] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            t += __shfl_xor_sync(0xffffffffu, t, off);
    }
    return t;
}

// ---------------------------------------------------------------------------
// Warp form, for short rows (at most 32 * VPL 16-byte vectors per operand):
// one warp per row, eight rows per CTA.  Each lane holds VPL vectors of its
// row in registers (128-bit loads straight from global memory), the row's
// reductions are warp shuffles, and pass 2 works from the registers: one read
// and one write per element, no shared memory and no CTA barrier.
constexpr int kWarpRowsPerCta = 8;

template <Op OP, typename T, int VPL>
__global__ void __launch_bounds__(kWarpRowsPerCta * 32) rows_warp_kernel(const RowArgs a)
{
    using E = Elem<T>;
    constexpr int VEC = E::kPerVec;
    constexpr int NBUF = (OP == Op::SoftmaxBwd) ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpRowsPerCta + (threadIdx.x >> 5);
    if (OP == Op::CE && threadIdx.x == 0)  // the mean kernel may be scheduled (it waits for this grid)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (row >= a.M)
        return;

    const T *in0 = static_cast<const T *>(a.in0) + row * a.s0;
    const T *in1 = nullptr;
    if constexpr (NBUF == 2)
        in1 = static_cast<const T *>(a.in1) + row * a.s1;
    T *out = static_cast<T *>(a.out) + row * a.so;
    const RowGeom g = row_geom(in0, a.cols);
    const int cnt = static_cast<int>(g.nvec);
    const bool head_here = lane < g.head;
    const bool tail_here = lane < g.tail;
    const uint4 *src0 = reinterpret_cast<const uint4 *>(in0 + g.head);
    uint4 *o = reinterpret_cast<uint4 *>(out + g.head);

    int64_t y = -1;
    if constexpr (OP == Op::CE) {
        y = a.targets[row];
        if (y == a.ignore_index) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                if (lane + 32 * v < cnt)
                    __stcs(o + lane + 32 * v, z);
            if (head_here)
                E::store(out + lane, 0.f);
            if (tail_here)
                E::store(out + g.tail_start + lane, 0.f);
            if (lane == 0)
                a.row_loss[row] = 0.f;
            wait_prerequisite_grid();  // see ce_row_exit_order
            return;
        }
        if (y < 0 || y >= a.cols) {
            if (lane == 0) {
                a.row_loss[row] = __int_as_float(0x7fc00000);
                atomicOr(&g_flags, kFlagBadTarget);
            }
            wait_prerequisite_grid();
            return;
        }
    }

    // the row, straight into registers
    uint4 r0[VPL], r1[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        const int j = lane + 32 * v;
        r0[v] = j < cnt ? __ldcs(src0 + j)
                        : make_uint4(E::kNegInfPair, E::kNegInfPair, E::kNegInfPair, E::kNegInfPair);
        if constexpr (NBUF == 2)
            r1[v] = j < cnt ? __ldcs(reinterpret_cast<const uint4 *>(in1 + g.head) + j)
                            : make_uint4(0u, 0u, 0u, 0u);
    }
    float h0 = 0.f, h1 = 0.f, t0 = 0.f, t1 = 0.f;
    if (head_here) {
        h0 = E::load(in0 + lane);
        if constexpr (NBUF == 2)
            h1 = E::load(in1 + lane);
    }
    if (tail_here) {
        t0 = E::load(in0 + g.tail_start + lane);
        if constexpr (NBUF == 2)
            t1 = E::load(in1 + g.tail_start + lane);
    }

    if constexpr (OP == Op::SoftmaxBwd) {
        float sdot = 0.f;
        if (head_here)
            sdot = fmaf(h0, h1, sdot);
        if (tail_here)
            sdot = fmaf(t0, t1, sdot);
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            if (lane + 32 * v < cnt) {
                float fy[VEC], fd[VEC];
                E::unpack(r0[v], fy);
                E::unpack(r1[v], fd);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    sdot = fmaf(fy[e], fd[e], sdot);
            }
        }
        sdot = warp_sum(sdot);
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            if (lane + 32 * v < cnt) {
                float fy[VEC], fd[VEC];
                E::unpack(r0[v], fy);
                E::unpack(r1[v], fd);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    fy[e] = fy[e] * (fd[e] - sdot);
                __stcs(o + lane + 32 * v, E::pack(fy));
            }
        }
        if (head_here)
            E::store(out + lane, h0 * (h1 - sdot));
        if (tail_here)
            E::store(out + g.tail_start + lane, t0 * (t1 - sdot));
        return;
    } else {
        // the row maximum (vectors past the end read as -inf), then the normaliser
        float m = -INFINITY;
        if (head_here)
            m = h0;
        if (tail_here)
            m = fmaxf(m, t0);
        if constexpr (VEC == 8) {
            uint32_t mm = E::kNegInfPair;
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                mm = E::max2(E::max2(mm, r0[v].x), E::max2(r0[v].y, E::max2(r0[v].z, r0[v].w)));
            m = fmaxf(m, E::pair_max(mm));
        } else {
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                if (lane + 32 * v < cnt) {
                    float f[VEC];
                    E::unpack(r0[v], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        m = fmaxf(m, f[e]);
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        // the row's shift in log2 units (0 for an all -inf row, whose terms are 0)
        const float sL = (m == -INFINITY) ? 0.f : shift_of(m);
        float d = 0.f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            if (lane + 32 * v < cnt) {
                float f[VEC];
                E::unpack(r0[v], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    d += exp2_shift(f[e], sL);
            }
        }
        if (head_here)
            d += exp2_shift(h0, sL);
        if (tail_here)
            d += exp2_shift(t0, sL);
        d = warp_sum(d);

        float scale, sub = 0.f;
        if constexpr (OP == Op::CE) {
            wait_prerequisite_grid();  // n comes from the count kernel
            ce_row_factor(a, row, d, static_cast<float>(*a.n_ptr), scale, sub);
        } else {
            scale = 1.f / d;
        }
        const int64_t ycol = y - g.head;
        float xy = 0.f;  // the target logit, from the registers of the lane that holds it
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const int j = lane + 32 * v;
            if (j < cnt) {
                float f[VEC];
                E::unpack(r0[v], f);
                float gr[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    gr[e] = exp2_shift(f[e], sL) * scale;
                if constexpr (OP == Op::CE) {
                    const int64_t rel = ycol - static_cast<int64_t>(j) * VEC;
                    if (rel >= 0 && rel < VEC) {  // the target column: (p_y - 1) / n
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (e == rel) {
                                gr[e] = fmaf(exp2_shift(f[e], sL), scale, -sub);
                                xy = f[e];
                            }
                    }
                }
                __stcs(o + j, E::pack(gr));
            }
        }
        if (head_here) {
            const float ex = exp2_shift(h0, sL);
            E::store(out + lane, (OP == Op::CE && y == lane) ? fmaf(ex, scale, -sub) : ex * scale);
            if (OP == Op::CE && y == lane)
                xy = h0;
        }
        if (tail_here) {
            const float ex = exp2_shift(t0, sL);
            const bool at_y = OP == Op::CE && y == g.tail_start + lane;
            E::store(out + g.tail_start + lane, at_y ? fmaf(ex, scale, -sub) : ex * scale);
            if (at_y)
                xy = t0;
        }
        if constexpr (OP == Op::CE) {
            // exactly one lane holds the target logit; the others contribute 0
            xy = warp_sum(xy);
            if (lane == 0)
                a.row_loss[row] = row_loss_from(sL, d, xy);
        }
    }
}

// ---------------------------------------------------------------------------
// Resident form, for rows whose operands fit one CTA's shared memory (<= 64 KB
// per row in all): one CTA per row, three CTAs per SM.  The CTA stages its row
// with up to kMaxChunks bulk copies (one mbarrier each), runs pass 1 as the
// chunks land, and pass 2 from the staged copy.
// Residency: 128-thread CTAs serve short softmax-forward rows, 16 of them per
// SM; otherwise 1536 threads per SM, except the fp32 softmax backward with
// 1280 (48 registers: at 40 it spilled 28 bytes; measured on 4096 x 4096 fp32,
// 1280 and 1536 threads run alike, while 1024 threads, 64 registers, ran 8%
// slower).
// DROP: the instance for failure-path tests only (a.drop_copy may name a copy
// CTA 0 leaves out); the others carry no trace of the test (the check in the
// issue loop alone cost 4% on 4096 x 4096 fp32 rows).
template <Op OP, typename T, int NT, bool DROP>
__global__ void __launch_bounds__(NT, (OP == Op::SoftmaxFwd && NT == 128) ? 16
                                      : ((OP == Op::SoftmaxBwd && sizeof(T) == 4) ? 1280 / NT
                                                                                 : 1536 / NT))
    rows_resident_kernel(const RowArgs a)
{
    using E = Elem<T>;
    using P = Partial<OP>;
    constexpr int VEC = E::kPerVec;
    constexpr int NW = NT / 32;
    constexpr int NBUF = (OP == Op::SoftmaxBwd) ? 2 : 1;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kMaxChunks];
    __shared__ float2 red[NW];
    __shared__ float4 fin;

    const int64_t row = blockIdx.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    if constexpr (OP == Op::CE)  // the mean kernel may be scheduled (it waits for this grid)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const T *in0 = static_cast<const T *>(a.in0) + row * a.s0;
    const T *in1 = nullptr;
    if constexpr (NBUF == 2)
        in1 = static_cast<const T *>(a.in1) + row * a.s1;
    T *out = static_cast<T *>(a.out) + row * a.so;

    // Every operand of a row shares this geometry (the host checks that their
    // row starts agree modulo 16 bytes).
    const RowGeom g = row_geom(in0, a.cols);
    const int cnt = static_cast<int>(g.nvec);
    const bool head_here = tid < g.head;
    const bool tail_here = tid < g.tail;
    uint4 *o = reinterpret_cast<uint4 *>(out + g.head);

    int64_t y = -1;
    if constexpr (OP == Op::CE) {
        y = a.targets[row];
        if (y == a.ignore_index) {
            // ignored row: zero gradient, zero loss, nothing read
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int j = tid; j < cnt; j += NT)
                __stcs(o + j, z);
            if (head_here)
                E::store(out + tid, 0.f);
            if (tail_here)
                E::store(out + g.tail_start + tid, 0.f);
            if (tid == 0)
                a.row_loss[row] = 0.f;
            wait_prerequisite_grid();  // see ce_row_exit_order
            return;
        }
        if (y < 0 || y >= a.cols) {
            // out-of-range target: flag it, NaN loss, leave the row as it is
            if (tid == 0) {
                a.row_loss[row] = __int_as_float(0x7fc00000);
                atomicOr(&g_flags, kFlagBadTarget);
            }
            wait_prerequisite_grid();
            return;
        }
    }

    // ---- issue the bulk copies of the row (one mbarrier per chunk)
    const int nch = cnt ? (cnt + a.chunk_vec - 1) / a.chunk_vec : 0;
    const uint32_t buf0 = smem_addr(smem);
    const uint32_t buf1 = buf0 + static_cast<uint32_t>(a.per_vec) * 16u;
    if (tid == 0) {
        for (int k = 0; k < nch; ++k)
            mbar_init(smem_addr(&bars[k]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint64_t pol = policy_evict_first();
        const int drop = (DROP && blockIdx.x == 0) ? a.drop_copy : -1;
        for (int k = 0; k < nch; ++k) {
            if (DROP && k == drop)
                continue;  // failure-path test: this chunk never lands
            const int c0 = k * a.chunk_vec;
            const int c1 = c0 + a.chunk_vec < cnt ? c0 + a.chunk_vec : cnt;
            const uint32_t bytes = static_cast<uint32_t>(c1 - c0) * 16u;
            const uint32_t bar = smem_addr(&bars[k]);
            mbar_arrive_expect_tx(bar, bytes * NBUF);
            bulk_load(buf0 + c0 * 16u, in0 + g.head + static_cast<int64_t>(c0) * VEC, bytes, bar,
                      pol);
            if constexpr (NBUF == 2)
                bulk_load(buf1 + c0 * 16u, in1 + g.head + static_cast<int64_t>(c0) * VEC, bytes, bar,
                          pol);
        }
    }

    // scalar head / tail elements (fewer than one vector each)
    float h0 = 0.f, h1 = 0.f, t0 = 0.f, t1 = 0.f;
    if (head_here) {
        h0 = E::load(in0 + tid);
        if constexpr (NBUF == 2)
            h1 = E::load(in1 + tid);
    }
    if (tail_here) {
        t0 = E::load(in0 + g.tail_start + tid);
        if constexpr (NBUF == 2)
            t1 = E::load(in1 + g.tail_start + tid);
    }
    float xy = 0.f;  // the target logit, read before this CTA stores anything
    if constexpr (OP == Op::CE) {
        if (tid == 0)
            xy = E::load(in0 + y);
    }

    // ---- pass 1
    bool ok = true;
    float pa, pb;  // (m, d) for CE / softmax fwd, (sum y*dy, unused) for softmax bwd
    if constexpr (OP == Op::SoftmaxBwd) {
        float sdot = 0.f;
        for (int k = 0; k < nch && ok; ++k) {
            ok = mbar_wait_bounded(smem_addr(&bars[k]), 0);
            const int c1 = (k + 1) * a.chunk_vec < cnt ? (k + 1) * a.chunk_vec : cnt;
            if (ok) {
                for (int j = k * a.chunk_vec + tid; j < c1; j += NT) {
                    float fy[VEC], fd[VEC];
                    E::unpack(ld_shared_v4(buf0 + j * 16u), fy);
                    E::unpack(ld_shared_v4(buf1 + j * 16u), fd);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        sdot = fmaf(fy[e], fd[e], sdot);
                }
            }
        }
        // head and tail (loaded before the chunks landed) last: their load latency
        // overlaps the chunk waits
        if (head_here)
            sdot = fmaf(h0, h1, sdot);
        if (tail_here)
            sdot = fmaf(t0, t1, sdot);
        ok = __syncthreads_and(ok);
        pa = sdot;
        pb = 0.f;
    } else {
        float m = -INFINITY;
        for (int k = 0; k < nch && ok; ++k) {
            ok = mbar_wait_bounded(smem_addr(&bars[k]), 0);
            const int c1 = (k + 1) * a.chunk_vec < cnt ? (k + 1) * a.chunk_vec : cnt;
            if (ok) {
                if constexpr (VEC == 8) {
                    // 16-bit types: packed max of element pairs, no unpacking
                    uint32_t mm = E::kNegInfPair;
                    for (int j = k * a.chunk_vec + tid; j < c1; j += NT) {
                        const uint4 v = ld_shared_v4(buf0 + j * 16u);
                        mm = E::max2(E::max2(mm, v.x), E::max2(v.y, E::max2(v.z, v.w)));
                    }
                    m = fmaxf(m, E::pair_max(mm));
                } else {
                    for (int j = k * a.chunk_vec + tid; j < c1; j += NT) {
                        float f[VEC];
                        E::unpack(ld_shared_v4(buf0 + j * 16u), f);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            m = fmaxf(m, f[e]);
                    }
                }
            }
        }
        // head and tail (loaded before the chunks landed) last: their load latency
        // overlaps the chunk waits
        if (head_here)
            m = fmaxf(m, h0);
        if (tail_here)
            m = fmaxf(m, t0);
        // every chunk has landed once all threads passed the loop above
        ok = __syncthreads_and(ok);
        float d = 0.f;
        if (ok) {
            // this thread's shift in log2 units (0 if it saw only -inf: its terms are 0)
            const float sL = (m == -INFINITY) ? 0.f : shift_of(m);
#pragma unroll 2
            for (int j = tid; j < cnt; j += NT) {
                float f[VEC];
                E::unpack(ld_shared_v4(buf0 + j * 16u), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    d += exp2_shift(f[e], sL);
            }
            if (head_here)
                d += exp2_shift(h0, sL);
            if (tail_here)
                d += exp2_shift(t0, sL);
        }
        pa = shift_of(m);  // (shift, sum) partial; (-inf, 0) when empty
        pb = d;
    }

    // ---- CTA reduction of the partials
    P::warp_reduce(pa, pb);
    if (lane == 0)
        red[warp] = make_float2(pa, pb);
    __syncthreads();
    if (warp == 0) {
        const float2 e = P::empty();
        pa = lane < NW ? red[lane].x : e.x;
        pb = lane < NW ? red[lane].y : e.y;
        P::warp_reduce(pa, pb);
        if (lane == 0)
            fin = make_float4(pa, pb, 0.f, 0.f);
    }
    __syncthreads();
    const float4 r = fin;

    // ---- pass 2: results from the staged copy, one store per element
    if (ok) {
        if constexpr (OP == Op::SoftmaxBwd) {
            const float sdot = r.x;
#pragma unroll 2
            for (int j = tid; j < cnt; j += NT) {
                float fy[VEC], fd[VEC];
                E::unpack(ld_shared_v4(buf0 + j * 16u), fy);
                E::unpack(ld_shared_v4(buf1 + j * 16u), fd);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    fy[e] = fy[e] * (fd[e] - sdot);
                __stcs(o + j, E::pack(fy));
            }
            if (head_here)
                E::store(out + tid, h0 * (h1 - sdot));
            if (tail_here)
                E::store(out + g.tail_start + tid, t0 * (t1 - sdot));
        } else {
            const float SL = r.x, D = r.y;  // the row's shift (log2 units) and sum
            float scale, sub = 0.f;
            if constexpr (OP == Op::CE) {
                wait_prerequisite_grid();  // n comes from the count kernel
                ce_row_factor(a, row, D, static_cast<float>(*a.n_ptr), scale, sub);
            } else {
                scale = 1.f / D;
            }
            const int64_t ycol = y - g.head;  // target position relative to the vectors
#pragma unroll 2
            for (int j = tid; j < cnt; j += NT) {
                float f[VEC];
                E::unpack(ld_shared_v4(buf0 + j * 16u), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    f[e] = exp2_shift(f[e], SL);
                float gr[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    gr[e] = f[e] * scale;
                if constexpr (OP == Op::CE) {
                    const int64_t rel = ycol - static_cast<int64_t>(j) * VEC;
                    if (rel >= 0 && rel < VEC) {  // the target column: (p_y - 1) / n
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (e == rel)
                                gr[e] = fmaf(f[e], scale, -sub);
                    }
                }
                __stcs(o + j, E::pack(gr));
            }
            if (head_here) {
                const float ex = exp2_shift(h0, SL);
                E::store(out + tid, (OP == Op::CE && y == tid) ? fmaf(ex, scale, -sub) : ex * scale);
            }
            if (tail_here) {
                const float ex = exp2_shift(t0, SL);
                E::store(out + g.tail_start + tid,
                         (OP == Op::CE && y == g.tail_start + tid) ? fmaf(ex, scale, -sub)
                                                                    : ex * scale);
            }
            if constexpr (OP == Op::CE) {
                if (tid == 0)
                    a.row_loss[row] = row_loss_from(SL, D, xy);
            }
        }
    } else {
        if (tid == 0) {
            if constexpr (OP == Op::CE) {
                wait_prerequisite_grid();  // the count kernel has cleared the failure word
                a.row_loss[row] = __int_as_float(0x7fc00000);
            }
            raise_timeout(a.fail);
            // copies still in flight land before the CTA exits (a fixed budget)
            const int drop = (DROP && blockIdx.x == 0) ? a.drop_copy : -1;
            const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
            for (int k = 0; k < nch; ++k)
                if (k != drop)
                    mbar_wait_until(smem_addr(&bars[k]), 0, deadline);
        }
    }
}

// ---------------------------------------------------------------------------
template <Op OP>
__device__ __forceinline__ bool row_is_live(const RowArgs &a, int64_t y)
{
    if constexpr (OP == Op::CE)
        return y != a.ignore_index && y >= 0 && y < a.cols;
    return true;
}

// ---------------------------------------------------------------------------
// Warp-specialised ring form (one CTA, or a cluster of a.C CTAs, per row;
// persistent over rows).
//
// A producer warp streams each live row slice through a ring of shared-memory
// chunks with 1-D bulk copies: first the whole slice for pass 1, then the
// slice again, chunks in order, for pass 2 (or once, held for both passes,
// when it fits half the ring).  The consumer warps reduce the pass-1 chunks
// online, merge (shift, sum) pairs across the CTA and the cluster, and write
// the pass-2 results.  The ring keeps up to its whole capacity of loads in
// flight through every phase (including the reduction), and the second read
// of a slice follows the first by one slice-time, so it is served by L2: HBM
// sees one read and one write per element, as with a row held on chip.
// full[s] (count 1 + bytes) and empty[s] (one arrival per consumer warp) hand
// each slot back and forth.  Every wait is bounded: a consumer warp that gives
// up stops releasing slots, a row any warp gave up on gets no stores, and the
// producer waits for every copy it issued before the CTA exits.
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// L2 policy for data that will be read again soon.
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

constexpr int kRingMaxSlots = 32;

constexpr int kRingMaxCluster = 16;

// CLUSTER: rows are split across a cluster of a.C CTAs (else one CTA per row).
// HOLD: every row slice fills at most half the ring and is loaded once, held
// for pass 2 (the host checks this bound for the whole launch).  Both are
// template parameters so that the common path carries no code of the other.
template <Op OP, typename T, int NCW, int VPT, bool CLUSTER, bool HOLD>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) rows_ring_kernel(const RowArgs a)
{
    using E = Elem<T>;
    using P = Partial<OP>;
    constexpr int VEC = E::kPerVec;
    constexpr int NBUF = (OP == Op::SoftmaxBwd) ? 2 : 1;
    constexpr int NC = NCW * 32;            // consumer threads
    constexpr int CHUNK = NC * VPT;         // 16-byte vectors per ring slot and operand
    constexpr uint32_t kChunkBytes = CHUNK * 16u;
    constexpr uint32_t kSlotBytes = kChunkBytes * NBUF;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[kRingMaxSlots];
    __shared__ __align__(8) uint64_t empty[kRingMaxSlots];
    __shared__ __align__(8) uint64_t xbar[2];  // cluster exchange, by live-row parity
    __shared__ __align__(16) float4 xslot[2][kRingMaxCluster];
    __shared__ float2 red[NCW];
    __shared__ int wbad[NCW];  // a consumer warp whose wait gave up (this row or before)
    __shared__ float4 fin;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int C = CLUSTER ? a.C : 1;
    const int rank = CLUSTER ? static_cast<int>(cluster_rank()) : 0;
    // 32-bit row and vector indices throughout (rows < 2^27 and columns < 2^31
    // are checked on the host); only the row base addresses are 64-bit
    const int cid = static_cast<int>(blockIdx.x) / C;
    const int G = static_cast<int>(gridDim.x) / C;
    const int M = static_cast<int>(a.M);
    const int nslot = a.nslot;
    const uint32_t ring = smem_addr(smem);

    if (tid == 0) {
        for (int s = 0; s < nslot; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), NCW);
        }
        mbar_init(smem_addr(&xbar[0]), 1);
        mbar_init(smem_addr(&xbar[1]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if constexpr (CLUSTER) {  // every peer's barriers exist before anyone signals them
        cluster_arrive_any();
        cluster_wait_any();
    }

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
            uint32_t slot = 0, ph = 0;
            bool ok = true;
            // slots filled at least once, and the phase of each slot's last fill
            uint32_t filled = 0, fill_ph = 0;
            uint32_t issued = 0;  // copies issued so far, the left-out one included
            const int drop = blockIdx.x == 0 ? a.drop_copy : -1;
            int64_t ynext = (OP == Op::CE && cid < M) ? a.targets[cid] : 0;
            for (int row = cid; row < M && ok; row += G) {
                const int64_t y = ynext;
                if (OP == Op::CE && row + G < M)
                    ynext = a.targets[row + G];
                if (!row_is_live<OP>(a, y))
                    continue;  // ignored or invalid target: nothing to read
                const T *in0 = static_cast<const T *>(a.in0) + row * a.s0;
                const T *in1 = nullptr;
                if constexpr (NBUF == 2)
                    in1 = static_cast<const T *>(a.in1) + row * a.s1;
                const RowGeom g = row_geom(in0, a.cols);
                const int nvec = static_cast<int>(g.nvec);
                const int per = (nvec + C - 1) / C;
                const int v0 = rank * per;
                const int cnt = v0 < nvec ? (v0 + per < nvec ? per : nvec - v0) : 0;
                const int body = g.head + v0 * VEC;
                const int nch = (cnt + CHUNK - 1) / CHUNK;
                if (HOLD && 2 * nch > nslot)
                    continue;  // outside the launch's bound: the consumers skip it too
                // a held slice is loaded once; otherwise the row is streamed twice
                constexpr int passes = HOLD ? 1 : 2;
                for (int pass = 0; pass < passes && ok; ++pass) {
                    for (int kk = 0; kk < nch; ++kk) {
                        const int c0 = kk * CHUNK;
                        const int c1 = c0 + CHUNK < cnt ? c0 + CHUNK : cnt;
                        const uint32_t bytes = static_cast<uint32_t>(c1 - c0) * 16u;
                        if (!mbar_wait_bounded(smem_addr(&empty[slot]), ph ^ 1u)) {
                            ok = false;
                            atomicOr(&g_flags, kFlagTimeout);
                            break;
                        }
                        const uint32_t fb = smem_addr(&full[slot]);
                        const uint32_t dst = ring + slot * kSlotBytes;
                        if (drop >= 0 && issued == static_cast<uint32_t>(drop)) {
                            // failure-path test: this fill is left out, its phase never completes
                        } else {
                            mbar_arrive_expect_tx(fb, bytes * NBUF);
                            bulk_load(dst, in0 + body + c0 * VEC, bytes, fb,
                                      pass == 0 ? keep : stream);
                            if constexpr (NBUF == 2)
                                bulk_load(dst + kChunkBytes, in1 + body + c0 * VEC, bytes, fb,
                                          pass == 0 ? keep : stream);
                            filled |= 1u << slot;
                            fill_ph = (fill_ph & ~(1u << slot)) | (ph << slot);
                        }
                        ++issued;
                        if (++slot == static_cast<uint32_t>(nslot)) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            // Every copy issued here lands before the CTA may exit (consumers
            // that gave up no longer wait for them): the last fill of each slot
            // completes the phase recorded for it (a left-out fill records
            // nothing; the slot's earlier fill, if any, has long landed).  A
            // fixed budget bounds the whole drain.
            const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
            for (int s = 0; s < nslot; ++s)
                if ((filled >> s) & 1u)
                    mbar_wait_until(smem_addr(&full[s]), (fill_ph >> s) & 1u, deadline);
        }
    } else {
        // ------------------------------------------------------------ consumers
        // Thread tid owns vectors tid + v * NC (v < VPT) of every chunk: VPT
        // independent 128-bit shared loads per chunk, issued back to back.
        uint32_t slot = 0, ph = 0, xph = 0;
        int live = 0;
        bool ok = true;
        if constexpr (OP == Op::CE)
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // n (from the count kernel) is first needed by a row's pass 2: pass 1 of
        // the first row overlaps the count kernel
        bool have_n = OP != Op::CE;
        float nf = 1.f;
        int64_t ynext = (OP == Op::CE && cid < M) ? a.targets[cid] : 0;
        for (int row = cid; row < M; row += G) {
            const int64_t y = ynext;  // loaded one row ahead
            if (OP == Op::CE && row + G < M)
                ynext = a.targets[row + G];
            const T *in0 = static_cast<const T *>(a.in0) + row * a.s0;
            const T *in1 = nullptr;
            if constexpr (NBUF == 2)
                in1 = static_cast<const T *>(a.in1) + row * a.s1;
            T *out = static_cast<T *>(a.out) + row * a.so;
            const RowGeom g = row_geom(in0, a.cols);
            const int nvec = static_cast<int>(g.nvec);
            const int tail_start = static_cast<int>(g.tail_start);
            const int per = (nvec + C - 1) / C;
            const int v0 = rank * per;
            const int cnt = v0 < nvec ? (v0 + per < nvec ? per : nvec - v0) : 0;
            const int body = g.head + v0 * VEC;
            const bool head_here = rank == 0 && tid < g.head;
            const bool tail_here = rank == C - 1 && tid < g.tail;
            uint4 *o = reinterpret_cast<uint4 *>(out + body);
            if constexpr (OP == Op::CE) {
                if (y == a.ignore_index) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    for (int j = tid; j < cnt; j += NC)
                        __stcs(o + j, z);
                    if (head_here)
                        E::store(out + tid, 0.f);
                    if (tail_here)
                        E::store(out + tail_start + tid, 0.f);
                    if (rank == 0 && tid == 0)
                        a.row_loss[row] = 0.f;
                    continue;
                }
                if (y < 0 || y >= a.cols) {
                    if (rank == 0 && tid == 0) {
                        a.row_loss[row] = __int_as_float(0x7fc00000);
                        atomicOr(&g_flags, kFlagBadTarget);
                    }
                    continue;
                }
            }
            const int nch = (cnt + CHUNK - 1) / CHUNK;
            if (HOLD && 2 * nch > nslot) {  // cannot happen for a valid plan: flag, skip
                if (tid == 0) {
                    atomicOr(&g_flags, kFlagTimeout);
                    if (OP == Op::CE && rank == 0)
                        a.row_loss[row] = __int_as_float(0x7fc00000);
                }
                continue;
            }
            constexpr bool hold = HOLD;  // loaded once, kept for pass 2
            const uint32_t slot0 = slot, ph0 = ph;
            float h0 = 0.f, h1 = 0.f, t0 = 0.f, t1 = 0.f;
            if (head_here) {
                h0 = E::load(in0 + tid);
                if constexpr (NBUF == 2)
                    h1 = E::load(in1 + tid);
            }
            if (tail_here) {
                t0 = E::load(in0 + tail_start + tid);
                if constexpr (NBUF == 2)
                    t1 = E::load(in1 + tail_start + tid);
            }
            float xy = 0.f;
            if constexpr (OP == Op::CE) {
                if (rank == 0 && tid == 0)
                    xy = E::load(in0 + y);  // completes before this row's partial is published
            }

            // ---- pass 1: online over the chunks as they arrive
            float pa, pb;
            if constexpr (OP == Op::SoftmaxBwd) {
                float sdot = 0.f;
                for (int kk = 0; kk < nch; ++kk) {
                    const int c0 = kk * CHUNK;
                    const int cn = (c0 + CHUNK < cnt ? c0 + CHUNK : cnt) - c0;
                    if (ok)
                        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&full[slot]), ph));
                    if (ok) {
                        const uint32_t b0 = ring + slot * kSlotBytes;
                        uint4 ry[VPT], rd[VPT];
#pragma unroll
                        for (int v = 0; v < VPT; ++v) {
                            const int j = tid + v * NC;
                            if (j < cn) {
                                ry[v] = ld_shared_v4(b0 + j * 16u);
                                rd[v] = ld_shared_v4(b0 + kChunkBytes + j * 16u);
                            }
                        }
#pragma unroll
                        for (int v = 0; v < VPT; ++v) {
                            if (tid + v * NC < cn) {
                                float fy[VEC], fd[VEC];
                                E::unpack(ry[v], fy);
                                E::unpack(rd[v], fd);
#pragma unroll
                                for (int e = 0; e < VEC; ++e)
                                    sdot = fmaf(fy[e], fd[e], sdot);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0 && ok && !hold)  // a warp that gave up stops releasing slots
                        mbar_arrive(smem_addr(&empty[slot]));
                    if (++slot == static_cast<uint32_t>(nslot)) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
                // head and tail, loaded at the row start, are added after the chunks:
                // their load latency hides behind the chunk waits instead of delaying them
                if (head_here)
                    sdot = fmaf(h0, h1, sdot);
                if (tail_here)
                    sdot = fmaf(t0, t1, sdot);
                pa = sdot;
                pb = 0.f;
            } else {
                float m = -INFINITY, d = 0.f;  // running shift (log2 units) and sum
                for (int kk = 0; kk < nch; ++kk) {
                    const int c0 = kk * CHUNK;
                    const int cn = (c0 + CHUNK < cnt ? c0 + CHUNK : cnt) - c0;
                    if (ok)
                        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&full[slot]), ph));
                    // A full chunk (every one but a slice's last) needs no per-vector
                    // bound.  Only the clustered instances (128 registers) take that
                    // unchecked path: in the 96-register unclustered ones the second
                    // copy of the loop cost 3% (measured), while the clustered fp32
                    // rows gained 1.7%.
                    auto chunk1 = [&](auto full_tag) {
                        constexpr bool FULL = decltype(full_tag)::value;
                        const uint32_t b0 = ring + slot * kSlotBytes;
                        uint4 raw[VPT];
#pragma unroll
                        for (int v = 0; v < VPT; ++v) {
                            const int j = tid + v * NC;
                            // a vector past the slice end reads as -inf pairs (fp32 code skips it)
                            raw[v] = (FULL || j < cn) ? ld_shared_v4(b0 + j * 16u)
                                                      : make_uint4(E::kNegInfPair, E::kNegInfPair,
                                                                   E::kNegInfPair, E::kNegInfPair);
                        }
                        // the chunk's max first (packed pairs for bf16), then one rescale and the sum
                        float cm = -INFINITY;
                        if constexpr (VEC == 8) {
                            uint32_t mm = E::kNegInfPair;
#pragma unroll
                            for (int v = 0; v < VPT; ++v)
                                mm = E::max2(E::max2(mm, raw[v].x),
                                             E::max2(raw[v].y, E::max2(raw[v].z, raw[v].w)));
                            cm = E::pair_max(mm);
                        } else {
#pragma unroll
                            for (int v = 0; v < VPT; ++v) {
                                if (FULL || tid + v * NC < cn) {
                                    float f[VEC];
                                    E::unpack(raw[v], f);
#pragma unroll
                                    for (int e = 0; e < VEC; ++e)
                                        cm = fmaxf(cm, f[e]);
                                }
                            }
                        }
                        // the running shift in log2 units: fl(x log2 e) is monotonic,
                        // so the shift of the larger maximum is the larger shift
                        const float mn = fmaxf(m, shift_of(cm));
                        if (mn != -INFINITY) {
                            float s = 0.f;
#pragma unroll
                            for (int v = 0; v < VPT; ++v) {
                                if (FULL || tid + v * NC < cn) {
                                    float f[VEC];
                                    E::unpack(raw[v], f);
#pragma unroll
                                    for (int e = 0; e < VEC; ++e)
                                        s += exp2_shift(f[e], mn);
                                }
                            }
                            d = d * exp2f(m - mn) + s;
                            m = mn;
                        }
                    };
                    if (ok) {
                        if (CLUSTER && cn == CHUNK)
                            chunk1(std::integral_constant<bool, CLUSTER>{});
                        else
                            chunk1(std::false_type{});
                    }
                    __syncwarp();
                    if (lane == 0 && ok && !hold)
                        mbar_arrive(smem_addr(&empty[slot]));
                    if (++slot == static_cast<uint32_t>(nslot)) {
                        slot = 0;
                        ph ^= 1u;
                    }
                }
                // head and tail, loaded at the row start, are merged after the chunks:
                // their load latency hides behind the chunk waits instead of delaying them
                float hm = -INFINITY;
                if (head_here)
                    hm = h0;
                if (tail_here)
                    hm = fmaxf(hm, t0);
                if (hm != -INFINITY) {
                    const float hL = shift_of(hm);
                    float hd = 0.f;
                    if (head_here)
                        hd += exp2_shift(h0, hL);
                    if (tail_here)
                        hd += exp2_shift(t0, hL);
                    md_merge(m, d, hL, hd);
                }
                pa = m;
                pb = d;
            }

            // ---- merge across the consumer warps; a row is good only if every
            // warp's waits succeeded up to here (a warp that gave up stays out)
            P::warp_reduce(pa, pb);
            if (lane == 0) {
                red[warp] = make_float2(pa, pb);
                wbad[warp] = ok ? 0 : 1;
            }
            named_barrier_sync(1, NC);
            if (warp == 0) {
                const float2 e = P::empty();
                pa = lane < NCW ? red[lane].x : e.x;
                pb = lane < NCW ? red[lane].y : e.y;
                const bool bad = __any_sync(0xffffffffu, lane < NCW && wbad[lane] != 0);
                P::warp_reduce(pa, pb);
                if (lane == 0)
                    fin = make_float4(pa, pb, bad ? 1.f : 0.f, 0.f);
            }
            named_barrier_sync(1, NC);
            float4 r = fin;

            // ---- merge across the cluster: each CTA sends its partial to every
            // peer's slot (st.async, counted on the peer's exchange barrier) and
            // folds the C partials in rank order, so all CTAs get the same bits.
            if constexpr (CLUSTER) {
                const int pi = live & 1;
                if (tid == 0) {
                    asm volatile("" ::"f"(xy));  // the target logit was read before peers store
                    mbar_arrive_expect_tx(smem_addr(&xbar[pi]), 16u * static_cast<uint32_t>(C - 1));
                    const uint32_t slot_addr = smem_addr(&xslot[pi][rank]);
                    const uint32_t bar_addr = smem_addr(&xbar[pi]);
                    for (int q = 0; q < C; ++q)
                        if (q != rank)
                            st_async_f4(map_to_rank(slot_addr, q), r, map_to_rank(bar_addr, q));
                }
                bool xok = ok;
                if (xok)
                    xok = __all_sync(0xffffffffu,
                                     mbar_wait_bounded(smem_addr(&xbar[pi]), (xph >> pi) & 1u));
                xph ^= 1u << pi;
                const float2 e = P::empty();
                float qa = e.x, qb = e.y, qf = xok ? 0.f : 1.f;
                for (int q = 0; q < C; ++q) {
                    const float4 v = q == rank ? r : xslot[pi][q];
                    P::merge(qa, qb, v.x, v.y);
                    qf += v.z;
                }
                r = make_float4(qa, qb, qf, 0.f);
                ok = ok && xok;
            }
            ++live;

            // ---- pass 2: the slice again (the same slots when held, else a
            // second read that L2 serves), chunks in order
            float scale = 0.f, sub = 0.f;
            if constexpr (OP == Op::CE) {
                if (!have_n) {
                    wait_prerequisite_grid();
                    nf = static_cast<float>(*a.n_ptr);
                    have_n = true;
                }
            }
            if constexpr (OP != Op::SoftmaxBwd) {
                if constexpr (OP == Op::CE)
                    ce_row_factor(a, row, r.y, nf, scale, sub);
                else
                    scale = 1.f / r.y;
            }
            const bool all_ok = r.z == 0.f;
            const int ycol = static_cast<int>(y) - body;  // y is in [0, cols) here
            // the vector of the slice that holds the target, and its element (-1:
            // none here); the clustered instances test that index per vector
            const int yv = ycol >= 0 ? ycol / VEC : -1;
            const int ye = ycol - yv * VEC;
            if (hold) {  // revisit the slots pass 1 read
                slot = slot0;
                ph = ph0;
            }
            for (int kk = 0; kk < nch; ++kk) {
                const int c0 = kk * CHUNK;
                const int cn = (c0 + CHUNK < cnt ? c0 + CHUNK : cnt) - c0;
                if (ok && !hold)
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&full[slot]), ph));
                auto chunk2 = [&](auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
                    const uint32_t b0 = ring + slot * kSlotBytes;
                    uint4 raw[VPT];
                    [[maybe_unused]] uint4 raw2[VPT];  // the second operand (softmax backward)
#pragma unroll
                    for (int v = 0; v < VPT; ++v) {
                        const int j = tid + v * NC;
                        if (FULL || j < cn) {
                            raw[v] = ld_shared_v4(b0 + j * 16u);
                            if constexpr (NBUF == 2)
                                raw2[v] = ld_shared_v4(b0 + kChunkBytes + j * 16u);
                        }
                    }
#pragma unroll
                    for (int v = 0; v < VPT; ++v) {
                        const int j = tid + v * NC;
                        if (!FULL && j >= cn)
                            continue;
                        const int vj = c0 + j;  // vector index within the slice
                        if constexpr (OP == Op::SoftmaxBwd) {
                            float fy[VEC], fd[VEC];
                            E::unpack(raw[v], fy);
                            E::unpack(raw2[v], fd);
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                fy[e] = fy[e] * (fd[e] - r.x);
                            o[vj] = E::pack(fy);
                        } else {
                            float f[VEC];
                            E::unpack(raw[v], f);
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                f[e] = exp2_shift(f[e], r.x);
                            float gr[VEC];
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                gr[e] = f[e] * scale;
                            if constexpr (OP == Op::CE) {
                                if constexpr (CLUSTER) {
                                    if (vj == yv) {  // the target column: (p_y - 1) / n
#pragma unroll
                                        for (int e = 0; e < VEC; ++e)
                                            if (e == ye)
                                                gr[e] = fmaf(f[e], scale, -sub);
                                    }
                                } else {
                                    const int rel = ycol - vj * VEC;
                                    if (rel >= 0 && rel < VEC) {  // the target column: (p_y - 1) / n
#pragma unroll
                                        for (int e = 0; e < VEC; ++e)
                                            if (e == rel)
                                                gr[e] = fmaf(f[e], scale, -sub);
                                    }
                                }
                            }
                            o[vj] = E::pack(gr);
                        }
                    }
                };
                if (ok && all_ok) {
                    if (CLUSTER && cn == CHUNK)
                        chunk2(std::integral_constant<bool, CLUSTER>{});
                    else
                        chunk2(std::false_type{});
                }
                __syncwarp();
                if (lane == 0 && ok)
                    mbar_arrive(smem_addr(&empty[slot]));
                if (++slot == static_cast<uint32_t>(nslot)) {
                    slot = 0;
                    ph ^= 1u;
                }
            }
            if (ok && all_ok) {
                if constexpr (OP == Op::SoftmaxBwd) {
                    if (head_here)
                        E::store(out + tid, h0 * (h1 - r.x));
                    if (tail_here)
                        E::store(out + tail_start + tid, t0 * (t1 - r.x));
                } else {
                    if (head_here) {
                        const float ex = exp2_shift(h0, r.x);
                        E::store(out + tid,
                                 (OP == Op::CE && y == tid) ? fmaf(ex, scale, -sub) : ex * scale);
                    }
                    if (tail_here) {
                        const float ex = exp2_shift(t0, r.x);
                        E::store(out + tail_start + tid,
                                 (OP == Op::CE && y == tail_start + tid) ? fmaf(ex, scale, -sub)
                                                                            : ex * scale);
                    }
                    if constexpr (OP == Op::CE) {
                        if (rank == 0 && tid == 0)
                            a.row_loss[row] = row_loss_from(r.x, r.y, xy);
                    }
                }
            } else if (tid == 0) {
                raise_timeout(a.fail);
                if constexpr (OP == Op::CE) {
                    if (rank == 0)
                        a.row_loss[row] = __int_as_float(0x7fc00000);
                }
            }
        }
        if constexpr (OP == Op::CE) {
            if (!have_n)  // the count kernel has cleared the failure word; see ce_row_exit_order
                wait_prerequisite_grid();
        }
        if (!ok && lane == 0)  // this warp gave up (perhaps in a last pass 2 no row vote saw)
            raise_timeout(a.fail);
        if constexpr (CLUSTER) {
            // a CTA that gave up stopped waiting for its peers' partials: let the
            // last one of each exchange barrier land before the CTA may exit
            if (tid == 0 && live > 0) {
                const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
                for (int pi = 0; pi < 2 && pi < live; ++pi)
                    mbar_wait_until(smem_addr(&xbar[pi]), ((xph >> pi) & 1u) ^ 1u, deadline);
            }
        }
    }
    if constexpr (CLUSTER) {  // no CTA leaves while a peer may still signal it
        cluster_arrive_any();
        cluster_wait_any();
    }
}

// ---------------------------------------------------------------------------
// General fallback for rows whose operands do not share a 16-byte phase or
// whose slices would not fit in shared memory: the same cluster-per-row
// reduction, with plain element loads from global memory (the row is read
// from HBM / L2 in every pass).
template <Op OP, typename T, int NT>
__global__ void __launch_bounds__(NT) rows_streaming_kernel(const RowArgs a)
{
    using E = Elem<T>;
    using P = Partial<OP>;
    constexpr int NW = NT / 32;
    __shared__ float2 red[NW];
    __shared__ __align__(16) float4 part;
    __shared__ float4 fin;

    const int C = a.C;
    const int64_t row = blockIdx.x / C;
    const int rank = C > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if constexpr (OP == Op::CE)  // the mean kernel may be scheduled (it waits for this grid)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const T *in0 = static_cast<const T *>(a.in0) + row * a.s0;
    const T *in1 = OP == Op::SoftmaxBwd ? static_cast<const T *>(a.in1) + row * a.s1 : nullptr;
    T *out = static_cast<T *>(a.out) + row * a.so;
    const int64_t per = (a.cols + C - 1) / C;
    const int64_t e0 = rank * per;
    const int64_t e1 = e0 + per < a.cols ? e0 + per : a.cols;

    int64_t y = -1;
    if constexpr (OP == Op::CE) {
        y = a.targets[row];
        if (y == a.ignore_index) {
            for (int64_t i = e0 + tid; i < e1; i += NT)
                E::store(out + i, 0.f);
            if (rank == 0 && tid == 0)
                a.row_loss[row] = 0.f;
            wait_prerequisite_grid();  // see ce_row_exit_order
            return;
        }
        if (y < 0 || y >= a.cols) {
            if (rank == 0 && tid == 0) {
                a.row_loss[row] = __int_as_float(0x7fc00000);
                atomicOr(&g_flags, kFlagBadTarget);
            }
            wait_prerequisite_grid();
            return;
        }
    }
    float xy = 0.f;
    if constexpr (OP == Op::CE) {
        if (rank == 0 && tid == 0)
            xy = E::load(in0 + y);
    }
    float pa, pb;
    if constexpr (OP == Op::SoftmaxBwd) {
        float s = 0.f;
        for (int64_t i = e0 + tid; i < e1; i += NT)
            s = fmaf(E::load(in0 + i), E::load(in1 + i), s);
        pa = s;
        pb = 0.f;
    } else {
        float m = -INFINITY;
        for (int64_t i = e0 + tid; i < e1; i += NT)
            m = fmaxf(m, E::load(in0 + i));
        const float sL = (m == -INFINITY) ? 0.f : shift_of(m);  // all -inf: every term 0
        float d = 0.f;
        for (int64_t i = e0 + tid; i < e1; i += NT)
            d += exp2_shift(E::load(in0 + i), sL);
        pa = shift_of(m);  // (shift, sum) partial; (-inf, 0) when empty
        pb = d;
    }
    P::warp_reduce(pa, pb);
    if (lane == 0)
        red[warp] = make_float2(pa, pb);
    __syncthreads();
    if (warp == 0) {
        const float2 e = P::empty();
        pa = lane < NW ? red[lane].x : e.x;
        pb = lane < NW ? red[lane].y : e.y;
        P::warp_reduce(pa, pb);
        if (lane == 0)
            part = make_float4(pa, pb, 0.f, 0.f);
    }
    __syncthreads();
    float4 r;
    if (C > 1) {
        cluster_arrive();
        cluster_wait();
        if (warp == 0) {
            const float2 e = P::empty();
            float qa = e.x, qb = e.y;
            if (lane < C) {
                const float2 ab =
                    ld_cluster_f2(map_to_rank(smem_addr(&part), static_cast<uint32_t>(lane)));
                qa = ab.x;
                qb = ab.y;
            }
            P::warp_reduce(qa, qb);
            if (lane == 0)
                fin = make_float4(qa, qb, 0.f, 0.f);
        }
        cluster_arrive();
        __syncthreads();
        r = fin;
    } else {
        r = part;
    }
    if constexpr (OP == Op::SoftmaxBwd) {
        for (int64_t i = e0 + tid; i < e1; i += NT) {
            const float yv = E::load(in0 + i);
            E::store(out + i, yv * (E::load(in1 + i) - r.x));
        }
    } else {
        float scale, sub = 0.f;
        if constexpr (OP == Op::CE) {
            wait_prerequisite_grid();  // n comes from the count kernel
            ce_row_factor(a, row, r.y, static_cast<float>(*a.n_ptr), scale, sub);
        } else {
            scale = 1.f / r.y;
        }
        // Read every element before this thread overwrites it (in place for CE);
        // each element is read and written by the same thread only.
        for (int64_t i = e0 + tid; i < e1; i += NT) {
            const float ex = exp2_shift(E::load(in0 + i), r.x);
            E::store(out + i, (OP == Op::CE && i == y) ? fmaf(ex, scale, -sub) : ex * scale);
        }
        if constexpr (OP == Op::CE) {
            if (rank == 0 && tid == 0)
                a.row_loss[row] = row_loss_from(r.x, r.y, xy);
        }
    }
    if (C > 1)
        cluster_wait();
}

// ---------------------------------------------------------------------------
// n = number of targets != ignore_index (one CTA); flags targets outside [0, V);
// for M == 0 writes the reduced loss itself (mean 0/0 = NaN, sum 0).  It lets the row kernel launch
// at once (programmatic dependent launch); the row kernel waits for it on the
// device before it reads n.
template <int NT>
__global__ void __launch_bounds__(NT) ce_count_kernel(const int64_t *targets, int64_t M, int64_t V,
                                                      int64_t ignore_index, int *n_out,
                                                      unsigned *fail, float *loss, int reduction)
{
    __shared__ int warp_n[NT / 32];
    __shared__ int any_bad;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0)
        any_bad = 0;
    __syncthreads();
    int n = 0;
    bool bad = false;
#pragma unroll 16
    for (int64_t i = threadIdx.x; i < M; i += NT) {
        const int64_t y = targets[i];
        if (y != ignore_index) {
            ++n;
            bad |= (y < 0 || y >= V);
        }
    }
    if (bad)
        any_bad = 1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        n += __shfl_xor_sync(0xffffffffu, n, off);
    if ((threadIdx.x & 31) == 0)
        warp_n[threadIdx.x >> 5] = n;
    __syncthreads();
    if (threadIdx.x < 32) {
        n = threadIdx.x < NT / 32 ? warp_n[threadIdx.x] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            n += __shfl_xor_sync(0xffffffffu, n, off);
        if (threadIdx.x == 0) {
            *n_out = n;
            *fail = 0u;  // no wait of this call has given up yet
            if (M == 0 && reduction != kReduceNone)  // the mean of nothing is 0/0, the sum 0
                *loss = reduction == kReduceMean ? __int_as_float(0x7fc00000) : 0.f;
            if (any_bad)
                atomicOr(&g_flags, kFlagBadTarget);
        }
    }
}

// L = sum_r row_loss[r] / n after the row kernel (one CTA; launched as its
// programmatic dependent, it waits for the row kernel to complete first).
// NaN when a bounded wait of the call gave up (its failure word is set).
template <int NT>
__global__ void __launch_bounds__(NT) ce_mean_kernel(const float *row_loss, int64_t M,
                                                     const int *n_ptr, const unsigned *fail,
                                                     float *loss, int reduction)
{
    wait_prerequisite_grid();
    const float s = sum_row_losses<NT>(row_loss, M, threadIdx.x, 1);
    if (threadIdx.x == 0) {
        const float L = reduction == kReduceMean ? s / static_cast<float>(__ldcg(n_ptr)) : s;
        *loss = __ldcg(fail) ? __int_as_float(0x7fc00000) : L;
    }
}

// x[r, :N] *= scale[per_row ? r : 0], in place (Liger-Kernel cross_entropy.py,
// element_mul, applied by LigerCrossEntropyFunction.backward when grad_output
// is not 1).  A single scale of exactly 1 returns at once on the device, so
// the caller needs no host-side test of grad_output.
template <typename T, int NT>
__global__ void __launch_bounds__(NT) scale_rows_kernel(void *x, int64_t stride, int64_t M,
                                                        int64_t N, const float *scale, int per_row)
{
    using E = Elem<T>;
    constexpr int VEC = E::kPerVec;
    if (!per_row && __ldg(scale) == 1.f)
        return;
    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const float sc = __ldg(scale + (per_row ? r : 0));
        T *row = static_cast<T *>(x) + r * stride;
        const RowGeom g = row_geom(row, N);
        if (static_cast<int>(threadIdx.x) < g.head)
            E::store(row + threadIdx.x, E::load(row + threadIdx.x) * sc);
        if (static_cast<int>(threadIdx.x) < g.tail)
            E::store(row + g.tail_start + threadIdx.x, E::load(row + g.tail_start + threadIdx.x) * sc);
        uint4 *v = reinterpret_cast<uint4 *>(row + g.head);
        for (int64_t j = threadIdx.x; j < g.nvec; j += NT) {
            float f[VEC];
            E::unpack(__ldcs(v + j), f);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                f[e] *= sc;
            __stcs(v + j, E::pack(f));
        }
    }
}

}  // namespace gbce
