// Row kernels: fused cross-entropy forward+backward, softmax forward, softmax
// backward.  One thread-block cluster of C CTAs handles one row; each CTA
// stages its contiguous slice of the row in shared memory with 1-D bulk (TMA)
// copies, so the row is read from HBM once and written once.
//
// Per row (cross-entropy; the softmax forward is the same without the target):
//   1. target load and ignore test (Liger-Kernel cross_entropy.py,
//      liger_cross_entropy_kernel, steps 1-2).  Ignored rows are zero-filled
//      with no read; a target outside [0, V) raises a flag and leaves the row.
//   2. pass 1, the online normaliser (same kernel, step 3, "Algorithm 3" of
//      the online-softmax paper it cites): each thread takes the max m of its
//      elements, then d = sum exp(x - m); the (m, d) pairs are merged by warp
//      shuffles, through shared memory, then across the cluster over
//      distributed shared memory, rescaling each sum to the larger max.
//   3. pass 2, the gradient in place (step 4 and step 6):
//      g_i = exp(x_i - M) / (D n), and (exp(x_y - M)/D - 1)/n at the target,
//      computed from the staged copy, so the second pass does not touch HBM.
//   4. the row loss M + ln D - x_y (step 5), x_y captured before any store.
#pragma once

#include "device.cuh"

namespace gbce {

constexpr int kMaxChunks = 8;  // bulk copies (one mbarrier each) per CTA slice

enum class Op { CE, SoftmaxFwd, SoftmaxBwd };

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
    // launch plan
    int C;          // CTAs per row (cluster size)
    int per_vec;    // 16-byte vectors per CTA slice (capacity of one staged buffer)
    int chunk_vec;  // vectors per bulk copy, a multiple of the CTA's thread count
};

// Sticky error flags of this device (kFlag* bits); defined once per library.
__device__ unsigned int g_flags = 0;

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

template <Op OP, typename T, int NT>
__global__ void __launch_bounds__(NT, 1536 / NT) rows_resident_kernel(const RowArgs a)
{
    using E = Elem<T>;
    using P = Partial<OP>;
    constexpr int VEC = E::kPerVec;
    constexpr int NW = NT / 32;
    constexpr int NBUF = (OP == Op::SoftmaxBwd) ? 2 : 1;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kMaxChunks];
    __shared__ float2 red[NW];
    __shared__ __align__(16) float4 part;  // this CTA's (a, b, failed): read by cluster peers
    __shared__ float4 fin;

    const int C = a.C;
    const int64_t row = blockIdx.x / C;
    const int rank = C > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;

    const T *in0 = static_cast<const T *>(a.in0) + row * a.s0;
    const T *in1 = nullptr;
    if constexpr (NBUF == 2)
        in1 = static_cast<const T *>(a.in1) + row * a.s1;
    T *out = static_cast<T *>(a.out) + row * a.so;

    // Every operand of a row shares this geometry (the host checks that their
    // row starts agree modulo 16 bytes).
    const RowGeom g = row_geom(in0, a.cols);
    const int64_t v0 = static_cast<int64_t>(rank) * a.per_vec;
    const int64_t vend = v0 + a.per_vec < g.nvec ? v0 + a.per_vec : g.nvec;
    const int cnt = vend > v0 ? static_cast<int>(vend - v0) : 0;
    const int64_t body = g.head + v0 * VEC;  // column of this CTA's first vector
    const bool head_here = rank == 0 && tid < g.head;
    const bool tail_here = rank == C - 1 && tid < g.tail;

    int64_t y = -1;
    if constexpr (OP == Op::CE) {
        y = a.targets[row];
        if (y == a.ignore_index) {
            // ignored row: zero gradient, zero loss, nothing read
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            uint4 *o = reinterpret_cast<uint4 *>(out + body);
            for (int j = tid; j < cnt; j += NT)
                __stcs(o + j, z);
            if (head_here)
                E::store(out + tid, 0.f);
            if (tail_here)
                E::store(out + g.tail_start + tid, 0.f);
            if (rank == 0 && tid == 0)
                a.row_loss[row] = 0.f;
            return;
        }
        if (y < 0 || y >= a.cols) {
            // out-of-range target: flag it, NaN loss, leave the row as it is
            if (rank == 0 && tid == 0) {
                a.row_loss[row] = __int_as_float(0x7fc00000);
                atomicOr(&g_flags, kFlagBadTarget);
            }
            return;
        }
    }

    // ---- issue the bulk copies of this CTA's slice (one mbarrier per chunk)
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
        for (int k = 0; k < nch; ++k) {
            const int c0 = k * a.chunk_vec;
            const int c1 = c0 + a.chunk_vec < cnt ? c0 + a.chunk_vec : cnt;
            const uint32_t bytes = static_cast<uint32_t>(c1 - c0) * 16u;
            const uint32_t bar = smem_addr(&bars[k]);
            mbar_arrive_expect_tx(bar, bytes * NBUF);
            bulk_load(buf0 + c0 * 16u, in0 + body + static_cast<int64_t>(c0) * VEC, bytes, bar, pol);
            if constexpr (NBUF == 2)
                bulk_load(buf1 + c0 * 16u, in1 + body + static_cast<int64_t>(c0) * VEC, bytes, bar,
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
    float xy = 0.f;  // the target logit, read before this cluster stores anything
    if constexpr (OP == Op::CE) {
        if (rank == 0 && tid == 0)
            xy = E::load(in0 + y);
    }

    // ---- pass 1
    bool ok = true;
    float pa, pb;  // (m, d) for CE / softmax fwd, (sum y*dy, unused) for softmax bwd
    if constexpr (OP == Op::SoftmaxBwd) {
        float s = 0.f;
        if (head_here)
            s = fmaf(h0, h1, s);
        if (tail_here)
            s = fmaf(t0, t1, s);
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
                        s = fmaf(fy[e], fd[e], s);
                }
            }
        }
        pa = s;
        pb = 0.f;
    } else {
        float m = -INFINITY;
        if (head_here)
            m = fmaxf(m, h0);
        if (tail_here)
            m = fmaxf(m, t0);
        for (int k = 0; k < nch && ok; ++k) {
            ok = mbar_wait_bounded(smem_addr(&bars[k]), 0);
            const int c1 = (k + 1) * a.chunk_vec < cnt ? (k + 1) * a.chunk_vec : cnt;
            if (ok) {
                for (int j = k * a.chunk_vec + tid; j < c1; j += NT) {
                    float f[VEC];
                    E::unpack(ld_shared_v4(buf0 + j * 16u), f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        m = fmaxf(m, f[e]);
                }
            }
        }
        // every chunk has landed once the loop above completed for all threads
        ok = __syncthreads_and(ok);
        float d = 0.f;
        if (ok) {
            const float mL = (m == -INFINITY) ? 0.f : m * kLog2e;
            for (int j = tid; j < cnt; j += NT) {
                float f[VEC];
                E::unpack(ld_shared_v4(buf0 + j * 16u), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    d += exp2f(fmaf(f[e], kLog2e, -mL));
            }
            if (head_here)
                d += exp2f(fmaf(h0, kLog2e, -mL));
            if (tail_here)
                d += exp2f(fmaf(t0, kLog2e, -mL));
        }
        pa = m;
        pb = d;
    }
    if constexpr (OP == Op::SoftmaxBwd)
        ok = __syncthreads_and(ok);

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
            part = make_float4(pa, pb, ok ? 0.f : 1.f, 0.f);
    }
    __syncthreads();

    // ---- cluster reduction over distributed shared memory
    float4 r;
    if (C > 1) {
        cluster_arrive();
        cluster_wait();  // every CTA's `part` is now visible
        if (warp == 0) {
            const float2 e = P::empty();
            float qa = e.x, qb = e.y, qf = 0.f;
            if (lane < C) {
                const uint32_t peer = map_to_rank(smem_addr(&part), static_cast<uint32_t>(lane));
                const float2 ab = ld_cluster_f2(peer);
                const float2 fl = ld_cluster_f2(peer + 8u);
                qa = ab.x;
                qb = ab.y;
                qf = fl.x;
            }
            P::warp_reduce(qa, qb);
            qf = warp_sum(qf);
            if (lane == 0)
                fin = make_float4(qa, qb, qf, 0.f);
        }
        cluster_arrive();  // done reading peers; the matching wait precedes exit
        __syncthreads();
        r = fin;
    } else {
        r = part;
    }
    const bool all_ok = r.z == 0.f;

    // ---- pass 2: results from the staged copy, one store per element
    if (all_ok) {
        uint4 *o = reinterpret_cast<uint4 *>(out + body);
        if constexpr (OP == Op::SoftmaxBwd) {
            const float s = r.x;
            for (int j = tid; j < cnt; j += NT) {
                float fy[VEC], fd[VEC];
                E::unpack(ld_shared_v4(buf0 + j * 16u), fy);
                E::unpack(ld_shared_v4(buf1 + j * 16u), fd);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    fy[e] = fy[e] * (fd[e] - s);
                __stcs(o + j, E::pack(fy));
            }
            if (head_here)
                E::store(out + tid, h0 * (h1 - s));
            if (tail_here)
                E::store(out + g.tail_start + tid, t0 * (t1 - s));
        } else {
            const float M = r.x, D = r.y;
            const float ML = M * kLog2e;
            float scale, sub = 0.f;
            if constexpr (OP == Op::CE) {
                const float n = static_cast<float>(*a.n_ptr);
                scale = 1.f / (D * n);
                sub = 1.f / n;
            } else {
                scale = 1.f / D;
            }
            const int64_t ycol = y - body;  // target position relative to this slice
            for (int j = tid; j < cnt; j += NT) {
                float f[VEC];
                E::unpack(ld_shared_v4(buf0 + j * 16u), f);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    f[e] = exp2f(fmaf(f[e], kLog2e, -ML));
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
                const float ex = exp2f(fmaf(h0, kLog2e, -ML));
                E::store(out + tid, (OP == Op::CE && y == tid) ? fmaf(ex, scale, -sub) : ex * scale);
            }
            if (tail_here) {
                const float ex = exp2f(fmaf(t0, kLog2e, -ML));
                E::store(out + g.tail_start + tid,
                         (OP == Op::CE && y == g.tail_start + tid) ? fmaf(ex, scale, -sub)
                                                                    : ex * scale);
            }
            if constexpr (OP == Op::CE) {
                if (rank == 0 && tid == 0)
                    a.row_loss[row] = M + logf(D) - xy;
            }
        }
    } else {
        if (tid == 0) {
            atomicOr(&g_flags, kFlagTimeout);
            // give copies still in flight a bounded chance to land before exit
            for (int k = 0; k < nch; ++k)
                mbar_wait_bounded(smem_addr(&bars[k]), 0);
        }
        if constexpr (OP == Op::CE) {
            if (rank == 0 && tid == 0)
                a.row_loss[row] = __int_as_float(0x7fc00000);
        }
    }
    if (C > 1)
        cluster_wait();
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
            return;
        }
        if (y < 0 || y >= a.cols) {
            if (rank == 0 && tid == 0) {
                a.row_loss[row] = __int_as_float(0x7fc00000);
                atomicOr(&g_flags, kFlagBadTarget);
            }
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
        const float mL = (m == -INFINITY) ? 0.f : m * kLog2e;
        float d = 0.f;
        for (int64_t i = e0 + tid; i < e1; i += NT)
            d += exp2f(fmaf(E::load(in0 + i), kLog2e, -mL));
        pa = m;
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
        const float ML = r.x * kLog2e;
        float scale, sub = 0.f;
        if constexpr (OP == Op::CE) {
            const float n = static_cast<float>(*a.n_ptr);
            scale = 1.f / (r.y * n);
            sub = 1.f / n;
        } else {
            scale = 1.f / r.y;
        }
        // Read every element before this thread overwrites it (in place for CE);
        // each element is read and written by the same thread only.
        for (int64_t i = e0 + tid; i < e1; i += NT) {
            const float ex = exp2f(fmaf(E::load(in0 + i), kLog2e, -ML));
            E::store(out + i, (OP == Op::CE && i == y) ? fmaf(ex, scale, -sub) : ex * scale);
        }
        if constexpr (OP == Op::CE) {
            if (rank == 0 && tid == 0)
                a.row_loss[row] = r.x + logf(r.y) - xy;
        }
    }
    if (C > 1)
        cluster_wait();
}

// ---------------------------------------------------------------------------
// n = number of targets != ignore_index (one CTA); flags targets outside [0, V).
template <int NT>
__global__ void __launch_bounds__(NT) ce_count_kernel(const int64_t *targets, int64_t M, int64_t V,
                                                      int64_t ignore_index, int *n_out)
{
    __shared__ int warp_n[NT / 32];
    __shared__ int any_bad;
    if (threadIdx.x == 0)
        any_bad = 0;
    __syncthreads();
    int n = 0;
    bool bad = false;
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
            if (any_bad)
                atomicOr(&g_flags, kFlagBadTarget);
        }
    }
}

// L = sum_r row_loss[r] / n, summed in fp64 in a fixed order (deterministic).
template <int NT>
__global__ void __launch_bounds__(NT) ce_mean_kernel(const float *row_loss, int64_t M,
                                                     const int *n_ptr, float *loss)
{
    __shared__ double part[NT];
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < M; i += NT)
        s += static_cast<double>(row_loss[i]);
    part[threadIdx.x] = s;
    __syncthreads();
#pragma unroll
    for (int w = NT / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w)
            part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        *loss = static_cast<float>(part[0] / static_cast<double>(*n_ptr));
}

}  // namespace gbce
