// Device-side building blocks for the row kernels: PTX wrappers for mbarriers,
// 1-D bulk (TMA) copies, thread-block clusters and distributed shared memory,
// element packing for fp32 / bf16, and the (max, rescaled-sum) pair algebra of
// the online softmax.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gbce {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): exp(x) = exp2(x * log2(e))
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a bulk copy that takes 2 s has failed

// Sticky per-device error flags (read and cleared by gbce_last_error()).
enum : unsigned { kFlagBadTarget = 1u, kFlagTimeout = 2u, kFlagBadTable = 4u };

// ---------------------------------------------------------------------------
// small PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return true;
}

// Wait for phase `parity` of an mbarrier until the %globaltimer value
// `deadline`: used before a CTA exits, for copies it issued that may still be
// in flight after a wait gave up.
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, uint64_t deadline)
{
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() > deadline)
            return false;
    }
    return true;
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Store 16 bytes into shared memory of a peer CTA (a shared::cluster address)
// and count them on that CTA's mbarrier (also a shared::cluster address).
__device__ __forceinline__ void st_async_f4(uint32_t remote, float4 v, uint32_t remote_bar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(remote),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ void cluster_arrive_any()
{
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_any()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ float2 ld_cluster_f2(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v.x), "=f"(v.y)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// element types: 16-byte vectors of fp32 (4), bf16 (8) or fp16 (8)

template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kPerVec = 4;
    static constexpr uint32_t kNegInfPair = 0xff800000u;  // -inf (never read as pairs)
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[4])
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
    __device__ static __forceinline__ float load(const float *p) { return *p; }
    __device__ static __forceinline__ void store(float *p, float v) { *p = v; }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    static constexpr uint32_t kNegInfPair = 0xff80ff80u;  // two bf16 -inf
    // element-wise max of two packed pairs, and the larger of a pair as fp32
    __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b)
    {
        __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    __device__ static __forceinline__ float pair_max(uint32_t p)
    {
        return fmaxf(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
    }
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[8])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[8])
    {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ static __forceinline__ float load(const __nv_bfloat16 *p)
    {
        return __bfloat162float(*p);
    }
    __device__ static __forceinline__ void store(__nv_bfloat16 *p, float v)
    {
        *p = __float2bfloat16_rn(v);
    }
};

template <>
struct Elem<__half> {
    static constexpr int kPerVec = 8;
    static constexpr uint32_t kNegInfPair = 0xfc00fc00u;  // two fp16 -inf
    __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b)
    {
        __half2 r = __hmax2(*reinterpret_cast<const __half2 *>(&a),
                            *reinterpret_cast<const __half2 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    __device__ static __forceinline__ float pair_max(uint32_t p)
    {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&p));
        return fmaxf(f.x, f.y);
    }
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[8])
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ static __forceinline__ uint32_t pack2(float lo, float hi)
    {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[8])
    {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
    __device__ static __forceinline__ float load(const __half *p) { return __half2float(*p); }
    __device__ static __forceinline__ void store(__half *p, float v) { *p = __float2half_rn(v); }
};

// ---------------------------------------------------------------------------
// Row geometry: a row of `cols` elements starting at `p` splits into a head of
// elements before the first 16-byte boundary, `nvec` whole 16-byte vectors,
// and a tail of fewer than one vector.  The head and tail are accessed with
// scalar loads and stores, the vectors with bulk copies / 128-bit accesses.
struct RowGeom {
    int head;           // elements before the first 16-byte-aligned address
    int tail;           // elements after the last whole vector
    int64_t nvec;       // whole vectors
    int64_t tail_start; // column of the first tail element
};

template <typename T>
__device__ __forceinline__ RowGeom row_geom(const T *p, int64_t cols)
{
    constexpr int VEC = Elem<T>::kPerVec;
    RowGeom g;
    const int mis = static_cast<int>(reinterpret_cast<uintptr_t>(p) & 15u);
    int64_t head = mis ? (16 - mis) / static_cast<int>(sizeof(T)) : 0;
    if (head > cols)
        head = cols;
    g.head = static_cast<int>(head);
    g.nvec = (cols - head) / VEC;
    g.tail_start = head + g.nvec * VEC;
    g.tail = static_cast<int>(cols - g.tail_start);
    return g;
}

// ---------------------------------------------------------------------------
// exp(x - m) as exp2(x log2(e) - sL), where sL = fl(m log2(e)) is the shift of a
// partial sum in log2 units.  The product x log2(e) is exact inside the FMA, so
// the exponent carries one rounding, relative to its own size |x - m| log2(e):
// the error of a term grows with its distance from the shift, not with the
// magnitude of the logits.  Every partial keeps its shift in these units and
// rescales by exp2(sL_a - sL_b) when merging, so numerator and denominator see
// the same shift and any rounding of m log2(e) cancels in exp(x - m) / sum.
// sL must be finite (0 for a part that holds only -inf, whose terms are 0).
__device__ __forceinline__ float exp2_shift(float x, float sL) { return exp2f(fmaf(x, kLog2e, -sL)); }

// The shift of a part whose maximum is m, in log2 units: -inf for an empty
// part (its sum is 0), else fl(m log2(e)).
__device__ __forceinline__ float shift_of(float m) { return m * kLog2e; }

// -log p_y = ln D - (x_y log2(e) - SL) ln 2 for the final shift SL and sum D:
// the difference is one FMA rounding relative to |x_y - m|, so the row loss
// keeps its relative accuracy whatever the logits' magnitude.
__device__ __forceinline__ float row_loss_from(float SL, float D, float xy)
{
    return logf(D) - fmaf(xy, kLog2e, -SL) * kLn2;
}

// ---------------------------------------------------------------------------
// (s, d) pairs of the online softmax: s = fl(m log2(e)) the shift of a running
// maximum m in log2 units, d = sum exp2(x log2(e) - s).  Merging two pairs
// rescales both sums to the larger shift by exp2 of the difference of the two
// stored shifts (exact when they are within a factor of two).  An empty pair
// is (-inf, 0); two empty pairs merge to an empty pair (no -inf - -inf).
__device__ __forceinline__ void md_merge(float &m, float &d, float m2, float d2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY)
        return;
    d = d * exp2f(m - mn) + d2 * exp2f(m2 - mn);
    m = mn;
}

// Butterfly merge across a warp; every lane ends with the same bits because
// md_merge is commutative.
__device__ __forceinline__ void warp_md_reduce(float &m, float &d)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float d2 = __shfl_xor_sync(0xffffffffu, d, off);
        md_merge(m, d, m2, d2);
    }
}

__device__ __forceinline__ float warp_sum(float s)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

}  // namespace gbce
