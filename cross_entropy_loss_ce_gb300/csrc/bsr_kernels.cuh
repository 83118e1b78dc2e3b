// Block-sparse softmax backward ("python sum function examples
// (triton.language)", _backward): dx = y * (dy - sum(y * dy)) * scale over the
// rows of a block-sparse matrix whose blocks are listed in a look-up table.
//
// Storage (per batch item z, at z * stride elements): block b is a
// block x block tile, row-major, at b * block^2.  The table starts with one
// (size, offset) pair per block-row; entry k of block-row rbm is 4 ints at
// offset + 4 k, the block id first.  Row rxm of block-row rbm is the
// concatenation of row rxm of its blocks.
//
// Two kernels, chosen on the host from the longest row (sizemax * block):
//   bsr_bwd_staged_kernel    one CTA (or 2 or 4, each with a share of the rows)
//                            per block-row and batch item, its rows in slabs of R.  A slab's piece of every listed block
//                            (R * block contiguous elements per operand) is
//                            gathered into shared memory with 16-byte
//                            asynchronous copies, each row's sum(y * dy) is
//                            reduced there, and dx is written from the staged
//                            copy (HBM sees 2 reads and 1 write per element);
//                            stages overlap the next slabs' copies with the
//                            current slab's work.
//   bsr_bwd_unstaged_kernel  rows too long to stage: one CTA per row, the sum
//                            in a first pass over global memory and dx in a
//                            second (the re-read mostly served by L2).
// Both validate the table before touching any element: a block-row whose size
// is negative or above sizemax, whose entries run past the table, or that
// names a block outside [0, nblocks) raises kFlagBadTable (and the call's
// status word, when it has one) and is left alone.
#pragma once

#include "device.cuh"

namespace gbce {

struct BsrArgs {
    const void *y;    // softmax output, batch stride ys elements
    int64_t ys;
    const void *dy;   // upstream gradient, batch stride dys
    int64_t dys;
    void *dx;         // result (may be dy), batch stride dxs
    int64_t dxs;
    const int32_t *lut;
    int64_t lut_len;
    int64_t nbr;      // block-rows (table headers)
    int64_t nblocks;  // blocks per batch item
    int log2_block;
    int log2_R;       // staged: a stage holds sizemax blocks of 2^log2_R rows per operand
    int max_log2_R;   // staged: largest rows per slab, log2 (<= log2_block, <= log2(NT / 4))
    int sizemax;      // largest valid size of a block-row
    int ids_bytes;    // staged: shared bytes reserved for the block ids (multiple of 16)
    int stage_bytes;  // staged: bytes of one stage (y slab, dy slab; multiple of 16)
    int log2_split;   // staged: CTAs per block-row and batch item (2^log2_split), each a share of its slabs
    float scale;
    unsigned *status; // the call's own status word (NULL: none); kStatusBadTable marks a bad entry
};

constexpr unsigned kStatusBadTable = 2u;  // GBCE_STATUS_BAD_TABLE

// A malformed table entry: the device flag, and the call's status word when it has one.
__device__ __forceinline__ void raise_bad_table(const BsrArgs &a)
{
    atomicOr(&g_flags, kFlagBadTable);
    if (a.status)
        atomicOr(a.status, kStatusBadTable);
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_pending()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int N>
struct Log2 {
    static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
    static constexpr int value = 0;
};

// Warp-wide check of block-row rbm's table entry (all 32 lanes call it).
// Returns the block-row's size, or -1 when the table is wrong for it.  With
// `ids`, the block ids are stored there (only meaningful when the result is
// >= 0).  `off` receives the entries' offset.
__device__ __forceinline__ int bsr_header(const BsrArgs &a, int64_t rbm, int32_t *ids, int lane,
                                          int &off)
{
    int size = 0, o = 0;
    if (lane == 0) {
        size = __ldg(a.lut + 2 * rbm);
        o = __ldg(a.lut + 2 * rbm + 1);
    }
    size = __shfl_sync(0xffffffffu, size, 0);
    o = __shfl_sync(0xffffffffu, o, 0);
    bool bad = size < 0 || size > a.sizemax ||
               (size > 0 && (o < 0 || int64_t{o} + 4 * int64_t{size - 1} >= a.lut_len));
    if (!bad) {
        for (int k = lane; k < size; k += 32) {
            const int id = __ldg(a.lut + int64_t{o} + 4 * int64_t{k});
            if (id < 0 || int64_t{id} >= a.nblocks)
                bad = true;
            if (ids)
                ids[k] = id;
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    off = o;
    return bad ? -1 : size;
}

// One CTA per task t = z * nbr + rbm (one block-row of one batch item).  The
// table entry is read once; the block-row's rows then stream, a slab of
// several rows at a time, through STAGES shared-memory stages: slabs s + 1 ..
// s + STAGES - 1 are in flight while slab s is reduced and written.
// VEC: elements per access, 16 / sizeof(T) (16-byte vectors) or 1.  STAGES:
// slab stages in shared memory (STAGES - 1 slabs in flight during the work).
template <typename T, int VEC, int NT, int STAGES>
__global__ void __launch_bounds__(NT) bsr_bwd_staged_kernel(const BsrArgs a)
{
    using E = Elem<T>;
    constexpr int LV = Log2<VEC>::value;
    constexpr int LNT = Log2<NT>::value;
    static_assert(VEC == 1 || VEC * sizeof(T) == 16, "VEC is one element or one 16-byte vector");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_size;
    __shared__ float s_warp[NT / 32];
    __shared__ float s_row[NT / 4];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t task = blockIdx.x >> a.log2_split;
    const int share = static_cast<int>(blockIdx.x & ((1u << a.log2_split) - 1));
    const int64_t rbm = task % a.nbr;
    const int64_t z = task / a.nbr;
    int32_t *ids = reinterpret_cast<int32_t *>(smem);
    if (warp == 0) {
        int off;
        const int size = bsr_header(a, rbm, ids, lane, off);
        if (lane == 0) {
            s_size = size;
            if (size < 0)
                raise_bad_table(a);
        }
    }
    __syncthreads();
    const int size = s_size;
    if (size <= 0)
        return;

    // A stage holds sizemax blocks of 2^log2_R rows per operand; a block-row of
    // `size` blocks takes slabs of 2^lr rows, the most that fit (at most
    // 2^max_log2_R, the block's rows or NT / 4).
    const int64_t seg_elems = static_cast<int64_t>(a.sizemax) << (a.log2_R + a.log2_block);
    int lr = a.log2_R;
    while (lr < a.max_log2_R && (int64_t{size} << (lr + 1)) <= (int64_t{a.sizemax} << a.log2_R))
        ++lr;
    const int log2_seg = lr + a.log2_block;  // elements of one block's slab
    const int64_t bb = int64_t{1} << (2 * a.log2_block);
    // this CTA's share of the block-row's slabs: sl0 .. sl0 + nslab - 1
    const int all_slabs = 1 << (a.log2_block - lr);
    int nslab, sl0;
    if (all_slabs >= (1 << a.log2_split)) {
        nslab = all_slabs >> a.log2_split;
        sl0 = share * nslab;
    } else {
        nslab = share < all_slabs ? 1 : 0;
        sl0 = share;
    }
    if (nslab == 0)
        return;
    const T *ybase = static_cast<const T *>(a.y) + z * a.ys;
    const T *dybase = static_cast<const T *>(a.dy) + z * a.dys;
    T *xbase = static_cast<T *>(a.dx) + z * a.dxs;
    auto ybuf = [&](int st) {
        return reinterpret_cast<T *>(smem + a.ids_bytes + st * a.stage_bytes);
    };

    // Gather slab sl into stage st: piece k = R rows of block ids[k],
    // contiguous in global memory (16-byte asynchronous copies).
    auto issue = [&](int sl, int st) {
        const int64_t slab_off = int64_t{sl0 + sl} << log2_seg;
        T *yb = ybuf(st);
        T *db = yb + seg_elems;
        if constexpr (VEC > 1) {
            const uint32_t ys_addr = smem_addr(yb), ds_addr = smem_addr(db);
            const int log2_segv = log2_seg - LV;
            const int nvec = size << log2_segv;
            for (int q = tid; q < nvec; q += NT) {
                const int64_t src = slab_off + ids[q >> log2_segv] * bb +
                                    (int64_t{q & ((1 << log2_segv) - 1)} << LV);
                cp_async_16(ys_addr + 16u * q, ybase + src);
                cp_async_16(ds_addr + 16u * q, dybase + src);
            }
        } else {
            const int n = size << log2_seg;
            for (int q = tid; q < n; q += NT) {
                const int64_t src = slab_off + ids[q >> log2_seg] * bb + (q & ((1 << log2_seg) - 1));
                yb[q] = ybase[src];
                db[q] = dybase[src];
            }
        }
    };

    // row r of a slab is served by 2^log2_tpr consecutive threads
    const int log2_tpr = LNT - lr;
    const int tpr = 1 << log2_tpr;
    const int r = tid >> log2_tpr;
    const int part = tid & (tpr - 1);
    const int log2_bv = a.log2_block - LV;  // accesses per row of one block
    const int rv = size << log2_bv;         // accesses per matrix row
    const float scale = a.scale;

    for (int sl = 0; sl < STAGES - 1; ++sl) {
        if (sl < nslab)
            issue(sl, sl);
        cp_async_commit();
    }
    for (int sl = 0; sl < nslab; ++sl) {
        const int st = sl % STAGES;
        if (sl + STAGES - 1 < nslab)
            issue(sl + STAGES - 1, (sl + STAGES - 1) % STAGES);
        cp_async_commit();
        cp_async_wait_pending<STAGES - 1>();  // slab sl has landed
        __syncthreads();

        const T *yb = ybuf(st);
        const T *db = yb + seg_elems;
        const uint32_t ys_addr = smem_addr(yb), ds_addr = smem_addr(db);
        float acc = 0.f;
        for (int j = part; j < rv; j += tpr) {
            const int e = ((((j >> log2_bv) << lr) + r) << a.log2_block) +
                          ((j & ((1 << log2_bv) - 1)) << LV);
            if constexpr (VEC > 1) {
                float fy[VEC], fd[VEC];
                E::unpack(ld_shared_v4(ys_addr + e * static_cast<uint32_t>(sizeof(T))), fy);
                E::unpack(ld_shared_v4(ds_addr + e * static_cast<uint32_t>(sizeof(T))), fd);
#pragma unroll
                for (int i = 0; i < VEC; ++i)
                    acc = fmaf(fy[i], fd[i], acc);
            } else {
                acc = fmaf(E::load(yb + e), E::load(db + e), acc);
            }
        }
        if (tpr <= 32) {
            for (int o = tpr >> 1; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (part == 0)
                s_row[r] = acc;
        } else {
            acc = warp_sum(acc);
            if (lane == 0)
                s_warp[warp] = acc;
            __syncthreads();
            if (part == 0) {
                float sum = 0.f;
                for (int i = 0; i < (tpr >> 5); ++i)
                    sum += s_warp[warp + i];
                s_row[r] = sum;
            }
        }
        __syncthreads();
        const float sr = s_row[r];
        T *xb = xbase + (int64_t{sl0 + sl} << log2_seg) + (int64_t{r} << a.log2_block);
        for (int j = part; j < rv; j += tpr) {
            const int k = j >> log2_bv;
            const int c = j & ((1 << log2_bv) - 1);
            const int e = (((k << lr) + r) << a.log2_block) + (c << LV);
            T *dst = xb + ids[k] * bb + (c << LV);
            if constexpr (VEC > 1) {
                float fy[VEC], fd[VEC];
                E::unpack(ld_shared_v4(ys_addr + e * static_cast<uint32_t>(sizeof(T))), fy);
                E::unpack(ld_shared_v4(ds_addr + e * static_cast<uint32_t>(sizeof(T))), fd);
#pragma unroll
                for (int i = 0; i < VEC; ++i)
                    fy[i] = fy[i] * (fd[i] - sr) * scale;
                __stcs(reinterpret_cast<uint4 *>(dst), E::pack(fy));
            } else {
                E::store(dst, E::load(yb + e) * (E::load(db + e) - sr) * scale);
            }
        }
        __syncthreads();  // stage st and s_row are free for slab sl + STAGES
    }
    cp_async_wait_all();
}

// One CTA per matrix row: u = (z * nbr + rbm) * block + rxm.
template <typename T, int VEC, int NT>
__global__ void __launch_bounds__(NT) bsr_bwd_unstaged_kernel(const BsrArgs a)
{
    using E = Elem<T>;
    constexpr int LV = Log2<VEC>::value;
    static_assert(VEC == 1 || VEC * sizeof(T) == 16, "VEC is one element or one 16-byte vector");
    __shared__ int s_size, s_off;
    __shared__ float s_warp[NT / 32];
    __shared__ float s_sum;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t u = blockIdx.x;
    const int64_t rxm = u & ((int64_t{1} << a.log2_block) - 1);
    const int64_t t = u >> a.log2_block;
    const int64_t rbm = t % a.nbr;
    const int64_t z = t / a.nbr;
    if (warp == 0) {
        int off;
        const int size = bsr_header(a, rbm, nullptr, lane, off);
        if (lane == 0) {
            s_size = size;
            s_off = off;
            if (size < 0)
                raise_bad_table(a);
        }
    }
    __syncthreads();
    const int size = s_size;
    if (size <= 0)
        return;
    const int64_t off = s_off;
    const int64_t bb = int64_t{1} << (2 * a.log2_block);
    const int64_t row_off = rxm << a.log2_block;
    const T *yb = static_cast<const T *>(a.y) + z * a.ys + row_off;
    const T *dyb = static_cast<const T *>(a.dy) + z * a.dys + row_off;
    T *xb = static_cast<T *>(a.dx) + z * a.dxs + row_off;
    const int log2_bv = a.log2_block - LV;
    const int64_t rv = int64_t{size} << log2_bv;

    float acc = 0.f;
    for (int64_t j = tid; j < rv; j += NT) {
        const int64_t k = j >> log2_bv;
        const int64_t p = __ldg(a.lut + off + 4 * k) * bb + ((j & ((1 << log2_bv) - 1)) << LV);
        if constexpr (VEC > 1) {
            float fy[VEC], fd[VEC];
            E::unpack(__ldcg(reinterpret_cast<const uint4 *>(yb + p)), fy);
            E::unpack(__ldcg(reinterpret_cast<const uint4 *>(dyb + p)), fd);
#pragma unroll
            for (int i = 0; i < VEC; ++i)
                acc = fmaf(fy[i], fd[i], acc);
        } else {
            acc = fmaf(E::load(yb + p), E::load(dyb + p), acc);
        }
    }
    acc = warp_sum(acc);
    if (lane == 0)
        s_warp[warp] = acc;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int i = 0; i < NT / 32; ++i)
            s += s_warp[i];
        s_sum = s;
    }
    __syncthreads();
    const float sr = s_sum;
    const float scale = a.scale;
    for (int64_t j = tid; j < rv; j += NT) {
        const int64_t k = j >> log2_bv;
        const int64_t p = __ldg(a.lut + off + 4 * k) * bb + ((j & ((1 << log2_bv) - 1)) << LV);
        if constexpr (VEC > 1) {
            float fy[VEC], fd[VEC];
            E::unpack(__ldcg(reinterpret_cast<const uint4 *>(yb + p)), fy);
            E::unpack(__ldcg(reinterpret_cast<const uint4 *>(dyb + p)), fd);
#pragma unroll
            for (int i = 0; i < VEC; ++i)
                fy[i] = fy[i] * (fd[i] - sr) * scale;
            __stcs(reinterpret_cast<uint4 *>(xb + p), E::pack(fy));
        } else {
            E::store(xb + p, E::load(yb + p) * (E::load(dyb + p) - sr) * scale);
        }
    }
}

}  // namespace gbce
