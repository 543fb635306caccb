// tcgen05 / TMA building blocks (sm_100-family PTX) shared by the tensor-core
// kernels: tensor-map encoding on the host, shared-memory matrix descriptors,
// instruction descriptors, TMEM allocation, MMA issue, commit and TMEM loads.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace k3 {
namespace tc {

// ---- host: tensor maps -----------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2D bf16 matrix [rows, cols] (cols contiguous, row pitch `pitch_elems`), box
// [box_rows, 64 cols] with 128-byte swizzle: the K-major operand tile layout of
// tcgen05 (8-row x 128-byte swizzle atoms). Out-of-range rows/cols read as 0.
inline bool make_map_bf16_sw128(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                                uint64_t pitch_elems, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_elems * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- device -------------------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle:
// start address >> 4 in [0,14), leading byte offset (unused for this layout)
// in [16,30), stride byte offset 1024 (one 8-row swizzle atom) in [32,46),
// descriptor version 1 in [46,48), swizzle mode 2 (128B) in [61,64).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(su32(bar))
        : "memory");
}

// 3D tile (x, y, z) with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(su32(bar)), "l"(policy)
        : "memory");
}

// A bf16 [rows, cols] row-major matrix viewed as (64 columns, cols / 64 blocks,
// rows), box {64, blocks, box_rows}: one copy lands box_rows rows of
// 64 * blocks columns each, row after row, unswizzled. cols % 64 == 0.
inline bool make_map_bf16_rows(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t blocks,
                               uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || cols % 64) return false;
    const cuuint64_t dims[3] = {64, cols / 64, rows};
    const cuuint64_t strides[2] = {128, cols * 2};
    const cuuint32_t box[3] = {64, blocks, box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// TMEM allocation by one full warp; the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     su32(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// Position in a ring of N slots: slot index and the parity of its current use.
template <int N>
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next()
    {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// One lane of a converged warp.
__device__ __forceinline__ bool elect_one()
{
    uint32_t p;
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
    return p != 0;
}

// A bounded barrier wait by every lane of a converged warp, which takes the
// outcome only if all lanes saw the phase complete. Needs k3moe_internal.cuh.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, int *err, int where)
{
    const bool ok = mbar_wait(bar, parity, err, where);
    return __all_sync(0xffffffffu, ok) != 0;
}

// A bounded barrier wait by lane 0 of a converged warp, its outcome
// broadcast: the other lanes wait at the shuffle instead of polling.
__device__ __forceinline__ bool lane0_wait(uint64_t *bar, uint32_t parity, int *err, int where)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err, where) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Work items handed out at run time. One thread of the CTA (the writer)
// claims the next item number from a counter in global memory that every CTA
// of the launch shares, when it is ready to start that item, and publishes it
// to the CTA's other roles through a ring of kQ entries in shared memory; -1
// ends the sequence. An SM that HBM
// serves faster than another thereby takes more items, instead of every SM
// taking a fixed share. Every role reads the same sequence, entry i at the
// start of its i-th item, and each reading warp frees the entry once it has
// read it; the writer refills an entry only after all of them have, and it
// runs less than one item ahead of the roles it feeds, so the ring never
// holds it up for long. Waits are bounded as everywhere else.
struct ItemQueue {
    static constexpr int kQ = 4;
    int *item;              // [kQ] in shared memory
    uint64_t *full, *empty; // [kQ] each: full by the writer, empty by the readers
    __device__ __forceinline__ void init(int readers)
    {
        for (int i = 0; i < kQ; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], (uint32_t)readers);
        }
    }
    // writer: claims the CTA's i-th item (-1 once the counter has passed n)
    __device__ __forceinline__ int claim(int *counter, int n, int i, int *err, int where)
    {
        const int v = atomicAdd(counter, 1);
        const int it = v < n ? v : -1;
        if (!mbar_wait(&empty[i % kQ], ((uint32_t)(i / kQ) & 1u) ^ 1u, err, where)) return -1;
        item[i % kQ] = it;
        mbar_arrive(&full[i % kQ]);
        return it;
    }
    // a reading warp (every lane gets the item; lane 0 frees the entry);
    // -1 at the end of the sequence or after a time-out
    __device__ __forceinline__ int read_warp(int i, int *err, int where)
    {
        if (!warp_wait(&full[i % kQ], (uint32_t)(i / kQ) & 1u, err, where)) return -1;
        const int it = *reinterpret_cast<volatile int *>(&item[i % kQ]);
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[i % kQ]);
        return it;
    }
    // a reading thread that stands for its warp (the warp's other lanes do not read)
    __device__ __forceinline__ int read_one(int i, int *err, int where)
    {
        if (!mbar_wait(&full[i % kQ], (uint32_t)(i / kQ) & 1u, err, where)) return -1;
        const int it = *reinterpret_cast<volatile int *>(&item[i % kQ]);
        mbar_arrive(&empty[i % kQ]);
        return it;
    }
};

}  // namespace tc
}  // namespace k3
