// Shared pieces of the tensor-core prefill kernels: canonical shared-memory
// operand layouts of tcgen05 (interleaved and 128-byte swizzled), bf16
// packing, block-wide bounded waits, and the host-side TMA descriptor setup.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace kda {
namespace tc {

constexpr uint32_t kWaitLimit = 1u << 22;   // polls before a wait gives up

// ---- canonical operand layouts --------------------------------------------
// interleaved K-major bf16: element (m, k)
__device__ __forceinline__ uint32_t km_bf16(int m, int k, uint32_t sbo) {
    return (uint32_t)(m >> 3) * sbo + (uint32_t)(k >> 3) * 128u + (uint32_t)(m & 7) * 16u +
           (uint32_t)(k & 7) * 2u;
}
// interleaved K-major tf32: element (m, k)
__device__ __forceinline__ uint32_t km_tf32(int m, int k, uint32_t sbo) {
    return (uint32_t)(m >> 3) * sbo + (uint32_t)(k >> 2) * 128u + (uint32_t)(m & 7) * 16u +
           (uint32_t)(k & 3) * 4u;
}
// interleaved MN-major bf16: element (k, mn)
__device__ __forceinline__ uint32_t mn_bf16(int k, int mn, uint32_t lbo) {
    return (uint32_t)(mn & 7) * 2u + (uint32_t)(mn >> 3) * 128u + (uint32_t)(k & 7) * 16u +
           (uint32_t)(k >> 3) * lbo;
}
// 128B-swizzled tile with 128-byte rows: 16-byte chunk `c` (0..15 across two
// 64-element halves, bf16) of row `row`; `half_bytes` = rows * 128.
__device__ __forceinline__ uint32_t sw_chunk(int row, int c, uint32_t half_bytes) {
    return (uint32_t)(c >> 3) * half_bytes + (uint32_t)row * 128u +
           ((uint32_t)((c & 7) ^ (row & 7)) << 4);
}
// element (row, col) of a bf16 sw tile with two 64-column halves of 64 rows
__device__ __forceinline__ uint32_t sw_elem64(int row, int col) {
    return sw_chunk(row, col >> 3, 8192) + (uint32_t)(col & 7) * 2u;
}

__device__ __forceinline__ float bf(const uint8_t *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack_h8(const float (&x)[8]) {
    return make_uint4(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]), pack_h2(x[4], x[5]), pack_h2(x[6], x[7]));
}
__device__ __forceinline__ uint4 pack_h8x2(const float2 (&x)[4]) {
    return make_uint4(pack_h2(x[0].x, x[0].y), pack_h2(x[1].x, x[1].y), pack_h2(x[2].x, x[2].y),
                      pack_h2(x[3].x, x[3].y));
}
__device__ __forceinline__ uint4 pack_bf8(const float (&x)[8]) {
    return make_uint4(pack_bf2(x[0], x[1]), pack_bf2(x[2], x[3]), pack_bf2(x[4], x[5]),
                      pack_bf2(x[6], x[7]));
}
__device__ __forceinline__ void unpack_bf8(uint4 u, float (&x)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}

// Bounded wait by every thread, then a block-wide verdict.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity, kWaitLimit);
    return __syncthreads_and(ok) != 0;
}

__device__ __forceinline__ void sync_tc() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// 32 consecutive TMEM columns of this thread's lane (two x16 loads, one wait)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    float a[16], b[16];
    tmem_ld16(taddr, a);
    tmem_ld16(taddr + 16, b);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        v[c] = a[c];
        v[16 + c] = b[c];
    }
}

// ---- host: TMA descriptors -----------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3D map over a [T, H, 128] bf16 tensor: dims (128, H, T), box (bw, 1, 64).
inline bool make_map_bf16(CUtensorMap *m, const void *base, int64_t T, int H, uint32_t bw,
                          bool swz) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
    cuuint32_t box[3] = {bw, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3D map over a [T, H, 128] fp32 tensor: dims (128, H, T), box (32, 1, 64), 128B swizzle.
inline bool make_map_f32(CUtensorMap *m, const void *base, int64_t T, int H) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128 * 4, (cuuint64_t)H * 128 * 4};
    cuuint32_t box[3] = {32, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3D map over a [T, H, 128] fp32 tensor: dims (128, H, T), box (32, 1, 64), no swizzle
// (for TMA stores of [64 rows][32 channels] tiles).
inline bool make_map_f32_plain(CUtensorMap *m, const void *base, int64_t T, int H) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128 * 4, (cuuint64_t)H * 128 * 4};
    cuuint32_t box[3] = {32, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---- host: a small cache of encoded maps ----------------------------------
// A serving loop calls the prefill again and again on the same buffers;
// encoding a map is pure host work but not free, so the last few maps are
// kept, keyed on everything that goes into them.
enum MapKind : int { kMapBf16Sw = 0, kMapF32Sw = 1, kMapF32Plain = 2 };

struct MapCache {
    struct Entry {
        const void *base = nullptr;
        int64_t T = -1;
        int H = 0, kind = -1;
        CUtensorMap map;
    };
    static constexpr int kEntries = 32;
    std::mutex mu;
    Entry e[kEntries];
    int next = 0;

    bool get(CUtensorMap *m, int kind, const void *base, int64_t T, int H) {
        {
            std::lock_guard<std::mutex> lk(mu);
            for (const Entry &x : e)
                if (x.kind == kind && x.base == base && x.T == T && x.H == H) {
                    *m = x.map;
                    return true;
                }
        }
        bool ok = kind == kMapBf16Sw   ? make_map_bf16(m, base, T, H, 64, true)
                  : kind == kMapF32Sw  ? make_map_f32(m, base, T, H)
                                       : make_map_f32_plain(m, base, T, H);
        if (!ok) return false;
        std::lock_guard<std::mutex> lk(mu);
        Entry &x = e[next];
        next = (next + 1) % kEntries;
        x.base = base;
        x.T = T;
        x.H = H;
        x.kind = kind;
        x.map = *m;
        return true;
    }
};

}  // namespace tc
}  // namespace kda
