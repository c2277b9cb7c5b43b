// Helpers shared by the tcgen05 first-order scan kernels (fo_tc.cu, d = dv = 128; fo64_tc.cu,
// d = dv = 64): bf16 packing, the masked decayed Gram block, the segment geometry of a CTA and
// the tensor maps of [BH][n][D] bf16 tensors.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace hla2 {
namespace {

namespace la_common {
constexpr int kW = 128;                // chunk width (tokens per chunk)
constexpr uint32_t kBlk = 128 * 128;   // one [128 rows][64 bf16] SW128 column block (16 KB)
}  // namespace la_common

__device__ __forceinline__ float la_bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float la_bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ uint4 la_scale_chunk(uint4 c, float s) {
    uint4 o;
    o.x = pack_bf16x2(s * la_bf_lo(c.x), s * la_bf_hi(c.x));
    o.y = pack_bf16x2(s * la_bf_lo(c.y), s * la_bf_hi(c.y));
    o.z = pack_bf16x2(s * la_bf_lo(c.z), s * la_bf_hi(c.z));
    o.w = pack_bf16x2(s * la_bf_lo(c.w), s * la_bf_hi(c.w));
    return o;
}

__device__ __forceinline__ uint4 la_pack8(const float* f) {
    uint4 o;
    o.x = pack_bf16x2(f[0], f[1]);
    o.y = pack_bf16x2(f[2], f[3]);
    o.z = pack_bf16x2(f[4], f[5]);
    o.w = pack_bf16x2(f[6], f[7]);
    return o;
}

// Byte offset of 16-byte chunk j (0..7) of row r in column block b of a [128][128] tile.
__device__ __forceinline__ uint32_t la_off(int b, int r, int j) { return (uint32_t)b * la_common::kBlk + tc::sw128_chunk(r, j); }

// Masked, decayed 32-column block [cb, cb + 32) of Gram row r (fp32 at src in tensor memory),
// packed to 16 bf16 pairs.  Forward keeps i <= r with g^(r - i); reverse keeps i >= r with
// g^(i - r).  cb and the warp's first row row0 are multiples of 32, so a block is entirely
// kept, entirely dropped (written as zeros without reading) or the diagonal block.
template <bool REV>
__device__ __forceinline__ void la_masked_pack(uint32_t src, int r, int cb, int row0, float log2g, float g,
                                               float ginv, uint32_t (&pk)[16]) {
    const bool dropped = REV ? cb < row0 : cb > row0;
    if (dropped) {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
        return;
    }
    const bool diag = cb == row0;
    float f = pow_decay(log2g, (float)(REV ? cb - r : r - cb));  // factor at column cb
    const float step = REV ? g : ginv;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // 16 columns at a time (register pressure)
        uint32_t v[16];
        tc::tmem_ld16(src + 16 * half, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            float a0 = f * __uint_as_float(v[j]);
            f *= step;
            float a1 = f * __uint_as_float(v[j + 1]);
            f *= step;
            if (diag) {
                const int i0 = cb + 16 * half + j, i1 = i0 + 1;
                a0 = (REV ? i0 >= r : i0 <= r) ? a0 : 0.f;
                a1 = (REV ? i1 >= r : i1 <= r) ? a1 : 0.f;
            }
            pk[8 * half + j / 2] = pack_bf16x2(a0, a1);
        }
    }
}

// Segment geometry of a CTA.
struct FoSeg {
    int c_begin, c_end, nit, t0, L;
};
__device__ __forceinline__ FoSeg la_seg(const FoArgs& a, int seg) {
    FoSeg s;
    s.c_begin = seg * a.seg_chunks;
    s.c_end = min(s.c_begin + a.seg_chunks, a.nchunks);
    s.nit = s.c_end - s.c_begin;
    s.t0 = s.c_begin * la_common::kW;
    s.L = min(s.c_end * la_common::kW, a.n) - s.t0;
    return s;
}


PFN_cuTensorMapEncodeTiled_v12000 la_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// [BH][n][D] bf16 (D = 64 or 128), box [1][128][64] (128-byte rows), 128-byte swizzle; rows
// past n read as zero and are not written by stores.
bool la_map(CUtensorMap* m, const void* ptr, int BH, int n, int D = 128) {
    auto fn = la_encode_fn();
    if (!fn || !ptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)n * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)la_common::kW, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace
}  // namespace hla2
