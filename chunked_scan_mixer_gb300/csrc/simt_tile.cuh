// Register-tiled float32 products for the SIMT chunk kernels (fwd_chunk_simt.cu,
// bwd_chunk_simt.cu).
//
// A thread owns an RM x 4 block of an M x N output: four consecutive columns n0 .. n0 + 3
// and RM consecutive rows m0 ..  Every step k of a product reads one float4 of B's row k
// (B row-major over the output's columns, leading dimension a multiple of 4, 16-byte
// aligned) and RM values of A through two strides, so A may sit in either orientation.
// Consecutive threads take consecutive column groups, so the lanes of a warp read one
// contiguous run of B (shared by the row groups of the warp: a broadcast) and the few A
// values of their row groups.  Tiles that are read as A with their rows spread over a warp
// are stored with the leading dimension pad(x) = x + 4, which starts consecutive rows four
// banks apart.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace hla2 {
namespace simt {

constexpr int kThreads = 256;

__host__ __device__ constexpr int pad(int x) { return x + 4; }

template <int RM>
using Acc = float[RM][4];

// acc += sum_{k0 <= k < k1} A(i, k) B(k, 0..3),  A(i, k) = A[i * sam + k * sak]
template <int RM>
__device__ __forceinline__ void mac(Acc<RM>& acc, const float* A, int sam, int sak, const float* B, int ldb, int k0,
                                    int k1) {
#pragma unroll 4
    for (int k = k0; k < k1; ++k) {
        const float4 b = *reinterpret_cast<const float4*>(B + (size_t)k * ldb);
#pragma unroll
        for (int i = 0; i < RM; ++i) {
            const float x = A[i * sam + k * sak];
            acc[i][0] = fmaf(x, b.x, acc[i][0]);
            acc[i][1] = fmaf(x, b.y, acc[i][1]);
            acc[i][2] = fmaf(x, b.z, acc[i][2]);
            acc[i][3] = fmaf(x, b.w, acc[i][3]);
        }
    }
}

// The same with a weight w(k) on every B row.
template <int RM, class Wk>
__device__ __forceinline__ void mac_w(Acc<RM>& acc, const float* A, int sam, int sak, const float* B, int ldb, int k0,
                                      int k1, Wk w) {
#pragma unroll 4
    for (int k = k0; k < k1; ++k) {
        float4 b = *reinterpret_cast<const float4*>(B + (size_t)k * ldb);
        const float s = w(k);
        b.x *= s;
        b.y *= s;
        b.z *= s;
        b.w *= s;
#pragma unroll
        for (int i = 0; i < RM; ++i) {
            const float x = A[i * sam + k * sak];
            acc[i][0] = fmaf(x, b.x, acc[i][0]);
            acc[i][1] = fmaf(x, b.y, acc[i][1]);
            acc[i][2] = fmaf(x, b.z, acc[i][2]);
            acc[i][3] = fmaf(x, b.w, acc[i][3]);
        }
    }
}

template <int RM>
__device__ __forceinline__ void zero(Acc<RM>& acc) {
#pragma unroll
    for (int i = 0; i < RM; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

template <int RM>
__device__ __forceinline__ void scale_row(Acc<RM>& acc, int i, float s) {
    acc[i][0] *= s;
    acc[i][1] *= s;
    acc[i][2] *= s;
    acc[i][3] *= s;
}

__device__ __forceinline__ float4 f4(const float (&r)[4]) { return make_float4(r[0], r[1], r[2], r[3]); }

__device__ __forceinline__ void st4(float* p, const float (&r)[4]) { *reinterpret_cast<float4*>(p) = f4(r); }

// dst[0..3] = rho * dst[0..3] + r
__device__ __forceinline__ void decay_add4(float* p, float rho, const float (&r)[4]) {
    float4 o = *reinterpret_cast<float4*>(p);
    o.x = fmaf(rho, o.x, r[0]);
    o.y = fmaf(rho, o.y, r[1]);
    o.z = fmaf(rho, o.z, r[2]);
    o.w = fmaf(rho, o.w, r[3]);
    *reinterpret_cast<float4*>(p) = o;
}

// four values to global memory (16-byte float4, or 8 bytes of bf16)
__device__ __forceinline__ void store4(float* p, const float (&r)[4]) { st4(p, r); }
__device__ __forceinline__ void store4(bf16* p, const float (&r)[4]) {
    uint2 u;
    u.x = pack_bf16x2(r[0], r[1]);
    u.y = pack_bf16x2(r[2], r[3]);
    *reinterpret_cast<uint2*>(p) = u;
}

// Rows per thread of an M x N output (N a multiple of 4): the largest of 4, 2, 1 that still
// gives every thread a block.
__device__ __forceinline__ int rows_per_thread(int M, int N) {
    const int nt = N >> 2;
    if ((M & 3) == 0 && (M >> 2) * nt >= kThreads) return 4;
    if ((M & 1) == 0 && (M >> 1) * nt >= kThreads) return 2;
    return 1;
}

// f(std::integral_constant<int, RM>) with RM = rows_per_thread(M, N)
template <class F>
__device__ __forceinline__ void with_rm(int M, int N, F&& f) {
    switch (rows_per_thread(M, N)) {
        case 4: f(std::integral_constant<int, 4>{}); break;
        case 2: f(std::integral_constant<int, 2>{}); break;
        default: f(std::integral_constant<int, 1>{}); break;
    }
}

// f(m0, n0) for every RM x 4 block of an M x N output that this thread owns
template <int RM, class F>
__device__ __forceinline__ void for_blocks(int M, int N, F&& f) {
    const int nt = N >> 2, blocks = (M / RM) * nt;
    for (int t = threadIdx.x; t < blocks; t += kThreads) f((t / nt) * RM, (t % nt) * 4);
}

}  // namespace simt
}  // namespace hla2
