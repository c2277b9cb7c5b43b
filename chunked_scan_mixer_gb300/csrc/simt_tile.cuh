// Register-tiled float32 products for the SIMT chunk kernels (fwd_chunk_simt.cu,
// bwd_chunk_simt.cu).
//
// A thread owns an RM x 4 block of an M x N output: four consecutive columns n0 .. n0 + 3
// and RM consecutive rows m0 ..  Every step k of a product reads one float4 of B's row k
// (B row-major over the output's columns, leading dimension a multiple of 4, 16-byte
// aligned) and the block's RM values of A: from a row-major A one float4 per row serves
// four steps (mac_r), from a column-major A one vector of RM floats serves a step (mac_c).
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

// Shared memory of an SM (228 KB) and the most one CTA may take (227 KB); the runtime keeps
// 1 KB per resident CTA.
constexpr size_t kSmemPerSm = 233472, kSmemPerCta = 232448, kSmemReserved = 1024;

// CTAs of `bytes` dynamic shared memory that fit on one SM (shared memory only).
__host__ __device__ constexpr int ctas_per_sm(size_t bytes) {
    return bytes > kSmemPerCta ? 0 : (int)(kSmemPerSm / (bytes + kSmemReserved));
}

// Whether `extra` more floats of shared memory beside `floats` are free for a kernel of at most
// `max_ctas` resident CTAs per SM: they fit, and as many CTAs stay resident.
__host__ __device__ constexpr int min_ctas(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr bool fits_beside(size_t floats, size_t extra, int max_ctas) {
    return ctas_per_sm((floats + extra) * 4) >= 1 &&
           min_ctas(ctas_per_sm((floats + extra) * 4), max_ctas) >= min_ctas(ctas_per_sm(floats * 4), max_ctas);
}

template <int RM>
using Acc = float[RM][4];

// RM values a[0 .. RM) from 16-byte aligned consecutive floats
template <int RM>
__device__ __forceinline__ void ldv(float (&a)[RM], const float* p) {
    if constexpr (RM == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        a[0] = t.x;
        a[1] = t.y;
        a[2] = t.z;
        a[3] = t.w;
    } else if constexpr (RM == 2) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        a[0] = t.x;
        a[1] = t.y;
    } else {
        a[0] = p[0];
    }
}

template <int RM>
__device__ __forceinline__ void fma_row(Acc<RM>& acc, const float (&a)[RM], const float4& b) {
#pragma unroll
    for (int i = 0; i < RM; ++i) {
        acc[i][0] = fmaf(a[i], b.x, acc[i][0]);
        acc[i][1] = fmaf(a[i], b.y, acc[i][1]);
        acc[i][2] = fmaf(a[i], b.z, acc[i][2]);
        acc[i][3] = fmaf(a[i], b.w, acc[i][3]);
    }
}

__device__ __forceinline__ float4 ldb4(const float* B, int ldb, int k) {
    return *reinterpret_cast<const float4*>(B + (size_t)k * ldb);
}

__device__ __forceinline__ float4 scale4(float4 b, float s) {
    b.x *= s;
    b.y *= s;
    b.z *= s;
    b.w *= s;
    return b;
}

struct NoWeight {
    __device__ __forceinline__ float operator()(int) const { return 1.f; }
};

// acc += sum_{0 <= k < k1} A[i][k] w(k) B(k, 0..3) with A row-major (lda, 16-byte aligned
// rows): four k at a time, one float4 of every A row.
template <int RM, class Wk = NoWeight>
__device__ __forceinline__ void mac_r(Acc<RM>& acc, const float* A, int lda, const float* B, int ldb, int k1,
                                      Wk w = Wk{}) {
    constexpr bool kW = !std::is_same<Wk, NoWeight>::value;
    const int k4 = k1 & ~3;
#pragma unroll 2
    for (int k = 0; k < k4; k += 4) {
        float4 a[RM];
#pragma unroll
        for (int i = 0; i < RM; ++i) a[i] = *reinterpret_cast<const float4*>(A + i * lda + k);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float4 b = ldb4(B, ldb, k + u);
            if (kW) b = scale4(b, w(k + u));
            float x[RM];
#pragma unroll
            for (int i = 0; i < RM; ++i) x[i] = u == 0 ? a[i].x : u == 1 ? a[i].y : u == 2 ? a[i].z : a[i].w;
            fma_row<RM>(acc, x, b);
        }
    }
    for (int k = k4; k < k1; ++k) {
        float4 b = ldb4(B, ldb, k);
        if (kW) b = scale4(b, w(k));
        float x[RM];
#pragma unroll
        for (int i = 0; i < RM; ++i) x[i] = A[i * lda + k];
        fma_row<RM>(acc, x, b);
    }
}

// acc += sum_{k0 <= k < k1} A[k][i] w(k) B(k, 0..3) with A column-major (row k of A holds the
// RM values of this block contiguously, 4 * RM-byte aligned): one vector load of A per k.
template <int RM, class Wk = NoWeight>
__device__ __forceinline__ void mac_c(Acc<RM>& acc, const float* A, int lda, const float* B, int ldb, int k0, int k1,
                                      Wk w = Wk{}) {
    constexpr bool kW = !std::is_same<Wk, NoWeight>::value;
#pragma unroll 4
    for (int k = k0; k < k1; ++k) {
        float4 b = ldb4(B, ldb, k);
        if (kW) b = scale4(b, w(k));
        float x[RM];
        ldv<RM>(x, A + (size_t)k * lda);
        fma_row<RM>(acc, x, b);
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
