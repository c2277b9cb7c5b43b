// Device helpers shared by the HLA-2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hla2.h"

namespace hla2 {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// Planning shared by host code and kernels.
// ---------------------------------------------------------------------------

// Segmentation of one head's sequence: `nseg` segments of `seg_chunks` chunks
// (the last one may be shorter, and the last chunk may be partial).
struct Plan {
    int BH, H, n, d, dv, W;
    int nchunks;     // ceil(n / W)
    int seg_chunks;  // chunks per segment
    int nseg;        // segments per head
};

// Float offsets of the forward workspace arrays (each 64-float aligned).  The first 64
// floats hold the status word (an int at offset 0): kernels with bounded waits write a
// nonzero code there when a wait gives up.
constexpr size_t kStatusFloats = 64;
struct FwdLayout {
    size_t SB, CB, ZB, mB, yB;   // summaries, [BH][nsum][...]
    size_t Sin, Zin, yin;        // carries,   [BH][nseg][...]
    size_t Clast, mlast;         // C, m carried into the last segment, [BH][...]
    size_t fin;                  // raw final (S, C, m, Z, y), [BH][...]
    size_t total;                // floats
};

__host__ __device__ inline size_t align64(size_t x) { return (x + 63) & ~size_t(63); }

__host__ __device__ inline size_t raw_state_floats(int d, int dv) {
    return (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d;
}

// nsum: summaries kept per head (the forward needs nseg - 1, the backward nseg).
inline FwdLayout fwd_layout(const Plan& p, int nsum) {
    FwdLayout L;
    const size_t BH = p.BH, ns = p.nseg, nsm = nsum > 0 ? nsum : 0;
    const size_t dd = (size_t)p.d * p.d, ddv = (size_t)p.d * p.dv, d = p.d;
    size_t o = kStatusFloats;
    L.SB = o;    o = align64(o + BH * nsm * dd);
    L.CB = o;    o = align64(o + BH * nsm * ddv);
    L.ZB = o;    o = align64(o + BH * nsm * ddv);
    L.mB = o;    o = align64(o + BH * nsm * d);
    L.yB = o;    o = align64(o + BH * nsm * d);
    L.Sin = o;   o = align64(o + BH * ns * dd);
    L.Zin = o;   o = align64(o + BH * ns * ddv);
    L.yin = o;   o = align64(o + BH * ns * d);
    L.Clast = o; o = align64(o + BH * ddv);
    L.mlast = o; o = align64(o + BH * d);
    L.fin = o;   o = align64(o + BH * raw_state_floats(p.d, p.dv));
    L.total = o;
    return L;
}

// Raw final-state block of one head, float offsets: S | C | m | Z | y.
struct RawOff {
    size_t S, C, m, Z, y;
};
__host__ __device__ inline RawOff raw_off(int d, int dv) {
    RawOff r;
    r.S = 0;
    r.C = (size_t)d * d;
    r.m = r.C + (size_t)d * dv;
    r.Z = r.m + d;
    r.y = r.Z + (size_t)d * dv;
    return r;
}

// Packed (public) state of one head, float offsets: S | C | G | m | h.
struct PackOff {
    size_t S, C, G, m, h;
};
__host__ __device__ inline PackOff pack_off(int d, int dv) {
    PackOff r;
    r.S = 0;
    r.C = (size_t)d * d;
    r.G = r.C + (size_t)d * dv;
    r.m = r.G + (size_t)d * dv;
    r.h = r.m + d;
    return r;
}

// Compact decode state of one head: S symmetric, stored block-triangularly -- row a holds
// S[a][b] for b = 4 floor(a/4) .. d-1 (the upper triangle plus the lower half of the 4 x 4
// diagonal blocks), rows back to back; then C, G, m, h as in the packed layout.  Every row
// starts on a multiple of 4 floats.  S takes d (d + 4) / 2 floats.
__host__ __device__ inline size_t compact_s_floats(int d) { return (size_t)d * (d + 4) / 2; }
__host__ __device__ inline size_t compact_state_floats(int d, int dv) {
    return compact_s_floats(d) + 2 * (size_t)d * dv + 2 * (size_t)d;
}
// float offset of row a of the compact S
//   block row j = a / 4 starts after 4 rows of d - 4 j' floats for every j' < j
__host__ __device__ inline size_t compact_row(int a, int d) {
    const long long j = a >> 2, r = a & 3;
    return (size_t)(4 * j * d - 8 * j * (j - 1) + r * (d - 4 * j));
}
__host__ __device__ inline PackOff compact_off(int d, int dv) {
    PackOff r;
    r.S = 0;
    r.C = compact_s_floats(d);
    r.G = r.C + (size_t)d * dv;
    r.m = r.G + (size_t)d * dv;
    r.h = r.m + d;
    return r;
}

// ---------------------------------------------------------------------------
// Debug build (compiled with -DHLA2_DEBUG).  HLA2_IN(cond, site) evaluates to cond; a
// false cond records `site` in this translation unit's debug word (the first site wins), and
// the caller skips the access it guards.  Nothing traps.  In the normal build HLA2_IN is
// `true` and costs nothing.  HLA2_DEBUG_READER(name) defines, at the end of a file that uses
// HLA2_IN, the host function that reads (and optionally clears) that file's word.
// ---------------------------------------------------------------------------
#ifdef HLA2_DEBUG
static __device__ int hla2_dbg_word;
__device__ __forceinline__ bool hla2_dbg_in(bool ok, int site) {
    if (!ok) atomicCAS(&hla2_dbg_word, 0, site);
    return ok;
}
#define HLA2_IN(cond, site) hla2_dbg_in((cond), (site))
#define HLA2_DEBUG_READER(name)                                                            \
    namespace hla2 {                                                                       \
    int dbg_read_##name(bool clear) {                                                      \
        int v = 0;                                                                         \
        if (cudaMemcpyFromSymbol(&v, hla2_dbg_word, sizeof(int)) != cudaSuccess) return -1; \
        if (clear) {                                                                       \
            const int z = 0;                                                               \
            if (cudaMemcpyToSymbol(hla2_dbg_word, &z, sizeof(int)) != cudaSuccess) return -1; \
        }                                                                                  \
        return v;                                                                          \
    }                                                                                      \
    }
#else
#define HLA2_IN(cond, site) true
#define HLA2_DEBUG_READER(name)
#endif

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// decay^k with k possibly fractional-free integer; log2 of the decay precomputed.
__device__ __forceinline__ float pow_decay(float log2g, float k) { return exp2f(k * log2g); }

__device__ __forceinline__ float head_decay(const float* gamma, int bh, int H) {
    return gamma ? __ldg(gamma + (bh % H)) : 1.0f;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with launch_pdl may start while the
// kernel before it on the stream is still running (once every CTA of that kernel has run
// pdl_trigger or exited); it must run pdl_wait before it reads or writes memory that an
// earlier kernel of the stream touches.  pdl_wait returns once the kernels before it have
// completed and their writes are visible; without the launch attribute it returns at once.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// cp.async (16-byte global -> shared copies)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

// ---------------------------------------------------------------------------
// Warp-level bf16 tensor-core tiles: mma.m16n8k16 with ldmatrix operand loads.
//
// Fragment ownership (g = lane / 4, c = lane % 4):
//   A 16x16: a0 (g, 2c..2c+1), a1 (g+8, 2c..), a2 (g, 2c+8..), a3 (g+8, 2c+8..)
//   B 16x8 : b0 (k 2c..2c+1, n g), b1 (k 2c+8.., n g)
//   D 16x8 : d0,d1 (g, 2c..2c+1), d2,d3 (g+8, 2c..2c+1)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc (16 x 16 tile, two n-halves of 8) += A[m0:m0+16, k0:k1] * B[k0:k1, n0:n0+16].
//   A_T = false: A stored [M][K] (row stride lda):   A(m,k) = A[m*lda + k]
//   A_T = true : A stored [K][M]:                    A(m,k) = A[k*lda + m]
//   B_T = false: B stored [N][K]:                    B(k,n) = B[n*ldb + k]
//   B_T = true : B stored [K][N]:                    B(k,n) = B[k*ldb + n]
// k0, k1 multiples of 16; all addresses 16-byte aligned (strides multiple of 8).
template <bool A_T, bool B_T>
__device__ __forceinline__ void warp_tile_mma(float (&acc)[2][4], const bf16* A, int lda, int m0,
                                              const bf16* B, int ldb, int n0, int k0, int k1) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, r = lane & 7;
    for (int k = k0; k < k1; k += 16) {
        uint32_t a[4];
        if (!A_T) {
            const bf16* p = A + (size_t)(m0 + r + (mi & 1) * 8) * lda + k + (mi >> 1) * 8;
            ldsm_x4(a[0], a[1], a[2], a[3], p);
        } else {
            const bf16* p = A + (size_t)(k + r + (mi >> 1) * 8) * lda + m0 + (mi & 1) * 8;
            ldsm_x4_t(a[0], a[1], a[2], a[3], p);
        }
        uint32_t b[4];
        if (!B_T) {
            const bf16* p = B + (size_t)(n0 + r + (mi >> 1) * 8) * ldb + k + (mi & 1) * 8;
            ldsm_x4(b[0], b[1], b[2], b[3], p);
        } else {
            const bf16* p = B + (size_t)(k + r + (mi & 1) * 8) * ldb + n0 + (mi >> 1) * 8;
            ldsm_x4_t(b[0], b[1], b[2], b[3], p);
        }
        mma_16816(acc[0], a, b[0], b[1]);
        mma_16816(acc[1], a, b[2], b[3]);
    }
}

__device__ __forceinline__ void zero_acc(float (&acc)[2][4]) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;
}

// Row / column of accumulator element (h, i) of a 16x16 tile at (m0, n0).
__device__ __forceinline__ int acc_row(int m0, int i) { return m0 + ((threadIdx.x & 31) >> 2) + (i >> 1) * 8; }
__device__ __forceinline__ int acc_col(int n0, int h, int i) {
    return n0 + h * 8 + ((threadIdx.x & 31) & 3) * 2 + (i & 1);
}

}  // namespace hla2
