// Element-wise steps of the ratio-normalised backward (page "Higher-order Linear
// Attention", section summary §2 and §5.1: the normalised output divides the masked
// output by the masked denominator).
//
// With o_t = num_t / (den_t + eps), num the unnormalised output and den the same pair sum
// with every v_j replaced by 1, the quotient rule gives
//     dL/dnum_t = dO_t / (den_t + eps),   dL/dden_t = -(dO_t . num_t) / (den_t + eps)^2.
// num and den are the unnormalised outputs of one recurrence for the widened value rows
// [v_j | 1 | 0 ...] (dv + w0 columns, column dv the unit), so one unnormalised forward gives
// [num | den] and one unnormalised backward with the upstream gradient [dL/dnum | dL/dden]
// gives dq, dk and [dv | .].  dq and dk are then the difference of a numerator part and a
// denominator part that can each be tens of times larger than their sum, so the composition
// runs in float32 (bf16 inputs are widened first and the gradients rounded at the end).
// The kernels below widen the values, apply the quotient rule, narrow the value gradient
// and convert between bf16 and float32.
#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld_f32(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_f32(const bf16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_val(float* p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_val(bf16* p, size_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// ve[t] = [v_t | 1 | 0 ...]: rows x w float32 from rows x dv values (w > dv).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    widen_values_kernel(const T* __restrict__ v, float* __restrict__ ve, size_t count, int dv, int w) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= count) return;
    const size_t t = i / (size_t)w;
    const int j = (int)(i - t * (size_t)w);
    ve[i] = j < dv ? ld_f32(v, t * dv + j) : (j == dv ? 1.f : 0.f);
}

// One warp per token row t of nd = [num | den | .] (w wide): den = nd[t][dv],
// s = dO_t . num_t, dnd[t] = [dO_t / (den + eps) | -s / (den + eps)^2 | 0 ...].
template <typename T>
__global__ void __launch_bounds__(kThreads)
    quotient_rule_kernel(const T* __restrict__ dout, const float* __restrict__ nd, float* __restrict__ dnd,
                         size_t rows, int dv, int w, float eps) {
    const size_t row = (size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* x = nd + row * w;
    float s = 0.f;
    for (int j = lane; j < dv; j += 32) s += ld_f32(dout, row * dv + j) * x[j];
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    const float inv = 1.f / (x[dv] + eps);
    for (int j = lane; j < w; j += 32)
        dnd[row * w + j] = j < dv ? ld_f32(dout, row * dv + j) * inv : (j == dv ? -s * inv * inv : 0.f);
}

// out[t][j] = dve[t][j] for j < dv (the value gradient out of [dv | .], w wide).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    narrow_values_kernel(const float* __restrict__ dve, T* __restrict__ out, size_t count, int dv, int w) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= count) return;
    const size_t t = i / (size_t)dv;
    const int j = (int)(i - t * (size_t)dv);
    st_val(out, i, dve[t * w + j]);
}

// 8 elements per thread; count a multiple of 8.
__global__ void __launch_bounds__(kThreads) bf16_to_f32_kernel(const bf16* __restrict__ src, float* __restrict__ dst,
                                                               size_t count8) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= count8) return;
    const uint4 c = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    float4 lo, hi;
    lo.x = __uint_as_float(w[0] << 16);
    lo.y = __uint_as_float(w[0] & 0xFFFF0000u);
    lo.z = __uint_as_float(w[1] << 16);
    lo.w = __uint_as_float(w[1] & 0xFFFF0000u);
    hi.x = __uint_as_float(w[2] << 16);
    hi.y = __uint_as_float(w[2] & 0xFFFF0000u);
    hi.z = __uint_as_float(w[3] << 16);
    hi.w = __uint_as_float(w[3] & 0xFFFF0000u);
    reinterpret_cast<float4*>(dst)[2 * i] = lo;
    reinterpret_cast<float4*>(dst)[2 * i + 1] = hi;
}

__global__ void __launch_bounds__(kThreads) f32_to_bf16_kernel(const float* __restrict__ src, bf16* __restrict__ dst,
                                                               size_t count8) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= count8) return;
    const float4 lo = reinterpret_cast<const float4*>(src)[2 * i];
    const float4 hi = reinterpret_cast<const float4*>(src)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16x2(lo.x, lo.y);
    o.y = pack_bf16x2(lo.z, lo.w);
    o.z = pack_bf16x2(hi.x, hi.y);
    o.w = pack_bf16x2(hi.z, hi.w);
    reinterpret_cast<uint4*>(dst)[i] = o;
}

unsigned blocks_for(size_t n, int per_block) { return (unsigned)((n + per_block - 1) / per_block); }

int done() { return cudaPeekAtLastError() == cudaSuccess ? 0 : -1; }

}  // namespace

int launch_widen_values(const void* v, float* ve, size_t rows, int dv, int w, bool is_bf16, cudaStream_t st) {
    const size_t c = rows * (size_t)w;
    if (c == 0) return 0;
    if (is_bf16)
        widen_values_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(static_cast<const bf16*>(v), ve, c, dv, w);
    else
        widen_values_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(static_cast<const float*>(v), ve, c, dv, w);
    return done();
}

int launch_quotient_rule(const void* dout, const float* nd, float* dnd, size_t rows, int dv, int w, float eps,
                         bool is_bf16, cudaStream_t st) {
    if (rows == 0) return 0;
    const unsigned g = blocks_for(rows, kThreads / 32);
    if (is_bf16)
        quotient_rule_kernel<<<g, kThreads, 0, st>>>(static_cast<const bf16*>(dout), nd, dnd, rows, dv, w, eps);
    else
        quotient_rule_kernel<<<g, kThreads, 0, st>>>(static_cast<const float*>(dout), nd, dnd, rows, dv, w, eps);
    return done();
}

int launch_narrow_values(const float* dve, void* out, size_t rows, int dv, int w, bool is_bf16, cudaStream_t st) {
    const size_t c = rows * (size_t)dv;
    if (c == 0) return 0;
    if (is_bf16)
        narrow_values_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(dve, static_cast<bf16*>(out), c, dv, w);
    else
        narrow_values_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(dve, static_cast<float*>(out), c, dv, w);
    return done();
}

int launch_convert_bf16_f32(const bf16* src, float* dst, size_t count, cudaStream_t st) {
    const size_t c = count / 8;
    if (c == 0) return 0;
    bf16_to_f32_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(src, dst, c);
    return done();
}

int launch_convert_f32_bf16(const float* src, bf16* dst, size_t count, cudaStream_t st) {
    const size_t c = count / 8;
    if (c == 0) return 0;
    f32_to_bf16_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(src, dst, c);
    return done();
}

}  // namespace hla2
