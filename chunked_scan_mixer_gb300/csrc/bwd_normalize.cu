// Element-wise steps of the ratio-normalised backward (page "Higher-order Linear
// Attention", section summary §2 and §5.1: the normalised output divides the masked
// output by the masked denominator).
//
// With o_t = num_t / (den_t + eps), num the unnormalised output and den the same pair sum
// with every v_j replaced by 1, the quotient rule gives
//     dL/dnum_t = dO_t / (den_t + eps),   dL/dden_t = -(dO_t . num_t) / (den_t + eps)^2.
// Both num and den are unnormalised outputs of the same recurrence: den is the output for
// the value rows e_0 = (1, 0, ..., 0). So the gradients are those of two unnormalised
// backward passes: one with (v, dL/dnum), and one with (e_0, dL/dden e_0^T), which adds to
// dq and dk only.  The two parts of dq and dk can each be tens of times larger than their
// sum, so the composition runs in float32 (bf16 inputs are widened first and the gradients
// rounded at the end).  The kernels below build e_0 and the two upstream gradients, add the
// second pass's dq, dk into the first's, and convert between bf16 and float32.
#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kThreads = 256;

// rows x w float32 with column 0 = 1 and every other column 0.
__global__ void __launch_bounds__(kThreads) unit_first_column_kernel(float* e0, size_t count, int w) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i < count) e0[i] = (i % (size_t)w) == 0 ? 1.f : 0.f;
}

// One warp per token row t: den = den_out[t][0], s = dO_t . num_t,
// dnum[t] = dO_t / (den + eps), dden[t] = (-s / (den + eps)^2, 0, ..., 0).
__global__ void __launch_bounds__(kThreads)
    quotient_rule_kernel(const float* __restrict__ dout, const float* __restrict__ num,
                         const float* __restrict__ den_out, float* __restrict__ dnum, float* __restrict__ dden,
                         size_t rows, int dv, int w, float eps) {
    const size_t row = (size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* o = dout + row * dv;
    const float* x = num + row * dv;
    float s = 0.f;
    for (int j = lane; j < dv; j += 32) s += o[j] * x[j];
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    const float inv = 1.f / (den_out[row * w] + eps);
    for (int j = lane; j < dv; j += 32) dnum[row * dv + j] = o[j] * inv;
    for (int j = lane; j < w; j += 32) dden[row * w + j] = j == 0 ? -s * inv * inv : 0.f;
}

// a += b, float32, count a multiple of 4.
__global__ void __launch_bounds__(kThreads) add_into_kernel(float* a, const float* b, size_t count4) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= count4) return;
    float4 x = reinterpret_cast<float4*>(a)[i];
    const float4 y = reinterpret_cast<const float4*>(b)[i];
    x.x += y.x;
    x.y += y.y;
    x.z += y.z;
    x.w += y.w;
    reinterpret_cast<float4*>(a)[i] = x;
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

int launch_unit_first_column(float* e0, size_t rows, int w, cudaStream_t st) {
    const size_t c = rows * (size_t)w;
    if (c == 0) return 0;
    unit_first_column_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(e0, c, w);
    return done();
}

int launch_quotient_rule(const float* dout, const float* num, const float* den_out, float* dnum, float* dden,
                         size_t rows, int dv, int w, float eps, cudaStream_t st) {
    if (rows == 0) return 0;
    quotient_rule_kernel<<<blocks_for(rows, kThreads / 32), kThreads, 0, st>>>(dout, num, den_out, dnum, dden, rows,
                                                                                dv, w, eps);
    return done();
}

int launch_add_into(float* a, const float* b, size_t count, cudaStream_t st) {
    const size_t c = count / 4;
    if (c == 0) return 0;
    add_into_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(a, b, c);
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
