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
// dq and dk only. The kernels below build e_0 and the two upstream gradients, and add the
// second pass's dq, dk into the first's.
#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kThreads = 256;

// rows x d bf16 with column 0 = 1 and every other column 0 (d a multiple of 8).
__global__ void __launch_bounds__(kThreads) unit_first_column_kernel(bf16* e0, size_t chunks8, int d) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= chunks8) return;
    uint4 z = make_uint4(0u, 0u, 0u, 0u);
    if ((i * 8) % (size_t)d == 0) z.x = 0x3F80u;  // bf16 1.0 in the low half: element 0
    reinterpret_cast<uint4*>(e0)[i] = z;
}

// One warp per token row t: den = den_out[t][0], s = dO_t . num_t,
// dnum[t] = dO_t / (den + eps), dden[t] = (-s / (den + eps)^2, 0, ..., 0).
__global__ void __launch_bounds__(kThreads)
    quotient_rule_kernel(const bf16* __restrict__ dout, const bf16* __restrict__ num,
                         const bf16* __restrict__ den_out, bf16* __restrict__ dnum, bf16* __restrict__ dden,
                         size_t rows, int dv, int d, float eps) {
    const size_t row = (size_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const bf16* o = dout + row * dv;
    const bf16* x = num + row * dv;
    float s = 0.f;
    for (int j = lane; j < dv; j += 32) s += to_f32(o[j]) * to_f32(x[j]);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    const float inv = 1.f / (to_f32(den_out[row * d]) + eps);
    for (int j = lane; j < dv; j += 32) dnum[row * dv + j] = from_f32<bf16>(to_f32(o[j]) * inv);
    for (int j = lane; j < d; j += 32) dden[row * d + j] = from_f32<bf16>(j == 0 ? -s * inv * inv : 0.f);
}

// a += b, bf16, count a multiple of 8.
__global__ void __launch_bounds__(kThreads) add_into_kernel(bf16* a, const bf16* b, size_t chunks8) {
    const size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (i >= chunks8) return;
    uint4 x = reinterpret_cast<uint4*>(a)[i];
    const uint4 y = reinterpret_cast<const uint4*>(b)[i];
    uint32_t* xs = reinterpret_cast<uint32_t*>(&x);
    const uint32_t* ys = reinterpret_cast<const uint32_t*>(&y);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float lo = __uint_as_float(xs[w] << 16) + __uint_as_float(ys[w] << 16);
        const float hi = __uint_as_float(xs[w] & 0xFFFF0000u) + __uint_as_float(ys[w] & 0xFFFF0000u);
        xs[w] = pack_bf16x2(lo, hi);
    }
    reinterpret_cast<uint4*>(a)[i] = x;
}

unsigned blocks_for(size_t n, int per_block) { return (unsigned)((n + per_block - 1) / per_block); }

}  // namespace

int launch_unit_first_column(bf16* e0, size_t rows, int d, cudaStream_t st) {
    const size_t c = rows * (size_t)d / 8;
    if (c == 0) return 0;
    unit_first_column_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(e0, c, d);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_quotient_rule(const bf16* dout, const bf16* num, const bf16* den_out, bf16* dnum, bf16* dden,
                         size_t rows, int dv, int d, float eps, cudaStream_t st) {
    if (rows == 0) return 0;
    quotient_rule_kernel<<<blocks_for(rows, kThreads / 32), kThreads, 0, st>>>(dout, num, den_out, dnum, dden, rows,
                                                                                dv, d, eps);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_add_into(bf16* a, const bf16* b, size_t count, cudaStream_t st) {
    const size_t c = count / 8;
    if (c == 0) return 0;
    add_into_kernel<<<blocks_for(c, kThreads), kThreads, 0, st>>>(a, b, c);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2
