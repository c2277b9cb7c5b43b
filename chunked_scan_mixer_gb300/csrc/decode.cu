// Single-token streaming decode step of masked HLA-2 (page "Higher-order Linear
// Attention", section summary §3.1: online updates at O(d^2 + d dv) per token with a
// constant-size state; technical summary item "1. Zweite Ordnung HLA").
//
// One CTA per head.  The state (S, C, G, m, h) is read and written exactly once, in
// three passes that each stream one matrix with 128-bit accesses:
//   pass S:  S' = g S + k k^T,                 u = S' q
//   pass C:  r = C^T k (old C),  C' = g C + q v^T,   w = C'^T u
//   pass G:  G' = g^2 G + g k r^T,             z = G'^T q
//   out = w - z  (= q^T (S' C' - G')),  den = u . m' - q . h'
// with m' = g m + q and h' = g^2 h + g k (k . m).  G and h use the pre-update C, m.
// The unmasked output (section summary §3: q^T S' C', denominator u . m') needs neither
// G nor h: that variant skips pass G and the h update and leaves both untouched, so its
// state traffic is S, C and m only.
#include <cooperative_groups.h>

#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDim = 128;

// 128-bit streaming state accesses.  Win is the state block the access must stay in: the
// debug build checks it (HLA2_IN) and skips an access outside it; the normal build ignores it.
struct Win {
    const float* lo;
    const float* hi;
};
__device__ __forceinline__ float4 ld_stream(const float* p, const Win& w) {
    if (!HLA2_IN(p >= w.lo && p + 4 <= w.hi, 301)) return make_float4(0.f, 0.f, 0.f, 0.f);
    return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_stream(float* p, float4 v, const Win& w) {
    if (HLA2_IN(p >= w.lo && p + 4 <= w.hi, 302)) __stcs(reinterpret_cast<float4*>(p), v);
}

template <int NT = kThreads>
__device__ __forceinline__ float block_sum(float x, float* red) {
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) s += red[w];
    return s;
}

// Column sums of a d x dv pass: each thread holds partial sums for 4 columns
// (column group tid % (dv/4)); combine threads that share a column group.
template <int NT = kThreads>
__device__ __forceinline__ void column_reduce(float4 p, int dv, float* red /*[NT / 32][kMaxDim]*/,
                                              float* result /*[dv]*/) {
    const int lpc = dv / 4;  // lanes per row (<= 32, power of two)
    for (int o = lpc; o < 32; o <<= 1) {
        p.x += __shfl_xor_sync(0xffffffffu, p.x, o);
        p.y += __shfl_xor_sync(0xffffffffu, p.y, o);
        p.z += __shfl_xor_sync(0xffffffffu, p.z, o);
        p.w += __shfl_xor_sync(0xffffffffu, p.w, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane < lpc) *reinterpret_cast<float4*>(&red[warp * kMaxDim + lane * 4]) = p;
    __syncthreads();
    for (int c = threadIdx.x; c < dv; c += NT) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) s += red[w * kMaxDim + c];
        result[c] = s;
    }
    __syncthreads();
}

// COMPACT: the state uses the compact layout (S block-triangular, see compact_off).
// UM: unmasked output (no G, h).
template <typename T, bool COMPACT, bool UM>
__global__ void __launch_bounds__(kThreads)
    decode_step_kernel(float* __restrict__ state, const T* __restrict__ q, const T* __restrict__ k,
                       const T* __restrict__ v, T* __restrict__ out, int H, int d, int dv,
                       const float* __restrict__ gamma, int normalize, float eps) {
    __shared__ __align__(16) float qs[kMaxDim], ks[kMaxDim], vs[kMaxDim], us[kMaxDim];
    __shared__ __align__(16) float rs[kMaxDim], ws[kMaxDim], zs[kMaxDim];
    __shared__ __align__(16) float red[kWarps * kMaxDim];
    const int head = blockIdx.x, tid = threadIdx.x;
    const float g = head_decay(gamma, head, H), g2 = g * g;
    const size_t sf = COMPACT ? compact_state_floats(d, dv) : raw_state_floats(d, dv);
    float* S = state + (size_t)head * sf;
    const Win win{S, S + sf};
    const PackOff po = COMPACT ? compact_off(d, dv) : pack_off(d, dv);
    float *C = S + po.C, *G = S + po.G, *m = S + po.m, *hh = S + po.h;

    for (int i = tid; i < d; i += kThreads) {
        qs[i] = to_f32(q[(size_t)head * d + i]);
        ks[i] = to_f32(k[(size_t)head * d + i]);
    }
    for (int i = tid; i < dv; i += kThreads) vs[i] = to_f32(v[(size_t)head * dv + i]);
    __syncthreads();

    // m' = g m + q;  h' = g^2 h + g k (k . m_old)
    float km = 0.f;
    if (!UM) {
        for (int i = tid; i < d; i += kThreads) km += ks[i] * m[i];
        km = block_sum(km, red);
        __syncthreads();  // every warp has read red before pass S may reuse it
    }
    float mh_dot = 0.f;  // this thread's part of u . m' - q . h', formed after pass S

    // ---- pass S ----------------------------------------------------------------------
    if (COMPACT) {
        // S' = g S + k k^T and u = S' q on the block-triangular storage.  As in the packed
        // pass, d/4 lanes share a row and lane l owns column chunk l (columns 4l..4l+3);
        // in row a it has data when l >= a/4 (the row's stored part starts at the diagonal
        // block).  The row part S'[a][4l..] . q[4l..] is reduced across the row's lanes;
        // right of the diagonal block the mirror S'[a][4l+e] q[a] (the entry S'[4l+e][a] of
        // the lower triangle) is summed per lane and reduced over the rows at the end.
        const int lpr = d / 4;
        const int l = tid % lpr, c = 4 * l;
        const int rows_per = kThreads / lpr;
        float4 mir = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int a0 = tid / lpr; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d && l >= (a >> 2)) x[u] = ld_stream(S + compact_row(a, d) + (size_t)(c - 4 * (a >> 2)), win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                float part = 0.f;
                if (a < d && l >= (a >> 2)) {
                    const float ka = ks[a];
                    float4 y = x[u];
                    y.x = g * y.x + ka * ks[c + 0];
                    y.y = g * y.y + ka * ks[c + 1];
                    y.z = g * y.z + ka * ks[c + 2];
                    y.w = g * y.w + ka * ks[c + 3];
                    st_stream(S + compact_row(a, d) + (size_t)(c - 4 * (a >> 2)), y, win);
                    part = y.x * qs[c] + y.y * qs[c + 1] + y.z * qs[c + 2] + y.w * qs[c + 3];
                    if (l > (a >> 2)) {
                        const float qa = qs[a];
                        mir.x += y.x * qa;
                        mir.y += y.y * qa;
                        mir.z += y.z * qa;
                        mir.w += y.w * qa;
                    }
                }
                for (int o = lpr >> 1; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (a < d && l == 0) us[a] = part;
            }
        }
        column_reduce(mir, d, red, zs);  // zs is free until pass G
        for (int i = tid; i < d; i += kThreads) us[i] += zs[i];
    } else {
        const int lpr = d / 4;               // lanes per row
        const int n4 = d * d / 4;
        for (int base = 0; base < n4; base += kThreads * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * kThreads + tid;
                if (i < n4) x[u] = ld_stream(S + (size_t)i * 4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * kThreads + tid;
                float part = 0.f;
                const int a = (i * 4) / d, c = (i * 4) % d;
                if (i < n4) {
                    const float ka = ks[a];
                    float4 y = x[u];
                    y.x = g * y.x + ka * ks[c + 0];
                    y.y = g * y.y + ka * ks[c + 1];
                    y.z = g * y.z + ka * ks[c + 2];
                    y.w = g * y.w + ka * ks[c + 3];
                    st_stream(S + (size_t)i * 4, y, win);
                    part = y.x * qs[c] + y.y * qs[c + 1] + y.z * qs[c + 2] + y.w * qs[c + 3];
                }
                // all lanes of a row group take part (rows are aligned to lpr lanes)
                for (int o = lpr >> 1; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (i < n4 && (i % lpr) == 0) us[a] = part;
            }
        }
    }
    __syncthreads();

    // m, h and the denominator's vector terms
    for (int i = tid; i < d; i += kThreads) {
        const float mn = g * m[i] + qs[i];
        m[i] = mn;
        mh_dot += us[i] * mn;
        if (!UM) {
            const float hn = g2 * hh[i] + g * ks[i] * km;
            hh[i] = hn;
            mh_dot -= qs[i] * hn;
        }
    }

    // ---- pass C ------------------------------------------------------------------------
    {
        const int lpc = dv / 4;
        const int rows_per = kThreads / lpc;
        const int c4 = (tid % lpc) * 4;
        float4 pr = make_float4(0.f, 0.f, 0.f, 0.f), pw = pr;
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(C + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float ka = ks[a], qa = qs[a], ua = us[a];
                float4 y = x[u];
                if (!UM) { pr.x += ka * y.x; pr.y += ka * y.y; pr.z += ka * y.z; pr.w += ka * y.w; }
                y.x = g * y.x + qa * vs[c4 + 0];
                y.y = g * y.y + qa * vs[c4 + 1];
                y.z = g * y.z + qa * vs[c4 + 2];
                y.w = g * y.w + qa * vs[c4 + 3];
                pw.x += ua * y.x; pw.y += ua * y.y; pw.z += ua * y.z; pw.w += ua * y.w;
                st_stream(C + (size_t)a * dv + c4, y, win);
            }
        }
        if (!UM) column_reduce(pr, dv, red, rs);
        column_reduce(pw, dv, red, ws);
    }

    // ---- pass G ------------------------------------------------------------------------
    if (!UM) {
        const int lpc = dv / 4;
        const int rows_per = kThreads / lpc;
        const int c4 = (tid % lpc) * 4;
        float4 pz = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 r4 = *reinterpret_cast<const float4*>(&rs[c4]);
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(G + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float gk = g * ks[a], qa = qs[a];
                float4 y = x[u];
                y.x = g2 * y.x + gk * r4.x;
                y.y = g2 * y.y + gk * r4.y;
                y.z = g2 * y.z + gk * r4.z;
                y.w = g2 * y.w + gk * r4.w;
                pz.x += qa * y.x; pz.y += qa * y.y; pz.z += qa * y.z; pz.w += qa * y.w;
                st_stream(G + (size_t)a * dv + c4, y, win);
            }
        }
        column_reduce(pz, dv, red, zs);
    }

    float inv = 1.f;
    if (normalize) {
        const float den = block_sum(mh_dot, red);
        inv = 1.f / (den + eps);
    }
    for (int e = tid; e < dv; e += kThreads)
        out[(size_t)head * dv + e] = from_f32<T>((UM ? ws[e] : ws[e] - zs[e]) * inv);
}

// AHLA decode step (technical summary item "2. ... (AHLA)": streaming summaries P^KV, m^K,
// E, n; section summary §6.1), one CTA per head, state [P d*dv | E d*dv | m d | n d]:
//   pass P:  P' = g P + k v^T,            inner = P'^T q
//   pass E:  E' = g E + k inner^T,        o = E'^T q
//   m' = g m + k,  n' = g n + k (q . m'),  den = q . n'
// Each matrix is read and written once with 128-bit accesses.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    ahla_decode_kernel(float* __restrict__ state, const T* __restrict__ q, const T* __restrict__ k,
                       const T* __restrict__ v, T* __restrict__ out, int H, int d, int dv,
                       const float* __restrict__ gamma, int normalize, float eps) {
    __shared__ __align__(16) float qs[kMaxDim], ks[kMaxDim], vs[kMaxDim], is[kMaxDim], os[kMaxDim];
    __shared__ __align__(16) float red[kWarps * kMaxDim];
    const int head = blockIdx.x, tid = threadIdx.x;
    const float g = head_decay(gamma, head, H);
    float* P = state + (size_t)head * (2 * (size_t)d * dv + 2 * (size_t)d);
    const Win win{P, P + 2 * (size_t)d * dv + 2 * (size_t)d};
    float* E = P + (size_t)d * dv;
    float* m = E + (size_t)d * dv;
    float* nn = m + d;
    for (int i = tid; i < d; i += kThreads) {
        qs[i] = to_f32(q[(size_t)head * d + i]);
        ks[i] = to_f32(k[(size_t)head * d + i]);
    }
    for (int i = tid; i < dv; i += kThreads) vs[i] = to_f32(v[(size_t)head * dv + i]);
    __syncthreads();

    const int lpc = dv / 4, rows_per = kThreads / lpc, c4 = (tid % lpc) * 4;
    // pass P: P' = g P + k v^T and inner = P'^T q
    {
        float4 pi = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(P + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float ka = ks[a], qa = qs[a];
                float4 y = x[u];
                y.x = g * y.x + ka * vs[c4 + 0];
                y.y = g * y.y + ka * vs[c4 + 1];
                y.z = g * y.z + ka * vs[c4 + 2];
                y.w = g * y.w + ka * vs[c4 + 3];
                pi.x += qa * y.x; pi.y += qa * y.y; pi.z += qa * y.z; pi.w += qa * y.w;
                st_stream(P + (size_t)a * dv + c4, y, win);
            }
        }
        column_reduce(pi, dv, red, is);
    }
    // pass E: E' = g E + k inner^T and o = E'^T q
    {
        float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 i4 = *reinterpret_cast<const float4*>(&is[c4]);
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(E + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float ka = ks[a], qa = qs[a];
                float4 y = x[u];
                y.x = g * y.x + ka * i4.x;
                y.y = g * y.y + ka * i4.y;
                y.z = g * y.z + ka * i4.z;
                y.w = g * y.w + ka * i4.w;
                po.x += qa * y.x; po.y += qa * y.y; po.z += qa * y.z; po.w += qa * y.w;
                st_stream(E + (size_t)a * dv + c4, y, win);
            }
        }
        column_reduce(po, dv, red, os);
    }
    // m' = g m + k;  n' = g n + k (q . m');  den = q . n'
    float qm = 0.f;
    for (int i = tid; i < d; i += kThreads) {
        const float mn = g * m[i] + ks[i];
        m[i] = mn;
        qm += qs[i] * mn;
    }
    qm = block_sum(qm, red);
    float qn = 0.f;
    for (int i = tid; i < d; i += kThreads) {
        const float nv = g * nn[i] + ks[i] * qm;
        nn[i] = nv;
        qn += qs[i] * nv;
    }
    float inv = 1.f;
    if (normalize) inv = 1.f / (block_sum(qn, red) + eps);
    for (int e = tid; e < dv; e += kThreads) out[(size_t)head * dv + e] = from_f32<T>(os[e] * inv);
}

// Packed [S d*d | C | G | m | h] -> compact (upper block triangle of S), one CTA per head.
__global__ void __launch_bounds__(kThreads) state_to_compact_kernel(const float* __restrict__ full,
                                                                   float* __restrict__ compact, int d, int dv) {
    const size_t head = blockIdx.x;
    const float* src = full + head * raw_state_floats(d, dv);
    float* dst = compact + head * compact_state_floats(d, dv);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int a = warp; a < d; a += kWarps) {
        const int b0 = 4 * (a >> 2);
        float* row = dst + compact_row(a, d);
        for (int b = b0 + lane; b < d; b += 32) row[b - b0] = src[(size_t)a * d + b];
    }
    const size_t tail = 2 * (size_t)d * dv + 2 * (size_t)d, cs = compact_s_floats(d), fs = (size_t)d * d;
    for (size_t i = threadIdx.x; i < tail; i += kThreads) dst[cs + i] = src[fs + i];
}

// Compact -> packed, S mirrored from its stored upper block triangle.
__global__ void __launch_bounds__(kThreads) state_from_compact_kernel(const float* __restrict__ compact,
                                                                     float* __restrict__ full, int d, int dv) {
    const size_t head = blockIdx.x;
    const float* src = compact + head * compact_state_floats(d, dv);
    float* dst = full + head * raw_state_floats(d, dv);
    for (int e = threadIdx.x; e < d * d; e += kThreads) {
        const int a = e / d, b = e % d;
        dst[e] = b >= 4 * (a >> 2) ? src[compact_row(a, d) + (b - 4 * (a >> 2))]
                                   : src[compact_row(b, d) + (a - 4 * (b >> 2))];
    }
    const size_t tail = 2 * (size_t)d * dv + 2 * (size_t)d, cs = compact_s_floats(d), fs = (size_t)d * d;
    for (size_t i = threadIdx.x; i < tail; i += kThreads) dst[fs + i] = src[cs + i];
}

// Streaming step of the masked third-order output at gamma = 1 (technical summary item
// "3. Dritte Ordnung HLA": masked streaming with the prefix moments S^K, P^KV; reading: the
// output is q^T Y with Y = sum_j (S^K_j q_j)(P_j^T q_j)^T).  One CTA per head, state
// [S d*d | P d*dv | Y d*dv | m d | y d], each matrix streamed once with 128-bit accesses:
//   pass S:  S' = S + k k^T,          p = S' q        (row form; S is symmetric)
//   pass P:  P' = P + k v^T,          u = P'^T q
//   pass Y:  Y' = Y + p u^T,          o = Y'^T q
//   m' = m + k,  y' = y + p (q . m'),  den = q . y'
template <typename T>
__global__ void __launch_bounds__(kThreads)
    hla3_decode_kernel(float* __restrict__ state, const T* __restrict__ q, const T* __restrict__ k,
                       const T* __restrict__ v, T* __restrict__ out, int d, int dv, int normalize, float eps) {
    __shared__ __align__(16) float qs[kMaxDim], ks[kMaxDim], vs[kMaxDim], ps[kMaxDim], us[kMaxDim], os[kMaxDim];
    __shared__ __align__(16) float red[kWarps * kMaxDim];
    const int head = blockIdx.x, tid = threadIdx.x;
    float* S = state + (size_t)head * ((size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d);
    const Win win{S, S + (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d};
    float* P = S + (size_t)d * d;
    float* Y = P + (size_t)d * dv;
    float* m = Y + (size_t)d * dv;
    float* y = m + d;
    for (int i = tid; i < d; i += kThreads) {
        qs[i] = to_f32(q[(size_t)head * d + i]);
        ks[i] = to_f32(k[(size_t)head * d + i]);
    }
    for (int i = tid; i < dv; i += kThreads) vs[i] = to_f32(v[(size_t)head * dv + i]);
    __syncthreads();

    // ---- pass S (row form, as the second-order step) ------------------------------------
    {
        const int lpr = d / 4, n4 = d * d / 4;
        for (int base = 0; base < n4; base += kThreads * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * kThreads + tid;
                if (i < n4) x[u] = ld_stream(S + (size_t)i * 4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * kThreads + tid;
                float part = 0.f;
                const int a = (i * 4) / d, c = (i * 4) % d;
                if (i < n4) {
                    const float ka = ks[a];
                    float4 z = x[u];
                    z.x += ka * ks[c + 0];
                    z.y += ka * ks[c + 1];
                    z.z += ka * ks[c + 2];
                    z.w += ka * ks[c + 3];
                    st_stream(S + (size_t)i * 4, z, win);
                    part = z.x * qs[c] + z.y * qs[c + 1] + z.z * qs[c + 2] + z.w * qs[c + 3];
                }
                for (int o = lpr >> 1; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (i < n4 && (i % lpr) == 0) ps[a] = part;
            }
        }
    }
    // m' = m + k and q . m'
    float qm = 0.f;
    for (int i = tid; i < d; i += kThreads) {
        const float mn = m[i] + ks[i];
        m[i] = mn;
        qm += qs[i] * mn;
    }
    qm = block_sum(qm, red);  // also orders pass S's writes of ps before their reads below
    __syncthreads();          // every warp has read red before pass P reuses it

    const int lpc = dv / 4, rows_per = kThreads / lpc, c4 = (tid % lpc) * 4;
    // ---- pass P: P' = P + k v^T, u = P'^T q -------------------------------------------------
    {
        float4 pu = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(P + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float ka = ks[a], qa = qs[a];
                float4 z = x[u];
                z.x += ka * vs[c4 + 0];
                z.y += ka * vs[c4 + 1];
                z.z += ka * vs[c4 + 2];
                z.w += ka * vs[c4 + 3];
                pu.x += qa * z.x; pu.y += qa * z.y; pu.z += qa * z.z; pu.w += qa * z.w;
                st_stream(P + (size_t)a * dv + c4, z, win);
            }
        }
        column_reduce(pu, dv, red, us);
    }
    // ---- pass Y: Y' = Y + p u^T, o = Y'^T q ---------------------------------------------------
    {
        float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 u4 = *reinterpret_cast<const float4*>(&us[c4]);
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(Y + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float pa = ps[a], qa = qs[a];
                float4 z = x[u];
                z.x += pa * u4.x;
                z.y += pa * u4.y;
                z.z += pa * u4.z;
                z.w += pa * u4.w;
                po.x += qa * z.x; po.y += qa * z.y; po.z += qa * z.z; po.w += qa * z.w;
                st_stream(Y + (size_t)a * dv + c4, z, win);
            }
        }
        column_reduce(po, dv, red, os);
    }
    float qy = 0.f;
    for (int i = tid; i < d; i += kThreads) {
        const float yn = y[i] + ps[i] * qm;
        y[i] = yn;
        qy += qs[i] * yn;
    }
    float inv = 1.f;
    if (normalize) inv = 1.f / (block_sum(qy, red) + eps);
    for (int e = tid; e < dv; e += kThreads) out[(size_t)head * dv + e] = from_f32<T>(os[e] * inv);
}

// Decode step with multi-query sharing (section summary §5.2: one key moment per group of
// query heads, state O(d^2 + h d dv) per group).  One CTA per query head; the `group` CTAs
// of a key group form a thread-block cluster.  Each CTA advances one block of rows of the
// group's S, so S is streamed once per group:
//   pass S (rows a of this CTA's block):  S'[a] = g S[a] + k_a k^T,  u_i[a] = S'[a] . q_i
// for every head i of the group (u = S' q; S' is symmetric).  The row blocks of u are then
// gathered through distributed shared memory, and each CTA streams its own head's C and G
// as the single-head step does, with the group's k and v.  With one CTA per head the grid
// is as large as the single-head step's (8192 CTAs for 256 sequences x 32 heads), which
// keeps the waves short; one CTA per group (2048) ran 1.7 waves with the last one two-thirds
// full.  key_state [N*Hk][d*d]; head_state [N*Hk*group][C | G | m | h].
constexpr int kMaxGroup = 8;

template <typename T, bool UM>
__global__ void __launch_bounds__(kThreads)
    decode_mq_kernel(float* __restrict__ key_state, float* __restrict__ head_state, const T* __restrict__ q,
                     const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ out, int Hk, int group,
                     int d, int dv, const float* __restrict__ gamma, int normalize, float eps) {
    __shared__ __align__(16) float qs[kMaxGroup][kMaxDim], us[kMaxGroup][kMaxDim];
    __shared__ __align__(16) float ks[kMaxDim], vs[kMaxDim], uo[kMaxDim], rs[kMaxDim], ws[kMaxDim], zs[kMaxDim];
    __shared__ __align__(16) float red[kWarps * kMaxDim];
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    const int head = blockIdx.x;           // query head (sequence-major)
    const int grp = head / group;          // its key group
    const int r = (int)cluster.block_rank();  // == head % group
    const float g = head_decay(gamma, grp, Hk), g2 = g * g;
    float* S = key_state + (size_t)grp * d * d;
    Win win{S, S + (size_t)d * d};  // the key group's S; the head's block from pass C on

    for (int i = tid; i < d; i += kThreads) ks[i] = to_f32(k[(size_t)grp * d + i]);
    for (int i = tid; i < dv; i += kThreads) vs[i] = to_f32(v[(size_t)grp * dv + i]);
    for (int i = tid; i < group * d; i += kThreads) qs[i / d][i % d] = to_f32(q[(size_t)grp * group * d + i]);
    __syncthreads();

    // ---- pass S over this CTA's rows [lo, hi) ----------------------------------------------
    {
        const int lo = r * d / group, hi = (r + 1) * d / group;
        const int lpr = d / 4;  // lanes per row; a warp holds 32 / lpr whole rows
        const int rows_per = kThreads / lpr;
        const int c4 = (tid % lpr) * 4;
        const int iters = (hi - lo + rows_per * 4 - 1) / (rows_per * 4);  // the same for every thread
        for (int it = 0; it < iters; ++it) {
            const int a0 = lo + it * rows_per * 4 + tid / lpr;
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < hi) x[u] = ld_stream(S + (size_t)a * d + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                const bool ok = a < hi;
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ok) {
                    const float ka = ks[a];
                    y = x[u];
                    y.x = g * y.x + ka * ks[c4 + 0];
                    y.y = g * y.y + ka * ks[c4 + 1];
                    y.z = g * y.z + ka * ks[c4 + 2];
                    y.w = g * y.w + ka * ks[c4 + 3];
                    st_stream(S + (size_t)a * d + c4, y, win);
                }
                for (int i = 0; i < group; ++i) {  // every lane takes part in the shuffles
                    float part = y.x * qs[i][c4] + y.y * qs[i][c4 + 1] + y.z * qs[i][c4 + 2] + y.w * qs[i][c4 + 3];
                    for (int o = lpr >> 1; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                    if (ok && (tid % lpr) == 0) us[i][a] = part;
                }
            }
        }
    }
    // The other CTAs' row blocks of u are read after the cluster barrier; its arrival is
    // split from the wait so that the m and h updates fill the gap.
    auto arrived = cluster.barrier_arrive();

    // ---- this head: m, h, pass C, pass G, output ----------------------------------------------
    const size_t hsf = 2 * (size_t)d * dv + 2 * (size_t)d;
    float* C = head_state + (size_t)head * hsf;
    win = Win{C, C + hsf};
    float* G = C + (size_t)d * dv;
    float* m = G + (size_t)d * dv;
    float* hh = m + d;
    const float* qi = qs[r];
    float km = 0.f;
    if (!UM) {
        for (int a = tid; a < d; a += kThreads) km += ks[a] * m[a];
        km = block_sum(km, red);
        __syncthreads();  // every warp has read red before pass C reuses it
    }
    float mh_dot = 0.f;  // q . (S' m' - h') = u . m' - q . h'; the u part once u is here
    for (int a = tid; a < d; a += kThreads) {
        const float mn = g * m[a] + qi[a];
        m[a] = mn;
        if (!UM) {
            const float hn = g2 * hh[a] + g * ks[a] * km;
            hh[a] = hn;
            mh_dot -= qi[a] * hn;
        }
    }
    cluster.barrier_wait(std::move(arrived));
    for (int a = tid; a < d; a += kThreads) {
        int owner = 0;
        while (owner + 1 < group && (owner + 1) * d / group <= a) ++owner;
        const float* src = cluster.map_shared_rank(&us[0][0], owner);
        uo[a] = src[r * kMaxDim + a];
        mh_dot += uo[a] * m[a];  // m[a] was written by this thread above
    }
    auto gathered = cluster.barrier_arrive();  // this CTA's reads of the others are done
    __syncthreads();
    const int lpc = dv / 4;
    const int rows_per = kThreads / lpc;
    const int c4 = (tid % lpc) * 4;
    {  // pass C
        float4 pr = make_float4(0.f, 0.f, 0.f, 0.f), pw = pr;
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(C + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float ka = ks[a], qa = qi[a], ua = uo[a];
                float4 y = x[u];
                if (!UM) { pr.x += ka * y.x; pr.y += ka * y.y; pr.z += ka * y.z; pr.w += ka * y.w; }
                y.x = g * y.x + qa * vs[c4 + 0];
                y.y = g * y.y + qa * vs[c4 + 1];
                y.z = g * y.z + qa * vs[c4 + 2];
                y.w = g * y.w + qa * vs[c4 + 3];
                pw.x += ua * y.x; pw.y += ua * y.y; pw.z += ua * y.z; pw.w += ua * y.w;
                st_stream(C + (size_t)a * dv + c4, y, win);
            }
        }
        if (!UM) column_reduce(pr, dv, red, rs);
        column_reduce(pw, dv, red, ws);
    }
    if (!UM) {  // pass G
        float4 pz = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 r4 = *reinterpret_cast<const float4*>(&rs[c4]);
        for (int a0 = tid / lpc; a0 < d; a0 += rows_per * 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a < d) x[u] = ld_stream(G + (size_t)a * dv + c4, win);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int a = a0 + u * rows_per;
                if (a >= d) continue;
                const float gk = g * ks[a], qa = qi[a];
                float4 y = x[u];
                y.x = g2 * y.x + gk * r4.x;
                y.y = g2 * y.y + gk * r4.y;
                y.z = g2 * y.z + gk * r4.z;
                y.w = g2 * y.w + gk * r4.w;
                pz.x += qa * y.x; pz.y += qa * y.y; pz.z += qa * y.z; pz.w += qa * y.w;
                st_stream(G + (size_t)a * dv + c4, y, win);
            }
        }
        column_reduce(pz, dv, red, zs);
    }
    float inv = 1.f;
    if (normalize) inv = 1.f / (block_sum(mh_dot, red) + eps);
    for (int e = tid; e < dv; e += kThreads) out[(size_t)head * dv + e] = from_f32<T>((UM ? ws[e] : ws[e] - zs[e]) * inv);
    cluster.barrier_wait(std::move(gathered));  // no CTA leaves while another may still read it
}

template <bool COMPACT, bool UM>
void launch_decode_t(float* state, const void* q, const void* k, const void* v, void* out, long heads, int H, int d,
                     int dv, const float* gamma, int normalize, float eps, bool is_bf16, cudaStream_t st) {
    if (is_bf16)
        decode_step_kernel<bf16, COMPACT, UM><<<(unsigned)heads, kThreads, 0, st>>>(
            state, static_cast<const bf16*>(q), static_cast<const bf16*>(k), static_cast<const bf16*>(v),
            static_cast<bf16*>(out), H, d, dv, gamma, normalize, eps);
    else
        decode_step_kernel<float, COMPACT, UM><<<(unsigned)heads, kThreads, 0, st>>>(
            state, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            static_cast<float*>(out), H, d, dv, gamma, normalize, eps);
}

}  // namespace

int launch_decode_step(float* state, const void* q, const void* k, const void* v, void* out,
                       int N, int H, int d, int dv, const float* gamma, int normalize, float eps,
                       bool is_bf16, bool compact, bool unmasked, cudaStream_t st) {
    const long heads = (long)N * H;
    if (heads <= 0) return 0;
    if (compact && unmasked)
        launch_decode_t<true, true>(state, q, k, v, out, heads, H, d, dv, gamma, normalize, eps, is_bf16, st);
    else if (compact)
        launch_decode_t<true, false>(state, q, k, v, out, heads, H, d, dv, gamma, normalize, eps, is_bf16, st);
    else if (unmasked)
        launch_decode_t<false, true>(state, q, k, v, out, heads, H, d, dv, gamma, normalize, eps, is_bf16, st);
    else
        launch_decode_t<false, false>(state, q, k, v, out, heads, H, d, dv, gamma, normalize, eps, is_bf16, st);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_decode_mq(float* key_state, float* head_state, const void* q, const void* k, const void* v, void* out,
                     int N, int Hk, int group, int d, int dv, const float* gamma, int normalize, float eps,
                     bool is_bf16, bool unmasked, cudaStream_t st) {
    const long heads = (long)N * Hk * group;
    if (heads <= 0) return 0;
    if (group < 1 || group > kMaxGroup) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)heads);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)group;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
#define HLA2_MQ(T, UMV)                                                                                  \
    e = cudaLaunchKernelEx(&cfg, decode_mq_kernel<T, UMV>, key_state, head_state, static_cast<const T*>(q), \
                           static_cast<const T*>(k), static_cast<const T*>(v), static_cast<T*>(out), Hk, group, d, \
                           dv, gamma, normalize, eps)
    if (is_bf16 && unmasked) {
        HLA2_MQ(bf16, true);
    } else if (is_bf16) {
        HLA2_MQ(bf16, false);
    } else if (unmasked) {
        HLA2_MQ(float, true);
    } else {
        HLA2_MQ(float, false);
    }
#undef HLA2_MQ
    if (e != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_hla3_decode_step(float* state, const void* q, const void* k, const void* v, void* out, long heads, int d,
                            int dv, int normalize, float eps, bool is_bf16, cudaStream_t st) {
    if (heads <= 0) return 0;
    if (is_bf16)
        hla3_decode_kernel<bf16><<<(unsigned)heads, kThreads, 0, st>>>(
            state, static_cast<const bf16*>(q), static_cast<const bf16*>(k), static_cast<const bf16*>(v),
            static_cast<bf16*>(out), d, dv, normalize, eps);
    else
        hla3_decode_kernel<float><<<(unsigned)heads, kThreads, 0, st>>>(
            state, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            static_cast<float*>(out), d, dv, normalize, eps);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_ahla_decode_step(float* state, const void* q, const void* k, const void* v, void* out, int N, int H,
                            int d, int dv, const float* gamma, int normalize, float eps, bool is_bf16,
                            cudaStream_t st) {
    const long heads = (long)N * H;
    if (heads <= 0) return 0;
    if (is_bf16)
        ahla_decode_kernel<bf16><<<(unsigned)heads, kThreads, 0, st>>>(
            state, static_cast<const bf16*>(q), static_cast<const bf16*>(k), static_cast<const bf16*>(v),
            static_cast<bf16*>(out), H, d, dv, gamma, normalize, eps);
    else
        ahla_decode_kernel<float><<<(unsigned)heads, kThreads, 0, st>>>(
            state, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            static_cast<float*>(out), H, d, dv, gamma, normalize, eps);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_state_compact(const float* src, float* dst, long heads, int d, int dv, bool to_compact, cudaStream_t st) {
    if (heads <= 0) return 0;
    if (to_compact)
        state_to_compact_kernel<<<(unsigned)heads, kThreads, 0, st>>>(src, dst, d, dv);
    else
        state_from_compact_kernel<<<(unsigned)heads, kThreads, 0, st>>>(src, dst, d, dv);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2

HLA2_DEBUG_READER(decode)
