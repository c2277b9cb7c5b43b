// tcgen05 chunk kernel of the masked HLA-2 forward for d = dv = 64 and chunk width 128
// (bf16 inputs, fp32 state, unnormalised).  Same per-chunk algebra as the mma.sync kernel
// (fwd_chunk_mma.cuh: p_t = S_t q_t, Z_t = g^2 Z_{t-1} + p_t v_t^T, o_t = q_t^T Z_t), with
// the chunk products on the 5th-generation tensor cores.  Tensor memory holds four 64-column
// regions T0 | T1 | T3 | T2 (T1T3 contiguous):
//
//   MMA1  A   = Q K^T                                   -> T0T1 (128 x 128 fp32)
//   EPI1  A~  = A * [i <= r] g^(r-i)  (bf16, packed)    -> T3 (A operand of MMA2)
//         K~  = diag(g^(Wc-1-i)) K                      (bf16, shared memory)
//   MMA2  A~ K -> T2;   Q S0 -> T0
//   EPI2  P   = g^(r+1) Q S0 + A~ K;  P (bf16, K-major), P~ = diag(g^(2(Wc-1-j))) P  (smem)
//   MMA3  B   = Q P^T -> T0T1;   Q Z0 -> T2
//   EPI3  B~  = B * [j <= r] g^(2(r-j))  (bf16)        -> T3
//   MMA4  B~ V -> T0;  then ST = [K~^T ; P~^T] [K | V]  -> T1T3 (dS = K~^T K, dZ = P~^T V)
//   EPI4  out = g^(2(r+1)) Q Z0 + B~ V  (bf16, global);
//         S <- g^Wc S + dS,  Z <- g^(2Wc) Z + dZ  (fp32 registers); bf16 S0, Z0 (smem)
//
// Summary mode (segment summaries for the inter-segment scan) keeps EPI1/MMA2/EPI2 and then
// computes [Q~^T ; P~^T] V -> T1 (dC, dZ; Q~ = diag(g^(Wc-1-j)) Q) and [K~^T ; K~^T] K -> T3
// (dS twice, so that every thread owns 16 of its columns), accumulating S, C, Z from zero.
//
// UM (unmasked output q^T S C = p^T C, section summary §3 and §4.1): MMA3 forms P Q^T and
// P C0 (C0 in the Z0 slot), EPI3 masks with g^(r-j), out = g^(r+1) P C0 + B~ V, EPI2 writes
// Q~ = diag(g^(Wc-1-j)) Q in place of P~ so that the state product gives dC, and the
// summary pass needs no A~ or P: after the scaled copies it forms [Q~^T ; Q~^T] V (dC
// twice) and [K~^T ; K~^T] K (dS), so C lands in both the C and the Z slots.
//
// Roles: warp 0 allocates tensor memory and one of its threads issues the TMA loads and every
// MMA; warps 1..8 move data between tensor memory, registers and shared memory (warp w reads
// TMEM lanes 32*(w%4)..+31, i.e. token/feature rows, and half (w-1)/4 of the columns).  Two
// CTAs share an SM (256 TMEM columns, ~107 KB of shared memory each).  Every wait is bounded;
// on a timeout the kernel records where in a status word, drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace hla2 {

namespace {

constexpr int kW = 128, kD = 64;
constexpr int kThreads = 288;  // 1 control warp + 8 epilogue warps
constexpr uint32_t kTile = 128 * 128;  // bytes of one [128][64] bf16 SW128 tile
// shared memory slots (byte offsets from the 1024-aligned base)
constexpr uint32_t oQ = 0, oK = kTile, oV = 2 * kTile, oP = 3 * kTile, oKt = 4 * kTile, oPt = 5 * kTile;
constexpr uint32_t oZ0 = 6 * kTile;            // [64][64] bf16 (8 KB); S0 shares the P~ slot
constexpr uint32_t oGP = oZ0 + 8192;           // decay table g^0 .. g^(2W), 257 floats
constexpr uint32_t oBar = oGP + 1088;
constexpr uint32_t oMisc = oBar + 16 * 8;      // tmem base, abort flag
constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;  // + alignment slack
// TMEM columns
constexpr uint32_t T0 = 0, T1 = 64, T3 = 128, T2 = 192, kTmemCols = 256;

enum Bar { FULLQ = 0, FULLKV, BA, BAT, BP, BPS, BB, BBT, BO, BST, BS, kBarCount };

struct TcMaps {
    CUtensorMap q, k, v;
};

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// 8 bf16 of a 16-byte chunk, scaled, repacked
__device__ __forceinline__ uint4 scale_chunk(uint4 c, float s) {
    uint4 o;
    o.x = pack_bf16x2(s * bf_lo(c.x), s * bf_hi(c.x));
    o.y = pack_bf16x2(s * bf_lo(c.y), s * bf_hi(c.y));
    o.z = pack_bf16x2(s * bf_lo(c.z), s * bf_hi(c.z));
    o.w = pack_bf16x2(s * bf_lo(c.w), s * bf_hi(c.w));
    return o;
}

__device__ __forceinline__ uint4 pack8(const float* f, float s) {
    uint4 o;
    o.x = pack_bf16x2(s * f[0], s * f[1]);
    o.y = pack_bf16x2(s * f[2], s * f[3]);
    o.z = pack_bf16x2(s * f[4], s * f[5]);
    o.w = pack_bf16x2(s * f[6], s * f[7]);
    return o;
}

// Masked, decayed 32-column block of a 128 x 128 chunk product for row r:
//   out[i] = [i <= r] base^(r - i) * in[i],  i = cb .. cb + 31,
// with base = g (A~) or g^2 (B~), read from src (TMEM, fp32) and written packed (16 columns)
// to dst.  Blocks entirely above the diagonal of this warp's rows are written as zeros
// without reading; the factors are stepped multiplicatively from base^(r - cb).  rs, when
// given, accumulates the block's fp32 row sum (the normalised output's denominator).
__device__ __forceinline__ void masked_pack(uint32_t src, int r, int cb, int warp_row0, float first, float step_up,
                                            uint32_t (&pk)[16], float* rs = nullptr) {
    if (cb > warp_row0 + 31) {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
    } else {
        uint32_t v[32];
        tc::tmem_ld32(src, v);
        tc::tmem_wait_ld();
        float f = first;  // base^(r - cb)
        const bool diag = cb + 31 > warp_row0;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            float a0 = f * __uint_as_float(v[j]);
            f *= step_up;
            float a1 = f * __uint_as_float(v[j + 1]);
            f *= step_up;
            if (diag) {
                a0 = cb + j <= r ? a0 : 0.f;
                a1 = cb + j + 1 <= r ? a1 : 0.f;
            }
            if (rs) *rs += a0 + a1;
            pk[j / 2] = pack_bf16x2(a0, a1);
        }
    }
}

// Sums over a warp's 32 rows of a 16-column block held one row per lane (cs[c], column c):
// halving steps leave lane l with column l & 15 summed over the 16 lanes that share bit 4, the
// last step adds the other 16.  Every lane returns the sum of column l & 15.
__device__ __forceinline__ float warp_colsum16(float (&cs)[16], int lane) {
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = up ? cs[i] : cs[i + off];
            const float keep = up ? cs[i + off] : cs[i];
            cs[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return cs[0] + __shfl_xor_sync(0xffffffffu, cs[0], 16);
}

__device__ __forceinline__ void masked_block(uint32_t src, uint32_t dst, int r, int cb, int warp_row0,
                                             float first, float step_up, float* rs = nullptr) {
    uint32_t pk[16];
    masked_pack(src, r, cb, warp_row0, first, step_up, pk, rs);
    tc::tmem_st16(dst, pk);
}

template <int MODE, bool UM>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_chunk_tc_kernel(const __grid_constant__ TcMaps maps, const ChunkArgs a, int* status) {
    constexpr bool SUMMARY = MODE == kSummary;
    constexpr bool CHAIN = !(UM && SUMMARY);  // A~ and P are formed
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gp = reinterpret_cast<float*>(sm + oGP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + oMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const float g = head_decay(a.gamma, bh, a.H);
    const float log2g = log2f(g);

    for (int i = tid; i < 2 * kW + 1; i += kThreads) gp[i] = pow_decay(log2g, (float)i);
    if (tid == 0) {
        for (int b = 0; b < kBarCount; ++b) {
            const bool from_epilogue = (b == BAT || b == BPS || b == BBT || b == BS);
            tc::mbar_init(&bars[b], from_epilogue ? 8 : 1);
        }
        *abort = 0;
        tc::mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    const int nit = c_end - c_begin;

    if (warp == 0) {
        // ------------------------------------------------------------ control thread
        if (lane == 0 && nit > 0) {
            const uint32_t sQ = smem_u32(sm + oQ), sK = smem_u32(sm + oK), sV = smem_u32(sm + oV);
            const uint32_t sP = smem_u32(sm + oP), sKt = smem_u32(sm + oKt), sPt = smem_u32(sm + oPt);
            const uint32_t sS0 = sPt, sZ0 = smem_u32(sm + oZ0);
            auto load_q = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FULLQ], kTile);
                tc::tma_load_3d(sm + oQ, &maps.q, 0, c * kW, bh, &bars[FULLQ]);
            };
            auto load_kv = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FULLKV], 2 * kTile);
                tc::tma_load_3d(sm + oK, &maps.k, 0, c * kW, bh, &bars[FULLKV]);
                tc::tma_load_3d(sm + oV, &maps.v, 0, c * kW, bh, &bars[FULLKV]);
            };
            constexpr uint32_t I_AB = tc::idesc_bf16(128, 128, 0, 0);   // K-major x K-major, N = 128
            constexpr uint32_t I_QX = tc::idesc_bf16(128, 64, 0, 1);    // K-major x MN-major, N = 64
            constexpr uint32_t I_TS64 = tc::idesc_bf16(128, 64, 0, 1);  // A (TMEM) x MN-major B, N = 64
            constexpr uint32_t I_ST = tc::idesc_bf16(128, 128, 1, 1);   // MN-major x MN-major, N = 128
            constexpr uint32_t I_ST64 = tc::idesc_bf16(128, 64, 1, 1);  // MN-major x MN-major, N = 64
            load_q(c_begin);
            load_kv(c_begin);
            int loads = 1;
            for (int it = 0; it < nit; ++it) {
                const uint32_t ph = it & 1;
                tc::mbar_wait(&bars[FULLQ], ph, abort, status, 1);
                tc::mbar_wait(&bars[FULLKV], ph, abort, status, 2);
                if (it > 0) tc::mbar_wait(&bars[BS], ph ^ 1, abort, status, 3);
                tc::fence_after_sync();
                if (CHAIN) {
                    // MMA1: A = Q K^T -> T0T1
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024),
                                   tc::smem_desc(sK + 32 * ks, 16, 1024), I_AB, ks > 0);
                    tc::mma_commit(&bars[BA]);
                    tc::mbar_wait(&bars[BAT], ph, abort, status, 4);
                    tc::fence_after_sync();
                    // MMA2: A~ K -> T2;  Q S0 -> T0
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + T2, tmem + T3 + 8 * ks, tc::smem_desc(sK + 2048 * ks, 16, 1024), I_TS64,
                                   ks > 0);
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024),
                                   tc::smem_desc(sS0 + 2048 * ks, 16, 1024), I_QX, ks > 0);
                    tc::mma_commit(&bars[BP]);
                }
                tc::mbar_wait(&bars[BPS], ph, abort, status, 5);
                tc::fence_after_sync();
                if (!SUMMARY) {
                    // MMA3: B = Q P^T -> T0T1;  Q Z0 -> T2   (unmasked: P Q^T and P C0)
                    const uint32_t sL = UM ? sP : sQ, sR = UM ? sQ : sP;
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T0, tc::smem_desc(sL + 32 * ks, 16, 1024), tc::smem_desc(sR + 32 * ks, 16, 1024),
                                   I_AB, ks > 0);
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T2, tc::smem_desc(sL + 32 * ks, 16, 1024),
                                   tc::smem_desc(sZ0 + 2048 * ks, 16, 1024), I_QX, ks > 0);
                    tc::mma_commit(&bars[BB]);
                    tc::mbar_wait(&bars[BBT], ph, abort, status, 6);
                    tc::fence_after_sync();
                    if (it + 1 < nit) load_q(c_begin + it + 1);  // Q is no longer read
                    // MMA4: B~ V -> T0, then ST once B~ (T3) has been read
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + T0, tmem + T3 + 8 * ks, tc::smem_desc(sV + 2048 * ks, 16, 1024), I_TS64, ks > 0);
                    tc::mma_commit(&bars[BO]);
                    tc::mbar_wait(&bars[BO], ph, abort, status, 7);
                    tc::fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T1, tc::smem_desc(sKt + 2048 * ks, kTile, 1024),
                                   tc::smem_desc(sK + 2048 * ks, kTile, 1024), I_ST, ks > 0);
                } else {
                    if (it + 1 < nit) load_q(c_begin + it + 1);  // Q~ (P slot) is used below, not Q
                    // [Q~^T ; P~^T] V -> T1 (dC, dZ);  [K~^T ; K~^T] K -> T3 (dS twice)
                    // (unmasked: [Q~^T ; Q~^T] V, dC twice)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T1, tc::smem_desc(sP + 2048 * ks, UM ? 0 : 2 * kTile, 1024),
                                   tc::smem_desc(sV + 2048 * ks, 16, 1024), I_ST64, ks > 0);
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T3, tc::smem_desc(sKt + 2048 * ks, 0, 1024),
                                   tc::smem_desc(sK + 2048 * ks, 16, 1024), I_ST64, ks > 0);
                }
                tc::mma_commit(&bars[BST]);
                tc::mbar_wait(&bars[BST], ph, abort, status, 8);  // K, V free
                if (it + 1 < nit) {
                    load_kv(c_begin + it + 1);
                    ++loads;
                }
            }
            // drain (bounded, ignoring the abort flag) so that nothing is in flight at exit
            volatile int never = 0;
            tc::mbar_wait(&bars[BST], (nit - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FULLKV], (loads - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FULLQ], (SUMMARY || !*abort ? nit - 1 : loads - 1) & 1, &never, nullptr, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q4 = warp & 3, h = (warp - 1) >> 2;
        const int r = 32 * q4 + lane;  // TMEM lane = row
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        unsigned char* sQ = sm + oQ;
        unsigned char* sK = sm + oK;
        unsigned char* sP = sm + oP;
        unsigned char* sKt = sm + oKt;
        unsigned char* sPt = sm + oPt;
        unsigned char* sZ0 = sm + oZ0;
        const float ginv = g > 0.f ? 1.f / g : 0.f;
        // fp32 state: output: S row r (r < 64) or Z row r - 64, columns 32h..32h+31.
        //             summary: C row r (r < 64) or Z row r - 64, columns 32h..; and
        //                      S row r % 64, columns 32h + 16 (r / 64) .. +15.
        float st[32];
        float ss[16];
        const size_t sidx = (size_t)bh * a.nseg + seg;
        if (!SUMMARY) {
            const float* src = r < 64 ? a.ws + a.L.Sin + sidx * kD * kD + (size_t)r * kD
                                      : a.ws + a.L.Zin + sidx * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j] = src[32 * h + j];
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) ss[j] = 0.f;
        }
        // bf16 copies of S (P~ slot) and Z (Z0 slot): the B operands of Q S0 and Q Z0
        auto publish_state = [&]() {
            if (!SUMMARY) {
                unsigned char* base = r < 64 ? sPt : sZ0;
                const int row = r & 63;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(base + tc::sw128_chunk(row, 4 * h + j)) = pack8(&st[8 * j], 1.f);
            } else {
                const int row = r & 63, cb = 32 * h + 16 * (r >> 6);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    *reinterpret_cast<uint4*>(sPt + tc::sw128_chunk(row, cb / 8 + j)) = pack8(&ss[8 * j], 1.f);
            }
        };
        publish_state();
        tc::fence_proxy_async();

        for (int it = 0; it < nit; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            // ---- EPI1: A~ -> T3;  K~ (and Q~) -> smem -----------------------------------
            tc::mbar_wait(&bars[FULLQ], ph, abort, status, 11);
            tc::mbar_wait(&bars[FULLKV], ph, abort, status, 12);
            if (CHAIN) {
                tc::mbar_wait(&bars[BA], ph, abort, status, 13);
                tc::fence_after_sync();
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int cb = 64 * h + 32 * p;
                    const float first = r >= cb ? gp[r - cb] : 0.f;
                    masked_block(lrow + T0 + cb, lrow + T3 + cb / 2, r, cb, row0, first, ginv);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[BAT]);
            }
            // K~ (and Q~ in summary mode) rows, features 32h .. 32h+31, while MMA2 runs; they
            // are first read by the MMAs issued after EPI2 / EPI3 (fenced there)
            {
                const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                    *reinterpret_cast<uint4*>(sKt + off) = scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w1);
                    if (SUMMARY)
                        *reinterpret_cast<uint4*>(sP + off) = scale_chunk(*reinterpret_cast<const uint4*>(sQ + off), w1);
                }
            }

            // ---- EPI2: P = g^(r+1) Q S0 + A~ K;  P, P~ -> smem ---------------------------
            // (unmasked: P -> smem and Q~ in the P~ slot; the unmasked summary skips this)
            if (CHAIN) {
                tc::mbar_wait(&bars[BP], ph, abort, status, 14);
                tc::fence_after_sync();
                const float s1 = gp[r + 1];
                const float w2 = r < Wc ? gp[2 * (Wc - 1 - r)] : 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qs[16], ak[16];
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, qs);
                    tc::tmem_ld16(lrow + T2 + 32 * h + 16 * half, ak);
                    tc::tmem_wait_ld();
                    float pv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) pv[j] = s1 * __uint_as_float(qs[j]) + __uint_as_float(ak[j]);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t off = tc::sw128_chunk(r, 4 * h + 2 * half + j);
                        if (!SUMMARY) *reinterpret_cast<uint4*>(sP + off) = pack8(&pv[8 * j], 1.f);
                        if (!UM) *reinterpret_cast<uint4*>(sPt + off) = pack8(&pv[8 * j], w2);
                    }
                }
                if (UM) {  // Q~ rows, features 32h .. 32h+31 (S0 in this slot has been read by MMA2)
                    const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                        *reinterpret_cast<uint4*>(sPt + off) = scale_chunk(*reinterpret_cast<const uint4*>(sQ + off), w1);
                    }
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BPS]);
            if (!SUMMARY) {
                // ---- EPI3: B~ -> T3 ----------------------------------------------------------
                tc::mbar_wait(&bars[BB], ph, abort, status, 15);
                tc::fence_after_sync();
                constexpr int BP2 = UM ? 1 : 2;  // decay power of the second product
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int cb = 64 * h + 32 * p;
                    const float first = r >= cb ? gp[BP2 * (r - cb)] : 0.f;
                    masked_block(lrow + T0 + cb, lrow + T3 + cb / 2, r, cb, row0, first, UM ? ginv : ginv * ginv);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[BBT]);

                // ---- EPI4a: out = g^(2(r+1)) Q Z0 + B~ V ---------------------------------------
                tc::mbar_wait(&bars[BO], ph, abort, status, 16);
                tc::fence_after_sync();
                const float s2 = gp[BP2 * (r + 1)];
                bf16* out = static_cast<bf16*>(a.out) + ((size_t)bh * a.n + (size_t)c * kW + r) * kD + 32 * h;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qz[16], bv[16];
                    tc::tmem_ld16(lrow + T2 + 32 * h + 16 * half, qz);
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, bv);
                    tc::tmem_wait_ld();
                    if (r < Wc) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            float o[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                o[u] = s2 * __uint_as_float(qz[8 * j + u]) + __uint_as_float(bv[8 * j + u]);
                            *reinterpret_cast<uint4*>(out + 16 * half + 8 * j) = pack8(o, 1.f);
                        }
                    }
                }
            }

            // ---- EPI4b: state update ---------------------------------------------------------
            tc::mbar_wait(&bars[BST], ph, abort, status, 17);
            tc::fence_after_sync();
            {
                const float rho = gp[Wc], rho2 = gp[2 * Wc];
                uint32_t v[32];
                if (!SUMMARY) {
                    // ST rows < 64: dS in ST columns 0..63 (T1); rows >= 64: dZ in columns 64..127 (T3)
                    tc::tmem_ld32(lrow + (r < 64 ? T1 : T3) + 32 * h, v);
                    tc::tmem_wait_ld();
                    const float decay = r < 64 || UM ? rho : rho2;  // unmasked: the Z slot holds C
#pragma unroll
                    for (int j = 0; j < 32; ++j) st[j] = decay * st[j] + __uint_as_float(v[j]);
                } else {
                    // T1 rows < 64: dC, rows >= 64: dZ;  T3: dS (rows r and r + 64 identical)
                    tc::tmem_ld32(lrow + T1 + 32 * h, v);
                    uint32_t w[16];
                    tc::tmem_ld16(lrow + T3 + 32 * h + 16 * (r >> 6), w);
                    tc::tmem_wait_ld();
                    const float decay = r < 64 || UM ? rho : rho2;
#pragma unroll
                    for (int j = 0; j < 32; ++j) st[j] = decay * st[j] + __uint_as_float(v[j]);
#pragma unroll
                    for (int j = 0; j < 16; ++j) ss[j] = rho * ss[j] + __uint_as_float(w[j]);
                }
                publish_state();
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BS]);
        }

        if (SUMMARY && seg < a.nsum) {  // (a launch that stores p also covers the last segment)
            const size_t si = (size_t)bh * a.nsum + seg;
            float* dst = r < 64 ? a.ws + a.L.CB + si * kD * kD + (size_t)r * kD
                                : a.ws + a.L.ZB + si * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[32 * h + j] = st[j];
            float* ds = a.ws + a.L.SB + si * kD * kD + (size_t)(r & 63) * kD + 32 * h + 16 * (r >> 6);
#pragma unroll
            for (int j = 0; j < 16; ++j) ds[j] = ss[j];
            if (h == 0 && r < 64) {
                a.ws[a.L.mB + si * kD + r] = 0.f;
                a.ws[a.L.yB + si * kD + r] = 0.f;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Output pass from the stored segment-local p (kOutputP; UM = unmasked, NORM = ratio-normalised).
//
// The summary pass stores, for every token t of segment s, p^sl_t = S^sl_t q_t, where S^sl is
// the key moment accumulated from zero at the segment start (bf16, in the output buffer).
// With the segment's carry-in S_in (section summary §4: the carry enters by one decayed
// product),
//     p_t = p^sl_t + g^(t - t0 + 1) S_in q_t,         t0 = the segment's first token,
// so the key moment leaves the chunk-to-chunk chain: this pass reads q, p^sl and v (no k) and
// carries only Z from chunk to chunk.  Per chunk (local row r, it = chunk index in the segment):
//   MMA-a  Q S_in -> T0                                          (no dependence on Z)
//   EPI-a  P = P^sl + g^(it W + r + 1) Q S_in  (bf16, in place);  P~ = diag(g^(2(Wc-1-r))) P
//   MMA-b  B = Q P^T -> T0T1;  Q Z0 -> T2;  then [P~^T ; P~^T] V -> T3 (dZ, rows 0..63 and again
//          64..127), which runs while EPI-b masks B
//   EPI-b  B~ = B * [j <= r] g^(2(r-j))  (bf16, packed in place over T0; the two warps of a lane
//          quarter order their reads and writes with a named barrier)
//   MMA-c  B~ V -> T1
//   EPI-c  out = g^(2(r+1)) Q Z0 + B~ V  (bf16 tile in smem; one TMA tile store writes it over
//          this chunk's p^sl, already consumed);  Z <- g^(2Wc) Z + dZ  (fp32, 16 columns a
//          thread);  bf16 Z0 (smem)
// MMA-a of the next chunk and the next loads overlap EPI-c.  The unmasked output (UM) forms
// P Q^T and P C0 instead (C0 in the Z0 slot), masks with g^(r-j), scales by g^(r+1), carries
// C (decay g^Wc) and takes dC = [Q~^T ; Q~^T] V with Q~ = diag(g^(Wc-1-r)) Q in the P~ slot.
//
// NORM (masked; section summary §3: the denominator is the same recurrence with every value
// row replaced by 1) divides each output row by den + eps, with
//     den_r = g^(2(r+1)) q_r . y0 + sum_j B~[r][j],     y <- g^(2Wc) y0 + sum_r P~[r],
// y0 the p moment at the chunk start (the segment's carry-in y_in, then updated chunk by
// chunk).  All of it is epilogue arithmetic in fp32: q_r . y0 and the column sums of P~ in
// EPI-a (the column sums by a shuffle reduction over the warp's 32 rows, then per lane
// quarter in shared memory), the row sums of B~ in EPI-b, the division and the y update in
// EPI-c.  The partial sums are added in a fixed order (results reproducible bit for bit).
// Same roles, bounded waits and two CTAs per SM as the kernel above.
namespace outp {

constexpr uint32_t oQ = 0, oP = kTile, oV = 2 * kTile, oPt = 3 * kTile;
constexpr uint32_t oO = 4 * kTile;        // output tile, written by one TMA tile store
constexpr uint32_t oS = 5 * kTile;        // S_in, [64][64] bf16 (8 KB), B operand of Q S_in
constexpr uint32_t oZ0 = oS + 8192;       // Z0, [64][64] bf16 (8 KB), B operand of Q Z0
constexpr uint32_t oGP = oZ0 + 8192;      // decay table g^0 .. g^(2W)
constexpr uint32_t oBar = oGP + 1088;
constexpr uint32_t oMisc = oBar + 16 * 8;
constexpr uint32_t oY = oMisc + 16;       // NORM: y0 [64] fp32
constexpr uint32_t oYP = oY + 256;        // NORM: column sums of P~ per lane quarter [4][64]
constexpr uint32_t oDP = oYP + 1024;      // NORM: denominator partials per column half [2][128]
constexpr uint32_t kSmemBytes = oDP + 1024 + 1024;
constexpr uint32_t T0 = 0, T1 = 64, T2 = 128, T3 = 192;

enum Bar { FQP = 0, FV, BA, BAT, BB, BBT, BC, BOS, kBarCount };

struct Maps {
    CUtensorMap q, p, v;
};

}  // namespace outp

template <bool UM, bool NORM>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_out_p_tc_kernel(const __grid_constant__ outp::Maps maps, const ChunkArgs a, int* status) {
    static_assert(!(UM && NORM), "the unmasked normalised output runs on the other kernels");
    pdl_trigger();
    // this pass's layout (shadows the kernel above)
    constexpr uint32_t oQ = outp::oQ, oP = outp::oP, oV = outp::oV, oPt = outp::oPt, oO = outp::oO, oS = outp::oS,
                       oZ0 = outp::oZ0;
    constexpr uint32_t oGP = outp::oGP, oBar = outp::oBar, oMisc = outp::oMisc;
    constexpr uint32_t T0 = outp::T0, T1 = outp::T1, T2 = outp::T2, T3 = outp::T3;
    constexpr int FQP = outp::FQP, FV = outp::FV, BA = outp::BA, BAT = outp::BAT, BB = outp::BB, BBT = outp::BBT,
                  BC = outp::BC, BOS = outp::BOS, kBarCount = outp::kBarCount;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gp = reinterpret_cast<float*>(sm + oGP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + oMisc + 4);
    float* y0 = reinterpret_cast<float*>(sm + outp::oY);
    float* ypart = reinterpret_cast<float*>(sm + outp::oYP);
    float* dpart = reinterpret_cast<float*>(sm + outp::oDP);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const float g = head_decay(a.gamma, bh, a.H);
    const float log2g = log2f(g);
    const int nit = c_end - c_begin;

    // epilogue thread: TMEM lane / token row r, column half h; Z row zr, columns zc .. zc+15
    const int q4 = warp & 3, h = (warp - 1) >> 2;
    const int r = 32 * q4 + lane;
    const int zr = r & 63, zc = 32 * h + 16 * (r >> 6);
    float zz[16];
    auto publish_z = [&]() {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint4*>(sm + oZ0 + tc::sw128_chunk(zr, zc / 8 + j)) = pack8(&zz[8 * j], 1.f);
    };

    for (int i = tid; i < 2 * kW + 1; i += kThreads) gp[i] = pow_decay(log2g, (float)i);
    if (tid == 0) {
        for (int b = 0; b < kBarCount; ++b) tc::mbar_init(&bars[b], (b == BAT || b == BBT || b == BOS) ? 8 : 1);
        *abort = 0;
        tc::mbar_fence_init();
    }
    pdl_wait();  // everything below reads what the earlier kernels of the forward wrote
    if (warp == 0) {
        tc::tmem_alloc(tmem_holder, kTmemCols);
    } else {
        // carry-in of the segment: S_in (bf16, smem) and Z_in (fp32 registers, bf16 copy in smem)
        const size_t sidx = (size_t)bh * a.nseg + seg;
        if (r < 64) {
            const float* src = a.ws + a.L.Sin + sidx * kD * kD + (size_t)r * kD + 32 * h;
            float t[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) t[j] = src[j];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(sm + oS + tc::sw128_chunk(r, 4 * h + j)) = pack8(&t[8 * j], 1.f);
        }
        const float* zsrc = a.ws + a.L.Zin + sidx * kD * kD + (size_t)zr * kD + zc;
#pragma unroll
        for (int j = 0; j < 16; ++j) zz[j] = zsrc[j];
        publish_z();
        if (NORM && h == 0 && r < 64) y0[r] = a.ws[a.L.yin + sidx * kD + r];
        tc::fence_proxy_async();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ control thread
        if (lane == 0 && nit > 0) {
            const uint32_t sQ = smem_u32(sm + oQ), sP = smem_u32(sm + oP), sV = smem_u32(sm + oV);
            const uint32_t sPt = smem_u32(sm + oPt), sS = smem_u32(sm + oS), sZ0 = smem_u32(sm + oZ0);
            auto load_qp = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FQP], 2 * kTile);
                tc::tma_load_3d(sm + oQ, &maps.q, 0, c * kW, bh, &bars[FQP]);
                tc::tma_load_3d(sm + oP, &maps.p, 0, c * kW, bh, &bars[FQP]);
            };
            auto load_v = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FV], kTile);
                tc::tma_load_3d(sm + oV, &maps.v, 0, c * kW, bh, &bars[FV]);
            };
            constexpr uint32_t I_AB = tc::idesc_bf16(128, 128, 0, 0);   // K-major x K-major, N = 128
            constexpr uint32_t I_QX = tc::idesc_bf16(128, 64, 0, 1);    // K-major x MN-major, N = 64
            constexpr uint32_t I_TS64 = tc::idesc_bf16(128, 64, 0, 1);  // A (TMEM) x MN-major B, N = 64
            constexpr uint32_t I_ST64 = tc::idesc_bf16(128, 64, 1, 1);  // MN-major x MN-major, N = 64
            load_qp(c_begin);
            load_v(c_begin);
            int lqp = 1, lv = 1;
            for (int it = 0; it < nit; ++it) {
                const uint32_t ph = it & 1;
                tc::mbar_wait(&bars[FQP], ph, abort, status, 41);
                tc::fence_after_sync();
                // MMA-a: Q S_in -> T0 (T0's B~ of the previous chunk was read: its MMA-c completed)
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sS + 2048 * ks, 16, 1024),
                               I_QX, ks > 0);
                tc::mma_commit(&bars[BA]);
                tc::mbar_wait(&bars[BAT], ph, abort, status, 42);  // P, P~ written; previous EPI-c done
                tc::fence_after_sync();
                // MMA-b: B = Q P^T -> T0T1;  Q Z0 -> T2   (unmasked: P Q^T and P C0)
                const uint32_t sL = UM ? sP : sQ, sR = UM ? sQ : sP;
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T0, tc::smem_desc(sL + 32 * ks, 16, 1024), tc::smem_desc(sR + 32 * ks, 16, 1024),
                               I_AB, ks > 0);
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T2, tc::smem_desc(sL + 32 * ks, 16, 1024), tc::smem_desc(sZ0 + 2048 * ks, 16, 1024),
                               I_QX, ks > 0);
                tc::mma_commit(&bars[BB]);
                // dZ: [P~^T ; P~^T] V -> T3 (unmasked: [Q~^T ; Q~^T] V), while EPI-b masks B
                tc::mbar_wait(&bars[FV], ph, abort, status, 45);
                tc::fence_after_sync();
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + T3, tc::smem_desc(sPt + 2048 * ks, 0, 1024), tc::smem_desc(sV + 2048 * ks, 16, 1024),
                               I_ST64, ks > 0);
                if (it > 0) {  // the previous chunk's output tile (staged by its EPI-c) -> out
                    tc::mbar_wait(&bars[BOS], ph ^ 1, abort, status, 47);
                    tc::tma_store_3d(&maps.p, sm + oO, 0, (c_begin + it - 1) * kW, bh);
                    tc::bulk_commit();
                }
                tc::mbar_wait(&bars[BB], ph, abort, status, 43);  // Q and P no longer read (Q~ was copied)
                if (it + 1 < nit) {
                    load_qp(c_begin + it + 1);
                    ++lqp;
                }
                tc::mbar_wait(&bars[BBT], ph, abort, status, 44);
                tc::bulk_wait_read_all();  // the output tile slot is free before this chunk's EPI-c
                tc::fence_after_sync();
                // MMA-c: B~ V -> T1 (B~ packed in T0)
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + T1, tmem + T0 + 8 * ks, tc::smem_desc(sV + 2048 * ks, 16, 1024), I_TS64, ks > 0);
                tc::mma_commit(&bars[BC]);
                tc::mbar_wait(&bars[BC], ph, abort, status, 46);  // V, P~ and T0 free
                if (it + 1 < nit) {
                    load_v(c_begin + it + 1);
                    ++lv;
                }
            }
            tc::mbar_wait(&bars[BOS], (nit - 1) & 1, abort, status, 48);  // the last output tile
            tc::tma_store_3d(&maps.p, sm + oO, 0, (c_begin + nit - 1) * kW, bh);
            tc::bulk_commit();
            // drain (bounded, ignoring the abort flag) so that nothing is in flight at exit
            volatile int never = 0;
            tc::mbar_wait(&bars[BC], (nit - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FQP], (lqp - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FV], (lv - 1) & 1, &never, nullptr, 0);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        unsigned char* sP = sm + oP;
        unsigned char* sPt = sm + oPt;
        const float ginv = g > 0.f ? 1.f / g : 0.f;
        for (int it = 0; it < nit; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            // ---- EPI-a: P = P^sl + g^(it W + r + 1) Q S_in;  P (in place), P~ -> smem ----------
            tc::mbar_wait(&bars[FQP], ph, abort, status, 51);
            tc::mbar_wait(&bars[BA], ph, abort, status, 52);
            tc::fence_after_sync();
            float qy = 0.f;  // NORM: q_r . y0 over this thread's 32 columns
            {
                const float f = pow_decay(log2g, (float)(it * kW + r + 1));
                const float w2 = r < Wc ? gp[2 * (Wc - 1 - r)] : 0.f;
                if (NORM) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 qc = *reinterpret_cast<const uint4*>(sm + oQ + tc::sw128_chunk(r, 4 * h + j));
                        const uint32_t qw[4] = {qc.x, qc.y, qc.z, qc.w};
                        const float* yy = y0 + 32 * h + 8 * j;
#pragma unroll
                        for (int u = 0; u < 4; ++u) qy += bf_lo(qw[u]) * yy[2 * u] + bf_hi(qw[u]) * yy[2 * u + 1];
                    }
                }
                if (UM) {  // the state product forms dC = Q~^T V: Q~ = diag(g^(Wc-1-r)) Q in the P~ slot
                    const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                        *reinterpret_cast<uint4*>(sPt + off) =
                            scale_chunk(*reinterpret_cast<const uint4*>(sm + oQ + off), w1);
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qs[16];
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, qs);
                    tc::tmem_wait_ld();
                    float cs[16];  // NORM: this row's P~ over the half's 16 columns
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t off = tc::sw128_chunk(r, 4 * h + 2 * half + j);
                        const uint4 pl = *reinterpret_cast<const uint4*>(sP + off);
                        const uint32_t pw[4] = {pl.x, pl.y, pl.z, pl.w};
                        float pv[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            pv[2 * u] = bf_lo(pw[u]) + f * __uint_as_float(qs[8 * j + 2 * u]);
                            pv[2 * u + 1] = bf_hi(pw[u]) + f * __uint_as_float(qs[8 * j + 2 * u + 1]);
                        }
                        *reinterpret_cast<uint4*>(sP + off) = pack8(pv, 1.f);
                        if (!UM) *reinterpret_cast<uint4*>(sPt + off) = pack8(pv, w2);
#pragma unroll
                        for (int u = 0; u < 8; ++u) cs[8 * j + u] = w2 * pv[u];
                    }
                    if (NORM) {  // column sums over the warp's 32 rows
                        const float t = warp_colsum16(cs, lane);
                        if (lane < 16) ypart[64 * q4 + 32 * h + 16 * half + lane] = t;
                    }
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BAT]);

            // ---- EPI-b: B~ packed over T0 (unmasked: decay g^(r-j)) -------------------------------
            // Warp h of a lane quarter reads B's columns 64h .. 64h+63 and writes their packed
            // pairs to T0 columns 32h .. 32h+31.  Warp h = 1's writes land on columns warp h = 0
            // reads, so warp h = 0 signals (named barrier 1 + q4) once it has read them.
            tc::mbar_wait(&bars[BB], ph, abort, status, 53);
            tc::fence_after_sync();
            constexpr int BP2 = UM ? 1 : 2;  // decay power of the second product
            const float step2 = UM ? ginv : ginv * ginv;
            float rs = 0.f;  // NORM: row sum of B~ over this warp's 64 columns
            if (h == 0) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const float first = r >= 32 * p ? gp[BP2 * (r - 32 * p)] : 0.f;
                    masked_block(lrow + T0 + 32 * p, lrow + T0 + 16 * p, r, 32 * p, row0, first, step2,
                                 NORM ? &rs : nullptr);
                }
                tc::fence_before_sync();
                switch (q4) {  // constant barrier ids
                    case 0: tc::named_arrive(1, 64); break;
                    case 1: tc::named_arrive(2, 64); break;
                    case 2: tc::named_arrive(3, 64); break;
                    default: tc::named_arrive(4, 64); break;
                }
            } else {
                uint32_t pk0[16], pk1[16];
                masked_pack(lrow + T0 + 64, r, 64, row0, r >= 64 ? gp[BP2 * (r - 64)] : 0.f, step2, pk0,
                            NORM ? &rs : nullptr);
                masked_pack(lrow + T0 + 96, r, 96, row0, r >= 96 ? gp[BP2 * (r - 96)] : 0.f, step2, pk1,
                            NORM ? &rs : nullptr);
                switch (q4) {
                    case 0: tc::named_bar(1, 64); break;
                    case 1: tc::named_bar(2, 64); break;
                    case 2: tc::named_bar(3, 64); break;
                    default: tc::named_bar(4, 64); break;
                }
                tc::fence_after_sync();
                tc::tmem_st16(lrow + T0 + 32, pk0);
                tc::tmem_st16(lrow + T0 + 48, pk1);
            }
            tc::tmem_wait_st();
            if (NORM) dpart[128 * h + r] = gp[2 * (r + 1)] * qy + rs;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BBT]);

            // ---- EPI-c: out = g^(2(r+1)) Q Z0 + B~ V;  Z <- g^(2Wc) Z + dZ ------------------------
            tc::mbar_wait(&bars[BC], ph, abort, status, 54);
            tc::fence_after_sync();
            float inv = 1.f;
            if (NORM) {  // every epilogue warp's partials of this chunk are written, and y0 read
                tc::named_bar(5, 256);
                inv = 1.f / ((dpart[r] + dpart[128 + r]) + a.eps);
            }
            {
                const float s2 = gp[BP2 * (r + 1)];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qz[16], bv[16];
                    tc::tmem_ld16(lrow + T2 + 32 * h + 16 * half, qz);
                    tc::tmem_ld16(lrow + T1 + 32 * h + 16 * half, bv);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {  // output tile (rows >= Wc fall outside the tensor)
                        float o[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            o[u] = s2 * __uint_as_float(qz[8 * j + u]) + __uint_as_float(bv[8 * j + u]);
                        *reinterpret_cast<uint4*>(sm + oO + tc::sw128_chunk(r, 4 * h + 2 * half + j)) = pack8(o, inv);
                    }
                }
                uint32_t dz[16];
                tc::tmem_ld16(lrow + T3 + zc, dz);
                tc::tmem_wait_ld();
                const float rho2 = gp[BP2 * Wc];  // (unmasked: C decays by g per token)
#pragma unroll
                for (int j = 0; j < 16; ++j) zz[j] = rho2 * zz[j] + __uint_as_float(dz[j]);
                publish_z();  // read by MMA-b of the next chunk, after its EPI-a arrives
                if (NORM) {  // y0 for the next chunk, then every warp sees it before its EPI-a
                    if (q4 == 0) {
                        const int cy = 32 * h + lane;
                        y0[cy] = rho2 * y0[cy] + (((ypart[cy] + ypart[64 + cy]) + ypart[128 + cy]) + ypart[192 + cy]);
                    }
                    tc::named_bar(6, 256);
                }
            }
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BOS]);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Summary pass that also stores the segment-local p (unnormalised; kSummaryP; UM = unmasked).
//
// Same sums as the summary mode above (S, C, Z of the segment from zero), and it writes
// p^sl_t = S^sl_t q_t (bf16) into the output buffer for the kOutputP pass.  The launch covers
// every segment (the last one for its p, and for the final combine when a final state is
// wanted).  Work taken off the chunk-to-chunk chain:
//   * the key-moment increment is formed as K^T D K = K^^T K^ with K^ = diag(g^((Wc-1-i)/2)) K,
//     so the raw K slot is free once A~ K has run and the next chunk's K loads early;
//   * P is staged in the raw Q slot (free after A~ K and Q S0) and written by one TMA tile
//     store; the next chunk's Q loads once that store has read the slot;
//   * the state products land in T2 | T3, so the next chunk's Q K^T (T0T1) is issued while this
//     chunk's state update still reads them.
// Per chunk (local row r):
//   MMA1  A = Q K^T -> T0T1              (issued during the previous chunk's EPI4)
//   EPI1  A~ = A * [i <= r] g^(r-i) -> T3;  then Q~ = diag(g^(Wc-1-r)) Q, K^ (smem)
//   MMA2  A~ K -> T2;  Q S0 -> T0
//   EPI2  P = g^(r+1) Q S0 + A~ K;  P~ = diag(g^(2(Wc-1-r))) P and P (smem);  P -> out (TMA)
//   ST    [Q~^T ; P~^T] V -> T2 (dC, dZ; unmasked: [Q~^T ; Q~^T] V, dC twice);
//         [K^^T ; K^^T] K^ -> T3 (dS twice)
//   EPI4  S <- g^Wc S + dS,  C <- g^Wc C + dC,  Z <- g^(2Wc) Z + dZ;  bf16 S0 (smem)
// MOM (masked; a final state or the normalised output) also forms the segment's query and p
// moments, m_B = sum_t g^(L-1-t) q_t and y_B = sum_t g^(2(L-1-t)) p^sl_t: per chunk the column
// sums of Q~ (EPI1) and P~ (EPI2), each reduced over a warp's 32 rows by shuffles into lane l's
// running sum of column 32h + l (decayed by g^Wc and g^(2Wc) like C and Z), and at the end
// summed over the four lane quarters in a fixed order.
namespace sump {

constexpr uint32_t oQ = 0, oK = kTile, oV = 2 * kTile, oQt = 3 * kTile, oKh = 4 * kTile, oPt = 5 * kTile;
constexpr uint32_t oS0 = 6 * kTile;   // S0, [64][64] bf16 (8 KB)
constexpr uint32_t oGP = oS0 + 8192;  // decay table g^0 .. g^(2W)
constexpr uint32_t oBar = oGP + 1088;
constexpr uint32_t oMisc = oBar + 16 * 8;
constexpr uint32_t oMom = oMisc + 16;  // MOM: m and y partials per lane quarter [2][4][64] fp32
constexpr uint32_t kSmemBytes = oMom + 2048 + 1024;
constexpr uint32_t T0 = 0, T2 = 128, T3 = 192;  // T0 .. T0+127: A = Q K^T (N = 128)

enum Bar { FQK = 0, FV, BA, BAT, BP, BPS, BST, kBarCount };

struct Maps {
    CUtensorMap q, k, v, p;  // p: the output buffer, where P is stored
};

}  // namespace sump

template <bool UM, bool MOM>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_sum_p_tc_kernel(const __grid_constant__ sump::Maps maps, const ChunkArgs a, int* status) {
    static_assert(!(UM && MOM), "the unmasked moments come from the moments kernel");
    pdl_trigger();
    // this pass's layout (shadows the first kernel's)
    constexpr uint32_t oQ = sump::oQ, oK = sump::oK, oV = sump::oV, oQt = sump::oQt, oKh = sump::oKh,
                       oPt = sump::oPt, oS0 = sump::oS0;
    constexpr uint32_t oGP = sump::oGP, oBar = sump::oBar, oMisc = sump::oMisc;
    constexpr uint32_t T0 = sump::T0, T2 = sump::T2, T3 = sump::T3;
    constexpr int FQK = sump::FQK, FV = sump::FV, BA = sump::BA, BAT = sump::BAT, BP = sump::BP, BPS = sump::BPS,
                  BST = sump::BST, kBarCount = sump::kBarCount;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gp = reinterpret_cast<float*>(sm + oGP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + oMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const float g = head_decay(a.gamma, bh, a.H);
    const float log2g = log2f(g);
    const int nit = c_end - c_begin;

    for (int i = tid; i < 2 * kW + 1; i += kThreads) gp[i] = pow_decay(log2g, (float)i);
    if (tid == 0) {
        for (int b = 0; b < kBarCount; ++b) tc::mbar_init(&bars[b], (b == BAT || b == BPS) ? 8 : 1);
        *abort = 0;
        tc::mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    pdl_wait();  // the status word and the workspace are written by the kernel before
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ control thread
        if (lane == 0 && nit > 0) {
            const uint32_t sQ = smem_u32(sm + oQ), sK = smem_u32(sm + oK), sV = smem_u32(sm + oV);
            const uint32_t sQt = smem_u32(sm + oQt), sKh = smem_u32(sm + oKh), sS0 = smem_u32(sm + oS0);
            auto load_qk = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FQK], 2 * kTile);
                tc::tma_load_3d(sm + oQ, &maps.q, 0, c * kW, bh, &bars[FQK]);
                tc::tma_load_3d(sm + oK, &maps.k, 0, c * kW, bh, &bars[FQK]);
            };
            // the next chunk's K at once, its Q once the P tile (staged in the Q slot) is read
            auto load_k_first = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FQK], 2 * kTile);
                tc::tma_load_3d(sm + oK, &maps.k, 0, c * kW, bh, &bars[FQK]);
            };
            auto load_q_second = [&](int c) { tc::tma_load_3d(sm + oQ, &maps.q, 0, c * kW, bh, &bars[FQK]); };
            auto load_v = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FV], kTile);
                tc::tma_load_3d(sm + oV, &maps.v, 0, c * kW, bh, &bars[FV]);
            };
            constexpr uint32_t I_AB = tc::idesc_bf16(128, 128, 0, 0);   // K-major x K-major, N = 128
            constexpr uint32_t I_QX = tc::idesc_bf16(128, 64, 0, 1);    // K-major x MN-major, N = 64
            constexpr uint32_t I_TS64 = tc::idesc_bf16(128, 64, 0, 1);  // A (TMEM) x MN-major B, N = 64
            constexpr uint32_t I_ST64 = tc::idesc_bf16(128, 64, 1, 1);  // MN-major x MN-major, N = 64
            auto mma1 = [&]() {  // A = Q K^T -> T0T1
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sK + 32 * ks, 16, 1024),
                               I_AB, ks > 0);
                tc::mma_commit(&bars[BA]);
            };
            load_qk(c_begin);
            load_v(c_begin);
            int lqk = 1, lv = 1;
            tc::mbar_wait(&bars[FQK], 0, abort, status, 61);
            tc::fence_after_sync();
            mma1();
            for (int it = 0; it < nit; ++it) {
                const uint32_t ph = it & 1;
                if (it + 1 < nit) {  // next chunk's tiles into L2, so that their loads below are short
                    const int cn = (c_begin + it + 1) * kW;
                    tc::tma_prefetch_3d(&maps.q, 0, cn, bh);
                    tc::tma_prefetch_3d(&maps.k, 0, cn, bh);
                    tc::tma_prefetch_3d(&maps.v, 0, cn, bh);
                }
                tc::mbar_wait(&bars[BAT], ph, abort, status, 62);  // A~, and the previous chunk's S0
                tc::fence_after_sync();
                // MMA2: A~ K -> T2;  Q S0 -> T0
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + T2, tmem + T3 + 8 * ks, tc::smem_desc(sK + 2048 * ks, 16, 1024), I_TS64, ks > 0);
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sS0 + 2048 * ks, 16, 1024),
                               I_QX, ks > 0);
                tc::mma_commit(&bars[BP]);
                tc::mbar_wait(&bars[BPS], ph, abort, status, 64);  // P (Q slot), P~, Q~, K^ written; T0, T2 read
                // P -> out (one tile store); raw K is free (MMA2 and EPI1's scaled copy are done)
                tc::tma_store_3d(&maps.p, sm + oQ, 0, (c_begin + it) * kW, bh);
                tc::bulk_commit();
                if (it + 1 < nit) {
                    load_k_first(c_begin + it + 1);
                    ++lqk;
                }
                tc::mbar_wait(&bars[FV], ph, abort, status, 65);
                tc::fence_after_sync();
                // ST: [Q~^T ; P~^T] V -> T2 (unmasked: [Q~^T ; Q~^T] V, dC twice);  [K^^T ; K^^T] K^ -> T3
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + T2, tc::smem_desc(sQt + 2048 * ks, UM ? 0 : oPt - oQt, 1024),
                               tc::smem_desc(sV + 2048 * ks, 16, 1024), I_ST64, ks > 0);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + T3, tc::smem_desc(sKh + 2048 * ks, 0, 1024),
                               tc::smem_desc(sKh + 2048 * ks, 16, 1024), I_ST64, ks > 0);
                tc::mma_commit(&bars[BST]);
                tc::bulk_wait_read_all();  // the P tile has left the Q slot
                if (it + 1 < nit) {
                    load_q_second(c_begin + it + 1);
                    // next chunk's Q K^T while this chunk's state update runs
                    tc::mbar_wait(&bars[FQK], ph ^ 1, abort, status, 66);
                    tc::fence_after_sync();
                    mma1();
                }
                tc::mbar_wait(&bars[BST], ph, abort, status, 67);  // V, Q~, K^ free
                if (it + 1 < nit) {
                    load_v(c_begin + it + 1);
                    ++lv;
                }
            }
            volatile int never = 0;
            tc::mbar_wait(&bars[BST], (nit - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FQK], (lqk - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FV], (lv - 1) & 1, &never, nullptr, 0);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q4 = warp & 3, h = (warp - 1) >> 2;
        const int r = 32 * q4 + lane;
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        unsigned char* sQ = sm + oQ;  // raw Q, then this chunk's P tile (after MMA2)
        unsigned char* sK = sm + oK;
        unsigned char* sQt = sm + oQt;
        unsigned char* sKh = sm + oKh;
        unsigned char* sPt = sm + oPt;
        const float ginv = g > 0.f ? 1.f / g : 0.f;
        // fp32 sums: C row r (r < 64) or Z row r - 64, columns 32h ..; S row r % 64, columns sc ..
        const int sc = 32 * h + 16 * (r >> 6);
        float st[32], ss[16];
#pragma unroll
        for (int j = 0; j < 32; ++j) st[j] = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) ss[j] = 0.f;
        auto publish_s = [&]() {
#pragma unroll
            for (int j = 0; j < 2; ++j)
                *reinterpret_cast<uint4*>(sm + oS0 + tc::sw128_chunk(r & 63, sc / 8 + j)) = pack8(&ss[8 * j], 1.f);
        };
        publish_s();
        tc::fence_proxy_async();
        float mw = 0.f, yw = 0.f;  // MOM: this warp's rows' moments of column 32h + lane

        for (int it = 0; it < nit; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            // ---- EPI1: A~ -> T3;  Q~, K^ -> smem ----------------------------------------------
            tc::mbar_wait(&bars[FQK], ph, abort, status, 71);
            tc::mbar_wait(&bars[BA], ph, abort, status, 72);
            tc::fence_after_sync();
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const int cb = 64 * h + 32 * p;
                const float first = r >= cb ? gp[r - cb] : 0.f;
                masked_block(lrow + T0 + cb, lrow + T3 + cb / 2, r, cb, row0, first, ginv);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BAT]);
            {  // first read by ST, after EPI2's fence
                const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
                const float wh = r < Wc ? pow_decay(log2g, 0.5f * (float)(Wc - 1 - r)) : 0.f;
                float cs[16];  // MOM: this row's w1 q over a 16-column half
                float dm = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                    const uint4 qc = *reinterpret_cast<const uint4*>(sQ + off);
                    *reinterpret_cast<uint4*>(sQt + off) = scale_chunk(qc, w1);
                    *reinterpret_cast<uint4*>(sKh + off) = scale_chunk(*reinterpret_cast<const uint4*>(sK + off), wh);
                    if (MOM) {
                        const uint32_t qw[4] = {qc.x, qc.y, qc.z, qc.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            cs[8 * (j & 1) + 2 * u] = w1 * bf_lo(qw[u]);
                            cs[8 * (j & 1) + 2 * u + 1] = w1 * bf_hi(qw[u]);
                        }
                        if (j & 1) {
                            const float t = warp_colsum16(cs, lane);
                            if ((lane >> 4) == (j >> 1)) dm = t;  // lane l keeps column 32h + l
                        }
                    }
                }
                if (MOM) mw = gp[Wc] * mw + dm;
            }
            // ---- EPI2: P = g^(r+1) Q S0 + A~ K;  P~ -> smem, P -> out ---------------------------
            tc::mbar_wait(&bars[BP], ph, abort, status, 73);
            tc::fence_after_sync();
            {
                const float s1 = gp[r + 1];
                const float w2 = r < Wc ? gp[2 * (Wc - 1 - r)] : 0.f;
                float dy = 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qs[16], ak[16];
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, qs);
                    tc::tmem_ld16(lrow + T2 + 32 * h + 16 * half, ak);
                    tc::tmem_wait_ld();
                    float pv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) pv[j] = s1 * __uint_as_float(qs[j]) + __uint_as_float(ak[j]);
                    if (MOM) {  // P~ column sums (P as stored: rounded to bf16 first, as the output pass reads it)
                        float cs[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) cs[j] = w2 * __bfloat162float(__float2bfloat16(pv[j]));
                        const float t = warp_colsum16(cs, lane);
                        if ((lane >> 4) == half) dy = t;
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t off = tc::sw128_chunk(r, 4 * h + 2 * half + j);
                        if (!UM) *reinterpret_cast<uint4*>(sPt + off) = pack8(&pv[8 * j], w2);
                        *reinterpret_cast<uint4*>(sQ + off) = pack8(&pv[8 * j], 1.f);  // rows >= Wc: not stored
                    }
                }
                if (MOM) yw = gp[2 * Wc] * yw + dy;
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BPS]);
            // ---- EPI4: state update --------------------------------------------------------------
            tc::mbar_wait(&bars[BST], ph, abort, status, 74);
            tc::fence_after_sync();
            {
                const float rho = gp[Wc], rho2 = gp[2 * Wc];
                uint32_t v[32], w[16];
                tc::tmem_ld32(lrow + T2 + 32 * h, v);
                tc::tmem_ld16(lrow + T3 + sc, w);
                tc::tmem_wait_ld();
                const float decay = r < 64 || UM ? rho : rho2;  // unmasked: rows >= 64 hold C again
#pragma unroll
                for (int j = 0; j < 32; ++j) st[j] = decay * st[j] + __uint_as_float(v[j]);
#pragma unroll
                for (int j = 0; j < 16; ++j) ss[j] = rho * ss[j] + __uint_as_float(w[j]);
                publish_s();  // read by the next chunk's MMA2, after its EPI1 arrives
            }
            tc::fence_proxy_async();
        }

        if (seg < a.nsum) {  // (the launch also covers the last segment, for its p)
            const size_t si = (size_t)bh * a.nsum + seg;
            float* dst = r < 64 ? a.ws + a.L.CB + si * kD * kD + (size_t)r * kD
                                : a.ws + a.L.ZB + si * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[32 * h + j] = st[j];
            float* ds = a.ws + a.L.SB + si * kD * kD + (size_t)(r & 63) * kD + sc;
#pragma unroll
            for (int j = 0; j < 16; ++j) ds[j] = ss[j];
            if (MOM) {  // the four lane quarters' moments, added in a fixed order
                float* mom = reinterpret_cast<float*>(sm + sump::oMom);
                mom[64 * q4 + 32 * h + lane] = mw;
                mom[256 + 64 * q4 + 32 * h + lane] = yw;
                tc::named_bar(5, 256);
                if (q4 == 0) {
                    const int c = 32 * h + lane;
                    a.ws[a.L.mB + si * kD + c] = ((mom[c] + mom[64 + c]) + mom[128 + c]) + mom[192 + c];
                    a.ws[a.L.yB + si * kD + c] = ((mom[256 + c] + mom[320 + c]) + mom[384 + c]) + mom[448 + c];
                }
            } else if (h == 0 && r < 64) {
                a.ws[a.L.mB + si * kD + r] = 0.f;
                a.ws[a.L.yB + si * kD + r] = 0.f;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [BH][n][64] bf16, box [1][128][64], 128-byte swizzle; rows past n read as zero.
bool make_map(CUtensorMap* m, const void* ptr, int BH, int n) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)n, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)n * kD * 2};
    cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kW, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fwd_chunk_tc_available() { return encode_fn() != nullptr; }

size_t fwd_chunk_tc_smem() { return kSmemBytes; }

int launch_fwd_chunk_tc(const ChunkArgs& a, int mode, int* status, cudaStream_t st) {
    if (a.nseg_launch <= 0 || a.BH <= 0) return 0;
    if (mode == kOutputP) {
        outp::Maps pm;
        if (!make_map(&pm.q, a.q, a.BH, a.n) || !make_map(&pm.p, a.out, a.BH, a.n) || !make_map(&pm.v, a.v, a.BH, a.n))
            return -2;
        auto kfn = a.unmasked ? fwd_out_p_tc_kernel<true, false>
                              : (a.normalize ? fwd_out_p_tc_kernel<false, true> : fwd_out_p_tc_kernel<false, false>);
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, outp::kSmemBytes);
        if (e != cudaSuccess) return -1;
        if (launch_pdl(kfn, dim3(a.nseg_launch, a.BH), dim3(kThreads), outp::kSmemBytes, st, pm, a, status) !=
            cudaSuccess)
            return -1;
        return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
    }
    TcMaps maps;
    if (!make_map(&maps.q, a.q, a.BH, a.n) || !make_map(&maps.k, a.k, a.BH, a.n) || !make_map(&maps.v, a.v, a.BH, a.n))
        return -2;
    if (mode == kSummaryP) {
        sump::Maps sm4;
        sm4.q = maps.q;
        sm4.k = maps.k;
        sm4.v = maps.v;
        if (!make_map(&sm4.p, a.out, a.BH, a.n)) return -2;
        // masked with a final state or normalised: the segment moments come from this pass
        auto kfn = a.unmasked ? fwd_sum_p_tc_kernel<true, false>
                              : (a.want_final || a.normalize ? fwd_sum_p_tc_kernel<false, true>
                                                             : fwd_sum_p_tc_kernel<false, false>);
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, sump::kSmemBytes);
        if (e != cudaSuccess) return -1;
        if (launch_pdl(kfn, dim3(a.nseg_launch, a.BH), dim3(kThreads), sump::kSmemBytes, st, sm4, a, status) !=
            cudaSuccess)
            return -1;
        return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
    }
    dim3 grid(a.nseg_launch, a.BH);
    auto kfn = mode == kSummary ? (a.unmasked ? fwd_chunk_tc_kernel<kSummary, true> : fwd_chunk_tc_kernel<kSummary, false>)
                                : (a.unmasked ? fwd_chunk_tc_kernel<kOutput, true> : fwd_chunk_tc_kernel<kOutput, false>);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) kfn<<<grid, kThreads, kSmemBytes, st>>>(maps, a, status);
    if (e != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2
