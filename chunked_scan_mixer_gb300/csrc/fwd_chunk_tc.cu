// tcgen05 chunk kernel of the masked HLA-2 forward for d = dv = 64 and chunk width 128
// (bf16 inputs, fp32 state, unnormalised).  Same per-chunk algebra as the mma.sync kernel
// (fwd_chunk_mma.cuh: p_t = S_t q_t, Z_t = g^2 Z_{t-1} + p_t v_t^T, o_t = q_t^T Z_t), with
// the chunk products on the 5th-generation tensor cores:
//
//   MMA1  A   = Q K^T                                  -> TMEM R1 (128 x 128 fp32)
//   EPI1  A~  = A * [i <= r] g^(r-i)  (bf16, in place in R1, the A operand of MMA2)
//         Qh  = diag(g^(r+1)) Q,  Qh2 = diag(g^(2(r+1))) Q   (bf16, in R1 next to A~)
//         K~  = diag(g^(Wc-1-i)) K                     (bf16, shared memory)
//   MMA2  P   = [A~ | Qh] [K ; S0]                     -> R2 (128 x 64)
//         O   = Qh2 Z0                                 -> R3 (128 x 64)
//   EPI2  P (bf16, K-major), P~ = diag(g^(2(Wc-1-j))) P (bf16)          (shared memory)
//   MMA3  B   = Q P^T                                  -> R1
//   EPI3  B~  = B * [j <= r] g^(2(r-j))                (bf16, in place in R1)
//   MMA4  O  += B~ V                                   -> R3
//         ST  = [K~^T ; P~^T] [K | V]: dS = K~^T K, dZ = P~^T V   -> R1
//   EPI4  out = O (bf16, global);  S <- g^Wc S + dS,  Z <- g^(2Wc) Z + dZ  (fp32 registers),
//         S0, Z0 = bf16(S), bf16(Z) for the next chunk (shared memory)
//
// Summary mode (segment summaries for the inter-segment scan) keeps EPI1/MMA2/EPI2 and then
// computes ST = [Q~^T ; K~^T] [K | V] (dC = Q~^T V, dS = K~^T K, Q~ = diag(g^(Wc-1-j)) Q) and
// dZ = P~^T V as an M = 64 MMA, accumulating S, C, Z from zero.
//
// Roles: warp 0 allocates tensor memory and one of its threads issues the TMA loads and every
// MMA; warps 1..8 move data between tensor memory, registers and shared memory (warp w reads
// TMEM lanes 32*(w%4)..+31, i.e. token/feature rows, and half (w-1)/4 of the columns).  Two
// CTAs share an SM (256 TMEM columns, ~99 KB of shared memory each).  Every wait is bounded;
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
constexpr uint32_t oGP = 6 * kTile;  // decay table g^0 .. g^(2W), 257 floats
constexpr uint32_t oBar = oGP + 1088;
constexpr int kNumBars = 11;
constexpr uint32_t oMisc = oBar + kNumBars * 8;  // tmem base, abort flag
constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;  // + alignment slack
// TMEM columns
constexpr uint32_t R1 = 0, R2 = 128, R3 = 192, kTmemCols = 256;

enum Bar { FULL = 0, BA, BAT, BP, BPS, BB, BBT, BO, BST, BS, kBarCount };

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

template <int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_chunk_tc_kernel(const __grid_constant__ TcMaps maps, const ChunkArgs a, int* status) {
    constexpr bool SUMMARY = MODE == kSummary;
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
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));

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
            const uint32_t sS0 = sPt, sZ0 = sPt + 8192;
            auto load = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FULL], 3 * kTile);
                tc::tma_load_3d(sm + oQ, &maps.q, 0, c * kW, bh, &bars[FULL]);
                tc::tma_load_3d(sm + oK, &maps.k, 0, c * kW, bh, &bars[FULL]);
                tc::tma_load_3d(sm + oV, &maps.v, 0, c * kW, bh, &bars[FULL]);
            };
            constexpr uint32_t I_AB = tc::idesc_bf16(128, 128, 0, 0);   // K-major x K-major, N = 128
            constexpr uint32_t I_TS64 = tc::idesc_bf16(128, 64, 0, 1);  // A (TMEM) x MN-major B, N = 64
            constexpr uint32_t I_ST = tc::idesc_bf16(128, 128, 1, 1);   // MN-major x MN-major, N = 128
            constexpr uint32_t I_Z64 = tc::idesc_bf16(64, 64, 1, 1);    // M = 64, MN-major x MN-major
            load(c_begin);
            for (int it = 0; it < nit; ++it) {
                const uint32_t ph = it & 1;
                tc::mbar_wait(&bars[FULL], ph, abort, status, 1);
                if (it > 0) tc::mbar_wait(&bars[BS], ph ^ 1, abort, status, 2);
                tc::fence_after_sync();
                // MMA1: A = Q K^T
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + R1, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sK + 32 * ks, 16, 1024),
                               I_AB, ks > 0);
                tc::mma_commit(&bars[BA]);
                tc::mbar_wait(&bars[BAT], ph, abort, status, 3);
                tc::fence_after_sync();
                // MMA2: P = [A~ | Qh] [K ; S0];  O = Qh2 Z0
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + R2, tmem + R1 + 8 * ks, tc::smem_desc(sK + 2048 * ks, 16, 1024), I_TS64, ks > 0);
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ts(tmem + R2, tmem + R1 + 64 + 8 * ks, tc::smem_desc(sS0 + 2048 * ks, 16, 1024), I_TS64, 1);
                if (!SUMMARY)
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ts(tmem + R3, tmem + R1 + 96 + 8 * ks, tc::smem_desc(sZ0 + 2048 * ks, 16, 1024), I_TS64,
                                   ks > 0);
                tc::mma_commit(&bars[BP]);
                tc::mbar_wait(&bars[BPS], ph, abort, status, 4);
                tc::fence_after_sync();
                if (!SUMMARY) {
                    // MMA3: B = Q P^T
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + R1, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sP + 32 * ks, 16, 1024),
                                   I_AB, ks > 0);
                    tc::mma_commit(&bars[BB]);
                    tc::mbar_wait(&bars[BBT], ph, abort, status, 5);
                    tc::fence_after_sync();
                    // MMA4: O += B~ V, then ST (after O has read B~ out of R1)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + R3, tmem + R1 + 8 * ks, tc::smem_desc(sV + 2048 * ks, 16, 1024), I_TS64, 1);
                    tc::mma_commit(&bars[BO]);
                    tc::mbar_wait(&bars[BO], ph, abort, status, 6);
                    tc::fence_after_sync();
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + R1, tc::smem_desc(sKt + 2048 * ks, kTile, 1024),
                                   tc::smem_desc(sK + 2048 * ks, kTile, 1024), I_ST, ks > 0);
                } else {
                    // ST = [Q~^T ; K~^T] [K | V] (Q~ in the P slot);  dZ = P~^T V (M = 64)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + R1, tc::smem_desc(sP + 2048 * ks, kTile, 1024),
                                   tc::smem_desc(sK + 2048 * ks, kTile, 1024), I_ST, ks > 0);
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + R3, tc::smem_desc(sPt + 2048 * ks, 16, 1024),
                                   tc::smem_desc(sV + 2048 * ks, 16, 1024), I_Z64, ks > 0);
                }
                tc::mma_commit(&bars[BST]);
                tc::mbar_wait(&bars[BST], ph, abort, status, 7);  // Q, K, V free
                if (it + 1 < nit) load(c_begin + it + 1);
            }
            // drain (bounded, ignoring the abort flag) so nothing is in flight at exit
            volatile int never = 0;
            tc::mbar_wait(&bars[BST], (nit - 1) & 1, &never, nullptr, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q4 = warp & 3, h = (warp - 1) >> 2;
        const int r = 32 * q4 + lane;                       // TMEM lane = row
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        unsigned char* sQ = sm + oQ;
        unsigned char* sK = sm + oK;
        unsigned char* sP = sm + oP;
        unsigned char* sKt = sm + oKt;
        unsigned char* sPt = sm + oPt;
        // state rows owned by this thread (32 columns each)
        float st[32];   // output: S (r < 64) or Z (r >= 64); summary: C (r < 64) or S (r >= 64)
        float stz[32];  // summary only: Z row m = 16*q4 + lane for lane < 16
        const size_t sidx = (size_t)bh * a.nseg + seg;
        if (!SUMMARY) {
            const float* src = r < 64 ? a.ws + a.L.Sin + sidx * kD * kD + (size_t)r * kD
                                      : a.ws + a.L.Zin + sidx * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j] = src[32 * h + j];
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j] = stz[j] = 0.f;
        }
        // bf16 copies of the initial S (and Z) for MMA2 of the first chunk
        auto publish_state = [&]() {
            const bool s_row = SUMMARY ? r >= 64 : r < 64;
            if (SUMMARY && !s_row) return;
            const int row = r < 64 ? r : r - 64;
            unsigned char* base = sPt + (s_row ? 0 : 8192);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 o;
                o.x = pack_bf16x2(st[8 * j + 0], st[8 * j + 1]);
                o.y = pack_bf16x2(st[8 * j + 2], st[8 * j + 3]);
                o.z = pack_bf16x2(st[8 * j + 4], st[8 * j + 5]);
                o.w = pack_bf16x2(st[8 * j + 6], st[8 * j + 7]);
                *reinterpret_cast<uint4*>(base + tc::sw128_chunk(row, 4 * h + j)) = o;
            }
        };
        publish_state();
        tc::fence_proxy_async();

        for (int it = 0; it < nit; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            // ---- EPI1 -------------------------------------------------------------------
            tc::mbar_wait(&bars[FULL], ph, abort, status, 11);
            tc::mbar_wait(&bars[BA], ph, abort, status, 12);
            tc::fence_after_sync();
            {
                uint32_t pk[32];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t v[32];
                    tc::tmem_ld32(tmem + lane_off + R1 + 64 * h + 32 * p, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int i = 64 * h + 32 * p + j;
                        const float a0 = i <= r ? gp[r - i] * __uint_as_float(v[j]) : 0.f;
                        const float a1 = i + 1 <= r ? gp[r - i - 1] * __uint_as_float(v[j + 1]) : 0.f;
                        pk[16 * p + j / 2] = pack_bf16x2(a0, a1);
                    }
                }
                tc::named_bar(1, 256);  // every read of A is done before R1 is overwritten
                uint32_t lo[16], hi[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    lo[j] = pk[j];
                    hi[j] = pk[16 + j];
                }
                tc::tmem_st16(tmem + lane_off + R1 + 32 * h, lo);
                tc::tmem_st16(tmem + lane_off + R1 + 32 * h + 16, hi);
            }
            {
                // Qh (h = 0) / Qh2 (h = 1, output only) rows into R1 columns 64 + 32 h
                if (h == 0 || !SUMMARY) {
                    const float s = h == 0 ? gp[r + 1] : gp[2 * (r + 1)];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t qh[16];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 cq = scale_chunk(*reinterpret_cast<const uint4*>(sQ + tc::sw128_chunk(r, 4 * half + j)), s);
                            qh[4 * j + 0] = cq.x;
                            qh[4 * j + 1] = cq.y;
                            qh[4 * j + 2] = cq.z;
                            qh[4 * j + 3] = cq.w;
                        }
                        tc::tmem_st16(tmem + lane_off + R1 + 64 + 32 * h + 16 * half, qh);
                    }
                }
                // K~ (and Q~ in summary mode) rows: features 32h .. 32h+31
                const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                    *reinterpret_cast<uint4*>(sKt + off) = scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w1);
                    if (SUMMARY)
                        *reinterpret_cast<uint4*>(sP + off) = scale_chunk(*reinterpret_cast<const uint4*>(sQ + off), w1);
                }
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BAT]);

            // ---- EPI2: P, P~ -------------------------------------------------------------
            tc::mbar_wait(&bars[BP], ph, abort, status, 13);
            tc::fence_after_sync();
            {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + R2 + 32 * h, v);
                tc::tmem_wait_ld();
                const float w2 = r < Wc ? gp[2 * (Wc - 1 - r)] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                    const float* f = reinterpret_cast<const float*>(&v[8 * j]);
                    if (!SUMMARY) {
                        uint4 o;
                        o.x = pack_bf16x2(f[0], f[1]);
                        o.y = pack_bf16x2(f[2], f[3]);
                        o.z = pack_bf16x2(f[4], f[5]);
                        o.w = pack_bf16x2(f[6], f[7]);
                        *reinterpret_cast<uint4*>(sP + off) = o;
                    }
                    uint4 t;
                    t.x = pack_bf16x2(w2 * f[0], w2 * f[1]);
                    t.y = pack_bf16x2(w2 * f[2], w2 * f[3]);
                    t.z = pack_bf16x2(w2 * f[4], w2 * f[5]);
                    t.w = pack_bf16x2(w2 * f[6], w2 * f[7]);
                    *reinterpret_cast<uint4*>(sPt + off) = t;
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BPS]);

            if (!SUMMARY) {
                // ---- EPI3: B~ in place ---------------------------------------------------------
                tc::mbar_wait(&bars[BB], ph, abort, status, 14);
                tc::fence_after_sync();
                uint32_t pk[32];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t v[32];
                    tc::tmem_ld32(tmem + lane_off + R1 + 64 * h + 32 * p, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int i = 64 * h + 32 * p + j;
                        const float b0 = i <= r ? gp[2 * (r - i)] * __uint_as_float(v[j]) : 0.f;
                        const float b1 = i + 1 <= r ? gp[2 * (r - i - 1)] * __uint_as_float(v[j + 1]) : 0.f;
                        pk[16 * p + j / 2] = pack_bf16x2(b0, b1);
                    }
                }
                tc::named_bar(1, 256);
                uint32_t lo[16], hi[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    lo[j] = pk[j];
                    hi[j] = pk[16 + j];
                }
                tc::tmem_st16(tmem + lane_off + R1 + 32 * h, lo);
                tc::tmem_st16(tmem + lane_off + R1 + 32 * h + 16, hi);
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[BBT]);

                // ---- EPI4a: output rows --------------------------------------------------------
                tc::mbar_wait(&bars[BO], ph, abort, status, 15);
                tc::fence_after_sync();
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + R3 + 32 * h, v);
                tc::tmem_wait_ld();
                if (r < Wc) {
                    bf16* out = static_cast<bf16*>(a.out) + ((size_t)bh * a.n + (size_t)c * kW + r) * kD + 32 * h;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float* f = reinterpret_cast<const float*>(&v[8 * j]);
                        uint4 o;
                        o.x = pack_bf16x2(f[0], f[1]);
                        o.y = pack_bf16x2(f[2], f[3]);
                        o.z = pack_bf16x2(f[4], f[5]);
                        o.w = pack_bf16x2(f[6], f[7]);
                        *reinterpret_cast<uint4*>(out + 8 * j) = o;
                    }
                }
            }

            // ---- EPI4b: state update -----------------------------------------------------------
            tc::mbar_wait(&bars[BST], ph, abort, status, 16);
            tc::fence_after_sync();
            {
                const float rho = gp[Wc], rho2 = gp[2 * Wc];
                uint32_t v[32];
                // output: rows < 64 hold dS (cols 0..63), rows >= 64 dZ (cols 64..127)
                // summary: rows < 64 hold dC (cols 64..127), rows >= 64 dS (cols 0..63)
                const uint32_t col = (SUMMARY ? (r < 64 ? 64 : 0) : (r < 64 ? 0 : 64)) + 32 * h;
                tc::tmem_ld32(tmem + lane_off + R1 + col, v);
                tc::tmem_wait_ld();
                const float decay = SUMMARY ? rho : (r < 64 ? rho : rho2);
#pragma unroll
                for (int j = 0; j < 32; ++j) st[j] = decay * st[j] + __uint_as_float(v[j]);
                if (SUMMARY) {
                    tc::tmem_ld32(tmem + lane_off + R3 + 32 * h, v);  // dZ, M = 64 layout
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) stz[j] = rho2 * stz[j] + __uint_as_float(v[j]);
                }
                publish_state();
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BS]);
        }

        if (SUMMARY) {
            const size_t si = (size_t)bh * a.nsum + seg;
            float* dst = r < 64 ? a.ws + a.L.CB + si * kD * kD + (size_t)r * kD
                                : a.ws + a.L.SB + si * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[32 * h + j] = st[j];
            if (lane < 16) {
                float* dz = a.ws + a.L.ZB + si * kD * kD + (size_t)(16 * q4 + lane) * kD;
#pragma unroll
                for (int j = 0; j < 32; ++j) dz[32 * h + j] = stz[j];
            }
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
    TcMaps maps;
    if (!make_map(&maps.q, a.q, a.BH, a.n) || !make_map(&maps.k, a.k, a.BH, a.n) || !make_map(&maps.v, a.v, a.BH, a.n))
        return -2;
    dim3 grid(a.nseg_launch, a.BH);
    cudaError_t e;
    if (mode == kSummary) {
        e = cudaFuncSetAttribute(fwd_chunk_tc_kernel<kSummary>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e == cudaSuccess) fwd_chunk_tc_kernel<kSummary><<<grid, kThreads, kSmemBytes, st>>>(maps, a, status);
    } else {
        e = cudaFuncSetAttribute(fwd_chunk_tc_kernel<kOutput>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e == cudaSuccess) fwd_chunk_tc_kernel<kOutput><<<grid, kThreads, kSmemBytes, st>>>(maps, a, status);
    }
    if (e != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2
