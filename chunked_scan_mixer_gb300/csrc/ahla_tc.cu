// tcgen05 chunk kernel of the AHLA forward for d = dv = 64 and chunk width 128 (bf16
// inputs, fp32 state, unnormalised).  Same per-chunk algebra as the mma.sync kernel
// (ahla.cu: Inner = g^(r+1) Q P0 + A~ V, O = g^(r+1) Q E0 + A~ Inner with one masked matrix
// A~[r, j] = [j <= r] g^(r-j) (q_r . k_j)), with the chunk products on the 5th-generation
// tensor cores.  A~ is written once to tensor memory and is the A operand of both cascaded
// products.  Tensor memory holds four 64-column regions T0 | T1 | T3 | T2 (T1T3 and T3T2
// contiguous):
//
//   MMA1  A     = Q K^T                                -> T0T1 (128 x 128 fp32)
//   EPI1  A~    = A * [j <= r] g^(r-j)  (bf16, packed) -> T3;  K~ = diag(g^(Wc-1-i)) K (smem)
//   MMA2  A~ V  -> T2;  Q P0 -> T0
//   EPI2  Inner = g^(r+1) Q P0 + A~ V  (bf16, smem)
//   MMA3  A~ Inner -> T0;  Q E0 -> T1;   then ST = [K~^T ; K~^T] [V | Inner] -> T3T2
//   EPI3  out = g^(r+1) Q E0 + A~ Inner  (bf16, global)
//   EPI4  P <- g^Wc P + dP (rows < 64 of ST, T3),  E <- g^Wc E + dE (rows >= 64, T2);
//         bf16 P0, E0 (smem)
//
// Summary mode keeps MMA1, EPI1, MMA2, EPI2, then computes ST and R = [K^T ; K^T] Q -> T0
// (undecayed), accumulating P, E, R from zero.
//
// FO (first-order mode) serves the third-order output's inner pass, masked first-order linear
// attention u = Inner: the output pass writes Inner itself (one TMA tile store a chunk from the
// Inner slot) and skips MMA3 and EPI3, and the
// summary pass skips MMA1 to EPI2 and the R product, keeping only the scaled keys and the
// state product, whose P half is the segment's P (the E and R summaries are then unused).
//
// Roles as in the symmetric kernel (fwd_chunk_tc.cu): warp 0 allocates tensor memory and one
// of its threads issues the TMA loads and every MMA; warps 1..8 move data between tensor
// memory, registers and shared memory.  Two CTAs share an SM.  Every wait is bounded; on a
// timeout the kernel records where in the workspace status word, drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tc_common.cuh"

namespace hla2 {

namespace {

constexpr int kW = 128, kD = 64;
constexpr int kThreads = 288;          // 1 control warp + 8 epilogue warps
constexpr uint32_t kTile = 128 * 128;  // bytes of one [128][64] bf16 SW128 tile
// shared memory slots (byte offsets from the 1024-aligned base); Inner follows V so that
// [V | Inner] is one MN-major operand
constexpr uint32_t oQ = 0, oK = kTile, oV = 2 * kTile, oIn = 3 * kTile, oKt = 4 * kTile;
constexpr uint32_t oP0 = 5 * kTile, oE0 = oP0 + 8192;  // [64][64] bf16 each
constexpr uint32_t oGP = oE0 + 8192;                   // decay table g^0 .. g^(2W)
constexpr uint32_t oBar = oGP + 1088;
constexpr uint32_t oMisc = oBar + 16 * 8;
constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
constexpr uint32_t T0 = 0, T1 = 64, T3 = 128, T2 = 192, kTmemCols = 256;

enum Bar { FULLQ = 0, FULLKV, BA, BAT, BP, BPS, BO, BST, BS, kBarCount };

struct TcMaps {
    CUtensorMap q, k, v, o;  // o: the output buffer (stored Inner, summary pass with store_inner)
};

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

__device__ __forceinline__ uint4 scale_chunk(uint4 c, float s) {
    uint4 o;
    o.x = pack_bf16x2(s * bf_lo(c.x), s * bf_hi(c.x));
    o.y = pack_bf16x2(s * bf_lo(c.y), s * bf_hi(c.y));
    o.z = pack_bf16x2(s * bf_lo(c.z), s * bf_hi(c.z));
    o.w = pack_bf16x2(s * bf_lo(c.w), s * bf_hi(c.w));
    return o;
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 o;
    o.x = pack_bf16x2(f[0], f[1]);
    o.y = pack_bf16x2(f[2], f[3]);
    o.z = pack_bf16x2(f[4], f[5]);
    o.w = pack_bf16x2(f[6], f[7]);
    return o;
}

// Masked, decayed 32-column block of A for row r: out[j] = [j <= r] g^(r - j) in[j],
// j = cb .. cb + 31, read from src (TMEM fp32), written packed (16 columns) to dst.
__device__ __forceinline__ void masked_block(uint32_t src, uint32_t dst, int r, int cb, int warp_row0,
                                             float first, float step_up) {
    uint32_t pk[16];
    if (cb > warp_row0 + 31) {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
    } else {
        uint32_t v[32];
        tc::tmem_ld32(src, v);
        tc::tmem_wait_ld();
        float f = first;
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
            pk[j / 2] = pack_bf16x2(a0, a1);
        }
    }
    tc::tmem_st16(dst, pk);
}

template <bool SUMMARY, bool FO>
__global__ void __launch_bounds__(kThreads, 2)
    ahla_tc_kernel(const __grid_constant__ TcMaps maps, const AhlaArgs a, int* status) {
    constexpr bool CHAIN = !(FO && SUMMARY);  // A~ and Inner are formed
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
            const bool from_epilogue = (b == BAT || b == BPS || b == BS);
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
            const uint32_t sIn = smem_u32(sm + oIn), sKt = smem_u32(sm + oKt);
            const uint32_t sP0 = smem_u32(sm + oP0), sE0 = smem_u32(sm + oE0);
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
                tc::mbar_wait(&bars[FULLQ], ph, abort, status, 31);
                tc::mbar_wait(&bars[FULLKV], ph, abort, status, 32);
                if (it > 0) tc::mbar_wait(&bars[BS], ph ^ 1, abort, status, 33);
                tc::fence_after_sync();
                if (CHAIN) {
                    // MMA1: A = Q K^T -> T0T1
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024),
                                   tc::smem_desc(sK + 32 * ks, 16, 1024), I_AB, ks > 0);
                    tc::mma_commit(&bars[BA]);
                    tc::mbar_wait(&bars[BAT], ph, abort, status, 34);
                    // the previous chunk's Inner tile store has read the slot before this chunk's
                    // EPI2 (which follows MMA2) rewrites it
                    if ((SUMMARY && !FO && a.store_inner) || (FO && !SUMMARY)) tc::bulk_wait_read_all();
                    tc::fence_after_sync();
                    // MMA2: A~ V -> T2;  Q P0 -> T0
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + T2, tmem + T3 + 8 * ks, tc::smem_desc(sV + 2048 * ks, 16, 1024), I_TS64,
                                   ks > 0);
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024),
                                   tc::smem_desc(sP0 + 2048 * ks, 16, 1024), I_QX, ks > 0);
                    tc::mma_commit(&bars[BP]);
                }
                tc::mbar_wait(&bars[BPS], ph, abort, status, 35);  // Inner and K~ written
                tc::fence_after_sync();
                if ((SUMMARY && !FO && a.store_inner) || (FO && !SUMMARY)) {
                    // segment-local Inner (first-order mode: the pass's output) -> out, one tile store
                    tc::tma_store_3d(&maps.o, sm + oIn, 0, (c_begin + it) * kW, bh);
                    tc::bulk_commit();
                }
                if (FO) {
                    if (it + 1 < nit) load_q(c_begin + it + 1);  // Q is no longer read
                    // [K~^T ; K~^T] [V | Inner] -> T3T2 (dP; dE is not used)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T3, tc::smem_desc(sKt + 2048 * ks, 0, 1024),
                                   tc::smem_desc(sV + 2048 * ks, oIn - oV, 1024), I_ST, ks > 0);
                } else if (!SUMMARY) {
                    // MMA3: A~ Inner -> T0;  Q E0 -> T1
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + T0, tmem + T3 + 8 * ks, tc::smem_desc(sIn + 2048 * ks, 16, 1024), I_TS64,
                                   ks > 0);
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + T1, tc::smem_desc(sQ + 32 * ks, 16, 1024),
                                   tc::smem_desc(sE0 + 2048 * ks, 16, 1024), I_QX, ks > 0);
                    tc::mma_commit(&bars[BO]);
                    tc::mbar_wait(&bars[BO], ph, abort, status, 36);  // A~ (T3) read; Q no longer read
                    tc::fence_after_sync();
                    if (it + 1 < nit) load_q(c_begin + it + 1);
                    // [K~^T ; K~^T] [V | Inner] -> T3T2 (dP, dE)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T3, tc::smem_desc(sKt + 2048 * ks, 0, 1024),
                                   tc::smem_desc(sV + 2048 * ks, oIn - oV, 1024), I_ST, ks > 0);
                } else {
                    // [K~^T ; K~^T] [V | Inner] -> T3T2 (dP, dE);  [K^T ; K^T] Q -> T0 (dR, undecayed)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T3, tc::smem_desc(sKt + 2048 * ks, 0, 1024),
                                   tc::smem_desc(sV + 2048 * ks, oIn - oV, 1024), I_ST, ks > 0);
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + T0, tc::smem_desc(sK + 2048 * ks, 0, 1024),
                                   tc::smem_desc(sQ + 2048 * ks, 16, 1024), I_ST64, ks > 0);
                }
                tc::mma_commit(&bars[BST]);
                tc::mbar_wait(&bars[BST], ph, abort, status, 37);  // K, V (and Q) free
                if (SUMMARY && !FO && it + 1 < nit) load_q(c_begin + it + 1);
                if (it + 1 < nit) {
                    load_kv(c_begin + it + 1);
                    ++loads;
                }
            }
            volatile int never = 0;
            tc::mbar_wait(&bars[BST], (nit - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FULLKV], (loads - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FULLQ], (loads - 1) & 1, &never, nullptr, 0);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int q4 = warp & 3, h = (warp - 1) >> 2;
        const int r = 32 * q4 + lane;  // TMEM lane = row
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        unsigned char* sK = sm + oK;
        unsigned char* sIn = sm + oIn;
        unsigned char* sKt = sm + oKt;
        unsigned char* sP0 = sm + oP0;
        unsigned char* sE0 = sm + oE0;
        const float ginv = g > 0.f ? 1.f / g : 0.f;
        // fp32 state: P row r (r < 64) or E row r - 64, columns 32h..32h+31; in summary mode
        // also R row r % 64, columns 32h + 16 (r / 64) .. +15
        float st[32];
        float rr[16];
        const size_t cidx = (size_t)bh * a.nseg + seg;
        if (!SUMMARY) {
            const float* src = r < 64 ? a.ws + a.L.Pin + cidx * kD * kD + (size_t)r * kD
                                      : a.ws + a.L.Ein + cidx * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j] = src[32 * h + j];
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) st[j] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) rr[j] = 0.f;
        }
        // bf16 copies of P (P0 slot) and E (E0 slot): the B operands of Q P0 and Q E0
        auto publish_state = [&]() {
            unsigned char* base = r < 64 ? sP0 : sE0;
            if (SUMMARY && r >= 64) return;  // summaries read P0 only
            const int row = r & 63;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(base + tc::sw128_chunk(row, 4 * h + j)) = pack8(&st[8 * j]);
        };
        publish_state();
        tc::fence_proxy_async();

        for (int it = 0; it < nit; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            // ---- EPI1: A~ -> T3;  K~ -> smem ----------------------------------------------
            tc::mbar_wait(&bars[FULLKV], ph, abort, status, 41);
            if (CHAIN) {
                tc::mbar_wait(&bars[BA], ph, abort, status, 42);
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
            {
                const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                    *reinterpret_cast<uint4*>(sKt + off) = scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w1);
                }
            }

            // ---- EPI2: Inner = g^(r+1) Q P0 + A~ V -> smem (first-order mode: the output tile) ----
            if (CHAIN) {
                tc::mbar_wait(&bars[BP], ph, abort, status, 43);
                tc::fence_after_sync();
                const float s1 = r < Wc ? gp[r + 1] : 0.f;
                const float keep = r < Wc ? 1.f : 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qp[16], av[16];
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, qp);
                    tc::tmem_ld16(lrow + T2 + 32 * h + 16 * half, av);
                    tc::tmem_wait_ld();
                    float in[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) in[j] = s1 * __uint_as_float(qp[j]) + keep * __uint_as_float(av[j]);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        *reinterpret_cast<uint4*>(sIn + tc::sw128_chunk(r, 4 * h + 2 * half + j)) = pack8(&in[8 * j]);
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BPS]);

            if (!SUMMARY && !FO) {
                // ---- EPI3: out = g^(r+1) Q E0 + A~ Inner ------------------------------------
                tc::mbar_wait(&bars[BO], ph, abort, status, 44);
                tc::fence_after_sync();
                const float s1 = gp[r + 1];
                bf16* out = static_cast<bf16*>(a.out) + ((size_t)bh * a.n + (size_t)c * kW + r) * kD + 32 * h;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qe[16], ai[16];
                    tc::tmem_ld16(lrow + T1 + 32 * h + 16 * half, qe);
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, ai);
                    tc::tmem_wait_ld();
                    if (r < Wc) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            float o[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                o[u] = s1 * __uint_as_float(qe[8 * j + u]) + __uint_as_float(ai[8 * j + u]);
                            *reinterpret_cast<uint4*>(out + 16 * half + 8 * j) = pack8(o);
                        }
                    }
                }
            }

            // ---- EPI4: state update ------------------------------------------------------------
            tc::mbar_wait(&bars[BST], ph, abort, status, 45);
            tc::fence_after_sync();
            {
                const float rho = gp[Wc];
                uint32_t v[32];
                // ST rows < 64: dP in columns 0..63 (T3); rows >= 64: dE in columns 64..127 (T2)
                tc::tmem_ld32(lrow + (r < 64 ? T3 : T2) + 32 * h, v);
                if (SUMMARY && !FO) {
                    uint32_t w[16];
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * (r >> 6), w);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) rr[j] += __uint_as_float(w[j]);
                } else {
                    tc::tmem_wait_ld();
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) st[j] = rho * st[j] + __uint_as_float(v[j]);
                publish_state();
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BS]);
        }

        if (FO && !SUMMARY && a.final_state && seg == a.nseg - 1 && r < 64) {  // P after the last token
            float* dst = a.final_state + (size_t)bh * kD * kD + (size_t)r * kD + 32 * h;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[j] = st[j];
        }
        if (SUMMARY && seg < a.nsum) {  // (a launch that stores Inner also covers the last segment)
            const size_t si = (size_t)bh * a.nsum + seg;
            float* dst = r < 64 ? a.ws + a.L.PB + si * kD * kD + (size_t)r * kD
                                : a.ws + a.L.EB + si * kD * kD + (size_t)(r - 64) * kD;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[32 * h + j] = st[j];
            float* dr = a.ws + a.L.RB + si * kD * kD + (size_t)(r & 63) * kD + 32 * h + 16 * (r >> 6);
#pragma unroll
            for (int j = 0; j < 16; ++j) dr[j] = rr[j];
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------------
// Output pass from the stored segment-local Inner (chunk 128, more than one segment).
//
// The summary pass stores, for every token of a segment, Inner^sl_t = P^sl_t^T q_t with the
// value moment P^sl accumulated from zero at the segment start (bf16, in the output buffer).
// With the segment's carry P_in,
//     Inner_t = Inner^sl_t + g^(t - t0 + 1) P_in^T q_t,        t0 = the segment's first token,
// so P leaves the chunk-to-chunk chain: only E is carried, and this pass reads q, k and
// Inner^sl (no v).  Per chunk (local row r, it = chunk index in the segment):
//   MMA1  A = Q K^T -> T0T1;  Q P_in -> T2                       (no dependence on E)
//   EPI1  A~ = A * [j <= r] g^(r-j) -> T3;  Inner = Inner^sl + g^(it W + r + 1) Q P_in (bf16, in
//         place);  K~ = diag(g^(Wc-1-i)) K (smem)
//   MMA2  A~ Inner -> T0;  Q E0 -> T1;  [K~^T ; K~^T] Inner -> T2 (dE, rows 0..63 and 64..127)
//   EPI2  out = g^(r+1) Q E0 + A~ Inner  (bf16 tile in smem, one TMA tile store over this
//         chunk's Inner^sl, already consumed);  E <- g^Wc E + dE;  bf16 E0 (smem)
namespace aout {

constexpr uint32_t oQ = 0, oK = kTile, oI = 2 * kTile, oKt = 3 * kTile, oO = 4 * kTile;
constexpr uint32_t oPi = 5 * kTile, oE0 = oPi + 8192;  // P_in, E0: [64][64] bf16 each
constexpr uint32_t oGP = oE0 + 8192;
constexpr uint32_t oBar = oGP + 1088;
constexpr uint32_t oMisc = oBar + 16 * 8;
constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
constexpr uint32_t T0 = 0, T1 = 64, T2 = 128, T3 = 192;

enum Bar { FQK = 0, FI, BA, BAT, BB, BOS, kBarCount };

struct Maps {
    CUtensorMap q, k, i;  // i: the output buffer, holding Inner^sl, then out
};

}  // namespace aout

__global__ void __launch_bounds__(kThreads, 2)
    ahla_out_i_tc_kernel(const __grid_constant__ aout::Maps maps, const AhlaArgs a, int* status) {
    // this pass's layout (shadows the kernel above)
    constexpr uint32_t oQ = aout::oQ, oK = aout::oK, oI = aout::oI, oKt = aout::oKt, oO = aout::oO,
                       oPi = aout::oPi, oE0 = aout::oE0;
    constexpr uint32_t oGP = aout::oGP, oBar = aout::oBar, oMisc = aout::oMisc;
    constexpr uint32_t T0 = aout::T0, T1 = aout::T1, T2 = aout::T2, T3 = aout::T3;
    constexpr int FQK = aout::FQK, FI = aout::FI, BA = aout::BA, BAT = aout::BAT, BB = aout::BB, BOS = aout::BOS,
                  kBarCount = aout::kBarCount;
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

    // epilogue thread: TMEM lane / token row r, column half h; E row er, columns ec .. ec+15
    const int q4 = warp & 3, h = (warp - 1) >> 2;
    const int r = 32 * q4 + lane;
    const int er = r & 63, ec = 32 * h + 16 * (r >> 6);
    float ee[16];
    auto publish_e = [&]() {
#pragma unroll
        for (int j = 0; j < 2; ++j)
            *reinterpret_cast<uint4*>(sm + oE0 + tc::sw128_chunk(er, ec / 8 + j)) = pack8(&ee[8 * j]);
    };

    for (int i = tid; i < 2 * kW + 1; i += kThreads) gp[i] = pow_decay(log2g, (float)i);
    if (tid == 0) {
        for (int b = 0; b < kBarCount; ++b) tc::mbar_init(&bars[b], (b == BAT || b == BOS) ? 8 : 1);
        *abort = 0;
        tc::mbar_fence_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_holder, kTmemCols);
    } else {
        // carry-in of the segment: P_in (bf16, smem) and E_in (fp32 registers, bf16 copy in smem)
        const size_t cidx = (size_t)bh * a.nseg + seg;
        if (r < 64) {
            const float* src = a.ws + a.L.Pin + cidx * kD * kD + (size_t)r * kD + 32 * h;
            float t[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) t[j] = src[j];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(sm + oPi + tc::sw128_chunk(r, 4 * h + j)) = pack8(&t[8 * j]);
        }
        const float* esrc = a.ws + a.L.Ein + cidx * kD * kD + (size_t)er * kD + ec;
#pragma unroll
        for (int j = 0; j < 16; ++j) ee[j] = esrc[j];
        publish_e();
        tc::fence_proxy_async();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ control thread
        if (lane == 0 && nit > 0) {
            const uint32_t sQ = smem_u32(sm + oQ), sK = smem_u32(sm + oK), sI = smem_u32(sm + oI);
            const uint32_t sKt = smem_u32(sm + oKt), sPi = smem_u32(sm + oPi), sE0 = smem_u32(sm + oE0);
            auto load_qk = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FQK], 2 * kTile);
                tc::tma_load_3d(sm + oQ, &maps.q, 0, c * kW, bh, &bars[FQK]);
                tc::tma_load_3d(sm + oK, &maps.k, 0, c * kW, bh, &bars[FQK]);
            };
            auto load_i = [&](int c) {
                tc::mbar_arrive_expect_tx(&bars[FI], kTile);
                tc::tma_load_3d(sm + oI, &maps.i, 0, c * kW, bh, &bars[FI]);
            };
            constexpr uint32_t I_AB = tc::idesc_bf16(128, 128, 0, 0);   // K-major x K-major, N = 128
            constexpr uint32_t I_QX = tc::idesc_bf16(128, 64, 0, 1);    // K-major x MN-major, N = 64
            constexpr uint32_t I_TS64 = tc::idesc_bf16(128, 64, 0, 1);  // A (TMEM) x MN-major B, N = 64
            constexpr uint32_t I_ST64 = tc::idesc_bf16(128, 64, 1, 1);  // MN-major x MN-major, N = 64
            load_qk(c_begin);
            load_i(c_begin);
            int loads = 1;
            for (int it = 0; it < nit; ++it) {
                const uint32_t ph = it & 1;
                tc::mbar_wait(&bars[FQK], ph, abort, status, 81);
                if (it > 0) {  // previous chunk's EPI2 done: T0..T2 read, its output tile staged
                    tc::mbar_wait(&bars[BOS], ph ^ 1, abort, status, 82);
                    tc::tma_store_3d(&maps.i, sm + oO, 0, (c_begin + it - 1) * kW, bh);
                    tc::bulk_commit();
                }
                tc::fence_after_sync();
                // MMA1: A = Q K^T -> T0T1;  Q P_in -> T2
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T0, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sK + 32 * ks, 16, 1024),
                               I_AB, ks > 0);
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T2, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sPi + 2048 * ks, 16, 1024),
                               I_QX, ks > 0);
                tc::mma_commit(&bars[BA]);
                tc::mbar_wait(&bars[BAT], ph, abort, status, 83);  // A~, Inner, K~ written
                tc::bulk_wait_read_all();  // the output tile slot is free before this chunk's EPI2
                tc::fence_after_sync();
                // MMA2: A~ Inner -> T0;  Q E0 -> T1;  [K~^T ; K~^T] Inner -> T2
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + T0, tmem + T3 + 8 * ks, tc::smem_desc(sI + 2048 * ks, 16, 1024), I_TS64, ks > 0);
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + T1, tc::smem_desc(sQ + 32 * ks, 16, 1024), tc::smem_desc(sE0 + 2048 * ks, 16, 1024),
                               I_QX, ks > 0);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + T2, tc::smem_desc(sKt + 2048 * ks, 0, 1024), tc::smem_desc(sI + 2048 * ks, 16, 1024),
                               I_ST64, ks > 0);
                tc::mma_commit(&bars[BB]);
                tc::mbar_wait(&bars[BB], ph, abort, status, 84);  // Q, K, Inner and K~ no longer read
                if (it + 1 < nit) {
                    load_qk(c_begin + it + 1);
                    load_i(c_begin + it + 1);
                    ++loads;
                }
            }
            tc::mbar_wait(&bars[BOS], (nit - 1) & 1, abort, status, 85);  // the last output tile
            tc::tma_store_3d(&maps.i, sm + oO, 0, (c_begin + nit - 1) * kW, bh);
            tc::bulk_commit();
            volatile int never = 0;
            tc::mbar_wait(&bars[BB], (nit - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FQK], (loads - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[FI], (loads - 1) & 1, &never, nullptr, 0);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        unsigned char* sK = sm + oK;
        unsigned char* sI = sm + oI;
        unsigned char* sKt = sm + oKt;
        const float ginv = g > 0.f ? 1.f / g : 0.f;
        for (int it = 0; it < nit; ++it) {
            const uint32_t ph = it & 1;
            const int c = c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            // ---- EPI1: A~ -> T3;  Inner (in place);  K~ -----------------------------------------
            tc::mbar_wait(&bars[FQK], ph, abort, status, 91);
            tc::mbar_wait(&bars[FI], ph, abort, status, 92);
            tc::mbar_wait(&bars[BA], ph, abort, status, 93);
            tc::fence_after_sync();
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const int cb = 64 * h + 32 * p;
                const float first = r >= cb ? gp[r - cb] : 0.f;
                masked_block(lrow + T0 + cb, lrow + T3 + cb / 2, r, cb, row0, first, ginv);
            }
            {
                const float f = pow_decay(log2g, (float)(it * kW + r + 1));
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qp[16];
                    tc::tmem_ld16(lrow + T2 + 32 * h + 16 * half, qp);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t off = tc::sw128_chunk(r, 4 * h + 2 * half + j);
                        const uint4 il = *reinterpret_cast<const uint4*>(sI + off);
                        const uint32_t iw[4] = {il.x, il.y, il.z, il.w};
                        float in[8];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            in[2 * u] = bf_lo(iw[u]) + f * __uint_as_float(qp[8 * j + 2 * u]);
                            in[2 * u + 1] = bf_hi(iw[u]) + f * __uint_as_float(qp[8 * j + 2 * u + 1]);
                        }
                        *reinterpret_cast<uint4*>(sI + off) = pack8(in);
                    }
                }
                const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = tc::sw128_chunk(r, 4 * h + j);
                    *reinterpret_cast<uint4*>(sKt + off) = scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w1);
                }
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BAT]);

            // ---- EPI2: out = g^(r+1) Q E0 + A~ Inner;  E <- g^Wc E + dE --------------------------
            tc::mbar_wait(&bars[BB], ph, abort, status, 94);
            tc::fence_after_sync();
            {
                const float s1 = gp[r + 1];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t qe[16], ai[16];
                    tc::tmem_ld16(lrow + T1 + 32 * h + 16 * half, qe);
                    tc::tmem_ld16(lrow + T0 + 32 * h + 16 * half, ai);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {  // output tile (rows >= Wc fall outside the tensor)
                        float o[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            o[u] = s1 * __uint_as_float(qe[8 * j + u]) + __uint_as_float(ai[8 * j + u]);
                        *reinterpret_cast<uint4*>(sm + oO + tc::sw128_chunk(r, 4 * h + 2 * half + j)) = pack8(o);
                    }
                }
                uint32_t de[16];
                tc::tmem_ld16(lrow + T2 + ec, de);
                tc::tmem_wait_ld();
                const float rho = gp[Wc];
#pragma unroll
                for (int j = 0; j < 16; ++j) ee[j] = rho * ee[j] + __uint_as_float(de[j]);
                publish_e();  // read by the next chunk's MMA2, after its EPI1 arrives
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[BOS]);
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

bool ahla_tc_available() { return encode_fn() != nullptr; }

size_t ahla_tc_smem() { return kSmemBytes; }

int launch_ahla_tc(const AhlaArgs& a, bool summary, int* status, cudaStream_t st, bool first_order) {
    if (a.nseg_launch <= 0 || a.BH <= 0) return 0;
    TcMaps maps;
    if (!make_map(&maps.q, a.q, a.BH, a.n) || !make_map(&maps.k, a.k, a.BH, a.n) || !make_map(&maps.v, a.v, a.BH, a.n))
        return -2;
    if (((summary && !first_order && a.store_inner) || (first_order && !summary)) &&
        !make_map(&maps.o, a.out, a.BH, a.n))
        return -2;
    dim3 grid(a.nseg_launch, a.BH);
    auto kfn = summary ? (first_order ? ahla_tc_kernel<true, true> : ahla_tc_kernel<true, false>)
                       : (first_order ? ahla_tc_kernel<false, true> : ahla_tc_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) kfn<<<grid, kThreads, kSmemBytes, st>>>(maps, a, status);
    if (e != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_ahla_tc_out_i(const AhlaArgs& a, int* status, cudaStream_t st) {
    if (a.nseg_launch <= 0 || a.BH <= 0) return 0;
    aout::Maps maps;
    if (!make_map(&maps.q, a.q, a.BH, a.n) || !make_map(&maps.k, a.k, a.BH, a.n) || !make_map(&maps.i, a.out, a.BH, a.n))
        return -2;
    cudaError_t e = cudaFuncSetAttribute(ahla_out_i_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         aout::kSmemBytes);
    if (e != cudaSuccess) return -1;
    ahla_out_i_tc_kernel<<<dim3(a.nseg_launch, a.BH), kThreads, aout::kSmemBytes, st>>>(maps, a, status);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2
