// First-order chunked linear attention on the 5th-generation tensor cores, d = dv = 128,
// chunk width 128 (bf16 tiles, fp32 state).  It is the building block of the d = 128
// training path: the masked HLA-2 output is two chained first-order scans, and so is its
// reverse mode (page "Higher-order Linear Attention", section summary §4.2: the reverse-mode
// scan gives the serial recurrence's gradients).
//
// With decay g (= gamma or gamma^2 of the head), one launch computes over every segment of
// every head
//   forward:  Y_t = sum_{i <= t} g^(t-i) (x_t . k_i) v_i   (+ g^(t-t0+1) x_t^T Sig_in)
//   reverse:  Y_t = sum_{i >= t} g^(i-t) (x_t . k_i) v_i   (+ g^(t1-t) x_t^T Sig_in)
// with Sig = sum_i k_i v_i^T decayed to the segment's start (forward) or end (reverse);
// Sig_in is the carry from the other segments.  Per chunk of W = 128 rows r (Wc valid):
//   MMA-G  G = X K^T                                     (128 x 128 fp32, tensor memory)
//   EPI-1  G~ = mask(G) (forward [i <= r] g^(r-i), reverse [i >= r] g^(i-r)), bf16 packed
//          in tensor memory beside fX = diag(f_r) X (forward f = g^(r+1), reverse
//          g^(Wc-r)): the A operand of the next product;  K~ = diag(w_i) K in shared memory
//          (forward w = g^(Wc-1-i), reverse g^i)
//   MMA-Y  Y = [G~ | fX] [V ; Sig0]                       (one accumulation, K = 256)
//   MMA-S  dSig = K~^T V
//   EPI-S  Sig <- g^Wc Sig + dSig  (fp32 registers, 64 a thread), bf16 Sig0 for the next chunk
//   EPI-Y  Y (+ a partial sum read from global) -> bf16 tile -> one TMA tile store
// Optional parts, chosen per launch:
//   * a second key/value pair with the values and keys swapped, (K2, V2) = (V, K), sharing
//     X and the state: Y = G~1 V + G~2 K + fX Sig0, Sig = sum_i (k_i v_i^T + v_i k_i^T)
//     (the symmetric pair of the key-gradient scan);
//   * the next summary: Sig'_B = sum_t w'_t y_t u_t^T over the segment, keys = this launch's
//     own (bf16) output and values u = one of its inputs or an extra tile, decayed with g'
//     to the segment's end (forward) or start (reverse) -- the segment summary of the scan
//     that takes Y as its keys, so that scan needs no cross term;
//   * a partial output (bf16, same layout) added before the store.
// The carry Sig_in is read as stored, transposed, or symmetrised (Sig + Sig^T).
//
// A second kernel forms segment summaries only: Sig_B = sum_i w_i k_i v_i^T with no chain,
// the keys scaled in shared memory and the products accumulated in tensor memory.
//
// Roles: warp 0 allocates tensor memory and one of its threads issues the TMA loads and every
// MMA; warps 1..8 move data between tensor memory, registers and shared memory (warp w holds
// TMEM lanes 32 (w % 4) .. +31 = token / feature rows, and half (w - 1) / 4 of the columns).
// One CTA per SM (up to 192 KB of shared memory, all 512 tensor-memory columns).  Every
// wait is bounded; on a timeout the kernel records the site in the status word, drains and
// exits.
#include "fo_common.cuh"

namespace hla2 {

namespace {

namespace la {

constexpr int kW = 128, kD = 128;
constexpr int kThreads = 288;          // 1 control warp + 8 epilogue warps
// the output kernel adds warp 9: with G / Y double-buffered it issues the tile loads and stores
// while warp 0 issues only the MMAs
constexpr int kThreadsOut = 320, kLoadWarp = 9;
constexpr uint32_t kBlk = 128 * 128;   // one [128 rows][64 bf16] SW128 column block (16 KB)
constexpr uint32_t kTile = 2 * kBlk;   // a [128][128] bf16 tile: column blocks 0 (cols 0..63) and 1
constexpr uint32_t kTmemCols = 512;

// Shared-memory plan of the output kernel (byte offsets of 32 KB slots from the 1024-aligned
// base).  Two key slots (chunk j in slot j % 2) let the next chunk's keys load while this
// chunk's products still read its own; with KVS the key slot also serves as the value tile.
template <bool R2, bool KVS, bool XVS, bool ADD>
struct OutLayout {
    static constexpr uint32_t oQ = 0;
    static constexpr uint32_t oK = kTile;                                     // slots oK, oK + kTile
    static constexpr uint32_t oV = KVS ? oK : oK + 2 * kTile;                 // KVS: the key slot
    static constexpr uint32_t oEnd0 = KVS ? oK + 2 * kTile : oV + kTile;
    static constexpr uint32_t oXV = XVS ? oEnd0 : oV;                         // next summary's values
    static constexpr uint32_t oAD = XVS ? oXV + kTile : oEnd0;                // partial (ADD)
    static constexpr uint32_t oKt = ADD ? oAD + kTile : oAD;                  // K~ (and V~ for R2)
    static constexpr uint32_t oKt2 = oKt + kTile;
    static constexpr uint32_t oS0 = R2 ? oKt2 + kTile : oKt + kTile;         // bf16 Sig0
    static constexpr bool kStageInQ = R2;                                     // no room for a stage slot
    static constexpr uint32_t oST = kStageInQ ? oQ : oS0 + kTile;             // output tile
    static constexpr uint32_t oGP = (kStageInQ ? oS0 : oST) + kTile;          // g^0 .. g^(2W)
    static constexpr uint32_t oBar = oGP + 1088;
    static constexpr uint32_t oMisc = oBar + 16 * 8;
    static constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;  // + alignment slack
    __host__ __device__ static constexpr uint32_t key(int j) { return oK + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t val(int j) { return KVS ? key(j) : oV; }
};

// Tensor-memory columns.  R = 1: G / Y of chunk j in [0,128) or, without a next summary,
// alternately [384,512); A operands [128,256) (G~ | fX); dSig [256,384); next summary
// [384,512).  R = 2: G1 [0,128), G2 [128,256); after EPI-1 Y [0,128) and dSig [128,256);
// A operands [256,448) (G~1 | G~2 | fX).
template <bool R2, bool NSUM>
struct Cols {
    static constexpr bool kTwoG = !R2 && !NSUM;  // G / Y double-buffered
    static constexpr uint32_t TA = R2 ? 256 : 128;
    static constexpr uint32_t TX = TA + (R2 ? 128 : 64);  // fX
    static constexpr uint32_t TS = R2 ? 128 : 256;
    static constexpr uint32_t TN = 384;
    __device__ static constexpr uint32_t TG(int j) { return kTwoG && (j & 1) ? 384u : 0u; }
};

// BSU1: with G / Y double-buffered BSU serves even chunks and BSU1 odd ones (two waiters)
enum Bar { FQ = 0, FK0, FK1, FV, BG, BGT, BSU, BS, BYT, BN, BSF, BSU1, kBarCount };

struct Maps {
    CUtensorMap x, k, v, xv, ad, out;
};

}  // namespace la

// ----------------------------------------------------------------------------------------
// Output kernel.  REV: reverse direction.  NSUM: next summary of the output.  R2: the swapped
// second pair.  KVS: keys and values are the same tensor (one tile).  XVS: the next
// summary's values are a separate tensor (else the value tile).  ADD: partial added.
//
// Schedule per chunk j (control thread / epilogue warps):
//   MMA-G(j) -> EPI-1(j) -> MMA-Y(j), MMA-S(j) (one commit) -> EPI-S(j) -> ...
// With G / Y double-buffered (no next summary, one pair) the epilogue runs EPI-S(j), EPI-1(j+1),
// EPI-Y(j): MMA-G(j+1) is issued as soon as chunk j's products are, and MMA-Y(j+1) runs while
// chunk j's output is staged.  Otherwise the order is EPI-S(j), EPI-Y(j), EPI-1(j+1).
template <bool REV, bool NSUM, bool R2, bool KVS, bool XVS, bool ADD>
__global__ void __launch_bounds__(la::kThreadsOut, 1)
    fo_out_tc_kernel(const __grid_constant__ la::Maps maps, const FoArgs a) {
    using Lay = la::OutLayout<R2, KVS, XVS, ADD>;
    using C = la::Cols<R2, NSUM>;
    constexpr bool kTwoG = C::kTwoG;
    constexpr int kW = la::kW;
    pdl_trigger();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gp = reinterpret_cast<float*>(sm + Lay::oGP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Lay::oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::oMisc + 4);
    int* status = a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const FoSeg sg = la_seg(a, seg);
    const int nit = sg.nit;
    const float gam = head_decay(a.gamma, bh, a.H);
    const float log2g = (float)a.pow * log2f(gam);
    const float log2gn = (float)a.pow_next * log2f(gam);
    const float g = exp2f(log2g);

    for (int i = tid; i < 2 * kW + 1; i += la::kThreadsOut) gp[i] = pow_decay(log2g, (float)i);
    if (tid == 0) {
        for (int b = 0; b < la::kBarCount; ++b) {
            const bool from_epilogue = (b == la::BGT || b == la::BS || b == la::BYT);
            tc::mbar_init(&bars[b], from_epilogue ? 8 : 1);
        }
        *abort = 0;
        tc::mbar_fence_init();
    }
    pdl_wait();  // everything below reads what earlier kernels of the stream wrote

    // epilogue thread: TMEM lane / row r, column half h (columns 64h .. 64h+63)
    const int q4 = warp & 3, h = (warp - 1) >> 2;
    const int r = 32 * q4 + lane;
    float sig[64];  // Sig row r, columns 64h ..
    auto publish_sig = [&]() {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(sm + Lay::oS0 + la_off(h, r, j)) = la_pack8(&sig[8 * j]);
    };

    if (warp == 0) {
        tc::tmem_alloc(tmem_holder, la::kTmemCols);
    } else if (warp <= 8) {
        // carry-in of the segment (zero without one), as stored, transposed or symmetrised
        if (a.carry && HLA2_IN(bh < a.BH && seg < a.nseg, 801)) {
            const float* src = a.carry + ((size_t)bh * a.nseg + seg) * la::kD * la::kD;
            if (a.carry_mode == 0) {
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src + (size_t)r * la::kD + 64 * h + j);
                    sig[j] = x.x, sig[j + 1] = x.y, sig[j + 2] = x.z, sig[j + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) sig[j] = src[(size_t)(64 * h + j) * la::kD + r];
                if (a.carry_mode == 2) {
#pragma unroll
                    for (int j = 0; j < 64; ++j) sig[j] += src[(size_t)r * la::kD + 64 * h + j];
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) sig[j] = 0.f;
        }
        publish_sig();
        tc::fence_proxy_async();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    auto chunk_of = [&](int it) { return REV ? sg.c_end - 1 - it : sg.c_begin + it; };
    auto fk = [&](int j) { return &bars[(j & 1) ? la::FK1 : la::FK0]; };
    // the products' barrier: with G / Y double-buffered a pair by chunk parity (the epilogue and
    // the load thread wait on it, and neither may see a later phase)
    auto bsu = [&](int j) { return &bars[kTwoG && (j & 1) ? la::BSU1 : la::BSU]; };
    auto bsu_par = [&](int j) { return (uint32_t)(kTwoG ? (j >> 1) & 1 : j & 1); };

    if (warp == 0 || warp == la::kLoadWarp) {
        // ------------------------------------------------------------ control threads
        const bool mma_role = warp == 0;
        if (lane == 0 && nit > 0 && (kTwoG || mma_role)) {
            auto load2 = [&](uint32_t slot, const CUtensorMap* m, int c, uint64_t* bar) {
                tc::tma_load_3d(sm + slot, m, 0, c * kW, bh, bar);
                tc::tma_load_3d(sm + slot + la::kBlk, m, 64, c * kW, bh, bar);
            };
            auto load_x = [&](int j) {
                tc::mbar_arrive_expect_tx(&bars[la::FQ], la::kTile);
                load2(Lay::oQ, &maps.x, chunk_of(j), &bars[la::FQ]);
            };
            auto load_k = [&](int j) {
                tc::mbar_arrive_expect_tx(fk(j), la::kTile);
                load2(Lay::key(j), &maps.k, chunk_of(j), fk(j));
            };
            constexpr int kVTiles = (KVS ? 0 : 1) + (XVS ? 1 : 0) + (ADD ? 1 : 0);
            auto load_v = [&](int j) {
                if (kVTiles == 0) return;
                tc::mbar_arrive_expect_tx(&bars[la::FV], kVTiles * la::kTile);
                if (!KVS) load2(Lay::oV, &maps.v, chunk_of(j), &bars[la::FV]);
                if (XVS) load2(Lay::oXV, &maps.xv, chunk_of(j), &bars[la::FV]);
                if (ADD) load2(Lay::oAD, &maps.ad, chunk_of(j), &bars[la::FV]);
            };
            constexpr bool v_late = NSUM || ADD;  // the value group is still read after the products
            const uint32_t sX = smem_u32(sm + Lay::oQ), sV = smem_u32(sm + Lay::oV);
            const uint32_t sKt = smem_u32(sm + Lay::oKt), sKt2 = smem_u32(sm + Lay::oKt2);
            const uint32_t sS0 = smem_u32(sm + Lay::oS0), sST = smem_u32(sm + Lay::oST);
            const uint32_t sXV = smem_u32(sm + Lay::oXV);
            constexpr uint32_t I_KK = tc::idesc_bf16(128, 128, 0, 0);  // K-major x K-major
            constexpr uint32_t I_TM = tc::idesc_bf16(128, 128, 0, 1);  // A (TMEM, K-major) x MN-major B
            constexpr uint32_t I_MM = tc::idesc_bf16(128, 128, 1, 1);  // MN-major x MN-major
            // K-major operand, K = 128 features in two column blocks; MN-major, K = 128 tokens
            auto kdesc = [](uint32_t base, int ks) {
                return tc::smem_desc(base + (uint32_t)(ks >> 2) * la::kBlk + (uint32_t)(ks & 3) * 32, 16, 1024);
            };
            auto mdesc = [](uint32_t base, int ks) { return tc::smem_desc(base + 2048u * ks, la::kBlk, 1024); };
            int lx = 0, lk = 0, lv = 0;
            // MMA-G: G = X K^T (R2: and X V^T), chunk j
            auto mma_g = [&](int j) {
                const uint32_t sK = smem_u32(sm + Lay::key(j));
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + C::TG(j), kdesc(sX, ks), kdesc(sK, ks), I_KK, ks > 0);
                if (R2)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + C::TG(j) + 128, kdesc(sX, ks), kdesc(sV, ks), I_KK, ks > 0);
                tc::mma_commit(&bars[la::BG]);
            };
            auto wait_g_inputs = [&](int j) {
                tc::mbar_wait(&bars[la::FQ], j & 1, abort, status, 101);
                tc::mbar_wait(fk(j), (j >> 1) & 1, abort, status, 102);
                if (R2) tc::mbar_wait(&bars[la::FV], j & 1, abort, status, 103);
                tc::fence_after_sync();
            };
            // after EPI-Y(j): the tile store and the next summary's products (finish_store); then
            // the late loads and the stage freed (finish_release), which the two-region order
            // runs after the next Gram is issued
            auto finish_store = [&](int j) {
                tc::mbar_wait(&bars[la::BYT], j & 1, abort, status, 108);
                tc::fence_after_sync();
                const int c = chunk_of(j);
                tc::tma_store_3d(&maps.out, sm + Lay::oST, 0, c * kW, bh);
                tc::tma_store_3d(&maps.out, sm + Lay::oST + la::kBlk, 64, c * kW, bh);
                tc::bulk_commit();
                if (NSUM) {  // next summary: T_N += Y^T (w' U)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + C::TN, mdesc(sST, ks), mdesc(sXV, ks), I_MM, (j > 0 || ks > 0) ? 1u : 0u);
                    tc::mma_commit(&bars[la::BN]);
                }
            };
            auto finish_release = [&](int j) {
                if (NSUM) tc::mbar_wait(&bars[la::BN], j & 1, abort, status, 109);
                if (v_late && j + 1 < nit && kVTiles > 0) {
                    load_v(j + 1);
                    ++lv;
                }
                tc::bulk_wait_read_all();  // the output tile has been read
                if (Lay::kStageInQ && j + 1 < nit) {
                    load_x(j + 1);
                    ++lx;
                }
                tc::mbar_arrive(&bars[la::BSF]);
            };
            auto finish = [&](int j) {
                finish_store(j);
                finish_release(j);
            };

            auto prologue_loads = [&]() {
                load_x(0);
                ++lx;
                load_k(0);
                ++lk;
                if (kVTiles > 0) {
                    load_v(0);
                    ++lv;
                }
                if (nit > 1) {
                    load_k(1);
                    ++lk;
                }
            };
            if constexpr (kTwoG) {
                // warp 0 issues the MMAs; warp 9 the loads and the tile stores
                if (mma_role) {
                    wait_g_inputs(0);
                    mma_g(0);
                    for (int j = 0; j < nit; ++j) {
                        tc::mbar_wait(&bars[la::BGT], j & 1, abort, status, 104);  // G read; G~, fX, K~ written
                        if (j > 0) tc::mbar_wait(&bars[la::BS], (j - 1) & 1, abort, status, 106);  // Sig0 of chunk j
                        if (!KVS) tc::mbar_wait(&bars[la::FV], j & 1, abort, status, 105);  // the value tile
                        tc::fence_after_sync();
                        const uint32_t sVj = smem_u32(sm + Lay::val(j));
                        // MMA-Y: Y = [G~ | fX] [V ; Sig0];  MMA-S: dSig = K~^T V
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_ts(tmem + C::TG(j), tmem + C::TA + 8 * ks, mdesc(sVj, ks), I_TM, ks > 0);
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_ts(tmem + C::TG(j), tmem + C::TX + 8 * ks, mdesc(sS0, ks), I_TM, 1);
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_ss(tmem + C::TS, mdesc(sKt, ks), mdesc(sVj, ks), I_MM, ks > 0);
                        tc::mma_commit(bsu(j));
                        if (j + 1 < nit) {  // G / Y region (j + 1) % 2: EPI-Y(j - 1) has read it
                            if (j > 0) tc::mbar_wait(&bars[la::BYT], (j - 1) & 1, abort, status, 110);
                            wait_g_inputs(j + 1);
                            mma_g(j + 1);
                        }
                    }
                    volatile int never = 0;  // drain (bounded, ignoring the abort flag)
                    tc::mbar_wait(bsu(nit - 1), bsu_par(nit - 1), &never, nullptr, 0);
                } else {
                    prologue_loads();
                    for (int j = 0; j < nit; ++j) {
                        tc::mbar_wait(&bars[la::BGT], j & 1, abort, status, 111);  // X and key slot j % 2 read
                        if (j + 1 < nit) {
                            load_x(j + 1);
                            ++lx;
                        }
                        if (!KVS && j + 2 < nit) {
                            load_k(j + 2);
                            ++lk;
                        }
                        if (j > 0) finish(j - 1);  // after EPI-Y(j - 1)
                        tc::mbar_wait(bsu(j), bsu_par(j), abort, status, 107);  // chunk j's products done
                        if (KVS && j + 2 < nit) {
                            load_k(j + 2);
                            ++lk;
                        }
                        if (!v_late && !KVS && j + 1 < nit) {
                            load_v(j + 1);
                            ++lv;
                        }
                    }
                    finish(nit - 1);
                    volatile int never = 0;  // drain (bounded, ignoring the abort flag)
                    tc::mbar_wait(&bars[la::FQ], (lx - 1) & 1, &never, nullptr, 0);
                    tc::mbar_wait(&bars[la::FK0], ((lk + 1) / 2 - 1) & 1, &never, nullptr, 0);
                    if (lk > 1) tc::mbar_wait(&bars[la::FK1], (lk / 2 - 1) & 1, &never, nullptr, 0);
                    if (lv > 0) tc::mbar_wait(&bars[la::FV], (lv - 1) & 1, &never, nullptr, 0);
                    tc::bulk_wait_all();
                }
            } else {
            prologue_loads();
            wait_g_inputs(0);
            mma_g(0);
            for (int j = 0; j < nit; ++j) {
                tc::mbar_wait(&bars[la::BGT], j & 1, abort, status, 104);  // G read; G~, fX, K~ written
                if (j > 0) tc::mbar_wait(&bars[la::BS], (j - 1) & 1, abort, status, 106);  // Sig0 of chunk j
                if (!Lay::kStageInQ && j + 1 < nit) {  // X no longer read
                    load_x(j + 1);
                    ++lx;
                }
                if (!R2 && !KVS && j + 2 < nit) {  // key slot j % 2 no longer read (unless MMA-Y reads it:
                    load_k(j + 2);                    // the swapped pair, or keys as values)
                    ++lk;
                }
                if (!KVS) tc::mbar_wait(&bars[la::FV], j & 1, abort, status, 105);  // the value tile
                tc::fence_after_sync();
                const uint32_t sK = smem_u32(sm + Lay::key(j)), sVj = smem_u32(sm + Lay::val(j));
                // MMA-Y: Y = [G~ | (G~2) | fX] [V ; (K) ; Sig0]
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + C::TG(j), tmem + C::TA + 8 * ks, mdesc(sVj, ks), I_TM, ks > 0);
                if (R2)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + C::TG(j), tmem + C::TA + 64 + 8 * ks, mdesc(sK, ks), I_TM, 1);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + C::TG(j), tmem + C::TX + 8 * ks, mdesc(sS0, ks), I_TM, 1);
                // MMA-S: dSig = K~^T V (R2: + V~^T K)
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + C::TS, mdesc(sKt, ks), mdesc(sVj, ks), I_MM, ks > 0);
                if (R2)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + C::TS, mdesc(sKt2, ks), mdesc(sK, ks), I_MM, 1);
                tc::mma_commit(&bars[la::BSU]);
                if (kTwoG) {
                    // EPI-Y(j - 1) has read G / Y region (j + 1) % 2: the next Gram goes before the
                    // wait for the previous tile store to leave the stage
                    if (j > 0) finish_store(j - 1);
                    if (j + 1 < nit) {
                        wait_g_inputs(j + 1);
                        mma_g(j + 1);
                    }
                    if (j > 0) finish_release(j - 1);
                    tc::mbar_wait(&bars[la::BSU], j & 1, abort, status, 107);  // chunk j's products done
                    if ((R2 || KVS) && j + 2 < nit) {
                        load_k(j + 2);
                        ++lk;
                    }
                    if (!v_late && !KVS && j + 1 < nit) {
                        load_v(j + 1);
                        ++lv;
                    }
                } else {
                    finish(j);  // after EPI-Y(j), so chunk j's products are done
                    if ((R2 || KVS) && j + 2 < nit) {
                        load_k(j + 2);
                        ++lk;
                    }
                    if (!v_late && !KVS && j + 1 < nit) {
                        load_v(j + 1);
                        ++lv;
                    }
                    if (j + 1 < nit) {
                        wait_g_inputs(j + 1);
                        mma_g(j + 1);
                    }
                }
            }
            // drain (bounded, ignoring the abort flag) so that nothing is in flight at exit
            volatile int never = 0;
            tc::mbar_wait(&bars[la::BSU], (nit - 1) & 1, &never, nullptr, 0);
            if (NSUM) tc::mbar_wait(&bars[la::BN], (nit - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[la::FQ], (lx - 1) & 1, &never, nullptr, 0);
            tc::mbar_wait(&bars[la::FK0], ((lk + 1) / 2 - 1) & 1, &never, nullptr, 0);
            if (lk > 1) tc::mbar_wait(&bars[la::FK1], (lk / 2 - 1) & 1, &never, nullptr, 0);
            if (lv > 0) tc::mbar_wait(&bars[la::FV], (lv - 1) & 1, &never, nullptr, 0);
            tc::bulk_wait_all();
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        const float ginv = g > 0.f ? 1.f / g : 0.f;
        unsigned char* sX = sm + Lay::oQ;
        unsigned char* sV = sm + Lay::oV;

        // ---- EPI-1(j): G~ (and G~2), fX -> tensor memory;  K~ (and V~) -> shared memory ------------
        auto epi1 = [&](int j) {
            const int c = chunk_of(j);
            const int Wc = min(kW, a.n - c * kW);
            const bool live = r < Wc;
            unsigned char* sK = sm + Lay::key(j);
            tc::mbar_wait(&bars[la::FQ], j & 1, abort, status, 111);
            tc::mbar_wait(fk(j), (j >> 1) & 1, abort, status, 112);
            if (R2) tc::mbar_wait(&bars[la::FV], j & 1, abort, status, 113);
            tc::mbar_wait(&bars[la::BG], j & 1, abort, status, 114);
            tc::fence_after_sync();
#pragma unroll
            for (int gi = 0; gi < (R2 ? 2 : 1); ++gi) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int cb = 64 * h + 32 * p;
                    uint32_t pk[16];
                    la_masked_pack<REV>(lrow + C::TG(j) + 128 * gi + cb, r, cb, row0, log2g, g, ginv, pk);
                    tc::tmem_st16(lrow + C::TA + 64 * gi + cb / 2, pk);
                }
            }
            const float f = live ? (REV ? gp[Wc - r] : gp[r + 1]) : 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 x = la_scale_chunk(*reinterpret_cast<const uint4*>(sX + la_off(h, r, 4 * half + i)), f);
                    pk[4 * i] = x.x, pk[4 * i + 1] = x.y, pk[4 * i + 2] = x.z, pk[4 * i + 3] = x.w;
                }
                tc::tmem_st16(lrow + C::TX + 32 * h + 16 * half, pk);
            }
            const float w = live ? (REV ? gp[r] : gp[Wc - 1 - r]) : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t off = la_off(h, r, i);
                *reinterpret_cast<uint4*>(sm + Lay::oKt + off) = la_scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w);
                if (R2)
                    *reinterpret_cast<uint4*>(sm + Lay::oKt2 + off) =
                        la_scale_chunk(*reinterpret_cast<const uint4*>(sV + off), w);
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[la::BGT]);
        };

        // ---- EPI-S(j): Sig <- g^Wc Sig + dSig;  bf16 Sig0 for chunk j + 1 ---------------------------
        auto epis = [&](int j) {
            const int c = chunk_of(j);
            const int Wc = min(kW, a.n - c * kW);
            tc::mbar_wait(bsu(j), bsu_par(j), abort, status, 115);  // chunk j's products are done
            tc::fence_after_sync();
            const float rho = gp[Wc];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t v[16];
                tc::tmem_ld16(lrow + C::TS + 64 * h + 16 * p, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) sig[16 * p + i] = rho * sig[16 * p + i] + __uint_as_float(v[i]);
            }
            if (j + 1 < nit) publish_sig();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[la::BS]);
        };

        // ---- EPI-Y(j): Y (+ partial) -> bf16 output tile;  next summary's values scaled -------------
        auto epiy = [&](int j) {
            const int c = chunk_of(j);
            const int Wc = min(kW, a.n - c * kW);
            const bool live = r < Wc;
            if (j > 0) tc::mbar_wait(&bars[la::BSF], (j - 1) & 1, abort, status, 116);  // previous tile read
            if (ADD || (NSUM && XVS)) tc::mbar_wait(&bars[la::FV], j & 1, abort, status, 117);
            tc::fence_after_sync();
#pragma unroll
            for (int p = 0; p < 4; ++p) {  // 16 columns = 2 chunks of the tile at a time
                uint32_t v[16];
                tc::tmem_ld16(lrow + C::TG(j) + 64 * h + 16 * p, v);
                tc::tmem_wait_ld();
                float y[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) y[i] = __uint_as_float(v[i]);
                if (ADD) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 x = *reinterpret_cast<const uint4*>(sm + Lay::oAD + la_off(h, r, 2 * p + i));
                        y[8 * i + 0] += la_bf_lo(x.x), y[8 * i + 1] += la_bf_hi(x.x);
                        y[8 * i + 2] += la_bf_lo(x.y), y[8 * i + 3] += la_bf_hi(x.y);
                        y[8 * i + 4] += la_bf_lo(x.z), y[8 * i + 5] += la_bf_hi(x.z);
                        y[8 * i + 6] += la_bf_lo(x.w), y[8 * i + 7] += la_bf_hi(x.w);
                    }
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    *reinterpret_cast<uint4*>(sm + Lay::oST + la_off(h, r, 2 * p + i)) = la_pack8(&y[8 * i]);
            }
            if (NSUM) {
                const int pos = (c - sg.c_begin) * kW + r;  // token position in the segment
                const float wn = live ? pow_decay(log2gn, (float)(REV ? pos : sg.L - 1 - pos)) : 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t off = la_off(h, r, i);
                    *reinterpret_cast<uint4*>(sm + Lay::oXV + off) =
                        la_scale_chunk(*reinterpret_cast<const uint4*>(sm + Lay::oXV + off), wn);
                }
            }
            tc::tmem_wait_ld();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[la::BYT]);
        };

        if (nit > 0) epi1(0);
        for (int j = 0; j < nit; ++j) {
            epis(j);
            if (kTwoG) {
                if (j + 1 < nit) epi1(j + 1);
                epiy(j);
            } else {
                epiy(j);
                if (j + 1 < nit) epi1(j + 1);
            }
        }
        if (NSUM && nit > 0 && HLA2_IN(bh < a.BH && seg < a.nseg, 802)) {  // the segment's next summary (fp32)
            tc::mbar_wait(&bars[la::BN], (nit - 1) & 1, abort, status, 118);
            tc::fence_after_sync();
            float* dst = a.summary + ((size_t)bh * a.nseg + seg) * la::kD * la::kD + (size_t)r * la::kD + 64 * h;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t v[32];
                tc::tmem_ld32(lrow + C::TN + 64 * h + 32 * p, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(dst + 32 * p + i) =
                        make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                    __uint_as_float(v[i + 3]));
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, la::kTmemCols);
}

// ----------------------------------------------------------------------------------------
// Summary kernel: Sig_B[s] = sum_{i in s} w_i k_i v_i^T, w_i = g^(t1-1-i) (forward, decayed
// to the segment's end) or g^(i-t0) (reverse, to its start).  Three stages of tiles (loads run
// three chunks ahead); per chunk the epilogue scales K into K~ (in place, unless the keys are
// also the values) and the control thread accumulates K~^T V in tensor memory.
namespace las {
constexpr int kStages = 3;
template <bool KVS>
struct Layout {
    static constexpr uint32_t oK = 0;                                       // kStages stages
    static constexpr uint32_t oV = KVS ? oK : oK + kStages * la::kTile;     // kStages stages
    static constexpr uint32_t oKt = KVS ? oK + kStages * la::kTile : oK;    // KVS: its own stages
    static constexpr uint32_t oBar = (KVS ? oKt : oV) + kStages * la::kTile;
    static constexpr uint32_t oMisc = oBar + 16 * 8;
    static constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
};
enum Bar { F0 = 0, T0 = F0 + kStages, N0 = T0 + kStages, kBarCount = N0 + kStages };
}  // namespace las

template <bool REV, bool KVS>
__global__ void __launch_bounds__(la::kThreads, 1)
    fo_sum_tc_kernel(const __grid_constant__ la::Maps maps, const FoArgs a) {
    using Lay = las::Layout<KVS>;
    constexpr int kW = la::kW;
    pdl_trigger();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Lay::oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::oMisc + 4);
    int* status = a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const FoSeg sg = la_seg(a, seg);
    const int nit = sg.nit;
    const float log2g = (float)a.pow * log2f(head_decay(a.gamma, bh, a.H));

    if (tid == 0) {
        for (int b = 0; b < las::kBarCount; ++b) tc::mbar_init(&bars[b], (b >= las::T0 && b < las::N0) ? 8 : 1);
        *abort = 0;
        tc::mbar_fence_init();
    }
    pdl_wait();
    if (warp == 0) tc::tmem_alloc(tmem_holder, 128);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    auto chunk_of = [&](int it) { return REV ? sg.c_end - 1 - it : sg.c_begin + it; };

    if (warp == 0) {
        if (lane == 0 && nit > 0) {
            auto load = [&](int it) {
                const int s = it % las::kStages, c = chunk_of(it);
                uint64_t* bar = &bars[las::F0 + s];
                tc::mbar_arrive_expect_tx(bar, (KVS ? 1 : 2) * la::kTile);
                const uint32_t ok = Lay::oK + s * la::kTile, ov = Lay::oV + s * la::kTile;
                tc::tma_load_3d(sm + ok, &maps.k, 0, c * kW, bh, bar);
                tc::tma_load_3d(sm + ok + la::kBlk, &maps.k, 64, c * kW, bh, bar);
                if (!KVS) {
                    tc::tma_load_3d(sm + ov, &maps.v, 0, c * kW, bh, bar);
                    tc::tma_load_3d(sm + ov + la::kBlk, &maps.v, 64, c * kW, bh, bar);
                }
            };
            constexpr uint32_t I_MM = tc::idesc_bf16(128, 128, 1, 1);
            auto mdesc = [](uint32_t base, int ks) { return tc::smem_desc(base + 2048u * ks, la::kBlk, 1024); };
            for (int it = 0; it < las::kStages && it < nit; ++it) load(it);
            for (int it = 0; it < nit; ++it) {
                const int s = it % las::kStages;
                const uint32_t ph = (it / las::kStages) & 1;
                tc::mbar_wait(&bars[las::T0 + s], ph, abort, status, 121);  // K~ of this chunk written
                tc::fence_after_sync();
                const uint32_t sKt = smem_u32(sm + Lay::oKt + s * la::kTile);
                const uint32_t sV = smem_u32(sm + Lay::oV + s * la::kTile);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem, mdesc(sKt, ks), mdesc(sV, ks), I_MM, (it > 0 || ks > 0) ? 1u : 0u);
                tc::mma_commit(&bars[las::N0 + s]);
                if (it + las::kStages < nit) {  // this stage's tiles are free once its product has run
                    tc::mbar_wait(&bars[las::N0 + s], ph, abort, status, 122);
                    load(it + las::kStages);
                }
            }
            volatile int never = 0;  // the products not yet waited for (the last kStages chunks)
            for (int it = nit - las::kStages < 0 ? 0 : nit - las::kStages; it < nit; ++it)
                tc::mbar_wait(&bars[las::N0 + it % las::kStages], (it / las::kStages) & 1, &never, nullptr, 0);
        }
        __syncwarp();
    } else {
        const int q4 = warp & 3, h = (warp - 1) >> 2;
        const int r = 32 * q4 + lane;
        const uint32_t lrow = tmem + ((uint32_t)(32 * q4) << 16);
        for (int it = 0; it < nit; ++it) {
            const int s = it % las::kStages;
            const uint32_t ph = (it / las::kStages) & 1;
            const int c = chunk_of(it);
            const int Wc = min(kW, a.n - c * kW);
            tc::mbar_wait(&bars[las::F0 + s], ph, abort, status, 123);
            const int pos = (c - sg.c_begin) * kW + r;
            const float w = r < Wc ? pow_decay(log2g, (float)(REV ? pos : sg.L - 1 - pos)) : 0.f;
            unsigned char* sK = sm + Lay::oK + s * la::kTile;
            unsigned char* sKt = sm + Lay::oKt + s * la::kTile;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t off = la_off(h, r, j);
                *reinterpret_cast<uint4*>(sKt + off) = la_scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w);
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[las::T0 + s]);
        }
        if (nit > 0 && HLA2_IN(bh < a.BH && seg < a.nseg, 803)) {
            tc::mbar_wait(&bars[las::N0 + (nit - 1) % las::kStages], ((nit - 1) / las::kStages) & 1, abort, status,
                          124);
            tc::fence_after_sync();
            float* dst = a.summary + ((size_t)bh * a.nseg + seg) * la::kD * la::kD + (size_t)r * la::kD + 64 * h;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t v[32];
                tc::tmem_ld32(lrow + 64 * h + 32 * p, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(dst + 32 * p + j) =
                        make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                    __uint_as_float(v[j + 3]));
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// Final-state summaries in one pass over (q, p, v): per segment
//   C_B = sum_i w_i q_i v_i^T,  Z_B = sum_i w_i^2 p_i v_i^T,  m_B = sum_i w_i q_i,  y_B = sum_i w_i^2 p_i,
// with w_i = g^(t1-1-i) (decayed to the segment's end).  Two stages of (q, p, v) tiles; per chunk
// the epilogue scales q by w and p by w^2 in place and keeps the moments' partial sums, and the
// control thread accumulates Q~^T V (tensor-memory columns [0, 128)) and P~^T V ([128, 256)).
// Epilogue thread e owns the 8-column group 8 (e % 16) .. of rows e / 16 + 16 i (i < 8).
namespace las2 {
constexpr uint32_t oQ = 0, oP = 2 * la::kTile, oV = 4 * la::kTile;  // 2 stages each
constexpr uint32_t oRed = 6 * la::kTile;                             // moment partials [2][16][128] fp32
constexpr uint32_t oBar = oRed + 2 * 16 * 128 * 4;
constexpr uint32_t oMisc = oBar + 16 * 8;
constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
}  // namespace las2

__global__ void __launch_bounds__(la::kThreads, 1)
    fo_sum_final_tc_kernel(const __grid_constant__ la::Maps maps, const FoArgs a, float* zsum, float* msum,
                           float* ysum) {
    using namespace las2;
    constexpr int kW = la::kW, kD = la::kD;
    pdl_trigger();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + oMisc + 4);
    float* red = reinterpret_cast<float*>(sm + oRed);
    int* status = a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const FoSeg sg = la_seg(a, seg);
    const int nit = sg.nit;
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));

    if (tid == 0) {
        for (int b = 0; b < las::kBarCount; ++b) tc::mbar_init(&bars[b], (b >= las::T0 && b < las::N0) ? 8 : 1);
        *abort = 0;
        tc::mbar_fence_init();
    }
    pdl_wait();
    if (warp == 0) tc::tmem_alloc(tmem_holder, 256);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0 && nit > 0) {
            auto load = [&](int it) {
                const int s = it & 1, c = sg.c_begin + it;
                uint64_t* bar = &bars[las::F0 + s];
                tc::mbar_arrive_expect_tx(bar, 3 * la::kTile);
                const uint32_t o = s * la::kTile;
                tc::tma_load_3d(sm + oQ + o, &maps.x, 0, c * kW, bh, bar);
                tc::tma_load_3d(sm + oQ + o + la::kBlk, &maps.x, 64, c * kW, bh, bar);
                tc::tma_load_3d(sm + oP + o, &maps.k, 0, c * kW, bh, bar);
                tc::tma_load_3d(sm + oP + o + la::kBlk, &maps.k, 64, c * kW, bh, bar);
                tc::tma_load_3d(sm + oV + o, &maps.v, 0, c * kW, bh, bar);
                tc::tma_load_3d(sm + oV + o + la::kBlk, &maps.v, 64, c * kW, bh, bar);
            };
            constexpr uint32_t I_MM = tc::idesc_bf16(128, 128, 1, 1);
            auto mdesc = [](uint32_t base, int ks) { return tc::smem_desc(base + 2048u * ks, la::kBlk, 1024); };
            load(0);
            if (nit > 1) load(1);
            for (int it = 0; it < nit; ++it) {
                const int s = it & 1;
                const uint32_t ph = (it >> 1) & 1;
                tc::mbar_wait(&bars[las::T0 + s], ph, abort, status, 131);  // Q~, P~ of this chunk written
                tc::fence_after_sync();
                const uint32_t o = s * la::kTile;
                const uint32_t sQ = smem_u32(sm + oQ + o), sP = smem_u32(sm + oP + o), sV = smem_u32(sm + oV + o);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem, mdesc(sQ, ks), mdesc(sV, ks), I_MM, (it > 0 || ks > 0) ? 1u : 0u);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + 128, mdesc(sP, ks), mdesc(sV, ks), I_MM, (it > 0 || ks > 0) ? 1u : 0u);
                tc::mma_commit(&bars[las::N0 + s]);
                if (it + 2 < nit) {  // this stage's tiles are free once its products have run
                    tc::mbar_wait(&bars[las::N0 + s], ph, abort, status, 132);
                    load(it + 2);
                }
            }
            volatile int never = 0;
            tc::mbar_wait(&bars[las::N0 + ((nit - 1) & 1)], ((nit - 1) >> 1) & 1, &never, nullptr, 0);
            if (nit > 1) tc::mbar_wait(&bars[las::N0 + ((nit - 2) & 1)], ((nit - 2) >> 1) & 1, &never, nullptr, 0);
        }
        __syncwarp();
    } else {
        const int e = tid - 32, cc = e % 16, b = cc / 8, j = cc % 8, r0 = e / 16;
        float mq[8], yp[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mq[u] = yp[u] = 0.f;
        for (int it = 0; it < nit; ++it) {
            const int s = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const int c = sg.c_begin + it;
            const int Wc = min(kW, a.n - c * kW);
            tc::mbar_wait(&bars[las::F0 + s], ph, abort, status, 133);
            unsigned char* sQ = sm + oQ + s * la::kTile;
            unsigned char* sP = sm + oP + s * la::kTile;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = r0 + 16 * i;
                const int pos = (c - sg.c_begin) * kW + r;
                const float w1 = r < Wc ? pow_decay(log2g, (float)(sg.L - 1 - pos)) : 0.f, w2 = w1 * w1;
                const uint32_t off = la_off(b, r, j);
                const uint4 qc = *reinterpret_cast<const uint4*>(sQ + off);
                const uint4 pc = *reinterpret_cast<const uint4*>(sP + off);
                const uint32_t qw[4] = {qc.x, qc.y, qc.z, qc.w}, pw[4] = {pc.x, pc.y, pc.z, pc.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    mq[2 * u] += w1 * __uint_as_float(qw[u] << 16);
                    mq[2 * u + 1] += w1 * __uint_as_float(qw[u] & 0xFFFF0000u);
                    yp[2 * u] += w2 * __uint_as_float(pw[u] << 16);
                    yp[2 * u + 1] += w2 * __uint_as_float(pw[u] & 0xFFFF0000u);
                }
                *reinterpret_cast<uint4*>(sQ + off) = la_scale_chunk(qc, w1);
                *reinterpret_cast<uint4*>(sP + off) = la_scale_chunk(pc, w2);
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[las::T0 + s]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            red[r0 * kD + 64 * b + 8 * j + u] = mq[u];
            red[16 * kD + r0 * kD + 64 * b + 8 * j + u] = yp[u];
        }
        if (nit > 0 && HLA2_IN(bh < a.BH && seg < a.nseg, 805)) {  // C_B and Z_B rows of this warp's lanes
            const int q4 = warp & 3, h = (warp - 1) >> 2;
            const int r = 32 * q4 + lane;
            const uint32_t lrow = tmem + ((uint32_t)(32 * q4) << 16);
            tc::mbar_wait(&bars[las::N0 + ((nit - 1) & 1)], ((nit - 1) >> 1) & 1, abort, status, 134);
            tc::fence_after_sync();
            const size_t si = (size_t)bh * a.nseg + seg;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float* dst = (part ? zsum : a.summary) + si * kD * kD + (size_t)r * kD + 64 * h;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint32_t v[32];
                    tc::tmem_ld32(lrow + 128 * part + 64 * h + 32 * p, v);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + 32 * p + i) =
                            make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                        __uint_as_float(v[i + 3]));
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid < 2 * kD && HLA2_IN(bh < a.BH && seg < a.nseg, 806)) {  // moments: the 16 row groups in a fixed order
        const int part = tid / kD, col = tid % kD;
        float t = 0.f;
        for (int g = 0; g < 16; ++g) t += red[part * 16 * kD + g * kD + col];
        (part ? ysum : msum)[((size_t)bh * a.nseg + seg) * kD + col] = t;
    }
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// Zeroes the carry into segment 0 of every head ([BH][nseg][E], segment 0; E = d * d) and
// clears the status word, before a forward linear scan fills the other segments.
__global__ void fo_zero_first_kernel(float* carry, int nseg, int E, int BH, int* status) {
    pdl_trigger();
    pdl_wait();
    const int bh = blockIdx.x;
    if (!HLA2_IN(bh < BH && E % 4 == 0, 804)) return;
    float4* dst = reinterpret_cast<float4*>(carry + (size_t)bh * nseg * E);
    for (int i = threadIdx.x; i < E / 4; i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (bh == 0 && threadIdx.x == 0 && status) *status = 0;
}

template <typename K>
int la_launch(K kfn, uint32_t smem, const la::Maps& maps, const FoArgs& a, cudaStream_t st,
              int threads = la::kThreads) {
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -1;
    if (launch_pdl(kfn, dim3(a.nseg, a.BH), dim3(threads), smem, st, maps, a) != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

bool fo_tc_available() { return la_encode_fn() != nullptr; }

// The largest shared-memory plan among the instantiated output kernels (and the summary kernels).
size_t fo_tc_max_smem() {
    const uint32_t sizes[] = {la::OutLayout<false, true, true, false>::kSmemBytes,    // p
                              la::OutLayout<false, false, false, false>::kSmemBytes,  // o, Z dO, dv
                              la::OutLayout<true, false, false, false>::kSmemBytes,   // dk
                              la::OutLayout<false, true, false, true>::kSmemBytes,    // dq
                              las::Layout<false>::kSmemBytes, las::Layout<true>::kSmemBytes, las2::kSmemBytes};
    uint32_t m = 0;
    for (uint32_t x : sizes) m = x > m ? x : m;
    return m;
}

int launch_fo_zero_first(float* carry, int BH, int nseg, int E, int* status, cudaStream_t st) {
    if (BH <= 0) return 0;
    if (launch_pdl(fo_zero_first_kernel, dim3(BH), dim3(256), 0, st, carry, nseg, E, BH, status) != cudaSuccess)
        return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_fo_tc_summary_final(const FoArgs& a, const void* q, const void* p, const void* v, float* zsum,
                               float* msum, float* ysum, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    if (!a.summary || !zsum || !msum || !ysum) return -2;
    la::Maps m{};
    if (!la_map(&m.x, q, a.BH, a.n) || !la_map(&m.k, p, a.BH, a.n) || !la_map(&m.v, v, a.BH, a.n)) return -2;
    if (cudaFuncSetAttribute(fo_sum_final_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)las2::kSmemBytes) != cudaSuccess)
        return -1;
    if (launch_pdl(fo_sum_final_tc_kernel, dim3(a.nseg, a.BH), dim3(la::kThreads), las2::kSmemBytes, st, m, a, zsum,
                   msum, ysum) != cudaSuccess)
        return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_fo_tc_summary(const FoArgs& a, const void* k, const void* v, bool reverse, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    la::Maps m{};
    if (!la_map(&m.k, k, a.BH, a.n) || !la_map(&m.v, v ? v : k, a.BH, a.n)) return -2;
    const bool kvs = !v || v == k;
    if (kvs)
        return reverse ? la_launch(fo_sum_tc_kernel<true, true>, las::Layout<true>::kSmemBytes, m, a, st)
                       : la_launch(fo_sum_tc_kernel<false, true>, las::Layout<true>::kSmemBytes, m, a, st);
    return reverse ? la_launch(fo_sum_tc_kernel<true, false>, las::Layout<false>::kSmemBytes, m, a, st)
                   : la_launch(fo_sum_tc_kernel<false, false>, las::Layout<false>::kSmemBytes, m, a, st);
}

// Output launch.  x, k, v: queries, keys, values ([BH][n][128] bf16); v == nullptr: the values
// are the key tile.  r2: the swapped second pair.  next_sum: 0 none, 1 over (out, the value
// tile), 2 over (out, xv).  add: partial added to the output (nullptr: none).
int launch_fo_tc_out(const FoArgs& a, const void* x, const void* k, const void* v, bool r2, int next_sum,
                     const void* xv, const void* add, void* out, bool reverse, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    la::Maps m{};
    const bool kvs = v == nullptr, nsum = next_sum != 0, xvs = next_sum == 2, addp = add != nullptr;
    if (!la_map(&m.x, x, a.BH, a.n) || !la_map(&m.k, k, a.BH, a.n) || !la_map(&m.v, kvs ? k : v, a.BH, a.n) ||
        !la_map(&m.out, out, a.BH, a.n))
        return -2;
    if (xvs && !la_map(&m.xv, xv, a.BH, a.n)) return -2;
    if (addp && !la_map(&m.ad, add, a.BH, a.n)) return -2;
    if (nsum && !a.summary) return -2;
#define HLA2_LA(REV, NSUM, R2, KVS, XVS, ADD)                                                               \
    if (reverse == REV && nsum == NSUM && r2 == R2 && kvs == KVS && xvs == XVS && addp == ADD)             \
        return la_launch(fo_out_tc_kernel<REV, NSUM, R2, KVS, XVS, ADD>,                                      \
                         la::OutLayout<R2, KVS, XVS, ADD>::kSmemBytes, m, a, st, la::kThreadsOut);
    // the passes of the d = 128 training path
    HLA2_LA(false, true, false, true, true, false)    // p = LA(q, k, k), next summary over (p, v)
    HLA2_LA(false, false, false, true, false, false)   // p = LA(q, k, k) (the summary over (p, v) apart)
    HLA2_LA(false, false, false, false, false, false) // o = LA(q, p, v);  dq_a = LA(dO, v, p)
    HLA2_LA(true, true, false, false, false, false)   // dp = RLA(v, dO, q), next summary over (dp, q)
    HLA2_LA(true, false, false, false, false, false)  // dv = RLA(p, q, dO)
    HLA2_LA(true, false, true, false, false, false)   // dk = RLA(k, dp, q) + RLA(k, q, dp)
    HLA2_LA(false, false, false, true, false, true)   // dq = LA(dp, k, k) + dq_a
#undef HLA2_LA
    return -3;  // combination not instantiated
}

}  // namespace hla2

HLA2_DEBUG_READER(fo_tc)
