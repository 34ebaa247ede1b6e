// gdn_k1_contract.cuh -- phase 1 of the frame-wise GDN forward.
//
// For every (batch b, latent frame f, head h) -- one "item" -- the two
// frame-parallel contractions of the delta rule
//     A_f = K_f^T B_f K_f = sum_n beta_n k_n k_n^T      (dk x dk)
//     U_f = V_f^T B_f K_f = sum_n beta_n v_n k_n^T      (dv x dk)
// (SANA-WM article, "The Architecture": the state is updated once per latent
// frame by a decay gate and a delta-rule correction; these two matrices are
// everything the frame contributes to that update).
//
// Formulation on the tensor core: one MMA  D = (B K)^T [K | V]  with
//     M = 128   rows j of (beta k)^T      (dk, zero-padded to 128)
//     N = 256   columns [k (128) | v (128)]
//     K = tokens, 16 per instruction, 64 per pipeline stage
// so that TMEM lane j holds row j of A (columns 0..127) and column j of U
// (columns 128..255).  Both operands are read straight from the TMA tiles
// of q/k/v's natural token-major layout, i.e. MN-major in the MMA's terms.
// beta is applied in fp32 to a copy of the K tile (rounded to bf16 once).
//
// Warp roles (320 threads): warp 0 TMA producer; warp 1 TMEM owner and MMA
// issuer; warps 2-5 beta scalers (two adjacent lanes per token row); warps
// 6-9 epilogue (TMEM lane quarter = warp % 4).  The K/V tiles stream through a
// 5-deep TMA ring; the scaled copy of K has its own 3-deep ring, so a K/V slot
// is released as soon as its MMAs retire.  beta reaches the scalers through a
// small per-thread shared-memory ring filled by cp.async four chunks ahead.
// TMEM holds two 256-column accumulators so one item's epilogue overlaps the
// next item's MMAs.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace k1 {

#ifndef GDN_K1_STAGES
#define GDN_K1_STAGES 5
#endif
#ifndef GDN_K1_BK_BUFS
#define GDN_K1_BK_BUFS 3
#endif
#ifndef GDN_K1_SCALER_WARPS
#define GDN_K1_SCALER_WARPS 4
#endif
#ifndef GDN_K1_CHUNK
#define GDN_K1_CHUNK 64
#endif
constexpr int CHUNK = GDN_K1_CHUNK;         // tokens per stage (MMA K extent per stage)
constexpr int STAGES = GDN_K1_STAGES;       // K/V ring depth
constexpr int BK_BUFS = GDN_K1_BK_BUFS;     // beta*K buffers
constexpr int BOX_BYTES = CHUNK * 128;      // 64 token rows x 128 B (64 bf16)
constexpr int TILE_BYTES = 2 * BOX_BYTES;   // d padded to 128 -> two 64-column boxes
constexpr int STAGE_BYTES = 2 * TILE_BYTES; // K tile, V tile
constexpr int SCALER_WARPS = GDN_K1_SCALER_WARPS;
constexpr int SCALER_THREADS = SCALER_WARPS * 32;
constexpr int EPI_WARP0 = 2 + SCALER_WARPS;  // four epilogue warps follow the scalers
constexpr int THREADS = (EPI_WARP0 + 4) * 32;
// a pair of adjacent scaler lanes owns one token row (one 64-column box each)
static_assert(SCALER_THREADS == 2 * CHUNK, "two scaler threads per token row");
// beta is copied global -> shared by each scaler thread BETA_AHEAD chunks before
// its use, into a per-thread ring of BETA_AHEAD + 1 slots
constexpr int BETA_AHEAD = 4;
constexpr int BETA_RING_BYTES = (BETA_AHEAD + 1) * SCALER_THREADS * 4;
static_assert(1024 + STAGES * STAGE_BYTES + BK_BUFS * TILE_BYTES + BETA_RING_BYTES + 256 <= 232448, "shared memory");
constexpr int TMEM_COLS = 512;
constexpr int ACC_COLS = 256;
// MN-major operand with 128-byte swizzle: 64 MN-elements per 128-byte row,
// 8 K-rows per 1024-byte swizzle atom.  LBO = distance between 64-element
// MN blocks (the two 64-column TMA boxes), SBO = distance between 8-row K
// groups.
constexpr uint32_t MN_LBO = BOX_BYTES;
constexpr uint32_t MN_SBO = 1024;
// fp8 (e4m3) k and v: one 128-byte box (128 columns, zero-filled past d) per
// token row and input, STAGES8-deep.  The scalers decode each stage into one
// f16 buffer [sqrt(beta) K | sqrt(beta) V] and the MMA (kind::f16, f16
// operands) reads it as both operands,
//     D = (sqrt(B) K)^T [sqrt(B) K | sqrt(B) V] = [K^T B K | (V^T B K)^T],
// which writes a third less shared memory than separate beta*K, K and V
// copies (the fp8 path is bound by shared-memory traffic, not HBM).  e4m3 ->
// f16 is exact (one conversion per pair); the sqrt(beta) product is formed in
// f16 arithmetic, so beta must lie in [0, FP8_BETA_MAX] (sqrt(beta) * 448 below
// the f16 maximum); anything else is reported as GDN_ERR_RANGE.
constexpr int STAGES8 = 7;
constexpr int BOX8_BYTES = CHUNK * 128;        // 64 token rows x 128 fp8
constexpr int STAGE8_BYTES = 2 * BOX8_BYTES;   // K, V
constexpr int CBUFS8 = 3;
constexpr int CBUF8_BYTES = 2 * TILE_BYTES;    // sqrt(beta) K | sqrt(beta) V, f16
constexpr float FP8_BETA_MAX = 16384.0f;
// NVFP4 k and v: one box of d/2 bytes (64 codes of a 128-column row: at most
// 64 bytes, d = 64 or 128) per token row and input, unswizzled, STAGES4-deep;
// their E4M3 block scales (d/16 per row) reach the decoders like beta, by
// cp.async a few chunks ahead.  The decoders form e2m1 * scale exactly in
// f16, then scale by sqrt(beta) like the 8-bit path; with values up to
// 6 * 448 = 2688, beta must lie in [0, FP4_BETA_MAX] for sqrt(beta) * 2688 to
// stay below the f16 maximum.
constexpr int STAGES4 = 8;
constexpr int RAW4_BYTES = CHUNK * 64;          // 64 token rows x up to 64 B
constexpr int STAGE4_BYTES = 2 * RAW4_BYTES;    // K, V
constexpr float FP4_BETA_MAX = 512.0f;
constexpr int SF_RING_BYTES = (BETA_AHEAD + 1) * SCALER_THREADS * 8;   // two scale words per thread
template <int FMT>
struct Lay {
    static constexpr int NST = FMT == FMT_FP8 ? STAGES8 : FMT == FMT_FP4 ? STAGES4 : STAGES;   // TMA ring slots
    static constexpr int ST_BYTES = FMT == FMT_FP8 ? STAGE8_BYTES : FMT == FMT_FP4 ? STAGE4_BYTES : STAGE_BYTES;
    static constexpr int NBK = FMT != FMT_BF16 ? CBUFS8 : BK_BUFS;              // MMA operand buffers
    static constexpr int BK_BYTES = FMT != FMT_BF16 ? CBUF8_BYTES : TILE_BYTES;
    static constexpr int SF_BYTES = FMT == FMT_FP4 ? SF_RING_BYTES : 0;
    static constexpr size_t SMEM =
        1024 /*align slack*/ + NST * ST_BYTES + NBK * BK_BYTES + BETA_RING_BYTES + SF_BYTES + 256 /*barriers*/;
    static_assert(SMEM <= 232448, "shared memory");
    static_assert((2 * NST + 2 * NBK + 5) * 8 + 8 <= 256, "barrier area");
};
constexpr size_t SMEM_BYTES = Lay<FMT_BF16>::SMEM;
constexpr size_t SMEM_BYTES_FP8 = Lay<FMT_FP8>::SMEM;
constexpr size_t SMEM_BYTES_FP4 = Lay<FMT_FP4>::SMEM;

struct Params {
    const float* beta;     // [B, F, N, H]
    __nv_bfloat16* A_ws;   // [items][dk][dk]
    float* U_ws;           // [items][dv][dk]
    float* partial;        // [items - whole][split_per][dk*dk + dv*dk] fp32 partial sums
    int* counters;         // [items - whole] finished splits per split item (zero on entry)
    int H, N, dk, dv;
    int items;             // B * F * H, item = (b*F + f)*H + h
    int whole;             // items 0..whole-1 are processed whole (full rounds of the grid)
    int split_per;         // each remaining item is split into this many token ranges
    int chunks;            // ceil(N / CHUNK)
    int work;              // whole + (items - whole) * split_per
    int norm_k;            // fused prologue: k <- k / max(|k|, 1e-12) per (token, head)
    int beta_sigmoid;      // fused prologue: beta <- sigmoid(beta)
    float a_scale;         // A = a_scale * D[:, :dk]  (fp8 inputs: k_scale^2; else 1)
    float u_scale;         // U = u_scale * D[:, 128:] (fp8 inputs: k_scale * v_scale; else 1)
    const uint8_t* k_sf;   // NVFP4: E4M3 block scales of k [B, F, N, H, dk/16]
    const uint8_t* v_sf;   //        and of v [B, F, N, H, dv/16]
    // Ring mode (single-pass forward; 0 = off): units are whole items in scan
    // order -- step s of the scan (frame s, or F-1-s when reversed) for every
    // (b, h) -- and A_f, U_f go to ring slot (b * ring + s % ring) * H + h of
    // A_ws / U_ws instead of the item's own place, as whole zero-padded ring
    // tiles (RING_TILE_BF16 / RING_TILE_F32 bytes, the swizzled layout of
    // ring_off in gdn_ptx.cuh).  Before a slot is
    // rewritten the scan must have read its previous frame (au_free counts
    // frames read per slot); after the stores au_ready counts one more frame.
    int ring;
    int B, F, reverse;
    int* au_ready;
    const int* au_free;
    unsigned long long wait_limit_ns;
};

// x * s on packed bf16 pairs with s = hi + lo split into two bf16: fma(x, hi, x*lo)
// rounds the product essentially once, like an fp32 product rounded to bf16
struct BSplit {
    __nv_bfloat162 hi, lo;
};
__device__ __forceinline__ BSplit bsplit(float s) {
    const __nv_bfloat16 h = __float2bfloat16_rn(s);
    const __nv_bfloat16 l = __float2bfloat16_rn(s - __bfloat162float(h));
    return BSplit{__halves2bfloat162(h, h), __halves2bfloat162(l, l)};
}
__device__ __forceinline__ uint4 bscale(uint4 x, const BSplit& s) {
    uint32_t* xs = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 k2 = *reinterpret_cast<const __nv_bfloat162*>(&xs[e]);
        const __nv_bfloat162 r2 = __hfma2(k2, s.hi, __hmul2(k2, s.lo));
        xs[e] = *reinterpret_cast<const uint32_t*>(&r2);
    }
    return x;
}

// The same split product on packed f16 pairs (fp8 inputs).
struct HSplit {
    __half2 hi, lo;
};
__device__ __forceinline__ HSplit hsplit(float s) {
    const __half h = __float2half_rn(s);
    const __half l = __float2half_rn(s - __half2float(h));
    return HSplit{__halves2half2(h, h), __halves2half2(l, l)};
}
__device__ __forceinline__ uint32_t hscale(uint32_t x, const HSplit& s) {
    const __half2 k2 = *reinterpret_cast<const __half2*>(&x);
    const __half2 r2 = __hfma2(k2, s.hi, __hmul2(k2, s.lo));
    return *reinterpret_cast<const uint32_t*>(&r2);
}

// Work units: the first `whole` items whole, then every remaining item split
// into `split_per` contiguous token ranges (so the last round of the grid is
// as long as the others); split == -1 marks a whole item.  In ring mode every
// unit is a whole item in scan order; `slot` is where its A and U go and
// `use` how many frames went through that slot before it.
struct Unit {
    int item, split, c_begin, c_end, slot, use;
};
__device__ __forceinline__ Unit unit_of(const Params& p, int w) {
    Unit u;
    if (p.ring > 0) {
        const int BH = p.B * p.H;
        const int st = w / BH, r = w % BH, b = r / p.H, h = r % p.H;
        const int f = p.reverse ? p.F - 1 - st : st;
        u.item = (b * p.F + f) * p.H + h;
        u.split = -1;
        u.c_begin = 0;
        u.c_end = p.chunks;
        u.slot = (b * p.ring + st % p.ring) * p.H + h;
        u.use = st / p.ring;
        return u;
    }
    u.slot = -1;
    u.use = 0;
    if (w < p.whole) {
        u.item = w;
        u.split = -1;
        u.c_begin = 0;
        u.c_end = p.chunks;
        return u;
    }
    const int r = w - p.whole;
    u.item = p.whole + r / p.split_per;
    u.split = r % p.split_per;
    u.c_begin = static_cast<int>((static_cast<long long>(u.split) * p.chunks) / p.split_per);
    u.c_end = static_cast<int>((static_cast<long long>(u.split + 1) * p.chunks) / p.split_per);
    return u;
}

// The contraction of work units w_begin, w_begin + w_step, ... < p.work, in
// a block of at least THREADS threads (warps past the epilogue stay idle).
template <int FMT>
__device__ __forceinline__ void contract_role(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const Params& p,
                                              int w_begin, int w_step, uint8_t* smem) {
    constexpr bool FP8 = FMT == FMT_FP8;
    constexpr bool FP4 = FMT == FMT_FP4;
    constexpr bool LP = FMT != FMT_BF16;   // decoded into one f16 operand buffer [sqrt(beta) K | sqrt(beta) V]
    using L = Lay<FMT>;
    constexpr int NST = L::NST, NBK = L::NBK;
    uint8_t* stage_base = smem;                                   // [NST][K tile | V tile]
    uint8_t* bk_base = smem + NST * L::ST_BYTES;                  // [NBK][beta*K tile (| K | V when FP8)]
    float* beta_ring = reinterpret_cast<float*>(bk_base + NBK * L::BK_BYTES);  // [BETA_AHEAD+1][SCALER_THREADS]
    uint32_t* sf_ring = reinterpret_cast<uint32_t*>(bk_base + NBK * L::BK_BYTES + BETA_RING_BYTES);  // FP4: [..][2]
    uint64_t* bars = reinterpret_cast<uint64_t*>(bk_base + NBK * L::BK_BYTES + BETA_RING_BYTES + L::SF_BYTES);
    uint64_t* full = bars;                          // [NST]  TMA landed K and V
    uint64_t* empty = full + NST;                   // [NST]  stage consumed (MMA, or FP8 decoders)
    uint64_t* bk_full = empty + NST;                // [NBK]  MMA operand buffer written
    uint64_t* bk_empty = bk_full + NBK;             // [NBK]  MMA finished reading it
    uint64_t* tfull = bk_empty + NBK;               // [2]       accumulator ready
    uint64_t* tempty = tfull + 2;                   // [2]       accumulator drained
    uint64_t* final_bar = tempty + 2;               // [1]       every issued MMA retired
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // Work units round-robin over the grid: at any time the CTAs work on
    // consecutive items, i.e. all heads of the same few frames, so together
    // they read whole token rows (all heads) of k and v.  The split units come
    // last and number at most gridDim.x, so each CTA holds at most one.
    const int w_end = p.work;
    const int kboxes = p.dk > 64 ? 2 : 1;
    const int vboxes = p.dv > 64 ? 2 : 1;

    // Boxes that are never loaded (d <= 64) must read as 0; with d > 64 every
    // byte is written before it is read.
    // (FP8: the decoders write every byte of every operand buffer.)
    if (!LP && (kboxes < 2 || vboxes < 2))
        for (int i = threadIdx.x; i < (NST * L::ST_BYTES + NBK * L::BK_BYTES) / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], LP ? SCALER_THREADS : 1);
        }
        for (int b = 0; b < NBK; ++b) {
            mbar_init(&bk_full[b], SCALER_THREADS);
            mbar_init(&bk_empty[b], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            for (int w = w_begin; w < w_end && !*abort_flag; w += w_step) {
                const Unit u = unit_of(p, w);
                const int frame = u.item / p.H, h = u.item % p.H;
                for (int c = u.c_begin; c < u.c_end; ++c) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_limit_ns, abort_flag)) break;
                    uint8_t* st = stage_base + stage * L::ST_BYTES;
                    if constexpr (FP8) {
                        mbar_arrive_expect_tx(&full[stage], STAGE8_BYTES);
                        tma_load_4d(st, &tm_k, &full[stage], 0, h, c * CHUNK, frame);
                        tma_load_4d(st + BOX8_BYTES, &tm_v, &full[stage], 0, h, c * CHUNK, frame);
                    } else if constexpr (FP4) {
                        mbar_arrive_expect_tx(&full[stage], CHUNK * (p.dk / 2 + p.dv / 2));
                        tma_load_4d(st, &tm_k, &full[stage], 0, h, c * CHUNK, frame);
                        tma_load_4d(st + RAW4_BYTES, &tm_v, &full[stage], 0, h, c * CHUNK, frame);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], (kboxes + vboxes) * BOX_BYTES);
                        for (int bx = 0; bx < kboxes; ++bx)
                            tma_load_4d(st + bx * BOX_BYTES, &tm_k, &full[stage], 64 * bx, h, c * CHUNK, frame);
                        for (int bx = 0; bx < vboxes; ++bx)
                            tma_load_4d(st + TILE_BYTES + bx * BOX_BYTES, &tm_v, &full[stage], 64 * bx, h,
                                        c * CHUNK, frame);
                    }
                    ++issued;
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
            }
            // Drain: the most recent fill of every stage must have landed before exit
            // (only matters when a wait gave up; otherwise the MMA issuer consumed all).
            for (long long kf = (issued > NST ? issued - NST : 0); kf < issued; ++kf)
                mbar_wait_drain(&full[kf % NST], static_cast<uint32_t>((kf / NST) & 1), p.wait_limit_ns);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = LP ? idesc_f16(128, 256, 1, 1) : idesc_bf16(128, 256, 1, 1);
            int stage = 0, bk = 0;
            uint32_t phase = 0, bk_phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int w = w_begin; w < w_end && !*abort_flag; w += w_step) {
                const Unit u = unit_of(p, w);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.wait_limit_ns, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                bool ok = true;
                for (int c = u.c_begin; c < u.c_end; ++c) {
                    if ((!LP && !mbar_wait(&full[stage], phase, p.wait_limit_ns, abort_flag)) ||
                        !mbar_wait(&bk_full[bk], bk_phase, p.wait_limit_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // A = beta*K (FP8: sqrt(beta) K); B = [K | V] from the TMA stage, or (FP8)
                    // [sqrt(beta) K | sqrt(beta) V], the same buffer as A
                    const uint32_t a_base = smem_u32(bk_base + bk * L::BK_BYTES);
                    const uint32_t b_base = LP ? a_base : smem_u32(stage_base + stage * L::ST_BYTES);
#pragma unroll
                    for (int kk = 0; kk < CHUNK / 16; ++kk) {
                        const uint64_t ad = smem_desc(a_base + kk * 2048, MN_LBO, MN_SBO);
                        const uint64_t bd = smem_desc(b_base + kk * 2048, MN_LBO, MN_SBO);
                        mma_bf16(d_tmem, ad, bd, IDESC, (c > u.c_begin || kk > 0) ? 1u : 0u);
                    }
                    if (!LP) mma_commit(&empty[stage]);
                    mma_commit(&bk_empty[bk]);
                    if (++bk == NBK) { bk = 0; bk_phase ^= 1; }
                    if (++stage == NST) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            mma_commit(final_bar);
            mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
        }
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------ beta scalers
        const int t = threadIdx.x - 64;     // 0..SCALER_THREADS-1
        const int r = t >> 1;               // token row within the stage
        const int bx = t & 1;               // which 64-column box of the row
        // beta is copied to shared memory BETA_AHEAD chunks ahead of its use (a
        // cursor walks the same unit/chunk sequence), so its global-load
        // latency never sits between a landed K tile and its MMA.  Each thread
        // reads back only the values it copied itself.  The cursor's unit and
        // the row of its first token are computed once per unit: the integer
        // divisions of unit_of, done per chunk by these four warps, had cost
        // the contraction a third of its speed.
        int pw = w_begin, pc = 0;
        Unit pu{};
        size_t prow0 = 0;   // beta row of token 0 of the cursor's item
        auto enter_unit = [&]() {
            pu = unit_of(p, pw);
            prow0 = static_cast<size_t>(pu.item / p.H) * p.N * p.H + (pu.item % p.H);
            pc = pu.c_begin;
        };
        if (pw < w_end) enter_unit();
        int pslot = 0;
        auto beta_prefetch = [&]() {
            float* dst = beta_ring + pslot * SCALER_THREADS + t;
            uint32_t* sdst = sf_ring + (pslot * SCALER_THREADS + t) * 2;
            if (pw < w_end) {
                const int tok = pc * CHUNK + r;
                const size_t row = prow0 + static_cast<size_t>(tok) * p.H;
                if (tok < p.N)
                    cp_async_4(dst, p.beta + row);
                else
                    *dst = 0.0f;
                if constexpr (FP4) {
                    // scale word of this thread's 64 columns (4 scales of 16), if they exist
                    if (tok < p.N && 64 * bx < p.dk) cp_async_4(sdst, p.k_sf + row * (p.dk / 16) + 4 * bx);
                    else sdst[0] = 0u;
                    if (tok < p.N && 64 * bx < p.dv) cp_async_4(sdst + 1, p.v_sf + row * (p.dv / 16) + 4 * bx);
                    else sdst[1] = 0u;
                }
                if (++pc >= pu.c_end) {
                    pw += w_step;
                    if (pw < w_end) enter_unit();
                }
            }
            cp_async_commit();
            if (++pslot == BETA_AHEAD + 1) pslot = 0;
        };
        for (int i = 0; i < BETA_AHEAD; ++i) beta_prefetch();
        int cslot = 0;
        int stage = 0, bk = 0;
        uint32_t phase = 0, bk_phase = 0;
        for (int w = w_begin; w < w_end && !*abort_flag; w += w_step) {
            const Unit u = unit_of(p, w);
            bool ok = true;
            for (int c = u.c_begin; c < u.c_end; ++c) {
                beta_prefetch();                       // chunk BETA_AHEAD ahead
                cp_async_wait<BETA_AHEAD>();           // this chunk's copy has landed
                const float bval = beta_ring[cslot * SCALER_THREADS + t];
                uint32_t ksf = 0, vsf = 0;
                if constexpr (FP4) {
                    ksf = sf_ring[(cslot * SCALER_THREADS + t) * 2];
                    vsf = sf_ring[(cslot * SCALER_THREADS + t) * 2 + 1];
                }
                if (++cslot == BETA_AHEAD + 1) cslot = 0;
                if (!mbar_wait(&full[stage], phase, p.wait_limit_ns, abort_flag) ||
                    !mbar_wait(&bk_empty[bk], bk_phase ^ 1, p.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                if constexpr (FP8) {
                    // Thread pair (2r, 2r+1) owns token row r; this thread decodes the
                    // row's 64 columns of box bx (fp8 chunks 4bx..4bx+3, 16 columns
                    // each) of K and V to f16 and scales them by sqrt(beta) =
                    // hi + lo split into two f16: fma(x, hi, x*lo).
                    if (!(bval >= 0.0f && bval <= FP8_BETA_MAX)) record_error(GDN_ERR_RANGE);
                    const uint8_t* src = stage_base + stage * L::ST_BYTES + r * 128;
                    uint8_t* dst = bk_base + bk * L::BK_BYTES + bx * BOX_BYTES + r * 128;
                    const HSplit b2 = hsplit(sqrtf(fmaxf(bval, 0.0f)));
#pragma unroll
                    for (int i0 = 0; i0 < 4; ++i0) {
                        // box 1 walks its chunks in the order 2,3,0,1 so that the 8 threads of
                        // a quarter warp (4 rows x 2 boxes) hit 8 distinct bank groups
                        const int i = bx ? (i0 ^ 2) : i0;
                        const int c = 4 * bx + i;                    // fp8 chunk: columns 16c..16c+15
                        const int so = (c ^ (r & 7)) << 4;           // 128-byte swizzle of the TMA box
                        const uint4 k16 = *reinterpret_cast<const uint4*>(src + so);
                        const uint4 v16 = *reinterpret_cast<const uint4*>(src + BOX8_BYTES + so);
                        const uint32_t* kw = reinterpret_cast<const uint32_t*>(&k16);
                        const uint32_t* vw = reinterpret_cast<const uint32_t*>(&v16);
                        uint32_t kh[8], vh[8];
#pragma unroll
                        for (int wd = 0; wd < 4; ++wd) {
                            kh[2 * wd] = hscale(e4m3x2_to_f16x2(static_cast<uint16_t>(kw[wd] & 0xffffu)), b2);
                            kh[2 * wd + 1] = hscale(e4m3x2_to_f16x2(static_cast<uint16_t>(kw[wd] >> 16)), b2);
                            vh[2 * wd] = hscale(e4m3x2_to_f16x2(static_cast<uint16_t>(vw[wd] & 0xffffu)), b2);
                            vh[2 * wd + 1] = hscale(e4m3x2_to_f16x2(static_cast<uint16_t>(vw[wd] >> 16)), b2);
                        }
                        // columns 16i..16i+15 of box bx = its 16-bit chunks 2i and 2i+1
                        const int o0 = ((2 * i) ^ (r & 7)) << 4, o1 = ((2 * i + 1) ^ (r & 7)) << 4;
                        *reinterpret_cast<uint4*>(dst + o0) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
                        *reinterpret_cast<uint4*>(dst + o1) = make_uint4(kh[4], kh[5], kh[6], kh[7]);
                        *reinterpret_cast<uint4*>(dst + TILE_BYTES + o0) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
                        *reinterpret_cast<uint4*>(dst + TILE_BYTES + o1) = make_uint4(vh[4], vh[5], vh[6], vh[7]);
                    }
                } else if constexpr (FP4) {
                    // Thread pair (2r, 2r+1) owns token row r; this thread decodes the
                    // row's 64 columns of box bx: e2m1 codes (bytes 32bx..32bx+31 of
                    // the row, two per byte) times their E4M3 block scale (one per 16
                    // columns), exactly in f16, then times sqrt(beta) split hi + lo.
                    if (!(bval >= 0.0f && bval <= FP4_BETA_MAX)) record_error(GDN_ERR_RANGE);
                    const uint8_t* st = stage_base + stage * L::ST_BYTES;
                    uint8_t* dst = bk_base + bk * L::BK_BYTES + bx * BOX_BYTES + r * 128;
                    const HSplit b2 = hsplit(sqrtf(fmaxf(bval, 0.0f)));
                    const bool kin = 64 * bx < p.dk, vin = 64 * bx < p.dv;
                    uint32_t kw[8], vw[8];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 kx = kin ? *reinterpret_cast<const uint4*>(st + r * (p.dk / 2) + 32 * bx + 16 * q)
                                             : make_uint4(0, 0, 0, 0);
                        const uint4 vx = vin ? *reinterpret_cast<const uint4*>(st + RAW4_BYTES + r * (p.dv / 2) +
                                                                                 32 * bx + 16 * q)
                                             : make_uint4(0, 0, 0, 0);
                        kw[4 * q] = kx.x; kw[4 * q + 1] = kx.y; kw[4 * q + 2] = kx.z; kw[4 * q + 3] = kx.w;
                        vw[4 * q] = vx.x; vw[4 * q + 1] = vx.y; vw[4 * q + 2] = vx.z; vw[4 * q + 3] = vx.w;
                    }
#pragma unroll
                    for (int i0 = 0; i0 < 4; ++i0) {
                        const int i = bx ? (i0 ^ 2) : i0;    // columns 16i..16i+15 of box bx
                        const uint32_t ks2 = e4m3_to_f16x2_bcast(ksf >> (8 * i));
                        const uint32_t vs2 = e4m3_to_f16x2_bcast(vsf >> (8 * i));
                        uint32_t kh[8], vh[8];
                        fp4x8_to_f16(kw[2 * i], ks2, *reinterpret_cast<uint32_t(*)[4]>(&kh[0]));
                        fp4x8_to_f16(kw[2 * i + 1], ks2, *reinterpret_cast<uint32_t(*)[4]>(&kh[4]));
                        fp4x8_to_f16(vw[2 * i], vs2, *reinterpret_cast<uint32_t(*)[4]>(&vh[0]));
                        fp4x8_to_f16(vw[2 * i + 1], vs2, *reinterpret_cast<uint32_t(*)[4]>(&vh[4]));
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            kh[e] = hscale(kh[e], b2);
                            vh[e] = hscale(vh[e], b2);
                        }
                        const int o0 = ((2 * i) ^ (r & 7)) << 4, o1 = ((2 * i + 1) ^ (r & 7)) << 4;
                        *reinterpret_cast<uint4*>(dst + o0) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
                        *reinterpret_cast<uint4*>(dst + o1) = make_uint4(kh[4], kh[5], kh[6], kh[7]);
                        *reinterpret_cast<uint4*>(dst + TILE_BYTES + o0) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
                        *reinterpret_cast<uint4*>(dst + TILE_BYTES + o1) = make_uint4(vh[4], vh[5], vh[6], vh[7]);
                    }
                } else {
                    // thread pair (2r, 2r+1) owns token row r: box 0 and box 1 (64 columns each)
                    uint8_t* src = stage_base + stage * L::ST_BYTES + bx * BOX_BYTES + r * 128;
                    uint8_t* dst = bk_base + bk * L::BK_BYTES + bx * BOX_BYTES + r * 128;
                    const bool mine = bx < kboxes;
                    uint4 x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // rotate the 16-byte chunk order by row, and by 4 more for box 1, so
                        // the 8 threads of a quarter warp (4 rows x 2 boxes) hit 8 distinct
                        // bank groups
                        const int off = ((i + r + 4 * bx) & 7) << 4;
                        if (mine) x[i] = *reinterpret_cast<const uint4*>(src + off);
                        else x[i] = make_uint4(0, 0, 0, 0);
                    }
                    float sb = p.beta_sigmoid ? 1.0f / (1.0f + expf(-bval)) : bval;
                    if (p.norm_k) {
                        // k <- k / max(|k|, eps): the row's sum of squares over both halves
                        float ss = 0.0f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t* xs = reinterpret_cast<const uint32_t*>(&x[i]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
                                ss = fmaf(f2.x, f2.x, fmaf(f2.y, f2.y, ss));
                            }
                        }
                        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                        const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
                        sb *= inv;
                        if (mine) {
                            const BSplit n2 = bsplit(inv);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const uint4 y = bscale(x[i], n2);   // normalized k, the B operand
                                *reinterpret_cast<uint4*>(src + (((i + r + 4 * bx) & 7) << 4)) = y;
                            }
                        }
                    }
                    if (mine) {
                        // beta*k = fma(k, hi, k*lo) with beta = hi + lo split into two bf16
                        const BSplit b2 = bsplit(sb);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<uint4*>(dst + (((i + r + 4 * bx) & 7) << 4)) = bscale(x[i], b2);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&bk_full[bk]);
                if (LP) mbar_arrive(&empty[stage]);    // the decoders were the stage's last readers
                if (++bk == NBK) { bk = 0; bk_phase ^= 1; }
                if (++stage == NST) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
        }
        cp_async_wait<0>();  // no copy into the beta ring may outlive the CTA
    } else if (warp < EPI_WARP0 + 4) {
        // ----------------------------------------------------------- epilogue
        const int quarter = warp & 3;       // warps EPI_WARP0..EPI_WARP0+3 cover the four lane quarters
        const int j = quarter * 32 + lane;  // TMEM lane = row j of (beta K)^T = dk index
        int acc = 0;
        uint32_t acc_phase = 0;
        // The four epilogue warps take every decision together (the AND barrier), so
        // the named barriers of the split-item fixup below can never be left waiting.
        for (int w = w_begin; w < w_end; w += w_step) {
            const Unit u = unit_of(p, w);
            bool ok = mbar_wait(&tfull[acc], acc_phase, p.wait_limit_ns, abort_flag, 2010000 + (w & 0xffff));
            // ring mode: the scan has read the slot's previous frame (one scan CTA per head)
            if (ok && u.slot >= 0 && u.use > 0 && j == 0)
                ok = wait_count_geq(p.au_free + u.slot, u.use, p.wait_limit_ns, abort_flag, 2020000 + (w & 0xffff));
            if (!bar_and(1, 128, ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(quarter * 32) << 16);
            const bool jv = j < p.dk;
            const size_t per = static_cast<size_t>(p.dk) * p.dk + static_cast<size_t>(p.dv) * p.dk;
            // whole item: A (bf16) and U (fp32) straight to the workspace; split item: fp32
            // partial sums in the same element order
            float* part = u.split < 0 ? nullptr
                                      : p.partial + (static_cast<size_t>(u.item - p.whole) * p.split_per + u.split) * per;
            const size_t dst = static_cast<size_t>(u.item);   // A/U destination outside ring mode
            if (u.slot >= 0) {
                // ring slot: the whole zero-padded 128 x 128 tiles (D is exactly 0
                // past dk and dv), laid out as the scan's shared-memory image
                uint8_t* At = reinterpret_cast<uint8_t*>(p.A_ws) + static_cast<size_t>(u.slot) * RING_TILE_BF16;
                uint8_t* Ut = reinterpret_cast<uint8_t*>(p.U_ws) + static_cast<size_t>(u.slot) * RING_TILE_F32;
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t r32[32];
                    tmem_ld32(tbase + c0, r32);
                    tmem_wait_ld();
                    const float sa = LP ? p.a_scale : 1.0f;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4*>(At + ring_off(j, 2 * (c0 + 8 * q8))) = make_uint4(
                            pack_bf16x2(sa * __uint_as_float(r32[8 * q8 + 0]), sa * __uint_as_float(r32[8 * q8 + 1])),
                            pack_bf16x2(sa * __uint_as_float(r32[8 * q8 + 2]), sa * __uint_as_float(r32[8 * q8 + 3])),
                            pack_bf16x2(sa * __uint_as_float(r32[8 * q8 + 4]), sa * __uint_as_float(r32[8 * q8 + 5])),
                            pack_bf16x2(sa * __uint_as_float(r32[8 * q8 + 6]), sa * __uint_as_float(r32[8 * q8 + 7])));
                }
                // U[i][j] (row i = D column 128 + i): a warp writes one 128-byte line per i
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t r32[32];
                    tmem_ld32(tbase + 128 + c0, r32);
                    tmem_wait_ld();
                    const float su = LP ? p.u_scale : 1.0f;
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        *reinterpret_cast<float*>(Ut + ring_off(c0 + t, 4 * j)) = su * __uint_as_float(r32[t]);
                }
            } else {
                // A: row j of D holds A[j][0..dk); stored as row j (A is symmetric)
                for (int c0 = 0; c0 < p.dk; c0 += 32) {
                    uint32_t r32[32];
                    tmem_ld32(tbase + c0, r32);
                    tmem_wait_ld();
                    if (!jv) continue;
                    if (LP) {
#pragma unroll
                        for (int t = 0; t < 32; ++t) r32[t] = __float_as_uint(__uint_as_float(r32[t]) * p.a_scale);
                    }
                    if (part == nullptr) {
                        __nv_bfloat16* Arow = p.A_ws + (dst * p.dk + j) * p.dk;
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            uint4 v4 = make_uint4(
                                pack_bf16x2(__uint_as_float(r32[8 * q8 + 0]), __uint_as_float(r32[8 * q8 + 1])),
                                pack_bf16x2(__uint_as_float(r32[8 * q8 + 2]), __uint_as_float(r32[8 * q8 + 3])),
                                pack_bf16x2(__uint_as_float(r32[8 * q8 + 4]), __uint_as_float(r32[8 * q8 + 5])),
                                pack_bf16x2(__uint_as_float(r32[8 * q8 + 6]), __uint_as_float(r32[8 * q8 + 7])));
                            if (c0 + 8 * q8 < p.dk) *reinterpret_cast<uint4*>(Arow + c0 + 8 * q8) = v4;
                        }
                    } else {
                        float* prow = part + static_cast<size_t>(j) * p.dk;
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            if (c0 + 4 * q4 < p.dk)
                                *reinterpret_cast<uint4*>(prow + c0 + 4 * q4) =
                                    make_uint4(r32[4 * q4], r32[4 * q4 + 1], r32[4 * q4 + 2], r32[4 * q4 + 3]);
                    }
                }
                // U: row j of D holds U[0..dv)[j]; coalesced along j
                float* Uout = part == nullptr ? p.U_ws + dst * p.dv * p.dk
                                              : part + static_cast<size_t>(p.dk) * p.dk;
                for (int c0 = 0; c0 < p.dv; c0 += 32) {
                    uint32_t r32[32];
                    tmem_ld32(tbase + 128 + c0, r32);
                    tmem_wait_ld();
                    if (LP) {
#pragma unroll
                        for (int t = 0; t < 32; ++t) r32[t] = __float_as_uint(__uint_as_float(r32[t]) * p.u_scale);
                    }
                    if (jv) {
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (c0 + t < p.dv) Uout[static_cast<size_t>(c0 + t) * p.dk + j] = __uint_as_float(r32[t]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            if (u.slot >= 0) {
                // ring mode: every epilogue thread's stores, then one release (read
                // by the scan's copies through the async proxy after its acquire)
                fence_proxy_async_global();
                __threadfence();
                named_bar_sync(1, 128);
                if (j == 0) red_release_add(p.au_ready + u.slot, 1);
            }
            if (part != nullptr) {
                // Split item: once every split of the item has written its
                // partial sums, each split reduces its own share of the
                // elements, adding the partials in split order (deterministic).
                // The splits of an item are consecutive units, so they run on
                // distinct CTAs, each as its CTA's last unit, and the
                // cooperative launch keeps all of them resident: the wait ends.
                __threadfence();
                named_bar_sync(1, 128);
                const int r_item = u.item - p.whole;
                bool ready = true;
                if (j == 0) {
                    red_release_add(p.counters + r_item, 1);
                    ready = wait_count_geq(p.counters + r_item, p.split_per, p.wait_limit_ns, abort_flag);
                }
                if (!bar_and(1, 128, ready)) break;
                __threadfence();
                const float4* base = reinterpret_cast<const float4*>(
                    p.partial + static_cast<size_t>(r_item) * p.split_per * per);
                const size_t per4 = per / 4;                                   // dk, dv are multiples of 16
                const size_t a4 = static_cast<size_t>(p.dk) * p.dk / 4;        // A occupies [0, a4)
                const size_t e_begin = per4 * u.split / p.split_per;
                const size_t e_end = per4 * (u.split + 1) / p.split_per;
                // two elements per thread and up to eight splits per batch of
                // loads, all issued before the adds: 16 L2 reads in flight per thread
                const int S = p.split_per;
                auto store4 = [&](size_t e, const float4& v) {
                    if (e < a4) {
                        *reinterpret_cast<uint2*>(p.A_ws + static_cast<size_t>(u.item) * p.dk * p.dk + 4 * e) =
                            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                    } else {
                        *reinterpret_cast<float4*>(p.U_ws + static_cast<size_t>(u.item) * p.dv * p.dk +
                                                   4 * (e - a4)) = v;
                    }
                };
                for (size_t e0 = e_begin + j; e0 < e_end; e0 += 256) {
                    const size_t e1 = e0 + 128;
                    const bool has1 = e1 < e_end;
                    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
                    for (int sb = 0; sb < S; sb += 8) {
                        float4 t0[8], t1[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (sb + i < S) {
                                t0[i] = __ldcg(base + static_cast<size_t>(sb + i) * per4 + e0);
                                if (has1) t1[i] = __ldcg(base + static_cast<size_t>(sb + i) * per4 + e1);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (sb + i < S) {  // splits added in order
                                s0.x += t0[i].x; s0.y += t0[i].y; s0.z += t0[i].z; s0.w += t0[i].w;
                                if (has1) { s1.x += t1[i].x; s1.y += t1[i].y; s1.z += t1[i].z; s1.w += t1[i].w; }
                            }
                        }
                    }
                    store4(e0, s0);
                    if (has1) store4(e1, s1);
                }
            }
        }
    }

    // Wait for all outstanding MMAs before releasing TMEM.
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Standalone phase 1: a persistent grid, work units round-robin.
template <int FMT>
__global__ void __launch_bounds__(THREADS, 1)
    contract_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    contract_role<FMT>(tm_k, tm_v, p, blockIdx.x, gridDim.x, smem);
}

}  // namespace k1
}  // namespace gdn
