// gdn_k1_pair.cuh -- phase 1 of the frame-wise GDN forward for two heads at a
// time:  A_f = K_f^T B_f K_f,  U_f = V_f^T B_f K_f  for heads 2p and 2p + 1 of
// one (b, f) (SANA-WM article, "The Architecture": everything one latent frame
// contributes to the state's decay-gate / delta-rule update).
//
// Why pairs.  The tensor-memory accelerator's cost is per box row, not per
// byte: a box whose rows are the 256 B of one head (two 128-byte halves) per
// token streams at about 45-50 GB/s per CTA on B300, a box that covers the
// 512 contiguous bytes of two heads per token at about 100 GB/s (measured).
// The k and v boxes of a stage therefore cover two heads.  They are cut so
// that shared memory receives the operands in the canonical MN-major 128-byte
// swizzled layout directly: the token index is split into (t8, group) with
// t8 the second box dimension, so each (head, half, 8-token group) lands as
// one 1024-byte swizzle atom; for head hd the MMA reads 64-column blocks at
// a 1 KB stride and 8-token groups at a 4 KB stride.  The split needs the
// whole token sequence in groups of 8 (N % 8 == 0); a chunk that ends a frame
// also reads the first tokens of the next frame, whose rows the scalers
// clear (beta = 0 there, and the K and V rows are zeroed) so they add nothing.
//
// Per chunk of 64 tokens and head: D_hd += (beta K)^T K and D_hd += (beta K)^T V
// (two MMAs of M = 128, N = 128 per 16 tokens); the two heads' accumulators
// fill TMEM (2 x 256 columns), so the epilogue drains them before the next
// pair starts.  Warp roles as in gdn_k1_contract.cuh (320 threads): warp 0
// TMA producer, warp 1 TMEM owner and MMA issuer, warps 2-5 scalers, warps
// 6-9 epilogue.  Parameters, ring mode and results as k1::Params /
// k1::contract_role (bf16 inputs; dk = dv = 128; H even).
#pragma once

#include "gdn_k1_contract.cuh"

namespace gdn {
namespace k1p {

using k1::Params;
constexpr int CHUNK = 64;                    // tokens per stage
constexpr int GROUPS = CHUNK / 8;            // 8-token groups per stage
constexpr int ATOM = 1024;                   // 8 rows x 128 B
constexpr int PAIR_BYTES = CHUNK * 512;      // 64 tokens x 2 heads x 256 B = 32 KB
constexpr int STAGE_BYTES = 2 * PAIR_BYTES;  // k pair | v pair
constexpr int STAGES = 2;
constexpr int BK_HEAD = CHUNK * 256;         // beta K of one head: 64 tokens x 128 columns bf16
constexpr int BK_BYTES = 2 * BK_HEAD;
constexpr int NBK = 2;
constexpr int SCALER_THREADS = 128;
constexpr int EPI_WARP0 = 6;
constexpr int THREADS = 320;
constexpr int BETA_AHEAD = 4;
constexpr int BETA_RING_BYTES = (BETA_AHEAD + 1) * SCALER_THREADS * 8;   // beta of both heads
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NBK * BK_BYTES + BETA_RING_BYTES + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert((2 * STAGES + 2 * NBK + 3) * 8 + 8 <= 256, "barrier area");
// stage layout of a pair box: ((g * 2 + hd) * 2 + half) * ATOM + t8 * 128
constexpr uint32_t ST_LBO = ATOM;            // 64-column blocks of one head
constexpr uint32_t ST_SBO = 4 * ATOM;        // 8-token groups
// beta K of head hd: hd * BK_HEAD + (g * 2 + half) * ATOM + t8 * 128
constexpr uint32_t BK_LBO = ATOM;
constexpr uint32_t BK_SBO = 2 * ATOM;

// Work units: whole pairs (b, f, p) in scan order when p.ring > 0, else in
// item order (b, f) major; `item0` is the first head's item, `slot0` its ring
// slot (the second head's are item0 + 1 and slot0 + 1).
struct Unit {
    int item0, slot0, use;
};
__device__ __forceinline__ Unit pair_unit_of(const Params& p, int w) {
    const int P = p.H / 2;
    Unit u;
    if (p.ring > 0) {
        const int BP = p.B * P;
        const int st = w / BP, r = w % BP, b = r / P, pr = r % P;
        const int f = p.reverse ? p.F - 1 - st : st;
        u.item0 = (b * p.F + f) * p.H + 2 * pr;
        u.slot0 = (b * p.ring + st % p.ring) * p.H + 2 * pr;
        u.use = st / p.ring;
        return u;
    }
    u.item0 = (w / P) * p.H + 2 * (w % P);
    u.slot0 = -1;
    u.use = 0;
    return u;
}

// tm_k, tm_v: 5-D maps {64, 8, 2, H, B*F*N/8} (columns, token in group, half,
// head, 8-token group) with box {64, 8, 2, 2, CHUNK / 8}.  Units w_begin,
// w_begin + w_step, ... < p.work (p.work = number of pairs).
__device__ __forceinline__ void contract_pair_role(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                                   const Params& p, int w_begin, int w_step, uint8_t* smem) {
    uint8_t* stage_base = smem;
    uint8_t* bk_base = smem + STAGES * STAGE_BYTES;
    float2* beta_ring = reinterpret_cast<float2*>(bk_base + NBK * BK_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(bk_base + NBK * BK_BYTES + BETA_RING_BYTES);
    uint64_t* full = bars;              // [STAGES]
    uint64_t* empty = full + STAGES;    // [STAGES]
    uint64_t* bk_full = empty + STAGES; // [NBK]
    uint64_t* bk_empty = bk_full + NBK; // [NBK]
    uint64_t* tfull = bk_empty + NBK;   // the pair's accumulators are complete
    uint64_t* tempty = tfull + 1;       // drained by the epilogue
    uint64_t* final_bar = tempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int w_end = p.work;
    const int chunks = p.chunks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NBK; ++b) {
            mbar_init(&bk_full[b], SCALER_THREADS);
            mbar_init(&bk_empty[b], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 128);
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
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
                const Unit u = pair_unit_of(p, w);
                const int bf = u.item0 / p.H, h0 = u.item0 % p.H;
                for (int c = 0; c < chunks; ++c) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_limit_ns, abort_flag)) break;
                    uint8_t* st = stage_base + stage * STAGE_BYTES;
                    const int g = (bf * p.N + c * CHUNK) / 8;   // first 8-token group of the chunk
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_5d(st, &tm_k, &full[stage], 0, 0, 0, h0, g);
                    tma_load_5d(st + PAIR_BYTES, &tm_v, &full[stage], 0, 0, 0, h0, g);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            for (long long kf = (issued > STAGES ? issued - STAGES : 0); kf < issued; ++kf)
                mbar_wait_drain(&full[kf % STAGES], static_cast<uint32_t>((kf / STAGES) & 1), p.wait_limit_ns);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16(128, 128, 1, 1);
            int stage = 0, bk = 0;
            uint32_t phase = 0, bk_phase = 0, t_phase = 0;
            for (int w = w_begin; w < w_end && !*abort_flag; w += w_step) {
                if (!mbar_wait(tempty, t_phase ^ 1, p.wait_limit_ns, abort_flag)) break;
                tc_fence_after();
                bool ok = true;
                for (int c = 0; c < chunks; ++c) {
                    if (!mbar_wait(&full[stage], phase, p.wait_limit_ns, abort_flag) ||
                        !mbar_wait(&bk_full[bk], bk_phase, p.wait_limit_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(stage_base + stage * STAGE_BYTES);
                    const uint32_t bkb = smem_u32(bk_base + bk * BK_BYTES);
#pragma unroll
                    for (int hd = 0; hd < 2; ++hd) {
#pragma unroll
                        for (int kk = 0; kk < CHUNK / 16; ++kk) {   // 16 tokens = two 8-token groups
                            const uint64_t ad = smem_desc(bkb + hd * BK_HEAD + kk * 2 * BK_SBO, BK_LBO, BK_SBO);
                            const uint64_t kd = smem_desc(st + hd * 2 * ATOM + kk * 2 * ST_SBO, ST_LBO, ST_SBO);
                            const uint64_t vd =
                                smem_desc(st + PAIR_BYTES + hd * 2 * ATOM + kk * 2 * ST_SBO, ST_LBO, ST_SBO);
                            const uint32_t acc = (c > 0 || kk > 0) ? 1u : 0u;
                            mma_bf16(tmem_base + hd * 256, ad, kd, IDESC, acc);
                            mma_bf16(tmem_base + hd * 256 + 128, ad, vd, IDESC, acc);
                        }
                    }
                    mma_commit(&empty[stage]);
                    mma_commit(&bk_empty[bk]);
                    if (++bk == NBK) { bk = 0; bk_phase ^= 1; }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(tfull);
                t_phase ^= 1;
            }
            mma_commit(final_bar);
            mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
        }
    } else if (warp < EPI_WARP0) {
        // ------------------------------------------------------ beta scalers
        // thread pair (2r, 2r+1): token row r of the chunk, column half bx of
        // both heads; beta of both heads (adjacent in memory) by an 8-byte
        // cp.async BETA_AHEAD chunks ahead
        const int t = threadIdx.x - 64;
        const int r = t >> 1, bx = t & 1;
        const int g = r >> 3, t8 = r & 7;
        int pw = w_begin, pc = 0, pslot = 0;
        size_t prow0 = 0;   // beta row of token 0 of the cursor's pair (unit index math once per unit)
        auto enter_unit = [&]() {
            const Unit u = pair_unit_of(p, pw);
            prow0 = static_cast<size_t>(u.item0 / p.H) * p.N * p.H + (u.item0 % p.H);
        };
        if (pw < w_end) enter_unit();
        auto beta_prefetch = [&]() {
            float2* dst = beta_ring + pslot * SCALER_THREADS + t;
            if (pw < w_end) {
                const int tok = pc * CHUNK + r;
                if (tok < p.N)
                    cp_async_8(dst, p.beta + prow0 + static_cast<size_t>(tok) * p.H);
                else
                    *dst = make_float2(0.0f, 0.0f);
                if (++pc >= chunks) {
                    pc = 0;
                    pw += w_step;
                    if (pw < w_end) enter_unit();
                }
            }
            cp_async_commit();
            if (++pslot == BETA_AHEAD + 1) pslot = 0;
        };
        for (int i = 0; i < BETA_AHEAD; ++i) beta_prefetch();
        int cslot = 0, stage = 0, bk = 0;
        uint32_t phase = 0, bk_phase = 0;
        for (int w = w_begin; w < w_end && !*abort_flag; w += w_step) {
            bool ok = true;
            for (int c = 0; c < chunks; ++c) {
                beta_prefetch();
                cp_async_wait<BETA_AHEAD>();
                const float2 bv = beta_ring[cslot * SCALER_THREADS + t];
                if (++cslot == BETA_AHEAD + 1) cslot = 0;
                if (!mbar_wait(&full[stage], phase, p.wait_limit_ns, abort_flag) ||
                    !mbar_wait(&bk_empty[bk], bk_phase ^ 1, p.wait_limit_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const bool live = c * CHUNK + r < p.N;   // rows past the frame belong to the next frame
                uint8_t* st = stage_base + stage * STAGE_BYTES;
#pragma unroll
                for (int hd = 0; hd < 2; ++hd) {
                    const int atom = (g * 2 + hd) * 2 + bx;
                    uint8_t* krow = st + atom * ATOM + t8 * 128;
                    uint8_t* dst = bk_base + bk * BK_BYTES + hd * BK_HEAD + (g * 2 + bx) * ATOM + t8 * 128;
                    uint4 x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        x[i] = live ? *reinterpret_cast<const uint4*>(krow + (((i + r + 4 * bx) & 7) << 4))
                                    : make_uint4(0, 0, 0, 0);
                    float sb = hd ? bv.y : bv.x;
                    if (p.beta_sigmoid) sb = 1.0f / (1.0f + expf(-sb));
                    if (!live) sb = 0.0f;
                    if (p.norm_k) {
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
                        sb *= inv;   // beta K = k * (beta / |k|), from the raw k (one rounding)
                        if (live) {
                            const k1::BSplit n2 = k1::bsplit(inv);
#pragma unroll
                            for (int i = 0; i < 8; ++i)   // normalized k, the B operand
                                *reinterpret_cast<uint4*>(krow + (((i + r + 4 * bx) & 7) << 4)) = k1::bscale(x[i], n2);
                        }
                    }
                    if (!live) {
                        // clear this row's K and V halves: the next frame's tokens add nothing
                        uint8_t* vrow = krow + PAIR_BYTES;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            *reinterpret_cast<uint4*>(krow + (i << 4)) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4*>(vrow + (i << 4)) = make_uint4(0, 0, 0, 0);
                        }
                    }
                    const k1::BSplit b2 = k1::bsplit(sb);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<uint4*>(dst + (((i + r + 4 * bx) & 7) << 4)) = k1::bscale(x[i], b2);
                }
                fence_proxy_async_smem();
                mbar_arrive(&bk_full[bk]);
                if (++bk == NBK) { bk = 0; bk_phase ^= 1; }
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
        }
        cp_async_wait<0>();
    } else if (warp < EPI_WARP0 + 4) {
        // ----------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int j = quarter * 32 + lane;   // TMEM lane = row j of A = column j of U
        uint32_t t_phase = 0;
        for (int w = w_begin; w < w_end; w += w_step) {
            const Unit u = pair_unit_of(p, w);
            bool ok = mbar_wait(tfull, t_phase, p.wait_limit_ns, abort_flag);
            // ring mode: the scan has read both slots' previous frames
            if (ok && u.slot0 >= 0 && u.use > 0 && j == 0)
                ok = wait_count_geq(p.au_free + u.slot0, u.use, p.wait_limit_ns, abort_flag) &&
                     wait_count_geq(p.au_free + u.slot0 + 1, u.use, p.wait_limit_ns, abort_flag);
            if (!bar_and(1, 128, ok)) break;
            tc_fence_after();
#pragma unroll 1
            for (int hd = 0; hd < 2; ++hd) {
                const size_t dst = static_cast<size_t>(u.slot0 >= 0 ? u.slot0 + hd : u.item0 + hd);
                const uint32_t tb = tmem_base + hd * 256 + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t a32[32], u32[32];
                    tmem_ld32(tb + c0, a32);
                    tmem_ld32(tb + 128 + c0, u32);
                    tmem_wait_ld();
                    // ring mode: the tiles in the scan's shared-memory image (ring_off)
                    const bool rm = u.slot0 >= 0;
                    uint8_t* At = reinterpret_cast<uint8_t*>(p.A_ws) + dst * RING_TILE_BF16;
                    uint8_t* Ut = reinterpret_cast<uint8_t*>(p.U_ws) + dst * RING_TILE_F32;
                    __nv_bfloat16* Arow = p.A_ws + (dst * 128 + j) * 128 + c0;
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        const uint4 v4 = make_uint4(
                            pack_bf16x2(__uint_as_float(a32[8 * q8 + 0]), __uint_as_float(a32[8 * q8 + 1])),
                            pack_bf16x2(__uint_as_float(a32[8 * q8 + 2]), __uint_as_float(a32[8 * q8 + 3])),
                            pack_bf16x2(__uint_as_float(a32[8 * q8 + 4]), __uint_as_float(a32[8 * q8 + 5])),
                            pack_bf16x2(__uint_as_float(a32[8 * q8 + 6]), __uint_as_float(a32[8 * q8 + 7])));
                        if (rm)
                            *reinterpret_cast<uint4*>(At + ring_off(j, 2 * (c0 + 8 * q8))) = v4;
                        else
                            *reinterpret_cast<uint4*>(Arow + 8 * q8) = v4;
                    }
                    float* Ucol = p.U_ws + dst * 128 * 128 + j;
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        if (rm)
                            *reinterpret_cast<float*>(Ut + ring_off(c0 + t, 4 * j)) = __uint_as_float(u32[t]);
                        else
                            Ucol[static_cast<size_t>(c0 + t) * 128] = __uint_as_float(u32[t]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty);
            t_phase ^= 1;
            if (u.slot0 >= 0) {
                fence_proxy_async_global();
                __threadfence();
                named_bar_sync(1, 128);
                if (j == 0) {
                    red_release_add(p.au_ready + u.slot0, 1);
                    red_release_add(p.au_ready + u.slot0 + 1, 1);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// Standalone phase 1 on head pairs: a persistent grid, units round-robin.
__global__ void __launch_bounds__(THREADS, 1)
    contract_pair_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    contract_pair_role(tm_k, tm_v, p, blockIdx.x, gridDim.x, smem);
}

}  // namespace k1p
}  // namespace gdn
