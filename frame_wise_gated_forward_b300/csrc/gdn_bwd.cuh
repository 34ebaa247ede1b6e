// gdn_bwd.cuh -- the backward pass of the frame-wise GDN forward: the two
// frame-parallel gradient kernels.  The reverse recurrence of the state
// gradient runs on the forward's scan kernel (see gdn_frame_backward in
// gdn_api.cu); these kernels turn its per-frame results into the gradients.
//
// Per (b, f, h) with S_{f-1} the state before frame f, G_f = dL/dS_f, and the
// forward S_f = alpha_f (S_{f-1} - S_{f-1} A_f) + U_f, o_n = S_f q_n
// (SANA-WM article, "The Architecture": a decay gate and a delta-rule
// correction of a fixed-size state, one latent frame per step), the chain
// rule gives
//     P_f = S_{f-1}^T G_f,  dalpha_f = tr P_f - <P_f, A_f>,
//     W_f = dA_f + dA_f^T = -alpha_f (P_f + P_f^T)
// (frame_grad_kernel) and, per token n of frame f,
//     dk_n = beta_n (W_f k_n + G_f^T v_n),  dv_n = beta_n G_f k_n,
//     dbeta_n = k_n^T W_f k_n / 2 + v_n^T G_f k_n       (token_grad_kernel)
//     dq_n = S_f^T do_n           (the forward's output kernel, S_f MN-major).  Both are tcgen05 MMAs on operands TMA-loaded into
// 128-byte-swizzled shared memory; the bf16 per-frame states S and G are read
// MN-major or K-major from the same tile as each product needs.
//
// Both kernels take one batch row (items f*H + h); each CTA runs one work
// unit's MMAs and epilogue at a time while the next unit's copies are in
// flight.  Every wait is bounded.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace bwd {

constexpr int THREADS = 128;                 // four warps: TMEM lane quarters
constexpr int BOX = 128 * 128;               // 128 rows x 64 bf16 columns
constexpr int TILE = 2 * BOX;                // 128 x 128 bf16, two 64-column boxes
constexpr uint32_t MN_LBO = BOX;             // MN-major: distance between 64-column blocks
constexpr uint32_t SBO = 1024;               // 8 rows x 128 B
constexpr int PT_STRIDE = 129;               // fp32 staging of P^T, padded against bank conflicts

// ------------------------------------------------------------ frame grads
constexpr size_t FRAME_SMEM = 1024 + 4 * TILE + 128 * PT_STRIDE * 4 + 256;
static_assert(FRAME_SMEM <= 232448, "shared memory");

struct FrameParams {
    const float* alpha;       // [F, H] forward decay
    float* d_alpha;           // [F, H] out
    __nv_bfloat16* W;         // [F*H][dk][dk] out: -alpha (P + P^T)
    int H, F, dk, dv;
    unsigned long long wait_limit_ns;
};

// One CTA per SM; item f*H + h: P = S_{f-1}^T G_f with M = dk, N = dk, K = dv,
// both operands MN-major straight from the [dv][dk] state images.
//   tm_Sx: per-frame states, slot f holds S_{f-1} (slot 0 = S_0)
//   tm_Gx: state gradients, slot f + 1 holds G_f
//   tm_A:  A_f (bf16 [dk][dk])
__global__ void __launch_bounds__(THREADS, 1)
    frame_grad_kernel(const __grid_constant__ CUtensorMap tm_Sx, const __grid_constant__ CUtensorMap tm_Gx,
                      const __grid_constant__ CUtensorMap tm_A, const FrameParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sS = smem;
    uint8_t* sG = sS + TILE;
    uint8_t* sA2 = sG + TILE;                                          // [2]: A_f is read by the epilogue
    float* Pt = reinterpret_cast<float*>(sA2 + 2 * TILE);              // Pt[c * 129 + j] = P[j][c]
    uint64_t* bars = reinterpret_cast<uint64_t*>(Pt + 128 * PT_STRIDE);
    uint64_t* load_bar = bars;
    uint64_t* mma_bar = bars + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* red = reinterpret_cast<float*>(tmem_slot + 2);               // [4] per-warp partial sums

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kboxes = p.dk > 64 ? 2 : 1;
    const int items = p.F * p.H;
    if (kboxes < 2)  // box 1 of every tile is never loaded and must read as zero
        for (int i = tid; i < 4 * TILE / 16; i += THREADS) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(load_bar, 1);
        mbar_init(mma_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_Sx);
        prefetch_tmap(&tm_Gx);
        prefetch_tmap(&tm_A);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    uint32_t phase = 0;
    bool load_pending = false, mma_pending = false;

    // thread 0: copies of item `it` (S_{f-1}, G_f, and A_f into buffer `ab`); the
    // next item's copies are issued as soon as this item's MMAs have completed
    auto issue_loads = [&](int it, int ab) {
        const int f = it / p.H, h = it % p.H;
        mbar_arrive_expect_tx(load_bar, 3 * kboxes * BOX);
        for (int bx = 0; bx < kboxes; ++bx) {
            tma_load_3d(sS + bx * BOX, &tm_Sx, load_bar, 64 * bx, 0, f * p.H + h);
            tma_load_3d(sG + bx * BOX, &tm_Gx, load_bar, 64 * bx, 0, (f + 1) * p.H + h);
            tma_load_3d(sA2 + ab * TILE + bx * BOX, &tm_A, load_bar, 64 * bx, 0, it);
        }
    };
    if (tid == 0 && static_cast<int>(blockIdx.x) < items) issue_loads(blockIdx.x, 0);
    load_pending = static_cast<int>(blockIdx.x) < items;
    int ab = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ab ^= 1) {
        uint8_t* sA = sA2 + ab * TILE;
        bool ok = mbar_wait(load_bar, phase, p.wait_limit_ns, abort_flag);
        if (!__syncthreads_and(ok)) break;
        load_pending = false;
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t IDESC = idesc_bf16(128, 128, 1, 1);
            const int nk = (p.dv + 15) / 16;
            for (int kk = 0; kk < nk; ++kk) {
                const uint64_t ad = smem_desc(smem_u32(sS) + kk * 2048, MN_LBO, SBO);
                const uint64_t bd = smem_desc(smem_u32(sG) + kk * 2048, MN_LBO, SBO);
                mma_bf16(tmem_base, ad, bd, IDESC, kk > 0 ? 1u : 0u);
            }
            mma_commit(mma_bar);
        }
        mma_pending = true;
        ok = mbar_wait(mma_bar, phase, p.wait_limit_ns, abort_flag);
        if (!__syncthreads_and(ok)) break;
        mma_pending = false;
        phase ^= 1;
        tc_fence_after();
        if (it + static_cast<int>(gridDim.x) < items) {
            if (tid == 0) issue_loads(it + gridDim.x, ab ^ 1);
            load_pending = true;
        }

        // thread j holds row j of P (TMEM lane j): the trace term, <P, A> with
        // row j of A from shared memory, and P^T staged for the transpose
        const int j = tid;
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        float part = 0.0f;
        for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t r32[32];
            tmem_ld32(trow + c0, r32);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const int c = c0 + t;
                const float pv = __uint_as_float(r32[t]);
                Pt[c * PT_STRIDE + j] = pv;
                if (j < p.dk && c < p.dk) {
                    // A[j][c] in the swizzled K-major tile: box c/64, 16-byte chunk (c%64)/8
                    const int cc = c & 63;
                    const __nv_bfloat16* ap = reinterpret_cast<const __nv_bfloat16*>(
                        sA + (c >> 6) * BOX + j * 128 + ((((cc >> 3) ^ (j & 7))) << 4)) + (cc & 7);
                    part += (c == j ? pv : 0.0f) - pv * __bfloat162float(*ap);
                }
            }
        }
        tc_fence_before();
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red[warp] = part;
        __syncthreads();
        const float af = p.alpha[it];
        if (tid == 0) p.d_alpha[it] = (red[0] + red[1]) + (red[2] + red[3]);
        if (j < p.dk) {
            __nv_bfloat16* wrow = p.W + (static_cast<size_t>(it) * p.dk + j) * p.dk;
            for (int c0 = 0; c0 < p.dk; c0 += 8) {
                float w[8];
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    w[t] = -af * (Pt[(c0 + t) * PT_STRIDE + j] + Pt[j * PT_STRIDE + c0 + t]);
                *reinterpret_cast<uint4*>(wrow + c0) =
                    make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                               pack_bf16x2(w[6], w[7]));
            }
        }
        __syncthreads();  // tiles, Pt and red are reused by the next item
    }
    // an abandoned item's copies or MMAs must land before the CTA leaves
    if (tid == 0) {
        if (load_pending) mbar_wait_drain(load_bar, phase, p.wait_limit_ns);
        if (mma_pending) mbar_wait_drain(mma_bar, phase, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 128);
    }
}

// ------------------------------------------------------------ token grads
// dq = dO S_f runs on the forward's output kernel with the state read
// MN-major (k3::Params::b_mn); this kernel forms dk, dv and dbeta from two
// accumulators per 128-token tile, M = 128 tokens each:
//     T12 = K W_f + V G_f     T3 = K G_f^T
// so dk = beta T12, dv = beta T3, and, since T12 . k_n = k_n^T W_f k_n +
// v_n^T G_f k_n and T3 . v_n = v_n^T G_f k_n,
//     dbeta_n = (T12 . k_n + T3 . v_n) / 2.
// Two accumulator pairs fill TMEM's 512 columns, so one tile's MMAs run while
// the previous tile's epilogue drains.  Warp roles (320 threads): warp 0 TMA
// producer, warp 1 TMEM owner and MMA issuer, warps 2-9 epilogue (two warps
// per TMEM lane quarter, one per half of the columns).  Token tiles (k, v)
// stream through a 2-deep ring; a slot is released when the epilogue has read
// its k and v rows.  G_f (K-major for T3, MN-major for T12) and W_f (K-major,
// symmetric) are reloaded when the item changes.
constexpr int TOKEN_THREADS = 320;
constexpr int TOKEN_EPI = 256;
constexpr int KV_STAGES = 2;
constexpr size_t TOKEN_SMEM = 1024 + (2 * KV_STAGES + 2) * TILE + 256 + 2 * 128 * 4;
static_assert(TOKEN_SMEM <= 232448, "shared memory");

struct TokenParams {
    const float* beta;         // [F, N, H]
    __nv_bfloat16 *dk_out, *dv_out;  // [F, N, H, d] out
    float* d_beta;             // [F, N, H] out
    int H, F, N, dk, dv;
    int ntile;                 // ceil(N / 128)
    long long units;           // F * H * ntile
    unsigned long long wait_limit_ns;
};

__global__ void __launch_bounds__(TOKEN_THREADS, 1)
    token_grad_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_Gx, const __grid_constant__ CUtensorMap tm_W,
                      const TokenParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;                              // [KV_STAGES][K tile | V tile]
    uint8_t* sG = ring + KV_STAGES * 2 * TILE;
    uint8_t* sW = sG + TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sW + TILE);
    uint64_t* kfull = bars;                            // [2] TMA landed k, v
    uint64_t* kempty = kfull + KV_STAGES;              // [2] epilogue read the rows
    uint64_t* tfull = kempty + KV_STAGES;              // [2] accumulator pair ready
    uint64_t* tempty = tfull + 2;                      // [2] accumulator pair drained
    uint64_t* gw_full = tempty + 2;                    // G_f, W_f landed
    uint64_t* gw_empty = gw_full + 1;                  // the item's last MMAs retired
    uint64_t* final_bar = gw_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* dbh = reinterpret_cast<float*>(sW + TILE + 256);   // [2][128] upper column half's dbeta part

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kb = p.dk > 64 ? 2 : 1, vb = p.dv > 64 ? 2 : 1;
    if (kb < 2 || vb < 2)  // boxes that are never loaded must read as zero
        for (int i = tid; i < (2 * KV_STAGES + 2) * TILE / 16; i += TOKEN_THREADS)
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(&kfull[s], 1);
            mbar_init(&kempty[s], TOKEN_EPI);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], TOKEN_EPI);
        }
        mbar_init(gw_full, 1);
        mbar_init(gw_empty, 1);
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_Gx);
        prefetch_tmap(&tm_W);
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

    // contiguous unit ranges: a CTA's consecutive tiles mostly share an item
    const long long u_begin = (static_cast<long long>(blockIdx.x) * p.units) / gridDim.x;
    const long long u_end = (static_cast<long long>(blockIdx.x + 1) * p.units) / gridDim.x;
    // (item, tile, frame row, head) of unit u, stepped once per unit: the 64-bit
    // divisions that give them directly cost every thread of the epilogue
    // more than a little of each tile's work
    struct TileCursor {
        int item, tile, f, h;
        __device__ TileCursor(long long u, int ntile, int H) {
            item = static_cast<int>(u / ntile);
            tile = static_cast<int>(u - static_cast<long long>(item) * ntile);
            f = item / H;
            h = item - f * H;
        }
        __device__ void next(int ntile, int H) {
            if (++tile == ntile) {
                tile = 0;
                ++item;
                if (++h == H) { h = 0; ++f; }
            }
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int gw_item = -1, gw_loads = 0;
            long long issued = 0;
            TileCursor cur(u_begin, p.ntile, p.H);
            for (long long u = u_begin; u < u_end; ++u, cur.next(p.ntile, p.H)) {
                const long long i = u - u_begin;
                const int s = static_cast<int>(i % KV_STAGES);
                const int item = cur.item, tile = cur.tile;
                const int f = cur.f, h = cur.h;
                if (!mbar_wait(&kempty[s], static_cast<uint32_t>(((i / KV_STAGES) & 1) ^ 1), p.wait_limit_ns,
                               abort_flag))
                    break;
                if (item != gw_item) {
                    if (!mbar_wait(gw_empty, static_cast<uint32_t>((gw_loads & 1) ^ 1), p.wait_limit_ns, abort_flag))
                        break;
                    mbar_arrive_expect_tx(gw_full, 2 * kb * BOX);
                    for (int bx = 0; bx < kb; ++bx) {
                        tma_load_3d(sG + bx * BOX, &tm_Gx, gw_full, 64 * bx, 0, (f + 1) * p.H + h);  // G_f
                        tma_load_3d(sW + bx * BOX, &tm_W, gw_full, 64 * bx, 0, item);
                    }
                    gw_item = item;
                    ++gw_loads;
                }
                uint8_t* dst = ring + s * 2 * TILE;
                mbar_arrive_expect_tx(&kfull[s], (kb + vb) * BOX);
                for (int bx = 0; bx < kb; ++bx) tma_load_4d(dst + bx * BOX, &tm_k, &kfull[s], 64 * bx, h, tile * 128, f);
                for (int bx = 0; bx < vb; ++bx)
                    tma_load_4d(dst + TILE + bx * BOX, &tm_v, &kfull[s], 64 * bx, h, tile * 128, f);
                ++issued;
            }
            // copies in flight must land before the CTA leaves (only when a wait gave up)
            for (long long kq = (issued > KV_STAGES ? issued - KV_STAGES : 0); kq < issued; ++kq)
                mbar_wait_drain(&kfull[kq % KV_STAGES], static_cast<uint32_t>((kq / KV_STAGES) & 1), p.wait_limit_ns);
            if (gw_loads > 0) mbar_wait_drain(gw_full, static_cast<uint32_t>((gw_loads - 1) & 1), p.wait_limit_ns);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_KK = idesc_bf16(128, 128, 0, 0);   // A K-major, B K-major
            constexpr uint32_t ID_KM = idesc_bf16(128, 128, 0, 1);   // A K-major, B MN-major
            const int nkk = (p.dk + 15) / 16, nkv = (p.dv + 15) / 16;
            const uint32_t bG = smem_u32(sG), bW = smem_u32(sW);
            int gw_item = -1, gw_used = 0;
            TileCursor cur(u_begin, p.ntile, p.H);
            for (long long u = u_begin; u < u_end; ++u, cur.next(p.ntile, p.H)) {
                const long long i = u - u_begin;
                const int s = static_cast<int>(i % KV_STAGES), a = static_cast<int>(i & 1);
                const int item = cur.item;
                if (!mbar_wait(&tempty[a], static_cast<uint32_t>(((i >> 1) & 1) ^ 1), p.wait_limit_ns, abort_flag) ||
                    !mbar_wait(&kfull[s], static_cast<uint32_t>((i / KV_STAGES) & 1), p.wait_limit_ns, abort_flag))
                    break;
                if (item != gw_item) {
                    if (!mbar_wait(gw_full, static_cast<uint32_t>(gw_used & 1), p.wait_limit_ns, abort_flag)) break;
                    gw_item = item;
                    ++gw_used;
                }
                tc_fence_after();
                const uint32_t aK = smem_u32(ring + s * 2 * TILE), aV = aK + TILE;
                const uint32_t t12 = tmem_base + a * 256, t3 = t12 + 128;
                for (int kk = 0; kk < nkk; ++kk) {   // K W and K G^T: K-steps over dk
                    const uint32_t ko = (kk >> 2) * BOX + (kk & 3) * 32;
                    const uint64_t ad = smem_desc(aK + ko, 16, SBO);
                    mma_bf16(t12, ad, smem_desc(bW + ko, 16, SBO), ID_KK, kk > 0 ? 1u : 0u);
                    mma_bf16(t3, ad, smem_desc(bG + ko, 16, SBO), ID_KK, kk > 0 ? 1u : 0u);
                }
                for (int kk = 0; kk < nkv; ++kk) {   // + V G: K-steps over dv, into the same accumulator
                    const uint32_t ko = (kk >> 2) * BOX + (kk & 3) * 32;
                    mma_bf16(t12, smem_desc(aV + ko, 16, SBO), smem_desc(bG + kk * 2048, MN_LBO, SBO), ID_KM, 1u);
                }
                mma_commit(&tfull[a]);
                if (u + 1 == u_end || cur.tile + 1 == p.ntile) mma_commit(gw_empty);   // the item's last tile
            }
            mma_commit(final_bar);
            mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        // thread (n, half): token row n (TMEM lane n), columns [64 half, 64 half + 64)
        const int et = tid - 64;                 // 0..255
        const int half = et >> 7;
        const int n = (warp & 3) * 32 + lane;
        const uint32_t trow_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        // 8 bf16 of row n of a K-major token tile, columns c..c+7 (c % 8 == 0)
        auto row8 = [&](const uint8_t* tilep, int c, float* x) {
            const int cc = c & 63;
            const uint4 w = *reinterpret_cast<const uint4*>(tilep + (c >> 6) * BOX + n * 128 +
                                                            (((cc >> 3) ^ (n & 7)) << 4));
            const uint32_t* ws = reinterpret_cast<const uint32_t*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
                x[2 * e] = f2.x;
                x[2 * e + 1] = f2.y;
            }
        };
        TileCursor cur(u_begin, p.ntile, p.H);
        for (long long u = u_begin; u < u_end; ++u, cur.next(p.ntile, p.H)) {
            const long long i = u - u_begin;
            const int s = static_cast<int>(i % KV_STAGES), a = static_cast<int>(i & 1);
            const int tile = cur.tile;
            const int f = cur.f, h = cur.h;
            // both halves decide together: the named barrier below is never left waiting
            const bool ok = bar_and(1, TOKEN_EPI,
                                    mbar_wait(&tfull[a], static_cast<uint32_t>((i >> 1) & 1), p.wait_limit_ns,
                                              abort_flag));
            if (!ok) break;
            tc_fence_after();
            const uint8_t* sK = ring + s * 2 * TILE;
            const uint8_t* sV = sK + TILE;
            const int token = tile * 128 + n;
            const bool valid = token < p.N;
            const size_t th = (static_cast<size_t>(f) * p.N + (valid ? token : 0)) * p.H + h;
            const float bn = valid ? p.beta[th] : 0.0f;
            const uint32_t trow = tmem_base + a * 256 + trow_off;
            float dbeta = 0.0f;
            // dk = beta T12, dbeta += T12 . k / 2
            for (int c0 = 64 * half; c0 < p.dk && c0 < 64 * half + 64; c0 += 32) {
                uint32_t t[32];
                tmem_ld32(trow + c0, t);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float kx[8];
                    row8(sK, c0 + 8 * q8, kx);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float a0 = __uint_as_float(t[8 * q8 + e]), a1 = __uint_as_float(t[8 * q8 + e + 1]);
                        dbeta += 0.5f * (a0 * kx[e] + a1 * kx[e + 1]);
                        pk[(8 * q8 + e) / 2] = pack_bf16x2(bn * a0, bn * a1);
                    }
                }
                if (valid) {
                    __nv_bfloat16* dst = p.dk_out + th * p.dk + c0;
                    for (int q4 = 0; q4 < 4; ++q4)
                        if (c0 + 8 * q4 < p.dk)
                            *reinterpret_cast<uint4*>(dst + 8 * q4) =
                                make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                }
            }
            // dv = beta T3, dbeta += T3 . v / 2
            for (int c0 = 64 * half; c0 < p.dv && c0 < 64 * half + 64; c0 += 32) {
                uint32_t t[32];
                tmem_ld32(trow + 128 + c0, t);
                tmem_wait_ld();
                uint32_t pv[16];
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float vx[8];
                    row8(sV, c0 + 8 * q8, vx);
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        const float a0 = __uint_as_float(t[8 * q8 + e]), a1 = __uint_as_float(t[8 * q8 + e + 1]);
                        dbeta += 0.5f * (a0 * vx[e] + a1 * vx[e + 1]);
                        pv[(8 * q8 + e) / 2] = pack_bf16x2(bn * a0, bn * a1);
                    }
                }
                if (valid) {
                    __nv_bfloat16* dst = p.dv_out + th * p.dv + c0;
                    for (int q4 = 0; q4 < 4; ++q4)
                        if (c0 + 8 * q4 < p.dv)
                            *reinterpret_cast<uint4*>(dst + 8 * q4) =
                                make_uint4(pv[4 * q4], pv[4 * q4 + 1], pv[4 * q4 + 2], pv[4 * q4 + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[a]);
            mbar_arrive(&kempty[s]);
            if (half == 1) dbh[a * 128 + n] = dbeta;
            named_bar_sync(1, TOKEN_EPI);
            if (half == 0 && valid) p.d_beta[th] = dbeta + dbh[a * 128 + n];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace bwd
}  // namespace gdn
