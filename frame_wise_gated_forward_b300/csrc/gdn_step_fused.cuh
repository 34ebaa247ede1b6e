// gdn_step_fused.cuh -- one frame of the frame-wise GDN forward on a resident
// state in a single launch (the interactive step: the pipeline advances by
// one latent frame at a time, WorldFoundry model card "What it is for").
//
// One thread-block cluster of CS = 4 CTAs per (b, h) head.  The frame's
// contraction D = K^T B [K | V] (dk x (dk + dv)) is split by its columns, not
// by tokens, so no CTA ever adds another CTA's partial sums:
//   CTA 0, 1: columns [64 r, 64 r + 64) of A = K^T B K   (B operand: K box r)
//   CTA 2, 3: rows [64 (r-2), + 64) of U = V^T B K        (B operand: V box r-2)
// each over all N tokens of the frame (a 4-deep ring of 64-token chunks; the
// U CTAs' state-row loads are issued before it and used after it).  The MMA's
// A operand is the raw K tile; each CTA scales only its own 64 B-operand
// columns by beta (the fp32 product rounded once to bf16), so the rounding
// sits on the other factor than in phase 1 -- the same sum to bf16 accuracy.
// Then
//   - CTAs 0 and 1 write their columns of A (bf16) into CTAs 2 and 3's copy of
//     A through distributed shared memory (A is symmetric: row = column);
//   - CTAs 2 and 3 advance their 64 state rows, S <- alpha (S - S A) + U, with
//     one tcgen05 MMA (M = 128, N = 64), write state_out, and send the rows
//     (bf16) into every CTA's copy of S;
//   - every CTA computes o_n = S q_n for a quarter of the frame's 128-token
//     tiles, staged in shared memory and written by a TMA store.
// Nothing but the inputs, the state and the outputs touches HBM, and every
// sum is taken in one accumulator in token order, as in phase 1.
//
// The cluster barriers are executed by every thread of every CTA exactly the
// same number of times on every path: a bounded wait that gives up only marks
// the CTA as failed (GDN_ERR_TIMEOUT is recorded) and skips the work that
// depends on it.  160 threads: warps 0-3 (thread j is TMEM lane j) scale the
// B operand and run every later phase; warp 4's first lane issues the
// contraction's ring loads and MMAs, so a chunk's MMAs and the refill of its
// stage overlap the scaling of the next chunk (mbarriers, no block barrier).
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace step {

// Programmatic dependent launch: wait until the grids this one depends on in
// the stream have completed and their memory is visible (a no-op for a grid
// launched without the programmatic-serialization attribute), and let the
// next such grid in the stream be scheduled before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int CS = 4;                       // CTAs per cluster (one head)
constexpr int NWORK = 128;                  // warps 0-3
constexpr int THREADS = NWORK + 32;         // + the contraction's issuer warp
constexpr int CHUNK = 64;                   // tokens per ring stage
constexpr int NST = 4;                      // ring depth
constexpr int NBK = 2;                      // scaled B boxes in flight (workers run up to NBK chunks ahead of the MMAs)
constexpr int KBOX = CHUNK * 128;           // 64 token rows x 128 B
constexpr int STAGE = 3 * KBOX;             // K box 0 | K box 1 | this CTA's V box
constexpr int QBOX = 128 * 128;             // 128 rows x 128 B
constexpr int TILE = 2 * QBOX;              // 128 x 128 bf16, K-major
constexpr int SR = 64;                      // state rows per scan CTA
constexpr int SRBOX = SR * 128;
// shared memory, in order (1024-byte aligned pieces)
constexpr int OFF_RING = 0;                              // [NST] stages; later two q tiles
constexpr int OFF_OSTG = OFF_RING + 2 * TILE;            // (after the contraction) output staging tile;
                                                         // before it, the scan CTA's fp32 state rows
constexpr int OFF_BK = OFF_RING + NST * STAGE;           // [NBK] beta-scaled B boxes (64 rows x 64 columns)
constexpr int OFF_A = OFF_BK + NBK * KBOX;               // A, K-major 128 x 128 (scan CTAs)
constexpr int OFF_S = OFF_A + TILE;                      // S after the frame, K-major 128 x 128
constexpr int OFF_SIMG = OFF_S + TILE;                   // scan CTA's 64 rows of S before the frame, K-major
constexpr int OFF_BETA = OFF_SIMG + 2 * SRBOX;           // per-thread beta rings of the contraction
constexpr int BETA_BYTES = 4096;
constexpr int BETA_AHEAD = 4;                            // beta copies in flight per thread
static_assert((BETA_AHEAD + 1) * NWORK * 4 <= BETA_BYTES, "beta rings");
constexpr int OFF_BAR = OFF_BETA + BETA_BYTES;
constexpr int NBARS = 2 * NST + 2 + 2 * 2 + 2 * NBK;     // full, empty; d, c; qfull, o_bar; bk_empty, scaled
constexpr int BAR_BYTES = 256;                           // the barriers, the TMEM address and the abort flag
static_assert(NBARS * 8 + 8 <= BAR_BYTES, "barrier area");
constexpr size_t SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES;
static_assert(NST * STAGE >= 3 * TILE, "two q tiles and the output staging tile fit in the ring");
static_assert(SR * 128 * 4 <= TILE, "the fp32 state rows fit in the output staging tile");
static_assert(SMEM_BYTES <= 232448, "shared memory");
// TMEM columns
constexpr uint32_t T_D = 0;                 // 64: this CTA's columns of D
constexpr uint32_t T_C = 64;                // 64: S_rows A (scan CTAs)
constexpr uint32_t T_S = 128;               // 64: the scan CTA's fp32 state rows before the frame
constexpr uint32_t T_O = 256;               // [2] x 128: Q S^T

struct Params {
    const float* alpha;     // [B, H]
    const float* beta;      // [B, N, H]
    const float* state_in;  // [B, H, dv, dk] or nullptr
    float* state_out;       // [B, H, dv, dk] or nullptr
    int H, N, dk, dv;
    unsigned long long wait_limit_ns;
};

// byte offset of bf16 element (row, col) in a K-major, 128-byte-swizzled tile
// whose 64-column boxes hold `box_bytes` each
__device__ __forceinline__ uint32_t kmaj(int row, int col, int box_bytes) {
    return (col >> 6) * box_bytes + row * 128 + (((((col & 63) >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

// tm_k, tm_v: [B, N, H, d] token tensors, box (64, 1, 64, 1); tm_q, tm_o: box (64, 1, 128, 1);
// tm_s: state_out as [B H, dv, dk] fp32, box (128, 64, 1), unswizzled (unused when state_out is null)
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(THREADS, 1)
    step_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                const __grid_constant__ CUtensorMap tm_s, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;                  // [NST] stage landed
    uint64_t* empty = full + NST;           // [NST] the stage's MMAs retired
    uint64_t* bk_empty = empty + NST;       // [NBK] the scaled box's MMAs retired
    uint64_t* d_bar = bk_empty + NBK;       // every contraction MMA retired
    uint64_t* c_bar = d_bar + 1;            // scan MMA retired
    uint64_t* qfull = c_bar + 1;            // [2] q tile landed
    uint64_t* o_bar = qfull + 2;            // [2] output MMA retired
    uint64_t* scaled = o_bar + 2;           // [NBK] every worker has written its part of the scaled box
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(scaled + NBK);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5;
    const bool worker = tid < NWORK;   // owns TMEM lane tid
    const bool issuer = tid == NWORK;  // contraction loads and MMAs
    const int rank = static_cast<int>(cluster_ctarank());
    const bool scan_cta = rank >= 2;
    const int bh = blockIdx.x / CS;
    const int b = bh / p.H, h = bh % p.H;
    const int C = (p.N + CHUNK - 1) / CHUNK;
    const int kb = p.dk > 64 ? 2 : 1, vb = p.dv > 64 ? 2 : 1;
    const bool vload = scan_cta && rank - 2 < vb;          // this CTA's V box exists
    const uint32_t sbase = smem_u32(smem);
    const int j = tid;
    const int i0 = (rank - 2) * SR;                        // scan CTAs: first state row
    const size_t soff = (static_cast<size_t>(b) * p.H + h) * p.dv * p.dk;

    // ring boxes that are never loaded must read as zero: with dk <= 64 (no k
    // box 1) or a U CTA without a v box, clear the ring and the scaled boxes
    // once (A, S and the state images are always written whole)
    if (kb == 1 || (scan_cta && !vload))
        for (int i = tid; i < OFF_A / 16; i += THREADS) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&qfull[x], 1);
            mbar_init(&o_bar[x], 1);
        }
        for (int x = 0; x < NBK; ++x) {
            mbar_init(&bk_empty[x], 1);
            mbar_init(&scaled[x], NWORK);
        }
        mbar_init(d_bar, 1);
        mbar_init(c_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_o);
        if (p.state_out != nullptr) prefetch_tmap(&tm_s);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Everything above touches no global memory, so with programmatic launch
    // it overlaps the end of the previous step; every global access comes
    // after the wait (the previous grid may have written this step's inputs).
    griddep_wait();
    griddep_launch_dependents();
    const float af = p.alpha[static_cast<size_t>(b) * p.H + h];
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);   // workers only
    bool good = true;
    int loads_issued = 0;   // issuer: ring loads issued (for the drain)

    auto load_chunk = [&](int c) {   // issuer
        const int s = c % NST;
        uint8_t* st = smem + OFF_RING + s * STAGE;
        mbar_arrive_expect_tx(&full[s], (kb + (vload ? 1 : 0)) * KBOX);
        for (int bx = 0; bx < kb; ++bx) tma_load_4d(st + bx * KBOX, &tm_k, &full[s], 64 * bx, h, c * CHUNK, b);
        if (vload) tma_load_4d(st + 2 * KBOX, &tm_v, &full[s], 64 * (rank - 2), h, c * CHUNK, b);
        ++loads_issued;
    };
    if (issuer)
        for (int c = 0; c < NST && c < C; ++c) load_chunk(c);

    // scan CTAs: their state rows before the frame, loaded now (all 64 loads in
    // flight, addresses clamped into the matrix) and used after the
    // contraction, so the loads' latency hides behind it
    const bool load_state = scan_cta && worker && p.state_in != nullptr;
    uint32_t sv[SR];
    if (load_state) {
        const int jc = j < p.dk ? j : p.dk - 1;
#pragma unroll
        for (int t = 0; t < SR; ++t) {
            const int ic = i0 + t < p.dv ? i0 + t : p.dv - 1;
            sv[t] = __float_as_uint(p.state_in[soff + static_cast<size_t>(ic) * p.dk + jc]);
        }
    }

    // ------------------------------------------------ 1. the contraction slice
    constexpr uint32_t ID_D = idesc_bf16(128, 64, 1, 1);
    int c_done = 0;          // workers: chunks scaled; issuer: chunks whose MMAs were issued
    bool d_issued = false;   // issuer: the final commit of the contraction
    if (worker) {
        // thread pair (2 row, 2 row + 1): token row `row` of the chunk, 16-byte
        // pieces 4 half .. 4 half + 3 of this CTA's B box
        const int row = tid >> 1, half = tid & 1;
        // beta of this thread's token row: a per-thread ring in shared memory
        // filled by cp.async BETA_AHEAD chunks ahead (each thread reads back
        // only what it copied), so no global-load latency sits inside a chunk
        float* beta_ring = reinterpret_cast<float*>(smem + OFF_BETA);
        int pslot = 0, cslot = 0;
        auto beta_prefetch = [&](int c) {
            float* dst = beta_ring + pslot * NWORK + tid;
            const int tok = c * CHUNK + row;
            if (c < C && tok < p.N)
                cp_async_4(dst, p.beta + (static_cast<size_t>(b) * p.N + tok) * p.H + h);
            else
                *dst = 0.0f;
            cp_async_commit();
            if (++pslot == BETA_AHEAD + 1) pslot = 0;
        };
        for (int c = 0; c < BETA_AHEAD; ++c) beta_prefetch(c);
        for (int c = 0; c < C; ++c) {
            const int s = c % NST, bkb = c % NBK;
            beta_prefetch(c + BETA_AHEAD);
            cp_async_wait<BETA_AHEAD>();   // this chunk's copy has landed
            const float bval = beta_ring[cslot * NWORK + tid];
            if (++cslot == BETA_AHEAD + 1) cslot = 0;
            if (!mbar_wait(&full[s], static_cast<uint32_t>((c / NST) & 1), p.wait_limit_ns, abort_flag) ||
                (c >= NBK &&
                 !mbar_wait(&bk_empty[bkb], static_cast<uint32_t>(((c / NBK) - 1) & 1), p.wait_limit_ns, abort_flag))) {
                good = false;
                break;
            }
            c_done = c + 1;
            // B box of this CTA: K box `rank` or its V box (a box never loaded is zero)
            const uint8_t* src = smem + OFF_RING + s * STAGE + (scan_cta ? 2 : rank) * KBOX + row * 128;
            uint8_t* dst = smem + OFF_BK + bkb * KBOX + row * 128;
            // pieces rotated by the row: the 8 threads of a quarter-warp touch 8
            // different 16-byte bank groups; all loads issue before any store
            uint4 x[4];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) x[c4] = *reinterpret_cast<const uint4*>(src + (((c4 + 4 * half + row) & 7) << 4));
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const uint32_t* xs = reinterpret_cast<const uint32_t*>(&x[c4]);
                uint32_t y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
                    y[e] = pack_bf16x2(f2.x * bval, f2.y * bval);   // fp32 product rounded once
                }
                *reinterpret_cast<uint4*>(dst + (((c4 + 4 * half + row) & 7) << 4)) = make_uint4(y[0], y[1], y[2], y[3]);
            }
            fence_proxy_async_smem();   // the scaled pieces are visible to the MMA
            mbar_arrive(&scaled[bkb]);
        }
        cp_async_wait<0>();   // no beta copy outlives the loop
        // scan CTAs: the state rows -- fp32 into TMEM (lane j, column T_S + r)
        // for the update, bf16 image in shared memory for S A (zero outside
        // dv x dk, and for a null state_in)
        if (scan_cta) {
#pragma unroll
            for (int r0 = 0; r0 < SR; r0 += 16) {
                uint32_t w[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    w[t] = (load_state && j < p.dk && i0 + r0 + t < p.dv) ? sv[r0 + t] : 0u;
                    *reinterpret_cast<__nv_bfloat16*>(smem + OFF_SIMG + kmaj(r0 + t, j, SRBOX)) =
                        __float2bfloat16_rn(__uint_as_float(w[t]));
                }
                tmem_st16(tlane + T_S + r0, w);
            }
            tmem_wait_st();
        }
    } else if (issuer) {
        for (int c = 0; c < C; ++c) {
            const int s = c % NST, bkb = c % NBK;
            if (!mbar_wait(&scaled[bkb], static_cast<uint32_t>((c / NBK) & 1), p.wait_limit_ns, abort_flag)) {
                good = false;
                break;
            }
            tc_fence_after();
            // A: the raw K tile (both boxes); B: this CTA's scaled 64 columns
            const uint32_t a_base = sbase + OFF_RING + s * STAGE;
            const uint32_t b_base = sbase + OFF_BK + bkb * KBOX;
            for (int kk = 0; kk < CHUNK / 16; ++kk)
                mma_bf16(tmem + T_D, smem_desc(a_base + kk * 2048, KBOX, 1024), smem_desc(b_base + kk * 2048, KBOX, 1024),
                         ID_D, (c > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
            mma_commit(&bk_empty[bkb]);
            c_done = c + 1;
            // refill the previous chunk's stage (its MMAs have most likely retired by now)
            if (c >= 1 && c - 1 + NST < C) {
                if (!mbar_wait(&empty[(c - 1) % NST], static_cast<uint32_t>(((c - 1) / NST) & 1), p.wait_limit_ns,
                               abort_flag)) {
                    good = false;
                    break;
                }
                load_chunk(c - 1 + NST);
            }
        }
        mma_commit(d_bar);   // tracks every contraction MMA issued, also after a given-up wait
        d_issued = true;
    }
    good = good && mbar_wait(d_bar, 0, p.wait_limit_ns, abort_flag);
    good = __syncthreads_and(good);
    tc_fence_after();

    // q tiles of this CTA's quarter of the tokens into the (now idle) ring
    const int ntiles = (p.N + 127) / 128;
    const int tile0 = (rank * ntiles) / CS, nq = ((rank + 1) * ntiles) / CS - tile0;
    int q_issued = 0;   // thread 0
    if (tid == 0 && good)
        for (int t = 0; t < nq && t < 2; ++t) {
            mbar_arrive_expect_tx(&qfull[t], kb * QBOX);
            for (int bx = 0; bx < kb; ++bx)
                tma_load_4d(smem + OFF_RING + t * TILE + bx * QBOX, &tm_q, &qfull[t], 64 * bx, h, (tile0 + t) * 128, b);
            ++q_issued;
        }

    // ------------------------------------------ 2. A columns to the scan CTAs
    if (!scan_cta && worker) {
        // thread j: row j of D = A[j][64 rank .. + 63] = A[64 rank .. + 63][j] (A symmetric);
        // both TMEM loads in flight before the one wait (a TMEM load's latency
        // is long next to the work between loads)
        uint32_t v[64];
        if (good) {
            tmem_ld32(tlane + T_D, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tlane + T_D + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int t = 0; t < 64; ++t) v[t] = 0u;
        }
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
            const uint4 w = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * q8 + 0]), __uint_as_float(v[8 * q8 + 1])),
                pack_bf16x2(__uint_as_float(v[8 * q8 + 2]), __uint_as_float(v[8 * q8 + 3])),
                pack_bf16x2(__uint_as_float(v[8 * q8 + 4]), __uint_as_float(v[8 * q8 + 5])),
                pack_bf16x2(__uint_as_float(v[8 * q8 + 6]), __uint_as_float(v[8 * q8 + 7])));
            const uint32_t o = sbase + OFF_A + kmaj(j, 64 * rank + 8 * q8, QBOX);
            st_dsmem_v4(mapa_shared(o, 2), w);
            st_dsmem_v4(mapa_shared(o, 3), w);
        }
    }
    fence_proxy_async_cluster();
    cluster_sync();  // ---------------------------------------------- (1) A complete in CTAs 2, 3

    // -------------------------------------------------- 3. the state rows
    if (scan_cta) {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && good) {
            tc_fence_after();
            constexpr uint32_t ID_C = idesc_bf16(128, SR, 0, 0);
            const int nk = (p.dk + 15) / 16;
            for (int kk = 0; kk < nk; ++kk)
                mma_bf16(tmem + T_C, smem_desc(sbase + OFF_A + (kk >> 2) * QBOX + (kk & 3) * 32, 16, 1024),
                         smem_desc(sbase + OFF_SIMG + (kk >> 2) * SRBOX + (kk & 3) * 32, 16, 1024), ID_C,
                         kk > 0 ? 1u : 0u);
            mma_commit(c_bar);
        }
        if (good) good = mbar_wait(c_bar, 0, p.wait_limit_ns, abort_flag);
        good = __syncthreads_and(good);
        tc_fence_after();
        // thread j, rows i0 + r: S' = alpha (S - C[j][r]) + U[r][j], U = D column r,
        // into fp32 staging rows (zero outside dv x dk); state_out by one TMA store
        float* fstg = reinterpret_cast<float*>(smem + OFF_OSTG);
        const bool col_ok = j < p.dk;
        for (int r0 = 0; r0 < SR && worker; r0 += 32) {   // 32 rows: three TMEM loads, one wait
            uint32_t cc[32], uu[32], so[32];
            tmem_ld32(tlane + T_S + r0, so);
            if (good) {
                tmem_ld32(tlane + T_C + r0, cc);
                tmem_ld32(tlane + T_D + r0, uu);
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) cc[t] = uu[t] = 0u;
            }
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float sn = af * (__uint_as_float(so[t]) - __uint_as_float(cc[t])) + __uint_as_float(uu[t]);
                fstg[(r0 + t) * 128 + j] = (col_ok && i0 + r0 + t < p.dv) ? sn : 0.0f;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && good && p.state_out != nullptr && i0 < p.dv) {   // rows past dv, columns past dk clipped
            tma_store_3d(&tm_s, fstg, 0, i0, b * p.H + h);
            bulk_commit();
        }
        // this CTA's 64 rows of the state, rounded to bf16, into every CTA's copy of S
        for (int k = tid; k < SR * 16; k += THREADS) {
            const int rr = k / 16, ch = k % 16;   // 16 pieces of 8 columns per row
            const float4 f0 = *reinterpret_cast<const float4*>(fstg + rr * 128 + ch * 8);
            const float4 f1 = *reinterpret_cast<const float4*>(fstg + rr * 128 + ch * 8 + 4);
            const uint4 w = make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f0.z, f0.w), pack_bf16x2(f1.x, f1.y),
                                       pack_bf16x2(f1.z, f1.w));
            const uint32_t o = sbase + OFF_S + kmaj(i0 + rr, ch * 8, QBOX);
            for (int q = 0; q < CS; ++q) st_dsmem_v4(mapa_shared(o, q), w);
        }
    }
    fence_proxy_async_cluster();
    cluster_sync();  // ---------------------------------------------- (2) S complete everywhere
    fence_proxy_async_smem();

    // ------------------------------------------------------- 4. the outputs
    int q_done = 0;
    for (int t = 0; t < nq; ++t) {
        const int x = t & 1;
        if (t >= 2 && tid == 0 && good) {  // the tile two back has been consumed: refill its buffer
            mbar_arrive_expect_tx(&qfull[x], kb * QBOX);
            for (int bx = 0; bx < kb; ++bx)
                tma_load_4d(smem + OFF_RING + x * TILE + bx * QBOX, &tm_q, &qfull[x], 64 * bx, h, (tile0 + t) * 128, b);
            ++q_issued;
        }
        if (good) good = mbar_wait(&qfull[x], static_cast<uint32_t>((t >> 1) & 1), p.wait_limit_ns, abort_flag);
        good = __syncthreads_and(good);
        if (!good) break;
        q_done = t + 1;
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID_O = idesc_bf16(128, 128, 0, 0);
            const int nk = (p.dk + 15) / 16;
            for (int kk = 0; kk < nk; ++kk) {
                const uint32_t ko = (kk >> 2) * QBOX + (kk & 3) * 32;
                mma_bf16(tmem + T_O + x * 128, smem_desc(sbase + OFF_RING + x * TILE + ko, 16, 1024),
                         smem_desc(sbase + OFF_S + ko, 16, 1024), ID_O, kk > 0 ? 1u : 0u);
            }
            mma_commit(&o_bar[x]);
        }
        good = mbar_wait(&o_bar[x], static_cast<uint32_t>((t >> 1) & 1), p.wait_limit_ns, abort_flag);
        good = __syncthreads_and(good);
        if (!good) break;
        tc_fence_after();
        // the previous store out of the staging tile (a tile's outputs, or the
        // state rows) has finished reading it
        if (tid == 0) bulk_wait_read<0>();
        __syncthreads();
        // thread j: token row j of the tile, bf16, into the swizzled staging boxes
        for (int c0 = 0; c0 < p.dv && worker; c0 += 64) {   // 64 columns: two TMEM loads, one wait
            uint32_t v[64];
            tmem_ld32(tlane + T_O + x * 128 + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tlane + T_O + x * 128 + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_wait_ld();
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8)
                *reinterpret_cast<uint4*>(smem + OFF_OSTG + kmaj(j, c0 + 8 * q8, QBOX)) = make_uint4(
                    pack_bf16x2(__uint_as_float(v[8 * q8 + 0]), __uint_as_float(v[8 * q8 + 1])),
                    pack_bf16x2(__uint_as_float(v[8 * q8 + 2]), __uint_as_float(v[8 * q8 + 3])),
                    pack_bf16x2(__uint_as_float(v[8 * q8 + 4]), __uint_as_float(v[8 * q8 + 5])),
                    pack_bf16x2(__uint_as_float(v[8 * q8 + 6]), __uint_as_float(v[8 * q8 + 7])));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();  // buffer x and its accumulator are reused two tiles on
        if (tid == 0) {   // tokens past N and columns past dv are clipped by the store
            for (int bx = 0; bx < vb; ++bx)
                tma_store_4d(&tm_o, smem + OFF_OSTG + bx * QBOX, 64 * bx, h, (tile0 + t) * 128, b);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait<0>();   // the output stores are complete before the CTA leaves
    // copies or MMAs of a given-up wait must land before the CTA leaves
    if (issuer && !good) {
        for (int k = c_done; k < loads_issued; ++k)
            mbar_wait_drain(&full[k % NST], static_cast<uint32_t>((k / NST) & 1), p.wait_limit_ns);
        if (d_issued) mbar_wait_drain(d_bar, 0, p.wait_limit_ns);
    }
    if (tid == 0 && !good) {
        for (int k = q_done; k < q_issued; ++k)
            mbar_wait_drain(&qfull[k & 1], static_cast<uint32_t>((k >> 1) & 1), p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    cluster_sync();  // no CTA leaves while another may still address its shared memory
}

}  // namespace step
}  // namespace gdn
