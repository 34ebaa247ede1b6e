// gdn_step_fused.cuh -- one frame of the frame-wise GDN forward on a resident
// state in a single launch (the interactive step: the pipeline advances by
// one latent frame at a time, WorldFoundry model card "What it is for").
//
// One thread-block cluster of CS CTAs per (b, h) head; CTA r of the
// cluster owns token chunks [r C / CS, (r + 1) C / CS) of the frame (C chunks
// of 64 tokens, at most two per CTA) and state rows [16 r, 16 r + 16).
//   1. D_r = (beta K)^T [K | V] over its tokens on tcgen05 (TMEM, fp32), as
//      phase 1 does for a whole frame;
//   2. the CTAs reduce the partial sums through distributed shared memory in
//      a fixed rank order: CTA r sums rows [16 r, 16 r + 16) of A and sends
//      them (bf16) into every CTA's copy of A; then it sums its rows of U;
//   3. its state rows: S_r <- alpha (S_r - S_r A) + U_r (one tcgen05 MMA,
//      M = 128, N = 16), written to state_out and, as bf16, into every CTA's
//      copy of S;
//   4. o_n = S q_n for its tokens (tcgen05, M = 128 tokens, N = dv), bf16.
// No workspace: nothing but the inputs, state and outputs touches HBM.
//
// The cluster barriers are executed by every thread of every CTA exactly the
// same number of times on every path: a bounded wait that gives up only marks
// the CTA as failed (GDN_ERR_TIMEOUT is recorded) and skips the work that
// depended on it.  128 threads; thread j is TMEM lane j.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace step {

constexpr int CS = 8;                       // CTAs per cluster (one head)
constexpr int THREADS = 128;
constexpr int CHUNK = 64;                   // tokens per contraction chunk
constexpr int MAX_CHUNKS = 2 * CS;          // frames of up to 1024 tokens
constexpr int KBOX = CHUNK * 128;           // 64 rows x 128 B
constexpr int KTILE = 2 * KBOX;             // 64 tokens x 128 columns, bf16
constexpr int QBOX = 128 * 128;             // 128 rows x 128 B
constexpr int QTILE = 2 * QBOX;             // 128 x 128 bf16
constexpr int SROWS = 16;                   // state rows per CTA
constexpr int SBOX = SROWS * 128;
// shared memory, in order
constexpr int OFF_KV = 0;                               // [2][K tile | V tile]; then fp32 partials [128][128]
constexpr int OFF_BK = OFF_KV + 4 * KTILE;              // [2] beta*K tiles
constexpr int OFF_Q = OFF_BK + 2 * KTILE;               // q tile, K-major (128 tokens)
constexpr int OFF_A = OFF_Q + QTILE;                    // A, K-major (128 x 128)
constexpr int OFF_S = OFF_A + QTILE;                    // S after the frame, K-major (128 x 128)
constexpr int OFF_SIMG = OFF_S + QTILE;                 // this CTA's rows of S before the frame, K-major
constexpr int OFF_SROW = OFF_SIMG + 2 * SBOX;           // this CTA's rows of S after the frame, row-major bf16
constexpr int OFF_BAR = OFF_SROW + SROWS * 128 * 2;
constexpr size_t SMEM_BYTES = 1024 + OFF_BAR + 64;
static_assert(4 * KTILE >= 128 * 128 * 4, "the partial sums fit in the K/V region");
static_assert(SMEM_BYTES <= 232448, "shared memory");
// TMEM columns
constexpr uint32_t T_D = 0;                 // 256: A part [0, 128), U part [128, 256)
constexpr uint32_t T_C = 256;               // 16: S_r A
constexpr uint32_t T_O = 384;               // 128: Q S^T

struct Params {
    const float* alpha;     // [B, H]
    const float* beta;      // [B, N, H]
    const float* state_in;  // [B, H, dv, dk] or nullptr
    float* state_out;       // [B, H, dv, dk] or nullptr
    __nv_bfloat16* out;     // [B, N, H, dv]
    int H, N, dk, dv;
    int chunks;             // ceil(N / 64) <= MAX_CHUNKS
    unsigned long long wait_limit_ns;
};

// byte offset of bf16 element (row, col) in a K-major, 128-byte-swizzled tile
// whose 64-column boxes hold `box_bytes` each
__device__ __forceinline__ uint32_t kmaj(int row, int col, int box_bytes) {
    return (col >> 6) * box_bytes + row * 128 + (((((col & 63) >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

// tm_k, tm_v: [B, N, H, d] token tensors, box (64, 1, 64, 1); tm_q: box (64, 1, 128, 1)
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(THREADS, 1)
    step_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_q, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* ld_bar = bars;
    uint64_t* mma_bar = bars + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int rank = static_cast<int>(cluster_ctarank());
    const int bh = blockIdx.x / CS;
    const int b = bh / p.H, h = bh % p.H;
    const int c_begin = (rank * p.chunks) / CS, c_end = ((rank + 1) * p.chunks) / CS;
    const int nch = c_end - c_begin;                       // 0, 1 or 2
    const int t0 = c_begin * CHUNK;
    const int t1 = min(c_end * CHUNK, p.N);
    const int kb = p.dk > 64 ? 2 : 1, vb = p.dv > 64 ? 2 : 1;
    const uint32_t sbase = smem_u32(smem);

    // boxes that are never loaded (d <= 64) must read as zero in the contraction's
    // operands; the A, S and S-row tiles are written whole before they are read
    if (kb < 2 || vb < 2)
        for (int i = tid; i < OFF_Q / 16; i += THREADS) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(ld_bar, 1);
        mbar_init(mma_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool good = true;
    uint32_t mma_phase = 0;
    bool mma_pending = false;   // thread 0: a commit not yet waited for

    // ------------------------------------------------------------- loads
    if (tid == 0 && nch > 0) {
        mbar_arrive_expect_tx(ld_bar, nch * (kb + vb) * KBOX + kb * QBOX);
        for (int c = 0; c < nch; ++c) {
            uint8_t* kv = smem + OFF_KV + c * 2 * KTILE;
            const int tok = (c_begin + c) * CHUNK;
            for (int bx = 0; bx < kb; ++bx) tma_load_4d(kv + bx * KBOX, &tm_k, ld_bar, 64 * bx, h, tok, b);
            for (int bx = 0; bx < vb; ++bx) tma_load_4d(kv + KTILE + bx * KBOX, &tm_v, ld_bar, 64 * bx, h, tok, b);
        }
        for (int bx = 0; bx < kb; ++bx) tma_load_4d(smem + OFF_Q + bx * QBOX, &tm_q, ld_bar, 64 * bx, h, t0, b);
    }
    // thread r: token t0 + r (beta), and column j = tid of this CTA's state rows
    const int r = tid;
    const bool tok_ok = nch > 0 && t0 + r < t1;
    const float bval = tok_ok ? p.beta[(static_cast<size_t>(b) * p.N + t0 + r) * p.H + h] : 0.0f;
    const float af = p.alpha[static_cast<size_t>(b) * p.H + h];
    const int j = tid;
    const int i0 = rank * SROWS;                            // this CTA's state rows
    const size_t soff = (static_cast<size_t>(b) * p.H + h) * p.dv * p.dk;
    float S[SROWS];
#pragma unroll
    for (int rr = 0; rr < SROWS; ++rr) {
        const bool v = p.state_in != nullptr && j < p.dk && i0 + rr < p.dv;
        S[rr] = v ? p.state_in[soff + static_cast<size_t>(i0 + rr) * p.dk + j] : 0.0f;
    }
    // image of this CTA's rows of S (before the frame): B operand of S_r A
#pragma unroll
    for (int rr = 0; rr < SROWS; ++rr)
        *reinterpret_cast<__nv_bfloat16*>(smem + OFF_SIMG + kmaj(rr, j, SBOX)) = __float2bfloat16_rn(S[rr]);

    if (nch > 0) good = mbar_wait(ld_bar, 0, p.wait_limit_ns, abort_flag);
    good = __syncthreads_and(good);

    // ------------------------------------------------- 1. partial contraction
    if (good && nch > 0) {
        // thread r scales token row r (chunk r / 64, row r % 64) by beta into the beta*K tile
        if (r < nch * CHUNK) {
            const int c = r / CHUNK, rw = r % CHUNK;
            const uint8_t* src = smem + OFF_KV + c * 2 * KTILE + rw * 128;
            uint8_t* dst = smem + OFF_BK + c * KTILE + rw * 128;
            for (int bx = 0; bx < kb; ++bx)
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 x = *reinterpret_cast<const uint4*>(src + bx * KBOX + ch * 16);
                    const uint32_t* xs = reinterpret_cast<const uint32_t*>(&x);
                    uint32_t y[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
                        y[e] = pack_bf16x2(f2.x * bval, f2.y * bval);   // fp32 product rounded once
                    }
                    *reinterpret_cast<uint4*>(dst + bx * KBOX + ch * 16) = make_uint4(y[0], y[1], y[2], y[3]);
                }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t ID = idesc_bf16(128, 256, 1, 1);
            for (int c = 0; c < nch; ++c) {
                const uint32_t a_base = sbase + OFF_BK + c * KTILE;
                const uint32_t b_base = sbase + OFF_KV + c * 2 * KTILE;
                for (int kk = 0; kk < CHUNK / 16; ++kk)
                    mma_bf16(tmem + T_D, smem_desc(a_base + kk * 2048, KBOX, 1024),
                             smem_desc(b_base + kk * 2048, KBOX, 1024), ID, (c > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(mma_bar);
            mma_pending = true;
        }
        good = mbar_wait(mma_bar, mma_phase, p.wait_limit_ns, abort_flag);
        if (good) {
            mma_phase ^= 1;
            mma_pending = false;
        }
        good = __syncthreads_and(good);
        tc_fence_after();
    }
    // the A part of D (row j = TMEM lane j) -> fp32 partials part[c][j] = A_r[j][c]
    // (column-major: consecutive threads write consecutive words); zeros without tokens
    float* part = reinterpret_cast<float*>(smem + OFF_KV);
    for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        if (good && nch > 0) {
            tmem_ld32(tlane + T_D + c0, v);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = 0u;
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) part[(c0 + t) * 128 + j] = __uint_as_float(v[t]);
    }
    cluster_sync();  // ---------------------------------------------- (1)

    // ---------------------------------------- 2a. A: reduce rows, share them
    // rows of the CTA's 16-row block are written to a local bf16 staging block,
    // then sent to every CTA's copy of A in 16-byte pieces
    __nv_bfloat16* blk = reinterpret_cast<__nv_bfloat16*>(smem + OFF_SROW);   // [16][128]
    auto send_rows = [&](uint32_t dst_off) {
        for (int k = tid; k < SROWS * 16; k += THREADS) {
            const int rr = k / 16, ch = k % 16;   // 16 pieces of 8 columns per row
            const uint4 w = *reinterpret_cast<const uint4*>(blk + rr * 128 + ch * 8);
            const uint32_t o = sbase + dst_off + kmaj(i0 + rr, ch * 8, QBOX);
            for (int q = 0; q < CS; ++q) st_dsmem_v4(mapa_shared(o, q), w);
        }
    };
    {
        // thread c: column c of rows i0 .. i0 + 15, i.e. part[c][i0 .. i0 + 15] of every rank, summed in order
        const int c = tid;
        float acc[SROWS];
#pragma unroll
        for (int e = 0; e < SROWS; ++e) acc[e] = 0.0f;
        const uint32_t local = sbase + OFF_KV + static_cast<uint32_t>(c * 128 + i0) * 4;
        // all 32 loads in flight at once, then the adds in rank order
        float4 x[CS][4];
#pragma unroll
        for (int q = 0; q < CS; ++q) {
            const uint32_t remote = mapa_shared(local, q);
#pragma unroll
            for (int e = 0; e < 4; ++e) x[q][e] = ld_dsmem_f32x4(remote + e * 16);
        }
#pragma unroll
        for (int q = 0; q < CS; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[4 * e] += x[q][e].x;
                acc[4 * e + 1] += x[q][e].y;
                acc[4 * e + 2] += x[q][e].z;
                acc[4 * e + 3] += x[q][e].w;
            }
#pragma unroll
        for (int e = 0; e < SROWS; ++e) blk[e * 128 + c] = __float2bfloat16_rn(acc[e]);
    }
    __syncthreads();
    send_rows(OFF_A);
    // the U part of D -> fp32 partials [i][j] (U[i][j] = D[j][128 + i]); the A
    // partials it overwrites have been read by every CTA only after barrier (2)
    fence_proxy_async_cluster();
    cluster_sync();  // ---------------------------------------------- (2)
    for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        if (good && nch > 0) {
            tmem_ld32(tlane + T_D + 128 + c0, v);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = 0u;
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) part[(c0 + t) * 128 + j] = __uint_as_float(v[t]);
    }
    cluster_sync();  // ---------------------------------------------- (3)

    // ------------------------------- 2b. U: this CTA's rows, summed in rank order
    // thread t sums row t / 8, columns 16 (t % 8) .. + 15 (16-byte remote loads)
    // into a local fp32 block; thread j then takes column j of it
    float* ured = reinterpret_cast<float*>(smem + OFF_BK);   // [16][128] (the beta*K tiles are done)
    {
        const int rr = tid / 8, col0 = (tid % 8) * 16;
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
        const uint32_t local = sbase + OFF_KV + static_cast<uint32_t>((i0 + rr) * 128 + col0) * 4;
        float4 x[CS][4];
#pragma unroll
        for (int q = 0; q < CS; ++q) {
            const uint32_t remote = mapa_shared(local, q);
#pragma unroll
            for (int e = 0; e < 4; ++e) x[q][e] = ld_dsmem_f32x4(remote + e * 16);
        }
#pragma unroll
        for (int q = 0; q < CS; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[4 * e] += x[q][e].x;
                acc[4 * e + 1] += x[q][e].y;
                acc[4 * e + 2] += x[q][e].z;
                acc[4 * e + 3] += x[q][e].w;
            }
#pragma unroll
        for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(ured + rr * 128 + col0 + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    }
    __syncthreads();
    float U[SROWS];
#pragma unroll
    for (int rr = 0; rr < SROWS; ++rr) U[rr] = ured[rr * 128 + j];

    // ------------------------------------------ 3. the state rows of this CTA
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && good) {
        tc_fence_after();
        constexpr uint32_t ID = idesc_bf16(128, SROWS, 0, 0);
        const int nk = (p.dk + 15) / 16;
        for (int kk = 0; kk < nk; ++kk) {
            const uint32_t ko = (kk >> 2) * QBOX + (kk & 3) * 32;
            const uint32_t so = (kk >> 2) * SBOX + (kk & 3) * 32;
            mma_bf16(tmem + T_C, smem_desc(sbase + OFF_A + ko, 16, 1024), smem_desc(sbase + OFF_SIMG + so, 16, 1024),
                     ID, kk > 0 ? 1u : 0u);
        }
        mma_commit(mma_bar);
        mma_pending = true;
    }
    if (good) {
        good = mbar_wait(mma_bar, mma_phase, p.wait_limit_ns, abort_flag);
        if (good) {
            mma_phase ^= 1;
            mma_pending = false;
        }
    }
    good = __syncthreads_and(good);
    tc_fence_after();
    {
        uint32_t c16[16];
        if (good) {
            tmem_ld16(tlane + T_C, c16);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) c16[t] = 0u;
        }
#pragma unroll
        for (int rr = 0; rr < SROWS; ++rr) {
            const float sn = af * (S[rr] - __uint_as_float(c16[rr])) + U[rr];
            if (good && p.state_out != nullptr && j < p.dk && i0 + rr < p.dv)
                p.state_out[soff + static_cast<size_t>(i0 + rr) * p.dk + j] = sn;
            blk[rr * 128 + j] = __float2bfloat16_rn(j < p.dk && i0 + rr < p.dv ? sn : 0.0f);
        }
    }
    __syncthreads();
    send_rows(OFF_S);   // this CTA's 16 rows of the bf16 state into every CTA's copy of S
    fence_proxy_async_cluster();
    cluster_sync();  // ---------------------------------------------- (4)
    fence_proxy_async_smem();

    // --------------------------------------------- 4. outputs of this CTA's tokens
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && good && nch > 0) {
        tc_fence_after();
        constexpr uint32_t ID = idesc_bf16(128, 128, 0, 0);
        const int nk = (p.dk + 15) / 16;
        for (int kk = 0; kk < nk; ++kk) {
            const uint32_t ko = (kk >> 2) * QBOX + (kk & 3) * 32;
            mma_bf16(tmem + T_O, smem_desc(sbase + OFF_Q + ko, 16, 1024), smem_desc(sbase + OFF_S + ko, 16, 1024), ID,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit(mma_bar);
        mma_pending = true;
    }
    if (good && nch > 0) {
        good = mbar_wait(mma_bar, mma_phase, p.wait_limit_ns, abort_flag);
        if (good) {
            mma_phase ^= 1;
            mma_pending = false;
        }
    }
    good = __syncthreads_and(good);
    tc_fence_after();
    if (good && nch > 0) {
        // thread r: output row of token t0 + r
        __nv_bfloat16* orow = p.out + ((static_cast<size_t>(b) * p.N + (tok_ok ? t0 + r : 0)) * p.H + h) * p.dv;
        for (int c0 = 0; c0 < p.dv; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tlane + T_O + c0, v);
            tmem_wait_ld();
            if (tok_ok) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    if (c0 + 8 * q8 < p.dv)
                        *reinterpret_cast<uint4*>(orow + c0 + 8 * q8) = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 0]), __uint_as_float(v[8 * q8 + 1])),
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 2]), __uint_as_float(v[8 * q8 + 3])),
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 4]), __uint_as_float(v[8 * q8 + 5])),
                            pack_bf16x2(__uint_as_float(v[8 * q8 + 6]), __uint_as_float(v[8 * q8 + 7])));
            }
        }
    }
    // a copy or MMA of a given-up wait must land before the CTA leaves
    if (tid == 0 && !good) {
        if (nch > 0) mbar_wait_drain(ld_bar, 0, p.wait_limit_ns);
        if (mma_pending) mbar_wait_drain(mma_bar, mma_phase, p.wait_limit_ns);
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
