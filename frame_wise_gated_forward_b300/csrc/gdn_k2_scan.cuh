// gdn_k2_scan.cuh -- phase 2 of the frame-wise GDN forward: the sequential
// per-head scan over latent frames
//     S_f = alpha_f * (S_{f-1} - S_{f-1} A_f) + U_f
// (SANA-WM article, "The Architecture": a fixed-size state matrix updated
// once per latent frame by a decay gate and a delta-rule correction; wispaper
// summary, "Methodology" 1: frames scanned one by one).
//
// Rows of S are independent (row i only needs row i of S_{f-1} and U_f and
// all of A_f), so the dv rows of each head are split over CTAs, R rows each,
// with no communication.  Per frame one CTA computes its slice of S A_f on
// the tensor core as C^T = A_f S_slice^T:
//     M = 128 (dk index j, zero-padded), N = R (rows of the slice), K = dk
// with both operands K-major in 128-byte-swizzled shared memory: A_f comes
// from the bf16 workspace by TMA together with the CTA's R rows of U_f
// (fp32, unswizzled) through a 4-deep prefetch ring, so no global load sits
// on the per-frame critical path; S_slice is the bf16 image of the state that
// the threads rewrite every frame.  The fp32 master
// state stays in registers: thread j (TMEM lane j) owns column j of the
// slice, which is exactly the layout tcgen05.ld returns C in.  Each frame's
// bf16 state image is also stored by TMA to the per-frame state buffer that
// phase 3 reads.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace k2 {

constexpr int THREADS = 128;
constexpr int ASTAGES = 4;
constexpr int ABOX_BYTES = 128 * 128;        // 128 rows x 128 B
constexpr int ATILE_BYTES = 2 * ABOX_BYTES;  // A_f, dk padded to 128
constexpr int TMEM_COLS = 32;

template <int R>
struct Cfg {
    static constexpr int SBOX_BYTES = R * 128;
    static constexpr int STILE_BYTES = 2 * SBOX_BYTES;
    static constexpr int UTILE_BYTES = R * 128 * 4;            // R rows x 128 fp32 (dk padded)
    static constexpr int STAGE_BYTES = ATILE_BYTES + UTILE_BYTES;
    static constexpr size_t SMEM_BYTES = 1024 + ASTAGES * STAGE_BYTES + 2 * STILE_BYTES + 256;
};

struct Params {
    const float* alpha;     // [B, F, H]
    const float* state_in;  // [B, H, dv, dk] or nullptr
    float* state_out;       // [B, H, dv, dk] or nullptr
    int H, F, dk, dv;
    int rsplit;             // dv / R CTAs per head
    unsigned long long wait_limit_ns;
};

template <int R>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&c)[R]);
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&c)[16]) { tmem_ld16(taddr, c); }
template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t (&c)[32]) { tmem_ld32(taddr, c); }

// bf16 element (r, j) of a K-major, 128-byte-swizzled [R rows x 128 cols] tile
template <int R>
__device__ __forceinline__ uint32_t sop_offset(int r, int j) {
    const int box = j >> 6, col = j & 63;
    return box * Cfg<R>::SBOX_BYTES + r * 128 + ((((col >> 3) ^ (r & 7))) << 4) + ((col & 7) << 1);
}

template <int R>
__global__ void __launch_bounds__(THREADS, 1)
    scan_kernel(const __grid_constant__ CUtensorMap tm_A, const __grid_constant__ CUtensorMap tm_U,
                const __grid_constant__ CUtensorMap tm_S, const Params p) {
    using C = Cfg<R>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* aring = smem;                                  // [ASTAGES][A tile | U rows]
    uint8_t* sop = smem + ASTAGES * C::STAGE_BYTES;         // [2][STILE_BYTES]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sop + 2 * C::STILE_BYTES);
    uint64_t* afull = bars;                                 // [ASTAGES]
    uint64_t* mma_done = bars + ASTAGES;                    // [1]
    uint64_t* final_bar = bars + ASTAGES + 1;               // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + ASTAGES + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int j = tid;  // TMEM lane = dk index = column of S owned by this thread
    const int bh = blockIdx.x / p.rsplit;
    const int r0 = (blockIdx.x % p.rsplit) * R;
    const int b = bh / p.H, h = bh % p.H;
    const int aboxes = p.dk > 64 ? 2 : 1;
    const int sboxes = aboxes;
    const int nk = (p.dk + 15) / 16;
    const bool jv = j < p.dk;

    for (int i = tid; i < (ASTAGES * C::STAGE_BYTES + 2 * C::STILE_BYTES) / 16; i += THREADS)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < ASTAGES; ++s) mbar_init(&afull[s], 1);
        mbar_init(mma_done, 1);
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_A);
        prefetch_tmap(&tm_U);
        prefetch_tmap(&tm_S);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }

    // S_0 slice: thread j holds S[r0 + r][j] for r < R
    float S[R];
    const size_t state_off = (static_cast<size_t>(b) * p.H + h) * p.dv * p.dk;
#pragma unroll
    for (int r = 0; r < R; ++r)
        S[r] = (p.state_in != nullptr && jv) ? p.state_in[state_off + static_cast<size_t>(r0 + r) * p.dk + j] : 0.0f;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();  // zero-fill done before the first state image is written
    tc_fence_after();
    const uint32_t tmem = *tmem_slot + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
    for (int r = 0; r < R; ++r)
        *reinterpret_cast<__nv_bfloat16*>(sop + sop_offset<R>(r, j)) = __float2bfloat16_rn(S[r]);

    auto item_of = [&](int f) { return (b * p.F + f) * p.H + h; };
    // one ring slot = A_f (bf16, 128x128 swizzled) followed by U_f rows r0..r0+R-1 (fp32)
    auto issue_load = [&](int frame, int slot) {
        uint8_t* st = aring + slot * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&afull[slot], aboxes * ABOX_BYTES + C::UTILE_BYTES);
        for (int bx = 0; bx < aboxes; ++bx)
            tma_load_3d(st + bx * ABOX_BYTES, &tm_A, &afull[slot], 64 * bx, 0, item_of(frame));
        tma_load_3d(st + ATILE_BYTES, &tm_U, &afull[slot], 0, r0, item_of(frame));
    };
    int loaded = 0;  // frames whose loads have been issued (thread 0 only)
    if (tid == 0)
        for (; loaded < ASTAGES && loaded < p.F; ++loaded) issue_load(loaded, loaded);
    float a_next = __ldg(p.alpha + static_cast<size_t>(b * p.F) * p.H + h);

    fence_proxy_async_smem();
    __syncthreads();

    constexpr uint32_t IDESC = idesc_bf16(128, R, 0, 0);
    int consumed = 0;  // frames whose A_f has been waited for
    int f = 0;
    for (; f < p.F; ++f) {
        const int cur = f & 1;
        const int slot = f % ASTAGES;
        if (tid == 0) {
            if (mbar_wait(&afull[slot], static_cast<uint32_t>((f / ASTAGES) & 1), p.wait_limit_ns, abort_flag)) {
                ++consumed;
                tc_fence_after();
                const uint32_t a_base = smem_u32(aring + slot * C::STAGE_BYTES);
                const uint32_t b_base = smem_u32(sop + cur * C::STILE_BYTES);
                for (int kk = 0; kk < nk; ++kk) {
                    const uint64_t ad = smem_desc(a_base + (kk >> 2) * ABOX_BYTES + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc(b_base + (kk >> 2) * C::SBOX_BYTES + (kk & 3) * 32, 16, 1024);
                    mma_bf16(*tmem_slot, ad, bd, IDESC, kk > 0 ? 1u : 0u);
                }
                mma_commit(mma_done);
            }
        }
        // alpha of the next frame is fetched one frame ahead
        const float a_f = a_next;
        if (f + 1 < p.F) a_next = __ldg(p.alpha + static_cast<size_t>(b * p.F + f + 1) * p.H + h);

        bool ok = mbar_wait(&afull[slot], static_cast<uint32_t>((f / ASTAGES) & 1), p.wait_limit_ns, abort_flag) &&
                  mbar_wait(mma_done, static_cast<uint32_t>(f & 1), p.wait_limit_ns, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            uint32_t c[R];
            tmem_ld_cols<R>(tmem, c);
            const float* urow = reinterpret_cast<const float*>(aring + slot * C::STAGE_BYTES + ATILE_BYTES) + j;
            float u[R];
#pragma unroll
            for (int r = 0; r < R; ++r) u[r] = urow[r * 128];
            tmem_wait_ld();
            uint8_t* nxt = sop + (cur ^ 1) * C::STILE_BYTES;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                S[r] = a_f * (S[r] - __uint_as_float(c[r])) + u[r];
                *reinterpret_cast<__nv_bfloat16*>(nxt + sop_offset<R>(r, j)) = __float2bfloat16_rn(S[r]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        tc_fence_after();
        if (!ok) break;
        if (tid == 0) {
            // every thread has read slot `slot` and its MMA has retired: refill it
            if (loaded < p.F) {
                issue_load(loaded, slot);
                ++loaded;
            }
            // publish the bf16 state after frame f for phase 3
            const uint8_t* nxt = sop + (cur ^ 1) * C::STILE_BYTES;
            for (int bx = 0; bx < sboxes; ++bx)
                tma_store_3d(&tm_S, nxt + bx * C::SBOX_BYTES, 64 * bx, r0, item_of(f));
            bulk_commit();
            bulk_wait_read<1>();  // the store issued one frame ago no longer reads its buffer
        }
    }

    if (f == p.F && p.state_out != nullptr && jv) {
#pragma unroll
        for (int r = 0; r < R; ++r) p.state_out[state_off + static_cast<size_t>(r0 + r) * p.dk + j] = S[r];
    }
    if (tid == 0) {
        bulk_wait<0>();
        for (int fl = consumed; fl < loaded; ++fl)
            mbar_wait_drain(&afull[fl % ASTAGES], static_cast<uint32_t>((fl / ASTAGES) & 1), p.wait_limit_ns);
        mma_commit(final_bar);
        mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, TMEM_COLS);
    }
}

}  // namespace k2
}  // namespace gdn
