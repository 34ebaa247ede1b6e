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
//     M = 128 (dk index j, zero-padded), N = rows of the slice, K = dk
// with both operands K-major in 128-byte-swizzled shared memory: A_f comes
// from the bf16 workspace by TMA together with the CTA's R rows of U_f
// (fp32, unswizzled) through a prefetch ring, so no global load sits on the
// per-frame critical path; S_slice is the bf16 image of the state that the
// compute threads rewrite every frame.  The fp32 master state stays in
// registers: thread j (TMEM lane j) owns column j of the slice, which is
// exactly the layout tcgen05.ld returns C in.
//
// A slice of more than 32 rows is split into independent chains of 32 rows,
// each with its own MMA (N = 32), accumulator columns and image-ready
// barrier: while one chain's MMA runs, the compute threads update another.
//
// Warp roles (224 threads): warps 0-3 compute; warp 4 publishes each frame's
// bf16 state image with a TMA store to the per-frame state buffer that phase
// 3 reads (and, when the scan runs fused with phase 3, then raises that item's
// ready count); warp 5 refills the A_f/U_f ring; warp 6 issues the MMAs.
// Compute hands each image to the publisher and the MMA issuer through
// mbarriers and keeps up to NIMG images in flight, so neither store latency
// nor load issue sits on the frame-to-frame chain.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace k2 {

constexpr int COMPUTE_THREADS = 128;
constexpr int THREADS = 224;                 // + publisher, loader and MMA-issuer warps
constexpr int ABOX_BYTES = 128 * 128;        // 128 rows x 128 B
constexpr int ATILE_BYTES = 2 * ABOX_BYTES;  // A_f, dk padded to 128

template <int R>
struct Cfg {
    static constexpr int RS = R < 32 ? R : 32;                 // rows per independent chain (MMA N)
    static constexpr int NC = R / RS;                          // chains per slice
    static constexpr int ASTAGES = R >= 64 ? 2 : 4;
    static constexpr int NIMG = 4;                             // bf16 state images in flight
    static constexpr int SBOX_BYTES = R * 128;
    static constexpr int STILE_BYTES = 2 * SBOX_BYTES;
    static constexpr int UTILE_BYTES = R * 128 * 4;            // R rows x 128 fp32 (dk padded)
    static constexpr int STAGE_BYTES = ATILE_BYTES + UTILE_BYTES;
    static constexpr int TMEM_COLS = R < 32 ? 32 : R;
    static constexpr size_t SMEM_BYTES = 1024 + ASTAGES * STAGE_BYTES + NIMG * STILE_BYTES + 512;
    static_assert(R % RS == 0, "whole chains");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert((2 * ASTAGES + NC + NIMG * NC + NIMG + 1) * 8 + 8 <= 512, "barrier area");
};

struct Params {
    const float* alpha;     // [B, F, H]
    const float* state_in;  // [B, H, dv, dk] or nullptr
    float* state_out;       // [B, H, dv, dk] or nullptr
    int H, F, dk, dv;
    int rsplit;             // dv / R CTAs per head
    int reverse;            // nonzero: scan the frames from F-1 down to 0
    int alpha_gate;         // fused prologue: alpha <- exp(-softplus(alpha) * alpha_scale)
    float alpha_scale;
    unsigned long long wait_limit_ns;
};

__device__ __forceinline__ float decay_gate(const Params& p, float x) {
    if (!p.alpha_gate) return x;
    const float sp = x > 20.0f ? x : log1pf(expf(x));  // softplus
    return expf(-sp * p.alpha_scale);
}

// bf16 element (r, j) of a K-major, 128-byte-swizzled [R rows x 128 cols] tile
template <int R>
__device__ __forceinline__ uint32_t sop_offset(int r, int j) {
    const int box = j >> 6, col = j & 63;
    return box * Cfg<R>::SBOX_BYTES + r * 128 + ((((col >> 3) ^ (r & 7))) << 4) + ((col & 7) << 1);
}

// The scan of one R-row slice of one head.  `cta` selects (b, h, slice);
// `flags` (may be null) receives one increment per published frame state.
// Needs THREADS threads.
template <int R>
__device__ __forceinline__ void scan_role(const CUtensorMap* tm_A, const CUtensorMap* tm_U, const CUtensorMap* tm_S,
                                          const Params& p, int cta, int* flags, uint8_t* smem) {
    using C = Cfg<R>;
    constexpr int AS = C::ASTAGES;
    constexpr int NI = C::NIMG;
    constexpr int NC = C::NC;
    constexpr int RS = C::RS;
    uint8_t* aring = smem;                                  // [AS][A tile | U rows]
    uint8_t* sop = smem + AS * C::STAGE_BYTES;              // [NI][STILE_BYTES] bf16 state images
    uint64_t* bars = reinterpret_cast<uint64_t*>(sop + NI * C::STILE_BYTES);
    uint64_t* afull = bars;                                 // [AS] loader -> compute, MMA
    uint64_t* slot_free = afull + AS;                       // [AS] compute -> loader
    uint64_t* mma_done = slot_free + AS;                    // [NC] MMA -> compute
    uint64_t* img_ready = mma_done + NC;                    // [NI][NC] compute -> MMA, publisher
    uint64_t* img_free = img_ready + NI * NC;               // [NI] publisher -> compute
    uint64_t* final_bar = img_free + NI;                    // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int j = tid;  // compute threads: TMEM lane = dk index = column of S owned by this thread
    const int bh = cta / p.rsplit;
    const int r0 = (cta % p.rsplit) * R;
    const int b = bh / p.H, h = bh % p.H;
    const int aboxes = p.dk > 64 ? 2 : 1;
    const int sboxes = aboxes;
    const int nk = (p.dk + 15) / 16;
    const bool jv = j < p.dk;
    // step f of the scan handles latent frame fr(f): f itself, or F-1-f when reversed
    auto fr = [&](int f) { return p.reverse ? p.F - 1 - f : f; };
    auto item_of = [&](int f) { return (b * p.F + fr(f)) * p.H + h; };

    // A_f's second box is never loaded when dk <= 64 and must read as zero;
    // everything else is written before it is read
    if (aboxes < 2)
        for (int i = tid; i < (AS * C::STAGE_BYTES + NI * C::STILE_BYTES) / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < AS; ++s) {
            mbar_init(&afull[s], 1);
            mbar_init(&slot_free[s], COMPUTE_THREADS);
        }
        for (int c = 0; c < NC; ++c) mbar_init(&mma_done[c], 1);
        for (int x = 0; x < NI; ++x) {
            for (int c = 0; c < NC; ++c) mbar_init(&img_ready[x * NC + c], COMPUTE_THREADS);
            mbar_init(&img_free[x], 1);
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(tm_A);
        prefetch_tmap(tm_U);
        prefetch_tmap(tm_S);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();  // zero-fill and barrier init done
    tc_fence_after();

    if (warp < 4) {
        // ---------------------------------------------------------- compute
        float S[R];
        const size_t state_off = (static_cast<size_t>(b) * p.H + h) * p.dv * p.dk;
#pragma unroll
        for (int r = 0; r < R; ++r)
            S[r] = (p.state_in != nullptr && jv) ? p.state_in[state_off + static_cast<size_t>(r0 + r) * p.dk + j]
                                                 : 0.0f;
        const uint32_t tmem_warp = *tmem_slot + (static_cast<uint32_t>(warp * 32) << 16);
        // image of the state before frame 0 in buffer 0; the state after frame f goes to buffer (f + 1) % NI
#pragma unroll
        for (int r = 0; r < R; ++r)
            *reinterpret_cast<__nv_bfloat16*>(sop + sop_offset<R>(r, j)) = __float2bfloat16_rn(S[r]);
        fence_proxy_async_smem();
        for (int c = 0; c < NC; ++c) mbar_arrive(&img_ready[c]);  // initial image (never stored)
        float a_next = decay_gate(p, __ldg(p.alpha + static_cast<size_t>(b * p.F + fr(0)) * p.H + h));

        int f = 0;
        for (; f < p.F; ++f) {
            const int slot = f % AS;
            const int nxt = (f + 1) % NI;  // image of the state after frame f
            const float a_f = a_next;
            if (f + 1 < p.F) a_next = decay_gate(p, __ldg(p.alpha + static_cast<size_t>(b * p.F + fr(f + 1)) * p.H + h));

            // the buffer this frame's image goes to was last stored NI frames ago
            bool ok = f < NI || mbar_wait(&img_free[nxt], static_cast<uint32_t>(((f / NI) - 1) & 1),
                                          p.wait_limit_ns, abort_flag);
            ok = ok && mbar_wait(&afull[slot], static_cast<uint32_t>((f / AS) & 1), p.wait_limit_ns, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const float* urow = reinterpret_cast<const float*>(aring + slot * C::STAGE_BYTES + ATILE_BYTES) + j;
            uint8_t* img = sop + nxt * C::STILE_BYTES;
            // chain by chain: read the chain's U rows and accumulator, update its
            // rows of the state, write them to the image and hand the chain on
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float u[RS];
#pragma unroll
                for (int r = 0; r < RS; ++r) u[r] = urow[(c * RS + r) * 128];
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&mma_done[c], static_cast<uint32_t>(f & 1), p.wait_limit_ns, abort_flag));
                if (!ok) break;
                tc_fence_after();
                uint32_t cc[RS];
#pragma unroll
                for (int q = 0; q < RS; q += 16)
                    tmem_ld16(tmem_warp + c * RS + q, *reinterpret_cast<uint32_t(*)[16]>(&cc[q]));
                tmem_wait_ld();
#pragma unroll
                for (int r = 0; r < RS; ++r) {
                    const int row = c * RS + r;
                    S[row] = a_f * (S[row] - __uint_as_float(cc[r])) + u[r];
                    *reinterpret_cast<__nv_bfloat16*>(img + sop_offset<R>(row, j)) = __float2bfloat16_rn(S[row]);
                }
                tc_fence_before();
                fence_proxy_async_smem();
                mbar_arrive(&img_ready[nxt * NC + c]);
            }
            if (!ok) break;
            mbar_arrive(&slot_free[slot]);  // U read, the MMAs that read A_f retired
        }
        if (f == p.F && p.state_out != nullptr && jv) {
#pragma unroll
            for (int r = 0; r < R; ++r) p.state_out[state_off + static_cast<size_t>(r0 + r) * p.dk + j] = S[r];
        }
    } else if (warp == 6) {
        // -------------------------------------------------------- MMA issuer
        if ((tid & 31) == 0) {
            constexpr uint32_t IDESC = idesc_bf16(128, RS, 0, 0);
            bool stop = false;
            for (int f = 0; f < p.F && !stop; ++f) {
                const int slot = f % AS;
                const int cur = f % NI;  // image of the state after frame f - 1
                if (!mbar_wait(&afull[slot], static_cast<uint32_t>((f / AS) & 1), p.wait_limit_ns, abort_flag))
                    break;
                for (int c = 0; c < NC; ++c) {
                    if (!mbar_wait(&img_ready[cur * NC + c], static_cast<uint32_t>((f / NI) & 1), p.wait_limit_ns,
                                   abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(aring + slot * C::STAGE_BYTES);
                    const uint32_t b_base = smem_u32(sop + cur * C::STILE_BYTES) + c * RS * 128;
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint64_t ad = smem_desc(a_base + (kk >> 2) * ABOX_BYTES + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = smem_desc(b_base + (kk >> 2) * C::SBOX_BYTES + (kk & 3) * 32, 16, 1024);
                        mma_bf16(*tmem_slot + c * RS, ad, bd, IDESC, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&mma_done[c]);
                }
            }
            mma_commit(final_bar);
            mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
        }
    } else if (warp == 4) {
        // -------------------------------------------------------- publisher
        // Stores are pipelined: a frame's ready count is raised once at most
        // two newer stores are still in flight.
        if ((tid & 31) == 0) {
            int published = 0;
            auto publish_upto = [&](int f_end) {
                if (flags == nullptr || published >= f_end) return;
                fence_proxy_async_global();  // async-proxy writes ordered before the release below
                for (; published < f_end; ++published) red_release_add(flags + item_of(published), 1);
            };
            int f = 0;
            bool stop = false;
            for (; f < p.F; ++f) {
                const int x = (f + 1) % NI;  // buffer holding the image of the state after frame f
                for (int c = 0; c < NC && !stop; ++c)
                    stop = !mbar_wait(&img_ready[x * NC + c], static_cast<uint32_t>(((f + 1) / NI) & 1),
                                      p.wait_limit_ns, abort_flag);
                if (stop) break;
                const uint8_t* img = sop + x * C::STILE_BYTES;
                for (int bx = 0; bx < sboxes; ++bx)
                    tma_store_3d(tm_S, img + bx * C::SBOX_BYTES, 64 * bx, r0, item_of(f));
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(&img_free[x]);
                bulk_wait<2>();  // stores of frames <= f - 2 are complete
                publish_upto(f - 1);
            }
            bulk_wait<0>();
            publish_upto(f);
        }
    } else if (warp == 5) {
        // ----------------------------------------------------------- loader
        if ((tid & 31) == 0) {
            // one ring slot = A_f (bf16, 128x128 swizzled) followed by U_f rows r0..r0+R-1 (fp32)
            int issued = 0;
            for (int f = 0; f < p.F; ++f) {
                const int slot = f % AS;
                if (f >= AS && !mbar_wait(&slot_free[slot], static_cast<uint32_t>(((f / AS) - 1) & 1),
                                          p.wait_limit_ns, abort_flag))
                    break;
                uint8_t* st = aring + slot * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&afull[slot], aboxes * ABOX_BYTES + C::UTILE_BYTES);
                for (int bx = 0; bx < aboxes; ++bx)
                    tma_load_3d(st + bx * ABOX_BYTES, tm_A, &afull[slot], 64 * bx, 0, item_of(f));
                tma_load_3d(st + ATILE_BYTES, tm_U, &afull[slot], 0, r0, item_of(f));
                ++issued;
            }
            // no copy may outlive the CTA (only matters when a wait gave up)
            for (int k = (issued > AS ? issued - AS : 0); k < issued; ++k)
                mbar_wait_drain(&afull[k % AS], static_cast<uint32_t>((k / AS) & 1), p.wait_limit_ns);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, C::TMEM_COLS);
    }
}

// Standalone phase 2: one CTA per R-row slice of each head.
template <int R>
__global__ void __launch_bounds__(THREADS, 1)
    scan_kernel(const __grid_constant__ CUtensorMap tm_A, const __grid_constant__ CUtensorMap tm_U,
                const __grid_constant__ CUtensorMap tm_S, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    scan_role<R>(&tm_A, &tm_U, &tm_S, p, blockIdx.x, nullptr, smem);
}

}  // namespace k2
}  // namespace gdn
