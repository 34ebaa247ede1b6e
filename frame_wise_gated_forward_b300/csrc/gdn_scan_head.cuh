// gdn_scan_head.cuh -- the sequential scan of the frame-wise GDN forward with
// one CTA per (b, h) head, for the single-pass forward (gdn_fwd_single.cuh):
//     S_f = alpha_f * (S_{f-1} - S_{f-1} A_f) + U_f
// (SANA-WM article, "The Architecture": a fixed-size state matrix updated
// once per latent frame by a decay gate and a delta-rule correction; wispaper
// summary, "Methodology" 1: frames scanned one by one).
//
// The state's rows live in tensor-memory lanes: lane i holds row i of the
// fp32 master state (columns [128, 256)) and row i of C = S_img A_f (columns
// [0, 128)), where S_img is the bf16 image of the state before the frame.
// Per frame one MMA chain on the tensor core
//     D[i][j] = sum_k S_img[i][k] A_f[k][j]      M = 128 (i), N = 128 (j), K = dk
// reads S_img (K-major: row i, k contiguous) and A_f (row j of the symmetric
// A_f, also K-major) from 128-byte-swizzled shared memory.  Eight compute
// warps update the state: warp w owns the lanes (rows) of quarter w % 4 and
// the 64 columns of half w / 4, so each thread reads its row of C and S from
// tensor memory, its row of U_f from the TMA-loaded tile, writes the new fp32
// row back to tensor memory and its bf16 row into the image with 16-byte
// stores.  One image buffer suffices: the image is rewritten only after the
// MMA that reads it has retired and the bulk store that publishes it has read
// it; the update itself runs before that wait, the new row held in registers.
//
// A_f and U_f come from ring slots of the workspace that contraction CTAs of
// the same launch fill (a per-slot count of frames written, raised with
// release semantics after the slot's stores); the loader warp waits (bounded,
// acquire) for the count, then copies the slot's two tiles with one bulk
// copy each: the contraction writes them in this role's shared-memory image
// (ring_off in gdn_ptx.cuh), so 96 KB move as two contiguous runs instead of
// 768 separate 128-byte rows, which bounded the scan at about 2 us a frame.
// Once the copy has landed the MMA warp hands the slot back (a count of
// frames read).  The publisher warp stores each frame's image into the ring
// slot of the output CTAs the same way (one 32 KB bulk store), after they
// have loaded the slot's previous occupant, and raises the slot's ready count
// once the store has completed.
//
// Warp roles (352 threads): warps 0-7 compute, warp 8 loads A_f / U_f, warp 9
// issues the MMAs, warp 10 publishes the images.  The image of the initial
// state has a barrier of its own, so the publisher's phase count starts with
// the image after frame 0.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace k2h {

constexpr int COMPUTE_THREADS = 256;
constexpr int LOADER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int PUB_WARP = 10;
constexpr int THREADS = 352;
constexpr int AS = 2;                      // A_f / U_f stages
constexpr int ABOX = 128 * 128;            // 128 rows x 128 B (64 bf16)
constexpr int ATILE = 2 * ABOX;            // A_f bf16 [128][128], two 64-column boxes
constexpr int UBOX = 128 * 128;            // 128 rows x 32 fp32
constexpr int UTILE = 4 * UBOX;            // U_f fp32 [128][128], four 32-column boxes
constexpr int STAGE = ATILE + UTILE;
constexpr int OFF_IMG = AS * STAGE;        // bf16 image of the state, two 64-column boxes
constexpr int OFF_BAR = OFF_IMG + ATILE;
constexpr int BAR_BYTES = 256;
constexpr size_t SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(ATILE == RING_TILE_BF16 && UTILE == RING_TILE_F32, "a stage holds one ring tile of each");
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t T_C = 0;                // C = S_img A_f
constexpr uint32_t T_S = 128;              // fp32 master state

struct Params {
    const __nv_bfloat16* A_ring;   // [B][W][H] ring tiles of A_f (RING_TILE_BF16 bytes each)
    const float* U_ring;           // [B][W][H] ring tiles of U_f (RING_TILE_F32 bytes each)
    __nv_bfloat16* S_ring;         // [B][W][H] ring tiles of the state images (RING_TILE_BF16 bytes each)
    const float* alpha;     // [B, F, H]
    const float* state_in;  // [B, H, dv, dk] or nullptr
    float* state_out;       // [B, H, dv, dk] or nullptr
    int B, H, F, dk, dv;
    int reverse;            // scan the frames from F-1 down to 0
    int alpha_gate;         // fused prologue: alpha <- exp(-softplus(alpha) * alpha_scale)
    float alpha_scale;
    int ring;               // W: ring slots per (b, h); step s of the scan uses slot s % W
    const int* au_ready;    // [B][W][H] frames of A/U written into the slot
    int* au_free;           // [B][W][H] frames of A/U read out of the slot
    int* s_ready;           // [B][W][H] frames of state images stored into the slot
    const int* s_free;      // [B][W][H] loads of the slot's image by output CTAs
    int s_units;            // output CTA loads per image
    unsigned long long wait_limit_ns;
};

__device__ __forceinline__ float decay_gate(const Params& p, float x) {
    if (!p.alpha_gate) return x;
    const float sp = x > 20.0f ? x : log1pf(expf(x));  // softplus
    return expf(-sp * p.alpha_scale);
}

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled box
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + (((c ^ (r & 7))) << 4); }

// The scan of head `cta` = b * H + h.  Needs THREADS threads.
__device__ __forceinline__ void scan_head_role(const Params& p, int cta, uint8_t* smem) {
    uint8_t* ring = smem;
    uint8_t* img = smem + OFF_IMG;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* afull = bars;                 // [AS] loader -> MMA: A_f landed
    uint64_t* ufull = afull + AS;           // [AS] loader -> compute, MMA: U_f landed
    uint64_t* slot_free = ufull + AS;       // [AS] compute -> loader
    uint64_t* mma_done = slot_free + AS;    // MMA -> compute
    uint64_t* img_init = mma_done + 1;      // compute -> MMA: the image of the state before frame 0
    uint64_t* img_ready = img_init + 1;     // compute -> MMA, publisher: the image after frame f
    uint64_t* img_free = img_ready + 1;     // publisher -> compute
    uint64_t* final_bar = img_free + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int b = cta / p.H, h = cta % p.H;
    const int nk = (p.dk + 15) / 16;
    auto fr = [&](int s) { return p.reverse ? p.F - 1 - s : s; };
    auto rslot = [&](int s) { return (b * p.ring + s % p.ring) * p.H + h; };

    if (tid == 0) {
        for (int s = 0; s < AS; ++s) {
            mbar_init(&afull[s], 1);
            mbar_init(&ufull[s], 1);
            mbar_init(&slot_free[s], COMPUTE_THREADS);
        }
        mbar_init(mma_done, 1);
        mbar_init(img_init, COMPUTE_THREADS);
        mbar_init(img_ready, COMPUTE_THREADS);
        mbar_init(img_free, 1);
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 8) {
        // ---------------------------------------------------------- compute
        const int i = (warp & 3) * 32 + lane;           // state row = TMEM lane
        const int ch = warp >> 2;                       // column half
        const uint32_t tw = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const size_t srow = ((static_cast<size_t>(b) * p.H + h) * p.dv + i) * p.dk;
        const bool iv = i < p.dv;
        // the state before frame 0: fp32 into TMEM, bf16 into the image
#pragma unroll
        for (int sc = 0; sc < 2; ++sc) {
            const int c0 = 64 * ch + 32 * sc;
            uint32_t v[32];
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p.state_in != nullptr && iv && c0 + 4 * q4 < p.dk)
                    x = *reinterpret_cast<const float4*>(p.state_in + srow + c0 + 4 * q4);
                v[4 * q4] = __float_as_uint(x.x);
                v[4 * q4 + 1] = __float_as_uint(x.y);
                v[4 * q4 + 2] = __float_as_uint(x.z);
                v[4 * q4 + 3] = __float_as_uint(x.w);
            }
            tmem_st32(tw + T_S + c0, v);
            uint8_t* row = img + (c0 >> 6) * ABOX;
            const int cb = (c0 & 63) >> 3;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                *reinterpret_cast<uint4*>(row + sw128(i, cb + t)) = make_uint4(
                    pack_bf16x2(__uint_as_float(v[8 * t + 0]), __uint_as_float(v[8 * t + 1])),
                    pack_bf16x2(__uint_as_float(v[8 * t + 2]), __uint_as_float(v[8 * t + 3])),
                    pack_bf16x2(__uint_as_float(v[8 * t + 4]), __uint_as_float(v[8 * t + 5])),
                    pack_bf16x2(__uint_as_float(v[8 * t + 6]), __uint_as_float(v[8 * t + 7])));
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(img_init);   // the initial image (never published)
        float a_next = decay_gate(p, __ldg(p.alpha + static_cast<size_t>(b * p.F + fr(0)) * p.H + h));
        int f = 0;
        for (; f < p.F; ++f) {
            const int slot = f % AS;
            const float a_f = a_next;
            if (f + 1 < p.F) a_next = decay_gate(p, __ldg(p.alpha + static_cast<size_t>(b * p.F + fr(f + 1)) * p.H + h));
            bool ok = mbar_wait(&ufull[slot], static_cast<uint32_t>((f / AS) & 1), p.wait_limit_ns, abort_flag,
                                1010000 + f);
            ok = ok && mbar_wait(mma_done, static_cast<uint32_t>(f & 1), p.wait_limit_ns, abort_flag, 1020000 + f);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint8_t* ut = ring + slot * STAGE + ATILE;
            uint4 im[2][4];   // the new row's bf16 image, written once the previous image is stored
#pragma unroll
            for (int sc = 0; sc < 2; ++sc) {
                const int c0 = 64 * ch + 32 * sc;
                uint32_t cc[32], ss[32];
                tmem_ld32(tw + T_C + c0, cc);
                tmem_ld32(tw + T_S + c0, ss);
                float4 u[8];
                const uint8_t* ub = ut + (c0 >> 5) * UBOX;
#pragma unroll
                for (int t = 0; t < 8; ++t) u[t] = *reinterpret_cast<const float4*>(ub + sw128(i, t));
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float uu[4] = {u[t].x, u[t].y, u[t].z, u[t].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int x = 4 * t + e;
                        ss[x] = __float_as_uint(a_f * (__uint_as_float(ss[x]) - __uint_as_float(cc[x])) + uu[e]);
                    }
                }
                tmem_st32(tw + T_S + c0, ss);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    im[sc][t] = make_uint4(
                        pack_bf16x2(__uint_as_float(ss[8 * t + 0]), __uint_as_float(ss[8 * t + 1])),
                        pack_bf16x2(__uint_as_float(ss[8 * t + 2]), __uint_as_float(ss[8 * t + 3])),
                        pack_bf16x2(__uint_as_float(ss[8 * t + 4]), __uint_as_float(ss[8 * t + 5])),
                        pack_bf16x2(__uint_as_float(ss[8 * t + 6]), __uint_as_float(ss[8 * t + 7])));
            }
            mbar_arrive(&slot_free[slot]);   // U_f read, the MMA that read A_f retired
            // the image may be rewritten once the store of the previous one has read it
            ok = f == 0 || mbar_wait(img_free, static_cast<uint32_t>((f - 1) & 1), p.wait_limit_ns, abort_flag,
                                     1030000 + f);
            if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll
            for (int sc = 0; sc < 2; ++sc) {
                const int c0 = 64 * ch + 32 * sc;
                uint8_t* row = img + (c0 >> 6) * ABOX;
                const int cb = (c0 & 63) >> 3;
#pragma unroll
                for (int t = 0; t < 4; ++t) *reinterpret_cast<uint4*>(row + sw128(i, cb + t)) = im[sc][t];
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(img_ready);
        }
        // tcgen05.ld is warp-collective: every lane loads, only rows < dv are stored
        if (__all_sync(0xffffffffu, f == p.F) && p.state_out != nullptr) {
            tc_fence_after();
#pragma unroll
            for (int sc = 0; sc < 2; ++sc) {
                const int c0 = 64 * ch + 32 * sc;
                uint32_t ss[32];
                tmem_ld32(tw + T_S + c0, ss);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    if (iv && c0 + 4 * q4 < p.dk)
                        *reinterpret_cast<float4*>(p.state_out + srow + c0 + 4 * q4) =
                            make_float4(__uint_as_float(ss[4 * q4]), __uint_as_float(ss[4 * q4 + 1]),
                                        __uint_as_float(ss[4 * q4 + 2]), __uint_as_float(ss[4 * q4 + 3]));
            }
        }
    } else if (warp == MMA_WARP) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16(128, 128, 0, 0);
            for (int f = 0; f < p.F; ++f) {
                const int slot = f % AS;
                if (!mbar_wait(&afull[slot], static_cast<uint32_t>((f / AS) & 1), p.wait_limit_ns, abort_flag,
                               1110000 + f))
                    break;
                // the image of the state before frame f
                if (!(f == 0 ? mbar_wait(img_init, 0, p.wait_limit_ns, abort_flag, 1120000)
                             : mbar_wait(img_ready, static_cast<uint32_t>((f - 1) & 1), p.wait_limit_ns, abort_flag,
                                         1120000 + f)))
                    break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(img);
                const uint32_t b_base = smem_u32(ring + slot * STAGE);
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t ko = (kk >> 2) * ABOX + (kk & 3) * 32;
                    mma_bf16(tmem + T_C, smem_desc(a_base + ko, 16, 1024), smem_desc(b_base + ko, 16, 1024), IDESC,
                             kk > 0 ? 1u : 0u);
                }
                mma_commit(mma_done);
                // both tiles of the slot are in shared memory: the contraction may
                // refill it (a release, which takes a while, so it follows the MMAs)
                if (!mbar_wait(&ufull[slot], static_cast<uint32_t>((f / AS) & 1), p.wait_limit_ns, abort_flag,
                               1130000 + f))
                    break;
                red_release_add(p.au_free + rslot(f), 1);
            }
            mma_commit(final_bar);
            mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
        }
    } else if (warp == PUB_WARP) {
        // -------------------------------------------------------- publisher
        if (lane == 0) {
            int published = 0;
            auto publish_upto = [&](int f_end) {
                if (published >= f_end) return;
                fence_proxy_async_global();  // the stores' writes ordered before the releases
                for (; published < f_end; ++published) red_release_add(p.s_ready + rslot(published), 1);
            };
            int f = 0;
            for (; f < p.F; ++f) {
                // the slot's previous image has been loaded by every output CTA that
                // reads it (asked before the image is ready, so that the round trip
                // to L2 overlaps the frame's update instead of delaying the store)
                if (f >= p.ring && !wait_count_geq(p.s_free + rslot(f), (f / p.ring) * p.s_units, p.wait_limit_ns,
                                                   abort_flag, 1220000 + f))
                    break;
                if (!mbar_wait(img_ready, static_cast<uint32_t>(f & 1), p.wait_limit_ns, abort_flag, 1210000 + f))
                    break;
                if (f >= p.ring) fence_proxy_async_global();
                bulk_store(reinterpret_cast<uint8_t*>(p.S_ring) + static_cast<size_t>(rslot(f)) * RING_TILE_BF16, img,
                           RING_TILE_BF16);
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(img_free);
                bulk_wait<1>();  // the stores of frames <= f - 1 are complete
                publish_upto(f);
            }
            bulk_wait<0>();
            publish_upto(f);
        }
    } else if (warp == LOADER_WARP) {
        // ----------------------------------------------------------- loader
        if (lane == 0) {
            int issued = 0;
            for (int f = 0; f < p.F; ++f) {
                const int slot = f % AS;
                // the contraction's count first (an L2 round trip that overlaps the
                // wait for the stage), then the stage
                if (!wait_count_geq(p.au_ready + rslot(f), f / p.ring + 1, p.wait_limit_ns, abort_flag, 1320000 + f))
                    break;
                if (f >= AS && !mbar_wait(&slot_free[slot], static_cast<uint32_t>(((f / AS) - 1) & 1),
                                          p.wait_limit_ns, abort_flag, 1310000 + f))
                    break;
                fence_proxy_async_global();  // the contraction's stores are read through the async proxy
                uint8_t* st = ring + slot * STAGE;
                const size_t rs = static_cast<size_t>(rslot(f));
                mbar_arrive_expect_tx(&afull[slot], RING_TILE_BF16);
                bulk_load(st, reinterpret_cast<const uint8_t*>(p.A_ring) + rs * RING_TILE_BF16, RING_TILE_BF16,
                          &afull[slot]);
                mbar_arrive_expect_tx(&ufull[slot], RING_TILE_F32);
                bulk_load(st + ATILE, reinterpret_cast<const uint8_t*>(p.U_ring) + rs * RING_TILE_F32, RING_TILE_F32,
                          &ufull[slot]);
                ++issued;
            }
            for (int k = (issued > AS ? issued - AS : 0); k < issued; ++k) {
                mbar_wait_drain(&afull[k % AS], static_cast<uint32_t>((k / AS) & 1), p.wait_limit_ns);
                mbar_wait_drain(&ufull[k % AS], static_cast<uint32_t>((k / AS) & 1), p.wait_limit_ns);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace k2h
}  // namespace gdn
