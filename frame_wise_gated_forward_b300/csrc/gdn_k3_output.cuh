// gdn_k3_output.cuh -- phase 3 of the frame-wise GDN forward: every token of
// latent frame f reads the state after frame f,
//     O_f = Q_f S_f^T        (o_n = S_f q_n)
// (SANA-WM article, "The Architecture": the layer processes one entire latent
// frame per step, so all tokens of a frame see the same state).
//
// Frame-parallel: tiles of 128 tokens of one (b, f, h) item.  Per tile one
// MMA chain D = Q_tile S_f^T with
//     M = 128 tokens, N = 128 (dv, zero-padded), K = dk (<= 128)
// both operands K-major in 128-byte-swizzled shared memory, loaded by TMA
// straight from q's token-major layout and from the bf16 per-frame states.
// S_f is loaded once per item (2-deep ring), q through a 3-deep ring, four
// 128-column accumulators in TMEM let the MMA run up to three tiles ahead of
// the epilogue.  Epilogue: each of four warps drains its 32-lane quarter,
// rounds to bf16 (RNE), writes a swizzled staging tile and stores it with its
// own TMA store (rows past N are clipped by the tensor map).
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2-5 epilogue (TMEM lane quarter = warp % 4), warps 6-7 row
// norms of q for the folded prologue (idle otherwise): they read each q tile
// from shared memory as soon as it lands, hand 1/max(|q_n|, eps) per row to
// the epilogue and co-sign the release of the ring slot.
//
// The role runs in two schedules:
//  - standalone (output_kernel): a persistent grid, each CTA a contiguous
//    range of tiles;
//  - fused with the scan (gdn_k23_fused.cuh): each worker CTA takes whole
//    items (single tiles when there are fewer than two items per worker, as
//    in a one-frame step) round-robin in frame-major order and, before loading
//    S_f, waits (bounded) until the scan has published that item's state.
#pragma once

#include "gdn_ptx.cuh"

namespace gdn {
namespace k3 {

constexpr int THREADS = 256;
constexpr int NORM_THREADS = 64;
constexpr int TILE_M = 128;                  // tokens per tile
constexpr int QSTAGES = 3;
constexpr int SSTAGES = 2;
constexpr int ACCS = 4;
constexpr int BOX_BYTES = TILE_M * 128;      // 128 rows x 128 B
constexpr int QTILE_BYTES = 2 * BOX_BYTES;   // dk padded to 128
constexpr int STILE_BYTES = 2 * BOX_BYTES;   // S_f: 128 rows (dv) x dk
constexpr int OBOX_BYTES = 32 * 128;         // one warp's 32 rows x 64 columns
constexpr int OSTAGE_BYTES = 2 * OBOX_BYTES; // 32 rows x 128 columns
constexpr int TMEM_COLS = 512;
constexpr int NSLOTS = 2;                    // row-norm buffers (folded prologue)
constexpr int BAR_BYTES = 256;
// fp8 (e4m3) q: TMA loads the raw 128x128-byte tile into the upper half of a
// q slot, and four decoder warps (6-9, so the block has 320 threads) decode
// it in place into the slot's two bf16 boxes: each thread owns one token row,
// reads its raw row whole before writing, and box 1's row is exactly the raw
// row it came from, so no thread overwrites bytes another one still reads.
constexpr int DEC_THREADS = 128;
template <int FMT>
__host__ __device__ constexpr int threads() { return FMT != FMT_BF16 ? 192 + DEC_THREADS : THREADS; }
constexpr int RAW_BYTES = TILE_M * 128;
static_assert(RAW_BYTES == BOX_BYTES, "a raw fp8 tile fills box 1 of a q slot");
static_assert((3 * QSTAGES + 2 * SSTAGES + 2 * ACCS + 1 + 2 * NSLOTS) * 8 + 8 <= BAR_BYTES, "barrier area");
constexpr size_t SMEM_BYTES =
    1024 + QSTAGES * QTILE_BYTES + SSTAGES * STILE_BYTES + 4 * 2 * OSTAGE_BYTES + BAR_BYTES + NSLOTS * TILE_M * 4;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(STILE_BYTES == RING_TILE_BF16, "a state stage holds one ring tile");

struct Params {
    int B, H, F, N, dk, dv;
    int ntile;              // ceil(N / 128) tiles per item
    long long total;        // items * ntile
    int reverse;            // fused schedule: follow a scan that runs from frame F-1 down
    int norm_q;             // fused prologue: scale each output row by 1/max(|q_n|, eps)
    float q_scale;          // fp8 / NVFP4 q: o_n = q_scale * S q_n (q decoded without it; 1 otherwise)
    const uint8_t* q_sf;    // NVFP4 q: E4M3 block scales [B, F, N, H, dk/16]
    int b_mn;               // 0: O = Q S^T (S K-major).  1: O = Q S with S read MN-major, for the
                            // backward's dq = dO S_f: then dk is dO's width (dv of S) and dv the
                            // output width (dk of S)
    unsigned long long wait_limit_ns;
};

// Which tiles a CTA processes, as a sequence of segments (item, nt_begin, nt_end).
struct Sched {
    // standalone: contiguous tile range [t0, t1)
    long long t0, t1;
    // fused: worker wi of nw takes frame-major item ranks wi, wi + nw, ...
    int wi, nw;
    bool fused;
    const int* flags;       // fused: per-item (ring: per-slot) count of published state slices
    int flag_target;        // fused: slices per item
    // ring mode (single-pass forward, 0 = off): the state of scan step s of
    // head (b, h) sits in slot (b * ring + s % ring) * H + h, which holds frames
    // s, s + ring, ... in turn; flags count published slices per slot, and
    // s_free counts this role's loads of each slot's image; the images are
    // whole ring tiles (RING_TILE_BF16 bytes, ring_off layout of gdn_ptx.cuh)
    // at s_ring, each loaded with one bulk copy
    int ring;
    int* s_free;
    const __nv_bfloat16* s_ring;

    __device__ __forceinline__ bool segment(const Params& p, int k, long long& item, int& nb, int& ne) const {
        long long slot;
        int use;
        return segment(p, k, item, nb, ne, slot, use);
    }
    __device__ __forceinline__ bool segment(const Params& p, int k, long long& item, int& nb, int& ne,
                                            long long& slot, int& use) const {
        use = 0;
        if (!fused) {
            // k-th segment of the contiguous range: walk items from t0
            long long t = t0;
            for (int i = 0; i < k && t < t1; ++i) t = (t / p.ntile + 1) * p.ntile;
            if (t >= t1) return false;
            item = t / p.ntile;
            nb = static_cast<int>(t % p.ntile);
            const long long end = (item + 1) * p.ntile < t1 ? (item + 1) * p.ntile : t1;
            ne = static_cast<int>(end - item * p.ntile);
            slot = item;
            return true;
        }
        // 32-bit unsigned arithmetic: every count here is below 2^31 (tiles of
        // one call), and several warps redo this per item, where 64-bit
        // divisions cost as much as some of the item's own work
        const unsigned BH = static_cast<unsigned>(p.B) * static_cast<unsigned>(p.H);
        const bool per_tile = static_cast<long long>(BH) * p.F < 2LL * nw;  // few items: spread single tiles instead
        const unsigned units = per_tile ? BH * p.F * p.ntile : BH * p.F;
        const long long rank64 = wi + static_cast<long long>(k) * nw;
        if (rank64 >= units) return false;
        const unsigned rank = static_cast<unsigned>(rank64);
        const unsigned nt = static_cast<unsigned>(p.ntile), H = static_cast<unsigned>(p.H);
        const unsigned ir = per_tile ? rank / nt : rank;
        const unsigned fs = ir / BH, bh = ir - fs * BH;
        const unsigned f = p.reverse ? static_cast<unsigned>(p.F) - 1u - fs : fs;
        const unsigned b = bh / H, h = bh - b * H;
        item = (static_cast<long long>(b) * p.F + f) * p.H + h;
        nb = per_tile ? static_cast<int>(rank - ir * nt) : 0;
        ne = per_tile ? nb + 1 : p.ntile;
        if (ring > 0) {
            const unsigned R = static_cast<unsigned>(ring), use_u = fs / R;
            slot = (static_cast<long long>(b) * ring + (fs - use_u * R)) * p.H + h;
            use = static_cast<int>(use_u);
        } else {
            slot = item;
        }
        return true;
    }
};

// FMT_FP8: q is e4m3 (tm_q maps bytes, one 128-column box per token row).
// FMT_FP4: q is NVFP4 (tm_q maps the packed codes, one box of dk/2 bytes per
// token row, unswizzled; dk = 64 or 128).
template <int FMT>
__device__ __forceinline__ void output_role(const CUtensorMap* tm_q, const CUtensorMap* tm_s,
                                            const CUtensorMap* tm_out, const Params& p, const Sched& sc,
                                            uint8_t* smem) {
    constexpr bool FP8 = FMT == FMT_FP8;
    constexpr bool FP4 = FMT == FMT_FP4;
    constexpr bool LP = FMT != FMT_BF16;
    constexpr int QS = QSTAGES;
    uint8_t* qring = smem;
    uint8_t* sring = qring + QSTAGES * QTILE_BYTES;
    uint8_t* ostage = sring + SSTAGES * STILE_BYTES;   // [4 warps][2][OSTAGE_BYTES]
    uint64_t* bars = reinterpret_cast<uint64_t*>(ostage + 4 * 2 * OSTAGE_BYTES);
    uint64_t* qfull = bars;
    uint64_t* qempty = qfull + QSTAGES;
    uint64_t* sfull = qempty + QSTAGES;
    uint64_t* sempty = sfull + SSTAGES;
    uint64_t* tfull = sempty + SSTAGES;
    uint64_t* tempty = tfull + ACCS;
    uint64_t* final_bar = tempty + ACCS;
    uint64_t* nready = final_bar + 1;                 // [NSLOTS] row norms of a tile written
    uint64_t* nfree = nready + NSLOTS;                // [NSLOTS] epilogue has read them
    uint64_t* qdec = nfree + NSLOTS;                  // [QSTAGES] FP8: q slot decoded (qfull: raw landed)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qdec + QSTAGES);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* rnorm = reinterpret_cast<float*>(smem + QSTAGES * QTILE_BYTES + SSTAGES * STILE_BYTES +
                                            4 * 2 * OSTAGE_BYTES + BAR_BYTES);   // [NSLOTS][TILE_M]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kboxes = p.dk > 64 ? 2 : 1;
    const int vboxes = p.dv > 64 ? 2 : 1;
    const int sboxes = p.b_mn ? vboxes : kboxes;   // 64-column boxes of the state tile

    // never-loaded boxes (dk <= 64) must read as zero
    if (!LP && (kboxes < 2 || sboxes < 2))
        for (int i = threadIdx.x; i < (QSTAGES * QTILE_BYTES + SSTAGES * STILE_BYTES) / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        // a q slot is released by the MMA commit and, with the folded prologue, by the norm threads
        for (int s = 0; s < QS; ++s) {
            mbar_init(&qfull[s], 1);
            mbar_init(&qempty[s], 1 + ((!LP && p.norm_q) ? NORM_THREADS : 0));
            mbar_init(&qdec[s], DEC_THREADS);
        }
        for (int s = 0; s < SSTAGES; ++s) { mbar_init(&sfull[s], 1); mbar_init(&sempty[s], 1); }
        for (int a = 0; a < ACCS; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        for (int n = 0; n < NSLOTS; ++n) {
            mbar_init(&nready[n], NORM_THREADS);
            mbar_init(&nfree[n], 128);
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(tm_q);
        if (sc.ring == 0) prefetch_tmap(tm_s);
        prefetch_tmap(tm_out);
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
            int qs = 0, ss = 0;
            uint32_t qph = 0, sph = 0;
            long long q_issued = 0, s_issued = 0;
            long long item, slot;
            int nb, ne, use;
            bool stop = false;
            for (int k = 0; !stop && !*abort_flag && sc.segment(p, k, item, nb, ne, slot, use); ++k) {
                const int frame = static_cast<int>(item / p.H), h = static_cast<int>(item % p.H);
                if (k > 0) { if (++ss == SSTAGES) { ss = 0; sph ^= 1; } }
                if (!mbar_wait(&sempty[ss], sph ^ 1, p.wait_limit_ns, abort_flag, 3010000 + (k & 0xffff))) break;
                if (sc.fused) {
                    if (!wait_count_geq(sc.flags + slot, (use + 1) * sc.flag_target, p.wait_limit_ns, abort_flag,
                                        3020000 + (k & 0xffff)))
                        break;
                    fence_proxy_async_global();  // the published state is read through the async proxy
                }
                if (sc.ring > 0) {
                    mbar_arrive_expect_tx(&sfull[ss], STILE_BYTES);
                    bulk_load(sring + ss * STILE_BYTES,
                              reinterpret_cast<const uint8_t*>(sc.s_ring) + static_cast<size_t>(slot) * RING_TILE_BF16,
                              STILE_BYTES, &sfull[ss]);
                } else {
                    mbar_arrive_expect_tx(&sfull[ss], sboxes * BOX_BYTES);
                    for (int bx = 0; bx < sboxes; ++bx)
                        tma_load_3d(sring + ss * STILE_BYTES + bx * BOX_BYTES, tm_s, &sfull[ss], 64 * bx, 0,
                                    static_cast<int>(slot));
                }
                ++s_issued;
                for (int nt = nb; nt < ne; ++nt) {
                    if constexpr (LP) {
                        // raw e4m3 / NVFP4 tile into box 1 of the slot, decoded there in place
                        if (!mbar_wait(&qempty[qs], qph ^ 1, p.wait_limit_ns, abort_flag)) { stop = true; break; }
                        mbar_arrive_expect_tx(&qfull[qs], FP8 ? RAW_BYTES : TILE_M * (p.dk / 2));
                        tma_load_4d(qring + qs * QTILE_BYTES + BOX_BYTES, tm_q, &qfull[qs], 0, h, nt * TILE_M,
                                    frame);
                        ++q_issued;
                        if (++qs == QS) { qs = 0; qph ^= 1; }
                    } else {
                        if (!mbar_wait(&qempty[qs], qph ^ 1, p.wait_limit_ns, abort_flag)) { stop = true; break; }
                        mbar_arrive_expect_tx(&qfull[qs], kboxes * BOX_BYTES);
                        for (int bx = 0; bx < kboxes; ++bx)
                            tma_load_4d(qring + qs * QTILE_BYTES + bx * BOX_BYTES, tm_q, &qfull[qs], 64 * bx, h,
                                        nt * TILE_M, frame);
                        ++q_issued;
                        if (++qs == QSTAGES) { qs = 0; qph ^= 1; }
                    }
                }
            }
            for (long long kq = (q_issued > QS ? q_issued - QS : 0); kq < q_issued; ++kq)
                mbar_wait_drain(&qfull[kq % QS], static_cast<uint32_t>((kq / QS) & 1), p.wait_limit_ns);
            for (long long ks = (s_issued > SSTAGES ? s_issued - SSTAGES : 0); ks < s_issued; ++ks)
                mbar_wait_drain(&sfull[ks % SSTAGES], static_cast<uint32_t>((ks / SSTAGES) & 1), p.wait_limit_ns);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t IDESC = p.b_mn ? idesc_bf16(128, 128, 0, 1) : idesc_bf16(128, 128, 0, 0);
            const int nk = (p.dk + 15) / 16;
            int qs = 0, ss = 0, acc = 0;
            uint32_t qph = 0, sph = 0, aph = 0;
            long long item;
            int nb, ne;
            bool stop = false;
            long long slot;
            int use;
            for (int k = 0; !stop && !*abort_flag && sc.segment(p, k, item, nb, ne, slot, use); ++k) {
                if (k > 0) { if (++ss == SSTAGES) { ss = 0; sph ^= 1; } }
                if (!mbar_wait(&sfull[ss], sph, p.wait_limit_ns, abort_flag, 3110000 + (k & 0xffff))) break;
                for (int nt = nb; nt < ne; ++nt) {
                    if (!mbar_wait(&tempty[acc], aph ^ 1, p.wait_limit_ns, abort_flag) ||
                        !mbar_wait(LP ? &qdec[qs] : &qfull[qs], qph, p.wait_limit_ns, abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(qring + qs * QTILE_BYTES);
                    const uint32_t b_base = smem_u32(sring + ss * STILE_BYTES);
                    const uint32_t d_tmem = tmem_base + acc * 128;
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint64_t ad = smem_desc(a_base + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = p.b_mn ? smem_desc(b_base + kk * 2048, BOX_BYTES, 1024)
                                                   : smem_desc(b_base + (kk >> 2) * BOX_BYTES + (kk & 3) * 32, 16, 1024);
                        mma_bf16(d_tmem, ad, bd, IDESC, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&qempty[qs]);
                    mma_commit(&tfull[acc]);
                    if (nt + 1 == ne) mma_commit(&sempty[ss]);
                    if (++qs == QS) { qs = 0; qph ^= 1; }
                    if (++acc == ACCS) { acc = 0; aph ^= 1; }
                }
                // ring mode: the image is in shared memory, the scan may reuse its slot
                // (a release, which takes a while, so it follows the item's MMAs)
                if (sc.ring > 0 && !stop) red_release_add(sc.s_free + slot, 1);
            }
            mma_commit(final_bar);
            mbar_wait_drain(final_bar, 0, p.wait_limit_ns);
        }
    } else if (warp >= 6 && warp < threads<FMT>() / 32) {
        if constexpr (FP4) {
            // --------------------------------------------- NVFP4 q decoders
            // Thread t owns token row t of each tile: its dk/2 raw bytes sit in
            // box 1 of the slot, packed (row pitch dk/2), so rows of different
            // threads overlap the decoded rows: every decoder reads its raw row
            // into registers, all meet at a named barrier, then each writes row t
            // of boxes 0 and 1 (bf16, K-major, 128-byte swizzle).  e2m1 times the
            // E4M3 block scale is exact in f16 and in bf16.  The row's block
            // scales (dk/16 bytes) are loaded one tile ahead.
            const int t = threadIdx.x - 192;
            const int nsc = p.dk / 16;                 // 4 or 8 scales per row
            int qs = 0;
            uint32_t qph = 0;
            long long item;
            int nb, ne;
            int k = 0;
            bool have = sc.segment(p, 0, item, nb, ne);
            int nt = nb;
            auto load_sf = [&](long long it, int ntile) -> uint2 {
                const int tok = ntile * TILE_M + t;
                if (tok >= p.N) return make_uint2(0u, 0u);
                const size_t row = (static_cast<size_t>(it / p.H) * p.N + tok) * p.H + (it % p.H);
                if (nsc == 8) return __ldg(reinterpret_cast<const uint2*>(p.q_sf + row * 8));
                return make_uint2(__ldg(reinterpret_cast<const uint32_t*>(p.q_sf + row * 4)), 0u);
            };
            uint2 sf_cur = have ? load_sf(item, nt) : make_uint2(0u, 0u);
            while (have && !*abort_flag) {
                // the next tile of this CTA, and its scales (consumed next round)
                long long item2 = item;
                int nt2 = nt + 1, nb2 = nb, ne2 = ne, k2 = k;
                bool have2 = true;
                if (nt2 >= ne) {
                    k2 = k + 1;
                    have2 = sc.segment(p, k2, item2, nb2, ne2);
                    nt2 = nb2;
                }
                const uint2 sf_next = have2 ? load_sf(item2, nt2) : make_uint2(0u, 0u);
                if (!bar_and(2, DEC_THREADS, mbar_wait(&qfull[qs], qph, p.wait_limit_ns, abort_flag))) break;
                uint8_t* tile = qring + qs * QTILE_BYTES;
                uint32_t w[16];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    if (q4 * 32 < p.dk) {
                        const uint4 x = *reinterpret_cast<const uint4*>(tile + BOX_BYTES + t * (p.dk / 2) + 16 * q4);
                        w[4 * q4] = x.x; w[4 * q4 + 1] = x.y; w[4 * q4 + 2] = x.z; w[4 * q4 + 3] = x.w;
                    }
                }
                named_bar_sync(2, DEC_THREADS);   // every raw row has been read
#pragma unroll
                for (int g = 0; g < 8; ++g) {     // 16 columns 16g..16g+15: raw words 2g, 2g+1
                    if (g < nsc) {
                        const uint32_t s2 = e4m3_to_f16x2_bcast((g < 4 ? sf_cur.x : sf_cur.y) >> (8 * (g & 3)));
                        uint32_t h[8];
                        fp4x8_to_f16(w[2 * g], s2, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
                        fp4x8_to_f16(w[2 * g + 1], s2, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
#pragma unroll
                        for (int e = 0; e < 8; ++e) h[e] = f16x2_to_bf16x2_exact(h[e]);
                        uint8_t* rowp = tile + (g >> 2) * BOX_BYTES + t * 128;
                        const int c8 = 2 * (g & 3);
                        *reinterpret_cast<uint4*>(rowp + ((c8 ^ (t & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                        *reinterpret_cast<uint4*>(rowp + (((c8 + 1) ^ (t & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&qdec[qs]);
                if (++qs == QS) { qs = 0; qph ^= 1; }
                item = item2; nt = nt2; nb = nb2; ne = ne2; k = k2; have = have2; sf_cur = sf_next;
            }
        } else if constexpr (FP8) {
            // ------------------------------------------------ e4m3 q decoders
            // row t of each raw tile (box 1 of the slot): 8 chunks of 16 columns,
            // all read first, then decoded exactly to bf16 into row t of the
            // slot's K-major, 128-byte-swizzled boxes 0 and 1
            const int t = threadIdx.x - 192;
            int qs = 0;
            uint32_t qph = 0;
            long long item;
            int nb, ne;
            bool stop = false;
            for (int k = 0; !stop && !*abort_flag && sc.segment(p, k, item, nb, ne); ++k) {
                for (int nt = nb; nt < ne; ++nt) {
                    if (!mbar_wait(&qfull[qs], qph, p.wait_limit_ns, abort_flag)) {
                        stop = true;
                        break;
                    }
                    uint8_t* tile = qring + qs * QTILE_BYTES;
                    const int row = t;
                    uint4 q16[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        q16[c] = *reinterpret_cast<const uint4*>(tile + BOX_BYTES + row * 128 + ((c ^ (row & 7)) << 4));
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t* qw = reinterpret_cast<const uint32_t*>(&q16[c]);
                        uint32_t qb[8];
#pragma unroll
                        for (int wd = 0; wd < 4; ++wd) {
                            qb[2 * wd] = e4m3x2_to_bf16x2(static_cast<uint16_t>(qw[wd] & 0xffffu));
                            qb[2 * wd + 1] = e4m3x2_to_bf16x2(static_cast<uint16_t>(qw[wd] >> 16));
                        }
                        // columns 16c..16c+15 = bf16 box c/4, chunks 2(c%4) and 2(c%4)+1
                        uint8_t* rowp = tile + (c >> 2) * BOX_BYTES + row * 128;
                        const int c8 = 2 * (c & 3);
                        *reinterpret_cast<uint4*>(rowp + ((c8 ^ (row & 7)) << 4)) = make_uint4(qb[0], qb[1], qb[2], qb[3]);
                        *reinterpret_cast<uint4*>(rowp + (((c8 + 1) ^ (row & 7)) << 4)) =
                            make_uint4(qb[4], qb[5], qb[6], qb[7]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&qdec[qs]);
                    if (++qs == QS) { qs = 0; qph ^= 1; }
                }
            }
        } else if (p.norm_q) {
            // ---------------------------------------------------------- q row norms
            const int t = threadIdx.x - 192;  // 0..63: rows t and t + 64 of each tile
            int qs = 0, ns = 0;
            uint32_t qph = 0, nph = 0;
            long long item;
            int nb, ne;
            bool stop = false;
            for (int k = 0; !stop && !*abort_flag && sc.segment(p, k, item, nb, ne); ++k) {
                for (int nt = nb; nt < ne; ++nt) {
                    // the tile has landed, and the epilogue has read this norm slot's last contents
                    if (!mbar_wait(&qfull[qs], qph, p.wait_limit_ns, abort_flag) ||
                        !mbar_wait(&nfree[ns], nph ^ 1, p.wait_limit_ns, abort_flag)) {
                        stop = true;
                        break;
                    }
                    const uint8_t* tile = qring + qs * QTILE_BYTES;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int row = t + 64 * h2;
                        float ss = 0.0f;
                        for (int bx = 0; bx < kboxes; ++bx) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                // any chunk order sums the same row; rotate for distinct bank groups
                                const uint4 v4 = *reinterpret_cast<const uint4*>(
                                    tile + bx * BOX_BYTES + row * 128 + (((c + row) & 7) << 4));
                                const uint32_t* vs = reinterpret_cast<const uint32_t*>(&v4);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f2 =
                                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vs[e]));
                                    ss = fmaf(f2.x, f2.x, fmaf(f2.y, f2.y, ss));
                                }
                            }
                        }
                        rnorm[ns * TILE_M + row] = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
                    }
                    mbar_arrive(&nready[ns]);
                    mbar_arrive(&qempty[qs]);
                    if (++qs == QSTAGES) { qs = 0; qph ^= 1; }
                    if (++ns == NSLOTS) { ns = 0; nph ^= 1; }
                }
            }
        }
    } else if (warp >= 2 && warp < 6) {
        // ----------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        uint8_t* my_stage = ostage + quarter * 2 * OSTAGE_BYTES;
        int acc = 0, ob = 0, ns = 0;
        uint32_t aph = 0, nph = 0;
        const int ncol32 = (p.dv + 31) / 32;
        long long item;
        int nb, ne;
        bool stop = false;
        for (int k = 0; !stop && !*abort_flag && sc.segment(p, k, item, nb, ne); ++k) {
            const int frame = static_cast<int>(item / p.H), h = static_cast<int>(item % p.H);
            for (int nt = nb; nt < ne; ++nt) {
                // fused prologue: o_n = S q_n / max(|q_n|, eps), norms from the norm warps
                float rs = LP ? p.q_scale : 1.0f;
                if (!LP && p.norm_q) {
                    const bool okn =
                        __all_sync(0xffffffffu, mbar_wait(&nready[ns], nph, p.wait_limit_ns, abort_flag));
                    if (!okn) { stop = true; break; }
                    rs = rnorm[ns * TILE_M + quarter * 32 + lane];
                    mbar_arrive(&nfree[ns]);
                    if (++ns == NSLOTS) { ns = 0; nph ^= 1; }
                }
                const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, p.wait_limit_ns, abort_flag));
                if (!ok) { stop = true; break; }
                tc_fence_after();
                const uint32_t tbase = tmem_base + acc * 128 + (static_cast<uint32_t>(quarter * 32) << 16);
                uint32_t packed[64];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c < ncol32) {
                        uint32_t r32[32];
                        tmem_ld32(tbase + c * 32, r32);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            packed[c * 16 + e] = pack_bf16x2(__uint_as_float(r32[2 * e]) * rs,
                                                             __uint_as_float(r32[2 * e + 1]) * rs);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) packed[c * 16 + e] = 0u;
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
                if (++acc == ACCS) { acc = 0; aph ^= 1; }

                // staging buffer `ob` was last read by the TMA store issued two tiles ago
                if (lane == 0) bulk_wait_read<1>();
                __syncwarp();
                uint8_t* stg = my_stage + ob * OSTAGE_BYTES;
                const int row = lane;  // token row within this warp's 32
#pragma unroll
                for (int ch = 0; ch < 16; ++ch) {
                    const int box = ch >> 3, c8 = ch & 7;
                    if (box < vboxes) {
                        uint4 v = make_uint4(packed[ch * 4 + 0], packed[ch * 4 + 1], packed[ch * 4 + 2],
                                             packed[ch * 4 + 3]);
                        *reinterpret_cast<uint4*>(stg + box * OBOX_BYTES + row * 128 + ((c8 ^ (row & 7)) << 4)) = v;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                const int row0 = nt * TILE_M + quarter * 32;
                if (lane == 0 && row0 < p.N) {
                    for (int bx = 0; bx < vboxes; ++bx)
                        tma_store_4d(tm_out, stg + bx * OBOX_BYTES, 64 * bx, h, row0, frame);
                }
                if (lane == 0) bulk_commit();
                ob ^= 1;
            }
        }
        if (lane == 0) bulk_wait<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Standalone phase 3: persistent grid, contiguous tile ranges.
template <int FMT>
__global__ void __launch_bounds__(threads<FMT>(), 1)
    output_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
                  const __grid_constant__ CUtensorMap tm_out, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Sched sc;
    sc.t0 = (static_cast<long long>(blockIdx.x) * p.total) / gridDim.x;
    sc.t1 = (static_cast<long long>(blockIdx.x + 1) * p.total) / gridDim.x;
    sc.wi = 0;
    sc.nw = 1;
    sc.fused = false;
    sc.flags = nullptr;
    sc.flag_target = 0;
    sc.ring = 0;
    sc.s_free = nullptr;
    sc.s_ring = nullptr;
    output_role<FMT>(&tm_q, &tm_s, &tm_out, p, sc, smem);
}

}  // namespace k3
}  // namespace gdn
