// gdn_fwd_single.cuh -- the whole frame-wise GDN forward in one cooperative
// launch: the frame-parallel contractions, the sequential scan and the
// frame-parallel output pass run side by side and hand each frame on through
// small ring buffers that stay in L2 (SANA-WM article, "The Architecture":
// one latent frame per step, a decay gate and a delta-rule correction;
// wispaper summary, "Methodology" 1: frames scanned one by one).
//
// CTA roles, one CTA per SM, all resident at once (cooperative launch):
//   [0, n_scan)                       the scan of one (b, h) head each
//                                     (gdn_scan_head.cuh)
//   [n_scan, n_scan + n_contract)     A_f = K_f^T B_f K_f, U_f = V_f^T B_f K_f
//                                     for whole (b, f, h) items, or head pairs,
//                                     in scan order (gdn_k1_contract.cuh,
//                                     gdn_k1_pair.cuh, ring mode)
//   the rest                          O_f = Q_f S_f^T for whole items in scan
//                                     order (gdn_k3_output.cuh, ring mode)
// Step s of the scan of head (b, h) uses ring slot (b * W + s % W) * H + h of
// three rings: A (bf16), U (fp32) and the bf16 state image S, each slot one
// zero-padded 128 x 128 tile in its consumer's shared-memory image (ring_off
// in gdn_ptx.cuh), copied in and out as one contiguous bulk copy.  Per slot four
// counts order the hand-offs (all raised with release semantics and read
// with bounded acquire waits):
//   au_ready  frames of A/U written by the contraction   -> the scan loads
//   au_free   frames of A/U loaded by the scan            -> the contraction
//                                                           rewrites the slot
//   s_ready   frames of S stored by the scan              -> output loads
//   s_free    loads of the slot's S by output CTAs        -> the scan rewrites
// Every wait is for an earlier role in the chain contraction -> scan ->
// output, or for a step at least W earlier, and every role walks its work in
// scan order, so the waits always end; they are still bounded, and one that
// runs out records GDN_ERR_TIMEOUT.  With W frames of ring (a few MB to a few
// tens of MB), what the three-launch schedule writes to HBM and reads back --
// A_f, U_f and the per-frame states -- stays in L2, and HBM carries only the
// layer's own bytes: q, k, v, beta and alpha in, out and the final state out.
#pragma once

#include "gdn_k1_contract.cuh"
#include "gdn_k1_pair.cuh"
#include "gdn_k3_output.cuh"
#include "gdn_scan_head.cuh"

namespace gdn {
namespace fwd {

constexpr int THREADS = k2h::THREADS;
static_assert(THREADS >= k1::THREADS && THREADS >= k3::threads<FMT_FP8>(), "the block covers every role's warps");

template <int FMT>
constexpr size_t smem_bytes() {
    constexpr size_t a = k2h::SMEM_BYTES > k1::Lay<FMT>::SMEM ? k2h::SMEM_BYTES : k1::Lay<FMT>::SMEM;
    constexpr size_t b = k3::SMEM_BYTES > k1p::SMEM_BYTES ? k3::SMEM_BYTES : k1p::SMEM_BYTES;
    return a > b ? a : b;
}

struct Counts {
    int* s_ready;   // [B][W][H]
    int* s_free;    // [B][W][H]
    const __nv_bfloat16* s_ring;   // [B][W][H] state image tiles
    int n_scan;     // = B * H
    int n_contract;
    int pair;       // bf16 only: the contraction CTAs take head pairs (gdn_k1_pair.cuh; tm_k, tm_v are pair maps)
};

template <int FMT>
__global__ void __launch_bounds__(THREADS, 1)
    forward_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out,
                   const k1::Params p1, const k2h::Params p2, const k3::Params p3, const Counts c) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int cta = static_cast<int>(blockIdx.x);
    if (cta < c.n_scan) {
        k2h::scan_head_role(p2, cta, smem);
    } else if (cta < c.n_scan + c.n_contract) {
        if constexpr (FMT == FMT_BF16) {
            if (c.pair) {
                k1p::contract_pair_role(tm_k, tm_v, p1, cta - c.n_scan, c.n_contract, smem);
                return;
            }
        }
        k1::contract_role<FMT>(tm_k, tm_v, p1, cta - c.n_scan, c.n_contract, smem);
    } else {
        k3::Sched sc;
        sc.t0 = 0;
        sc.t1 = 0;
        sc.wi = cta - c.n_scan - c.n_contract;
        sc.nw = static_cast<int>(gridDim.x) - c.n_scan - c.n_contract;
        sc.fused = true;
        sc.flags = c.s_ready;
        sc.flag_target = 1;   // one scan CTA per head
        sc.ring = p2.ring;
        sc.s_free = c.s_free;
        sc.s_ring = c.s_ring;
        k3::output_role<FMT>(&tm_q, nullptr, &tm_out, p3, sc, smem);
    }
}

}  // namespace fwd
}  // namespace gdn
