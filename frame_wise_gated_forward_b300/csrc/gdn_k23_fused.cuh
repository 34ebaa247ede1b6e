// gdn_k23_fused.cuh -- phases 2 and 3 of the frame-wise GDN forward in one
// cooperative launch.
//
// The scan (phase 2) is a chain of F dependent steps that keeps only a few
// SMs busy, while the output pass (phase 3) is bound by HBM bandwidth and
// still saturates it on fewer SMs than the GPU has.  So the first n_scan CTAs
// run the scan (one R-row slice of one head each) and the remaining CTAs run
// the output pass as soon as each frame's state is published: after storing
// the bf16 state of item (b, f, h) a scan CTA adds 1 to flags[item] with
// release semantics; an output CTA waits (bounded) until flags[item] counts
// every slice of the head, then loads the state through TMA.  Output CTAs
// take whole items round-robin in frame-major order, so they follow the scan
// front, and each frame's state is read while it is still in L2.
//
// The scan never waits on the output CTAs, and the cooperative launch makes
// every CTA resident at once, so the waits always end.
#pragma once

#include "gdn_k2_scan.cuh"
#include "gdn_k3_output.cuh"

namespace gdn {
namespace k23 {

constexpr int THREADS = k3::THREADS;
static_assert(k3::THREADS >= k2::THREADS, "the output role's block covers the scan role's warps");

template <int R>
constexpr size_t smem_bytes() {
    return k2::Cfg<R>::SMEM_BYTES > k3::SMEM_BYTES ? k2::Cfg<R>::SMEM_BYTES : k3::SMEM_BYTES;
}

template <int R, int FMT>
__global__ void __launch_bounds__(k3::threads<FMT>(), 1)
    scan_output_kernel(const __grid_constant__ CUtensorMap tm_A, const __grid_constant__ CUtensorMap tm_U,
                       const __grid_constant__ CUtensorMap tm_S_store, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_S_load, const __grid_constant__ CUtensorMap tm_out,
                       const k2::Params p2, const k3::Params p3, int* flags, int n_scan) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (static_cast<int>(blockIdx.x) < n_scan) {
        k2::scan_role<R>(&tm_A, &tm_U, &tm_S_store, p2, blockIdx.x, flags, smem);
    } else {
        k3::Sched sc;
        sc.t0 = 0;
        sc.t1 = 0;
        sc.wi = static_cast<int>(blockIdx.x) - n_scan;
        sc.nw = static_cast<int>(gridDim.x) - n_scan;
        sc.fused = true;
        sc.flags = flags;
        sc.flag_target = p2.rsplit;
        sc.ring = 0;
        sc.s_free = nullptr;
        sc.s_ring = nullptr;
        k3::output_role<FMT>(&tm_q, &tm_S_load, &tm_out, p3, sc, smem);
    }
}

}  // namespace k23
}  // namespace gdn
