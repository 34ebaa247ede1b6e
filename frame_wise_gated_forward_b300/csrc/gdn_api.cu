// gdn_api.cu -- the C ABI of libgdn_b300.so: argument validation, workspace,
// tensor-map encoding and the three-phase launch sequence of the frame-wise
// Gated DeltaNet forward (see include/gdn.h for the contract).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gdn.h"
#include "gdn_bwd.cuh"
#include "gdn_fwd_single.cuh"
#include "gdn_k1_contract.cuh"
#include "gdn_k23_fused.cuh"
#include "gdn_step_fused.cuh"

namespace {


constexpr int kMaxDevices = 64;
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ULL};
std::atomic<int> g_fused_scan{1};
std::atomic<int> g_max_split{0};  // 0: automatic; 1: never split; k > 1: up to k token ranges per item
std::atomic<int> g_fused_step{1};  // one-launch step (gdn_step_fused.cuh) where it applies
std::atomic<int> g_single_pass{1};     // whole forward in one launch (gdn_fwd_single.cuh) where it applies
std::atomic<int> g_single_contract{0}; // contraction CTAs of the single pass (0: automatic)
std::atomic<int> g_single_ring{0};     // ring frames of the single pass (0: automatic)
std::atomic<int> g_host_chunk{0};      // frames per chunk of the pipelined host call (0: automatic)
std::atomic<int> g_pairs{0};           // phase 1 on head pairs where the shape allows it (off by default)

// Kernels of each element format (gdn::FMT_BF16, FMT_FP8, FMT_FP4).
using gdn::FMT_BF16;
using gdn::FMT_FP4;
using gdn::FMT_FP8;
const void* k1_fn(int fmt) {
    return fmt == FMT_FP8   ? reinterpret_cast<const void*>(gdn::k1::contract_kernel<FMT_FP8>)
           : fmt == FMT_FP4 ? reinterpret_cast<const void*>(gdn::k1::contract_kernel<FMT_FP4>)
                            : reinterpret_cast<const void*>(gdn::k1::contract_kernel<FMT_BF16>);
}
size_t k1_smem(int fmt) {
    return fmt == FMT_FP8 ? gdn::k1::SMEM_BYTES_FP8 : fmt == FMT_FP4 ? gdn::k1::SMEM_BYTES_FP4 : gdn::k1::SMEM_BYTES;
}
const void* k3_fn(int fmt) {
    return fmt == FMT_FP8   ? reinterpret_cast<const void*>(gdn::k3::output_kernel<FMT_FP8>)
           : fmt == FMT_FP4 ? reinterpret_cast<const void*>(gdn::k3::output_kernel<FMT_FP4>)
                            : reinterpret_cast<const void*>(gdn::k3::output_kernel<FMT_BF16>);
}
int k3_threads(int fmt) { return fmt == FMT_BF16 ? gdn::k3::threads<FMT_BF16>() : gdn::k3::threads<FMT_FP8>(); }
template <int R>
const void* k23_fn_r(int fmt) {
    return fmt == FMT_FP8   ? reinterpret_cast<const void*>(gdn::k23::scan_output_kernel<R, FMT_FP8>)
           : fmt == FMT_FP4 ? reinterpret_cast<const void*>(gdn::k23::scan_output_kernel<R, FMT_FP4>)
                            : reinterpret_cast<const void*>(gdn::k23::scan_output_kernel<R, FMT_BF16>);
}
const void* k23_fn(int R, int fmt) { return R == 16 ? k23_fn_r<16>(fmt) : R == 32 ? k23_fn_r<32>(fmt) : k23_fn_r<64>(fmt); }
size_t k23_smem(int R) {
    return R == 16 ? gdn::k23::smem_bytes<16>() : R == 32 ? gdn::k23::smem_bytes<32>() : gdn::k23::smem_bytes<64>();
}
const void* fwd_fn(int fmt) {
    return fmt == FMT_FP8   ? reinterpret_cast<const void*>(gdn::fwd::forward_kernel<FMT_FP8>)
           : fmt == FMT_FP4 ? reinterpret_cast<const void*>(gdn::fwd::forward_kernel<FMT_FP4>)
                            : reinterpret_cast<const void*>(gdn::fwd::forward_kernel<FMT_BF16>);
}
size_t fwd_smem(int fmt) {
    return fmt == FMT_FP8   ? gdn::fwd::smem_bytes<FMT_FP8>()
           : fmt == FMT_FP4 ? gdn::fwd::smem_bytes<FMT_FP4>()
                            : gdn::fwd::smem_bytes<FMT_BF16>();
}

// ------------------------------------------------------------------ devices
struct DeviceState {
    bool probed = false;
    bool ok = false;
    int sms = 0;
    bool coop = false;     // cooperative launches possible with one fused CTA per SM
    bool coop_k1 = false;  // the same for the contraction kernel (needed to split items)
    bool coop_single = false;  // the same for the single-pass forward kernel
    cudaMemPool_t pool = nullptr;
    cudaStream_t copy_in = nullptr;   // host -> device copies of the pipelined host call
    cudaStream_t copy_out = nullptr;  // device -> host copies of the pipelined host call
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

gdn_status device_ready(int* dev_out, DeviceState** st_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GDN_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState& d = g_dev[dev];
    if (!d.probed) {
        d.probed = true;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) { cudaGetLastError(); return GDN_ERR_NO_DEVICE; }
        // the kernels are built for sm_103a only
        if (prop.major != 10 || prop.minor != 3) return GDN_ERR_NO_DEVICE;
        d.sms = prop.multiProcessorCount;
        if (g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                cudaGetLastError();
                return GDN_ERR_NO_DEVICE;
            }
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) { cudaGetLastError(); return GDN_ERR_ALLOC; }
        unsigned long long keep = ~0ULL;  // keep freed workspace cached in the pool
        cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (cudaStreamCreateWithFlags(&d.copy_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&d.copy_out, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_LAUNCH;
        }
        auto smem_attr = [](const void* fn, size_t bytes) {
            return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) ==
                   cudaSuccess;
        };
        using namespace gdn;
        bool fmt_ok = true;
        for (int fmt : {FMT_BF16, FMT_FP8, FMT_FP4}) {
            fmt_ok = fmt_ok && smem_attr(k1_fn(fmt), k1_smem(fmt)) && smem_attr(k3_fn(fmt), k3::SMEM_BYTES) &&
                     smem_attr(fwd_fn(fmt), fwd_smem(fmt));
            for (int R : {16, 32, 64}) fmt_ok = fmt_ok && smem_attr(k23_fn(R, fmt), k23_smem(R));
        }
        if (!fmt_ok ||
            !smem_attr(reinterpret_cast<const void*>(k2::scan_kernel<16>), k2::Cfg<16>::SMEM_BYTES) ||
            !smem_attr(reinterpret_cast<const void*>(k2::scan_kernel<32>), k2::Cfg<32>::SMEM_BYTES) ||
            !smem_attr(reinterpret_cast<const void*>(k2::scan_kernel<64>), k2::Cfg<64>::SMEM_BYTES) ||

            !smem_attr(reinterpret_cast<const void*>(k1p::contract_pair_kernel), k1p::SMEM_BYTES) ||
            !smem_attr(reinterpret_cast<const void*>(step::step_kernel), step::SMEM_BYTES) ||
            !smem_attr(reinterpret_cast<const void*>(bwd::frame_grad_kernel), bwd::FRAME_SMEM) ||
            !smem_attr(reinterpret_cast<const void*>(bwd::token_grad_kernel), bwd::TOKEN_SMEM)) {
            cudaGetLastError();
            return GDN_ERR_LAUNCH;
        }
        int coop = 0, per_sm = 0;
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k23::scan_output_kernel<64, FMT_BF16>, k23::THREADS,
                                                          k23::smem_bytes<64>()) != cudaSuccess)
            per_sm = 0;
        cudaGetLastError();
        d.coop = coop != 0 && per_sm >= 1;
        int per_sm_k1 = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_k1, k1::contract_kernel<FMT_BF16>, k1::THREADS,
                                                          k1::SMEM_BYTES) != cudaSuccess)
            per_sm_k1 = 0;
        cudaGetLastError();
        d.coop_k1 = coop != 0 && per_sm_k1 >= 1;
        int per_sm_single = 1;
        for (int fmt : {FMT_BF16, FMT_FP8, FMT_FP4}) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fwd_fn(fmt), fwd::THREADS, fwd_smem(fmt)) !=
                cudaSuccess)
                n = 0;
            per_sm_single = std::min(per_sm_single, n);
        }
        cudaGetLastError();
        d.coop_single = coop != 0 && per_sm_single >= 1;
        d.ok = true;
    }
    if (!d.ok) return GDN_ERR_NO_DEVICE;
    *dev_out = dev;
    *st_out = &d;
    return GDN_OK;
}

// ------------------------------------------------------------- validation
bool dim_ok(int d) { return d >= 16 && d <= 128 && d % 16 == 0; }

struct Range {
    uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// in_bits: bits per q/k/v element (16: bf16, 8: fp8, 4: NVFP4 codes); out is always bf16
gdn_status validate(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                    const float* state_in, const void* out, const float* state_out, int B, int H, int F, int N,
                    int dk, int dv, int in_bits = 16) {
    if (!q || !k || !v || !alpha || !beta || !out) return GDN_ERR_NULL_PTR;
    if (B < 1 || H < 1 || F < 1 || N < 1) return GDN_ERR_BAD_DIM;
    if (!dim_ok(dk) || !dim_ok(dv)) return GDN_ERR_UNSUPPORTED;
    const long long tok = static_cast<long long>(B) * F * N;
    const long long elems = tok * H * std::max(dk, dv);
    if (elems >= (1LL << 31) || static_cast<long long>(B) * F * H >= (1LL << 31)) return GDN_ERR_BAD_DIM;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return GDN_ERR_MISALIGNED;
    if (!a4(alpha) || !a4(beta) || (state_in && !a4(state_in)) || (state_out && !a4(state_out)))
        return GDN_ERR_MISALIGNED;
    const uintptr_t qb = reinterpret_cast<uintptr_t>(q), kb = reinterpret_cast<uintptr_t>(k),
                    vb = reinterpret_cast<uintptr_t>(v), ob = reinterpret_cast<uintptr_t>(out);
    const Range rq{qb, qb + static_cast<uintptr_t>(tok * H * dk * in_bits / 8)};
    const Range rk{kb, kb + static_cast<uintptr_t>(tok * H * dk * in_bits / 8)};
    const Range rv{vb, vb + static_cast<uintptr_t>(tok * H * dv * in_bits / 8)};
    const Range ro{ob, ob + static_cast<uintptr_t>(tok * H * dv * 2)};
    const uintptr_t ab = reinterpret_cast<uintptr_t>(alpha), bb = reinterpret_cast<uintptr_t>(beta);
    const Range ra{ab, ab + static_cast<uintptr_t>(static_cast<long long>(B) * F * H * 4)};
    const Range rb{bb, bb + static_cast<uintptr_t>(tok * H * 4)};
    const uintptr_t sbytes = static_cast<uintptr_t>(static_cast<long long>(B) * H * dv * dk * 4);
    if (overlap(ro, rq) || overlap(ro, rk) || overlap(ro, rv) || overlap(ro, ra) || overlap(ro, rb))
        return GDN_ERR_ALIAS;
    if (state_in) {
        const Range rs{reinterpret_cast<uintptr_t>(state_in), reinterpret_cast<uintptr_t>(state_in) + sbytes};
        if (overlap(ro, rs)) return GDN_ERR_ALIAS;
        if (state_out && state_out != state_in) {
            const Range rso{reinterpret_cast<uintptr_t>(state_out), reinterpret_cast<uintptr_t>(state_out) + sbytes};
            if (overlap(rs, rso)) return GDN_ERR_ALIAS;
        }
    }
    if (state_out) {
        const Range rso{reinterpret_cast<uintptr_t>(state_out), reinterpret_cast<uintptr_t>(state_out) + sbytes};
        if (overlap(ro, rso) || overlap(rq, rso) || overlap(rk, rso) || overlap(rv, rso) || overlap(ra, rso) ||
            overlap(rb, rso))
            return GDN_ERR_ALIAS;
    }
    return GDN_OK;
}

// Every pointer the kernels dereference must be device memory: a host pointer
// handed to a kernel would be an illegal access.
bool is_device_ptr(const void* p) {
    if (p == nullptr) return true;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// ------------------------------------------------------------- workspace
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Work plan of the contraction kernel on a grid of `grid` CTAs: whole items
// for as many full rounds as fit, then the remaining items, either whole or
// split into token ranges so that the last round is about as long as the
// others (see gdn::k1::unit_of).  A split costs a fixed few microseconds (the
// fp32 partial sums go through L2 and the splits wait for each other), which
// measured on B300 about what it saves at 14 chunks per item; so the automatic
// plan splits only items of at least kMinSplitChunks 64-token chunks.
constexpr int kMinSplitChunks = 32;
struct SplitPlan {
    int whole, rem, split_per, work;
};
SplitPlan plan_split(long long items, int chunks, int grid, bool allow_split) {
    SplitPlan sp;
    sp.whole = static_cast<int>(items >= grid ? (items / grid) * grid : 0);
    sp.rem = static_cast<int>(items - sp.whole);
    const int mode = g_max_split.load();
    int cap = mode == 0 ? (chunks >= kMinSplitChunks ? chunks : 1) : mode;
    sp.split_per = (sp.rem > 0 && allow_split) ? std::max(1, std::min({cap, chunks, grid / sp.rem})) : 1;
    if (sp.split_per == 1) {  // every item whole
        sp.whole = static_cast<int>(items);
        sp.rem = 0;
    }
    sp.work = sp.whole + sp.rem * sp.split_per;
    return sp;
}

struct Layout {
    size_t a_off, u_off, s_off, f_off, c_off, p_off, total;
};
Layout layout_of(long long items, int dk, int dv, const SplitPlan& sp) {
    Layout L;
    L.a_off = 0;
    L.u_off = align256(L.a_off + static_cast<size_t>(items) * dk * dk * 2);
    L.s_off = align256(L.u_off + static_cast<size_t>(items) * dv * dk * 4);
    L.f_off = align256(L.s_off + static_cast<size_t>(items) * dv * dk * 2);   // per-item ready counts
    L.c_off = L.f_off + static_cast<size_t>(items) * 4;                        // split-item counters
    L.p_off = align256(L.c_off + static_cast<size_t>(items) * 4);             // split partial sums
    L.total = align256(L.p_off + static_cast<size_t>(sp.rem) * sp.split_per * (dk * dk + dv * dk) * 4);
    return L;
}

int chunks_of(int N) { return (N + gdn::k1::CHUNK - 1) / gdn::k1::CHUNK; }

// ------------------------------------------------------------ tensor maps
bool encode(CUtensorMap* m, void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
            const cuuint32_t* box) {
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides_bytes, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
// token tensor [BF, N, H, d] bf16, box (64, 1, rows, 1)
bool encode_tokens(CUtensorMap* m, const void* base, int BF, int N, int H, int d, int rows) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BF)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                                   static_cast<cuuint64_t>(N) * H * d * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
    return encode(m, const_cast<void*>(base), 4, dims, strides, box);
}
// fp8 token tensor [BF, N, H, d] bytes, box (128, 1, rows, 1): one 128-byte
// row per token, columns past d zero-filled
bool encode_tokens8(CUtensorMap* m, const void* base, int BF, int N, int H, int d, int rows) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BF)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H) * d,
                                   static_cast<cuuint64_t>(N) * H * d};
    const cuuint32_t box[4] = {128, 1, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// NVFP4 token tensor [BF, N, H, d/2] bytes (two codes per byte), box (d/2, 1,
// rows, 1): one unswizzled row of d/2 bytes per token (d = 64 or 128)
bool encode_tokens4(CUtensorMap* m, const void* base, int BF, int N, int H, int d, int rows) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d / 2), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BF)};
    const cuuint64_t st[3] = {static_cast<cuuint64_t>(d / 2), static_cast<cuuint64_t>(H) * d / 2,
                              static_cast<cuuint64_t>(N) * H * d / 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(d / 2), 1, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, st, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// q, k, v token maps in the call's element format; rows_k: token rows per box of k and v
bool encode_inputs(CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tq, const void* q, const void* k, const void* v,
                   int fmt, int BF, int N, int H, int dk, int dv, int rows_k, int rows_q);

// bf16 token tensor of two-head rows: [T, H, 128] as {64 columns, 8 tokens,
// 2 halves, H heads, T / 8 groups}, box {64, 8, 2, 2, rows / 8}: each box row
// spans the 512 contiguous bytes of two heads, and shared memory receives
// 8-token x 128-byte swizzle atoms (gdn_k1_pair.cuh).  T % 8 == 0.
bool encode_pairs(CUtensorMap* m, const void* base, long long T, int H, int rows) {
    const cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T / 8)};
    const cuuint64_t strides[4] = {static_cast<cuuint64_t>(H) * 256, 128, 256, static_cast<cuuint64_t>(H) * 256 * 8};
    const cuuint32_t box[5] = {64, 8, 2, 2, static_cast<cuuint32_t>(rows / 8)};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per-item matrix [items, rows_total, cols] bf16, box (64, rows, 1)
bool encode_mats(CUtensorMap* m, const void* base, long long items, int rows_total, int cols, int rows) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows_total),
                                static_cast<cuuint64_t>(items)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                                   static_cast<cuuint64_t>(rows_total) * cols * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
    return encode(m, const_cast<void*>(base), 3, dims, strides, box);
}

// per-item fp32 matrix [items, rows_total, cols], no swizzle, box (128, rows, 1)
bool encode_mats_f32(CUtensorMap* m, const void* base, long long items, int rows_total, int cols, int rows) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows_total),
                                static_cast<cuuint64_t>(items)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 4,
                                   static_cast<cuuint64_t>(rows_total) * cols * 4};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_inputs(CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tq, const void* q, const void* k, const void* v,
                   int fmt, int BF, int N, int H, int dk, int dv, int rows_k, int rows_q) {
    if (fmt == FMT_FP8)
        return encode_tokens8(tk, k, BF, N, H, dk, rows_k) && encode_tokens8(tv, v, BF, N, H, dv, rows_k) &&
               encode_tokens8(tq, q, BF, N, H, dk, rows_q);
    if (fmt == FMT_FP4)
        return encode_tokens4(tk, k, BF, N, H, dk, rows_k) && encode_tokens4(tv, v, BF, N, H, dv, rows_k) &&
               encode_tokens4(tq, q, BF, N, H, dk, rows_q);
    return encode_tokens(tk, k, BF, N, H, dk, rows_k) && encode_tokens(tv, v, BF, N, H, dv, rows_k) &&
           encode_tokens(tq, q, BF, N, H, dk, rows_q);
}

// ------------------------------------------------------------- the pass
struct PassArgs {
    const void *q, *k, *v;
    const float *alpha, *beta, *state_in;
    void* out;
    float* state_out;
    int B, H, F, N, dk, dv;
    int reverse = 0;
    int prologue = 0;          // raw q, k and gate logits: normalize and apply the gates in the kernels
    float alpha_scale = 0.0f;  // prologue: alpha = exp(-softplus(a) * alpha_scale)
    int fmt = gdn::FMT_BF16;   // q, k, v element format (FMT_FP8: value = scale * e4m3; FMT_FP4: NVFP4)
    const uint8_t *q_sf = nullptr, *k_sf = nullptr, *v_sf = nullptr;   // NVFP4 block scales
    float q_scale = 1.0f, k_scale = 1.0f, v_scale = 1.0f;
    // forward with saved activations: A_f (bf16 [B, F, H, dk, dk]) and the
    // per-frame state images (bf16 [B, F, H, dv, dk]) go to these caller
    // buffers instead of the workspace (multi-launch schedule)
    void* ext_A = nullptr;
    void* ext_S = nullptr;
};

// Phase 1 on head pairs (gdn_k1_pair.cuh): bf16 inputs, d = 128, an even
// number of heads and frames of a multiple of 8 tokens.
bool pair_applies(const PassArgs& a) {
    return g_pairs.load() != 0 && a.fmt == gdn::FMT_BF16 && a.dk == 128 && a.dv == 128 && a.H % 2 == 0 &&
           a.N % 8 == 0;
}

// Rows of S per scan CTA.  Standalone scan: the smallest slice that keeps
// all scan CTAs in one wave.  Fused with the output pass: the smallest slice
// that leaves most SMs to the output pass (0: do not fuse).
int scan_rows_standalone(int B, int H, int dv, int sms) {
    for (int R : {16, 32, 64})
        if (dv % R == 0 && static_cast<long long>(B) * H * (dv / R) <= sms) return R;
    return dv % 64 == 0 ? 64 : (dv % 32 == 0 ? 32 : 16);
}
int scan_rows_fused(int B, int H, int dv, int sms) {
    const int forced = g_fused_scan.load();
    if (forced == 16 || forced == 32 || forced == 64)
        return (dv % forced == 0 && static_cast<long long>(B) * H * (dv / forced) < sms) ? forced : 0;
    // at most half of the SMs scan; the rest run the output pass
    for (int R : {16, 32, 64})
        if (dv % R == 0 && static_cast<long long>(B) * H * (dv / R) <= sms / 2) return R;
    return 0;
}

// Launch the three phases (and the step path's partial reduction) on `stream`
// with the workspace `ws` laid out as `L`.  Records ev[0..3] around the
// phases when `ev` is not null.
gdn_status launch_phases(const PassArgs& a, uint8_t* ws, const Layout& L, const SplitPlan& sp,
                         const DeviceState* ds, cudaStream_t stream, cudaEvent_t const* ev) {
    const long long items = static_cast<long long>(a.B) * a.F * a.H;
    const int BF = a.B * a.F;
    __nv_bfloat16* A_ws = reinterpret_cast<__nv_bfloat16*>(a.ext_A ? static_cast<uint8_t*>(a.ext_A) : ws + L.a_off);
    float* U_ws = reinterpret_cast<float*>(ws + L.u_off);
    __nv_bfloat16* S_all = reinterpret_cast<__nv_bfloat16*>(a.ext_S ? static_cast<uint8_t*>(a.ext_S) : ws + L.s_off);
    float* partial = reinterpret_cast<float*>(ws + L.p_off);
    const int Rf = (g_fused_scan.load() != 0 && ds->coop) ? scan_rows_fused(a.B, a.H, a.dv, ds->sms) : 0;
    const int R = Rf != 0 ? Rf : scan_rows_standalone(a.B, a.H, a.dv, ds->sms);
    int* flags = reinterpret_cast<int*>(ws + L.f_off);
    CUtensorMap tm_k, tm_v, tm_q, tm_out, tm_A, tm_U, tm_S_store, tm_S_load;
    const bool enc_in = encode_inputs(&tm_k, &tm_v, &tm_q, a.q, a.k, a.v, a.fmt, BF, a.N, a.H, a.dk, a.dv,
                                      gdn::k1::CHUNK, gdn::k3::TILE_M);
    const bool enc = enc_in &&
                     encode_tokens(&tm_out, a.out, BF, a.N, a.H, a.dv, 32) &&
                     encode_mats(&tm_A, A_ws, items, a.dk, a.dk, 128) &&
                     encode_mats_f32(&tm_U, U_ws, items, a.dv, a.dk, R) &&
                     encode_mats(&tm_S_store, S_all, items, a.dv, a.dk, R) &&
                     encode_mats(&tm_S_load, S_all, items, a.dv, a.dk, 128);
    if (!enc) return GDN_ERR_LAUNCH;
    const unsigned long long lim = g_wait_limit_ns.load();

    // ready counts of the fused scan/output launch and the split-item counters start at zero
    if (cudaMemsetAsync(ws + L.f_off, 0, static_cast<size_t>(items) * 8, stream) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    // phase 1
    gdn::k1::Params p1;
    std::memset(&p1, 0, sizeof(p1));   // ring mode off
    p1.beta = a.beta;
    p1.A_ws = A_ws;
    p1.U_ws = U_ws;
    p1.partial = partial;
    p1.counters = reinterpret_cast<int*>(ws + L.c_off);
    p1.H = a.H;
    p1.N = a.N;
    p1.dk = a.dk;
    p1.dv = a.dv;
    p1.items = static_cast<int>(items);
    p1.whole = sp.whole;
    p1.split_per = sp.split_per;
    p1.chunks = chunks_of(a.N);
    p1.work = sp.work;
    p1.norm_k = a.prologue;
    p1.beta_sigmoid = a.prologue;
    p1.a_scale = a.fmt != gdn::FMT_BF16 ? a.k_scale * a.k_scale : 1.0f;
    p1.u_scale = a.fmt != gdn::FMT_BF16 ? a.k_scale * a.v_scale : 1.0f;
    p1.k_sf = a.k_sf;
    p1.v_sf = a.v_sf;
    p1.wait_limit_ns = lim;
    if (ev) cudaEventRecord(ev[0], stream);
    const bool pairs = pair_applies(a);
    if (pairs) {
        // head pairs, whole: one unit per (b, f, head pair)
        if (!encode_pairs(&tm_k, a.k, static_cast<long long>(BF) * a.N, a.H, gdn::k1p::CHUNK) ||
            !encode_pairs(&tm_v, a.v, static_cast<long long>(BF) * a.N, a.H, gdn::k1p::CHUNK))
            return GDN_ERR_LAUNCH;
        p1.whole = p1.items;
        p1.split_per = 1;
        p1.work = p1.items / 2;
    }
    const int grid1 = std::min(p1.work, ds->sms);
    const void* fn1 = pairs ? reinterpret_cast<const void*>(gdn::k1p::contract_pair_kernel) : k1_fn(a.fmt);
    const size_t smem1 = pairs ? gdn::k1p::SMEM_BYTES : k1_smem(a.fmt);
    void* args1[] = {&tm_k, &tm_v, &p1};
    // split items wait for each other's partial sums: then all CTAs must be resident
    const cudaError_t e1 =
        (!pairs && sp.rem > 0)
            ? cudaLaunchCooperativeKernel(fn1, dim3(grid1), dim3(gdn::k1::THREADS), args1, smem1, stream)
            : cudaLaunchKernel(fn1, dim3(grid1), dim3(gdn::k1::THREADS), args1, smem1, stream);
    if (e1 != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_LAUNCH;
    }
    // phases 2 and 3
    if (ev) cudaEventRecord(ev[1], stream);
    gdn::k2::Params p2;
    p2.alpha = a.alpha;
    p2.state_in = a.state_in;
    p2.state_out = a.state_out;
    p2.H = a.H;
    p2.F = a.F;
    p2.dk = a.dk;
    p2.dv = a.dv;
    p2.rsplit = a.dv / R;
    p2.reverse = a.reverse;
    p2.alpha_gate = a.prologue;
    p2.alpha_scale = a.alpha_scale;
    p2.wait_limit_ns = lim;
    gdn::k3::Params p3;
    p3.B = a.B;
    p3.H = a.H;
    p3.F = a.F;
    p3.N = a.N;
    p3.dk = a.dk;
    p3.dv = a.dv;
    p3.ntile = (a.N + gdn::k3::TILE_M - 1) / gdn::k3::TILE_M;
    p3.total = items * p3.ntile;
    p3.reverse = a.reverse;
    p3.norm_q = a.prologue;
    p3.q_scale = a.fmt != gdn::FMT_BF16 ? a.q_scale : 1.0f;
    p3.q_sf = a.q_sf;
    p3.b_mn = 0;
    p3.wait_limit_ns = lim;
    const int n_scan = a.B * a.H * p2.rsplit;
    if (Rf != 0) {
        // one cooperative launch: scan CTAs publish per-frame states, output CTAs follow them
        const long long workers = std::min<long long>(ds->sms - n_scan, std::max<long long>(1, items * p3.ntile));
        int grid = n_scan + static_cast<int>(workers);
        int n_scan_arg = n_scan;
        void* args[] = {&tm_A, &tm_U, &tm_S_store, &tm_q, &tm_S_load, &tm_out, &p2, &p3, &flags, &n_scan_arg};
        const void* fn = k23_fn(Rf, a.fmt);
        const size_t smem = k23_smem(Rf);
        if (ev) cudaEventRecord(ev[2], stream);
        const int threads = k3_threads(a.fmt);
        if (cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(threads), args, smem, stream) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_LAUNCH;
        }
    } else {
        if (R == 16)
            gdn::k2::scan_kernel<16><<<n_scan, gdn::k2::THREADS, gdn::k2::Cfg<16>::SMEM_BYTES, stream>>>(
                tm_A, tm_U, tm_S_store, p2);
        else if (R == 32)
            gdn::k2::scan_kernel<32><<<n_scan, gdn::k2::THREADS, gdn::k2::Cfg<32>::SMEM_BYTES, stream>>>(
                tm_A, tm_U, tm_S_store, p2);
        else
            gdn::k2::scan_kernel<64><<<n_scan, gdn::k2::THREADS, gdn::k2::Cfg<64>::SMEM_BYTES, stream>>>(
                tm_A, tm_U, tm_S_store, p2);
        if (ev) cudaEventRecord(ev[2], stream);
        const int grid3 = static_cast<int>(std::min<long long>(p3.total, ds->sms));
        void* args3[] = {&tm_q, &tm_S_load, &tm_out, &p3};
        if (cudaLaunchKernel(k3_fn(a.fmt), dim3(grid3), dim3(k3_threads(a.fmt)), args3, gdn::k3::SMEM_BYTES, stream) !=
            cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_LAUNCH;
        }
    }
    if (ev) cudaEventRecord(ev[3], stream);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

// ------------------------------------------------ the single-pass forward
// Scan CTAs of the single pass for this shape (one per head), or 0 when the
// whole forward does not run as one launch: switched off, a one-frame call,
// no cooperative launch at one CTA per SM, or so many heads that fewer than
// three quarters of the SMs would be left to the contraction and the output.
int single_pass_heads(const PassArgs& a, const DeviceState* ds) {
    if (g_single_pass.load() == 0 || !ds->coop_single || a.F < 2) return 0;
    const long long heads = static_cast<long long>(a.B) * a.H;
    return heads * 4 <= ds->sms ? static_cast<int>(heads) : 0;
}

// Ring frames: as many as keep the three rings within ~24 MiB (so they stay
// in L2 next to the streaming inputs), at least 4, at most F.  A forced depth
// is at least 2: the scan publishes frame f's image only once frame f + 1's
// store is under way, so with one slot it would wait on itself.
int single_pass_ring(const PassArgs& a) {
    const int forced = g_single_ring.load();
    if (forced > 0) return std::min(std::max(forced, 2), a.F);
    const size_t per_frame = static_cast<size_t>(a.B) * a.H * (2 * gdn::RING_TILE_BF16 + gdn::RING_TILE_F32);
    const int w = static_cast<int>(std::max<size_t>(4, (size_t(24) << 20) / per_frame));
    return std::min(w, a.F);
}

struct SingleLayout {
    int ring;
    long long slots;
    size_t a_off, u_off, s_off, c_off, total;
};
SingleLayout single_layout(const PassArgs& a) {
    SingleLayout L;
    L.ring = single_pass_ring(a);
    L.slots = static_cast<long long>(a.B) * L.ring * a.H;
    L.a_off = 0;
    // whole 128 x 128 ring tiles (zero-padded for d = 64) in the consumers' shared-memory image
    L.u_off = align256(L.a_off + static_cast<size_t>(L.slots) * gdn::RING_TILE_BF16);
    L.s_off = align256(L.u_off + static_cast<size_t>(L.slots) * gdn::RING_TILE_F32);
    L.c_off = align256(L.s_off + static_cast<size_t>(L.slots) * gdn::RING_TILE_BF16);
    L.total = align256(L.c_off + static_cast<size_t>(L.slots) * 4 * 4);
    return L;
}

gdn_status launch_single(const PassArgs& a, uint8_t* ws, const SingleLayout& L, const DeviceState* ds,
                         cudaStream_t stream, cudaEvent_t const* ev) {
    using namespace gdn;
    const int BF = a.B * a.F;
    const long long items = static_cast<long long>(a.B) * a.F * a.H;
    __nv_bfloat16* A_r = reinterpret_cast<__nv_bfloat16*>(ws + L.a_off);
    float* U_r = reinterpret_cast<float*>(ws + L.u_off);
    __nv_bfloat16* S_r = reinterpret_cast<__nv_bfloat16*>(ws + L.s_off);
    int* cnt = reinterpret_cast<int*>(ws + L.c_off);
    int* au_ready = cnt;
    int* au_free = cnt + L.slots;
    int* s_ready = cnt + 2 * L.slots;
    int* s_free = cnt + 3 * L.slots;
    CUtensorMap tm_k, tm_v, tm_q, tm_out;
    const bool enc_in =
        encode_inputs(&tm_k, &tm_v, &tm_q, a.q, a.k, a.v, a.fmt, BF, a.N, a.H, a.dk, a.dv, k1::CHUNK, k3::TILE_M);
    if (!enc_in || !encode_tokens(&tm_out, a.out, BF, a.N, a.H, a.dv, 32)) return GDN_ERR_LAUNCH;
    const unsigned long long lim = g_wait_limit_ns.load();
    if (ev) cudaEventRecord(ev[0], stream);
    if (cudaMemsetAsync(cnt, 0, static_cast<size_t>(L.slots) * 16, stream) != cudaSuccess) return GDN_ERR_LAUNCH;
    if (ev) {
        cudaEventRecord(ev[1], stream);
        cudaEventRecord(ev[2], stream);
    }
    // roles: one scan CTA per head, the other SMs split between contraction and output
    fwd::Counts c;
    c.s_ready = s_ready;
    c.s_free = s_free;
    c.s_ring = S_r;
    c.n_scan = a.B * a.H;
    const int rest = ds->sms - c.n_scan;
    const int forced = g_single_contract.load();
    c.pair = pair_applies(a) ? 1 : 0;
    if (c.pair && (!encode_pairs(&tm_k, a.k, static_cast<long long>(BF) * a.N, a.H, k1p::CHUNK) ||
                   !encode_pairs(&tm_v, a.v, static_cast<long long>(BF) * a.N, a.H, k1p::CHUNK)))
        return GDN_ERR_LAUNCH;
    // automatic: the share of the free SMs that contract, per mille, where the
    // contraction and the output roles finish together (swept on B300 at the 60 s
    // shape, 132 free SMs): bf16 48.5 % (0.352 ms; 60 % gives 0.375 ms), the
    // folded prologue 60.6 % (normalizing k costs the scalers more than
    // normalizing q costs the output; 0.440 ms, against 0.480 ms at 63 %),
    // fp8 57.5 % and NVFP4 60.5 % (the decoders expand k and v in shared
    // memory); on head pairs 40 %
    const int share = c.pair ? 400 : a.prologue ? 606 : a.fmt == FMT_FP8 ? 575 : a.fmt == FMT_FP4 ? 605 : 485;
    c.n_contract = forced > 0 ? std::min(forced, rest - 1) : std::max(1, (rest * share + 500) / 1000);
    const int n_out = rest - c.n_contract;
    if (c.n_contract < 1 || n_out < 1) return GDN_ERR_LAUNCH;

    k1::Params p1;
    std::memset(&p1, 0, sizeof(p1));
    p1.beta = a.beta;
    p1.A_ws = A_r;
    p1.U_ws = U_r;
    p1.H = a.H;
    p1.N = a.N;
    p1.dk = a.dk;
    p1.dv = a.dv;
    p1.items = static_cast<int>(items);
    p1.whole = static_cast<int>(items);
    p1.split_per = 1;
    p1.chunks = chunks_of(a.N);
    p1.work = static_cast<int>(c.pair ? items / 2 : items);
    p1.norm_k = a.prologue;
    p1.beta_sigmoid = a.prologue;
    p1.a_scale = a.fmt != FMT_BF16 ? a.k_scale * a.k_scale : 1.0f;
    p1.u_scale = a.fmt != FMT_BF16 ? a.k_scale * a.v_scale : 1.0f;
    p1.k_sf = a.k_sf;
    p1.v_sf = a.v_sf;
    p1.ring = L.ring;
    p1.B = a.B;
    p1.F = a.F;
    p1.reverse = a.reverse;
    p1.au_ready = au_ready;
    p1.au_free = au_free;
    p1.wait_limit_ns = lim;

    k3::Params p3;
    p3.B = a.B;
    p3.H = a.H;
    p3.F = a.F;
    p3.N = a.N;
    p3.dk = a.dk;
    p3.dv = a.dv;
    p3.ntile = (a.N + k3::TILE_M - 1) / k3::TILE_M;
    p3.total = items * p3.ntile;
    p3.reverse = a.reverse;
    p3.norm_q = a.prologue;
    p3.q_scale = a.fmt != FMT_BF16 ? a.q_scale : 1.0f;
    p3.q_sf = a.q_sf;
    p3.b_mn = 0;
    p3.wait_limit_ns = lim;

    k2h::Params p2;
    p2.A_ring = A_r;
    p2.U_ring = U_r;
    p2.S_ring = S_r;
    p2.alpha = a.alpha;
    p2.state_in = a.state_in;
    p2.state_out = a.state_out;
    p2.B = a.B;
    p2.H = a.H;
    p2.F = a.F;
    p2.dk = a.dk;
    p2.dv = a.dv;
    p2.reverse = a.reverse;
    p2.alpha_gate = a.prologue;
    p2.alpha_scale = a.alpha_scale;
    p2.ring = L.ring;
    p2.au_ready = au_ready;
    p2.au_free = au_free;
    p2.s_ready = s_ready;
    p2.s_free = s_free;
    // the output role loads an item's state once per item, or once per tile when
    // items are fewer than two per output CTA (k3::Sched)
    p2.s_units = items < 2LL * n_out ? p3.ntile : 1;
    p2.wait_limit_ns = lim;

    const int grid = c.n_scan + c.n_contract + n_out;
    void* args[] = {&tm_k, &tm_v, &tm_q, &tm_out, &p1, &p2, &p3, &c};
    const void* fn = fwd_fn(a.fmt);
    const size_t smem = fwd_smem(a.fmt);
    if (cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(fwd::THREADS), args, smem, stream) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_LAUNCH;
    }
    if (ev) cudaEventRecord(ev[3], stream);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

bool all_device(const PassArgs& a) {
    return is_device_ptr(a.q) && is_device_ptr(a.k) && is_device_ptr(a.v) && is_device_ptr(a.alpha) &&
           is_device_ptr(a.beta) && is_device_ptr(a.state_in) && is_device_ptr(a.out) && is_device_ptr(a.state_out);
}

// The one-launch step: a plain bf16 frame (no folded prologue, no 8-bit inputs).
bool fused_step_applies(const PassArgs& a) {
    return g_fused_step.load() != 0 && a.F == 1 && a.fmt == gdn::FMT_BF16 && !a.prologue;
}
gdn_status launch_step_fused(const PassArgs& a, cudaStream_t stream) {
    CUtensorMap tm_k, tm_v, tm_q, tm_o;
    if (!encode_tokens(&tm_k, a.k, a.B, a.N, a.H, a.dk, gdn::step::CHUNK) ||
        !encode_tokens(&tm_v, a.v, a.B, a.N, a.H, a.dv, gdn::step::CHUNK) ||
        !encode_tokens(&tm_q, a.q, a.B, a.N, a.H, a.dk, 128) ||
        !encode_tokens(&tm_o, a.out, a.B, a.N, a.H, a.dv, 128))
        return GDN_ERR_LAUNCH;
    CUtensorMap tm_s;
    std::memset(&tm_s, 0, sizeof(tm_s));
    if (a.state_out != nullptr &&
        !encode_mats_f32(&tm_s, a.state_out, static_cast<long long>(a.B) * a.H, a.dv, a.dk, gdn::step::SR))
        return GDN_ERR_LAUNCH;
    gdn::step::Params ps;
    ps.alpha = a.alpha;
    ps.beta = a.beta;
    ps.state_in = a.state_in;
    ps.state_out = a.state_out;
    ps.H = a.H;
    ps.N = a.N;
    ps.dk = a.dk;
    ps.dv = a.dv;
    ps.wait_limit_ns = g_wait_limit_ns.load();
    // programmatic dependent launch: the kernel's prologue (barriers, TMEM,
    // tensor-map prefetch) overlaps the end of the previous grid in the
    // stream; the kernel waits for that grid before its first global access
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.H * gdn::step::CS));
    cfg.blockDim = dim3(gdn::step::THREADS);
    cfg.dynamicSmemBytes = gdn::step::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gdn::step::step_kernel, tm_k, tm_v, tm_q, tm_o, tm_s, ps) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_LAUNCH;
    }
    return GDN_OK;
}

// Pooled-workspace pass: gdn_frame_forward (step = false) and gdn_frame_step.
gdn_status run_pass(const PassArgs& a, bool step, cudaStream_t stream, cudaEvent_t const* ev = nullptr) {
    int dev;
    DeviceState* ds;
    gdn_status st = device_ready(&dev, &ds);
    if (st != GDN_OK) return st;
    if (!all_device(a)) return GDN_ERR_NULL_PTR;
    if (step && fused_step_applies(a) && ev == nullptr) return launch_step_fused(a, stream);
    if (!step && a.ext_A == nullptr && single_pass_heads(a, ds) > 0) {
        const SingleLayout L = single_layout(a);
        uint8_t* ws = nullptr;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), L.total, ds->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_ALLOC;
        }
        const gdn_status result = launch_single(a, ws, L, ds, stream, ev);
        cudaFreeAsync(ws, stream);
        return result;
    }
    const long long items = static_cast<long long>(a.B) * a.F * a.H;
    const SplitPlan sp = plan_split(items, chunks_of(a.N), ds->sms, ds->coop_k1);
    const Layout L = layout_of(items, a.dk, a.dv, sp);
    uint8_t* ws = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), L.total, ds->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_ALLOC;
    }
    const gdn_status result = launch_phases(a, ws, L, sp, ds, stream, ev);
    cudaFreeAsync(ws, stream);
    return result;
}

// ---------------------------------------------------------------- backward
__global__ void fill_f32_kernel(float* dst, long long n, float v) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = v;
}
__global__ void f32_to_bf16_kernel(const float* src, __nv_bfloat16* dst, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = __float2bfloat16_rn(src[i]);
}

struct BwdArgs {
    const void *q, *k, *v;
    const float *alpha, *beta, *state_in;
    const void* d_out;
    const float* d_state_out;
    void *dq, *dk, *dv;
    float *d_alpha, *d_beta, *d_state_in;
    int B, H, F, N, dk_, dv_;
    const void* saved_A = nullptr;   // forward activations (gdn_frame_forward_save), or null: recompute
    const void* saved_S = nullptr;
};

// Workspace of one batch row (reused row after row); F1 = F + 1 frame slots.
struct BwdLayout {
    size_t a_off, u_off, u2_off, sx_off, gx_off, w_off, al_off, one_off, c_off, total;
};
BwdLayout bwd_layout(int H, int F, int N, int dk, int dv) {
    const size_t F1 = static_cast<size_t>(F) + 1;
    BwdLayout L;
    L.a_off = 0;                                                               // A_f, bf16, slot F zero
    L.u_off = align256(L.a_off + F1 * H * dk * dk * 2);                        // U_f, fp32
    L.u2_off = align256(L.u_off + static_cast<size_t>(F) * H * dv * dk * 4);   // M_{f-1} in slot f, fp32
    L.sx_off = align256(L.u2_off + F1 * H * dv * dk * 4);                      // S_{f-1} in slot f, bf16
    L.gx_off = align256(L.sx_off + F1 * H * dv * dk * 2);                      // G_{f-1} in slot f, bf16
    L.w_off = align256(L.gx_off + F1 * H * dv * dk * 2);                       // W_f, bf16
    L.al_off = align256(L.w_off + static_cast<size_t>(F) * H * dk * dk * 2);   // alpha', fp32
    L.one_off = align256(L.al_off + F1 * H * 4);                               // ones [F, N, H]
    L.c_off = align256(L.one_off + static_cast<size_t>(F) * N * H * 4);        // phase-1 counters
    L.total = align256(L.c_off + F1 * H * 8);
    return L;
}

// Phase 1 on one batch row: A_f, U_f of (k, v, beta) for F frames, whole items.
gdn_status bwd_contract(const void* k, const void* v, const float* beta, __nv_bfloat16* A_out, float* U_out,
                        int* counters, int H, int F, int N, int dk, int dv, const DeviceState* ds, cudaStream_t st) {
    CUtensorMap tm_k, tm_v;
    if (!encode_tokens(&tm_k, k, F, N, H, dk, gdn::k1::CHUNK) || !encode_tokens(&tm_v, v, F, N, H, dv, gdn::k1::CHUNK))
        return GDN_ERR_LAUNCH;
    const long long items = static_cast<long long>(F) * H;
    gdn::k1::Params p1;
    std::memset(&p1, 0, sizeof(p1));   // ring mode off
    p1.beta = beta;
    p1.A_ws = A_out;
    p1.U_ws = U_out;
    p1.partial = nullptr;
    p1.counters = counters;
    p1.H = H;
    p1.N = N;
    p1.dk = dk;
    p1.dv = dv;
    p1.items = static_cast<int>(items);
    p1.whole = static_cast<int>(items);
    p1.split_per = 1;
    p1.chunks = chunks_of(N);
    p1.work = static_cast<int>(items);
    p1.norm_k = 0;
    p1.beta_sigmoid = 0;
    p1.a_scale = 1.0f;
    p1.u_scale = 1.0f;
    p1.wait_limit_ns = g_wait_limit_ns.load();
    gdn::k1::contract_kernel<gdn::FMT_BF16><<<std::min(p1.work, ds->sms), gdn::k1::THREADS, gdn::k1::SMEM_BYTES, st>>>(
        tm_k, tm_v, p1);
    return GDN_OK;
}

// The scan over `F` frames on one batch row (standalone kernel), state images
// stored through tm_S_store.
gdn_status bwd_scan(const __nv_bfloat16* A, const float* U, __nv_bfloat16* S_store, const float* alpha,
                    const float* state_in, float* state_out, int H, int F, int dk, int dv, int reverse,
                    const DeviceState* ds, cudaStream_t st) {
    const int R = scan_rows_standalone(1, H, dv, ds->sms);
    CUtensorMap tm_A, tm_U, tm_S;
    const long long items = static_cast<long long>(F) * H;
    if (!encode_mats(&tm_A, A, items, dk, dk, 128) || !encode_mats_f32(&tm_U, U, items, dv, dk, R) ||
        !encode_mats(&tm_S, S_store, items, dv, dk, R))
        return GDN_ERR_LAUNCH;
    gdn::k2::Params p2;
    p2.alpha = alpha;
    p2.state_in = state_in;
    p2.state_out = state_out;
    p2.H = H;
    p2.F = F;
    p2.dk = dk;
    p2.dv = dv;
    p2.rsplit = dv / R;
    p2.reverse = reverse;
    p2.alpha_gate = 0;
    p2.alpha_scale = 0.0f;
    p2.wait_limit_ns = g_wait_limit_ns.load();
    const int n_scan = H * p2.rsplit;
    if (R == 16)
        gdn::k2::scan_kernel<16><<<n_scan, gdn::k2::THREADS, gdn::k2::Cfg<16>::SMEM_BYTES, st>>>(tm_A, tm_U, tm_S, p2);
    else if (R == 32)
        gdn::k2::scan_kernel<32><<<n_scan, gdn::k2::THREADS, gdn::k2::Cfg<32>::SMEM_BYTES, st>>>(tm_A, tm_U, tm_S, p2);
    else
        gdn::k2::scan_kernel<64><<<n_scan, gdn::k2::THREADS, gdn::k2::Cfg<64>::SMEM_BYTES, st>>>(tm_A, tm_U, tm_S, p2);
    return GDN_OK;
}

// The backward of one batch row b (B = 1 views of every array).
gdn_status bwd_row(const BwdArgs& a, int b, uint8_t* ws, const BwdLayout& L, const DeviceState* ds,
                   cudaStream_t st) {
    const int H = a.H, F = a.F, N = a.N, dk = a.dk_, dv = a.dv_;
    const size_t tokH = static_cast<size_t>(F) * N * H;
    const size_t sd = static_cast<size_t>(dv) * dk, ad = static_cast<size_t>(dk) * dk;
    auto bf = [](const void* p, size_t elems) {
        return reinterpret_cast<const __nv_bfloat16*>(p) + elems;
    };
    const void* q = bf(a.q, b * tokH * dk);
    const void* k = bf(a.k, b * tokH * dk);
    const void* v = bf(a.v, b * tokH * dv);
    const void* dO = bf(a.d_out, b * tokH * dv);
    const float* alpha = a.alpha + static_cast<size_t>(b) * F * H;
    const float* beta = a.beta + b * tokH;
    const float* s0 = a.state_in ? a.state_in + static_cast<size_t>(b) * H * sd : nullptr;
    const float* dSF = a.d_state_out ? a.d_state_out + static_cast<size_t>(b) * H * sd : nullptr;
    __nv_bfloat16* A1 = reinterpret_cast<__nv_bfloat16*>(ws + L.a_off);
    float* U = reinterpret_cast<float*>(ws + L.u_off);
    float* U2 = reinterpret_cast<float*>(ws + L.u2_off);
    __nv_bfloat16* Sx = reinterpret_cast<__nv_bfloat16*>(ws + L.sx_off);
    __nv_bfloat16* Gx = reinterpret_cast<__nv_bfloat16*>(ws + L.gx_off);
    __nv_bfloat16* Wb = reinterpret_cast<__nv_bfloat16*>(ws + L.w_off);
    float* al = reinterpret_cast<float*>(ws + L.al_off);
    const float* ones = reinterpret_cast<const float*>(ws + L.one_off);
    int* counters = reinterpret_cast<int*>(ws + L.c_off);
    const int fill_grid = 2 * ds->sms;
    gdn_status r;

    // slots that no kernel writes: A_F = 0, M_{-1} = 0, S_{-1} image = S_0; alpha' = [alpha, 1]
    if (cudaMemsetAsync(A1 + static_cast<size_t>(F) * H * ad, 0, H * ad * 2, st) != cudaSuccess ||
        cudaMemsetAsync(U2, 0, H * sd * 4, st) != cudaSuccess ||
        cudaMemcpyAsync(al, alpha, static_cast<size_t>(F) * H * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    fill_f32_kernel<<<1, 128, 0, st>>>(al + static_cast<size_t>(F) * H, H, 1.0f);
    if (s0)
        f32_to_bf16_kernel<<<fill_grid, 256, 0, st>>>(s0, Sx, static_cast<long long>(H) * sd);
    else if (cudaMemsetAsync(Sx, 0, H * sd * 2, st) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    // forward recompute: A_f, U_f, and the states S_0..S_{F-1} into slots 1..F
    if (a.saved_A != nullptr) {
        // the forward's own A_f and state images, saved by gdn_frame_forward_save
        const size_t fa = static_cast<size_t>(F) * H * ad * 2, fs = static_cast<size_t>(F) * H * sd * 2;
        if (cudaMemcpyAsync(A1, static_cast<const uint8_t*>(a.saved_A) + b * fa, fa, cudaMemcpyDeviceToDevice, st) !=
                cudaSuccess ||
            cudaMemcpyAsync(Sx + H * sd, static_cast<const uint8_t*>(a.saved_S) + b * fs, fs,
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess)
            return GDN_ERR_LAUNCH;
    } else {
        if ((r = bwd_contract(k, v, beta, A1, U, counters, H, F, N, dk, dv, ds, st)) != GDN_OK) return r;
        if ((r = bwd_scan(A1, U, Sx + H * sd, alpha, s0, nullptr, H, F, dk, dv, 0, ds, st)) != GDN_OK) return r;
    }
    // M_f = dO_f^T Q_f into slots 1..F (the contraction with beta = 1; its A output is scratch)
    if ((r = bwd_contract(q, dO, ones, Wb, U2 + H * sd, counters, H, F, N, dk, dv, ds, st)) != GDN_OK) return r;
    // reverse scan over F + 1 slots: slot j >= 1 receives G_{j-1}, slot 0 dL/dS_0
    if ((r = bwd_scan(A1, U2, Gx, al, dSF, a.d_state_in ? a.d_state_in + static_cast<size_t>(b) * H * sd : nullptr,
                      H, F + 1, dk, dv, 1, ds, st)) != GDN_OK)
        return r;
    // per-frame gradients
    {
        CUtensorMap tm_Sx, tm_Gx, tm_A;
        const long long slots = static_cast<long long>(F + 1) * H;
        if (!encode_mats(&tm_Sx, Sx, slots, dv, dk, 128) || !encode_mats(&tm_Gx, Gx, slots, dv, dk, 128) ||
            !encode_mats(&tm_A, A1, slots, dk, dk, 128))
            return GDN_ERR_LAUNCH;
        gdn::bwd::FrameParams pf;
        pf.alpha = alpha;
        pf.d_alpha = a.d_alpha + static_cast<size_t>(b) * F * H;
        pf.W = Wb;
        pf.H = H;
        pf.F = F;
        pf.dk = dk;
        pf.dv = dv;
        pf.wait_limit_ns = g_wait_limit_ns.load();
        gdn::bwd::frame_grad_kernel<<<std::min(F * H, ds->sms), gdn::bwd::THREADS, gdn::bwd::FRAME_SMEM, st>>>(
            tm_Sx, tm_Gx, tm_A, pf);
    }
    // dq = dO S_f: the output kernel with the state read MN-major (A = dO, width dv; out width dk)
    {
        CUtensorMap tm_do, tm_S, tm_dq;
        if (!encode_tokens(&tm_do, dO, F, N, H, dv, gdn::k3::TILE_M) ||
            !encode_mats(&tm_S, Sx + H * sd, static_cast<long long>(F) * H, dv, dk, 128) ||
            !encode_tokens(&tm_dq, reinterpret_cast<__nv_bfloat16*>(a.dq) + b * tokH * dk, F, N, H, dk, 32))
            return GDN_ERR_LAUNCH;
        gdn::k3::Params p3;
        p3.B = 1;
        p3.H = H;
        p3.F = F;
        p3.N = N;
        p3.dk = dv;   // the A operand's (dO's) width
        p3.dv = dk;   // the output's (dq's) width
        p3.ntile = (N + gdn::k3::TILE_M - 1) / gdn::k3::TILE_M;
        p3.total = static_cast<long long>(F) * H * p3.ntile;
        p3.reverse = 0;
        p3.norm_q = 0;
        p3.q_scale = 1.0f;
        p3.b_mn = 1;
        p3.wait_limit_ns = g_wait_limit_ns.load();
        gdn::k3::output_kernel<gdn::FMT_BF16><<<static_cast<int>(std::min<long long>(p3.total, ds->sms)),
                                                gdn::k3::threads<gdn::FMT_BF16>(), gdn::k3::SMEM_BYTES, st>>>(
            tm_do, tm_S, tm_dq, p3);
    }
    // dk, dv, dbeta
    {
        CUtensorMap tm_k, tm_v, tm_Gx, tm_W;
        const long long slots = static_cast<long long>(F + 1) * H;
        if (!encode_tokens(&tm_k, k, F, N, H, dk, 128) || !encode_tokens(&tm_v, v, F, N, H, dv, 128) ||
            !encode_mats(&tm_Gx, Gx, slots, dv, dk, 128) ||
            !encode_mats(&tm_W, Wb, static_cast<long long>(F) * H, dk, dk, 128))
            return GDN_ERR_LAUNCH;
        gdn::bwd::TokenParams pt;
        pt.beta = beta;
        pt.dk_out = reinterpret_cast<__nv_bfloat16*>(a.dk) + b * tokH * dk;
        pt.dv_out = reinterpret_cast<__nv_bfloat16*>(a.dv) + b * tokH * dv;
        pt.d_beta = a.d_beta + b * tokH;
        pt.H = H;
        pt.F = F;
        pt.N = N;
        pt.dk = dk;
        pt.dv = dv;
        pt.ntile = (N + 127) / 128;
        pt.units = static_cast<long long>(F) * H * pt.ntile;
        pt.wait_limit_ns = g_wait_limit_ns.load();
        gdn::bwd::token_grad_kernel<<<static_cast<int>(std::min<long long>(pt.units, ds->sms)),
                                      gdn::bwd::TOKEN_THREADS, gdn::bwd::TOKEN_SMEM, st>>>(tm_k, tm_v, tm_Gx, tm_W, pt);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

__global__ void selftest_timeout_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        gdn::mbar_init(&bar, 1);  // nothing ever arrives on it
        abort_flag = 0;
        gdn::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) gdn::mbar_wait(&bar, 0, limit_ns, &abort_flag);
}

}  // namespace

extern "C" {

gdn_status gdn_frame_forward(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                             const float* state_in, void* out, float* state_out, int B, int H, int F, int N, int dk,
                             int dv, gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    return run_pass(PassArgs{q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv}, false,
                    reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_step(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                          const float* state_in, void* out, float* state_out, int B, int H, int N, int dk, int dv,
                          gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv);
    if (s != GDN_OK) return s;
    return run_pass(PassArgs{q, k, v, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv}, true,
                    reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_forward_reverse(const void* q, const void* k, const void* v, const float* alpha,
                                     const float* beta, const float* state_in, void* out, float* state_out, int B,
                                     int H, int F, int N, int dk, int dv, gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    PassArgs a{q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv};
    a.reverse = 1;
    return run_pass(a, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_forward_gated(const void* q, const void* k, const void* v, const float* a_logit,
                                   const float* b_logit, float alpha_scale, const float* state_in, void* out,
                                   float* state_out, int B, int H, int F, int N, int dk, int dv,
                                   gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, a_logit, b_logit, state_in, out, state_out, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    PassArgs a{q, k, v, a_logit, b_logit, state_in, out, state_out, B, H, F, N, dk, dv};
    a.prologue = 1;
    a.alpha_scale = alpha_scale;
    return run_pass(a, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_step_gated(const void* q, const void* k, const void* v, const float* a_logit,
                                const float* b_logit, float alpha_scale, const float* state_in, void* out,
                                float* state_out, int B, int H, int N, int dk, int dv, gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, a_logit, b_logit, state_in, out, state_out, B, H, 1, N, dk, dv);
    if (s != GDN_OK) return s;
    PassArgs a{q, k, v, a_logit, b_logit, state_in, out, state_out, B, H, 1, N, dk, dv};
    a.prologue = 1;
    a.alpha_scale = alpha_scale;
    return run_pass(a, true, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_forward_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                                 float v_scale, const float* alpha, const float* beta, const float* state_in,
                                 void* out, float* state_out, int B, int H, int F, int N, int dk, int dv,
                                 gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv, 8);
    if (s != GDN_OK) return s;
    PassArgs a{q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv};
    a.fmt = gdn::FMT_FP8;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return run_pass(a, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_step_fp8(const void* q, const void* k, const void* v, float q_scale, float k_scale,
                              float v_scale, const float* alpha, const float* beta, const float* state_in, void* out,
                              float* state_out, int B, int H, int N, int dk, int dv, gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv, 8);
    if (s != GDN_OK) return s;
    PassArgs a{q, k, v, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv};
    a.fmt = gdn::FMT_FP8;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return run_pass(a, true, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
// NVFP4 arguments: the common checks with 4 bits per element, then head sizes
// 64 or 128, the three block-scale arrays (device memory, 16-byte aligned,
// clear of every output).
gdn_status validate_nvfp4(const void* q4, const void* k4, const void* v4, const void* q_sf, const void* k_sf,
                          const void* v_sf, const float* alpha, const float* beta, const float* state_in,
                          const void* out, const float* state_out, int B, int H, int F, int N, int dk, int dv) {
    gdn_status s = validate(q4, k4, v4, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv, 4);
    if (s != GDN_OK) return s;
    if (!q_sf || !k_sf || !v_sf) return GDN_ERR_NULL_PTR;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return GDN_ERR_UNSUPPORTED;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(q_sf) || !a16(k_sf) || !a16(v_sf)) return GDN_ERR_MISALIGNED;
    const long long tok = static_cast<long long>(B) * F * N;
    auto R = [](const void* p, long long n) {
        return Range{reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(n)};
    };
    const Range sf[3] = {R(q_sf, tok * H * dk / 16), R(k_sf, tok * H * dk / 16), R(v_sf, tok * H * dv / 16)};
    const Range ro = R(out, tok * H * dv * 2);
    const Range rso = state_out ? R(state_out, static_cast<long long>(B) * H * dv * dk * 4) : Range{0, 0};
    for (const Range& r : sf)
        if (overlap(r, ro) || (state_out && overlap(r, rso))) return GDN_ERR_ALIAS;
    if (!is_device_ptr(q_sf) || !is_device_ptr(k_sf) || !is_device_ptr(v_sf)) return GDN_ERR_NULL_PTR;
    return GDN_OK;
}
}  // namespace

extern "C" {

gdn_status gdn_frame_forward_nvfp4(const void* q4, const void* k4, const void* v4, const void* q_sf,
                                   const void* k_sf, const void* v_sf, float q_gs, float k_gs, float v_gs,
                                   const float* alpha, const float* beta, const float* state_in, void* out,
                                   float* state_out, int B, int H, int F, int N, int dk, int dv,
                                   gdn_stream_t stream) {
    gdn_status s = validate_nvfp4(q4, k4, v4, q_sf, k_sf, v_sf, alpha, beta, state_in, out, state_out, B, H, F, N,
                                  dk, dv);
    if (s != GDN_OK) return s;
    PassArgs a{q4, k4, v4, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv};
    a.fmt = gdn::FMT_FP4;
    a.q_sf = static_cast<const uint8_t*>(q_sf);
    a.k_sf = static_cast<const uint8_t*>(k_sf);
    a.v_sf = static_cast<const uint8_t*>(v_sf);
    a.q_scale = q_gs;
    a.k_scale = k_gs;
    a.v_scale = v_gs;
    return run_pass(a, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_step_nvfp4(const void* q4, const void* k4, const void* v4, const void* q_sf, const void* k_sf,
                                const void* v_sf, float q_gs, float k_gs, float v_gs, const float* alpha,
                                const float* beta, const float* state_in, void* out, float* state_out, int B, int H,
                                int N, int dk, int dv, gdn_stream_t stream) {
    gdn_status s = validate_nvfp4(q4, k4, v4, q_sf, k_sf, v_sf, alpha, beta, state_in, out, state_out, B, H, 1, N,
                                  dk, dv);
    if (s != GDN_OK) return s;
    PassArgs a{q4, k4, v4, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv};
    a.fmt = gdn::FMT_FP4;
    a.q_sf = static_cast<const uint8_t*>(q_sf);
    a.k_sf = static_cast<const uint8_t*>(k_sf);
    a.v_sf = static_cast<const uint8_t*>(v_sf);
    a.q_scale = q_gs;
    a.k_scale = k_gs;
    a.v_scale = v_gs;
    return run_pass(a, true, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
gdn_status backward_impl(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                         const float* state_in, const void* saved_A, const void* saved_S, const void* d_out,
                         const float* d_state_out, void* dq_out, void* dk_out, void* dv_out, float* d_alpha,
                         float* d_beta, float* d_state_in, int B, int H, int F, int N, int dk, int dv,
                         gdn_stream_t stream) {
    if (!q || !k || !v || !alpha || !beta || !d_out || !dq_out || !dk_out || !dv_out || !d_alpha || !d_beta)
        return GDN_ERR_NULL_PTR;
    gdn_status s = validate(q, k, v, alpha, beta, state_in, d_out, nullptr, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!a16(dq_out) || !a16(dk_out) || !a16(dv_out) || !a4(d_alpha) || !a4(d_beta) || (d_state_in && !a4(d_state_in)) ||
        (d_state_out && !a4(d_state_out)))
        return GDN_ERR_MISALIGNED;
    // every gradient output must stay clear of every input
    {
        const long long tok = static_cast<long long>(B) * F * N;
        const uintptr_t sb = static_cast<uintptr_t>(static_cast<long long>(B) * H * dv * dk * 4);
        auto R = [](const void* p, uintptr_t n) { return Range{reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + n}; };
        const uintptr_t sab = static_cast<uintptr_t>(static_cast<long long>(B) * F * H * dk * dk * 2);
        const uintptr_t ssb = static_cast<uintptr_t>(static_cast<long long>(B) * F * H * dv * dk * 2);
        const Range ins[10] = {R(q, tok * H * dk * 2), R(k, tok * H * dk * 2), R(v, tok * H * dv * 2),
                               R(alpha, static_cast<uintptr_t>(B) * F * H * 4), R(beta, tok * H * 4),
                               R(d_out, tok * H * dv * 2), state_in ? R(state_in, sb) : Range{0, 0},
                               d_state_out ? R(d_state_out, sb) : Range{0, 0},
                               saved_A ? R(saved_A, sab) : Range{0, 0}, saved_S ? R(saved_S, ssb) : Range{0, 0}};
        const Range outs[6] = {R(dq_out, tok * H * dk * 2), R(dk_out, tok * H * dk * 2), R(dv_out, tok * H * dv * 2),
                               R(d_alpha, static_cast<uintptr_t>(B) * F * H * 4), R(d_beta, tok * H * 4),
                               d_state_in ? R(d_state_in, sb) : Range{0, 0}};
        for (const Range& o : outs)
            for (const Range& i : ins)
                if (o.hi > o.lo && i.hi > i.lo && overlap(o, i)) return GDN_ERR_ALIAS;
        for (int x = 0; x < 6; ++x)
            for (int y = x + 1; y < 6; ++y)
                if (outs[x].hi > outs[x].lo && outs[y].hi > outs[y].lo && overlap(outs[x], outs[y])) return GDN_ERR_ALIAS;
    }
    int dev;
    DeviceState* ds;
    s = device_ready(&dev, &ds);
    if (s != GDN_OK) return s;
    const void* ptrs[16] = {q, k, v, alpha, beta, state_in, d_out, d_state_out, dq_out, dk_out, dv_out, d_alpha, d_beta,
                            d_state_in, saved_A, saved_S};
    for (const void* p : ptrs)
        if (!is_device_ptr(p)) return GDN_ERR_NULL_PTR;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const BwdLayout L = bwd_layout(H, F, N, dk, dv);
    uint8_t* ws = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), L.total, ds->pool, st) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_ALLOC;
    }
    BwdArgs a{q, k, v, alpha, beta, state_in, d_out, d_state_out, dq_out, dk_out, dv_out, d_alpha, d_beta,
              d_state_in, B, H, F, N, dk, dv};
    a.saved_A = saved_A;
    a.saved_S = saved_S;
    fill_f32_kernel<<<2 * ds->sms, 256, 0, st>>>(reinterpret_cast<float*>(ws + L.one_off),
                                                 static_cast<long long>(F) * N * H, 1.0f);
    gdn_status r = GDN_OK;
    for (int b = 0; b < B && r == GDN_OK; ++b) r = bwd_row(a, b, ws, L, ds, st);
    cudaFreeAsync(ws, st);
    return r;
}
}  // namespace

extern "C" {

gdn_status gdn_frame_backward(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                              const float* state_in, const void* d_out, const float* d_state_out, void* dq_out,
                              void* dk_out, void* dv_out, float* d_alpha, float* d_beta, float* d_state_in, int B,
                              int H, int F, int N, int dk, int dv, gdn_stream_t stream) {
    return backward_impl(q, k, v, alpha, beta, state_in, nullptr, nullptr, d_out, d_state_out, dq_out, dk_out, dv_out,
                         d_alpha, d_beta, d_state_in, B, H, F, N, dk, dv, stream);
}

gdn_status gdn_frame_backward_saved(const void* q, const void* k, const void* v, const float* alpha,
                                    const float* beta, const float* state_in, const void* saved_A,
                                    const void* saved_S, const void* d_out, const float* d_state_out, void* dq_out,
                                    void* dk_out, void* dv_out, float* d_alpha, float* d_beta, float* d_state_in,
                                    int B, int H, int F, int N, int dk, int dv, gdn_stream_t stream) {
    if (!saved_A || !saved_S) return GDN_ERR_NULL_PTR;
    return backward_impl(q, k, v, alpha, beta, state_in, saved_A, saved_S, d_out, d_state_out, dq_out, dk_out, dv_out,
                         d_alpha, d_beta, d_state_in, B, H, F, N, dk, dv, stream);
}

gdn_status gdn_frame_forward_save(const void* q, const void* k, const void* v, const float* alpha, const float* beta,
                                  const float* state_in, void* out, float* state_out, void* saved_A, void* saved_S,
                                  int B, int H, int F, int N, int dk, int dv, gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    if (!saved_A || !saved_S) return GDN_ERR_NULL_PTR;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(saved_A) || !a16(saved_S)) return GDN_ERR_MISALIGNED;
    {
        const long long tok = static_cast<long long>(B) * F * N;
        auto R = [](const void* p, long long n) {
            return Range{reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(n)};
        };
        const Range ra = R(saved_A, static_cast<long long>(B) * F * H * dk * dk * 2);
        const Range rs = R(saved_S, static_cast<long long>(B) * F * H * dv * dk * 2);
        const Range others[7] = {R(q, tok * H * dk * 2), R(k, tok * H * dk * 2), R(v, tok * H * dv * 2),
                                 R(alpha, static_cast<long long>(B) * F * H * 4), R(beta, tok * H * 4),
                                 R(out, tok * H * dv * 2),
                                 state_out ? R(state_out, static_cast<long long>(B) * H * dv * dk * 4) : Range{0, 0}};
        if (overlap(ra, rs)) return GDN_ERR_ALIAS;
        for (const Range& o : others)
            if (o.hi > o.lo && (overlap(o, ra) || overlap(o, rs))) return GDN_ERR_ALIAS;
        if (state_in) {
            const Range ri = R(state_in, static_cast<long long>(B) * H * dv * dk * 4);
            if (overlap(ri, ra) || overlap(ri, rs)) return GDN_ERR_ALIAS;
        }
    }
    if (!is_device_ptr(saved_A) || !is_device_ptr(saved_S)) return GDN_ERR_NULL_PTR;
    PassArgs a{q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv};
    a.ext_A = saved_A;
    a.ext_S = saved_S;
    return run_pass(a, false, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status gdn_frame_forward_timed(const void* q, const void* k, const void* v, const float* alpha,
                                   const float* beta, const float* state_in, void* out, float* state_out, int B,
                                   int H, int F, int N, int dk, int dv, gdn_stream_t stream,
                                   void* const* phase_events) {
    if (phase_events == nullptr || !phase_events[0] || !phase_events[1] || !phase_events[2] || !phase_events[3])
        return GDN_ERR_NULL_PTR;
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    cudaEvent_t ev[4];
    for (int i = 0; i < 4; ++i) ev[i] = static_cast<cudaEvent_t>(phase_events[i]);
    return run_pass(PassArgs{q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv}, false,
                    reinterpret_cast<cudaStream_t>(stream), ev);
}

gdn_status gdn_frame_forward_host(const void* q, const void* k, const void* v, const float* alpha,
                                  const float* beta, const float* state_in, void* out, float* state_out, int B,
                                  int H, int F, int N, int dk, int dv, gdn_stream_t stream) {
    gdn_status s = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, F, N, dk, dv);
    if (s != GDN_OK) return s;
    int dev;
    DeviceState* ds;
    s = device_ready(&dev, &ds);
    if (s != GDN_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // Frame chunks of Fc frames, double-buffered on the device: chunk i's
    // host->device copy (copy_in stream), forward (the caller's stream, the
    // state carried in place from chunk to chunk, which is exact) and
    // device->host copy of its outputs (copy_out stream) overlap with the
    // neighbouring chunks'.  Events order the reuse of each buffer.
    const int forced = g_host_chunk.load();
    const int Fc = forced > 0 ? std::min(forced, F) : std::max(1, (F + 7) / 8);
    const int nch = (F + Fc - 1) / Fc;
    const size_t tokc = static_cast<size_t>(B) * Fc * N;
    const size_t per_f_q = static_cast<size_t>(N) * H * dk * 2, per_f_v = static_cast<size_t>(N) * H * dv * 2,
                 per_f_a = static_cast<size_t>(H) * 4, per_f_b = static_cast<size_t>(N) * H * 4;
    const size_t bs = static_cast<size_t>(B) * H * dv * dk * 4;
    // one slot: q, k, v, alpha, beta, out of Fc frames
    const size_t sz[6] = {tokc * H * dk * 2, tokc * H * dk * 2, tokc * H * dv * 2,
                          static_cast<size_t>(B) * Fc * H * 4, tokc * H * 4, tokc * H * dv * 2};
    size_t off[6], slot_bytes = 0;
    for (int i = 0; i < 6; ++i) { off[i] = slot_bytes; slot_bytes = align256(slot_bytes + sz[i]); }
    uint8_t* d = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&d), 2 * slot_bytes + bs, ds->pool, st) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_ALLOC;
    }
    float* dstate = reinterpret_cast<float*>(d + 2 * slot_bytes);
    cudaEvent_t ev[7];
    int made = 0;
    for (; made < 7; ++made)
        if (cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming) != cudaSuccess) break;
    cudaEvent_t* ev_in = ev;          // [2] a slot's inputs have landed
    cudaEvent_t* ev_comp = ev + 2;    // [2] the forward of a slot has finished
    cudaEvent_t* ev_out = ev + 4;     // [2] a slot's outputs have been copied out
    cudaEvent_t ev_start = ev[6];
    bool ok = made == 7;
    // B rows of `width` bytes (one per batch row); a plain copy when B = 1
    auto cp2 = [&](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, cudaMemcpyKind kind,
                   cudaStream_t s2) {
        ok = ok && (B == 1 ? cudaMemcpyAsync(dst, src, width, kind, s2)
                           : cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, B, kind, s2)) == cudaSuccess;
    };
    if (ok) {
        if (state_in)
            ok = cudaMemcpyAsync(dstate, state_in, bs, cudaMemcpyHostToDevice, st) == cudaSuccess;
        else
            ok = cudaMemsetAsync(dstate, 0, bs, st) == cudaSuccess;
        ok = ok && cudaEventRecord(ev_start, st) == cudaSuccess &&
             cudaStreamWaitEvent(ds->copy_in, ev_start, 0) == cudaSuccess &&
             cudaStreamWaitEvent(ds->copy_out, ev_start, 0) == cudaSuccess;
    }
    gdn_status r = GDN_OK;
    for (int i = 0; i < nch && ok && r == GDN_OK; ++i) {
        const int slot = i & 1;
        const int f0 = i * Fc, fc = std::min(Fc, F - f0);
        uint8_t* b = d + slot * slot_bytes;
        // inputs of chunk i (frames f0 .. f0 + fc - 1 of every batch row), dense [B, fc, ...]
        if (i >= 2) ok = ok && cudaStreamWaitEvent(ds->copy_in, ev_comp[slot], 0) == cudaSuccess;
        const uint8_t* hq = static_cast<const uint8_t*>(q);
        const uint8_t* hk = static_cast<const uint8_t*>(k);
        const uint8_t* hv = static_cast<const uint8_t*>(v);
        const uint8_t* ha = reinterpret_cast<const uint8_t*>(alpha);
        const uint8_t* hb = reinterpret_cast<const uint8_t*>(beta);
        cp2(b + off[0], fc * per_f_q, hq + f0 * per_f_q, F * per_f_q, fc * per_f_q, cudaMemcpyHostToDevice, ds->copy_in);
        cp2(b + off[1], fc * per_f_q, hk + f0 * per_f_q, F * per_f_q, fc * per_f_q, cudaMemcpyHostToDevice, ds->copy_in);
        cp2(b + off[2], fc * per_f_v, hv + f0 * per_f_v, F * per_f_v, fc * per_f_v, cudaMemcpyHostToDevice, ds->copy_in);
        cp2(b + off[3], fc * per_f_a, ha + f0 * per_f_a, F * per_f_a, fc * per_f_a, cudaMemcpyHostToDevice, ds->copy_in);
        cp2(b + off[4], fc * per_f_b, hb + f0 * per_f_b, F * per_f_b, fc * per_f_b, cudaMemcpyHostToDevice, ds->copy_in);
        ok = ok && cudaEventRecord(ev_in[slot], ds->copy_in) == cudaSuccess;
        // the forward of chunk i, once its inputs are in and the slot's previous outputs are out
        ok = ok && cudaStreamWaitEvent(st, ev_in[slot], 0) == cudaSuccess;
        if (i >= 2) ok = ok && cudaStreamWaitEvent(st, ev_out[slot], 0) == cudaSuccess;
        if (!ok) break;
        r = run_pass(PassArgs{b + off[0], b + off[1], b + off[2], reinterpret_cast<const float*>(b + off[3]),
                              reinterpret_cast<const float*>(b + off[4]), dstate, b + off[5], dstate, B, H, fc, N,
                              dk, dv},
                     false, st);
        ok = ok && cudaEventRecord(ev_comp[slot], st) == cudaSuccess;
        // its outputs back to the host
        ok = ok && cudaStreamWaitEvent(ds->copy_out, ev_comp[slot], 0) == cudaSuccess;
        cp2(static_cast<uint8_t*>(out) + f0 * per_f_v, F * per_f_v, b + off[5], fc * per_f_v, fc * per_f_v,
            cudaMemcpyDeviceToHost, ds->copy_out);
        ok = ok && cudaEventRecord(ev_out[slot], ds->copy_out) == cudaSuccess;
    }
    // the caller's stream waits for every copy, then returns the final state and frees
    for (int x = 0; x < 2 && made == 7; ++x) {
        cudaStreamWaitEvent(st, ev_in[x], 0);
        cudaStreamWaitEvent(st, ev_out[x], 0);
    }
    if (ok && r == GDN_OK && state_out)
        ok = cudaMemcpyAsync(state_out, dstate, bs, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    cudaFreeAsync(d, st);
    if (cudaStreamSynchronize(st) != cudaSuccess) ok = false;
    for (int x = 0; x < made; ++x) cudaEventDestroy(ev[x]);
    if (r == GDN_OK && !ok) r = GDN_ERR_LAUNCH;
    cudaGetLastError();
    return r;
}

void gdn_set_host_chunk_frames(int frames) { g_host_chunk.store(frames > 0 ? frames : 0); }

void gdn_set_contract_pairs(int on) { g_pairs.store(on != 0 ? 1 : 0); }

}  // extern "C"

namespace {
int current_sms() {
    int sms = 148;
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) sms = n;
    }
    cudaGetLastError();
    return sms;
}
}  // namespace

extern "C" {

size_t gdn_workspace_bytes(int B, int H, int F, int N, int dk, int dv) {
    if (B < 1 || H < 1 || F < 1 || N < 1 || !dim_ok(dk) || !dim_ok(dv)) return 0;
    const long long items = static_cast<long long>(B) * F * H;
    // on a usable device: exactly the plan a call would launch; otherwise the
    // plan with splitting allowed (an upper bound)
    int dev;
    DeviceState* ds;
    if (device_ready(&dev, &ds) == GDN_OK) {
        const PassArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, F, N, dk, dv};
        if (single_pass_heads(a, ds) > 0) return single_layout(a).total;
        return layout_of(items, dk, dv, plan_split(items, chunks_of(N), ds->sms, ds->coop_k1)).total;
    }
    return layout_of(items, dk, dv, plan_split(items, chunks_of(N), current_sms(), true)).total;
}

size_t gdn_step_workspace_bytes(int B, int H, int N, int dk, int dv) {
    return gdn_workspace_bytes(B, H, 1, N, dk, dv);   // a one-frame call never takes the single pass
}

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_NULL_PTR: return "GDN_ERR_NULL_PTR: a required pointer is NULL or not device memory";
        case GDN_ERR_BAD_DIM: return "GDN_ERR_BAD_DIM: B, H, F or N < 1, or a tensor is too large";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: dk and dv must be multiples of 16 in [16, 128]";
        case GDN_ERR_MISALIGNED: return "GDN_ERR_MISALIGNED: q/k/v/out need 16-byte, fp32 arrays 4-byte alignment";
        case GDN_ERR_ALLOC: return "GDN_ERR_ALLOC: workspace allocation failed";
        case GDN_ERR_LAUNCH: return "GDN_ERR_LAUNCH: a CUDA call or kernel launch failed";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a device-side bounded wait ran out";
        case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS: an output overlaps an input";
        case GDN_ERR_NO_DEVICE: return "GDN_ERR_NO_DEVICE: no usable sm_103 device is current";
        case GDN_ERR_TOO_LARGE: return "GDN_ERR_TOO_LARGE: the step needs more scratch than GDN_STEP_NOALLOC_SCRATCH_BYTES";
        case GDN_ERR_RANGE: return "GDN_ERR_RANGE: an input value is outside the entry point's range";
    }
    return "GDN_ERR_UNKNOWN";
}

gdn_status gdn_sync_status(gdn_stream_t stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GDN_ERR_NO_DEVICE; }
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_LAUNCH;
    }
    int code = 0;
    if (cudaMemcpyFromSymbol(&code, gdn::g_error, sizeof(int)) != cudaSuccess) { cudaGetLastError(); return GDN_ERR_LAUNCH; }
    if (code != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(gdn::g_error, &zero, sizeof(int));
        return static_cast<gdn_status>(code);
    }
    return GDN_OK;
}

gdn_status gdn_debug_last_timeout(int* info) {
    if (info == nullptr) return GDN_ERR_NULL_PTR;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return GDN_ERR_NO_DEVICE; }
    int zero[5] = {0, 0, 0, 0, 0};
    int taken = 0;
    if (cudaMemcpyFromSymbol(info, gdn::g_timeout_info, sizeof(zero)) != cudaSuccess ||
        cudaMemcpyToSymbol(gdn::g_timeout_info, zero, sizeof(zero)) != cudaSuccess ||
        cudaMemcpyToSymbol(gdn::g_timeout_taken, &taken, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return GDN_ERR_LAUNCH;
    }
    return GDN_OK;
}

void gdn_set_contract_split(int max_split) { g_max_split.store(max_split > 0 ? max_split : 0); }

void gdn_set_fused_step(int on) { g_fused_step.store(on != 0 ? 1 : 0); }

void gdn_set_single_pass(int on, int contract_ctas, int ring_frames) {
    g_single_pass.store(on != 0 ? 1 : 0);
    g_single_contract.store(contract_ctas > 0 ? contract_ctas : 0);
    g_single_ring.store(ring_frames > 0 ? ring_frames : 0);
}

int gdn_forward_schedule(int B, int H, int F, int N, int dk, int dv) {
    if (B < 1 || H < 1 || F < 1 || N < 1 || !dim_ok(dk) || !dim_ok(dv)) return -1;
    int dev;
    DeviceState* ds;
    if (device_ready(&dev, &ds) != GDN_OK) return -1;
    const PassArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, F, N, dk, dv};
    if (single_pass_heads(a, ds) > 0) return 2;
    return (g_fused_scan.load() != 0 && ds->coop && scan_rows_fused(B, H, dv, ds->sms) != 0) ? 1 : 0;
}

void gdn_set_fused_scan(int mode) {
    g_fused_scan.store((mode == 16 || mode == 32 || mode == 64) ? mode : (mode != 0 ? 1 : 0));
}

int gdn_scan_schedule(int B, int H, int dv) {
    if (B < 1 || H < 1 || !dim_ok(dv)) return 0;
    int dev;
    DeviceState* ds;
    if (device_ready(&dev, &ds) != GDN_OK) return 0;
    const int Rf = (g_fused_scan.load() != 0 && ds->coop) ? scan_rows_fused(B, H, dv, ds->sms) : 0;
    return Rf != 0 ? Rf : -scan_rows_standalone(B, H, dv, ds->sms);
}

void gdn_set_wait_limit_ns(unsigned long long limit_ns) {
    g_wait_limit_ns.store(limit_ns < 1000ULL ? 1000ULL : limit_ns);
}

gdn_status gdn_selftest_wait_timeout(unsigned long long limit_ns, gdn_stream_t stream) {
    int dev;
    DeviceState* ds;
    gdn_status st = device_ready(&dev, &ds);
    if (st != GDN_OK) return st;
    if (limit_ns < 1000ULL) limit_ns = 1000ULL;
    if (limit_ns > 5000000000ULL) limit_ns = 5000000000ULL;
    selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

const char* gdn_version(void) { return "gdn-b300 0.1 (sm_103a, tcgen05)"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free step (gdn_frame_step_noalloc).  For callers that cannot
// allocate device memory while they advance a resident state.  The workspace
// of the step path lives in one file-scope device array instead of a pool
// allocation; the kernels and their launch shapes are those of gdn_frame_step.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStepScratchBytes = GDN_STEP_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_step_scratch[kStepScratchBytes];

// Device address of g_step_scratch per device.  In host code the name
// g_step_scratch is only a host-side stand-in for the symbol, never a device
// address, so it is looked up once per device with that device current.
uint8_t* g_step_scratch_dev[kMaxDevices] = {};
std::mutex g_step_scratch_mu;

gdn_status step_scratch_address(int dev, uint8_t** out) {
    std::lock_guard<std::mutex> lk(g_step_scratch_mu);
    if (g_step_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return GDN_ERR_LAUNCH;
        }
        g_step_scratch_dev[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_step_scratch_dev[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_frame_step_noalloc(const void* q, const void* k, const void* v, const float* alpha,
                                             const float* beta, const float* state_in, void* out,
                                             float* state_out, int B, int H, int N, int dk, int dv,
                                             gdn_stream_t stream_handle) {
    gdn_status st = validate(q, k, v, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv);
    if (st != GDN_OK) return st;
    int dev;
    DeviceState* ds;
    st = device_ready(&dev, &ds);
    if (st != GDN_OK) return st;
    // the array's device address, looked up on the first call on this device
    // whichever step path the call takes
    uint8_t* ws = nullptr;
    st = step_scratch_address(dev, &ws);
    if (st != GDN_OK) return st;
    const PassArgs a{q, k, v, alpha, beta, state_in, out, state_out, B, H, 1, N, dk, dv};
    if (fused_step_applies(a)) {  // the one-launch step keeps everything on chip: no scratch at all
        if (!all_device(a)) return GDN_ERR_NULL_PTR;
        return launch_step_fused(a, reinterpret_cast<cudaStream_t>(stream_handle));
    }
    const long long items = static_cast<long long>(B) * H;
    const SplitPlan sp = plan_split(items, chunks_of(N), ds->sms, ds->coop_k1);
    const Layout L = layout_of(items, dk, dv, sp);
    if (L.total > kStepScratchBytes) return GDN_ERR_TOO_LARGE;
    if (!all_device(a)) return GDN_ERR_NULL_PTR;
    return launch_phases(a, ws, L, sp, ds, reinterpret_cast<cudaStream_t>(stream_handle), nullptr);
}
