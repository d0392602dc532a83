// fwd_sm103.cu -- launches of the forward (prefill) kernel over the tile
// orders of tile_order.cuh ("Optimizing Attention on GPUs by Exploiting GPU
// Architectural NUMA Effects", detail page, section 3 "before/after" table:
// head-first and block-first, their naive forms, and the die-split
// head-first order) and the grouped causal GQA mapping.  The kernel body,
// its roles and its TMEM plan are in fwd_kernel.cuh.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "attn_internal.h"
#include "fwd_kernel.cuh"

namespace attn {
namespace fwd {

template <int D>
int launch(const FwdLaunch &a, cudaStream_t stream) {
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const uint64_t dq = uint64_t(a.d);
    if (!encode_bf16_3d(&mq, a.q, dq, uint64_t(a.N), uint64_t(a.B) * a.Hq, 64, kTileM) ||
        !encode_bf16_3d(&mk, a.k, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN) ||
        !encode_bf16_3d(&mv, a.v, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN))
        return note_cuda_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (forward)");
    Params p;
    p.o = reinterpret_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.d_store = a.d;
    p.causal = a.causal ? 1 : 0;
    p.order = a.order;
    p.nb = unit_blocks(a.N);
    p.total_units = (long long)a.B * a.Hq * p.nb;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_ns = a.wait_ns;
    p.sched_slot = int(g_fwd_launch_seq.fetch_add(1) % kSchedSlots);
    p.die_of_sm = nullptr;
    if (a.order == kDieSplitHeadFirst) {
        const int rc = die_map_device(&p.die_of_sm);
        if (rc < 0) return rc;
    }
    p.order = effective_order(a.order, a.Hq, p.G, p.nb, p.causal);  // head-first over a whole entry
    const bool grouped = grouped_causal_order(p.order, p.G, p.causal);
    auto kernel = grouped ? fwd_kernel<D, kMapGrouped> : fwd_kernel<D, kMapOrder>;
    static bool attr_set[2][kMaxDevices] = {};  // per instantiation and device
    const int dev = slot_for_device();
    if (dev < 0 || !attr_set[grouped][dev]) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncGetAttributes(fwd_kernel)");
        // The setmaxnreg split assumes the launch register count; refuse to
        // launch a build that differs (its setmaxnreg.inc could never finish).
        if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
            return note_cuda_error(cudaErrorInvalidConfiguration,
                                   "fwd_kernel register count differs from the setmaxnreg split");
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(fwd_kernel)");
        if (dev >= 0) attr_set[grouped][dev] = true;
    }
    long long grid = p.total_units;
    if (a.order != kNaiveHeadFirst && grid > a.num_sms) grid = a.num_sms;
    if (grid > 0x7fffffffLL) return -2;
    kernel<<<dim3(unsigned(grid)), dim3(kThreads), C::kSmemBytes, stream>>>(mq, mk, mv, p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : note_cuda_error(e, "fwd_kernel launch");
}

}  // namespace fwd

int fwd_launch(const FwdLaunch &a, cudaStream_t stream) {
    if (a.d <= 64) return fwd::launch<64>(a, stream);
    return fwd::launch<128>(a, stream);
}

cudaError_t fwd_take_status(int *bits) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_fwd_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(int));
}

}  // namespace attn
