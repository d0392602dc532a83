// fwd_splitkv_sm103.cu -- forward attention with the key range of every head
// split into sub-ranges ("sub-ACC" split), then a log-sum-exp merge.
//
// "Optimizing Attention on GPUs by Exploiting GPU Architectural NUMA
// Effects" (related-work page, on the Attention Compute Cluster when one
// head's K/V outgrows an L2 slice) suggests splitting an ACC's keys so that
// the CTAs running together stream a piece of K/V that fits in L2.  Here the
// units of an ACC run key range 0 for all its heads and row blocks, then key
// range 1, and so on; each unit writes the fp32 partial (O_s normalised by
// its own l_s, lse_s) of its rows over its range, and a merge kernel combines
// the ranges of every row as the decode merge does (kernbench2 "Fused
// Grouped-Query Attention", Case 4: the (m, l, O) reduction):
//     L = max_s lse_s,  w_s = exp(lse_s - L),  O = sum_s w_s O_s / sum_s w_s,
//     lse = L + log(sum_s w_s).
// The unit kernel is the forward kernel of fwd_kernel.cuh (same roles, TMEM
// plan, softmax and bounded waits) instantiated with the split mapping; this
// translation unit holds its own copy of the kernel's work counters and
// status word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "fwd_kernel.cuh"

namespace attn {
namespace fwd {

// One warp per query row: combine the row's key ranges.  A causal row i
// attends range s only if it starts at or before i (s * C <= i); otherwise
// that range's partial is not read.  Lane l holds columns [4l, 4l + 4).
__global__ void __launch_bounds__(256)
    split_merge_kernel(const float *part_o, const float *part_lse, __nv_bfloat16 *o, float *lse, long long rows,
                       int N, int d, int splits, int chunk_keys, int causal) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = int(row % N);  // position of the row in its sequence
    const int ns = causal ? min(splits, i / chunk_keys + 1) : splits;
    const size_t stride = (size_t)rows;  // rows per split
    float L = -INFINITY;
    for (int s = 0; s < ns; ++s) L = fmaxf(L, part_lse[s * stride + row]);
    const int c0 = lane * 4;
    const bool active = c0 < d;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float ls = part_lse[s * stride + row];
        if (ls == -INFINITY) continue;
        const float w = __expf(ls - L);
        wsum += w;
        if (active) {
            const float4 v = *reinterpret_cast<const float4 *>(part_o + (s * stride + row) * d + c0);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (active) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(o + row * d + c0) = pk;
    }
    if (lane == 0 && lse) lse[row] = wsum > 0.f ? L + __logf(wsum) : -INFINITY;
}

template <int D>
int launch(const FwdSplitLaunch &a, cudaStream_t stream) {
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const uint64_t dq = uint64_t(a.d);
    if (!encode_bf16_3d(&mq, a.q, dq, uint64_t(a.N), uint64_t(a.B) * a.Hq, 64, kTileM) ||
        !encode_bf16_3d(&mk, a.k, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN) ||
        !encode_bf16_3d(&mv, a.v, dq, uint64_t(a.N), uint64_t(a.B) * a.Hkv, 64, kBlockN))
        return note_cuda_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (split-KV forward)");
    SplitParams p;
    p.o = nullptr;
    p.lse = nullptr;
    p.part_o = a.part_o;
    p.part_lse = a.part_lse;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.G = a.Hq / a.Hkv;
    p.d_store = a.d;
    p.causal = a.causal ? 1 : 0;
    p.order = kHeadFirst;  // one work counter; the split mapping orders the units
    p.die_of_sm = nullptr;
    p.nb = unit_blocks(a.N);
    p.splits = a.splits;
    p.chunk_blocks = a.chunk_keys / kBlockN;
    p.total_units = (long long)a.B * a.Hq * p.nb * a.splits;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_ns = a.wait_ns;
    p.sched_slot = int(g_fwd_launch_seq.fetch_add(1) % kSchedSlots);
    auto kernel = fwd_kernel<D, kMapSplit>;
    static bool attr_set[kMaxDevices] = {};
    const int dev = slot_for_device();
    if (dev < 0 || !attr_set[dev]) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncGetAttributes(fwd_kernel, split)");
        if (fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
            return note_cuda_error(cudaErrorInvalidConfiguration,
                                   "fwd_kernel (split) register count differs from the setmaxnreg split");
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(fwd_kernel, split)");
        if (dev >= 0) attr_set[dev] = true;
    }
    long long grid = p.total_units;
    if (grid > a.num_sms) grid = a.num_sms;
    kernel<<<dim3(unsigned(grid)), dim3(kThreads), C::kSmemBytes, stream>>>(mq, mk, mv, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return note_cuda_error(e, "fwd_kernel (split) launch");
    const long long rows = (long long)a.B * a.Hq * a.N;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return ATTN_ERR_ARG;
    split_merge_kernel<<<dim3(unsigned(blocks)), dim3(256), 0, stream>>>(
        a.part_o, a.part_lse, reinterpret_cast<__nv_bfloat16 *>(a.o), a.lse, rows, a.N, a.d, a.splits, a.chunk_keys,
        a.causal ? 1 : 0);
    e = cudaGetLastError();
    return e == cudaSuccess ? 0 : note_cuda_error(e, "split_merge_kernel launch");
}

}  // namespace fwd

int fwd_split_launch(const FwdSplitLaunch &a, cudaStream_t stream) {
    if (a.d <= 64) return fwd::launch<64>(a, stream);
    return fwd::launch<128>(a, stream);
}

cudaError_t fwd_split_take_status(int *bits) {
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_fwd_status, sizeof(int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(int));
}

}  // namespace attn
