// attn_internal.h -- interfaces between the C-ABI layer and the kernel
// translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Forward tile schemes: one 256-row unit per SM, or 512-row units on CTA
// pairs (cta_group::2 MMAs).
enum FwdScheme : int { kSchemeAuto = 0, kSchemeSingle = 1, kSchemePair = 2 };

struct FwdLaunch {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int B, Hq, Hkv, N, d;
    float scale;
    int causal, order;
    unsigned long long wait_ns;
    int num_sms;
    int scheme = kSchemeAuto;
};

struct BwdLaunch {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int B, Hq, Hkv, N, d;
    float scale;
    int causal, order;
    float *workspace;  // 2 * B * Hq * roundup(N, 128) floats
    int kv_split = 1;      // dK/dV query-head split (bwd_kv_split), used when part is set
    float *part = nullptr;  // its fp32 partials, bwd_part_bytes
    unsigned long long wait_ns;
    int num_sms;
};
int bwd_kv_split(int B, int Hq, int Hkv, int N, int causal);
size_t bwd_part_bytes(int B, int Hkv, int N, int d, int kv_split);

struct DecodeLaunch {
    const void *q, *kcache, *vcache;
    const int *seqlens;
    void *o;
    int B, Hq, Hkv, d, max_seqlen, num_splits;
    float scale;
    float *ws_o, *ws_lse;  // partial outputs / log-sum-exps (used when splits > 1)
    unsigned long long wait_ns;
    int num_sms = 0;       // SMs of the device (0: unknown); picks the ring depth
    // Varlen path (plan != null): work list, its capacity, and the chunk rule.
    int *plan = nullptr;
    int varlen_max_items = 0;
    long long varlen_target = 0;
    int varlen_min_chunk = 0;
};

// Forward on host-resident tensors (fwd_host.cu): `fwd` holds the problem
// (its q, k, v, o, lse pointers are unused), the rest the host buffers, the
// chunk size in KV heads and the device workspace of two chunk slots.
struct FwdHostLaunch {
    FwdLaunch fwd;
    const void *q_host, *k_host, *v_host;
    void *o_host;
    float *lse_host;  // may be null
    int kv_heads_per_chunk;
    void *workspace;
};

// Byte offsets of one workspace slot (one chunk of kv_heads_per_chunk KV
// heads and their query heads): q, k, v, o (bf16) and lse (fp32), each
// starting on a 256-byte boundary.
struct HostChunkLayout {
    size_t q_off, k_off, v_off, o_off, lse_off, slot_bytes;
};
HostChunkLayout host_chunk_layout(int Hq, int Hkv, int N, int d, int kv_heads_per_chunk);
int host_default_chunk(int Hq, int Hkv, int N);
int fwd_host_launch(const FwdHostLaunch &a, cudaStream_t stream);
// Per-chunk timeline of fwd_host_launch on the current device (see
// attn_fwd_host_trace in attn.h).  fwd_host_trace_read returns the chunk count
// of the last traced call, -1 when there is none, or an ATTN_ERR_* code.
int fwd_host_trace(int enable);
long long fwd_host_trace_read(float *ms, long long capacity);

// Kernel attributes (the dynamic shared-memory limit) belong to the current
// device, so the launchers set them once per device: slot_for_device()
// gives the current device's index into a per-device flag array, or -1 when
// it is out of range (then the attributes are set on every launch).
constexpr int kMaxDevices = 64;
inline int slot_for_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Record a failed CUDA call for attn_last_error() (this thread) and return
// ATTN_ERR_CUDA.
int note_cuda_error(cudaError_t e, const char *where);

// Each returns 0 or a negative ATTN_ERR_* code.
// fwd_run picks the launcher for a.scheme (fwd_launch: one CTA per unit;
// fwd_pair_launch: CTA pairs, d = 128 only).
int fwd_run(const FwdLaunch &a, cudaStream_t stream);
int fwd_launch(const FwdLaunch &a, cudaStream_t stream);
int fwd_pair_launch(const FwdLaunch &a, cudaStream_t stream);
int fwd_pair_units_per_head(int N);

// Split-KV forward (fwd_splitkv_sm103.cu): `fwd`'s problem with every head's
// keys cut into `splits` ranges of `chunk_keys` keys (a multiple of 128); the
// partials go to part_o ([splits][B * Hq][N][d] fp32) and part_lse
// ([splits][B * Hq][N] fp32), then a merge kernel writes o and lse.
struct FwdSplitLaunch {
    const void *q, *k, *v;
    void *o;
    float *lse;
    int B, Hq, Hkv, N, d;
    float scale;
    int causal;
    int splits, chunk_keys;
    float *part_o, *part_lse;
    unsigned long long wait_ns;
    int num_sms;
};
int fwd_split_launch(const FwdSplitLaunch &a, cudaStream_t stream);
int decode_launch(const DecodeLaunch &a, cudaStream_t stream);
int bwd_launch(const BwdLaunch &a, cudaStream_t stream);

// Size of the built-in scratch array used by attn_decode_noalloc.
constexpr size_t kDecodeNoAllocScratchBytes = size_t(4) << 20;
// Largest split count attn_decode accepts (the merge stages one lse per split
// in shared memory).
constexpr int kDecodeMaxSplits = 256;

// Device address of that array on the current device (looked up on the
// first call for each device).
cudaError_t decode_noalloc_scratch(void **ptr);

// SM -> die map of the current device for the die-split order (measured on
// the first call for each device; see die_map.cu).  die_map_device gives the
// device address of the map (kDieMapMaxSms ints, one per SM id);
// die_map_query copies it to the host with the calibration statistics and
// returns the SM count.  Both return a negative ATTN_ERR_* code on failure.
constexpr int kDieMapMaxSms = 256;
int die_map_device(const int **ptr);
int die_map_query(int *die_of_sm, int capacity, float *stats);

// Read and clear the status word of each kernel translation unit (OR of
// kStatus* bits).
cudaError_t fwd_take_status(int *bits);
cudaError_t fwd_pair_take_status(int *bits);
cudaError_t fwd_split_take_status(int *bits);
cudaError_t decode_take_status(int *bits);
cudaError_t bwd_take_status(int *bits);

// Tiled bf16 tensor map over a 3-D row-major tensor [dim2][dim1][dim0]
// (dim0 contiguous), box {box0, box1, 1}, 128-byte swizzle, zero fill out of
// bounds.  Returns false if the driver rejects it.
bool encode_bf16_3d(CUtensorMap *map, const void *base, uint64_t dim0, uint64_t dim1,
                    uint64_t dim2, uint32_t box0, uint32_t box1);

}  // namespace attn
