// fwd_host.cu -- forward attention on host-resident tensors: the copies of
// q, k, v to the device, the forward kernels and the copies of o and lse
// back, overlapped in chunks of KV heads.
//
// The tensors are cut into chunks of whole KV heads (each with the query
// heads that read it) of one batch entry, so every chunk is an independent
// forward problem with contiguous pieces of the host tensors.  Chunk c uses
// slot c % 2 of a caller-owned device workspace:
//   copy-in stream : H2D q, k, v of chunk c          (after chunk c-2's kernel)
//   compute stream : forward kernel of chunk c        (after its H2D and after
//                    chunk c-2's D2H); the caller's stream for even chunks,
//                    an internal one for odd chunks, so one chunk's tail
//                    overlaps the next chunk's start
//   copy-out stream: D2H o, lse of chunk c            (after its kernel)
// Every internal stream first waits for the work already on the caller's
// stream, and the caller's stream finally waits for the last copy back, so
// the whole call is ordered on the caller's stream like any other entry point.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "attn_internal.h"

namespace attn {

namespace {

constexpr int kSlots = 2;

struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr, comp = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
};

HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;  // one call enqueues at a time (the streams and events are shared)

// Per-chunk timeline of the last traced call on a device: ev[0] is recorded
// on the caller's stream when the call starts, then four events per chunk
// (copy-in done, kernel reached, kernel done, copy-out done).  Timing events
// are recorded only while tracing is on.
constexpr int kTracePerChunk = 4;
struct HostTrace {
    bool on = false;
    bool valid = false;  // a traced call has been enqueued since tracing was enabled
    long long chunks = 0;
    std::vector<cudaEvent_t> ev;
};
HostTrace g_trace[kMaxDevices];

cudaError_t trace_reserve(HostTrace &tr, long long chunks) {
    const size_t need = size_t(1 + kTracePerChunk * chunks);
    while (tr.ev.size() < need) {
        cudaEvent_t e;
        const cudaError_t rc = cudaEventCreate(&e);
        if (rc != cudaSuccess) return rc;
        tr.ev.push_back(e);
    }
    return cudaSuccess;
}

cudaError_t pipe_init(HostPipe &hp) {
    if (hp.ready) return cudaSuccess;
    cudaError_t e;
    for (cudaStream_t *s : {&hp.in, &hp.out, &hp.comp})
        if (!*s && (e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t *evs[] = {&hp.start, &hp.end, &hp.in_done[0], &hp.in_done[1], &hp.comp_done[0],
                          &hp.comp_done[1], &hp.out_done[0], &hp.out_done[1]};
    for (cudaEvent_t *ev : evs)
        if (!*ev && (e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    hp.ready = true;
    return cudaSuccess;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

HostChunkLayout host_chunk_layout(int Hq, int Hkv, int N, int d, int kv_heads_per_chunk) {
    HostChunkLayout L;
    const size_t G = size_t(Hq / Hkv);
    const size_t gc = size_t(kv_heads_per_chunk);
    const size_t q_bytes = gc * G * size_t(N) * size_t(d) * 2;
    const size_t kv_bytes = gc * size_t(N) * size_t(d) * 2;
    L.q_off = 0;
    L.k_off = round256(q_bytes);
    L.v_off = L.k_off + round256(kv_bytes);
    L.o_off = L.v_off + round256(kv_bytes);
    L.lse_off = L.o_off + round256(q_bytes);
    L.slot_bytes = L.lse_off + round256(gc * G * size_t(N) * 4);
    return L;
}

int host_default_chunk(int Hq, int Hkv, int N) {
    // The fewest KV heads whose chunk holds about two waves of forward work
    // units (256 query rows of one head) on a 152-SM GPU.  Small chunks keep
    // the first copy-in and the last copy-out, which nothing overlaps, short;
    // two waves keep each chunk's kernel busy, and the next chunk's kernel
    // (on the other compute stream) fills its tail.
    constexpr long long kChunkUnits = 2 * 152;
    const long long units_per_kv_head = static_cast<long long>(Hq / Hkv) * ((N + 255) / 256);
    const long long gc = (kChunkUnits + units_per_kv_head - 1) / units_per_kv_head;
    return int(std::max(1LL, std::min<long long>(gc, Hkv)));
}

int fwd_host_launch(const FwdHostLaunch &a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return note_cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return note_cuda_error(cudaErrorInvalidDevice, "device index");
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe &hp = g_pipe[dev];
    if ((e = pipe_init(hp)) != cudaSuccess) return note_cuda_error(e, "stream/event creation (host forward)");

    const FwdLaunch &f0 = a.fwd;
    const int G = f0.Hq / f0.Hkv;
    const int gc = a.kv_heads_per_chunk;
    const int per_b = (f0.Hkv + gc - 1) / gc;
    const long long chunks = static_cast<long long>(f0.B) * per_b;
    const HostChunkLayout L = host_chunk_layout(f0.Hq, f0.Hkv, f0.N, f0.d, gc);
    const size_t N = size_t(f0.N), d = size_t(f0.d);
    const uint8_t *hq = static_cast<const uint8_t *>(a.q_host);
    const uint8_t *hk = static_cast<const uint8_t *>(a.k_host);
    const uint8_t *hv = static_cast<const uint8_t *>(a.v_host);
    uint8_t *ho = static_cast<uint8_t *>(a.o_host);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);

    // On any failure after work was enqueued, the caller's stream still waits
    // for whatever the internal streams hold (best effort), so buffers the
    // caller releases after an error are not in use by a pending copy.
    auto join_internal = [&]() {
        for (cudaStream_t s : {hp.in, hp.comp, hp.out})
            if (cudaEventRecord(hp.end, s) == cudaSuccess) cudaStreamWaitEvent(stream, hp.end, 0);
    };
#define ATTN_CK(call, what)                                   \
    do {                                                      \
        const cudaError_t ck_ = (call);                       \
        if (ck_ != cudaSuccess) {                             \
            join_internal();                                  \
            return note_cuda_error(ck_, what);                \
        }                                                     \
    } while (0)

    HostTrace &tr = g_trace[dev];
    const bool tracing = tr.on;
    if (tracing) {
        tr.valid = false;
        ATTN_CK(trace_reserve(tr, chunks), "cudaEventCreate (host forward trace)");
        ATTN_CK(cudaEventRecord(tr.ev[0], stream), "cudaEventRecord (trace)");
    }
    auto trace_mark = [&](long long c, int k, cudaStream_t s) {
        return tracing ? cudaEventRecord(tr.ev[size_t(1 + kTracePerChunk * c + k)], s) : cudaSuccess;
    };
    ATTN_CK(cudaEventRecord(hp.start, stream), "cudaEventRecord (host forward)");
    for (cudaStream_t s : {hp.in, hp.comp, hp.out})
        ATTN_CK(cudaStreamWaitEvent(s, hp.start, 0), "cudaStreamWaitEvent (host forward)");
    for (long long c = 0; c < chunks; ++c) {
        const int s = int(c & 1);
        const int b = int(c / per_b);
        const int g0 = int(c % per_b) * gc;
        const int gn = std::min(gc, f0.Hkv - g0);
        const int h0 = g0 * G, hn = gn * G;
        uint8_t *slot = ws + size_t(s) * L.slot_bytes;
        const size_t q_bytes = size_t(hn) * N * d * 2, kv_bytes = size_t(gn) * N * d * 2;
        const size_t q_at = (size_t(b) * f0.Hq + h0) * N * d * 2;   // byte offset in q / o
        const size_t kv_at = (size_t(b) * f0.Hkv + g0) * N * d * 2;  // byte offset in k / v
        const size_t l_at = (size_t(b) * f0.Hq + h0) * N;            // float offset in lse

        if (c >= kSlots) ATTN_CK(cudaStreamWaitEvent(hp.in, hp.comp_done[s], 0), "wait (copy-in)");
        ATTN_CK(cudaMemcpyAsync(slot + L.q_off, hq + q_at, q_bytes, cudaMemcpyHostToDevice, hp.in), "copy q");
        ATTN_CK(cudaMemcpyAsync(slot + L.k_off, hk + kv_at, kv_bytes, cudaMemcpyHostToDevice, hp.in), "copy k");
        ATTN_CK(cudaMemcpyAsync(slot + L.v_off, hv + kv_at, kv_bytes, cudaMemcpyHostToDevice, hp.in), "copy v");
        // Each trace mark goes on its stream before the event other streams
        // wait on, so a time on one stream never follows one that depends on it.
        ATTN_CK(trace_mark(c, 0, hp.in), "cudaEventRecord (trace)");
        ATTN_CK(cudaEventRecord(hp.in_done[s], hp.in), "cudaEventRecord (copy-in)");

        cudaStream_t cs = (s == 0) ? stream : hp.comp;
        ATTN_CK(cudaStreamWaitEvent(cs, hp.in_done[s], 0), "wait (compute)");
        if (c >= kSlots) ATTN_CK(cudaStreamWaitEvent(cs, hp.out_done[s], 0), "wait (compute)");
        FwdLaunch f = f0;
        f.q = slot + L.q_off;
        f.k = slot + L.k_off;
        f.v = slot + L.v_off;
        f.o = slot + L.o_off;
        f.lse = a.lse_host ? reinterpret_cast<float *>(slot + L.lse_off) : nullptr;
        f.B = 1;
        f.Hq = hn;
        f.Hkv = gn;
        ATTN_CK(trace_mark(c, 1, cs), "cudaEventRecord (trace)");
        const int rc = fwd_run(f, cs);
        if (rc != 0) {
            join_internal();
            return rc;
        }
        ATTN_CK(trace_mark(c, 2, cs), "cudaEventRecord (trace)");
        ATTN_CK(cudaEventRecord(hp.comp_done[s], cs), "cudaEventRecord (compute)");

        ATTN_CK(cudaStreamWaitEvent(hp.out, hp.comp_done[s], 0), "wait (copy-out)");
        ATTN_CK(cudaMemcpyAsync(ho + q_at, slot + L.o_off, q_bytes, cudaMemcpyDeviceToHost, hp.out), "copy o");
        if (a.lse_host)
            ATTN_CK(cudaMemcpyAsync(a.lse_host + l_at, slot + L.lse_off, size_t(hn) * N * 4,
                                    cudaMemcpyDeviceToHost, hp.out),
                    "copy lse");
        ATTN_CK(trace_mark(c, 3, hp.out), "cudaEventRecord (trace)");
        ATTN_CK(cudaEventRecord(hp.out_done[s], hp.out), "cudaEventRecord (copy-out)");
    }
    if (tracing) {
        tr.chunks = chunks;
        tr.valid = true;
    }
    ATTN_CK(cudaEventRecord(hp.end, hp.out), "cudaEventRecord (host forward end)");
    ATTN_CK(cudaStreamWaitEvent(stream, hp.end, 0), "cudaStreamWaitEvent (host forward end)");
#undef ATTN_CK
    return 0;
}

int fwd_host_trace(int enable) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return note_cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return note_cuda_error(cudaErrorInvalidDevice, "device index");
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    g_trace[dev].on = enable != 0;
    if (enable) g_trace[dev].valid = false;  // switching off keeps the last timeline readable
    return 0;
}

long long fwd_host_trace_read(float *ms, long long capacity) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return note_cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return note_cuda_error(cudaErrorInvalidDevice, "device index");
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostTrace &tr = g_trace[dev];
    if (!tr.valid) return -1;
    const long long n = tr.chunks;
    // The copy-out stream's last event follows every other event of the call.
    if ((e = cudaEventSynchronize(tr.ev[size_t(kTracePerChunk * n)])) != cudaSuccess)
        return note_cuda_error(e, "cudaEventSynchronize (trace)");
    const long long m = std::min(n, capacity);
    for (long long c = 0; c < m; ++c)
        for (int k = 0; k < kTracePerChunk; ++k) {
            float t = 0.f;
            if ((e = cudaEventElapsedTime(&t, tr.ev[0], tr.ev[size_t(1 + kTracePerChunk * c + k)])) !=
                cudaSuccess)
                return note_cuda_error(e, "cudaEventElapsedTime (trace)");
            ms[kTracePerChunk * c + k] = t;
        }
    return n;
}

}  // namespace attn
