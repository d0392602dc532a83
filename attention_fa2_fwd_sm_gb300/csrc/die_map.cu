// die_map.cu -- which of the GPU's two dies each SM sits on, found by
// measurement, for the die-split tile order.
//
// GB300 is two dies behind one coherent L2.  Every global address has a home
// L2 partition on one of the dies, and an SM reaches lines homed on its own die
// faster than lines homed on the other die.  So the latency an SM sees to a
// fixed set of addresses has one pattern for all SMs of one die and the
// opposite pattern for the SMs of the other die.  SM ids do not follow the die
// boundary in any documented way, hence the calibration:
//   1. one thread per SM times chains of dependent L2-only loads to kProbes
//      words kProbeStride bytes apart, keeping per word the fastest of
//      kPasses passes after a warm-up pass (the lines are then in L2, and
//      the minimum drops the delays of other SMs' traffic);
//   2. the host removes from the latency matrix each SM's mean and each
//      word's mean over all SMs (so neither a slow SM nor a word that is slow
//      for everyone counts), normalises each SM's vector and splits the SMs
//      in two: first by the sign of their correlation with SM 0's vector,
//      then by repeatedly assigning each SM to the group whose mean vector it
//      correlates with more (two-means on correlation);
//   3. the split is accepted when every SM correlates with its own group's
//      mean by at least kMinMargin more than with the other group's, and both
//      dies hold at least a quarter of the SMs; otherwise the map falls back
//      to SM ids split in halves.  SM 0's group is die 0.
// The map is measured once per device, on first use, and kept in a device
// array that the forward kernel reads through %smid.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "attn_internal.h"

namespace attn {

namespace {
constexpr int kProbes = 128;         // probe words
constexpr int kProbeStride = 4096;   // bytes between probe words
constexpr int kChain = 16;           // dependent loads timed per word and pass
constexpr int kPasses = 3;           // timed passes (after one warm-up pass)
constexpr int kProbeSmem = 120 * 1024;  // forces one probe CTA per SM
constexpr double kMinMargin = 0.5;
}  // namespace

static __device__ int g_die_of_sm[kDieMapMaxSms];
static __device__ __align__(256) unsigned int g_probe_buf[kProbes * kProbeStride / 4];
static __device__ unsigned int g_probe_lat[kDieMapMaxSms * kProbes];
static __device__ unsigned int g_probe_seen[kDieMapMaxSms];

// One thread per CTA.  The loop bounds are kernel arguments and the chain
// loop is kept rolled: the clock reads then sit in other basic blocks than the
// loads they time, so the compiler cannot move them across the loads.
__global__ void __launch_bounds__(32) die_probe_kernel(int probes, int stride_words, int chain, int passes) {
    extern __shared__ unsigned char keep_one_cta_per_sm[];
    if (threadIdx.x != 0) return;
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    if (smid >= uint32_t(kDieMapMaxSms) || probes > kProbes) return;
    keep_one_cta_per_sm[0] = 0;
    for (int pr = 0; pr < probes; ++pr) {
        const unsigned int *a = g_probe_buf + (size_t)pr * stride_words;
        uint32_t best = 0xffffffffu;
        for (int pass = 0; pass <= passes; ++pass) {
            uint32_t x = 0;  // the buffer holds zeros: a + x is a, but each load waits for the last
            const long long t0 = clock64();
#pragma unroll 1
            for (int i = 0; i < chain; ++i)
                asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(x) : "l"(a + x) : "memory");
            keep_one_cta_per_sm[1] = (unsigned char)x;  // consumes the last load
            const long long t1 = clock64();
            const uint32_t v = uint32_t((t1 - t0) / chain);
            if (pass > 0 && v < best) best = v;
        }
        g_probe_lat[smid * kProbes + pr] = best;
    }
    g_probe_seen[smid] = 1u;
}

namespace {

struct DieState {
    bool done = false;
    int n = 0;                 // SM count
    std::vector<int> die;      // per SM id
    float stats[4] = {0, 0, 0, 0};
};

std::mutex g_die_mutex;
DieState g_die_state[kMaxDevices];

void halves(DieState &st) {
    st.die.assign(st.n, 0);
    for (int i = 0; i < st.n; ++i) st.die[i] = i < st.n / 2 ? 0 : 1;
}

// Split the SMs in two by their latency patterns (see the file comment).
// Returns true when the split is clean.
bool cluster(const std::vector<float> &lat, DieState &st) {
    const int n = st.n;
    std::vector<double> c(size_t(n) * kProbes);
    std::vector<double> row_mean(n, 0.0), col_mean(kProbes, 0.0);
    double all_mean = 0;
    for (int s = 0; s < n; ++s)
        for (int p = 0; p < kProbes; ++p) {
            const double v = lat[size_t(s) * kProbes + p];
            row_mean[s] += v / kProbes;
            col_mean[p] += v / n;
            all_mean += v / (double(n) * kProbes);
        }
    for (int s = 0; s < n; ++s) {
        double nn = 0;
        for (int p = 0; p < kProbes; ++p) {
            const double v = lat[size_t(s) * kProbes + p] - row_mean[s] - col_mean[p] + all_mean;
            c[size_t(s) * kProbes + p] = v;
            nn += v * v;
        }
        if (!(nn > 0)) return false;  // a flat pattern carries no die information
        const double inv = 1.0 / std::sqrt(nn);
        for (int p = 0; p < kProbes; ++p) c[size_t(s) * kProbes + p] *= inv;
    }
    auto dot = [&](const double *a, const double *b) {
        double r = 0;
        for (int p = 0; p < kProbes; ++p) r += a[p] * b[p];
        return r;
    };
    std::vector<int> die(n);
    for (int s = 0; s < n; ++s) die[s] = dot(&c[size_t(s) * kProbes], &c[0]) >= 0 ? 0 : 1;
    std::vector<double> cen(2 * kProbes);
    std::vector<double> margin(n, 0.0);
    int count[2] = {0, 0};
    for (int it = 0; it < 16; ++it) {
        std::fill(cen.begin(), cen.end(), 0.0);
        count[0] = count[1] = 0;
        for (int s = 0; s < n; ++s) {
            ++count[die[s]];
            for (int p = 0; p < kProbes; ++p) cen[die[s] * kProbes + p] += c[size_t(s) * kProbes + p];
        }
        if (count[0] == 0 || count[1] == 0) return false;
        for (int k = 0; k < 2; ++k) {
            double nn = 0;
            for (int p = 0; p < kProbes; ++p) nn += cen[k * kProbes + p] * cen[k * kProbes + p];
            if (!(nn > 0)) return false;
            const double inv = 1.0 / std::sqrt(nn);
            for (int p = 0; p < kProbes; ++p) cen[k * kProbes + p] *= inv;
        }
        bool moved = false;
        for (int s = 0; s < n; ++s) {
            const double r0 = dot(&c[size_t(s) * kProbes], &cen[0]);
            const double r1 = dot(&c[size_t(s) * kProbes], &cen[kProbes]);
            const int d = r1 > r0 ? 1 : 0;
            margin[s] = d ? r1 - r0 : r0 - r1;
            moved |= d != die[s];
            die[s] = d;
        }
        if (!moved) break;
    }
    if (die[0] != 0)  // SM 0's group is die 0
        for (int s = 0; s < n; ++s) die[s] ^= 1;
    count[0] = count[1] = 0;
    double min_margin = 2.0;
    for (int s = 0; s < n; ++s) {
        ++count[die[s]];
        min_margin = std::fmin(min_margin, margin[s]);
    }
    // Near / far latency: for each probe word, the lower and the higher of the
    // two dies' mean latencies.
    double near_sum = 0, far_sum = 0;
    if (count[0] > 0 && count[1] > 0) {
        for (int p = 0; p < kProbes; ++p) {
            double m[2] = {0, 0};
            for (int s = 0; s < n; ++s) m[die[s]] += lat[size_t(s) * kProbes + p];
            m[0] /= count[0];
            m[1] /= count[1];
            near_sum += std::fmin(m[0], m[1]);
            far_sum += std::fmax(m[0], m[1]);
        }
    }
    st.die = die;
    st.stats[1] = float(min_margin);
    st.stats[2] = float(near_sum / kProbes);
    st.stats[3] = float(far_sum / kProbes);
    return min_margin >= kMinMargin && count[0] >= n / 4 && count[1] >= n / 4;
}

// Measure (or fall back) and upload the map of device `dev`, which is current.
int calibrate(int dev, DieState &st) {
    int n = 0;
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return note_cuda_error(e, "device query (die map)");
    st.n = n < kDieMapMaxSms ? n : kDieMapMaxSms;
    bool measured = false;
    int reason = -2;  // fallback reason: -2 more SMs than the map holds
    if (n <= kDieMapMaxSms) {
        reason = -1;  // the probe did not run on every SM
        e = cudaFuncSetAttribute(die_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kProbeSmem);
        if (e != cudaSuccess) return note_cuda_error(e, "cudaFuncSetAttribute(die_probe_kernel)");
        std::vector<unsigned int> zeros(kProbes * kProbeStride / 4, 0u);
        e = cudaMemcpyToSymbol(g_probe_buf, zeros.data(), zeros.size() * sizeof(unsigned int));
        if (e != cudaSuccess) return note_cuda_error(e, "cudaMemcpyToSymbol(die probe buffer)");
        std::vector<unsigned int> seen(kDieMapMaxSms, 0u);
        std::vector<unsigned int> lat(size_t(kDieMapMaxSms) * kProbes, 0u);
        for (int attempt = 0; attempt < 3; ++attempt) {
            e = cudaMemcpyToSymbol(g_probe_seen, seen.data(), seen.size() * sizeof(unsigned int));
            if (e != cudaSuccess) return note_cuda_error(e, "cudaMemcpyToSymbol(die probe flags)");
            die_probe_kernel<<<n * (attempt + 1), 32, kProbeSmem>>>(kProbes, kProbeStride / 4, kChain, kPasses);
            e = cudaGetLastError();
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return note_cuda_error(e, "die_probe_kernel");
            std::vector<unsigned int> got(kDieMapMaxSms);
            e = cudaMemcpyFromSymbol(got.data(), g_probe_seen, got.size() * sizeof(unsigned int));
            if (e == cudaSuccess)
                e = cudaMemcpyFromSymbol(lat.data(), g_probe_lat, lat.size() * sizeof(unsigned int));
            if (e != cudaSuccess) return note_cuda_error(e, "cudaMemcpyFromSymbol(die probe)");
            int covered = 0;
            for (int s = 0; s < n; ++s) covered += got[s] ? 1 : 0;
            if (covered == n) {
                std::vector<float> f(size_t(n) * kProbes);
                for (size_t i = 0; i < f.size(); ++i) f[i] = float(lat[i]);
                measured = cluster(f, st);
                reason = 0;  // the split was not clean
                break;
            }
        }
    }
    if (!measured) halves(st);
    st.stats[0] = measured ? 1.f : float(reason);
    std::vector<int> up(kDieMapMaxSms, 0);
    for (int s = 0; s < st.n; ++s) up[s] = st.die[s];
    e = cudaMemcpyToSymbol(g_die_of_sm, up.data(), up.size() * sizeof(int));
    if (e != cudaSuccess) return note_cuda_error(e, "cudaMemcpyToSymbol(die map)");
    st.done = true;
    return 0;
}

int ensure(DieState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return note_cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return note_cuda_error(cudaErrorInvalidDevice, "device index (die map)");
    std::lock_guard<std::mutex> lock(g_die_mutex);
    DieState &st = g_die_state[dev];
    if (!st.done) {
        const int rc = calibrate(dev, st);
        if (rc < 0) return rc;
    }
    *out = &st;
    return 0;
}

}  // namespace

int die_map_device(const int **ptr) {
    DieState *st = nullptr;
    const int rc = ensure(&st);
    if (rc < 0) return rc;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_die_of_sm);
    if (e != cudaSuccess) return note_cuda_error(e, "cudaGetSymbolAddress(die map)");
    *ptr = static_cast<const int *>(p);
    return 0;
}

int die_map_query(int *die_of_sm, int capacity, float *stats) {
    DieState *st = nullptr;
    const int rc = ensure(&st);
    if (rc < 0) return rc;
    if (die_of_sm)
        for (int s = 0; s < capacity && s < st->n; ++s) die_of_sm[s] = st->die[s];
    if (stats) std::memcpy(stats, st->stats, sizeof(st->stats));
    return st->n;
}

}  // namespace attn
