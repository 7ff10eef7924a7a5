// xs_burst.cu -- Burst-Gap store microbenchmark (X-Stage paper, arXiv
// 2607.23264v1, section 3.1): K producers write bursts of B bytes separated by
// a producer-side gap, and each burst's sender-visible issue time and the
// start-to-start period are recorded with clock64. On one GPU the stores go to
// local memory: this is the pages' local-memory control path, used here to
// calibrate the drain rate, the backpressure-free issue time and the effective
// outstanding capacity of this GPU's own store path (sections 3.3-3.5).
//
// Producers are CTAs of `warps` warps, one per SM, launched cooperatively so that
// all of them are resident; the grid-wide barriers that align them are bounded
// in time and report a timeout instead of waiting forever.
#include "../../include/xs_burst.h"

#include <cmath>
#include <cstdio>
#include <mutex>
#include <vector>

#include "xs_internal.h"
#include "xs_ptx.cuh"

namespace xs {

namespace {

struct BurstParams {
    uint8_t *buf;
    uint32_t *hdr;                  // [0] barrier arrivals, [1] error flag
    unsigned long long *clk;        // [K][4]: globaltimer and clock64 at start and end
    unsigned long long *rec;        // [K][n_bursts][2]: clock64 at burst start and issue end
    uint32_t K, n_bursts;
    uint32_t warps;                 // warps per producer
    uint32_t chunks_per_warp;       // 16-byte chunks each warp stores per burst
    uint32_t cpr_log2;              // log2(16-byte chunks per row)
    uint32_t rows_per_burst, n_slots;
    uint64_t row_stride;
    uint64_t gap_cycles;
    int isolated;
};

constexpr uint32_t kBurstSmem = 120 * 1024;  // two producers cannot share an SM
constexpr unsigned long long kBarrierLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier number `target / K`; returns false if it ran out of time
// (or another producer's did), after raising the error flag.
__device__ bool grid_sync(const BurstParams &p, uint32_t &target) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        target += p.K;
        __threadfence();
        atomicAdd(p.hdr, 1u);
        const unsigned long long t0 = globaltimer_ns();
        int ok = 1;
        while (ld_acquire(p.hdr) < target) {
            if (ld_acquire(p.hdr + 1) != 0u || globaltimer_ns() - t0 > kBarrierLimitNs) {
                atomicOr(p.hdr + 1, 1u);
                ok = 0;
                break;
            }
        }
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

__device__ __forceinline__ void spin_cycles(unsigned long long cycles) {
    const unsigned long long t0 = clock64_now();
    while (clock64_now() - t0 < cycles) {
    }
}

__global__ void __launch_bounds__(1024, 1) burst_gap_kernel(const BurstParams p) {
    const uint32_t k = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t target = 0;
    if (threadIdx.x == 0) {
        p.clk[k * 4 + 0] = globaltimer_ns();
        p.clk[k * 4 + 1] = clock64_now();
    }
    if (!grid_sync(p, target)) return;
    const uint32_t x = k * 0x9E3779B9u ^ threadIdx.x;
    const uint32_t cmask = (1u << p.cpr_log2) - 1u;
    for (uint32_t n = 0; n < p.n_bursts; ++n) {
        if (p.isolated) {
            spin_cycles(p.gap_cycles);  // recovery, then all producers start together
            if (!grid_sync(p, target)) return;
        } else {
            __syncthreads();
        }
        const unsigned long long t0 = clock64_now();
        const uint64_t row0 = (uint64_t)((n * p.K + k) % p.n_slots) * p.rows_per_burst;
        for (uint32_t i = lane; i < p.chunks_per_warp; i += 32) {
            const uint32_t c = warp * p.chunks_per_warp + i;
            uint8_t *ptr = p.buf + (row0 + (c >> p.cpr_log2)) * p.row_stride + (uint64_t)(c & cmask) * 16u;
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(x), "r"(n), "r"(c), "r"(k)
                         : "memory");
        }
        __syncthreads();  // every warp of the producer has issued its stores
        const unsigned long long t1 = clock64_now();
        if (threadIdx.x == 0) {
            p.rec[((uint64_t)k * p.n_bursts + n) * 2 + 0] = t0;
            p.rec[((uint64_t)k * p.n_bursts + n) * 2 + 1] = t1;
        }
        if (!p.isolated) spin_cycles(p.gap_cycles);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        p.clk[k * 4 + 2] = globaltimer_ns();
        p.clk[k * 4 + 3] = clock64_now();
    }
}

// SM clock in MHz from a 2 ms spin (clock64 against %globaltimer).
__global__ void clock_probe_kernel(unsigned long long *out) {
    const unsigned long long g0 = globaltimer_ns(), c0 = clock64_now();
    while (globaltimer_ns() - g0 < 2000000ull) {
    }
    out[0] = globaltimer_ns() - g0;
    out[1] = clock64_now() - c0;
}

struct DevClock {
    bool ready = false;
    double mhz = 0.0;
};
DevClock g_clock[64];
std::mutex g_clock_mu;

int fail(int st, const char *msg) { return report_error(st, msg); }

int fail_cuda(const char *what, cudaError_t e) {
    char buf[256];
    snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return report_error(XS_ERR_CUDA, buf);
}

int measure_clock(int dev, unsigned long long *scratch, cudaStream_t s, double *mhz) {
    std::lock_guard<std::mutex> lk(g_clock_mu);
    if (dev < 0 || dev >= 64) return fail(XS_ERR_UNSUPPORTED, "device ordinal out of range");
    if (!g_clock[dev].ready) {
        clock_probe_kernel<<<1, 1, 0, s>>>(scratch);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda("clock probe launch", e);
        unsigned long long h[2] = {0, 0};
        if ((e = cudaMemcpyAsync(h, scratch, sizeof h, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
            (e = cudaStreamSynchronize(s)) != cudaSuccess)
            return fail_cuda("clock probe", e);
        if (h[0] == 0) return fail(XS_ERR_CUDA, "clock probe measured no time");
        g_clock[dev].mhz = 1e3 * (double)h[1] / (double)h[0];
        g_clock[dev].ready = true;
    }
    *mhz = g_clock[dev].mhz;
    return XS_OK;
}

size_t rec_bytes_for(int K, int n) { return 256 + (size_t)K * 32 + (size_t)K * n * 16; }

}  // namespace
}  // namespace xs

extern "C" {

size_t xs_burst_rec_bytes(int K, int n_bursts) {
    if (K < 1 || n_bursts < 1) return 0;
    return xs::rec_bytes_for(K, n_bursts);
}

xs_status xs_burst_gap(void *buf, size_t buf_bytes, void *rec, size_t rec_bytes, int K, int warps, int B,
                       double gap_ns, int n_bursts, int isolated, int row_bytes, int row_stride, xs_burst_stats *stats,
                       void *stream) {
    using namespace xs;
    if (!buf || !rec || !stats) return (xs_status)fail(XS_ERR_NULL, "buf, rec and stats must be non-NULL");
    if (((uintptr_t)buf & 15u) || ((uintptr_t)rec & 15u))
        return (xs_status)fail(XS_ERR_ALIGN, "buf and rec must be 16-byte aligned");
    if (row_bytes < 16 || row_bytes > 4096 || (row_bytes & (row_bytes - 1)))
        return (xs_status)fail(XS_ERR_SHAPE, "row_bytes must be a power of two in 16..4096");
    if (row_stride < row_bytes || row_stride % 16)
        return (xs_status)fail(XS_ERR_SHAPE, "row_stride must be >= row_bytes and a multiple of 16");
    if (warps < 1 || warps > 32) return (xs_status)fail(XS_ERR_SHAPE, "warps must be in 1..32");
    if (B < 512 * warps || B % (512 * warps) || B % row_bytes || B > (1 << 26))
        return (xs_status)fail(XS_ERR_SHAPE, "B must be a multiple of 512*warps and of row_bytes, at most 64 MiB");
    if (n_bursts < 2 || n_bursts > 4096) return (xs_status)fail(XS_ERR_SHAPE, "n_bursts must be in 2..4096");
    if (!(gap_ns >= 0.0 && gap_ns <= 1e6)) return (xs_status)fail(XS_ERR_SHAPE, "gap_ns must be in 0..1e6");
    if (K < 1) return (xs_status)fail(XS_ERR_SHAPE, "K must be >= 1");
    if (rec_bytes < rec_bytes_for(K, n_bursts))
        return (xs_status)fail(XS_ERR_SHAPE, "rec is smaller than xs_burst_rec_bytes(K, n_bursts)");
    const uint64_t rows_per_burst = (uint64_t)B / row_bytes;
    const uint64_t slot_bytes = rows_per_burst * (uint64_t)row_stride;
    if (buf_bytes < slot_bytes) return (xs_status)fail(XS_ERR_SHAPE, "buf is smaller than one burst slot");
    const uint64_t total_rows = buf_bytes / (uint64_t)row_stride;
    const uint64_t n_slots = total_rows / rows_per_burst;
    if (n_slots > 0xFFFFFFFFull) return (xs_status)fail(XS_ERR_SHAPE, "buf holds too many burst slots");

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (xs_status)fail_cuda("cudaGetDevice", e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return (xs_status)fail_cuda("cudaDeviceGetAttribute", e);
    if (K > sms) return (xs_status)fail(XS_ERR_SHAPE, "K exceeds the number of SMs");
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    uint8_t *r8 = static_cast<uint8_t *>(rec);
    double mhz = 0.0;
    int st = measure_clock(dev, reinterpret_cast<unsigned long long *>(r8 + 64), s, &mhz);
    if (st) return (xs_status)st;

    BurstParams p;
    p.buf = static_cast<uint8_t *>(buf);
    p.hdr = reinterpret_cast<uint32_t *>(r8);
    p.clk = reinterpret_cast<unsigned long long *>(r8 + 256);
    p.rec = reinterpret_cast<unsigned long long *>(r8 + 256 + (size_t)K * 32);
    p.K = (uint32_t)K;
    p.n_bursts = (uint32_t)n_bursts;
    p.warps = (uint32_t)warps;
    p.chunks_per_warp = (uint32_t)(B / 16 / warps);
    uint32_t l = 0;
    while ((16u << l) < (uint32_t)row_bytes) ++l;
    p.cpr_log2 = l;
    p.rows_per_burst = (uint32_t)rows_per_burst;
    p.n_slots = (uint32_t)n_slots;
    p.row_stride = (uint64_t)row_stride;
    p.gap_cycles = (uint64_t)llround(gap_ns * mhz / 1e3);
    p.isolated = isolated ? 1 : 0;

    if ((e = cudaMemsetAsync(rec, 0, 256, s)) != cudaSuccess) return (xs_status)fail_cuda("cudaMemsetAsync", e);
    if ((e = cudaFuncSetAttribute(burst_gap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBurstSmem)) !=
        cudaSuccess)
        return (xs_status)fail_cuda("cudaFuncSetAttribute", e);
    void *args[] = {&p};
    e = cudaLaunchCooperativeKernel((const void *)burst_gap_kernel, dim3(K), dim3(32 * warps), args, kBurstSmem, s);
    if (e != cudaSuccess) return (xs_status)fail_cuda("cooperative launch of the burst kernel", e);

    std::vector<unsigned long long> h((size_t)K * 4 + (size_t)K * n_bursts * 2);
    uint32_t hdr[2] = {0, 0};
    if ((e = cudaMemcpyAsync(hdr, rec, sizeof hdr, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(h.data(), r8 + 256, h.size() * 8, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return (xs_status)fail_cuda("reading the burst records", e);
    if (hdr[1]) return (xs_status)fail(XS_ERR_TIMEOUT, "a grid barrier of the burst kernel ran out of time");

    const unsigned long long *clk = h.data(), *r = h.data() + (size_t)K * 4;
    double mhz_run = 0.0;
    for (int k = 0; k < K; ++k)
        mhz_run += 1e3 * (double)(clk[k * 4 + 3] - clk[k * 4 + 1]) / (double)(clk[k * 4 + 2] - clk[k * 4 + 0]);
    mhz_run /= K;
    const int skip = isolated ? 0 : n_bursts / 4;
    double iss_mean = 0.0, iss_max = 0.0, period = 0.0;
    for (int n = skip; n < n_bursts; ++n) {
        double sum = 0.0, mx = 0.0;
        for (int k = 0; k < K; ++k) {
            const double span = (double)(r[((size_t)k * n_bursts + n) * 2 + 1] - r[((size_t)k * n_bursts + n) * 2]);
            sum += span;
            mx = span > mx ? span : mx;
        }
        iss_mean += sum / K;
        iss_max += mx;
    }
    const int nm = n_bursts - skip;
    if (!isolated && nm > 1) {
        for (int k = 0; k < K; ++k)
            period += (double)(r[((size_t)k * n_bursts + n_bursts - 1) * 2] - r[((size_t)k * n_bursts + skip) * 2]) /
                      (nm - 1);
        period /= K;
    }
    const double ns_per_cycle = 1e3 / mhz_run;
    stats->t_iss_mean_ns = iss_mean / nm * ns_per_cycle;
    stats->t_iss_max_ns = iss_max / nm * ns_per_cycle;
    stats->t_period_ns = period * ns_per_cycle;
    stats->sm_clock_mhz = mhz_run;
    stats->bursts_measured = nm;
    return XS_OK;
}

}  // extern "C"
