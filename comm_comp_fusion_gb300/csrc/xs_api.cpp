// xs_api.cpp -- the C ABI declared in include/xs.h: argument checks (done
// before any CUDA call, so they also run on machines without a GPU), per-device
// attributes, TMA tensor maps and kernel launches. No device memory is
// allocated here.
#include "../../include/xs.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "xs_internal.h"

namespace {

thread_local std::string g_last_error;

xs_status fail(xs_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

xs_status fail_cuda(const char *what, cudaError_t e) {
    return fail(XS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int major = 0, minor = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

xs_status current_device(int *dev, DeviceInfo *info) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
    if (*dev < 0 || *dev >= kMaxDevices) return fail(XS_ERR_UNSUPPORTED, "device ordinal %d out of range", *dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &d = g_dev[*dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess)
            return fail_cuda("cudaDeviceGetAttribute", e);
        d.ready = true;
    }
    *info = d;
    if (d.major != 10 || d.minor != 3)
        return fail(XS_ERR_UNSUPPORTED, "kernels are built for sm_103a only; device %d is sm_%d%d", *dev, d.major,
                    d.minor);
    return XS_OK;
}

xs_status check_device_pointer(const void *ptr, int dev, const char *name) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(XS_ERR_UNSUPPORTED, "%s is not a CUDA pointer (%s)", name, cudaGetErrorName(e));
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
        return fail(XS_ERR_UNSUPPORTED, "%s must be device memory", name);
    if (a.type == cudaMemoryTypeDevice && a.device != dev)
        return fail(XS_ERR_UNSUPPORTED, "%s lives on device %d, current device is %d", name, a.device, dev);
    return XS_OK;
}

// Host-buffer calls: the pointer must not be device memory (pinned or
// pageable host memory are both fine).
xs_status check_host_pointer(const void *ptr, const char *name) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(XS_ERR_CUDA, "cudaPointerGetAttributes(%s): %s", name, cudaGetErrorName(e));
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged)
        return fail(XS_ERR_UNSUPPORTED, "%s must be host memory", name);
    return XS_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

// Shape rules shared by every call.
xs_status check_shape(int B, int S, int H, int D, int P, bool attn, size_t *bytes) {
    (void)attn;
    if (B < 0 || S < 0) return fail(XS_ERR_SHAPE, "B and S must be >= 0 (got B=%d S=%d)", B, S);
    if (H < 1 || P < 1) return fail(XS_ERR_SHAPE, "H and P must be >= 1 (got H=%d P=%d)", H, P);
    if (H % P) return fail(XS_ERR_SHAPE, "H=%d is not a multiple of P=%d", H, P);
    if (S % P) return fail(XS_ERR_SHAPE, "S=%d is not a multiple of P=%d", S, P);
    if (D != 64 && D != 96 && D != 128 && D != 256)
        return fail(XS_ERR_UNSUPPORTED, "D=%d is not supported (64, 96, 128 or 256)", D);
    const unsigned long long rows = (unsigned long long)B * S * H;
    if (rows >= (1ull << 31)) return fail(XS_ERR_SHAPE, "B*S*H=%llu rows exceeds 2^31-1", rows);
    *bytes = (size_t)rows * D * 2;
    if (*bytes >= (1ull << 40)) return fail(XS_ERR_SHAPE, "tensor of %zu bytes exceeds 2^40", *bytes);
    return XS_OK;
}

bool misaligned(const void *p) { return ((uintptr_t)p & 15u) != 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

xs_status get_encoder(EncodeTiledFn *fn) {
    static EncodeTiledFn cached = nullptr;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!cached) return fail(XS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (%s)", cudaGetErrorName(err));
    *fn = cached;
    return XS_OK;
}

// Tensor map over a head-partitioned tensor [P*B][S][Hl][D] of bf16 (esize 2)
// or E4M3 bytes (esize 1), box = 128 bytes of columns x 128 tokens of one
// head, 128-byte swizzle (the tcgen05 K-major / MN-major operand layout with
// 128-byte rows).
xs_status make_head_map(CUtensorMap *m, const void *ptr, int B, int S, int H, int D, int P, const char *name,
                        int esize = 2) {
    EncodeTiledFn enc;
    xs_status st = get_encoder(&enc);
    if (st) return st;
    const int Hl = H / P;
    const cuuint64_t e = (cuuint64_t)esize;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hl, (cuuint64_t)S, (cuuint64_t)P * (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * e, (cuuint64_t)Hl * D * e, (cuuint64_t)S * Hl * D * e};
    const cuuint32_t box[4] = {(cuuint32_t)(128 / esize), 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(XS_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
    return XS_OK;
}

// Tensor map over rank r's slice [B][Sl][H][D] of a sequence-partitioned
// tensor [P][B][Sl][H][D], box = 64 columns x `rows` tokens of one head
// (`rows` divides Sl, so a box never crosses into the next rank's slice).
xs_status make_rank_map(CUtensorMap *m, const void *ptr, int r, int B, int S, int H, int D, int P, int rows,
                        const char *name) {
    EncodeTiledFn enc;
    xs_status st = get_encoder(&enc);
    if (st) return st;
    const int Sl = S / P;
    const size_t slice = (size_t)B * Sl * H * D * 2;
    void *base = static_cast<char *>(const_cast<void *>(ptr)) + (size_t)r * slice;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Sl, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)Sl * H * D * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS)
        return fail(XS_ERR_CUDA, "cuTensorMapEncodeTiled(%s, rank %d) failed with CUresult %d", name, r, (int)res);
    return XS_OK;
}

int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Generation stamps of balanced launches (48 bits are used; counting from 1, so
// the zero of fresh memory never matches).
std::atomic<unsigned long long> g_generation{1};
unsigned long long next_generation() { return g_generation.fetch_add(1, std::memory_order_relaxed) & ((1ull << 48) - 1ull); }

// What an attention call does besides the plain head-partitioned one.
struct CallOpts {
    int epi = 0;              // 0: head-partitioned output; 1: All-to-All scatter
    void *ws = nullptr;       // balanced-schedule workspace (NULL: whole-item schedule)
    size_t ws_bytes = 0;
    int layout = 0;           // 1: q, k, v and out sequence-partitioned (epi must be 1)
    void *trace = nullptr;    // epilogue trace buffer
    size_t trace_bytes = 0;
    bool causal = false;
    int f8 = 0;               // 1: q and k hold E4M3 bytes; 2: q, k and v do (D = 128, layout 0)
    // host buffers: copy in, compute and copy out pipelined over rank chunks
    // (q, k, v, out are then the device staging buffers)
    const void *hq = nullptr, *hk = nullptr, *hv = nullptr;
    void *hout = nullptr;
};

// Internal streams and events of the host-buffer pipeline, one set per device,
// created on first use. The mutex keeps one call's enqueue sequence whole.
constexpr int kMaxChunks = 16;
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, in[kMaxChunks] = {}, comp[kMaxChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

xs_status pipe_init(HostPipe &hp) {
    if (hp.ready) return XS_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming);
    for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c) {
        e = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.comp[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return fail_cuda("creating the host pipeline's streams and events", e);
    hp.ready = true;
    return XS_OK;
}

cudaError_t launch_any(const CallOpts &o, int D, const xs::OperandMaps<1> &maps, const xs::AttnParams &p, int grid,
                       cudaStream_t s) {
    if (o.causal) return xs::launch_causal(D, maps, p, grid, s);
    if (o.f8) return xs::launch_attention_f8_d128(o.f8, maps, p, grid, s);
    return xs::launch_attention(D, maps, p, grid, s);
}

// The host-buffer call: the (rank, batch) slices are split into up to kMaxChunks
// chunks. Chunk c's q, k, v slices (contiguous in the head-partitioned layout) are copied in on
// the pipeline's h2d stream; the caller's stream waits for them and runs the
// attention kernel over that chunk's work items only; the d2h stream then
// copies the chunk's output out: the columns of its heads in the rows of its
// batches of the sequence-partitioned output (one 2-D copy when the chunk holds
// whole ranks, one per slice and destination rank otherwise), or its contiguous
// part of the head-partitioned one. Copies of later chunks overlap the compute
// of earlier ones. The caller's stream finally waits for the last copy out.
xs_status host_pipeline(const CallOpts &o, const void *q, const void *k, const void *v, void *out, size_t qk_bytes,
                        size_t v_bytes, size_t bytes, int D, xs::AttnParams p, const xs::OperandMaps<1> &maps,
                        const DeviceInfo &info, int dev, cudaStream_t s) {
    HostPipe &hp = g_pipe[dev];
    std::lock_guard<std::mutex> lk(hp.mu);
    xs_status st = pipe_init(hp);
    if (st) return st;
    // Chunks over the call's units, one head of one (rank, batch) slice each, in
    // work-item order: a chunk's items are one contiguous range, and its rows are
    // whole slices (contiguous) and at most two partial slices (the same heads of
    // every row: one strided copy each).
    const int P = p.P, n_rb = P * p.B, Hl = p.Hl, units = n_rb * Hl, per_unit = p.n_items / units;
    int bounds[kMaxChunks + 1];
    const int chunks = xs::host_chunk_plan(units, (long long)((2 * qk_bytes + v_bytes) / units), 8ll << 20,
                                           kMaxChunks, bounds);
    const size_t q_rb = qk_bytes / n_rb, v_rb = v_bytes / n_rb, o_rb = bytes / n_rb;
    const size_t head_row = (size_t)D * 2, pitch = (size_t)p.H * head_row;
    const char *hq = static_cast<const char *>(o.hq), *hk = static_cast<const char *>(o.hk);
    const char *hv = static_cast<const char *>(o.hv);
    char *hout = static_cast<char *>(o.hout);
    const char *dq = static_cast<const char *>(q), *dk = static_cast<const char *>(k);
    const char *dv = static_cast<const char *>(v);
    char *dout = static_cast<char *>(out);
    // units [u0, u1) of a head-partitioned tensor ([P*B][S][Hl][*], `slice` bytes
    // per slice) from src to dst
    auto copy_units = [&](char *dst, const char *src, size_t slice, int u0, int u1, cudaMemcpyKind kind,
                          cudaStream_t st) -> cudaError_t {
        const size_t row = slice / (size_t)p.S, head = row / (size_t)Hl;
        cudaError_t err = cudaSuccess;
        for (int u = u0; u < u1 && err == cudaSuccess;) {
            const int sb = u / Hl, ha = u % Hl;
            if (ha == 0 && u + Hl <= u1) {  // whole slices [sb, sb1)
                int sb1 = sb + 1;
                while ((sb1 + 1) * Hl <= u1) ++sb1;
                err = cudaMemcpyAsync(dst + sb * slice, src + sb * slice, (size_t)(sb1 - sb) * slice, kind, st);
                u = sb1 * Hl;
            } else {  // heads [ha, hb) of every row of slice sb
                const int hb = ha + (u1 - u < Hl - ha ? u1 - u : Hl - ha);
                const size_t off = sb * slice + (size_t)ha * head;
                err = cudaMemcpy2DAsync(dst + off, row, src + off, row, (size_t)(hb - ha) * head, (size_t)p.S, kind, st);
                u += hb - ha;
            }
        }
        return err;
    };
    cudaError_t e = cudaEventRecord(hp.start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.h2d, hp.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.d2h, hp.start, 0);
    for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
        const int u0 = bounds[c], u1 = bounds[c + 1];
        e = copy_units((char *)dq, hq, q_rb, u0, u1, cudaMemcpyHostToDevice, hp.h2d);
        if (e == cudaSuccess) e = copy_units((char *)dk, hk, q_rb, u0, u1, cudaMemcpyHostToDevice, hp.h2d);
        if (e == cudaSuccess) e = copy_units((char *)dv, hv, v_rb, u0, u1, cudaMemcpyHostToDevice, hp.h2d);
        if (e == cudaSuccess) e = cudaEventRecord(hp.in[c], hp.h2d);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.in[c], 0);
        if (e != cudaSuccess) break;
        xs::AttnParams pc = p;
        pc.item0 = u0 * per_unit;
        pc.n_items = (u1 - u0) * per_unit;
        if (pc.ws_rec) pc.gen = next_generation();
        const int grid = xs::attn_schedule(pc, info.num_sms, pc.ws_rec != nullptr && !o.causal);
        e = launch_any(o, D, maps, pc, grid, s);
        if (e == cudaSuccess) e = cudaEventRecord(hp.comp[c], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.d2h, hp.comp[c], 0);
        if (e != cudaSuccess) break;
        if (!o.epi) {
            e = copy_units(hout, dout, o_rb, u0, u1, cudaMemcpyDeviceToHost, hp.d2h);
        } else if (u0 % (p.B * Hl) == 0 && u1 % (p.B * Hl) == 0) {
            // whole ranks: the columns of their heads in every row of the output
            const size_t col = (size_t)(u0 / Hl / p.B) * Hl * head_row;
            e = cudaMemcpy2DAsync(hout + col, pitch, dout + col, pitch, (size_t)((u1 - u0) / Hl / p.B) * Hl * head_row,
                                  (size_t)P * p.B * p.Sl, cudaMemcpyDeviceToHost, hp.d2h);
        } else {
            // heads [ha, hb) of slice (r, b): rank r's columns of those heads in the Sl
            // rows of batch b of each destination rank
            for (int u = u0; u < u1 && e == cudaSuccess;) {
                const int sb = u / Hl, ha = u % Hl, hb = ha + (u1 - u < Hl - ha ? u1 - u : Hl - ha);
                const int r = sb / p.B, b = sb % p.B;
                for (int rd = 0; rd < P && e == cudaSuccess; ++rd) {
                    const size_t off = ((size_t)(rd * p.B + b) * p.Sl) * pitch + ((size_t)r * Hl + ha) * head_row;
                    e = cudaMemcpy2DAsync(hout + off, pitch, dout + off, pitch, (size_t)(hb - ha) * head_row,
                                          (size_t)p.Sl, cudaMemcpyDeviceToHost, hp.d2h);
                }
                u += hb - ha;
            }
        }
    }
    if (e == cudaSuccess) e = cudaEventRecord(hp.done, hp.d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.done, 0);
    if (e != cudaSuccess) return fail_cuda("host-buffer pipeline", e);
    return XS_OK;
}

// layout 0: q, k, v head-partitioned, out as `epi` says. layout 1: q, k, v and
// out sequence-partitioned (both All-to-Alls fused; `epi` must be 1).
xs_status attention_call(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                         float scale, void *stream, const CallOpts &o) {
    const int epi = o.epi, layout = o.layout;
    void *const ws = o.ws, *const trace = o.trace;
    const size_t ws_bytes = o.ws_bytes, trace_bytes = o.trace_bytes;
    const bool causal = o.causal;
    if (!q || !k || !v || !out) return fail(XS_ERR_NULL, "q, k, v and out must be non-NULL");
    const bool host = o.hq || o.hk || o.hv || o.hout;
    if (host && (!o.hq || !o.hk || !o.hv || !o.hout))
        return fail(XS_ERR_NULL, "host q, k, v and out must all be non-NULL");
    size_t bytes = 0;
    xs_status st = check_shape(B, S, H, D, P, true, &bytes);
    if (st) return st;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(XS_ERR_SHAPE, "scale must be positive and finite");
    if (o.f8 && D != 128) return fail(XS_ERR_UNSUPPORTED, "E4M3 inputs are built for D=128 only (got D=%d)", D);
    const size_t qk_bytes = o.f8 ? bytes / 2 : bytes, v_bytes = o.f8 == 2 ? bytes / 2 : bytes;
    if (trace) {
        if (D != 128) return fail(XS_ERR_UNSUPPORTED, "epilogue tracing is built for D=128 only (got D=%d)", D);
        if (S % 128) return fail(XS_ERR_UNSUPPORTED, "epilogue tracing needs S a multiple of 128 (got S=%d)", S);
        if (misaligned(trace)) return fail(XS_ERR_ALIGN, "trace must be 16-byte aligned");
    }
    if (layout == 1) {
        if (P > xs::kMaxRanks) return fail(XS_ERR_UNSUPPORTED, "P=%d exceeds the %d ranks supported", P, xs::kMaxRanks);
        if ((S / P) % 8) return fail(XS_ERR_UNSUPPORTED, "S/P=%d tokens per rank is not a multiple of 8", S / P);
    }
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out))
        return fail(XS_ERR_ALIGN, "q, k, v and out must be 16-byte aligned");
    if (overlaps(out, bytes, q, qk_bytes) || overlaps(out, bytes, k, qk_bytes) || overlaps(out, bytes, v, v_bytes))
        return fail(XS_ERR_ALIAS, "out overlaps q, k or v");
    if (!ws && ws_bytes) return fail(XS_ERR_WORKSPACE, "workspace is NULL but workspace_bytes is %zu", ws_bytes);
    if (ws) {
        if (((uintptr_t)ws & 255u) != 0) return fail(XS_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        if (overlaps(ws, ws_bytes, q, qk_bytes) || overlaps(ws, ws_bytes, k, qk_bytes) || overlaps(ws, ws_bytes, v, v_bytes) ||
            overlaps(ws, ws_bytes, out, bytes))
            return fail(XS_ERR_WORKSPACE, "workspace overlaps q, k, v or out");
    }
    if (host) {
        if (layout || trace) return fail(XS_ERR_UNSUPPORTED, "host buffers take head-partitioned inputs, untraced");
        const void *hs[4] = {o.hq, o.hk, o.hv, o.hout};
        const size_t hb[4] = {qk_bytes, qk_bytes, v_bytes, bytes};
        const void *ds[4] = {q, k, v, out};
        for (int i = 0; i < 4; ++i)
            for (int j = 0; j < 4; ++j)
                if (overlaps(hs[i], hb[i], ds[j], hb[j]))
                    return fail(XS_ERR_ALIAS, "a host buffer overlaps a device buffer");
        if (overlaps(o.hout, bytes, o.hq, qk_bytes) || overlaps(o.hout, bytes, o.hk, qk_bytes) ||
            overlaps(o.hout, bytes, o.hv, v_bytes))
            return fail(XS_ERR_ALIAS, "host out overlaps host q, k or v");
    }
    if (bytes == 0) return XS_OK;

    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev, &info))) return st;
    if ((st = check_device_pointer(q, dev, "q")) || (st = check_device_pointer(k, dev, "k")) ||
        (st = check_device_pointer(v, dev, "v")) || (st = check_device_pointer(out, dev, "out")))
        return st;
    if (host && ((st = check_host_pointer(o.hq, "q_host")) || (st = check_host_pointer(o.hk, "k_host")) ||
                 (st = check_host_pointer(o.hv, "v_host")) || (st = check_host_pointer(o.hout, "out_host"))))
        return st;

    xs::AttnParams p;
    p.ld_rows = gcd_int(S / P, 128);
    xs::OperandMaps<1> head_maps;
    xs::OperandMaps<xs::kSeqMaps> rank_maps;
    if (layout == 0) {
        if ((st = make_head_map(&head_maps.q[0], q, B, S, H, D, P, "q", o.f8 ? 1 : 2)) ||
            (st = make_head_map(&head_maps.k[0], k, B, S, H, D, P, "k", o.f8 ? 1 : 2)) ||
            (st = make_head_map(&head_maps.v[0], v, B, S, H, D, P, "v", o.f8 == 2 ? 1 : 2)))
            return st;
    } else {
        memset(&rank_maps, 0, sizeof rank_maps);
        // entries r: boxes of ld_rows rows; entries kMaxRanks + r: 128-row boxes
        // for tiles inside one rank's slice (none when Sl < 128)
        for (int r = 0; r < P; ++r)
            for (int big = 0; big < (S / P >= 128 ? 2 : 1); ++big) {
                const int e = big * xs::kMaxRanks + r, rows = big ? 128 : p.ld_rows;
                if ((st = make_rank_map(&rank_maps.q[e], q, r, B, S, H, D, P, rows, "q")) ||
                    (st = make_rank_map(&rank_maps.k[e], k, r, B, S, H, D, P, rows, "k")) ||
                    (st = make_rank_map(&rank_maps.v[e], v, r, B, S, H, D, P, rows, "v")))
                    return st;
            }
    }
    p.B = B;
    p.S = S;
    p.H = H;
    p.P = P;
    p.Hl = H / P;
    p.Sl = S / P;
    p.n_qt = (S + 127) / 128;
    p.n_pairs = (p.n_qt + 1) / 2;
    p.n_kv = (S + 127) / 128;
    p.kv_tail = S - (p.n_kv - 1) * 128;
    const long long items = (long long)P * B * p.Hl * (xs::single_tile_items(D) ? p.n_qt : p.n_pairs);
    if (items >= (1ll << 31)) return fail(XS_ERR_SHAPE, "too many work items (%lld)", items);
    p.n_items = (int)items;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634073599246810019);
    p.out = static_cast<uint16_t *>(out);
    p.head_out = epi ? 0 : 1;
    p.ws_rec = nullptr;
    p.ws_cnt = nullptr;
    p.gen = 0;
    p.trace = static_cast<unsigned long long *>(trace);
    if (ws) {
        const size_t need = xs::attn_workspace_bytes(p.n_items, p.n_kv, D, info.num_sms);
        if (ws_bytes < need)
            return fail(XS_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
        if ((st = check_device_pointer(ws, dev, "workspace"))) return st;
        const size_t rec = ((size_t)2 * info.num_sms * xs::partial_record_bytes(D) + 255) & ~(size_t)255;
        p.ws_rec = static_cast<float *>(ws);
        p.ws_cnt = reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + rec);
        p.gen = next_generation();
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (host) return host_pipeline(o, q, k, v, out, qk_bytes, v_bytes, bytes, D, p, head_maps, info, dev, s);
    const int grid = xs::attn_schedule(p, info.num_sms, ws != nullptr && !causal);
    if (causal) {
        cudaError_t e = launch_any(o, D, head_maps, p, grid, s);
        if (e != cudaSuccess) return fail_cuda("causal attention launch", e);
        return XS_OK;
    }
    if (trace) {
        const size_t need = ((size_t)grid * p.n_dp * 8 + (size_t)grid * 4) * xs::kTraceWords * 8 + 2 * 2 * 64 * 4 * 8;
        if (trace_bytes < need)
            return fail(XS_ERR_SHAPE, "trace buffer of %zu bytes is smaller than the %zu bytes needed", trace_bytes,
                        need);
        if ((st = check_device_pointer(trace, dev, "trace"))) return st;
        cudaError_t e = cudaMemsetAsync(trace, 0, need, s);
        if (e == cudaSuccess) e = xs::launch_attention_traced(D, head_maps, p, grid, s);
        if (e != cudaSuccess) return fail_cuda("traced attention launch", e);
        return XS_OK;
    }
    cudaError_t e = layout == 0 ? launch_any(o, D, head_maps, p, grid, s) : xs::launch_ulysses(D, rank_maps, p, grid, s);
    if (e != cudaSuccess) return fail_cuda("attention launch", e);
    return XS_OK;
}

}  // namespace

namespace xs {
// Records `message` as this thread's last error and returns `status`; for the
// other translation units of the library.
int report_error(int status, const char *message) { return (int)fail((xs_status)status, "%s", message); }
}  // namespace xs

extern "C" {

xs_status xs_attn_a2a(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                      float scale, void *stream) {
    CallOpts o;
    o.epi = 1;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                  float scale, void *stream) {
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, CallOpts());
}

xs_status xs_attn_a2a_ws(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                         float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.epi = 1;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_ws(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                     float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_ulysses_attn(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                          float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.epi = 1;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.layout = 1;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_causal_a2a(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                             int P, float scale, void *stream) {
    CallOpts o;
    o.epi = 1;
    o.causal = true;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_causal(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D, int P,
                         float scale, void *stream) {
    CallOpts o;
    o.causal = true;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_a2a_q8(const void *q8, const void *k8, const void *v, void *out, int B, int S, int H, int D, int P,
                         float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.epi = 1;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.f8 = 1;
    return attention_call(q8, k8, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_q8(const void *q8, const void *k8, const void *v, void *out, int B, int S, int H, int D, int P,
                     float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.f8 = 1;
    return attention_call(q8, k8, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_a2a_qkv8(const void *q8, const void *k8, const void *v8, void *out, int B, int S, int H, int D,
                           int P, float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.epi = 1;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.f8 = 2;
    return attention_call(q8, k8, v8, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_qkv8(const void *q8, const void *k8, const void *v8, void *out, int B, int S, int H, int D, int P,
                       float scale, void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.f8 = 2;
    return attention_call(q8, k8, v8, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_a2a_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, void *q,
                           void *k, void *v, void *out, int B, int S, int H, int D, int P, float scale,
                           void *workspace, size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.epi = 1;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.hq = q_host;
    o.hk = k_host;
    o.hv = v_host;
    o.hout = out_host;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, void *q, void *k,
                       void *v, void *out, int B, int S, int H, int D, int P, float scale, void *workspace,
                       size_t workspace_bytes, void *stream) {
    CallOpts o;
    o.ws = workspace;
    o.ws_bytes = workspace_bytes;
    o.hq = q_host;
    o.hk = k_host;
    o.hv = v_host;
    o.hout = out_host;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_a2a_trace(const void *q, const void *k, const void *v, void *out, int B, int S, int H, int D,
                            int P, float scale, void *trace, size_t trace_bytes, void *stream) {
    if (!trace) return fail(XS_ERR_NULL, "trace must be non-NULL");
    CallOpts o;
    o.epi = 1;
    o.trace = trace;
    o.trace_bytes = trace_bytes;
    return attention_call(q, k, v, out, B, S, H, D, P, scale, stream, o);
}

xs_status xs_attn_trace_layout(int B, int S, int H, int D, int P, int *ctas, int *items_per_cta, size_t *bytes) {
    if (!ctas || !items_per_cta || !bytes) return fail(XS_ERR_NULL, "ctas, items_per_cta and bytes must be non-NULL");
    size_t tb = 0;
    xs_status st = check_shape(B, S, H, D, P, true, &tb);
    if (st) return st;
    if (tb == 0) {
        *ctas = *items_per_cta = 0;
        *bytes = 0;
        return XS_OK;
    }
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev, &info))) return st;
    xs::AttnParams p;
    p.n_qt = (S + 127) / 128;
    p.n_pairs = (p.n_qt + 1) / 2;
    p.n_kv = (S + 127) / 128;
    p.n_items = P * B * (H / P) * p.n_pairs;
    const int grid = xs::attn_schedule(p, info.num_sms, false);
    *ctas = grid;
    *items_per_cta = p.n_dp;
    *bytes = ((size_t)grid * p.n_dp * 8 + (size_t)grid * 4) * xs::kTraceWords * 8 + 2 * 2 * 64 * 4 * 8;
    return XS_OK;
}

xs_status xs_attn_workspace_size(int B, int S, int H, int D, int P, size_t *bytes) {
    if (!bytes) return fail(XS_ERR_NULL, "bytes must be non-NULL");
    size_t tb = 0;
    xs_status st = check_shape(B, S, H, D, P, true, &tb);
    if (st) return st;
    if (tb == 0) {
        *bytes = 0;
        return XS_OK;
    }
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev, &info))) return st;
    const int n_qt = (S + 127) / 128;
    const long long n_items = (long long)P * B * (H / P) * (xs::single_tile_items(D) ? n_qt : (n_qt + 1) / 2);
    *bytes = xs::attn_workspace_bytes((int)n_items, n_qt, D, info.num_sms);
    return XS_OK;
}

}  // extern "C"

namespace {

xs_status permute_call(const void *in, void *out, int B, int S, int H, int D, int P, void *stream, bool inverse) {
    if (!in || !out) return fail(XS_ERR_NULL, "in and out must be non-NULL");
    size_t bytes = 0;
    xs_status st = check_shape(B, S, H, D, P, false, &bytes);
    if (st) return st;
    if (misaligned(in) || misaligned(out)) return fail(XS_ERR_ALIGN, "in and out must be 16-byte aligned");
    if (overlaps(in, bytes, out, bytes)) return fail(XS_ERR_ALIAS, "in and out overlap");
    if (bytes == 0) return XS_OK;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev, &info))) return st;
    if ((st = check_device_pointer(in, dev, "in")) || (st = check_device_pointer(out, dev, "out"))) return st;

    xs::PermParams p;
    p.rows = (uint32_t)((unsigned long long)B * S * H);
    p.cpr = (uint32_t)(D / 8);
    p.cpr_log2 = D == 256 ? 5u : D == 128 ? 4u : 3u;
    xs::fastdiv_magic(p.cpr, &p.mC, &p.sC);
    if (D == 96 && (unsigned long long)p.rows * p.cpr >= (1ull << 31))
        return fail(XS_ERR_SHAPE, "a D=96 permute handles at most 2^31 16-byte chunks (tensor below 32 GiB)");
    p.B = (uint32_t)B;
    p.S = (uint32_t)S;
    p.H = (uint32_t)H;
    p.Hl = (uint32_t)(H / P);
    p.Sl = (uint32_t)(S / P);
    xs::fastdiv_magic(p.H, &p.mH, &p.sH);
    xs::fastdiv_magic(p.Sl, &p.mSl, &p.sSl);
    xs::fastdiv_magic(p.B, &p.mB, &p.sB);
    xs::fastdiv_magic(p.Hl, &p.mHl, &p.sHl);
    xs::fastdiv_magic(p.S, &p.mS, &p.sS);
    cudaError_t e = xs::launch_permute(in, out, p, inverse, info.num_sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda("permute launch", e);
    return XS_OK;
}

}  // namespace

extern "C" {

xs_status xs_a2a_permute(const void *in, void *out, int B, int S, int H, int D, int P, void *stream) {
    return permute_call(in, out, B, S, H, D, P, stream, false);
}

xs_status xs_a2a_permute_inverse(const void *in, void *out, int B, int S, int H, int D, int P, void *stream) {
    return permute_call(in, out, B, S, H, D, P, stream, true);
}

const char *xs_last_error(void) { return g_last_error.c_str(); }

xs_status xs_device_status(void *stream, int clear) {
    unsigned int word = 0;
    cudaError_t e = xs::read_device_error(&word, clear != 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda("reading the device error word", e);
    if (word) return fail(XS_ERR_TIMEOUT, "a bounded in-kernel wait ran out (device error word 0x%08x)", word);
    return XS_OK;
}

xs_status xs_selftest_wait_timeout(unsigned int timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 2000000u) return fail(XS_ERR_SHAPE, "timeout_us must be in 1..2000000");
    int dev;
    DeviceInfo info;
    xs_status st = current_device(&dev, &info);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = xs::launch_wait_selftest(1000ull * timeout_us, s);
    if (e != cudaSuccess) return fail_cuda("self-test launch", e);
    unsigned int word = 0;
    e = xs::read_device_error(&word, true, s);
    if (e != cudaSuccess) return fail_cuda("reading the device error word", e);
    if (word & 0x80000000u) return fail(XS_ERR_TIMEOUT, "self-test wait ran out as designed (word 0x%08x)", word);
    return XS_OK;
}

int xs_version(void) { return 100; }

}  // extern "C"
