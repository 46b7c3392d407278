// Status strings, launch planning and the Philox entry point.
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>
#include <vector>

#include "fs_host.h"

namespace fsd {

static thread_local char g_last_error[256] = "";

void set_last_error(const char* msg) { std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

fs_status cuda_fail(cudaError_t e) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return FS_ERR_CUDA;
}

fs_status device_limits(int& sm_count, size_t& smem_optin) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static std::mutex mu;
    static int cached_sm[64] = {0};
    static size_t cached_smem[64] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return FS_ERR_UNSUPPORTED;
    if (cached_sm[dev] == 0) {
        int v = 0;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        int s = 0;
        e = cudaDeviceGetAttribute(&s, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        cached_sm[dev] = v;
        cached_smem[dev] = size_t(s);
    }
    sm_count = cached_sm[dev];
    smem_optin = cached_smem[dev];
    return FS_OK;
}

fs_status prepare_kernel(const void* fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({fn, dev})) return FS_OK;
    size_t optin = 0;
    int sms = 0;
    fs_status st = device_limits(sms, optin);
    if (st != FS_OK) return st;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(optin));
    if (e != cudaSuccess) return cuda_fail(e);
    // Clusters of up to 16 CTAs (more than the portable 8) where the device has them;
    // make_plan only picks sizes the occupancy query says fit.
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e);
    done.insert({fn, dev});
    return FS_OK;
}

// How many clusters of C CTAs of `fn` (with `smem` bytes of dynamic shared memory)
// can be resident at once on the current device (cached).  This accounts for the
// placement of a cluster inside one GPC, which a per-SM occupancy count does not.
static fs_status active_clusters(const void* fn, size_t smem, int C, int& n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, size_t, int>, int> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find({fn, dev, smem, C});
        if (it != cache.end()) {
            n = it->second;
            return FS_OK;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(C), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int v = 0;
    e = cudaOccupancyMaxActiveClusters(&v, fn, &cfg);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(mu);
    cache[{fn, dev, smem, C}] = v;
    n = v;
    return FS_OK;
}

// Shared memory of one SM and the per-CTA reservation (cached per device).
static fs_status smem_per_sm(int& per_sm, int& reserved) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static std::mutex mu;
    static std::map<int, std::pair<int, int>> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it == cache.end()) {
        int a = 0, b = 0;
        e = cudaDeviceGetAttribute(&a, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaDeviceGetAttribute(&b, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        it = cache.insert({dev, {a, b}}).first;
    }
    per_sm = it->second.first;
    reserved = it->second.second;
    return FS_OK;
}

// The launch plan of `fn` for `rows` rows of `vocab` values.  The row-wide tables fix
// the shared memory a CTA needs.
//
// Kernels that stream the row about once (`single_pass`: the top-k-first samplers,
// sampling without filters, the top-k renormaliser and the logit mask) follow
// measurements of the top-k-first sampler on GB300 over 8..192 rows of 32000 to
// 256000 values: the fastest plans keep about 2.5 CTAs per SM (C near 2.5 x SMs /
// rows) with at most 3 CTAs per SM (a cap below the occupancy limit is enforced by
// asking for more shared memory than a 4th CTA leaves room for: with 4 per SM
// allowed, the block scheduler stacks 4 on some SMs and those SMs set the pass
// time), and clusters above 12 CTAs only pay off for 4 rows or fewer.  So C starts
// at ceil(2.5 x SMs / rows), capped at 12 (16 up to 4 rows), and steps down until
// all clusters are resident at once (one wave) at 3 per SM, else at the occupancy
// limit.
//
// Kernels that pass over the row several times with the whole cluster (rejection
// rounds of the joint order, top-p threshold searches) gain more from CTAs per row
// than from balance: the largest C (at most 16) whose clusters are all resident at
// the occupancy limit.
//
// C = 1 at the occupancy limit when no cluster size fits in one wave.  Plans are
// cached per (kernel, device, rows, vocab, kind).
fs_status make_plan(int rows, int vocab, const void* fn, bool single_pass, Plan& p, bool topp_hist) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int, int, bool>, Plan> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find({fn, dev, rows, vocab, single_pass});
        if (it != cache.end()) {
            p = it->second;
            return FS_OK;
        }
    }
    int sms = 0;
    size_t optin = 0;
    fs_status st = device_limits(sms, optin);
    if (st != FS_OK) return st;
    st = prepare_kernel(fn);
    if (st != FS_OK) return st;
    p.shift = seg_shift_for(vocab);
    p.ns = (vocab + (BLK << p.shift) - 1) / (BLK << p.shift);
    // row-wide tables in every CTA (and the top-p histograms of that filter)
    const size_t need = topp_hist ? Layout(p.ns).topp_total() : Layout(p.ns).total();
    if (need > optin) return FS_ERR_UNSUPPORTED;
    int per_sm = 0, reserved = 0;
    st = smem_per_sm(per_sm, reserved);
    if (st != FS_OK) return st;
    int natural = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&natural, fn, NT, need);
    if (e != cudaSuccess) return cuda_fail(e);
    int cmax = p.ns / 4;   // >= 4 segments per CTA
    if (cmax > MAX_CLUSTER) cmax = MAX_CLUSTER;
    auto nsc_of = [&](int C) { return ((p.ns + C - 1) / C + 3) & ~3; };   // a multiple of 4
    p.C = 1;
    p.smem = need;
    if (single_pass) {
        if (rows > 4 && cmax > 12) cmax = 12;
        int c0 = int((5L * sms + 2L * rows - 1) / (2L * rows));   // ceil(2.5 x SMs / rows)
        if (c0 > cmax) c0 = cmax;
        // The smallest request (a multiple of 16 bytes) that leaves no room for a 4th CTA.
        const size_t smem3 = std::max(need, (size_t(per_sm / 4 - reserved) + 16) & ~size_t(15));
        const bool cap3 = natural > 3 && smem3 <= optin;
        bool done = false;
        for (int C = c0; C >= 2 && !done; --C) {
            for (int pass = cap3 ? 0 : 1; pass < 2 && !done; ++pass) {
                const size_t smem = pass == 0 ? smem3 : need;
                int n = 0;
                st = active_clusters(fn, smem, C, n);
                if (st != FS_OK) return st;
                if (rows <= n) {
                    p.C = C;
                    p.smem = smem;
                    done = true;
                }
            }
        }
    } else {
        for (int C = cmax; C >= 2; --C) {
            int n = 0;
            st = active_clusters(fn, need, C, n);
            if (st != FS_OK) return st;
            if (rows <= n) {
                p.C = C;
                break;
            }
        }
    }
    p.nsc = nsc_of(p.C);
    p.per_sm = p.C == 1 ? natural : int(per_sm / (p.smem + reserved));
    if (p.per_sm > natural) p.per_sm = natural;
    std::lock_guard<std::mutex> lock(mu);
    cache[{fn, dev, rows, vocab, single_pass}] = p;
    return FS_OK;
}

// Scratch memory of the library, one buffer per (device, stream): calls on one stream
// run in order, so they can share it; calls on different streams get different
// buffers.  Allocated on first need and grown (to the next MiB) when a call needs
// more; a grown-out buffer may still be read by work in flight, so it is kept until
// fs_release_workspaces.  cudaMalloc runs in relaxed capture mode, so the first call
// on a stream may come while that stream is being captured into a CUDA graph (the
// buffer is allocated at capture time, outside the graph, and the graph's kernels
// use it on every replay).
struct WsEntry {
    void* ptr = nullptr;
    size_t bytes = 0;
};
static std::mutex g_ws_mu;
static std::map<std::pair<int, void*>, WsEntry> g_ws;
static std::vector<std::pair<int, void*>> g_ws_retired;

fs_status workspace(size_t bytes, void* stream, void** out) {
    *out = nullptr;
    if (bytes == 0) return FS_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_ws_mu);
    WsEntry& w = g_ws[{dev, stream}];
    if (w.bytes < bytes) {
        const size_t mib = size_t(1) << 20;
        const size_t want = (bytes + mib - 1) / mib * mib;
        cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
        e = cudaThreadExchangeStreamCaptureMode(&mode);
        if (e != cudaSuccess) return cuda_fail(e);
        void* p = nullptr;
        const cudaError_t ea = cudaMalloc(&p, want);
        e = cudaThreadExchangeStreamCaptureMode(&mode);
        if (ea != cudaSuccess) return cuda_fail(ea);
        if (e != cudaSuccess) return cuda_fail(e);
        // A new buffer starts at zero: the scan's claim counters must be zero at launch
        // (each finishing launch sets them back to zero afterwards).
        e = cudaMemsetAsync(p, 0, want, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            cudaFree(p);
            return cuda_fail(e);
        }
        if (w.ptr) g_ws_retired.push_back({dev, w.ptr});
        w.ptr = p;
        w.bytes = want;
    }
    *out = w.ptr;
    return FS_OK;
}

__global__ void philox_kernel(const uint32_t* __restrict__ ctr, const uint32_t* __restrict__ key, int64_t n,
                              uint32_t* __restrict__ out) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
    const uint2 k = make_uint2(key[2 * i], key[2 * i + 1]);
    const uint4 o = philox4x32_10(c, k);
    out[4 * i] = o.x;
    out[4 * i + 1] = o.y;
    out[4 * i + 2] = o.z;
    out[4 * i + 3] = o.w;
}

}  // namespace fsd

extern "C" {

fs_status fs_philox4x32_10(const uint32_t* ctr, const uint32_t* key, int64_t n, uint32_t* out, void* stream) {
    if (n < 0) return FS_ERR_INVALID_ARG;
    if (n == 0) return FS_OK;
    if (!ctr || !key || !out) return FS_ERR_INVALID_ARG;
    const int64_t threads = 256;
    const int64_t blocks = (n + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return FS_ERR_UNSUPPORTED;
    fsd::philox_kernel<<<unsigned(blocks), unsigned(threads), 0, static_cast<cudaStream_t>(stream)>>>(ctr, key, n,
                                                                                                      out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fsd::cuda_fail(e);
    return FS_OK;
}

const char* fs_status_string(int32_t status) {
    switch (status) {
        case FS_OK: return "FS_OK";
        case FS_ERR_INVALID_ARG: return "FS_ERR_INVALID_ARG: a required pointer is NULL or a size/enum is out of range";
        case FS_ERR_UNSUPPORTED: return "FS_ERR_UNSUPPORTED: vocab or launch size beyond what this build supports";
        case FS_ERR_CUDA: return "FS_ERR_CUDA: a CUDA call failed (see fs_last_error_string)";
        default: return "unknown fs_status";
    }
}

const char* fs_last_error_string(void) { return fsd::g_last_error; }

fs_status fs_workspace_bytes(int32_t batch_in, int32_t vocab, size_t* bytes) {
    if (!bytes || batch_in < 0 || vocab < 1) return FS_ERR_INVALID_ARG;
    if (vocab > FS_MAX_VOCAB) return FS_ERR_UNSUPPORTED;
    *bytes = fsd::scan_workspace_bytes(batch_in, vocab, true);
    return FS_OK;
}

fs_status fs_workspace_reserve(int32_t batch_in, int32_t vocab, void* stream) {
    size_t bytes = 0;
    const fs_status st = fs_workspace_bytes(batch_in, vocab, &bytes);
    if (st != FS_OK) return st;
    void* p = nullptr;
    return fsd::workspace(bytes, stream, &p);
}

fs_status fs_release_workspaces(void) {
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return fsd::cuda_fail(e);
    std::lock_guard<std::mutex> lock(fsd::g_ws_mu);
    std::vector<std::pair<int, void*>> all = fsd::g_ws_retired;
    for (auto& kv : fsd::g_ws) all.push_back({kv.first.first, kv.second.ptr});
    fs_status st = FS_OK;
    for (auto& d : all) {
        if (!d.second) continue;
        e = cudaSetDevice(d.first);
        if (e == cudaSuccess) e = cudaFree(d.second);
        if (e != cudaSuccess && st == FS_OK) st = fsd::cuda_fail(e);
    }
    fsd::g_ws.clear();
    fsd::g_ws_retired.clear();
    e = cudaSetDevice(cur);
    if (e != cudaSuccess && st == FS_OK) st = fsd::cuda_fail(e);
    return st;
}

int32_t fs_max_vocab(void) { return FS_MAX_VOCAB; }

}  // extern "C"
