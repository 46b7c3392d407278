// Status strings, launch planning and the Philox entry point.
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "fs_host.h"

namespace fsd {

static thread_local char g_last_error[256] = "";

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

fs_status make_plan(int rows, int vocab, const void* fn, Plan& p) {
    int sms = 0;
    size_t optin = 0;
    fs_status st = device_limits(sms, optin);
    if (st != FS_OK) return st;
    st = prepare_kernel(fn);
    if (st != FS_OK) return st;
    p.shift = seg_shift_for(vocab);
    p.ns = (vocab + (BLK << p.shift) - 1) / (BLK << p.shift);
    p.smem = Layout(p.ns).total();   // row-wide tables in every CTA
    if (p.smem > optin) return FS_ERR_UNSUPPORTED;
    // Largest C (<= MAX_CLUSTER, >= 4 segments per CTA) whose clusters are all
    // resident at once (one wave); C = 1 when none is.
    int cmax = p.ns / 4;
    if (cmax > MAX_CLUSTER) cmax = MAX_CLUSTER;
    if (cmax < 1) cmax = 1;
    int chosen = 1;
    for (int C = cmax; C >= 2; --C) {
        int n = 0;
        st = active_clusters(fn, p.smem, C, n);
        if (st != FS_OK) return st;
        if (rows <= n) {
            chosen = C;
            break;
        }
    }
    p.C = chosen;
    p.nsc = ((p.ns + chosen - 1) / chosen + 3) & ~3;   // a multiple of 4 segments per CTA
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

int32_t fs_max_vocab(void) { return FS_MAX_VOCAB; }

}  // extern "C"
