// Host-side launch planning shared by the entry points.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fs_device.cuh"
#include "fs_sampling.h"

namespace fsd {

// Cluster size, segments per CTA and shared-memory bytes of one launch.
struct Plan {
    int C;
    int nsc;
    int ns;
    size_t smem;
};

// Remember a CUDA error for fs_last_error_string() and turn it into a status.
fs_status cuda_fail(cudaError_t e);

// Number of SMs and the opt-in shared-memory limit of the current device.
fs_status device_limits(int& sm_count, size_t& smem_optin);

// Choose the cluster size for `rows` rows of `vocab` elements: enough CTAs to give
// every SM about two, at most MAX_CLUSTER per row and at least one segment each.
fs_status make_plan(int rows, int vocab, Plan& p);

// Opt the kernel into `smem` bytes of dynamic shared memory (once per device).
fs_status prepare_kernel(const void* fn, size_t smem);

template <typename Args>
fs_status launch_cluster(void (*kernel)(Args), const Plan& p, int rows, void* stream, const Args& a) {
    fs_status st = prepare_kernel(reinterpret_cast<const void*>(kernel), p.smem);
    if (st != FS_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(rows) * unsigned(p.C), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return cuda_fail(e);
    return FS_OK;
}

}  // namespace fsd
