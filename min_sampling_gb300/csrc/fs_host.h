// Host-side launch planning shared by the entry points.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fs_device.cuh"
#include "fs_sampling.h"

namespace fsd {

// Cluster size, segment geometry and shared-memory bytes of one launch.
struct Plan {
    int C;        // CTAs per row (cluster size)
    int shift;    // log2(blocks per segment)
    int ns;       // segments per row
    int nsc;      // segments per CTA
    size_t smem;  // dynamic shared memory per CTA (above the tables' need when it caps CTAs per SM)
    int per_sm;   // CTAs resident per SM at most
};

// Remember a CUDA error for fs_last_error_string() and turn it into a status.
fs_status cuda_fail(cudaError_t e);

// Set the text fs_last_error_string() returns to the calling host thread.
void set_last_error(const char* msg);

// Number of SMs and the opt-in shared-memory limit of the current device.
fs_status device_limits(int& sm_count, size_t& smem_optin);

// Choose the cluster size for `rows` rows of `vocab` elements so that the whole grid
// is resident at once (rows <= the device's resident clusters of that size for `fn`),
// with at most MAX_CLUSTER CTAs per row and at least four segments per CTA.
fs_status make_plan(int rows, int vocab, const void* fn, bool single_pass, Plan& p, bool topp_hist = false);

// The library's scratch buffer for the current device and `stream`, at least `bytes`
// long (allocated or grown on first need; see api.cu).
fs_status workspace(size_t bytes, void* stream, void** out);

// Bytes of scratch that the row summaries of `batch_in` rows of `vocab` values take
// (scan_kernel, sampling.cu); `codes`: with the joint order's run codes.
size_t scan_workspace_bytes(int batch_in, int vocab, bool codes);

// Opt the kernel into the device's maximum dynamic shared memory (once per device).
fs_status prepare_kernel(const void* fn);

template <typename Args>
fs_status launch_cluster(void (*kernel)(Args), const Plan& p, int rows, void* stream, const Args& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(rows) * unsigned(p.C), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the grid may be scheduled while the previous
    // kernel of the stream is still finishing; the kernel waits for that kernel's
    // completion (griddepcontrol.wait) before it touches global memory.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return cuda_fail(e);
    return FS_OK;
}

}  // namespace fsd
