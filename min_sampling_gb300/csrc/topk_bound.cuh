// Lower bound of the k-th largest value of a row from its segment maxima (leader).
#pragma once

#include "fs_device.cuh"

namespace fsd {

// Leader, block-collective: a lower bound L0 <= t_k of the row's k-th largest order key,
// from the segment maxima segkey[0..ns).  A histogram of the top bits of the keys
// (key >> bshift, 1024 bins) is scanned from the top bin down; the bin in which the
// count of segment maxima reaches k holds the k-th largest segment maximum, and its
// lower edge is at most that value.  The k-th largest of any subset of the row (here:
// the segment maxima) is at most the row's own k-th largest, so L0 <= t_k.  Every
// segment holding an element >= t_k then has its maximum >= L0.  Returns 0 when the
// row has fewer than k segments.  Uses lv as scratch.
FS_NOINLINE __device__ inline uint32_t topk_bound(const Smem& sm, int ns, int k, int bshift, int warp, int lane,
                                                  int tid) {
    if (ns < k) return 0;
    uint32_t* hist = reinterpret_cast<uint32_t*>(sm.lv);  // 1024 bins
    for (int i = tid; i < 1024; i += NT) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < ns; i += NT) atomicAdd(&hist[min(1023u, sm.segkey[i] >> bshift)], 1u);
    __syncthreads();
    // Thread t owns positions 4t..4t+3 counted from the top bin (bins 1023 - pos).
    uint32_t c[4];
    uint32_t own = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        c[q] = hist[1023 - (4 * tid + q)];
        own += c[q];
    }
    uint32_t incl = own;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) sm.red[warp] = int(incl);
    __syncthreads();
    uint32_t before = incl - own;
    for (int w = 0; w < warp; ++w) before += uint32_t(sm.red[w]);
    const uint32_t kk = uint32_t(k);
    if (before < kk && before + own >= kk) {
        uint32_t cum = before;
        int pos = 4 * tid;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            cum += c[q];
            if (cum >= kk) {
                pos = 4 * tid + q;
                break;
            }
        }
        sm.red[NW] = 1023 - pos;
    }
    __syncthreads();
    const uint32_t bin = uint32_t(sm.red[NW]);
    __syncthreads();
    return bin << bshift;
}

}  // namespace fsd
