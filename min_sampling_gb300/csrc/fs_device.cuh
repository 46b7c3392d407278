// Device building blocks shared by the sampling and filter kernels (sm_103a).
//
// Execution model: one thread-block cluster per row.  The C CTAs of a cluster
// split the row into contiguous ranges of SEG-element segments; every CTA streams
// its range from HBM exactly once (pass 1) and keeps, per segment, the maximum and
// the mass above the current lower pivot in shared memory.  Later work (rejection
// rounds, threshold searches) visits only the segments whose maximum can matter,
// re-reading them through L2, and switches to a compact in-shared-memory list of
// the surviving tokens as soon as it is small.  Cross-CTA reductions go through
// distributed shared memory (mapa + ld.shared::cluster) and hardware cluster
// barriers; every CTA of a cluster executes the same sequence of barriers because
// every branch that surrounds one depends only on cluster-wide reduced values.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fsd {

constexpr int NT = 512;                 // threads per CTA
constexpr int NW = NT / 32;             // warps per CTA
constexpr int SEG = 512;                // elements per segment
constexpr int SEG_IT = SEG / 128;       // warp iterations per segment (32 lanes x float4)
constexpr int CAP = 2048;               // compact-list capacity per row
constexpr int R_MAX = 256;              // rejection rounds before a row is invalid
constexpr int MAX_CLUSTER = 8;
constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------ shared layout

struct Slot {            // one cluster-exchange record (80 bytes)
    float f[8];
    uint32_t u[12];
};

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Byte offsets of the dynamic shared-memory carve-up.  `nsc` = segments per CTA,
// `ns` = segments per row (the whole row's segment maxima are gathered for the
// top-k lower bound).
struct Layout {
    size_t slot, gath, redf, redi, misc, segmax, mass0, mass1, mass2, off, lv, li, segall, total;
    __host__ __device__ Layout(int nsc, int ns) {
        size_t o = 0;
        slot = o;   o = align16(o + 2 * sizeof(Slot));
        gath = o;   o = align16(o + MAX_CLUSTER * sizeof(Slot));
        redf = o;   o = align16(o + NW * 4 * sizeof(float));
        redi = o;   o = align16(o + NW * 4 * sizeof(int));
        misc = o;   o = align16(o + 32 * sizeof(int));
        segmax = o; o = align16(o + size_t(nsc) * 4);
        mass0 = o;  o = align16(o + size_t(nsc) * 4);
        mass1 = o;  o = align16(o + size_t(nsc) * 4);
        mass2 = o;  o = align16(o + size_t(nsc) * 4);
        off = o;    o = align16(o + size_t(nsc + 1) * 4);
        lv = o;     o = align16(o + size_t(CAP) * 4);
        li = o;     o = align16(o + size_t(CAP) * 4);
        segall = o; o = align16(o + size_t(ns) * 4);
        total = o;
    }
};

extern __shared__ __align__(16) unsigned char smem_raw[];

struct Smem {
    Slot* slot;
    Slot* gath;
    float* redf;
    int* redi;
    int* misc;
    uint32_t* segkey;   // per-segment maximum order key
    float* mass[3];
    int* off;
    float* lv;
    int* li;
    uint32_t* segall;   // the whole row's segment keys (top-k lower bound)
    __device__ explicit Smem(const Layout& L) {
        slot = reinterpret_cast<Slot*>(smem_raw + L.slot);
        gath = reinterpret_cast<Slot*>(smem_raw + L.gath);
        redf = reinterpret_cast<float*>(smem_raw + L.redf);
        redi = reinterpret_cast<int*>(smem_raw + L.redi);
        misc = reinterpret_cast<int*>(smem_raw + L.misc);
        segkey = reinterpret_cast<uint32_t*>(smem_raw + L.segmax);
        mass[0] = reinterpret_cast<float*>(smem_raw + L.mass0);
        mass[1] = reinterpret_cast<float*>(smem_raw + L.mass1);
        mass[2] = reinterpret_cast<float*>(smem_raw + L.mass2);
        off = reinterpret_cast<int*>(smem_raw + L.off);
        lv = reinterpret_cast<float*>(smem_raw + L.lv);
        li = reinterpret_cast<int*>(smem_raw + L.li);
        segall = reinterpret_cast<uint32_t*>(smem_raw + L.segall);
    }
};

// ------------------------------------------------------------------ cluster PTX

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Hardware cluster barrier; release/acquire orders shared memory at cluster scope.
// All threads of all CTAs of the cluster must reach it (it also synchronises the CTA).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
    return __uint_as_float(ld_dsmem_u32(addr));
}

// ------------------------------------------------------------------ loads

// 16-byte read of row data; NC selects the read-only (non-coherent) path, which
// the samplers use (their input is never written during the kernel).  The filter
// kernels may run in place and use the coherent path.
template <bool NC>
__device__ __forceinline__ float4 ld_f4(const float* p) {
    float4 v;
    if (NC) {
        asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
            : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    } else {
        v = *reinterpret_cast<const float4*>(p);
    }
    return v;
}
template <bool NC>
__device__ __forceinline__ float ld_f1(const float* p) {
    float v;
    if (NC) {
        asm("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    } else {
        v = *p;
    }
    return v;
}

// The four elements [base, base+4) of a row; indices at or past V read as `fill`.
// VEC: the row start is 16-byte aligned and V % 4 == 0, so in-range quads are
// whole float4s.
template <bool VEC, bool NC>
__device__ __forceinline__ void load_quad(const float* __restrict__ row, int V, int base,
                                          float fill, float (&v)[4]) {
    if (VEC && base + 3 < V) {
        float4 f = ld_f4<NC>(row + base);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        return;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = (base + q < V) ? ld_f1<NC>(row + base + q) : fill;
}

// All SEG elements of segment s as seen by one lane: v[it][q] is element
// s*SEG + it*128 + lane*4 + q.
template <bool VEC, bool NC>
__device__ __forceinline__ void load_segment(const float* __restrict__ row, int V, int s, int lane,
                                             float fill, float (&v)[SEG_IT][4]) {
    const int base = s * SEG + lane * 4;
#pragma unroll
    for (int it = 0; it < SEG_IT; ++it) load_quad<VEC, NC>(row, V, base + it * 128, fill, v[it]);
}

// ------------------------------------------------------------------ warp helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
    return v;  // bitwise identical in every lane (each level adds a commuted pair)
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, m));
    return v;
}
__device__ __forceinline__ uint32_t warp_max_u(uint32_t v) {
#pragma unroll
    for (int m = 16; m; m >>= 1) v = max(v, __shfl_xor_sync(FULL, v, m));
    return v;
}
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        float o = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += o;
    }
    return v;
}
__device__ __forceinline__ int warp_incl_scan_i(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// Sum of a[0..n) in a fixed order (32-wide chunks, each tree-reduced, chunks added in
// order).  Warp-collective; the result is identical in all lanes.
__device__ __forceinline__ float ordered_sum(const float* a, int n, int lane) {
    float acc = 0.f;
    for (int base = 0; base < n; base += 32) {
        float v = (base + lane < n) ? a[base + lane] : 0.f;
        acc += warp_sum(v);
    }
    return acc;
}
__device__ __forceinline__ int ordered_sum_i(const int* a, int n, int lane) {
    int acc = 0;
    for (int base = 0; base < n; base += 32) acc += warp_sum_i((base + lane < n) ? a[base + lane] : 0);
    return acc;
}

// ------------------------------------------------------------------ keys

// Order key of a probability: its bit pattern when positive, 0 for +-0.  For
// non-negative floats the integer order of the bit pattern is the numeric order
// ([drill] section 3).
__device__ __forceinline__ uint32_t prob_key(float x) { return x > 0.f ? __float_as_uint(x) : 0u; }

// Order-preserving key of a signed float ([drill] section 8): negative patterns are
// flipped entirely, non-negative ones get their sign bit set.
__device__ __forceinline__ uint32_t logit_key(float x) {
    uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------------ Philox4x32-10

// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11:
// ten rounds of two 32x32->64 multiplies with a Weyl key schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k.x += W0; k.y += W1; }
        const uint32_t lo0 = M0 * c.x, hi0 = __umulhi(M0, c.x);
        const uint32_t lo1 = M1 * c.z, hi1 = __umulhi(M1, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    }
    return c;
}

// Uniform of output row `b`, round `r`: 24 random bits, exact in float32, in [0, 1).
__device__ __forceinline__ float sampler_uniform(unsigned long long seed, unsigned long long offset,
                                                 uint32_t b, uint32_t r) {
    const uint4 ctr = make_uint4(r, b, uint32_t(offset), uint32_t(offset >> 32));
    const uint2 key = make_uint2(uint32_t(seed), uint32_t(seed >> 32));
    return float(philox4x32_10(ctr, key).x >> 8) * 0x1p-24f;
}

// ------------------------------------------------------------------ cluster exchange

// Every CTA has filled slot[buf] (done by one thread before this call).  After the
// barrier, warp 0 copies the C slots into `gath` (rank order); the CTA barrier that
// follows makes them visible to every thread.
__device__ __forceinline__ void exchange(const Smem& sm, int buf, int C, int warp, int lane) {
    cluster_sync();
    if (warp == 0) {
        constexpr int WORDS = sizeof(Slot) / 4;
        for (int w = lane; w < C * WORDS; w += 32) {
            const int c = w / WORDS, o = w % WORDS;
            const uint32_t a = map_rank(smem_u32(reinterpret_cast<const uint32_t*>(&sm.slot[buf]) + o), c);
            reinterpret_cast<uint32_t*>(&sm.gath[c])[o] = ld_dsmem_u32(a);
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ draw inside a segment

// Inverse-transform locate inside one segment, warp-collective.  Eligible elements are
// x > low; `t` is the target measured from the segment start.  Returns the first
// eligible element whose running sum exceeds t; if rounding leaves none (t at or past
// the segment's computed mass), the last eligible element of the segment.  The
// segment must hold at least one eligible element.  ([blog] inverse transform and
// implementation details: a parallel float prefix sum need not be monotone, so the
// result is always forced onto an eligible token.)
template <bool VEC, bool NC>
__device__ __forceinline__ void locate_in_segment(const float* __restrict__ row, int V, int s, float low,
                                                  float t, int lane, int& j_out, float& x_out) {
    float run = 0.f;
    int last_j = -1;
    float last_x = 0.f;
    for (int it = 0; it < SEG_IT; ++it) {
        float v[4];
        const int base = s * SEG + it * 128 + lane * 4;
        load_quad<VEC, NC>(row, V, base, 0.f, v);
        float w[4];
        float lsum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[q] = v[q] > low ? v[q] : 0.f;
            lsum += w[q];
        }
        const bool any = (w[0] > 0.f) | (w[1] > 0.f) | (w[2] > 0.f) | (w[3] > 0.f);
        const float incl = warp_incl_scan(lsum, lane);
        const unsigned hit = __ballot_sync(FULL, any && (run + incl > t));
        const unsigned elig = __ballot_sync(FULL, any);
        if (elig) {
            const int l = 31 - __clz(elig);
            int lq = -1;
            float lx = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (w[q] > 0.f) { lq = q; lx = v[q]; }
            const int lq_l = __shfl_sync(FULL, lq, l);
            const float lx_l = __shfl_sync(FULL, lx, l);
            last_j = s * SEG + it * 128 + l * 4 + lq_l;
            last_x = lx_l;
        }
        if (hit) {
            const int l = __ffs(hit) - 1;
            int pq = -1, lastq = -1;
            float px = 0.f, lastx = 0.f;
            float acc = run + (incl - lsum);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (w[q] > 0.f) {
                    acc += w[q];
                    lastq = q;
                    lastx = v[q];
                    if (pq < 0 && acc > t) { pq = q; px = v[q]; }
                }
            }
            if (pq < 0) { pq = lastq; px = lastx; }
            j_out = s * SEG + it * 128 + l * 4 + __shfl_sync(FULL, pq, l);
            x_out = __shfl_sync(FULL, px, l);
            return;
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    j_out = last_j;
    x_out = last_x;
}

// Index of the first segment (0-based within the CTA) whose running mass over
// mass[0..n) exceeds t, with the mass before it in `before`; if none does, the last
// segment with positive mass (and `force_last` is set).  Warp-collective.
__device__ __forceinline__ int locate_segment(const float* mass, int n, float t, int lane,
                                              float& before, bool& force_last) {
    float run = 0.f;
    int last = -1;
    for (int base = 0; base < n; base += 32) {
        const float m = (base + lane < n) ? mass[base + lane] : 0.f;
        const float incl = warp_incl_scan(m, lane);
        const unsigned hit = __ballot_sync(FULL, m > 0.f && run + incl > t);
        const unsigned nz = __ballot_sync(FULL, m > 0.f);
        if (nz) last = base + 31 - __clz(nz);
        if (hit) {
            const int l = __ffs(hit) - 1;
            before = run + __shfl_sync(FULL, incl - m, l);
            force_last = false;
            return base + l;
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    before = 0.f;
    force_last = true;
    return last;
}

// Locate inside a compact list lv[0..n) (index order), eligible x > low.
__device__ __forceinline__ int locate_in_list(const float* lv, int n, float low, float t, int lane) {
    float run = 0.f;
    int last = -1;
    for (int base = 0; base < n; base += 128) {
        float w[4];
        float lsum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = base + lane * 4 + q;
            const float x = e < n ? lv[e] : 0.f;
            w[q] = x > low ? x : 0.f;
            lsum += w[q];
        }
        const bool any = (w[0] > 0.f) | (w[1] > 0.f) | (w[2] > 0.f) | (w[3] > 0.f);
        const float incl = warp_incl_scan(lsum, lane);
        const unsigned hit = __ballot_sync(FULL, any && (run + incl > t));
        const unsigned elig = __ballot_sync(FULL, any);
        if (elig) {
            const int l = 31 - __clz(elig);
            int lq = -1;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (w[q] > 0.f) lq = q;
            last = base + l * 4 + __shfl_sync(FULL, lq, l);
        }
        if (hit) {
            const int l = __ffs(hit) - 1;
            int pq = -1, lastq = -1;
            float acc = run + (incl - lsum);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (w[q] > 0.f) {
                    acc += w[q];
                    lastq = q;
                    if (pq < 0 && acc > t) pq = q;
                }
            }
            if (pq < 0) pq = lastq;
            return base + l * 4 + __shfl_sync(FULL, pq, l);
        }
        run += __shfl_sync(FULL, incl, 31);
    }
    return last;
}

// ------------------------------------------------------------------ compaction

// Collect, in index order, every element of this CTA's segments whose key is >= thr
// into lv/li (values and row indices).  KEYF maps a float to its order key.  Writes
// the local count to sm.misc[0] and returns it; nothing is written past CAP (the
// count is still exact, so the caller can see the overflow).  Block-collective.
template <bool VEC, bool NC, typename KEYF>
__device__ int compact_ge(const float* __restrict__ row, int V, int s0, int nsc, const uint32_t* segkey,
                          uint32_t thr, KEYF keyf, float fill, const Smem& sm, int warp, int lane, int tid) {
    // Phase A: per-segment counts.
    for (int ls = warp; ls < nsc; ls += NW) {
        int cnt = 0;
        if (segkey[ls] >= thr) {
            float v[SEG_IT][4];
            load_segment<VEC, NC>(row, V, s0 + ls, lane, fill, v);
#pragma unroll
            for (int it = 0; it < SEG_IT; ++it)
#pragma unroll
                for (int q = 0; q < 4; ++q) cnt += (keyf(v[it][q]) >= thr && s0 * SEG + ls * SEG + it * 128 + lane * 4 + q < V);
            cnt = warp_sum_i(cnt);
        }
        if (lane == 0) sm.off[ls] = cnt;
    }
    __syncthreads();
    // Exclusive scan of the counts in segment order.
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < nsc; base += 32) {
            const int c = (base + lane < nsc) ? sm.off[base + lane] : 0;
            const int incl = warp_incl_scan_i(c, lane);
            if (base + lane < nsc) sm.off[base + lane] = run + incl - c;
            run += __shfl_sync(FULL, incl, 31);
        }
        if (lane == 0) { sm.off[nsc] = run; sm.misc[0] = run; }
    }
    __syncthreads();
    const int total = sm.misc[0];
    // Phase B: ordered writes.
    for (int ls = warp; ls < nsc; ls += NW) {
        const int o0 = sm.off[ls], n = sm.off[ls + 1] - o0;
        if (n == 0) continue;
        float v[SEG_IT][4];
        load_segment<VEC, NC>(row, V, s0 + ls, lane, fill, v);
        int run = o0;
#pragma unroll
        for (int it = 0; it < SEG_IT; ++it) {
            const int base = (s0 + ls) * SEG + it * 128 + lane * 4;
            int c = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) c += (keyf(v[it][q]) >= thr && base + q < V);
            const int incl = warp_incl_scan_i(c, lane);
            int pos = run + incl - c;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (keyf(v[it][q]) >= thr && base + q < V) {
                    if (pos < CAP) { sm.lv[pos] = v[it][q]; sm.li[pos] = base + q; }
                    ++pos;
                }
            }
            run += __shfl_sync(FULL, incl, 31);
        }
    }
    __syncthreads();
    return total;
}

// Rank 0 appends the lists of ranks 1..C-1 after its own (counts from gath[].u[0]).
// Block-collective on rank 0; the caller guarantees the row total fits in CAP.
__device__ __forceinline__ void gather_lists(const Smem& sm, int C, int tid) {
    int offs = int(sm.gath[0].u[0]);
    for (int c = 1; c < C; ++c) {
        const int n = int(sm.gath[c].u[0]);
        const uint32_t rv = map_rank(smem_u32(sm.lv), c);
        const uint32_t ri = map_rank(smem_u32(sm.li), c);
        for (int e = tid; e < n && offs + e < CAP; e += NT) {
            sm.lv[offs + e] = ld_dsmem_f32(rv + 4u * e);
            sm.li[offs + e] = static_cast<int>(ld_dsmem_u32(ri + 4u * e));
        }
        offs += n;
    }
    __syncthreads();
}

// Largest key t among lv[0..n) with #{key >= t} >= k; 0 if no such key.
// Block-collective (rank counting; the list is small).
template <typename KEYF>
__device__ uint32_t kth_key_in_list(const Smem& sm, int n, int k, KEYF keyf, int warp, int lane, int tid) {
    uint32_t best = 0;
    for (int i = tid; i < n; i += NT) {
        const uint32_t ki = keyf(sm.lv[i]);
        int ge = 0;
        for (int j = 0; j < n; ++j) ge += (keyf(sm.lv[j]) >= ki);
        if (ge >= k) best = max(best, ki);
    }
    best = warp_max_u(best);
    if (lane == 0) sm.redi[warp] = static_cast<int>(best);
    __syncthreads();
    uint32_t r = 0;
    for (int w = 0; w < NW; ++w) r = max(r, static_cast<uint32_t>(sm.redi[w]));
    __syncthreads();
    return r;
}

// Largest key among a[0..n) (segment maxima) with #{>= it} >= k; 0 if none.
__device__ inline uint32_t kth_key_in_array(const uint32_t* a, int n, int k, const Smem& sm,
                                     int warp, int lane, int tid) {
    uint32_t best = 0;
    for (int i = tid; i < n; i += NT) {
        const uint32_t ki = a[i];
        int ge = 0;
        for (int j = 0; j < n; ++j) ge += (a[j] >= ki);
        if (ge >= k) best = max(best, ki);
    }
    best = warp_max_u(best);
    if (lane == 0) sm.redi[warp] = static_cast<int>(best);
    __syncthreads();
    uint32_t r = 0;
    for (int w = 0; w < NW; ++w) r = max(r, static_cast<uint32_t>(sm.redi[w]));
    __syncthreads();
    return r;
}

// Every CTA copies the segment keys of the whole row (rank order) into sm.segall.
// Must follow a cluster barrier after which no CTA changes its segkey array.
__device__ __forceinline__ void gather_segkeys(const Smem& sm, int nsc_max, int ns, int tid) {
    for (int s = tid; s < ns; s += NT) {
        const int c = s / nsc_max, ls = s % nsc_max;
        sm.segall[s] = ld_dsmem_u32(map_rank(smem_u32(sm.segkey + ls), c));
    }
    __syncthreads();
}

// ------------------------------------------------------------------ bisection

// Interval of a threshold search over order keys ([drill] sections 2-3: bisection on
// a monotone count or mass, done on the integer bit pattern so that it ends exactly
// on an existing value).  Invariant: crit(lo) holds, crit(hi) does not, where
// crit(t) = count(key >= t) >= k  or  mass(key >= t) >= target.  The answer is lo
// once hi = lo + 1.
struct Bisect {
    uint64_t lo, hi;
    int cnt_lo;       // count(key >= lo)
    float mass_lo;    // mass(key >= lo) (probabilities only)
};

// One pass over this CTA's segments with up to three pivots (several pivots per
// pass, as the drill page's section 5 describes for the production kernel).  For
// each pivot: count and (MASS) sum of elements with key >= pivot; for each of the
// four sub-intervals [lo,p0) [p0,p1) [p1,p2) [p2,hi): smallest and largest key
// present, so the next interval can shrink to the keys that exist (and the search
// stops when one distinct key is left).  Writes the CTA's record into slot[buf]
// (f[0..2] masses, u[0..2] counts, u[3..6] min keys, u[7..10] max keys).
template <bool VEC, bool NC, bool MASS, typename KEYF>
__device__ void bisect_pass(const float* __restrict__ row, int V, int s0, int nsc, const uint32_t* segkey,
                            const uint32_t (&piv)[3], uint64_t lo, uint64_t hi, KEYF keyf, float fill,
                            const Smem& sm, int buf, int warp, int lane, int tid) {
    float m[3] = {0.f, 0.f, 0.f};
    int c[3] = {0, 0, 0};
    uint32_t mn[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    uint32_t mx[4] = {0u, 0u, 0u, 0u};
    for (int ls = warp; ls < nsc; ls += NW) {
        if (uint64_t(segkey[ls]) < lo) continue;   // nothing at or above lo here
        float v[SEG_IT][4];
        load_segment<VEC, NC>(row, V, s0 + ls, lane, fill, v);
        const int base0 = (s0 + ls) * SEG + lane * 4;
#pragma unroll
        for (int it = 0; it < SEG_IT; ++it) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = v[it][q];
                const uint32_t key = keyf(x);
                const bool inr = base0 + it * 128 + q < V;
                const bool g0 = inr && key >= piv[0], g1 = inr && key >= piv[1], g2 = inr && key >= piv[2];
                if (MASS) {
                    m[0] += g0 ? x : 0.f;
                    m[1] += g1 ? x : 0.f;
                    m[2] += g2 ? x : 0.f;
                }
                c[0] += g0;
                c[1] += g1;
                c[2] += g2;
                const bool inlo = inr && uint64_t(key) >= lo && uint64_t(key) < hi;
                const int bkt = int(g0) + int(g1) + int(g2);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const bool sel = inlo && t == bkt;
                    mn[t] = sel ? min(mn[t], key) : mn[t];
                    mx[t] = sel ? max(mx[t], key) : mx[t];
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        m[i] = warp_sum(m[i]);
        c[i] = warp_sum_i(c[i]);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
#pragma unroll
        for (int d = 16; d; d >>= 1) {
            mn[t] = min(mn[t], __shfl_xor_sync(FULL, mn[t], d));
            mx[t] = max(mx[t], __shfl_xor_sync(FULL, mx[t], d));
        }
    }
    // Per-warp records in redf/redi (NW x 4 each): masses/counts, then min/max keys.
    if (lane == 0) {
        for (int i = 0; i < 3; ++i) { sm.redf[warp * 4 + i] = m[i]; sm.redi[warp * 4 + i] = c[i]; }
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) {
            float a = 0.f;
            uint32_t b = 0;
            for (int w = 0; w < NW; ++w) { a += sm.redf[w * 4 + i]; b += uint32_t(sm.redi[w * 4 + i]); }
            sm.slot[buf].f[i] = a;
            sm.slot[buf].u[i] = b;
        }
    }
    __syncthreads();
    if (lane == 0) {
        for (int t = 0; t < 4; ++t) {
            sm.redi[warp * 4 + t] = int(mn[t]);
            reinterpret_cast<uint32_t*>(sm.redf)[warp * 4 + t] = mx[t];
        }
    }
    __syncthreads();
    if (tid == 0) {
        for (int t = 0; t < 4; ++t) {
            uint32_t a = 0xffffffffu, b = 0u;
            for (int w = 0; w < NW; ++w) {
                a = min(a, uint32_t(sm.redi[w * 4 + t]));
                b = max(b, reinterpret_cast<const uint32_t*>(sm.redf)[w * 4 + t]);
            }
            sm.slot[buf].u[3 + t] = a;
            sm.slot[buf].u[7 + t] = b;
        }
    }
    // (the caller's exchange begins with a cluster barrier)
}

// Drive the search to the end: multi-pivot passes with a cluster-wide exchange after
// each.  All CTAs of the cluster call it with identical `st`; they leave it with
// identical results.  At most 40 passes (each removes at least a quarter of a
// non-empty key range, so the range of 2^32 keys is exhausted far earlier).
template <bool VEC, bool NC, bool MASS, typename KEYF>
__device__ void bisect_run(const float* __restrict__ row, int V, int s0, int nsc, const uint32_t* segkey,
                           Bisect& st, int kcrit, float target, KEYF keyf, float fill,
                           const Smem& sm, int& buf, int C, int warp, int lane, int tid) {
    for (int iter = 0; iter < 40 && st.hi - st.lo > 1; ++iter) {
        const uint64_t d = st.hi - st.lo;
        uint32_t piv[3];
        if (d >= 4) {
            for (int i = 0; i < 3; ++i) piv[i] = uint32_t(st.lo + (d * uint64_t(i + 1)) / 4);
        } else {
            piv[0] = uint32_t(st.lo + 1);
            piv[1] = uint32_t(d == 3 ? st.lo + 2 : st.hi);
            piv[2] = uint32_t(st.hi);
        }
        bisect_pass<VEC, NC, MASS>(row, V, s0, nsc, segkey, piv, st.lo, st.hi, keyf, fill, sm, buf,
                                   warp, lane, tid);
        exchange(sm, buf, C, warp, lane);
        buf ^= 1;
        float mass[3] = {0.f, 0.f, 0.f};
        int cnt[3] = {0, 0, 0};
        uint32_t kmin[4], kmax[4];
        for (int t = 0; t < 4; ++t) { kmin[t] = 0xffffffffu; kmax[t] = 0u; }
        for (int c = 0; c < C; ++c) {
            for (int i = 0; i < 3; ++i) {
                mass[i] += sm.gath[c].f[i];
                cnt[i] += int(sm.gath[c].u[i]);
            }
            for (int t = 0; t < 4; ++t) {
                kmin[t] = min(kmin[t], sm.gath[c].u[3 + t]);
                kmax[t] = max(kmax[t], sm.gath[c].u[7 + t]);
            }
        }
        // crit is monotone in the pivot: take the largest pivot where it holds.
        int best = -1;
        for (int i = 0; i < 3; ++i) {
            if (uint64_t(piv[i]) >= st.hi) break;
            const bool ok = MASS ? (mass[i] >= target) : (cnt[i] >= kcrit);
            if (ok) best = i;
        }
        uint64_t nlo = st.lo, nhi = st.hi;
        int bkt = 0;
        if (best >= 0) {
            nlo = piv[best];
            st.cnt_lo = cnt[best];
            st.mass_lo = mass[best];
            bkt = best + 1;
        }
        if (best + 1 < 3 && uint64_t(piv[best + 1]) < st.hi) nhi = piv[best + 1];
        if (kmin[bkt] <= kmax[bkt]) {            // keys present in the new interval
            nlo = max(nlo, uint64_t(kmin[bkt]));
            nhi = min(nhi, uint64_t(kmax[bkt]) + 1);
        }
        st.lo = nlo;
        st.hi = nhi;
        __syncthreads();   // gath is rewritten by the next exchange
    }
}

}  // namespace fsd
